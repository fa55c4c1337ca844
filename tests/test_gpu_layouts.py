"""Layout variants on the GPU against the oracle: FWHT block sizes 64 and 256,
a scale per 256 weights, and the residual two-pass ternarisation -- through
the C ABI (tq_fwht, tq_quantize_pack_layout, tq_gemv_layout, tq_gemm_layout)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import ternary_weight_fwht128_gb300 as tq
from ternary_weight_fwht128_gb300 import synth
from tq_testutil import check_y, guarded, to_dev_bf16, to_dev_f32, u16

pytestmark = pytest.mark.gpu

LAYOUTS = [(64, 128, False), (256, 128, False), (128, 256, False), (256, 256, False), (128, 128, True),
           (64, 256, True), (256, 128, True)]
IDS = [f"b{b}-g{g}{'-res' if r else ''}" for b, g, r in LAYOUTS]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def lor(orc):
    return oracle.LayoutOracle(orc)


@pytest.mark.parametrize("block", [64, 256])
@pytest.mark.parametrize("rows,K", [(1, 256), (37, 768), (3, 27648)])
def test_fwht_block_bitexact(lor, block, rows, K):
    rng = np.random.default_rng(rows * 7 + K + block)
    x = (rng.standard_normal((rows, K)) * rng.uniform(0.01, 30, size=(rows, 1))).astype(np.float32)
    ref = lor.fwht_f32(block, x)
    out, check = guarded((rows, K), torch.float32)
    tq.fwht(to_dev_f32(x), block, out=out)
    torch.cuda.synchronize()
    check()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    xb = synth.activations(rows, K, 5)
    refb = lor.fwht_f32(block, synth.bf16_bits_to_f32(xb))
    assert np.array_equal(u16(tq.fwht(to_dev_bf16(xb), block, out_dtype=torch.float16)),
                          refb.astype(np.float16).view(np.uint16))
    assert np.array_equal(u16(tq.fwht(to_dev_bf16(xb), block, out_dtype=torch.bfloat16)),
                          synth.f32_to_bf16_bits(refb))


def _quant_layout_check(lor, orc, W, lay_t, rows=None):
    b, g, res = lay_t
    lay = tq.layout(b, g, res)
    dev = to_dev_f32(W) if W.dtype == np.float32 else to_dev_bf16(W)
    c2, c3, s = tq.quantize_pack_layout(dev, lay, tq.TQ_PACK_BOTH)
    T, S = lor.quantize(W, b, g, res, rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    assert np.array_equal(u16(s[sel]), S), "scales differ"
    assert np.array_equal(c2[sel].cpu().numpy(), orc.pack2(T)), "2-bit codes differ"
    assert np.array_equal(c3[sel].cpu().numpy(), orc.pack3(T)), "base-3 codes differ"
    return c2, c3, s, T, S


@pytest.mark.parametrize("lay_t", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("N,K,dtype", [(37, 768, "f32"), (5, 5120, "bf16"), (3, 27648, "bf16")])
def test_quantize_layout_bitexact(lor, orc, lay_t, N, K, dtype):
    W = synth.weights(N, K, N + K + lay_t[0], dtype=dtype)
    _quant_layout_check(lor, orc, W, lay_t)


@pytest.mark.parametrize("lay_t", LAYOUTS, ids=IDS)
def test_quantize_layout_special_rows(lor, orc, lay_t):
    """Zero groups, fp16-underflowing groups, overflowing groups (s = inf),
    unit rows (rows of H)."""
    K = 512
    W = np.zeros((6, K), dtype=np.float32)
    W[1, :256] = 1e-9
    W[2, 256:] = 1e6
    W[3, 5] = 1.0
    W[4, 300] = -2.0
    W[5] = np.linspace(-1, 1, K, dtype=np.float32)
    _quant_layout_check(lor, orc, W, lay_t)


def test_layout_default_equals_plain(orc):
    """{128, 128, 0} through the layout entry points is the plain path."""
    N, K, M = 300, 1280, 2
    W = synth.weights(N, K, 3, dtype="bf16")
    c2, c3, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_BOTH)
    d2, d3, ds = tq.quantize_pack_layout(to_dev_bf16(W), tq.layout(), tq.TQ_PACK_BOTH)
    assert torch.equal(c2, d2) and torch.equal(c3, d3) and torch.equal(s, ds)
    x = to_dev_bf16(synth.activations(M, K, 4))
    assert torch.equal(tq.gemv(c2, s, x, K), tq.gemv_layout(c2, s, x, K, tq.layout()))


def _gemv_layout_case(lor, N, K, M, lay_t, fmt, seed, rows=None):
    b, g, res = lay_t
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    c2, c3, s = tq.quantize_pack_layout(to_dev_bf16(W), tq.layout(b, g, res), fmt)
    codes = c2 if fmt == tq.TQ_PACK_2BIT else c3
    out, check = guarded((M, N), torch.float32)
    tq.gemv_layout(codes, s, to_dev_bf16(xb), K, tq.layout(b, g, res), fmt, out=out)
    torch.cuda.synchronize()
    check()
    tq.device_fault()
    T, S = lor.quantize(W, b, g, res, rows)
    ref = lor.gemv(T, S, synth.bf16_bits_to_f32(xb), b, g, res)
    got = out.cpu().numpy()
    if rows is not None:
        got = got[:, rows]
    return check_y(got, ref)


@pytest.mark.parametrize("lay_t", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("fmt", [tq.TQ_PACK_2BIT, tq.TQ_PACK_BASE3], ids=["2bit", "base3"])
@pytest.mark.parametrize("N,K,M", [(300, 1280, 1), (513, 2560, 4), (200, 768, 16)])
def test_gemv_layout(lor, lay_t, fmt, N, K, M):
    _gemv_layout_case(lor, N, K, M, lay_t, fmt, seed=N + K + M)


@pytest.mark.parametrize("lay_t", [(128, 128, True), (256, 256, False), (64, 128, True)],
                         ids=["b128-g128-res", "b256-g256", "b64-g128-res"])
@pytest.mark.parametrize("fmt", [tq.TQ_PACK_2BIT, tq.TQ_PACK_BASE3], ids=["2bit", "base3"])
@pytest.mark.parametrize("N,K,M", [(27648, 5120, 1), (5120, 27648, 1), (27648, 5120, 8)])
def test_gemv_layout_full_size_sampled(lor, lay_t, fmt, N, K, M):
    rows = np.sort(np.random.default_rng(N + K + M).choice(N, size=40, replace=False))
    rows[-1] = N - 1
    _gemv_layout_case(lor, N, K, M, lay_t, fmt, seed=N + K + M + 9, rows=rows)


def _gemm_layout_case(lor, N, K, M, lay_t, seed, rows=None, out_rows=None):
    b, g, res = lay_t
    lay = tq.layout(b, g, res)
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    c2, _, s = tq.quantize_pack_layout(to_dev_bf16(W), lay, tq.TQ_PACK_2BIT)
    ws = torch.empty(tq.gemm_workspace_bytes_layout(M, K, lay), dtype=torch.uint8, device="cuda")
    out, check = guarded((M, N), torch.float32)
    tq.gemm_layout(c2, s, to_dev_bf16(xb), K, lay, workspace=ws, out=out)
    torch.cuda.synchronize()
    check()
    tq.gemm_check_range(ws)
    T, S = lor.quantize(W, b, g, res, rows)
    xs = synth.bf16_bits_to_f32(xb)
    if out_rows is not None:
        xs = xs[out_rows]
    ref = lor.gemv(T, S, xs, b, g, res)
    got = out.cpu().numpy()
    if out_rows is not None:
        got = got[out_rows]
    if rows is not None:
        got = got[:, rows]
    return check_y(got, ref, "gemm y")


@pytest.mark.parametrize("lay_t", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("N,K,M", [(256, 256, 256), (513, 1280, 300)])
def test_gemm_layout(lor, lay_t, N, K, M):
    _gemm_layout_case(lor, N, K, M, lay_t, seed=N + K + M)


@pytest.mark.parametrize("lay_t", [(128, 128, True), (256, 256, False)], ids=["b128-g128-res", "b256-g256"])
def test_gemm_layout_full_size_sampled(lor, lay_t):
    N, K, M = 5120, 5120, 2048
    rng = np.random.default_rng(17)
    rows = np.sort(rng.choice(N, size=24, replace=False))
    out_rows = np.sort(rng.choice(M, size=16, replace=False))
    _gemm_layout_case(lor, N, K, M, lay_t, seed=99, rows=rows, out_rows=out_rows)


def test_gemm_layout_reuse_rotated(lor):
    """With a residual layout the workspace holds x' and x; a second call on
    the same workspace may skip the pre-pass."""
    N, K, M = 512, 1280, 256
    lay = tq.layout(128, 128, True)
    W = synth.weights(N, K, 5, dtype="bf16")
    c2, _, s = tq.quantize_pack_layout(to_dev_bf16(W), lay, tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K, 6))
    ws = torch.empty(tq.gemm_workspace_bytes_layout(M, K, lay), dtype=torch.uint8, device="cuda")
    y0 = tq.gemm_layout(c2, s, x, K, lay, workspace=ws)
    y1 = tq.gemm_layout(c2, s, torch.zeros_like(x), K, lay, workspace=ws, flags=tq.TQ_GEMM_REUSE_ROTATED)
    assert torch.equal(y0, y1)
