"""The 2:4-sparse ternary format on the GPU against the oracle (mhpq.cn/news/
1159370 sec. 1.2), through the C ABI: tq_quantize_pack_sparse24 (codes and
scales bit-exact) and tq_gemv_sparse24 (y within the float tolerance)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import ternary_weight_fwht128_gb300 as tq
from ternary_weight_fwht128_gb300 import synth
from tq_testutil import check_y, guarded, to_dev_bf16, to_dev_f32, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def sp(orc):
    return oracle.Sparse24Oracle(orc)


def _dev(W):
    return to_dev_f32(W) if W.dtype == np.float32 else to_dev_bf16(W)


def _quant_check(sp, W, rows=None):
    N, K = W.shape
    codes, check_c = guarded((N, tq.sparse24_ld(K)), torch.uint8)
    scales, check_s = guarded((N, K // 128), torch.int16)
    tq.quantize_pack_sparse24(_dev(W), out=(codes, scales))
    torch.cuda.synchronize()
    check_c()
    check_s()
    T, KEEP, S = sp.quantize(W, rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    assert np.array_equal(u16(scales[sel]), S), "scales differ"
    assert np.array_equal(codes[sel].cpu().numpy(), sp.pack(T, KEEP)), "codes differ"
    return codes, scales


@pytest.mark.parametrize("N,K,dtype", [(1, 128, "f32"), (37, 768, "f32"), (300, 1280, "bf16"),
                                       (5, 27648, "bf16")])
def test_quantize_sparse24_bitexact(sp, N, K, dtype):
    W = synth.weights(N, K, N + K, dtype=dtype)
    _quant_check(sp, W)


@pytest.mark.parametrize("N,K", [(27648, 5120), (5120, 27648)])
def test_quantize_sparse24_full_layer_sampled(sp, N, K):
    """A full 27B-class layer, bf16 ~N(0, 0.02) with 0.1% outliers x20; the
    oracle checks 1% of the rows (first and last included)."""
    W = synth.weights(N, K, 7 + N, dtype="bf16")
    rows = np.sort(np.random.default_rng(N).choice(N, size=max(N // 100, 8), replace=False))
    rows[0], rows[-1] = 0, N - 1
    _quant_check(sp, W, rows)


def test_quantize_sparse24_special_rows(sp):
    """Zero groups (pattern (0,1) by the tie rule, scale 0), groups whose
    mean underflows fp16, overflowing groups (scale inf: trits 0), unit rows,
    all-equal quads (ties), and integer-valued rows (many ties)."""
    K = 512
    W = np.zeros((8, K), dtype=np.float32)
    W[1, :256] = 1e-9
    W[2, 256:] = 1e6
    W[3, 5] = 1.0
    W[4, 300] = -2.0
    W[5] = np.linspace(-1, 1, K, dtype=np.float32)
    W[6] = np.tile(np.array([1.0, -1.0, 1.0, -1.0], dtype=np.float32), K // 4)
    W[7] = np.random.default_rng(3).integers(-2, 3, size=K).astype(np.float32)
    _quant_check(sp, W)


def test_quantize_sparse24_codes_valid(sp):
    """The codes equal the oracle's, whose masks keep two of every four."""
    W = synth.weights(64, 1280, 11, dtype="bf16")
    codes, _ = tq.quantize_pack_sparse24(_dev(W))
    T, KEEP, _ = sp.quantize(W)
    assert np.all(KEEP.reshape(-1, 4).sum(1) == 2)
    assert np.array_equal(codes.cpu().numpy(), sp.pack(T, KEEP))


def _oracle_codes(sp, W, rows, codes, scales):
    """The oracle's codes and scales of W (rows: a sample); the GPU's, which
    the kernels under test read, must equal them bit for bit."""
    T, KEEP, S = sp.quantize(W, rows)
    c = sp.pack(T, KEEP)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    assert np.array_equal(codes[sel].cpu().numpy(), c) and np.array_equal(u16(scales[sel]), S)
    return c, S


def _gemv_case(sp, N, K, M, seed, rows=None):
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    out, check = guarded((M, N), torch.float32)
    y = tq.gemv_sparse24(codes, scales, to_dev_bf16(xb), K, out=out)
    torch.cuda.synchronize()
    check()
    c, S = _oracle_codes(sp, W, rows, codes, scales)
    ref = sp.gemv(c, S, synth.bf16_bits_to_f32(xb), K)
    got = out.cpu().numpy() if rows is None else out.cpu().numpy()[:, rows]
    check_y(got, ref)
    return codes, scales, to_dev_bf16(xb), y


@pytest.mark.parametrize("N,K,M", [(256, 256, 1), (300, 1280, 1), (33, 384, 3), (200, 768, 16), (1, 128, 2),
                                   (513, 2560, 5)])
def test_gemv_sparse24(sp, N, K, M):
    _gemv_case(sp, N, K, M, seed=N + 3 * K + M)


@pytest.mark.parametrize("N,K,M", [(27648, 5120, 1), (5120, 27648, 1), (5120, 27648, 16), (27648, 5120, 8)])
def test_gemv_sparse24_full_size_sampled(sp, N, K, M):
    """Bench shapes (K split into slices for 27648 and M > 1); the oracle
    checks 64 sampled rows (last row included)."""
    rows = np.sort(np.random.default_rng(N + K + M).choice(N, size=64, replace=False))
    rows[-1] = N - 1
    _gemv_case(sp, N, K, M, seed=N + K + M + 5, rows=rows)


def test_gemv_sparse24_path():
    """The tensor-memory kernel takes the shapes whose rows hold an even number
    (at least four) of groups; the others go to the CUDA-core kernel."""
    TM, CC = tq.TQ_GEMV_TENSOR_MEMORY, tq.TQ_GEMV_CUDA_CORES
    for N, K, M in [(27648, 5120, 1), (5120, 27648, 1), (5120, 27648, 16), (27648, 5120, 8), (300, 1280, 1),
                    (200, 768, 16), (1, 512, 1)]:
        assert tq.gemv_sparse24_path(N, K, M) == TM, (N, K, M)
    for N, K, M in [(256, 256, 1), (33, 384, 3), (1, 128, 2), (513, 2560 - 128, 1)]:
        assert tq.gemv_sparse24_path(N, K, M) == CC, (N, K, M)


@pytest.mark.parametrize("N,K,M", [(1000, 2560, 1), (4096, 5120, 2), (300, 6912, 7), (129, 512, 16)])
def test_gemv_sparse24_both_kernels(sp, N, K, M):
    """The same shape through both kernels: codes at the packed pitch (the
    tensor-memory kernel) and at a pitch 4 bytes longer (not a multiple of 16:
    the CUDA-core kernel); both within the tolerance of the oracle."""
    W = synth.weights(N, K, N + K + M + 9, dtype="bf16")
    xb = synth.activations(M, K, N + K + M + 10)
    ld = tq.sparse24_ld(K)
    wide = torch.zeros((N, ld + 4), dtype=torch.uint8, device="cuda")
    codes_a, scales = tq.quantize_pack_sparse24(_dev(W))
    codes_b = wide[:, :ld]
    scales_b = torch.empty_like(scales)
    tq.quantize_pack_sparse24(_dev(W), out=(codes_b, scales_b))
    assert tq.gemv_sparse24_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY
    c, S = _oracle_codes(sp, W, None, codes_a, scales)
    assert np.array_equal(codes_b.cpu().numpy(), c)
    ref = sp.gemv(c, S, synth.bf16_bits_to_f32(xb), K)
    x = to_dev_bf16(xb)
    ya = tq.gemv_sparse24(codes_a, scales, x, K)
    yb = tq.gemv_sparse24(codes_b, scales_b, x, K)
    torch.cuda.synchronize()
    check_y(ya.cpu().numpy(), ref, "tensor-memory kernel")
    check_y(yb.cpu().numpy(), ref, "CUDA-core kernel")


def test_gemv_sparse24_tensor_memory_repeatable():
    N, K, M = 27648, 5120, 1
    W = synth.weights(N, K, 19, dtype="bf16")
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    x = to_dev_bf16(synth.activations(M, K, 20))
    assert tq.gemv_sparse24_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY
    ys = [tq.gemv_sparse24(codes, scales, x, K) for _ in range(20)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_gemv_sparse24_repeatable():
    N, K, M = 5120, 27648, 4
    W = synth.weights(N, K, 17, dtype="bf16")
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    x = to_dev_bf16(synth.activations(M, K, 18))
    ys = [tq.gemv_sparse24(codes, scales, x, K) for _ in range(20)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_gemv_sparse24_invalid_codes_read_as_zero(sp):
    """Quads whose code is 54..63 contribute nothing (documented behaviour):
    the oracle's codes with one quad set to code 63, on both sides."""
    N, K, M = 64, 256, 2
    W = synth.weights(N, K, 21, dtype="bf16")
    T0, KEEP0, S = sp.quantize(W)
    c = sp.pack(T0, KEEP0).copy()
    c[5, 0] |= 0x0F   # quad 0 of row 5: low nibble 15 ...
    c[5, 16] |= 0x03  # ... and high bits 3: code 63
    xb = synth.activations(M, K, 22)
    scales = torch.from_numpy(S.view(np.int16)).cuda()
    y = tq.gemv_sparse24(torch.from_numpy(c).cuda(), scales, to_dev_bf16(xb), K)
    T, KEEP, bad = sp.unpack(c, K)
    assert bad == 1
    ref = oracle.load().gemv(T, S, synth.bf16_bits_to_f32(xb))
    check_y(y.cpu().numpy(), ref)


def test_gemv_sparse24_workspace_too_small():
    N, K, M = 64, 256, 1
    W = synth.weights(N, K, 23, dtype="bf16")
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    x = to_dev_bf16(synth.activations(M, K, 24))
    ws = torch.empty(tq.gemv_sparse24_workspace_bytes(N, K, M) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.gemv_sparse24(codes, scales, x, K, workspace=ws)
    assert e.value.status == tq.TQ_ERR_SHAPE


def test_gemv_sparse24_empty():
    K = 256
    codes = torch.empty((0, tq.sparse24_ld(K)), dtype=torch.uint8, device="cuda")
    scales = torch.empty((0, 2), dtype=torch.int16, device="cuda")
    x = to_dev_bf16(synth.activations(1, K, 1))
    y = tq.gemv_sparse24(codes, scales, x, K)
    assert y.shape == (1, 0)


def _gemm_case(sp, N, K, M, seed, rows=None):
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    out, check = guarded((M, N), torch.float32)
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    tq.gemm_sparse24(codes, scales, to_dev_bf16(xb), K, workspace=ws, out=out)
    torch.cuda.synchronize()
    check()
    tq.gemm_check_range(ws)
    c, S = _oracle_codes(sp, W, rows, codes, scales)
    ref = sp.gemv(c, S, synth.bf16_bits_to_f32(xb), K)
    got = out.cpu().numpy() if rows is None else out.cpu().numpy()[:, rows]
    check_y(got, ref)
    return codes, scales


@pytest.mark.parametrize("N,K,M", [(256, 256, 1), (300, 1280, 200), (513, 2560, 300), (64, 128, 1000)])
def test_gemm_sparse24(sp, N, K, M):
    _gemm_case(sp, N, K, M, seed=N + K + M + 1)


@pytest.mark.parametrize("N,K", [(5120, 5120), (27648, 5120), (5120, 27648)])
def test_gemm_sparse24_full_size_sampled(sp, N, K):
    """Prefill M = 2048 on the bench shapes; the oracle checks 24 sampled
    weight rows (last included) for all 2048 tokens."""
    rows = np.sort(np.random.default_rng(N + K).choice(N, size=24, replace=False))
    rows[-1] = N - 1
    _gemm_case(sp, N, K, 2048, seed=N + K + 13, rows=rows)


def test_gemm_sparse24_repeatable_and_gemv_agree(sp):
    """Repeated prefill calls give identical bits; the GEMM (fp16 x') and the
    GEMV (fp32 x') on the same skinny input are both within the tolerance of
    the oracle."""
    N, K, M = 1000, 2560, 8
    W = synth.weights(N, K, 31, dtype="bf16")
    xb = synth.activations(M, K, 32)
    codes, scales = tq.quantize_pack_sparse24(_dev(W))
    x = to_dev_bf16(xb)
    ys = [tq.gemm_sparse24(codes, scales, x, K) for _ in range(5)]
    yv = tq.gemv_sparse24(codes, scales, x, K)
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    c, S = _oracle_codes(sp, W, None, codes, scales)
    ref = sp.gemv(c, S, synth.bf16_bits_to_f32(xb), K)
    check_y(ys[0].cpu().numpy(), ref, "gemm")
    check_y(yv.cpu().numpy(), ref, "gemv")
