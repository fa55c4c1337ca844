"""CUDA path against the CPU oracle, through the C ABI (needs a GB300)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


# ------------------------------------------------------------------ FWHT

@pytest.mark.parametrize("rows,K", [(1, 128), (37, 384), (5, 5120), (3, 27648)])
def test_fwht_f32_bitexact(orc, rows, K):
    rng = np.random.default_rng(rows * 1000 + K)
    x = (rng.standard_normal((rows, K)) * rng.uniform(0.01, 30, size=(rows, 1))).astype(np.float32)
    ref = orc.fwht128_f32(x)
    out, check = guarded((rows, K), torch.float32)
    tq.fwht128(to_dev_f32(x), out=out)
    torch.cuda.synchronize()
    check()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_fwht_bf16_input_all_outputs(orc, out_dtype):
    xb = synth.activations(19, 1024, 7)
    ref = orc.fwht128_f32(synth.bf16_bits_to_f32(xb))
    got = tq.fwht128(to_dev_bf16(xb), out_dtype=out_dtype)
    if out_dtype == torch.float32:
        assert np.array_equal(got.cpu().numpy(), ref)
    elif out_dtype == torch.bfloat16:
        assert np.array_equal(u16(got), synth.f32_to_bf16_bits(ref))
    else:
        assert np.array_equal(u16(got), ref.astype(np.float16).view(np.uint16))


def test_fwht_in_place_and_strided(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 640)).astype(np.float32)
    ref = orc.fwht128_f32(x[:, :512])
    t = to_dev_f32(x)
    sub = t[:, :512]  # ld 640, K 512
    tq.fwht128(sub, out=sub)
    got = t.cpu().numpy()
    assert np.array_equal(got[:, :512], ref)
    assert np.array_equal(got[:, 512:], x[:, 512:])  # untouched tail of each row


def test_fwht_delta_rows(orc):
    x = np.zeros((128, 128), dtype=np.float32)
    x[np.arange(128), np.arange(128)] = 1.0
    got = tq.fwht128(to_dev_f32(x)).cpu().numpy()
    assert np.array_equal(got, orc.fwht128_f32(x))


# ------------------------------------------------------------- quantise

def _quant_check(orc, W, fmt=tq.TQ_PACK_BOTH, rows=None):
    dev = to_dev_f32(W) if W.dtype == np.float32 else to_dev_bf16(W)
    c2, c3, s = tq.quantize_pack(dev, fmt)
    T, S = orc.quantize(W, rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    assert np.array_equal(u16(s[sel]), S), "scales differ"
    K = W.shape[1]
    if c2 is not None:
        assert np.array_equal(c2[sel].cpu().numpy(), orc.pack2(T)), "2-bit codes differ"
    if c3 is not None:
        assert np.array_equal(c3[sel].cpu().numpy(), orc.pack3(T)), "base-3 codes differ"
    return c2, c3, s, T, S


def test_quantize_tiny_config(orc):
    W, _ = synth.tiny_config()
    _quant_check(orc, W)


@pytest.mark.parametrize("N,K,dtype,fmt", [
    (37, 384, "f32", tq.TQ_PACK_BOTH),
    (1, 128, "bf16", tq.TQ_PACK_2BIT),
    (3, 768, "bf16", tq.TQ_PACK_BASE3),   # six groups: a segment of five plus one
    (65, 5120, "bf16", tq.TQ_PACK_BOTH),
    (7, 27648, "bf16", tq.TQ_PACK_BOTH),  # 216 groups, last base-3 byte padded
])
def test_quantize_shapes(orc, N, K, dtype, fmt):
    W = synth.weights(N, K, N + K, dtype=dtype)
    _quant_check(orc, W, fmt)


@pytest.mark.parametrize("N,K", [(27648, 5120), (5120, 27648)])
def test_quantize_full_layer_sweep_shapes(orc, N, K):
    """The offline sweep's two large shapes at full size, in the launch
    configuration the sweep uses (2-bit and base-3 in one pass), with bf16
    weights ~N(0, 0.02) and 0.1 % of the entries (chosen without
    replacement) x20: one whole layer is compared bit for bit with the
    oracle, then 1 % of the rows of two further seeded layers."""
    W = synth.weights(N, K, 9000 + N + K, dtype="bf16")
    _quant_check(orc, W)
    del W
    for layer in (1, 2):
        W = synth.weights(N, K, 9000 + N + K + layer, dtype="bf16")
        rng = np.random.default_rng(layer * 7 + N)
        rows = np.sort(rng.choice(N, size=N // 100, replace=False))
        rows[-1] = N - 1
        _quant_check(orc, W, rows=rows)
        del W


def test_quantize_special_groups(orc):
    """All-zero groups (scale 0), tiny groups (fp16 underflow -> scale 0),
    huge groups (scale inf -> trits 0), delta rows (rows of H)."""
    K = 512
    W = np.zeros((6, K), dtype=np.float32)
    W[1, :128] = 1e-9
    W[2, 128:256] = 3e6
    W[3, 5] = 1.0
    W[3, 300] = -2.0
    W[4] = np.linspace(-1, 1, K, dtype=np.float32)
    W[5, ::2] = 0.25
    _quant_check(orc, W)


def test_quantize_guard_bytes(orc):
    N, K = 33, 640
    W = synth.weights(N, K, 5, dtype="bf16")
    c2, ck2 = guarded((N, K // 4), torch.uint8)
    ld3 = tq.packed_ld(K, tq.TQ_PACK_BASE3)
    c3, ck3 = guarded((N, ld3), torch.uint8)
    s, cks = guarded((N, K // 128), torch.int16)
    st = tq.lib().tq_quantize_pack(to_dev_bf16(W).data_ptr(), tq.TQ_BF16, N, K, K, tq.TQ_PACK_BOTH,
                                   c2.data_ptr(), K // 4, c3.data_ptr(), ld3, s.data_ptr(), K // 128,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == tq.TQ_OK
    torch.cuda.synchronize()
    ck2(); ck3(); cks()
    T, S = orc.quantize(W)
    assert np.array_equal(c2.cpu().numpy(), orc.pack2(T))
    assert np.array_equal(c3.cpu().numpy(), orc.pack3(T))


@pytest.mark.parametrize("extra", [3, 16])
def test_quantize_base3_row_pitch(orc, extra):
    """Base-3 rows with a pitch past the padded length: 4-byte stores where
    the pitch allows them (extra = 16), byte stores otherwise (extra = 3).
    Bytes up to the padded length match the oracle; the rest of each row
    keeps its poison."""
    N, K = 37, 1920  # 384 base-3 bytes per row: three units of 128
    W = synth.weights(N, K, 91, dtype="bf16")
    ld3min = tq.packed_ld(K, tq.TQ_PACK_BASE3)
    ld3 = ld3min + extra
    c3, ck3 = guarded((N, ld3), torch.uint8)
    s = torch.empty(N, K // 128, dtype=torch.int16, device="cuda")
    st = tq.lib().tq_quantize_pack(to_dev_bf16(W).data_ptr(), tq.TQ_BF16, N, K, K, tq.TQ_PACK_BASE3,
                                   None, 0, c3.data_ptr(), ld3, s.data_ptr(), K // 128,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == tq.TQ_OK
    torch.cuda.synchronize()
    ck3()
    got = c3.cpu().numpy()
    T, _ = orc.quantize(W)
    assert np.array_equal(got[:, :ld3min], orc.pack3(T))
    assert np.all(got[:, ld3min:] == 0x5A), "write past the padded row"


# ----------------------------------------------------------------- GEMV

def _gemv_case(orc, N, K, M, seed, fmt=tq.TQ_PACK_2BIT, rows=None):
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    c2, c3, s = tq.quantize_pack(to_dev_bf16(W), fmt)
    codes = c2 if fmt == tq.TQ_PACK_2BIT else c3
    out, check = guarded((M, N), torch.float32)
    tq.gemv(codes, s, to_dev_bf16(xb), K, fmt, out=out)
    torch.cuda.synchronize()
    check()
    T, S = orc.quantize(W, rows)
    ref = orc.gemv(T, S, synth.bf16_bits_to_f32(xb))
    got = out.cpu().numpy()
    if rows is not None:
        got = got[:, rows]
    return check_y(got, ref)


def test_gemv_tiny_config(orc):
    W, xb = synth.tiny_config()
    c2, _, s = tq.quantize_pack(to_dev_f32(W), tq.TQ_PACK_2BIT)
    y = tq.gemv(c2, s, to_dev_bf16(xb), 256)
    T, S = orc.quantize(W)
    check_y(y.cpu().numpy(), orc.gemv(T, S, synth.bf16_bits_to_f32(xb)))


@pytest.mark.parametrize("N,K,M", [
    (256, 256, 1), (37, 384, 3), (15, 128, 1), (1, 128, 16), (300, 1280, 2),
    (1000, 1280, 4), (513, 2560, 8), (200, 640, 16), (64, 27648 // 4, 5),
])
def test_gemv_shapes(orc, N, K, M):
    _gemv_case(orc, N, K, M, seed=N * 31 + K + M)


@pytest.mark.parametrize("N,K", [(5120, 5120), (27648, 5120), (5120, 27648)])
@pytest.mark.parametrize("M", [1, 16])
def test_gemv_full_size_sampled(orc, N, K, M):
    """The benchmark's shapes and launch configuration; the oracle checks a
    seeded sample of 48 output rows (it cannot do all of them quickly)."""
    rows = np.sort(np.random.default_rng(N + K + M).choice(N, size=48, replace=False))
    rows[-1] = N - 1
    _gemv_case(orc, N, K, M, seed=N + K + M, rows=rows)


@pytest.mark.parametrize("N,K,M", [
    (256, 256, 1), (37, 384, 3), (15, 128, 1), (100, 640, 16), (300, 1280, 2), (513, 2560, 8),
    (64, 27648 // 4, 5), (20, 27648, 1),
])
def test_gemv_base3_shapes(orc, N, K, M):
    """Base-3 codes (five trits per byte; a lane's 32 trits start anywhere in
    a byte and the last byte of a row is padded)."""
    _gemv_case(orc, N, K, M, seed=N * 17 + K + M, fmt=tq.TQ_PACK_BASE3)


@pytest.mark.parametrize("N,K", [(27648, 5120), (5120, 27648)])
@pytest.mark.parametrize("M", [1, 16])
def test_gemv_base3_full_size_sampled(orc, N, K, M):
    rows = np.sort(np.random.default_rng(N + K + M + 3).choice(N, size=32, replace=False))
    rows[-1] = N - 1
    _gemv_case(orc, N, K, M, seed=N + K + M + 3, fmt=tq.TQ_PACK_BASE3, rows=rows)


@pytest.mark.parametrize("N,K", [(19457, 2560), (20000, 2944), (4999, 27648), (19500, 4480)])
def test_gemv_tc_shapes(orc, N, K):
    """M = 1 GEMVs of more than about ten megabytes take the tensor-memory
    kernel: ragged last tiles (down to one row), group counts that leave
    padded four-group stages and odd K slices, few tiles with a deep K
    split, sampled rows including the tail."""
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([rng.choice(N, size=40, replace=False), np.arange(N - 130, N)]))
    _gemv_case(orc, N, K, 1, seed=N * 7 + K, rows=rows)


@pytest.mark.parametrize("N,K,M", [
    (27648, 5120, 2), (19457, 2560, 3), (20000, 2944, 5), (27648, 5120, 6), (4999, 27648, 8),
    (19500, 4480, 11), (5120, 27648, 13), (2049, 1152, 16),
])
def test_gemv_tc_skinny(orc, N, K, M):
    """Skinny M on the tensor-memory kernel: each B layout (M <= 2, 5, 8, 16
    rows of x: one, one, two and three MMA passes), ragged tiles and K
    slices, and a shape whose B for all M rows does not fit one CTA's share
    of shared memory (two launches of half the rows each)."""
    assert tq.gemv_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY
    rng = np.random.default_rng(N + K + M)
    rows = np.unique(np.concatenate([rng.choice(N, size=24, replace=False), np.arange(N - 130, N)]))
    _gemv_case(orc, N, K, M, seed=N * 5 + K + M, rows=rows)


# One shape per K split the planner can choose (1, 2, 3, 4, 6, 7, 8 CTAs per
# cluster at M = 3): 5120x128 has one group, 3000x2048 and 123x896 ragged
# tiles.
CLUSTER_SHAPES = [(5120, 128), (27648, 5120), (5120, 1536), (3000, 2048), (2048, 3072), (123, 896), (1024, 27648)]


def test_gemv_tc_plans_every_cluster_size():
    """At M = 3 the shapes of the next test reach every cluster size the
    planner has (the plan is queried through tq_gemv_plan, not assumed)."""
    sizes = [tq.gemv_plan(N, K, 3)[0] for N, K in CLUSTER_SHAPES]
    assert sizes == [1, 2, 3, 4, 6, 7, 8], sizes


@pytest.mark.parametrize("N,K", CLUSTER_SHAPES)
@pytest.mark.parametrize("M", [1, 3])
def test_gemv_tc_cluster_sizes(orc, N, K, M):
    """Each K split, including clusters of 3, 6 and 7 whose ranks own
    ceil(128 / kcl) rows of a tile (the last rank the rest) and floor-divided
    K slices: sampled rows and the tail against the oracle, and 20 repeats
    bit-identical to the first."""
    kcl, clusters, launches = tq.gemv_plan(N, K, M)
    assert 1 <= kcl <= 8 and clusters >= 1 and launches == 1
    rng = np.random.default_rng(N + K + M + 5)
    rows = np.unique(np.concatenate([rng.choice(N, size=min(N, 40), replace=False), np.arange(max(0, N - 130), N)]))
    _gemv_case(orc, N, K, M, seed=N * 11 + K + M, rows=rows)
    W = synth.weights(N, K, 91, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K, 92))
    outs = [tq.gemv(c2, s, x, K, weights_ready=True) for _ in range(20)]
    torch.cuda.synchronize()
    tq.device_fault()
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


@pytest.mark.parametrize("fmt", [tq.TQ_PACK_2BIT, tq.TQ_PACK_BASE3], ids=["2bit", "base3"])
def test_gemv_tc_cluster_of_16(orc, fmt):
    """5120x27648 at M = 16: no cluster of at most 8 CTAs fits the
    activations of all rows in shared memory, so the 2-bit plan is one launch
    on clusters of 16 (a non-portable size; 8 rows a rank); both formats
    against the oracle on sampled rows and the tail, and 10 repeats
    bit-identical to the first."""
    N, K, M = 5120, 27648, 16
    kcl, _, launches = tq.gemv_plan(N, K, M, fmt)
    if fmt == tq.TQ_PACK_2BIT:
        assert (kcl, launches) == (16, 1)
    rng = np.random.default_rng(97)
    rows = np.unique(np.concatenate([rng.choice(N, size=32, replace=False), np.arange(N - 130, N)]))
    _gemv_case(orc, N, K, M, seed=98, fmt=fmt, rows=rows)
    W = synth.weights(N, K, 99, dtype="bf16")
    c2, c3, s = tq.quantize_pack(to_dev_bf16(W), fmt)
    codes = c2 if fmt == tq.TQ_PACK_2BIT else c3
    x = to_dev_bf16(synth.activations(M, K, 100))
    outs = [tq.gemv(codes, s, x, K, fmt, weights_ready=True) for _ in range(10)]
    torch.cuda.synchronize()
    tq.device_fault()
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


@pytest.mark.parametrize("N,K", [(5120, 5120), (5120, 1536), (2560, 2560), (2048, 3072)])
def test_gemv_rotate_next_cluster_sizes(orc, N, K):
    """The chained form (rank 0 adds the partial sums of all 128 rows of
    its tiles) on shapes whose plan is not a power-of-two cluster: y against
    the oracle, x'_next bit for bit the staged transform of y."""
    kcl, _, _ = tq.gemv_plan(N, K, 1, chained=True)
    assert kcl in (3, 6, 7)
    W = synth.weights(N, K, 93, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    xb = synth.activations(1, K, 94)
    y, xn = tq.gemv_rotate_next(c2, s, to_dev_bf16(xb), K)
    torch.cuda.synchronize()
    tq.device_fault()
    yn = y.cpu().numpy()
    assert np.array_equal(xn.cpu().numpy().view(np.uint32), _staged_fwht128(yn).view(np.uint32))
    rows = np.arange(0, N, max(1, N // 64))
    T, S = orc.quantize(W, rows)
    check_y(yn[:, rows], orc.gemv(T, S, synth.bf16_bits_to_f32(xb)), f"chained y (clusters of {kcl})")


@pytest.mark.parametrize("N,K,M", [
    (27648, 5120, 1), (19457, 2560, 3), (20000, 2944, 5), (27648, 5120, 6), (4999, 27648, 8),
    (19500, 4480, 11), (5120, 27648, 13), (2049, 1152, 16), (300, 640, 1), (129, 768, 2), (1000, 27648, 16),
])
def test_gemv_tc_base3(orc, N, K, M):
    """Base-3 codes on the tensor-memory kernel: five-group stages whose K
    slices start on a code byte, group windows that share code bytes with
    their neighbours, a last stage of fewer than five groups (K = 768:
    six groups; K = 2944: 23; K = 27648: 216) reading the row's zero
    padding, every B layout, ragged tiles, and rows of x split over two to
    four launches (5120x27648 at M = 8, 13, 16)."""
    assert tq.gemv_path(N, K, M, tq.TQ_PACK_BASE3) == tq.TQ_GEMV_TENSOR_MEMORY
    rng = np.random.default_rng(N + K + M + 1)
    rows = np.unique(np.concatenate([rng.choice(N, size=min(N, 24), replace=False),
                                     np.arange(max(0, N - 130), N)]))
    _gemv_case(orc, N, K, M, seed=N * 3 + K + M, fmt=tq.TQ_PACK_BASE3, rows=rows)


def test_gemv_mma_sync_fallback_base3(orc):
    """Base-3 codes whose K slice of B does not fit shared memory even for
    a quarter of the rows of x take the mma.sync kernel."""
    N, K, M = 96, 262144, 16
    assert tq.gemv_path(N, K, M, tq.TQ_PACK_BASE3) == tq.TQ_GEMV_MMA_SYNC
    _gemv_case(orc, N, K, M, seed=78, fmt=tq.TQ_PACK_BASE3)


@pytest.mark.parametrize("N,K,M,fmt", [
    (27648, 5120, 1, tq.TQ_PACK_2BIT), (5120, 27648, 1, tq.TQ_PACK_2BIT), (5120, 5120, 4, tq.TQ_PACK_2BIT),
    (27648, 5120, 16, tq.TQ_PACK_2BIT), (27648, 5120, 1, tq.TQ_PACK_BASE3), (5120, 27648, 1, tq.TQ_PACK_BASE3),
    (5120, 27648, 16, tq.TQ_PACK_BASE3),
])
def test_gemv_tc_repeatable(N, K, M, fmt):
    """The tensor-memory kernel sums in a fixed order and its barriers admit
    one schedule of results: 200 back-to-back launches (each streaming its
    weights while the previous one finishes) give the same bits as the
    first, and no bounded wait ran out."""
    W = synth.weights(N, K, 41, dtype="bf16")
    c2, c3, s = tq.quantize_pack(to_dev_bf16(W), fmt)
    codes = c2 if fmt == tq.TQ_PACK_2BIT else c3
    x = to_dev_bf16(synth.activations(M, K, 42))
    outs = [torch.empty(M, N, device="cuda") for _ in range(200)]
    torch.cuda.synchronize()
    for y in outs:
        tq.gemv(codes, s, x, K, fmt, out=y, weights_ready=True)
    tq.device_fault()
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


@pytest.mark.parametrize("N,K,M", [(5120, 27648, 1), (27648, 5120, 2), (2049, 1152, 16)])
def test_gemv_tc_reads_no_stale_shared_memory(N, K, M):
    """Between launches a cuBLAS matmul of changing random operands leaves
    different data in every SM's shared memory; a kernel that read any of it
    before writing it would not reproduce its first result."""
    W = synth.weights(N, K, 51, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K, 52))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(53)
    scrib = [torch.randn(2048, 2048, device="cuda", generator=gen, dtype=torch.bfloat16) for _ in range(4)]
    outs = [torch.empty(M, N, device="cuda") for _ in range(40)]
    torch.cuda.synchronize()
    for i, y in enumerate(outs):
        _ = scrib[i % 4] @ scrib[(i + 1) % 4]
        tq.gemv(c2, s, x, K, out=y)
    tq.device_fault()
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


def test_gemv_mma_sync_fallback_2bit(orc):
    """2-bit codes whose K slice of B does not fit shared memory even for a
    quarter of the rows of x take the mma.sync kernel."""
    N, K, M = 96, 262144, 16
    assert tq.gemv_path(N, K, M) == tq.TQ_GEMV_MMA_SYNC
    _gemv_case(orc, N, K, M, seed=77)


def test_gemv_path_of_benchmark_shapes():
    """Both code formats take the tensor-memory kernel for every M of the
    benchmark."""
    for N, K in [(27648, 5120), (5120, 27648), (5120, 5120), (1, 128)]:
        for M in (1, 2, 4, 8, 16):
            assert tq.gemv_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY
            assert tq.gemv_path(N, K, M, tq.TQ_PACK_BASE3) == tq.TQ_GEMV_TENSOR_MEMORY


@pytest.mark.parametrize("N,K,M", [(27648, 5120, 1), (512, 1280, 1), (512, 1280, 4), (5120, 27648, 16)])
def test_gemv_weights_ready_matches(orc, N, K, M):
    """TQ_GEMV_WEIGHTS_READY only moves when codes are first read.  The
    tensor-memory kernel sums in a fixed order, so its result is
    bit-identical to the plain call; the mma.sync kernel adds partial tiles
    with shared-memory atomics (order varies), so both calls are checked
    against the oracle instead."""
    W = synth.weights(N, K, 21, dtype="bf16")
    xb = synth.activations(M, K, 22)
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(xb)
    torch.cuda.synchronize()
    y0 = tq.gemv(c2, s, x, K)
    y1 = tq.gemv(c2, s, x, K, weights_ready=True)
    if tq.gemv_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY:
        assert torch.equal(y0, y1)
    else:
        rows = np.arange(0, N, max(1, N // 64))
        T, S = orc.quantize(W, rows)
        ref = orc.gemv(T, S, synth.bf16_bits_to_f32(xb))
        check_y(y0.cpu().numpy()[:, rows], ref)
        check_y(y1.cpu().numpy()[:, rows], ref)


def test_gemv_weights_ready_chain(orc):
    """Back-to-back GEMVs whose x is the previous GEMV's output (converted to
    bf16 in between): with the flag, each kernel streams its fixed weights
    while the one before it finishes, and still reads x only afterwards."""
    K = 5120
    W1 = synth.weights(27648, K, 31, dtype="bf16")
    W2 = synth.weights(K, 27648, 32, dtype="bf16")
    c1, _, s1 = tq.quantize_pack(to_dev_bf16(W1), tq.TQ_PACK_2BIT)
    c2, _, s2 = tq.quantize_pack(to_dev_bf16(W2), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(1, K, 33))
    torch.cuda.synchronize()
    assert tq.gemv_path(27648, K) == tq.gemv_path(K, 27648) == tq.TQ_GEMV_TENSOR_MEMORY
    outs = []
    for flag in (False, True):
        h = tq.gemv(c1, s1, x, K, weights_ready=flag)
        h16 = (h * 0.05).to(torch.bfloat16)
        outs.append(tq.gemv(c2, s2, h16, 27648, weights_ready=flag))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_gemv_tc_zero_and_delta_activations(orc):
    N, K = 19456, 2560
    W = synth.weights(N, K, 11, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = np.zeros((1, K), dtype=np.uint16)
    y0 = tq.gemv(c2, s, to_dev_bf16(x), K).cpu().numpy()
    assert np.all(y0 == 0.0)
    x[0, 300] = synth.f32_to_bf16_bits(np.array([-2.5], dtype=np.float32))[0]
    y1 = tq.gemv(c2, s, to_dev_bf16(x), K).cpu().numpy()
    rows = np.arange(0, N, 97)
    T, S = orc.quantize(W, rows)
    check_y(y1[:, rows], orc.gemv(T, S, synth.bf16_bits_to_f32(x)))


def test_gemv_zero_and_delta_activations(orc):
    N, K = 96, 512
    W = synth.weights(N, K, 9, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = np.zeros((2, K), dtype=np.uint16)
    x[1, 77] = synth.f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    y = tq.gemv(c2, s, to_dev_bf16(x), K).cpu().numpy()
    assert np.all(y[0] == 0.0)
    T, S = orc.quantize(W)
    check_y(y[1:], orc.gemv(T, S, synth.bf16_bits_to_f32(x[1:])))


# ----------------------------------------------------------- prefill GEMM

def _gemm_case(orc, N, K, M, seed, rows=None, out_cols=None):
    W = synth.weights(N, K, seed, dtype="bf16")
    xb = synth.activations(M, K, seed + 1)
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    out, check = guarded((M, N), torch.float32)
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    tq.gemm(c2, s, to_dev_bf16(xb), K, tq.TQ_PACK_2BIT, workspace=ws, out=out)
    torch.cuda.synchronize()
    check()
    tq.gemm_check_range(ws)
    T, S = orc.quantize(W, rows)
    xs = synth.bf16_bits_to_f32(xb)
    if out_cols is not None:
        xs = xs[out_cols]
    ref = orc.gemv(T, S, xs)
    got = out.cpu().numpy()
    if out_cols is not None:
        got = got[out_cols]
    if rows is not None:
        got = got[:, rows]
    return check_y(got, ref, "gemm y")


@pytest.mark.parametrize("N,K,M", [(256, 128, 256), (256, 256, 256), (300, 384, 300), (513, 640, 77),
                                   (1024, 1280, 512), (64, 128, 1)])
def test_gemm_shapes(orc, N, K, M):
    _gemm_case(orc, N, K, M, seed=N + 3 * K + 7 * M)


@pytest.mark.parametrize("N,K", [(5120, 5120), (27648, 5120), (5120, 27648)])
def test_gemm_full_size_sampled(orc, N, K):
    """M = 2048 tokens at the benchmark's shapes; the oracle checks a seeded
    sample of output rows (weights) and tokens."""
    rng = np.random.default_rng(N + K)
    rows = np.sort(rng.choice(N, size=24, replace=False))
    rows[-1] = N - 1
    toks = np.sort(rng.choice(2048, size=12, replace=False))
    toks[-1] = 2047
    _gemm_case(orc, N, K, 2048, seed=N * 7 + K, rows=rows, out_cols=toks)


def test_gemm_row_pitch_and_ragged_edges(orc):
    """y with a row pitch wider than N (the output blocks leave by TMA store):
    the last weight tile and the last token block are ragged (N = 300 and
    M = 300 against 64-column and 256-token tiles), and the pitch's padding
    columns keep their poison bytes."""
    N, K, M, pad = 300, 384, 300, 12
    W = synth.weights(N, K, 71, dtype="bf16")
    xb = synth.activations(M, K, 72)
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    raw = torch.empty((M, N + pad), dtype=torch.float32, device="cuda")
    raw.view(torch.uint8).fill_(0x5A)
    out = raw[:, :N]
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    tq.gemm(c2, s, to_dev_bf16(xb), K, tq.TQ_PACK_2BIT, workspace=ws, out=out)
    torch.cuda.synchronize()
    tail = raw[:, N:].contiguous().view(torch.uint8).cpu().numpy()
    assert np.all(tail == 0x5A), "write into the row pitch's padding"
    T, S = orc.quantize(W)
    check_y(out.cpu().numpy(), orc.gemv(T, S, synth.bf16_bits_to_f32(xb)), "gemm y (row pitch)")


def test_gemm_tile_width_not_multiple_of_32(orc):
    """N = 152 x 208 weight rows at M = 256 fill 152 SMs with 208-row tiles:
    the last 16 columns of every tile's output leave by plain stores, the
    rest by TMA store.  Rows from both parts of every few tiles are checked."""
    N, K, M = 152 * 208, 256, 256
    rng = np.random.default_rng(83)
    tiles = rng.choice(152, size=6, replace=False)
    rows = np.sort(np.concatenate([t * 208 + np.array([0, 31, 191, 192, 200, 207]) for t in tiles]))
    _gemm_case(orc, N, K, M, seed=81, rows=rows)


def test_gemm_split_last_wave(orc):
    """5120 weight rows in 256-row tiles x 8 token blocks make 160 tiles on
    152 SMs; the last 8 (weight rows 4864..5119, every token) are computed
    as K segments (at K = 2048: 11 segments of 2 or 3 stages on 152 SMs)
    whose partial sums a second kernel adds in a fixed order.  Every output
    of those tiles is checked, plus rows of whole tiles, and a second call
    gives the same bits."""
    N, K, M = 5120, 2048, 2048
    W = synth.weights(N, K, 61, dtype="bf16")
    xb = synth.activations(M, K, 62)
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(xb)
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y0 = tq.gemm(c2, s, x, K, tq.TQ_PACK_2BIT, workspace=ws)
    y1 = tq.gemm(c2, s, x, K, tq.TQ_PACK_2BIT, workspace=ws)
    torch.cuda.synchronize()
    tq.gemm_check_range(ws)
    assert torch.equal(y0, y1)
    rows = np.concatenate([np.arange(4864, 5120), np.array([0, 255, 256, 2500, 4863])])
    T, S = orc.quantize(W, rows)
    ref = orc.gemv(T, S, synth.bf16_bits_to_f32(xb))
    check_y(y0.cpu().numpy()[:, rows], ref, "gemm y (split tiles)")


def test_gemm_reuse_rotated(orc):
    """Two projections of the same x (gate and up of a feed-forward block):
    the second call reuses the rotated x' in the workspace and skips the
    pre-pass.  Its output is bit-identical to a plain call (the GEMM is
    deterministic), and matches the oracle."""
    N, K, M = 768, 640, 300
    W1 = synth.weights(N, K, 101, dtype="bf16")
    W2 = synth.weights(N, K, 102, dtype="bf16")
    xb = synth.activations(M, K, 103)
    c1, _, s1 = tq.quantize_pack(to_dev_bf16(W1), tq.TQ_PACK_2BIT)
    c2, _, s2 = tq.quantize_pack(to_dev_bf16(W2), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(xb)
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    ref2 = tq.gemm(c2, s2, x, K, workspace=torch.empty_like(ws))
    tq.gemm(c1, s1, x, K, workspace=ws)
    junk = torch.zeros_like(x)  # not read when the rotation is reused
    y2 = tq.gemm(c2, s2, junk, K, workspace=ws, reuse_rotated=True)
    torch.cuda.synchronize()
    tq.gemm_check_range(ws)
    assert torch.equal(y2, ref2)
    T, S = orc.quantize(W2)
    check_y(y2.cpu().numpy(), orc.gemv(T, S, synth.bf16_bits_to_f32(xb)), "gemm y (reused x')")


def test_gemm_range_flag():
    """An activation block whose rotation exceeds the fp16 range is reported
    through the status word (tq_gemm_check_range -> TQ_ERR_RANGE)."""
    N, K, M = 256, 256, 256
    W = synth.weights(N, K, 1, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = torch.zeros(M, K, device="cuda", dtype=torch.bfloat16)
    x[3, :128] = 30000.0  # ||block||_2 = 30000 * sqrt(128) -> x'[0] far above 65504
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    tq.gemm(c2, s, x, K, workspace=ws)
    with pytest.raises(tq.TQError) as ei:
        tq.gemm_check_range(ws)
    assert ei.value.status == tq.TQ_ERR_RANGE
    x[3].zero_()
    tq.gemm(c2, s, x, K, workspace=ws)
    tq.gemm_check_range(ws)  # cleared on the next call


# ------------------------------------------- the rotation fused into the producer

def _unpermute16(xp: np.ndarray) -> np.ndarray:
    """Inverse of the GEMM k order inside each 16-chunk (slots 0, 8, 1, 9, ...)."""
    M, K = xp.shape
    v = xp.reshape(M, K // 16, 8, 2)
    return np.concatenate([v[:, :, :, 0], v[:, :, :, 1]], axis=2).reshape(M, K)


def _staged_fwht128(y: np.ndarray) -> np.ndarray:
    """FWHT-128 of each 128-block of the rows of fp32 y, stages h = 1 .. 64
    in order (the lower index keeps a + b), then times fp32(1/sqrt(128)),
    all in fp32 with round to nearest -- used to check that a kernel's fused
    transform of its own output is that output's transform (a property of
    two GPU results; the parity references below come from the oracle)."""
    v = np.ascontiguousarray(y, dtype=np.float32).reshape(y.shape[0], -1, 128).copy()
    h = 1
    while h < 128:
        w = v.reshape(v.shape[0], v.shape[1], 128 // (2 * h), 2, h)
        a, b = w[:, :, :, 0, :].copy(), w[:, :, :, 1, :].copy()
        w[:, :, :, 0, :] = a + b
        w[:, :, :, 1, :] = a - b
        h *= 2
    c = np.float32(1.0) / np.sqrt(np.float32(128.0), dtype=np.float32)
    return (v * np.float32(c)).reshape(y.shape).astype(np.float32)


@pytest.mark.parametrize("N1,K1,N2,M", [(1280, 640, 512, 300), (5120, 5120, 1024, 2048), (384, 256, 256, 257),
                                         (5376, 5120, 512, 2000)])
def test_gemm_rotate_next_chain(orc, N1, K1, N2, M):
    """The first GEMM writes FWHT-128 of its output as the second's fp16 x':
    bit for bit the rounded staged fp32 transform of y1, and both outputs
    match the oracle's chain (y1 = oracle GEMM of x, y2 = oracle GEMM of that
    y1) on sampled tokens.  At M = 2048 (and 2000) the 5120- and 5376-row
    outputs have more tiles than SMs: the last wave is split along K and its
    x' comes from the finished y (the 5376 case spans two column blocks and a
    short last row tile)."""
    W1 = synth.weights(N1, K1, 61, dtype="bf16")
    W2 = synth.weights(N2, N1, 62, dtype="bf16")
    c1, _, s1 = tq.quantize_pack(to_dev_bf16(W1), tq.TQ_PACK_2BIT)
    c2, _, s2 = tq.quantize_pack(to_dev_bf16(W2), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K1, 63))
    ws2 = torch.empty(tq.gemm_workspace_bytes(M, N1), dtype=torch.uint8, device="cuda")
    y1 = tq.gemm_rotate_next(c1, s1, x, K1, ws2)
    torch.cuda.synchronize()
    tq.gemm_check_range(ws2)
    y1n = y1.cpu().numpy()
    xr = ws2[256:256 + 2 * M * N1].view(torch.float16).view(M, N1).cpu().numpy()
    assert np.array_equal(_unpermute16(xr).view(np.uint16), _staged_fwht128(y1n).astype(np.float16).view(np.uint16))
    y2 = tq.gemm(c2, s2, torch.zeros(M, N1, dtype=torch.bfloat16, device="cuda"), N1, workspace=ws2,
                 reuse_rotated=True)
    torch.cuda.synchronize()
    mrows = np.arange(0, M, max(1, M // 48))
    T1, S1 = orc.quantize(W1)
    y1_ref = orc.gemv(T1, S1, synth.bf16_bits_to_f32(synth.activations(M, K1, 63))[mrows])
    check_y(y1n[mrows], y1_ref, "y1")
    rows = np.arange(0, N2, max(1, N2 // 64))
    T2, S2 = orc.quantize(W2, rows)
    check_y(y2.cpu().numpy()[np.ix_(mrows, rows)], orc.gemv(T2, S2, y1_ref), "chained y2")


def test_gemm_rotate_next_reports_overflow():
    """An output whose rotation overflows fp16 is reported on the next workspace."""
    N1, K1, M = 256, 256, 128
    # weights ~N(0, 2000): fp16 scales near 1600, outputs of a few 10^4 whose
    # rotation exceeds 65504; the activations' own rotation stays in range
    W1 = synth.weights(N1, K1, 64, dtype="f32", std=2000.0)
    c1, _, s1 = tq.quantize_pack(to_dev_f32(W1), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K1, 65))
    ws2 = torch.empty(tq.gemm_workspace_bytes(M, N1), dtype=torch.uint8, device="cuda")
    ws1 = torch.empty(tq.gemm_workspace_bytes(M, K1), dtype=torch.uint8, device="cuda")
    y1 = tq.gemm_rotate_next(c1, s1, x, K1, ws2, workspace=ws1)
    tq.gemm_check_range(ws1)
    assert torch.isfinite(y1).all()
    with pytest.raises(tq.TQError) as e:
        tq.gemm_check_range(ws2)
    assert e.value.status == tq.TQ_ERR_RANGE


@pytest.mark.parametrize("fmt", [tq.TQ_PACK_2BIT, tq.TQ_PACK_BASE3], ids=["2bit", "base3"])
@pytest.mark.parametrize("N1,K1,N2,M", [(5120, 5120, 1024, 1), (27648, 5120, 640, 1), (5120, 27648, 2048, 2),
                                         (1280, 640, 384, 4), (640, 1280, 256, 16)])
def test_gemv_rotate_next_chain(orc, fmt, N1, K1, N2, M):
    """Decode chain: the first GEMV writes FWHT-128 of its fp32 output as the
    next x' (bit for bit the staged fp32 transform of y1), the second GEMV
    reads it (TQ_GEMV_X_ROTATED), and both outputs match the oracle's chain
    (y1 = oracle GEMV of x, y2 = oracle GEMV of that y1).  The shapes reach
    every K split (5120x27648 uses clusters of 8, where rank 0 then adds all
    128 rows of each tile)."""
    W1 = synth.weights(N1, K1, 71, dtype="bf16")
    W2 = synth.weights(N2, N1, 72, dtype="bf16")
    c1a, c1b, s1 = tq.quantize_pack(to_dev_bf16(W1), fmt)
    c2a, c2b, s2 = tq.quantize_pack(to_dev_bf16(W2), fmt)
    c1 = c1a if fmt == tq.TQ_PACK_2BIT else c1b
    c2 = c2a if fmt == tq.TQ_PACK_2BIT else c2b
    xb = synth.activations(M, K1, 73)
    y1, xn = tq.gemv_rotate_next(c1, s1, to_dev_bf16(xb), K1, fmt)
    y2 = tq.gemv(c2, s2, xn, N1, fmt, x_rotated=True)
    torch.cuda.synchronize()
    tq.device_fault()
    y1n = y1.cpu().numpy()
    assert np.array_equal(xn.cpu().numpy().view(np.uint32), _staged_fwht128(y1n).view(np.uint32))
    T1, S1 = orc.quantize(W1)
    y1_ref = orc.gemv(T1, S1, synth.bf16_bits_to_f32(xb))
    check_y(y1n, y1_ref, "y1")
    rows = np.arange(0, N2, max(1, N2 // 48))
    T2, S2 = orc.quantize(W2, rows)
    check_y(y2.cpu().numpy()[:, rows], orc.gemv(T2, S2, y1_ref), "chained y2")


def test_gemv_rotate_next_repeatable():
    N1, K1, M = 5120, 27648, 1
    W1 = synth.weights(N1, K1, 74, dtype="bf16")
    c1, _, s1 = tq.quantize_pack(to_dev_bf16(W1), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K1, 75))
    outs = [tq.gemv_rotate_next(c1, s1, x, K1) for _ in range(30)]
    torch.cuda.synchronize()
    for y, xn in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(xn, outs[0][1])
