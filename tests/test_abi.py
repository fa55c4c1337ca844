"""The C ABI on the host: the library loads without a GPU, exports every
symbol include/tq.h declares, and rejects bad arguments before any launch.

Every call below fails host-side validation (or is an empty no-op), so the
fake device pointers are never dereferenced and no CUDA work is issued."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

import ternary_weight_fwht128_gb300 as tq
from ternary_weight_fwht128_gb300 import build as tqbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tq.h")
A = 0x10000   # 16-byte aligned fake device address (never dereferenced)
B = 0x20000
MIS = 0x10008  # 8-byte aligned only


@pytest.fixture(scope="module")
def L():
    tqbuild.build()
    return tq.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TQ_API[^;(]*?\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert len(syms) >= 9
    for s in syms:
        assert hasattr(L, s), f"{s} not exported"
    assert sorted(tq.EXPORTED) == syms


def test_status_strings_and_version(L):
    names = ["TQ_OK", "TQ_ERR_INVALID_ARG", "TQ_ERR_SHAPE", "TQ_ERR_ALIGN", "TQ_ERR_UNSUPPORTED", "TQ_ERR_CUDA",
             "TQ_ERR_RANGE", "TQ_ERR_TIMEOUT"]
    for st, name in enumerate(names):
        assert tq.status_string(st).startswith(name)
    assert tq.status_string(99) == "unknown tq_status"
    assert L.tq_version() == 100


def test_packed_ld(L):
    assert tq.packed_ld(5120, tq.TQ_PACK_2BIT) == 1280
    assert tq.packed_ld(5120, tq.TQ_PACK_BASE3) == 1024
    assert tq.packed_ld(27648, tq.TQ_PACK_BASE3) == 5536   # ceil(27648/5) = 5530 -> 5536
    assert tq.packed_ld(128, tq.TQ_PACK_BASE3) == 32       # 26 -> 32
    assert tq.packed_ld(0, tq.TQ_PACK_2BIT) == -1
    assert tq.packed_ld(128, 7) == -1


def test_gemm_workspace_bytes(L):
    # status word + fp16 rotated activations (rounded to 256 B) + 40 MiB of split partial tiles
    assert tq.gemm_workspace_bytes(2048, 5120) == 256 + 2048 * 5120 * 2 + 160 * 256 * 256 * 4
    assert tq.gemm_workspace_bytes(3, 128) == 1024 + 160 * 256 * 256 * 4
    assert tq.gemm_workspace_bytes(-1, 5) == 0


def test_fwht_validation(L):
    f = L.tq_fwht128
    assert f(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 0, 256, None) == tq.TQ_OK          # empty
    assert f(A, 7, 256, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_INVALID_ARG
    assert f(A, tq.TQ_F16, 256, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_INVALID_ARG
    assert f(A, tq.TQ_F32, 256, B, 9, 256, 4, 256, None) == tq.TQ_ERR_INVALID_ARG
    assert f(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, -1, 256, None) == tq.TQ_ERR_INVALID_ARG
    assert f(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 4, 200, None) == tq.TQ_ERR_SHAPE
    assert f(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 4, 0, None) == tq.TQ_ERR_SHAPE
    assert f(None, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_INVALID_ARG
    assert f(A, tq.TQ_F32, 128, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_SHAPE
    assert f(MIS, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_ALIGN
    assert f(A, tq.TQ_F32, 258, B, tq.TQ_F32, 256, 4, 256, None) == tq.TQ_ERR_ALIGN   # row stride not 16 B
    assert f(A, tq.TQ_F32, 256, A, tq.TQ_F16, 256, 4, 256, None) == tq.TQ_ERR_INVALID_ARG  # in place, dtypes differ


def test_quantize_validation(L):
    f = L.tq_quantize_pack
    ok = dict(W=A, wt=tq.TQ_BF16, N=4, K=256, ldw=256, fmt=tq.TQ_PACK_BOTH, c2=B, ld2=64, c3=B + 4096, ld3=64,
              s=B + 8192, lds=2)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["W"], a["wt"], a["N"], a["K"], a["ldw"], a["fmt"], a["c2"], a["ld2"], a["c3"], a["ld3"], a["s"],
                 a["lds"], None)

    assert call(N=0) == tq.TQ_OK
    assert call(wt=tq.TQ_F16) == tq.TQ_ERR_INVALID_ARG
    assert call(fmt=0) == tq.TQ_ERR_INVALID_ARG
    assert call(N=-2) == tq.TQ_ERR_INVALID_ARG
    assert call(K=100) == tq.TQ_ERR_SHAPE
    assert call(c2=None) == tq.TQ_ERR_INVALID_ARG
    assert call(c3=None) == tq.TQ_ERR_INVALID_ARG
    assert call(s=None) == tq.TQ_ERR_INVALID_ARG
    assert call(ld2=63) == tq.TQ_ERR_SHAPE
    assert call(ld3=52) == tq.TQ_ERR_SHAPE           # ceil(256/5) = 52, padded minimum is 64
    assert call(lds=1) == tq.TQ_ERR_SHAPE
    assert call(ldw=255) == tq.TQ_ERR_SHAPE
    assert call(W=MIS) == tq.TQ_ERR_ALIGN
    assert call(s=B + 8193) == tq.TQ_ERR_ALIGN
    # a format that does not write a layout does not need its pointer
    assert call(fmt=tq.TQ_PACK_2BIT, c3=None, N=0) == tq.TQ_OK


def test_gemv_ex_validation(L):
    f = L.tq_gemv_ex
    args = (A, 64, tq.TQ_PACK_2BIT, B, 2, 8, 256, B + 4096, 256, 1, B + 8192, 8)
    assert f(*args, 0x40, None) == tq.TQ_ERR_INVALID_ARG         # unknown flag bit
    assert f(*args[:5], 0, *args[6:], tq.TQ_GEMV_WEIGHTS_READY, None) == tq.TQ_OK   # N == 0
    assert f(*args[:9], 0, *args[10:], tq.TQ_GEMV_WEIGHTS_READY, None) == tq.TQ_ERR_SHAPE  # M == 0


def test_gemv_path_validation(L):
    f = L.tq_gemv_path
    assert f(8, 256, 1, 3) == -tq.TQ_ERR_INVALID_ARG
    assert f(-1, 256, 1, tq.TQ_PACK_2BIT) == -tq.TQ_ERR_INVALID_ARG
    assert f(8, 200, 1, tq.TQ_PACK_2BIT) == -tq.TQ_ERR_SHAPE
    assert f(8, 256, 0, tq.TQ_PACK_2BIT) == -tq.TQ_ERR_SHAPE
    assert f(8, 256, 17, tq.TQ_PACK_2BIT) == -tq.TQ_ERR_SHAPE
    # base-3 codes always take the mma.sync kernel (no device query needed)
    assert f(27648, 5120, 1, tq.TQ_PACK_BASE3) == tq.TQ_GEMV_MMA_SYNC
    assert f(5120, 27648, 16, tq.TQ_PACK_BASE3) == tq.TQ_GEMV_MMA_SYNC


def test_gemv_plan_validation(L):
    f = L.tq_gemv_plan
    v = (ctypes.c_int * 3)()
    a = ctypes.addressof(v)
    assert f(8, 256, 1, tq.TQ_PACK_2BIT, 0, None, a + 4, a + 8) == tq.TQ_ERR_INVALID_ARG
    assert f(8, 256, 1, tq.TQ_PACK_2BIT, 0, a, None, a + 8) == tq.TQ_ERR_INVALID_ARG
    assert f(8, 256, 1, tq.TQ_PACK_2BIT, 0, a, a + 4, None) == tq.TQ_ERR_INVALID_ARG
    assert f(8, 256, 1, 3, 0, a, a + 4, a + 8) == tq.TQ_ERR_INVALID_ARG
    assert f(8, 200, 1, tq.TQ_PACK_2BIT, 0, a, a + 4, a + 8) == tq.TQ_ERR_SHAPE
    assert f(8, 256, 17, tq.TQ_PACK_2BIT, 0, a, a + 4, a + 8) == tq.TQ_ERR_SHAPE
    # without a device every shape takes the other kernel (nothing to plan)
    if not torch.cuda.is_available():
        assert f(5120, 5120, 1, tq.TQ_PACK_2BIT, 0, a, a + 4, a + 8) == tq.TQ_ERR_UNSUPPORTED


def test_gemv_validation(L):
    f = L.tq_gemv
    ok = dict(c=A, ldc=64, fmt=tq.TQ_PACK_2BIT, s=B, lds=2, N=8, K=256, x=B + 4096, ldx=256, M=1, y=B + 8192, ldy=8)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                 a["ldy"], None)

    assert call(N=0) == tq.TQ_OK
    assert call(fmt=3) == tq.TQ_ERR_INVALID_ARG
    assert call(M=0) == tq.TQ_ERR_SHAPE
    assert call(M=17) == tq.TQ_ERR_SHAPE
    assert call(K=384 + 1) == tq.TQ_ERR_SHAPE
    assert call(ldc=48) == tq.TQ_ERR_SHAPE
    assert call(fmt=tq.TQ_PACK_BASE3, ldc=48) == tq.TQ_ERR_SHAPE   # base-3 needs 64 for K = 256
    assert call(ldy=7) == tq.TQ_ERR_SHAPE
    assert call(ldx=128) == tq.TQ_ERR_SHAPE
    assert call(x=None) == tq.TQ_ERR_INVALID_ARG
    assert call(c=MIS) == tq.TQ_ERR_ALIGN
    assert call(ldc=72) == tq.TQ_ERR_ALIGN
    assert call(x=MIS) == tq.TQ_ERR_ALIGN
    assert call(y=B + 8194) == tq.TQ_ERR_ALIGN


def test_gemm_validation(L):
    f = L.tq_gemm
    ws = tq.gemm_workspace_bytes(4, 256)
    ok = dict(c=A, ldc=64, fmt=tq.TQ_PACK_2BIT, s=B, lds=2, N=8, K=256, x=B + 4096, ldx=256, M=4, y=B + 8192, ldy=8,
              w=B + 65536, wsb=ws)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                 a["ldy"], a["w"], a["wsb"], None)

    assert call(M=0) == tq.TQ_OK
    assert call(N=0) == tq.TQ_OK
    assert call(fmt=tq.TQ_PACK_BASE3) == tq.TQ_ERR_UNSUPPORTED
    assert call(wsb=ws - 1) == tq.TQ_ERR_SHAPE
    assert call(w=None) == tq.TQ_ERR_INVALID_ARG
    assert call(w=B + 65544) == tq.TQ_ERR_ALIGN
    assert call(y=B + 8194) == tq.TQ_ERR_ALIGN
    assert call(K=0) == tq.TQ_ERR_SHAPE
    # tq_gemm_ex: the same validation, plus its flags
    fe = L.tq_gemm_ex

    def call_ex(flags, **kw):
        a = dict(ok, **kw)
        return fe(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                  a["ldy"], a["w"], a["wsb"], flags, None)

    assert call_ex(2, M=0) == tq.TQ_ERR_INVALID_ARG  # unknown flag bit, before anything else
    assert call_ex(tq.TQ_GEMM_REUSE_ROTATED, M=0) == tq.TQ_OK
    assert call_ex(tq.TQ_GEMM_REUSE_ROTATED, wsb=ws - 1) == tq.TQ_ERR_SHAPE
    assert call_ex(tq.TQ_GEMM_REUSE_ROTATED, w=B + 65544) == tq.TQ_ERR_ALIGN
    assert call_ex(0, fmt=tq.TQ_PACK_BASE3) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_gemm_check_range(None, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_gemm_check_range(MIS, None) == tq.TQ_ERR_ALIGN


def test_gemm_noalloc_validation(L):
    """tq_gemm_noalloc rejects bad arguments on the host, before it looks up
    its scratch array or launches anything (fake pointers, no GPU needed)."""
    f = L.tq_gemm_noalloc
    ok = dict(c=A, ldc=64, fmt=tq.TQ_PACK_2BIT, s=B, lds=2, N=8, K=256, x=B + 4096, ldx=256, M=4, y=B + 8192,
              ldy=8)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                 a["ldy"], None)

    assert call(M=0) == tq.TQ_OK
    assert call(N=0) == tq.TQ_OK
    assert call(fmt=7) == tq.TQ_ERR_INVALID_ARG
    assert call(fmt=tq.TQ_PACK_BOTH) == tq.TQ_ERR_INVALID_ARG
    assert call(fmt=tq.TQ_PACK_BASE3) == tq.TQ_ERR_UNSUPPORTED
    assert call(N=-1) == tq.TQ_ERR_INVALID_ARG
    assert call(M=-1) == tq.TQ_ERR_INVALID_ARG
    assert call(K=0) == tq.TQ_ERR_SHAPE
    assert call(K=200) == tq.TQ_ERR_SHAPE
    for name in ("c", "s", "x", "y"):
        assert call(**{name: None}) == tq.TQ_ERR_INVALID_ARG, name
    assert call(ldc=63) == tq.TQ_ERR_SHAPE
    assert call(lds=1) == tq.TQ_ERR_SHAPE
    assert call(ldx=255) == tq.TQ_ERR_SHAPE
    assert call(ldy=7) == tq.TQ_ERR_SHAPE
    assert call(c=A + 8) == tq.TQ_ERR_ALIGN
    assert call(ldc=72) == tq.TQ_ERR_ALIGN
    assert call(s=B + 1) == tq.TQ_ERR_ALIGN
    assert call(x=B + 4104) == tq.TQ_ERR_ALIGN
    assert call(ldx=260) == tq.TQ_ERR_ALIGN
    assert call(y=B + 8194) == tq.TQ_ERR_ALIGN
    # M * K above the fixed scratch array (2^24 rotated activations)
    assert call(M=2048, K=27648, ldx=27648, ldc=6912, lds=216) == tq.TQ_ERR_SHAPE
    assert call(M=(1 << 24) // 256 + 1) == tq.TQ_ERR_SHAPE


def test_layout_validation(L):
    """Layout entry points reject bad layouts and shapes on the host."""
    lay = tq.layout(256, 256, True)
    assert tq.layout_codes_ld(5120, tq.TQ_PACK_2BIT, lay) == 2560
    assert tq.layout_codes_ld(5120, tq.TQ_PACK_BASE3, lay) == 2048
    assert tq.layout_scales_ld(5120, lay) == 40
    assert tq.layout_scales_ld(5120, None) == 40
    assert tq.layout_codes_ld(5120 + 128, tq.TQ_PACK_2BIT, lay) == -1  # not a multiple of 256
    assert tq.layout_codes_ld(5120, tq.TQ_PACK_2BIT, tq.layout(96, 128, False)) == -1
    assert tq.gemm_workspace_bytes_layout(4, 256, lay) == tq.gemm_workspace_bytes(4, 512)
    ctypes = __import__("ctypes")
    bad = [tq.Layout(32, 128, 0), tq.Layout(128, 64, 0), tq.Layout(128, 128, 6)]
    for b in bad:
        assert L.tq_gemv_layout(A, 64, tq.TQ_PACK_2BIT, B, 2, 8, 256, B, 256, 1, B, 8, ctypes.byref(b), 0,
                                None) == tq.TQ_ERR_INVALID_ARG
        assert L.tq_quantize_pack_layout(A, tq.TQ_BF16, 8, 256, 256, tq.TQ_PACK_2BIT, B, 64, None, 0, B, 2,
                                         ctypes.byref(b), None) == tq.TQ_ERR_INVALID_ARG
    lp = ctypes.byref(lay)
    # K = 384 is not a multiple of 256
    assert L.tq_gemv_layout(A, 256, tq.TQ_PACK_2BIT, B, 8, 8, 384, B, 384, 1, B, 8, lp, 0, None) == tq.TQ_ERR_SHAPE
    # codes must hold both passes: ld >= 2K/4
    assert L.tq_gemv_layout(A, 64, tq.TQ_PACK_2BIT, B, 4, 8, 256, B, 256, 1, B, 8, lp, 0, None) == tq.TQ_ERR_SHAPE
    # scales must hold both passes: 2 x 256 / 256
    assert L.tq_gemv_layout(A, 128, tq.TQ_PACK_2BIT, B, 1, 8, 256, B, 256, 1, B, 8, lp, 0, None) == tq.TQ_ERR_SHAPE
    assert L.tq_gemv_layout(A, 128, tq.TQ_PACK_2BIT, B, 4, 0, 256, B, 256, 1, B, 8, lp, 0, None) == tq.TQ_OK
    assert L.tq_gemv_layout(A, 128, tq.TQ_PACK_2BIT, B, 4, 8, 256, B, 256, 17, B, 8, lp, 0, None) == tq.TQ_ERR_SHAPE
    assert L.tq_gemv_layout(A, 128, tq.TQ_PACK_2BIT, B, 4, 8, 256, MIS, 256, 1, B, 8, lp, 0, None) == tq.TQ_ERR_ALIGN
    assert L.tq_gemv_layout(A, 128, tq.TQ_PACK_2BIT, B, 4, 8, 256, B, 256, 1, B, 8, lp, 4, None) == \
        tq.TQ_ERR_INVALID_ARG
    assert L.tq_quantize_pack_layout(A, tq.TQ_BF16, 0, 256, 256, tq.TQ_PACK_2BIT, B, 128, None, 0, B, 4, lp,
                                     None) == tq.TQ_OK
    assert L.tq_quantize_pack_layout(A, tq.TQ_BF16, 8, 256, 256, tq.TQ_PACK_2BIT, B, 64, None, 0, B, 4, lp,
                                     None) == tq.TQ_ERR_SHAPE
    assert L.tq_quantize_pack_layout(A, tq.TQ_BF16, 8, 256, 256, tq.TQ_PACK_2BIT, B, 128, None, 0, B, 1, lp,
                                     None) == tq.TQ_ERR_SHAPE
    assert L.tq_quantize_pack_layout(A, tq.TQ_BF16, 8, 256, 256, tq.TQ_PACK_BASE3, None, 0, B, 96, B, 4, lp,
                                     None) == tq.TQ_ERR_SHAPE  # ld3 >= roundup16(ceil(512 / 5)) = 112
    ws = tq.gemm_workspace_bytes_layout(4, 256, lay)
    assert L.tq_gemm_layout(A, 128, tq.TQ_PACK_2BIT, B, 4, 8, 256, B, 256, 4, B, 8, B + 65536, ws - 1, lp, 0,
                            None) == tq.TQ_ERR_SHAPE
    assert L.tq_gemm_layout(A, 128, tq.TQ_PACK_BASE3, B, 4, 8, 256, B, 256, 4, B, 8, B + 65536, ws, lp, 0,
                            None) == tq.TQ_ERR_UNSUPPORTED
    assert L.tq_fwht(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 2, 256, 32, None) == tq.TQ_ERR_INVALID_ARG
    assert L.tq_fwht(A, tq.TQ_F32, 384, B, tq.TQ_F32, 384, 2, 384, 256, None) == tq.TQ_ERR_SHAPE
    assert L.tq_fwht(A, tq.TQ_F32, 256, B, tq.TQ_F32, 256, 0, 256, 64, None) == tq.TQ_OK


def test_gemm_rotate_next_validation(L):
    f = L.tq_gemm_rotate_next
    ws = tq.gemm_workspace_bytes(4, 256)
    wsn = tq.gemm_workspace_bytes(4, 128)
    W1, W2 = B + 65536, B + 65536 + (1 << 27)
    ok = dict(c=A, ldc=64, fmt=tq.TQ_PACK_2BIT, s=B, lds=2, N=128, K=256, x=B + 4096, ldx=256, M=4, y=B + 8192,
              ldy=128, w=W1, wsb=ws, fl=0, nw=W2, nwb=wsn)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                 a["ldy"], a["w"], a["wsb"], a["fl"], a["nw"], a["nwb"], None)

    assert call(M=0) == tq.TQ_OK
    assert call(N=192, ldy=192) == tq.TQ_ERR_SHAPE        # N not a multiple of 128
    assert call(nwb=wsn - 1) == tq.TQ_ERR_SHAPE
    assert call(nw=None) == tq.TQ_ERR_INVALID_ARG
    assert call(nw=W1 + 4096) == tq.TQ_ERR_INVALID_ARG      # overlaps the workspace
    assert call(nw=W2 + 8) == tq.TQ_ERR_ALIGN
    assert call(fl=4) == tq.TQ_ERR_INVALID_ARG
    assert call(fmt=tq.TQ_PACK_BASE3) == tq.TQ_ERR_UNSUPPORTED


def test_sparse24_validation(L):
    assert L.tq_sparse24_ld(5120) == 960 and L.tq_sparse24_ld(27648) == 5184
    assert L.tq_sparse24_ld(100) == -1 and L.tq_sparse24_ld(0) == -1
    assert L.tq_gemv_sparse24_path(5120, 100, 1) == -tq.TQ_ERR_SHAPE
    assert L.tq_gemv_sparse24_path(5120, 5120, 17) == -tq.TQ_ERR_SHAPE
    assert L.tq_gemv_sparse24_path(-1, 5120, 1) == -tq.TQ_ERR_INVALID_ARG
    # x' fp32 (rounded to 256 B), then partial sums when K is split into slices:
    # 55296x5120 needs one slice; 5120x5120 (160 row blocks, aiming at ~512
    # CTAs) is cut into 3 slices of 16 groups; 5120x27648 into 4 of 56
    assert L.tq_gemv_sparse24_workspace_bytes(55296, 5120, 1) == 5120 * 4
    assert L.tq_gemv_sparse24_workspace_bytes(5120, 5120, 1) == 5120 * 4 + 3 * 5120 * 4
    assert L.tq_gemv_sparse24_workspace_bytes(5120, 27648, 1) == 27648 * 4 + 4 * 5120 * 4
    # M = 16: 11 groups of x' per 96 KiB slice -> 20 slices over 216 groups
    assert L.tq_gemv_sparse24_workspace_bytes(5120, 27648, 16) == 16 * 27648 * 4 + 20 * 16 * 5120 * 4
    assert L.tq_gemv_sparse24_workspace_bytes(5120, 100, 1) == 0
    assert L.tq_gemv_sparse24_workspace_bytes(5120, 256, 17) == 0
    q = L.tq_quantize_pack_sparse24
    okq = dict(W=A, wt=tq.TQ_BF16, N=4, K=256, ldw=256, c=B, ldc=48, s=B + 4096, lds=2)

    def callq(**kw):
        a = dict(okq, **kw)
        return q(a["W"], a["wt"], a["N"], a["K"], a["ldw"], a["c"], a["ldc"], a["s"], a["lds"], None)

    assert callq(N=0) == tq.TQ_OK
    assert callq(wt=tq.TQ_F16) == tq.TQ_ERR_INVALID_ARG
    assert callq(N=-1) == tq.TQ_ERR_INVALID_ARG
    assert callq(K=200) == tq.TQ_ERR_SHAPE
    assert callq(c=None) == tq.TQ_ERR_INVALID_ARG
    assert callq(s=None) == tq.TQ_ERR_INVALID_ARG
    assert callq(ldc=47) == tq.TQ_ERR_SHAPE
    assert callq(lds=1) == tq.TQ_ERR_SHAPE
    assert callq(ldw=255) == tq.TQ_ERR_SHAPE
    assert callq(W=MIS) == tq.TQ_ERR_ALIGN
    assert callq(c=B + 2) == tq.TQ_ERR_ALIGN        # codes are written as 32-bit words
    assert callq(ldc=50) == tq.TQ_ERR_ALIGN
    assert callq(s=B + 4097) == tq.TQ_ERR_ALIGN
    g = L.tq_gemv_sparse24
    ws = L.tq_gemv_sparse24_workspace_bytes(64, 256, 2)
    okg = dict(c=B, ldc=48, s=B + 4096, lds=2, N=64, K=256, x=A, ldx=256, M=2, y=B + 8192, ldy=64, w=B + 65536,
               wb=ws)

    def callg(**kw):
        a = dict(okg, **kw)
        return g(a["c"], a["ldc"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"], a["ldy"],
                 a["w"], a["wb"], None)

    assert callg(N=0) == tq.TQ_OK
    assert callg(N=-1) == tq.TQ_ERR_INVALID_ARG
    assert callg(K=100) == tq.TQ_ERR_SHAPE
    assert callg(M=0) == tq.TQ_ERR_SHAPE and callg(M=17) == tq.TQ_ERR_SHAPE
    for k in ("c", "s", "x", "y", "w"):
        assert callg(**{k: None}) == tq.TQ_ERR_INVALID_ARG, k
    assert callg(ldc=47) == tq.TQ_ERR_SHAPE
    assert callg(lds=1) == tq.TQ_ERR_SHAPE
    assert callg(ldx=255) == tq.TQ_ERR_SHAPE
    assert callg(ldy=63) == tq.TQ_ERR_SHAPE
    assert callg(wb=ws - 1) == tq.TQ_ERR_SHAPE
    assert callg(x=MIS) == tq.TQ_ERR_ALIGN
    assert callg(ldx=260) == tq.TQ_ERR_ALIGN        # bf16 rows of x: 16-byte multiples
    assert callg(s=B + 4097) == tq.TQ_ERR_ALIGN
    assert callg(w=B + 65536 + 8) == tq.TQ_ERR_ALIGN
    assert callg(y=B + 8194) == tq.TQ_ERR_ALIGN
    assert callg(c=B + 2) == tq.TQ_ERR_ALIGN        # codes are read as 32-bit words
    assert callg(ldc=50) == tq.TQ_ERR_ALIGN


def test_gemm_sparse24_validation(L):
    f = L.tq_gemm_sparse24
    ws = tq.gemm_workspace_bytes(8, 256)
    ok = dict(c=B, ldc=48, s=B + 4096, lds=2, N=64, K=256, x=A, ldx=256, M=8, y=B + 8192, ldy=64, w=B + 65536, wb=ws)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"], a["ldy"],
                 a["w"], a["wb"], None)

    assert call(N=0) == tq.TQ_OK and call(M=0) == tq.TQ_OK
    assert call(N=-1) == tq.TQ_ERR_INVALID_ARG and call(M=-1) == tq.TQ_ERR_INVALID_ARG
    assert call(K=100) == tq.TQ_ERR_SHAPE
    for k in ("c", "s", "x", "y", "w"):
        assert call(**{k: None}) == tq.TQ_ERR_INVALID_ARG, k
    assert call(ldc=40) == tq.TQ_ERR_SHAPE
    assert call(lds=1) == tq.TQ_ERR_SHAPE
    assert call(ldx=255) == tq.TQ_ERR_SHAPE
    assert call(ldy=63) == tq.TQ_ERR_SHAPE
    assert call(wb=ws - 1) == tq.TQ_ERR_SHAPE
    assert call(c=B + 4) == tq.TQ_ERR_ALIGN          # codes are read as 8-byte words
    assert call(ldc=52) == tq.TQ_ERR_ALIGN
    assert call(x=MIS) == tq.TQ_ERR_ALIGN
    assert call(s=B + 4097) == tq.TQ_ERR_ALIGN
    assert call(y=B + 8194) == tq.TQ_ERR_ALIGN


def test_gemv_rotate_next_validation(L):
    f = L.tq_gemv_rotate_next
    ok = dict(c=B, ldc=64, fmt=tq.TQ_PACK_2BIT, s=B + 4096, lds=2, N=256, K=256, x=A, ldx=256, M=2, y=B + 8192,
              ldy=256, fl=0, xn=B + 65536, ldxn=256)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["c"], a["ldc"], a["fmt"], a["s"], a["lds"], a["N"], a["K"], a["x"], a["ldx"], a["M"], a["y"],
                 a["ldy"], a["fl"], a["xn"], a["ldxn"], None)

    assert call(N=0) == tq.TQ_OK
    assert call(fmt=7) == tq.TQ_ERR_INVALID_ARG
    assert call(fl=0x40) == tq.TQ_ERR_INVALID_ARG
    assert call(N=200, ldy=256, ldxn=256) == tq.TQ_ERR_SHAPE      # N a multiple of 128
    assert call(M=0) == tq.TQ_ERR_SHAPE and call(M=17) == tq.TQ_ERR_SHAPE
    assert call(xn=None) == tq.TQ_ERR_INVALID_ARG
    assert call(ldxn=255) == tq.TQ_ERR_SHAPE
    assert call(xn=B + 65538) == tq.TQ_ERR_ALIGN
    assert call(xn=B + 8192 + 512) == tq.TQ_ERR_INVALID_ARG      # overlaps y
    assert call(x=MIS) == tq.TQ_ERR_ALIGN                         # bf16 x: 16-byte rows
    # rotated fp32 x needs 4-byte alignment only
    g = L.tq_gemv_ex
    assert g(B, 64, tq.TQ_PACK_2BIT, B + 4096, 2, 0, 256, MIS, 256, 1, B + 8192, 256, tq.TQ_GEMV_X_ROTATED,
             None) == tq.TQ_OK
    assert g(B, 64, tq.TQ_PACK_2BIT, B + 4096, 2, 4, 256, A + 2, 256, 1, B + 8192, 256, tq.TQ_GEMV_X_ROTATED,
             None) == tq.TQ_ERR_ALIGN
