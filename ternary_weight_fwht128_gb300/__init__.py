"""Python binding of libtq (ternary weights after a block FWHT-128, on GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/tq.h``.  PyTorch provides the
device memory and the current CUDA stream.  There is no CPU fallback: if the
library is not built, every call raises.

Functions (names follow the C ABI):
  fwht128(x, out_dtype)                 x' = blockdiag(H_128)/sqrt(128) x along K
  quantize_pack(W, fmt)                 (codes2, codes3, scales)
  gemv(codes, scales, x, K, fmt)        y fp32 [M][N], M = 1..16
  gemm(codes, scales, x, K, fmt, ws)    y fp32 [M][N] on tcgen05 tensor cores
  gemm_workspace_bytes(M, K), gemm_check_range(ws)
  Layout variants (FWHT block 64/128/256, scale group 128/256, residual
  pass): fwht(x, block), quantize_pack_layout, gemv_layout, gemm_layout,
  layout_codes_ld, layout_scales_ld, gemm_workspace_bytes_layout
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as _LIB_PATH

(TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_SHAPE, TQ_ERR_ALIGN, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_RANGE,
 TQ_ERR_TIMEOUT) = range(8)
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
TQ_PACK_2BIT, TQ_PACK_BASE3, TQ_PACK_BOTH = 1, 2, 3

EXPORTED = ("tq_status_string", "tq_version", "tq_packed_ld", "tq_fwht128", "tq_quantize_pack", "tq_gemv",
            "tq_gemv_ex", "tq_gemv_path", "tq_gemv_plan", "tq_gemm_workspace_bytes", "tq_gemm", "tq_gemm_ex", "tq_gemm_check_range",
            "tq_device_fault", "tq_gemm_noalloc", "tq_layout_codes_ld", "tq_layout_scales_ld", "tq_fwht",
            "tq_quantize_pack_layout", "tq_gemv_layout", "tq_gemm_workspace_bytes_layout", "tq_gemm_layout",
            "tq_gemm_rotate_next", "tq_sparse24_ld", "tq_quantize_pack_sparse24",
            "tq_gemv_sparse24_workspace_bytes", "tq_gemv_sparse24", "tq_gemm_sparse24", "tq_gemv_rotate_next",
            "tq_gemv_sparse24_path")
TQ_GEMV_TENSOR_MEMORY, TQ_GEMV_MMA_SYNC, TQ_GEMV_CUDA_CORES = 1, 2, 3
TQ_GEMV_WEIGHTS_READY = 1
TQ_GEMV_X_ROTATED = 2
TQ_GEMM_REUSE_ROTATED = 1
TQ_GEMV_TEST_STALL = 0x100
TQ_GEMM_TEST_STALL = 0x100
TQ_LAYOUT_RESIDUAL = 1


class Layout(ctypes.Structure):
    """tq_layout: FWHT block size, weights per scale, flags (TQ_LAYOUT_RESIDUAL)."""
    _fields_ = [("block", ctypes.c_int32), ("group", ctypes.c_int32), ("flags", ctypes.c_uint32)]


def layout(block: int = 128, group: int = 128, residual: bool = False) -> Layout:
    return Layout(block, group, TQ_LAYOUT_RESIDUAL if residual else 0)

_lib = None
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_int = ctypes.c_int


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libtq.so is not built ({_LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        L.tq_status_string.restype = ctypes.c_char_p
        L.tq_status_string.argtypes = [_int]
        L.tq_version.restype = _int
        L.tq_packed_ld.restype = _i64
        L.tq_packed_ld.argtypes = [_i64, _int]
        L.tq_fwht128.restype = _int
        L.tq_fwht128.argtypes = [_vp, _int, _i64, _vp, _int, _i64, _i64, _i64, _vp]
        L.tq_quantize_pack.restype = _int
        L.tq_quantize_pack.argtypes = [_vp, _int, _i64, _i64, _i64, _int, _vp, _i64, _vp, _i64, _vp, _i64, _vp]
        L.tq_gemv.restype = _int
        L.tq_gemv.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp]
        L.tq_gemv_ex.restype = _int
        L.tq_gemv_ex.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, ctypes.c_uint,
                                 _vp]
        L.tq_gemv_path.restype = _int
        L.tq_gemv_path.argtypes = [_i64, _i64, _i64, _int]
        L.tq_gemv_plan.restype = _int
        L.tq_gemv_plan.argtypes = [_i64, _i64, _i64, _int, _int, _vp, _vp, _vp]
        L.tq_gemm_workspace_bytes.restype = ctypes.c_size_t
        L.tq_gemm_workspace_bytes.argtypes = [_i64, _i64]
        L.tq_gemm.restype = _int
        L.tq_gemm.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                              ctypes.c_size_t, _vp]
        L.tq_gemm_ex.restype = _int
        L.tq_gemm_ex.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                 ctypes.c_size_t, ctypes.c_uint, _vp]
        L.tq_gemm_check_range.restype = _int
        L.tq_gemm_check_range.argtypes = [_vp, _vp]
        L.tq_device_fault.restype = _int
        L.tq_device_fault.argtypes = []
        L.tq_gemm_noalloc.restype = _int
        L.tq_gemm_noalloc.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp]
        L.tq_gemm_rotate_next.restype = _int
        L.tq_gemm_rotate_next.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                          ctypes.c_size_t, ctypes.c_uint, _vp, ctypes.c_size_t, _vp]
        lp = ctypes.POINTER(Layout)
        L.tq_layout_codes_ld.restype = _i64
        L.tq_layout_codes_ld.argtypes = [_i64, _int, lp]
        L.tq_layout_scales_ld.restype = _i64
        L.tq_layout_scales_ld.argtypes = [_i64, lp]
        L.tq_fwht.restype = _int
        L.tq_fwht.argtypes = [_vp, _int, _i64, _vp, _int, _i64, _i64, _i64, _int, _vp]
        L.tq_quantize_pack_layout.restype = _int
        L.tq_quantize_pack_layout.argtypes = [_vp, _int, _i64, _i64, _i64, _int, _vp, _i64, _vp, _i64, _vp, _i64, lp,
                                              _vp]
        L.tq_gemv_layout.restype = _int
        L.tq_gemv_layout.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, lp,
                                     ctypes.c_uint, _vp]
        L.tq_gemm_workspace_bytes_layout.restype = ctypes.c_size_t
        L.tq_gemm_workspace_bytes_layout.argtypes = [_i64, _i64, lp]
        L.tq_gemm_layout.restype = _int
        L.tq_gemm_layout.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                     ctypes.c_size_t, lp, ctypes.c_uint, _vp]
        L.tq_sparse24_ld.restype = _i64
        L.tq_sparse24_ld.argtypes = [_i64]
        L.tq_quantize_pack_sparse24.restype = _int
        L.tq_quantize_pack_sparse24.argtypes = [_vp, _int, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
        L.tq_gemv_sparse24_workspace_bytes.restype = ctypes.c_size_t
        L.tq_gemv_sparse24_workspace_bytes.argtypes = [_i64, _i64, _i64]
        L.tq_gemv_rotate_next.restype = _int
        L.tq_gemv_rotate_next.argtypes = [_vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64,
                                          ctypes.c_uint, _vp, _i64, _vp]
        L.tq_gemm_sparse24.restype = _int
        L.tq_gemm_sparse24.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                       ctypes.c_size_t, _vp]
        L.tq_gemv_sparse24.restype = _int
        L.tq_gemv_sparse24.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp,
                                       ctypes.c_size_t, _vp]
        L.tq_gemv_sparse24_path.restype = _int
        L.tq_gemv_sparse24_path.argtypes = [_i64, _i64, _i64]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().tq_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != TQ_OK:
        raise TQError(status, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    if t.dtype == torch.float16:
        return TQ_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cuda2d(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit stride along its last dimension")


def packed_ld(K: int, fmt: int) -> int:
    return int(lib().tq_packed_ld(K, fmt))


def fwht128(x: torch.Tensor, out_dtype: torch.dtype = torch.float32, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Block FWHT-128 of every row of x (fp32 or bf16) along its last dimension."""
    _cuda2d(x, "x")
    rows, K = x.shape
    if out is None:
        out = torch.empty((rows, K), dtype=out_dtype, device=x.device)
    _cuda2d(out, "out")
    st = lib().tq_fwht128(x.data_ptr(), _dt(x), x.stride(0), out.data_ptr(), _dt(out), out.stride(0), rows, K,
                          _stream(stream))
    _check(st, "tq_fwht128")
    return out


def quantize_pack(W: torch.Tensor, fmt: int = TQ_PACK_BOTH, stream=None, out=None):
    """Rotate, ternarise and pack W [N][K] (fp32 or bf16).

    Returns (codes2 uint8 [N][K/4] or None, codes3 uint8 [N][ld3] or None,
    scales int16 [N][K/128] holding fp16 bit patterns).  out: an earlier
    (codes2, codes3, scales) triple of this shape and format to write into."""
    _cuda2d(W, "W")
    N, K = W.shape
    dev = W.device
    ld3 = packed_ld(K, TQ_PACK_BASE3) if K > 0 else 0
    if out is None:
        codes2 = torch.empty((N, K // 4), dtype=torch.uint8, device=dev) if fmt & TQ_PACK_2BIT else None
        codes3 = torch.empty((N, max(ld3, 0)), dtype=torch.uint8, device=dev) if fmt & TQ_PACK_BASE3 else None
        scales = torch.empty((N, K // 128), dtype=torch.int16, device=dev)
    else:
        codes2, codes3, scales = out
        for t, name in ((codes2, "codes2"), (codes3, "codes3"), (scales, "scales")):
            if t is not None:
                _cuda2d(t, name)
    st = lib().tq_quantize_pack(W.data_ptr(), _dt(W), N, K, W.stride(0), fmt,
                                codes2.data_ptr() if codes2 is not None else None,
                                codes2.stride(0) if codes2 is not None else 0,
                                codes3.data_ptr() if codes3 is not None else None,
                                codes3.stride(0) if codes3 is not None else 0,
                                scales.data_ptr(), scales.stride(0), _stream(stream))
    _check(st, "tq_quantize_pack")
    return codes2, codes3, scales


def gemv(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int, fmt: int = TQ_PACK_2BIT,
         out: torch.Tensor | None = None, stream=None, weights_ready: bool = False,
         x_rotated: bool = False) -> torch.Tensor:
    """y [M][N] fp32 = ternary GEMV/skinny GEMM of bf16 x [M][K] (M <= 16).
    weights_ready: codes and scales were complete before the work preceding
    this call on the stream started (tq_gemv_ex, TQ_GEMV_WEIGHTS_READY).
    x_rotated: x is the fp32 FWHT-128 of the activations, as gemv_rotate_next
    writes it (TQ_GEMV_X_ROTATED)."""
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    flags = (TQ_GEMV_WEIGHTS_READY if weights_ready else 0) | (TQ_GEMV_X_ROTATED if x_rotated else 0)
    st = lib().tq_gemv_ex(codes.data_ptr(), codes.stride(0), fmt, scales.data_ptr(), scales.stride(0), N, K,
                          x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), flags, _stream(stream))
    _check(st, "tq_gemv_ex")
    return out


def gemv_path(N: int, K: int, M: int = 1, fmt: int = TQ_PACK_2BIT) -> int:
    """Which kernel tq_gemv runs for the shape: TQ_GEMV_TENSOR_MEMORY or
    TQ_GEMV_MMA_SYNC (queries the current CUDA device; launches nothing)."""
    r = int(lib().tq_gemv_path(N, K, M, fmt))
    if r < 0:
        raise TQError(-r, "tq_gemv_path")
    return r


def gemv_plan(N: int, K: int, M: int = 1, fmt: int = TQ_PACK_2BIT, chained: bool = False) -> tuple[int, int, int]:
    """The tensor-memory kernel's split for the shape (tq_gemv_plan):
    (CTAs per cluster, clusters, launches)."""
    v = (ctypes.c_int * 3)()
    base = ctypes.addressof(v)
    st = lib().tq_gemv_plan(N, K, M, fmt, 1 if chained else 0, base, base + 4, base + 8)
    _check(st, "tq_gemv_plan")
    return int(v[0]), int(v[1]), int(v[2])


def gemm_workspace_bytes(M: int, K: int) -> int:
    return int(lib().tq_gemm_workspace_bytes(M, K))


def gemm(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int, fmt: int = TQ_PACK_2BIT,
         workspace: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None,
         reuse_rotated: bool = False) -> torch.Tensor:
    """y [M][N] fp32 = prefill GEMM of bf16 x [M][K] on tcgen05 tensor cores.
    reuse_rotated: `workspace` already holds the rotated x of the previous
    gemm call on it with this same x (tq_gemm_ex, TQ_GEMM_REUSE_ROTATED)."""
    if reuse_rotated and workspace is None:
        raise ValueError("reuse_rotated needs the workspace of the previous call")
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, K), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    flags = TQ_GEMM_REUSE_ROTATED if reuse_rotated else 0
    st = lib().tq_gemm_ex(codes.data_ptr(), codes.stride(0), fmt, scales.data_ptr(), scales.stride(0), N, K,
                          x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), flags, _stream(stream))
    _check(st, "tq_gemm_ex")
    return out


def device_fault() -> None:
    """Raises TQError(TQ_ERR_TIMEOUT) if a kernel gave up a bounded wait since
    the last call (synchronises the device)."""
    _check(lib().tq_device_fault(), "tq_device_fault")


def gemm_check_range(workspace: torch.Tensor, stream=None) -> None:
    """Raises TQError(TQ_ERR_RANGE) if the last tq_gemm saw an fp16 overflow."""
    _check(lib().tq_gemm_check_range(workspace.data_ptr(), _stream(stream)), "tq_gemm_check_range")


# ------------------------------------------------------------ layout variants

def _lp(lay: Layout | None):
    return None if lay is None else ctypes.byref(lay)


def layout_codes_ld(K: int, fmt: int, lay: Layout | None) -> int:
    return int(lib().tq_layout_codes_ld(K, fmt, _lp(lay)))


def layout_scales_ld(K: int, lay: Layout | None) -> int:
    return int(lib().tq_layout_scales_ld(K, _lp(lay)))


def fwht(x: torch.Tensor, block: int = 128, out_dtype: torch.dtype = torch.float32, out: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """Block FWHT (block 64, 128 or 256) of every row of x along its last dimension."""
    _cuda2d(x, "x")
    rows, K = x.shape
    if out is None:
        out = torch.empty((rows, K), dtype=out_dtype, device=x.device)
    _cuda2d(out, "out")
    st = lib().tq_fwht(x.data_ptr(), _dt(x), x.stride(0), out.data_ptr(), _dt(out), out.stride(0), rows, K, block,
                       _stream(stream))
    _check(st, "tq_fwht")
    return out


def quantize_pack_layout(W: torch.Tensor, lay: Layout, fmt: int = TQ_PACK_BOTH, stream=None):
    """quantize_pack under a layout: (codes2 [N][ld2] or None, codes3 [N][ld3] or
    None, scales int16 [N][Geff]); codes hold Keff = K (2K with the residual pass)."""
    _cuda2d(W, "W")
    N, K = W.shape
    dev = W.device
    ld2 = layout_codes_ld(K, TQ_PACK_2BIT, lay)
    ld3 = layout_codes_ld(K, TQ_PACK_BASE3, lay)
    lds = layout_scales_ld(K, lay)
    if min(ld2, ld3, lds) < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_layout_codes_ld")
    codes2 = torch.empty((N, ld2), dtype=torch.uint8, device=dev) if fmt & TQ_PACK_2BIT else None
    codes3 = torch.empty((N, ld3), dtype=torch.uint8, device=dev) if fmt & TQ_PACK_BASE3 else None
    scales = torch.empty((N, lds), dtype=torch.int16, device=dev)
    st = lib().tq_quantize_pack_layout(W.data_ptr(), _dt(W), N, K, W.stride(0), fmt,
                                       codes2.data_ptr() if codes2 is not None else None, ld2,
                                       codes3.data_ptr() if codes3 is not None else None, ld3,
                                       scales.data_ptr(), scales.stride(0), _lp(lay), _stream(stream))
    _check(st, "tq_quantize_pack_layout")
    return codes2, codes3, scales


def gemv_layout(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int, lay: Layout,
                fmt: int = TQ_PACK_2BIT, out: torch.Tensor | None = None, stream=None, flags: int = 0) -> torch.Tensor:
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().tq_gemv_layout(codes.data_ptr(), codes.stride(0), fmt, scales.data_ptr(), scales.stride(0), N, K,
                              x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), _lp(lay), flags,
                              _stream(stream))
    _check(st, "tq_gemv_layout")
    return out


def gemm_workspace_bytes_layout(M: int, K: int, lay: Layout | None) -> int:
    return int(lib().tq_gemm_workspace_bytes_layout(M, K, _lp(lay)))


def gemm_layout(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int, lay: Layout,
                fmt: int = TQ_PACK_2BIT, workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                stream=None, flags: int = 0) -> torch.Tensor:
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes_layout(M, K, lay), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().tq_gemm_layout(codes.data_ptr(), codes.stride(0), fmt, scales.data_ptr(), scales.stride(0), N, K,
                              x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _lp(lay), flags, _stream(stream))
    _check(st, "tq_gemm_layout")
    return out


def gemm_rotate_next(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int, next_ws: torch.Tensor,
                     workspace: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None,
                     flags: int = 0) -> torch.Tensor:
    """gemm that also writes FWHT-128(y) into next_ws as the x' of a following
    gemm(..., workspace=next_ws, reuse_rotated=True) whose x is this y."""
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, K), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().tq_gemm_rotate_next(codes.data_ptr(), codes.stride(0), TQ_PACK_2BIT, scales.data_ptr(),
                                   scales.stride(0), N, K, x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0),
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(), flags,
                                   next_ws.data_ptr(), next_ws.numel() * next_ws.element_size(), _stream(stream))
    _check(st, "tq_gemm_rotate_next")
    return out


# ---- 2:4-sparse ternary weights (tq_quantize_pack_sparse24, tq_gemv_sparse24)

def sparse24_ld(K: int) -> int:
    """Bytes of 2:4 codes per row (24 per group of 128)."""
    r = int(lib().tq_sparse24_ld(K))
    if r < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_sparse24_ld")
    return r


def quantize_pack_sparse24(W: torch.Tensor, out=None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """(codes uint8 [N][24 K/128], scales int16 [N][K/128] with fp16 bits) of
    W (fp32 or bf16 [N][K]) in the 2:4-sparse ternary format."""
    _cuda2d(W, "W")
    N, K = W.shape
    if out is None:
        codes = torch.empty((N, 24 * (K // 128)), dtype=torch.uint8, device=W.device)
        scales = torch.empty((N, K // 128), dtype=torch.int16, device=W.device)
    else:
        codes, scales = out
        _cuda2d(codes, "codes")
        _cuda2d(scales, "scales")
    st = lib().tq_quantize_pack_sparse24(W.data_ptr(), _dt(W), N, K, W.stride(0), codes.data_ptr(),
                                         codes.stride(0), scales.data_ptr(), scales.stride(0), _stream(stream))
    _check(st, "tq_quantize_pack_sparse24")
    return codes, scales


def gemv_sparse24_workspace_bytes(N: int, K: int, M: int) -> int:
    return int(lib().tq_gemv_sparse24_workspace_bytes(N, K, M))


def gemv_sparse24(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int,
                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """y [M][N] fp32 of the 2:4 codes and bf16 x [M][K] (M <= 16)."""
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(max(gemv_sparse24_workspace_bytes(N, K, M), 16), dtype=torch.uint8,
                                device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().tq_gemv_sparse24(codes.data_ptr(), codes.stride(0), scales.data_ptr(), scales.stride(0), N, K,
                                x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "tq_gemv_sparse24")
    return out


def gemm_sparse24(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int,
                  workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Prefill y [M][N] fp32 of the 2:4 codes and bf16 x [M][K] on the tensor cores."""
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, K), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().tq_gemm_sparse24(codes.data_ptr(), codes.stride(0), scales.data_ptr(), scales.stride(0), N, K,
                                x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "tq_gemm_sparse24")
    return out


def gemv_rotate_next(codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, K: int,
                     fmt: int = TQ_PACK_2BIT, xnext: torch.Tensor | None = None, out: torch.Tensor | None = None,
                     stream=None, weights_ready: bool = False, x_rotated: bool = False,
                     flags: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """(y, xnext): gemv that also writes FWHT-128(y) in fp32 as the x of a
    following gemv(..., x_rotated=True) (tq_gemv_rotate_next)."""
    _cuda2d(codes, "codes")
    _cuda2d(scales, "scales")
    _cuda2d(x, "x")
    N = codes.shape[0]
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if xnext is None:
        xnext = torch.empty((M, N), dtype=torch.float32, device=x.device)
    flags |= (TQ_GEMV_WEIGHTS_READY if weights_ready else 0) | (TQ_GEMV_X_ROTATED if x_rotated else 0)
    st = lib().tq_gemv_rotate_next(codes.data_ptr(), codes.stride(0), fmt, scales.data_ptr(), scales.stride(0), N, K,
                                   x.data_ptr(), x.stride(0), M, out.data_ptr(), out.stride(0), flags,
                                   xnext.data_ptr(), xnext.stride(0), _stream(stream))
    _check(st, "tq_gemv_rotate_next")
    return out, xnext


def gemv_sparse24_path(N: int, K: int, M: int = 1) -> int:
    """TQ_GEMV_TENSOR_MEMORY or TQ_GEMV_CUDA_CORES (tq_gemv_sparse24_path)."""
    return lib().tq_gemv_sparse24_path(N, K, M)
