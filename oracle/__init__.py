"""Plain CPU oracle for the ternary FWHT-128 linear layers (ctypes over tq_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

Each wrapper below marshals numpy arrays into the C functions; the arithmetic
lives in ``tq_oracle.c`` (documented there, with the page sections it follows).

Parity status of each function (what pins it, see ``tests/test_oracle.py``):
  hadamard_entry      pinned: equals the Sylvester recursion and scipy.linalg.hadamard
  fwht128_f32         pinned: equals the dense fp64 rotation within fp32 rounding,
                      delta inputs give exactly +-c, involution, energy
  fwht128_f64         pinned: equals scipy-built H @ v / sqrt(128) to 1e-13
  f32_to_f16 / back   pinned: equals numpy's IEEE conversion on every boundary case
  quantize_group      pinned: closed forms (constant magnitude, zero group, ties at
                      0.5 and 1.5 and their fp32 neighbours), compare-rule identity
  pack2/pack3         pinned: hand-worked bytes in tests/golden, round trip,
                      byte range, bit accounting
  gemv_f64            pinned: dense dequantised fp64 matmul with a scipy-built
                      block rotation, rotation invariance, delta activations
  Sparse24Oracle      2:4 pattern (two largest |w'| per quad), absmean over the
                      kept 64, joint 6-bit codes: pinned by a brute-force pattern
                      search, every one of the 54 codes by hand, closed-form
                      scales, order-sensitive sums over 64, the bit budget, and
                      a dense fp64 GEMV of the expanded trits
  LayoutOracle        block sizes 64/128/256, groups 128/256, residual pass:
                      pinned by scipy's H_n, the n = 128 functions above (bit
                      for bit), exact normalisation constants, order-sensitive
                      sums over 256, a closed-form residual of a delta row, the
                      residual's error reduction, and a dense fp64 GEMV
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()
_cache: dict[str, "Oracle"] = {}


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags: list[str] | None = None) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), "-I", _HERE, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _stale(lib: str, src: str) -> bool:
    if not os.path.exists(lib):
        return True
    m = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > m for p in (src, os.path.join(_HERE, "tq_oracle.h")))


_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_vp)


class Oracle:
    """One loaded copy of the oracle library (the tests also load mutated copies)."""

    def __init__(self, path: str):
        self.path = path
        L = ctypes.CDLL(path)
        self._L = L
        L.tqo_hadamard_entry.restype = ctypes.c_int
        L.tqo_hadamard_entry.argtypes = [ctypes.c_int, ctypes.c_int]
        L.tqo_sylvester.argtypes = [ctypes.c_int, _vp]
        L.tqo_norm_const_bits.restype = ctypes.c_uint32
        L.tqo_fwht128_f32.argtypes = [_vp, _vp]
        L.tqo_fwht128_f64.argtypes = [_vp, _vp]
        L.tqo_f32_to_f16.restype = ctypes.c_uint16
        L.tqo_f32_to_f16.argtypes = [ctypes.c_float]
        L.tqo_f16_to_f32.restype = ctypes.c_float
        L.tqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.tqo_quantize_group.restype = ctypes.c_uint16
        L.tqo_quantize_group.argtypes = [_vp, _vp]
        L.tqo_quantize_rows.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _i64, _vp, _vp]
        L.tqo_pack2.argtypes = [_vp, _i64, _i64, _vp, _i64]
        L.tqo_unpack2.argtypes = [_vp, _i64, _i64, _i64, _vp]
        L.tqo_ld3.restype = _i64
        L.tqo_ld3.argtypes = [_i64]
        L.tqo_pack3.argtypes = [_vp, _i64, _i64, _vp, _i64]
        L.tqo_unpack3.argtypes = [_vp, _i64, _i64, _i64, _vp]
        L.tqo_gemv_f64.argtypes = [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
        L.tqo_norm_const_bits_n.restype = ctypes.c_uint32
        L.tqo_norm_const_bits_n.argtypes = [ctypes.c_int]
        L.tqo_fwht_f32.argtypes = [ctypes.c_int, _vp, _vp]
        L.tqo_fwht_f64.argtypes = [ctypes.c_int, _vp, _vp]
        L.tqo_quantize_group_n.restype = ctypes.c_uint16
        L.tqo_quantize_group_n.argtypes = [ctypes.c_int, _vp, _vp]
        L.tqo_quantize_layout_rows.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _i64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, _vp, _vp]
        L.tqo_gemv_layout_f64.argtypes = [_vp, _vp, _i64, _vp, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _vp]
        L.tqo_quantize_group_24.restype = ctypes.c_uint16
        L.tqo_quantize_group_24.argtypes = [_vp, _vp, _vp]
        L.tqo_quantize_rows_24.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _i64, _vp, _vp, _vp]
        L.tqo_ld24.restype = _i64
        L.tqo_ld24.argtypes = [_i64]
        L.tqo_pack24.argtypes = [_vp, _vp, _i64, _i64, _vp, _i64]
        L.tqo_unpack24.restype = _i64
        L.tqo_unpack24.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]

    # -- Hadamard -------------------------------------------------------
    def hadamard_entry(self, i: int, j: int) -> int:
        return int(self._L.tqo_hadamard_entry(i, j))

    def hadamard(self, n: int) -> np.ndarray:
        return np.array([[self.hadamard_entry(i, j) for j in range(n)] for i in range(n)], dtype=np.int64)

    def sylvester(self, n: int) -> np.ndarray:
        h = np.zeros((n, n), dtype=np.int8)
        self._L.tqo_sylvester(n, _p(h))
        return h.astype(np.int64)

    def norm_const_bits(self) -> int:
        return int(self._L.tqo_norm_const_bits())

    def fwht128_f32(self, v: np.ndarray) -> np.ndarray:
        """Rotate every 128-block of the last axis (fp32 staged butterflies)."""
        a = np.ascontiguousarray(v, dtype=np.float32)
        flat = a.reshape(-1, 128)
        out = np.empty_like(flat)
        for r in range(flat.shape[0]):
            self._L.tqo_fwht128_f32(_p(flat[r]), _p(out[r]))
        return out.reshape(a.shape)

    def fwht128_f64(self, v: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float64)
        flat = a.reshape(-1, 128)
        out = np.empty_like(flat)
        for r in range(flat.shape[0]):
            self._L.tqo_fwht128_f64(_p(flat[r]), _p(out[r]))
        return out.reshape(a.shape)

    # -- fp16 -----------------------------------------------------------
    def f32_to_f16(self, f: float) -> int:
        return int(self._L.tqo_f32_to_f16(ctypes.c_float(f)))

    def f16_to_f32(self, h: int) -> float:
        return float(self._L.tqo_f16_to_f32(ctypes.c_uint16(h)))

    # -- quantiser ------------------------------------------------------
    def quantize_group(self, wrot: np.ndarray) -> tuple[int, np.ndarray]:
        w = np.ascontiguousarray(wrot, dtype=np.float32)
        assert w.shape == (128,)
        t = np.zeros(128, dtype=np.int8)
        s = self._L.tqo_quantize_group(_p(w), _p(t))
        return int(s), t

    def quantize(self, W: np.ndarray, rows: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
        """Quantise W (fp32 array, or uint16 array holding bf16 bits).

        Returns (T int8 [R][K], S uint16 fp16-bits [R][K/128]) for all rows or
        for the listed rows."""
        W = np.ascontiguousarray(W)
        if W.dtype == np.float32:
            wt = 0
        elif W.dtype == np.uint16:
            wt = 1
        else:
            raise TypeError("W must be float32 or uint16 (bf16 bits)")
        N, K = W.shape
        if K % 128:
            raise ValueError("K must be a multiple of 128")
        if rows is None:
            R, rp = N, None
        else:
            rp = np.ascontiguousarray(rows, dtype=np.int64)
            R = rp.shape[0]
        T = np.zeros((R, K), dtype=np.int8)
        S = np.zeros((R, K // 128), dtype=np.uint16)
        self._L.tqo_quantize_rows(_p(W), wt, K, K, _p(rp), R, _p(T), _p(S))
        return T, S

    # -- packing --------------------------------------------------------
    def ld3(self, K: int) -> int:
        return int(self._L.tqo_ld3(K))

    def pack2(self, T: np.ndarray, ld: int | None = None) -> np.ndarray:
        T = np.ascontiguousarray(T, dtype=np.int8)
        N, K = T.shape
        ld = K // 4 if ld is None else ld
        out = np.zeros((N, ld), dtype=np.uint8)
        self._L.tqo_pack2(_p(T), N, K, _p(out), ld)
        return out

    def unpack2(self, codes: np.ndarray, K: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, ld = codes.shape
        T = np.zeros((N, K), dtype=np.int8)
        self._L.tqo_unpack2(_p(codes), ld, N, K, _p(T))
        return T

    def pack3(self, T: np.ndarray, ld: int | None = None) -> np.ndarray:
        T = np.ascontiguousarray(T, dtype=np.int8)
        N, K = T.shape
        ld = self.ld3(K) if ld is None else ld
        out = np.zeros((N, ld), dtype=np.uint8)
        self._L.tqo_pack3(_p(T), N, K, _p(out), ld)
        return out

    def unpack3(self, codes: np.ndarray, K: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, ld = codes.shape
        T = np.zeros((N, K), dtype=np.int8)
        self._L.tqo_unpack3(_p(codes), ld, N, K, _p(T))
        return T

    # -- GEMV -----------------------------------------------------------
    def gemv(self, T: np.ndarray, S: np.ndarray, x: np.ndarray) -> np.ndarray:
        """fp64 y [M][R] from trits T [R][K], fp16-bit scales S [R][G] and
        activations x [M][K] (fp32 values, normally bf16-exact)."""
        T = np.ascontiguousarray(T, dtype=np.int8)
        S = np.ascontiguousarray(S, dtype=np.uint16)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
        R, K = T.shape
        M = x.shape[0]
        assert x.shape[1] == K and S.shape == (R, K // 128)
        y = np.zeros((M, R), dtype=np.float64)
        self._L.tqo_gemv_f64(_p(T), _p(S), R, K, _p(x), M, None, R, _p(y))
        return y


class LayoutOracle:
    """The transform / group / residual variants of the oracle (see
    tqo_quantize_layout_rows in tq_oracle.c), on a loaded Oracle."""

    def __init__(self, orc: Oracle):
        self._L = orc._L

    def norm_const_bits(self, n: int) -> int:
        return int(self._L.tqo_norm_const_bits_n(n))

    def fwht_f32(self, n: int, v: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float32)
        flat = a.reshape(-1, n)
        out = np.empty_like(flat)
        for r in range(flat.shape[0]):
            self._L.tqo_fwht_f32(n, _p(flat[r]), _p(out[r]))
        return out.reshape(a.shape)

    def fwht_f64(self, n: int, v: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float64)
        flat = a.reshape(-1, n)
        out = np.empty_like(flat)
        for r in range(flat.shape[0]):
            self._L.tqo_fwht_f64(n, _p(flat[r]), _p(out[r]))
        return out.reshape(a.shape)

    def quantize_group(self, g: int, wrot: np.ndarray) -> tuple[int, np.ndarray]:
        w = np.ascontiguousarray(wrot, dtype=np.float32)
        assert w.shape == (g,)
        t = np.zeros(g, dtype=np.int8)
        s = self._L.tqo_quantize_group_n(g, _p(w), _p(t))
        return int(s), t

    def quantize(self, W: np.ndarray, block: int = 128, group: int = 128, residual: bool = False,
                 rows: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
        """(T int8 [R][Keff], S uint16 [R][Geff]) of W (fp32, or uint16 bf16 bits)."""
        W = np.ascontiguousarray(W)
        wt = 0 if W.dtype == np.float32 else 1
        if W.dtype not in (np.float32, np.uint16):
            raise TypeError("W must be float32 or uint16 (bf16 bits)")
        N, K = W.shape
        if K % max(block, group):
            raise ValueError("K must be a multiple of the block and the group size")
        rp = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = N if rp is None else rp.shape[0]
        f = 2 if residual else 1
        T = np.zeros((R, f * K), dtype=np.int8)
        S = np.zeros((R, f * (K // group)), dtype=np.uint16)
        self._L.tqo_quantize_layout_rows(_p(W), wt, K, K, _p(rp), R, block, group, 1 if residual else 0, _p(T), _p(S))
        return T, S

    def gemv(self, T: np.ndarray, S: np.ndarray, x: np.ndarray, block: int = 128, group: int = 128,
             residual: bool = False) -> np.ndarray:
        T = np.ascontiguousarray(T, dtype=np.int8)
        S = np.ascontiguousarray(S, dtype=np.uint16)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
        R = T.shape[0]
        M, K = x.shape
        f = 2 if residual else 1
        assert T.shape == (R, f * K) and S.shape == (R, f * (K // group))
        y = np.zeros((M, R), dtype=np.float64)
        self._L.tqo_gemv_layout_f64(_p(T), _p(S), K, _p(x), M, R, block, group, 1 if residual else 0, _p(y))
        return y


class Sparse24Oracle:
    """The 2:4-sparse ternary format of the oracle (tqo_quantize_group_24 and
    the functions after it in tq_oracle.c), on a loaded Oracle."""

    def __init__(self, orc: Oracle):
        self._orc = orc
        self._L = orc._L

    def quantize_group(self, wrot: np.ndarray) -> tuple[int, np.ndarray, np.ndarray]:
        """(fp16 scale bits, t int8[128], keep uint8[128]) of one rotated group."""
        w = np.ascontiguousarray(wrot, dtype=np.float32)
        assert w.shape == (128,)
        t = np.zeros(128, dtype=np.int8)
        keep = np.zeros(128, dtype=np.uint8)
        s = self._L.tqo_quantize_group_24(_p(w), _p(t), _p(keep))
        return int(s), t, keep

    def quantize(self, W: np.ndarray, rows: np.ndarray | None = None
                 ) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """(T int8 [R][K], KEEP uint8 [R][K], S uint16 [R][K/128]) of W (fp32 or bf16 bits)."""
        W = np.ascontiguousarray(W)
        if W.dtype not in (np.float32, np.uint16):
            raise TypeError("W must be float32 or uint16 (bf16 bits)")
        wt = 0 if W.dtype == np.float32 else 1
        N, K = W.shape
        if K % 128:
            raise ValueError("K must be a multiple of 128")
        rp = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = N if rp is None else rp.shape[0]
        T = np.zeros((R, K), dtype=np.int8)
        KEEP = np.zeros((R, K), dtype=np.uint8)
        S = np.zeros((R, K // 128), dtype=np.uint16)
        self._L.tqo_quantize_rows_24(_p(W), wt, K, K, _p(rp), R, _p(T), _p(KEEP), _p(S))
        return T, KEEP, S

    def ld(self, K: int) -> int:
        return int(self._L.tqo_ld24(K))

    def pack(self, T: np.ndarray, KEEP: np.ndarray, ld: int | None = None) -> np.ndarray:
        T = np.ascontiguousarray(T, dtype=np.int8)
        KEEP = np.ascontiguousarray(KEEP, dtype=np.uint8)
        N, K = T.shape
        ld = self.ld(K) if ld is None else ld
        codes = np.zeros((N, ld), dtype=np.uint8)
        self._L.tqo_pack24(_p(T), _p(KEEP), N, K, _p(codes), ld)
        return codes

    def unpack(self, codes: np.ndarray, K: int) -> tuple[np.ndarray, np.ndarray, int]:
        """(T, KEEP, number of invalid codes) of a packed tensor."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        N, ld = codes.shape
        T = np.zeros((N, K), dtype=np.int8)
        KEEP = np.zeros((N, K), dtype=np.uint8)
        bad = self._L.tqo_unpack24(_p(codes), ld, N, K, _p(T), _p(KEEP))
        return T, KEEP, int(bad)

    def gemv(self, codes: np.ndarray, S: np.ndarray, x: np.ndarray, K: int) -> np.ndarray:
        """fp64 y [M][N] of the packed weights: the dense GEMV of the unpacked trits."""
        T, _, bad = self.unpack(codes, K)
        if bad:
            raise ValueError("invalid 2:4 codes")
        return self._orc.gemv(T, S, x)


def load(path: str | None = None) -> Oracle:
    """Load (building first if needed) the oracle library."""
    with _lock:
        if path is None:
            if _stale(_LIB_PATH, _SRC):
                build()
            path = _LIB_PATH
        if path not in _cache:
            _cache[path] = Oracle(path)
        return _cache[path]
