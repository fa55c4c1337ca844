"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Every ``check_*`` function takes a loaded oracle and raises AssertionError on a
mismatch.  ``test_oracle.py`` runs them against the real oracle;
``test_oracle_mutants.py`` runs them against deliberately broken copies of the
oracle source to show that each plausible mistake is caught by at least one.

Sources of truth used here (never the oracle itself):
  * scipy.linalg.hadamard (Sylvester-built) and numpy Kronecker products;
  * numpy's IEEE float16 conversion and fp32 division/rint;
  * exact rational arithmetic (fractions.Fraction);
  * hand-worked byte values in tests/golden/pack_cases.txt;
  * closed forms derived in the comments next to each check.
Page names: [mhpq] mhpq.cn/news/1159370, [dpshk] dpshk.com/news/5289456,
[xxqk] xxqk.cn/news/652513, [zwxr] zwxr.cn/news/303439.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import scipy.linalg

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
C_BITS = 0x3DB504F3  # RN_fp32(1/sqrt(128)), derived exactly in check_norm_const


def _f32(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def _block_h(K: int) -> np.ndarray:
    """blockdiag(H_128, ..., H_128) / sqrt(128) in fp64, H from scipy."""
    H = scipy.linalg.hadamard(128).astype(np.float64) / math.sqrt(128.0)
    return scipy.linalg.block_diag(*([H] * (K // 128)))


# --------------------------------------------------------------- Hadamard

def check_hadamard_definitions(orc):
    """[dpshk] sec. 2.1: the popcount entry rule equals the Sylvester recursion
    H_2n = [[H, H], [H, -H]] ([mhpq] sec. 2.2 writes it as H_n (x) H_2)."""
    h2 = np.array([[1, 1], [1, -1]], dtype=np.int64)
    kron = np.array([[1]], dtype=np.int64)
    n = 1
    while n <= 128:
        pop = orc.hadamard(n)
        assert np.array_equal(pop, kron), f"popcount H_{n} != Kronecker H_{n}"
        assert np.array_equal(orc.sylvester(n), kron), f"Sylvester H_{n} wrong"
        assert np.array_equal(pop, scipy.linalg.hadamard(n)), f"H_{n} != scipy"
        kron = np.kron(kron, h2)
        n *= 2


def check_hadamard_orthogonal(orc):
    """[mhpq] sec. 2.2 / [xxqk] sec. 2: H H^T = n I (and H = H^T, H^2 = n I)."""
    H = orc.hadamard(128)
    assert np.array_equal(H @ H.T, 128 * np.eye(128, dtype=np.int64))
    assert np.array_equal(H, H.T)


def check_norm_const(orc):
    """c = RN_fp32(1/sqrt(128)) = 0x3DB504F3, decided with exact rationals:
    among fp32 neighbours a < b around r = 2^-3.5, r is nearer to a iff
    r^2 = 1/128 < ((a + b) / 2)^2."""
    assert orc.norm_const_bits() == C_BITS, hex(orc.norm_const_bits())
    a = Fraction(float(_f32(C_BITS - 1)))
    c = Fraction(float(_f32(C_BITS)))
    b = Fraction(float(_f32(C_BITS + 1)))
    target = Fraction(1, 128)
    assert ((a + c) / 2) ** 2 < target < ((c + b) / 2) ** 2


def check_fwht_dense_f64(orc):
    """fp64 rotation = H_128 v / sqrt(128) with scipy's Sylvester H."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal((6, 256))
    ref = v @ _block_h(256).T
    out = orc.fwht128_f64(v)
    assert np.max(np.abs(out - ref)) <= 1e-13 * max(1.0, np.max(np.abs(ref)))


def check_fwht_f32_close(orc):
    """The fp32 staged transform equals the exact rotation within fp32
    rounding: 7 add stages and one multiply, |err| <= 8 u ||v||_2 per entry."""
    rng = np.random.default_rng(12)
    v = (rng.standard_normal((32, 128)) * rng.uniform(0.01, 100, size=(32, 1))).astype(np.float32)
    ref = v.astype(np.float64) @ _block_h(128).T
    out = orc.fwht128_f32(v).astype(np.float64)
    bound = 8 * 2.0 ** -24 * np.linalg.norm(v.astype(np.float64), axis=1, keepdims=True) * 2
    assert np.all(np.abs(out - ref) <= bound)


def check_fwht_delta(orc):
    """A unit input e_j is rotated to c * (column j of H) exactly: every
    butterfly of a delta is an exact +-1, and one multiply by c is exact."""
    H = scipy.linalg.hadamard(128)
    c = _f32(C_BITS)
    for j in (0, 1, 5, 64, 127):
        e = np.zeros(128, dtype=np.float32)
        e[j] = 1.0
        out = orc.fwht128_f32(e)
        assert np.array_equal(out, (H[:, j] * c).astype(np.float32)), j


def check_fwht_stage_order(orc):
    """The butterfly rounds run h = 1, 2, ..., 64 in fp32 (the fixed order that
    makes codes bit-reproducible).  Written here in tensor form: view the 128
    entries as a 2x2x...x2 array whose axis s is index bit s; round s
    combines the two slices along bit s."""
    rng = np.random.default_rng(13)
    v = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    w = v.copy()
    for s in range(7):
        h = 1 << s
        t = w.reshape(64, 128 // (2 * h), 2, h)
        a, b = t[:, :, 0, :].copy(), t[:, :, 1, :].copy()
        t[:, :, 0, :] = a + b
        t[:, :, 1, :] = a - b
        w = t.reshape(64, 128)
    w = (w * _f32(C_BITS)).astype(np.float32)
    assert np.array_equal(orc.fwht128_f32(v), w)


def check_fwht_involution_energy(orc):
    """The normalised rotation is its own inverse ([zwxr] sec. 2.1: the inverse
    is the same transform up to 1/n) and keeps the 2-norm ([mhpq] sec. 2.2)."""
    rng = np.random.default_rng(14)
    v = rng.standard_normal((8, 128))
    r = orc.fwht128_f64(v)
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(v, axis=1), rtol=1e-13, atol=0)
    assert np.max(np.abs(orc.fwht128_f64(r) - v)) <= 1e-13
    v32 = v.astype(np.float32)
    rr = orc.fwht128_f32(orc.fwht128_f32(v32)).astype(np.float64)
    assert np.all(np.abs(rr - v32) <= 1e-6 * np.linalg.norm(v32, axis=1, keepdims=True))


# ------------------------------------------------------------------ fp16

def _f16_cases() -> np.ndarray:
    """Every finite fp16 value, its fp32 neighbours, every midpoint between
    adjacent fp16 values and the midpoints' neighbours, plus edge values."""
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    f = h.view(np.float16).astype(np.float32)
    nxt = np.append(f[1:], np.float32(65520.0))
    mid = ((f.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)  # exact in fp32
    up = np.nextafter(f, np.float32(np.inf))
    dn = np.nextafter(f, np.float32(0))
    mu = np.nextafter(mid, np.float32(np.inf))
    md = np.nextafter(mid, np.float32(0))
    extra = np.array([2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 1e-30, 65504.0, 65519.996, 65520.0,
                      1e5, 3.4e38, np.inf], dtype=np.float32)
    allv = np.concatenate([f, up, dn, mid, mu, md, extra])
    return np.concatenate([allv, -allv])


def check_f16_conversion(orc):
    """fp32 -> binary16 round-to-nearest-even equals numpy's IEEE conversion
    on every rounding boundary; binary16 -> fp32 is exact for all patterns."""
    vals = _f16_cases()
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {vals[bad[0]]!r}: {got[bad[0]]:#x} vs {ref[bad[0]]:#x}"
    pats = np.arange(0, 0x10000, 7, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7C00) != 0x7C00]
    back = np.array([orc.f16_to_f32(int(p)) for p in pats], dtype=np.float32)
    assert np.array_equal(back.view(np.uint32), pats.view(np.float16).astype(np.float32).view(np.uint32))


# ------------------------------------------------------------- quantiser

def _fp16(x: float) -> int:
    return int(np.array([x], dtype=np.float32).astype(np.float16).view(np.uint16)[0])


def _fp16_val(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint16).view(np.float16).astype(np.float32)[0]


def check_quantize_constant_magnitude(orc):
    """[mhpq] sec. 1.1: a group whose |w'| all equal a has mean a, so the
    scale is fp16(a) and every weight maps to its sign (a / fp16(a) is within
    2^-11 of 1)."""
    rng = np.random.default_rng(21)
    for a in (0.02, 1.0, 0.0883883476, 3.7e-3, 1234.5):
        sign = np.where(rng.random(128) < 0.5, -1.0, 1.0).astype(np.float32)
        w = (sign * np.float32(a)).astype(np.float32)
        s, t = orc.quantize_group(w)
        assert s == _fp16(np.float32(a)), (a, hex(s))
        assert np.array_equal(t, sign.astype(np.int8))


def check_quantize_zero_and_extremes(orc):
    """All-zero group: scale 0, trits 0.  A group whose mean underflows fp16
    (< 2^-25) also gets scale 0 and trits 0.  A group whose mean reaches
    65520 rounds to an infinite scale and w'/inf = 0 gives trits 0."""
    s, t = orc.quantize_group(np.zeros(128, dtype=np.float32))
    assert s == 0 and not t.any()
    w = np.full(128, 2.0 ** -27, dtype=np.float32)
    w[::3] *= -1
    s, t = orc.quantize_group(w)
    assert s == 0 and not t.any()
    w = np.full(128, 70000.0, dtype=np.float32)
    s, t = orc.quantize_group(w)
    assert s == 0x7C00 and not t.any()


def _tie_group(s0: float):
    """A group whose mean rounds to the fp16 value s0, holding probe values at
    chosen multiples of s0.  The mean is about s0 * 1.0003, which still rounds
    to s0 in fp16 but differs from it in fp32."""
    s0 = np.float32(s0)
    probes = np.array([0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.0, 1.0, -1.0, 0.25], dtype=np.float32) * s0
    up = np.nextafter(np.float32(0.5) * s0, np.float32(np.inf))
    dn = np.nextafter(np.float32(0.5) * s0, np.float32(0))
    probes = np.concatenate([probes, [up, dn, -up, -dn]]).astype(np.float32)
    expect = np.array([0, 0, 1, -1, 1, -1, 0, 1, -1, 0, 1, 0, -1, 0], dtype=np.int8)
    nfill = 128 - probes.size
    fill_total = 128 * float(s0) * 1.0003 - float(np.sum(np.abs(probes.astype(np.float64))))
    fill = np.full(nfill, fill_total / nfill, dtype=np.float32)
    fill[1::2] *= -1
    return np.concatenate([probes, fill]).astype(np.float32), expect, probes.size


def check_quantize_ties(orc):
    """[mhpq] sec. 1.1 with round-half-even: w'/s = +-0.5 -> 0, +-1.5 -> +-2
    clipped to +-1, +-2.5 -> +-1; the fp32 neighbours of s/2 fall on either
    side.  The divisor is the stored fp16 scale, not the fp32 mean."""
    for s0 in (1.0, 0.01171875, 0.0234375, 6.103515625e-05):
        w, expect, n = _tie_group(s0)
        s, t = orc.quantize_group(w)
        assert s == _fp16(np.float32(s0)), (s0, hex(s))
        assert np.array_equal(t[:n], expect), (s0, t[:n], expect)


def check_quantize_rule_identity(orc):
    """For a finite scale s > 0, clamp(rint(fl(w/s)), -1, 1) equals
    sign(w) * [|w| > s/2] (exact fp32 reasoning: the quotient rounds above
    0.5 iff |w| exceeds s/2).  Checked on random groups with numpy's IEEE
    fp32 division and rint as the independent side."""
    rng = np.random.default_rng(23)
    for _ in range(200):
        w = (rng.standard_normal(128) * rng.uniform(1e-4, 10)).astype(np.float32)
        s, t = orc.quantize_group(w)
        sv = _fp16_val(s)
        q = np.rint(w / sv)
        ref = np.clip(q, -1, 1).astype(np.int8)
        assert np.array_equal(t, ref)
        rule = (np.sign(w) * (np.abs(w) > sv / np.float32(2))).astype(np.int8)
        assert np.array_equal(t, rule)


def check_quantize_mean_exact(orc):
    """When every partial sum is exact (small integers / 2^k), the scale is
    fp16 of the exact mean of |w'|."""
    rng = np.random.default_rng(24)
    for _ in range(20):
        ints = rng.integers(-64, 65, size=128)
        w = (ints / 16.0).astype(np.float32)
        s, _ = orc.quantize_group(w)
        mean = Fraction(int(np.sum(np.abs(ints))), 16 * 128)
        assert s == _fp16(np.float32(float(mean)))


def _sum_halving_tree_f32(a: np.ndarray) -> np.float32:
    """fp32 sum of 128 values in the order the scale's reduction fixes:
    for h = 64, 32, ..., 1 the first h partial sums take in the next h
    (element-wise, each addition rounded to fp32)."""
    s = a.astype(np.float32).copy()
    h = 64
    while h >= 1:
        s[:h] = s[:h] + s[h:2 * h]
        h //= 2
    return s[0]


def _sum_sequential_f32(a: np.ndarray) -> np.float32:
    acc = np.float32(0.0)
    for v in a.astype(np.float32):
        acc = np.float32(acc + v)
    return acc


def _sum_adjacent_tree_f32(a: np.ndarray) -> np.float32:
    s = a.astype(np.float32).copy()
    h = 1
    while h < 128:
        for i in range(0, 128, 2 * h):
            s[i] = np.float32(s[i] + s[i + h])
        h *= 2
    return s[0]


def _order_sensitive_groups(count: int = 4):
    """Groups whose exact sum of |w'| sits on an fp16 rounding midpoint of
    128 * scale, so that the fp32 rounding of the partial sums decides the
    scale; kept only where the halving tree lands on the other side from
    both a left-to-right sum and an adjacent-pair tree.  Magnitudes span
    e^-6 .. e^3 (a wide dynamic range makes the orders round differently)."""
    found = []
    for seed in range(4000):
        rng = np.random.default_rng(5000 + seed)
        mag = np.exp(rng.uniform(-6.0, 3.0, size=128)).astype(np.float32)
        sign = np.where(rng.random(128) < 0.5, -1.0, 1.0).astype(np.float32)
        others = sum(Fraction(float(v)) for v in mag[:-1])
        guess = np.float16(float(others + Fraction(float(mag[-1]))) / 128)
        lo = Fraction(float(guess))
        hi = Fraction(float(np.nextafter(guess, np.float16(np.inf))))
        need = 128 * (lo + hi) / 2 - others
        if need <= 0:
            continue
        mag[-1] = np.float32(float(need))
        f16 = [_fp16(np.float32(fn(mag) * np.float32(0.0078125)))
               for fn in (_sum_halving_tree_f32, _sum_sequential_f32, _sum_adjacent_tree_f32)]
        if f16[0] != f16[1] and f16[0] != f16[2]:
            found.append(((sign * mag).astype(np.float32), f16[0]))
            if len(found) == count:
                break
    assert len(found) == count, "too few order-sensitive groups"
    return found


def check_quantize_sum_order(orc):
    """The reduction order of mean |w'| (the pages are silent; the reading is
    the fixed halving tree, s[i] += s[i + h] for h = 64 .. 1, in fp32).  On
    groups whose exact sum lies on an fp16 rounding midpoint, the scale
    depends on the order of the fp32 additions; the expected scale is
    fp16_RN(tree sum * 2^-7) with the tree written out here, and the groups
    are chosen so that a left-to-right sum or an adjacent-pair tree gives a
    different scale.  The tree sum is also checked against the exact sum
    (fractions) within the error bound of 7 levels of fp32 additions."""
    for w, expect in _order_sensitive_groups():
        exact = sum(Fraction(abs(float(v))) for v in w)
        tree = _sum_halving_tree_f32(np.abs(w))
        assert abs(Fraction(float(tree)) - exact) <= Fraction(7, 2 ** 24) * exact
        s, _ = orc.quantize_group(w)
        assert s == expect, (hex(s), hex(expect))


def check_quantize_delta_rows(orc):
    """A weight row that is a unit vector in one group rotates to c * (column
    of H): all |w'| = c, mean = c exactly, scale = fp16(c), trits = that
    column of H; groups left at zero get scale 0."""
    H = scipy.linalg.hadamard(128)
    K = 256
    W = np.zeros((3, K), dtype=np.float32)
    W[0, 7] = 1.0
    W[1, 128 + 100] = 1.0
    W[2, 0] = 1.0
    W[2, 255] = 1.0
    T, S = orc.quantize(W)
    sc = _fp16(_f32(C_BITS))
    assert list(S[0]) == [sc, 0] and list(S[1]) == [0, sc] and list(S[2]) == [sc, sc]
    assert np.array_equal(T[0, :128], H[:, 7]) and not T[0, 128:].any()
    assert np.array_equal(T[1, 128:], H[:, 100]) and not T[1, :128].any()
    assert np.array_equal(T[2, :128], H[:, 0]) and np.array_equal(T[2, 128:], H[:, 127])


def check_quantize_bf16_input(orc):
    """bf16 weights are widened exactly: quantising bf16 bits equals
    quantising the same values given as fp32."""
    rng = np.random.default_rng(25)
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)
    wv = (bits.astype(np.uint32) << 16).view(np.float32)
    T1, S1 = orc.quantize(bits)
    T2, S2 = orc.quantize(wv)
    assert np.array_equal(T1, T2) and np.array_equal(S1, S2)


# --------------------------------------------------------------- packing

def _read_pack_cases():
    cases = []
    with open(os.path.join(GOLDEN, "pack_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, K, trits, bytes_ = line.split("|")
            cases.append((fmt.strip(), int(K), [int(v) for v in trits.split()],
                          [int(v) for v in bytes_.split()]))
    return cases


def check_pack_golden(orc):
    """Hand-worked bytes (tests/golden/pack_cases.txt) for both layouts."""
    for fmt, K, trits, expect in _read_pack_cases():
        T = np.array([trits], dtype=np.int8)
        assert T.shape[1] == K
        if fmt == "2bit":
            got = orc.pack2(T)[0]
            back = orc.unpack2(got[None, :], K)
        else:
            got = orc.pack3(T)[0]
            back = orc.unpack3(got[None, :], K)
        assert list(got) == expect, (fmt, trits, list(got), expect)
        assert np.array_equal(back, T)


def check_pack_roundtrip(orc):
    """unpack(pack(t)) = t for both layouts; base-3 bytes never exceed
    3^5 - 1 = 242; padding bytes are zero; the 2-bit layout never emits
    code 3."""
    rng = np.random.default_rng(31)
    for K in (128, 256, 640, 27648 // 8):
        T = rng.integers(-1, 2, size=(5, K)).astype(np.int8)
        c2 = orc.pack2(T)
        assert c2.shape == (5, K // 4)
        assert np.array_equal(orc.unpack2(c2, K), T)
        codes = np.stack([(c2 >> (2 * i)) & 3 for i in range(4)])
        assert codes.max() <= 2
        c3 = orc.pack3(T)
        ld = orc.ld3(K)
        assert c3.shape == (5, ld) and ld % 16 == 0 and ld >= -(-K // 5)
        assert c3.max() <= 242
        assert not c3[:, -(-K // 5):].any()
        assert np.array_equal(orc.unpack3(c3, K), T)


def check_bit_accounting(orc):
    """[mhpq] sec. 1.1: log2(3) = 1.585 bit per ternary weight; sec. 1.3: one
    fp16 scale per 128 weights adds 16/128 = 0.125 bit, 1.585 + 0.125 = 1.71.
    The layouts built here store 8/5 + 0.125 = 1.725 (base-3) and
    2 + 0.125 = 2.125 (2-bit) bits per weight at K = 5120."""
    assert round(math.log2(3), 3) == 1.585
    assert 16 / 128 == 0.125
    assert round(math.log2(3) + 0.125, 2) == 1.71
    K = 5120
    T = np.zeros((1, K), dtype=np.int8)
    assert orc.pack3(T).shape[1] * 8 / K + 16 / 128 == 1.725
    assert orc.pack2(T).shape[1] * 8 / K + 16 / 128 == 2.125


# ------------------------------------------------------------------ GEMV

def _dequant(T: np.ndarray, S: np.ndarray) -> np.ndarray:
    s = S.view(np.float16).astype(np.float64)
    return T.astype(np.float64) * np.repeat(s, 128, axis=1)


def check_gemv_dense(orc):
    """y equals the dense fp64 product of the dequantised weights
    (t * s per group) with the block-rotated activations (scipy H)."""
    rng = np.random.default_rng(41)
    for (N, K, M) in ((7, 128, 1), (33, 384, 3), (64, 512, 2)):
        T = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
        S = (rng.uniform(0.001, 0.1, size=(N, K // 128))).astype(np.float16).view(np.uint16)
        x = rng.standard_normal((M, K)).astype(np.float32)
        ref = (x.astype(np.float64) @ _block_h(K).T) @ _dequant(T, S).T
        got = orc.gemv(T, S, x)
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def check_gemv_delta_activation(orc):
    """x = e_k gives y[n] = (W_deq . blockdiag(H)/sqrt(128))[n, k]: the
    weight column k mapped back to the unrotated basis."""
    rng = np.random.default_rng(42)
    N, K = 9, 256
    T = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    S = rng.uniform(0.01, 0.05, size=(N, 2)).astype(np.float16).view(np.uint16)
    back = _dequant(T, S) @ _block_h(K)
    for k in (0, 77, 128, 255):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        assert np.max(np.abs(orc.gemv(T, S, x)[0] - back[:, k])) <= 1e-14


def check_rotation_invariance(orc):
    """[mhpq] sec. 2.3 (rotation absorbed): rotating the weight rows and the
    activations by the same normalised block transform leaves W x unchanged
    (fp64, before quantisation)."""
    rng = np.random.default_rng(43)
    W = rng.standard_normal((16, 384))
    x = rng.standard_normal(384)
    Wr = orc.fwht128_f64(W)
    xr = orc.fwht128_f64(x)
    assert np.max(np.abs(Wr @ xr - W @ x)) <= 1e-12 * np.max(np.abs(W @ x))


# --------------------------------------------- transform / group / residual

def _lay(orc):
    import oracle
    return oracle.LayoutOracle(orc)


def _block_h_n(K: int, n: int) -> np.ndarray:
    H = scipy.linalg.hadamard(n).astype(np.float64) / math.sqrt(float(n))
    return scipy.linalg.block_diag(*([H] * (K // n)))


def check_fwht_n_definitions(orc):
    """[dpshk] sec. 2.1 (H for any power of two) / [xxqk] sec. 2.2 (block size
    choices): the n-point transform for n = 64, 256 equals scipy's H_n / sqrt(n)
    (fp64 dense form to 1e-13, fp32 staged form within fp32 rounding), its
    normalisation constant is RN_fp32(1/sqrt(n)) -- exactly 1/8 and 1/16 --
    and at n = 128 both forms equal the pinned 128-point functions bit for
    bit."""
    L = _lay(orc)
    assert L.norm_const_bits(64) == 0x3E000000 and L.norm_const_bits(256) == 0x3D800000
    assert L.norm_const_bits(128) == C_BITS
    rng = np.random.default_rng(81)
    for n in (64, 256):
        v = rng.standard_normal((4, 2 * n))
        ref = v @ _block_h_n(2 * n, n).T
        assert np.max(np.abs(L.fwht_f64(n, v) - ref)) <= 1e-13 * max(1.0, np.max(np.abs(ref)))
        v32 = v.astype(np.float32)
        out = L.fwht_f32(n, v32).astype(np.float64)
        bound = 10 * 2.0 ** -24 * np.linalg.norm(v32.astype(np.float64), axis=1, keepdims=True) * 2
        assert np.all(np.abs(out - ref) <= bound)
    v = (rng.standard_normal((5, 256)) * 3).astype(np.float32)
    assert np.array_equal(L.fwht_f32(128, v), orc.fwht128_f32(v))
    assert np.array_equal(L.fwht_f64(128, v.astype(np.float64)), orc.fwht128_f64(v.astype(np.float64)))


def check_fwht_n_stage_order(orc):
    """The n-point fp32 transform runs its butterfly rounds h = 1, ..., n/2 in
    that order, then multiplies by the constant (tensor-form restatement, as
    for n = 128)."""
    L = _lay(orc)
    rng = np.random.default_rng(82)
    for n, cbits in ((64, 0x3E000000), (256, 0x3D800000)):
        v = (rng.standard_normal((16, n)) * 3).astype(np.float32)
        w = v.copy()
        h = 1
        while h < n:
            t = w.reshape(16, n // (2 * h), 2, h)
            a, b = t[:, :, 0, :].copy(), t[:, :, 1, :].copy()
            t[:, :, 0, :] = a + b
            t[:, :, 1, :] = a - b
            w = t.reshape(16, n)
            h *= 2
        w = (w * _f32(cbits)).astype(np.float32)
        assert np.array_equal(L.fwht_f32(n, v), w)


def check_group256_quantiser(orc):
    """[mhpq] sec. 1.4, a scale per 256 weights: constant-magnitude groups give
    s = fp16(a), t = sign; exact integer sums give fp16 of the exact mean
    (factor 2^-8); on groups whose exact sum of |w'| sits on an fp16 rounding
    midpoint the scale follows the halving tree over 256 (h = 128 .. 1) and
    not a left-to-right sum; at g = 128 the function equals the pinned
    128-group quantiser bit for bit."""
    L = _lay(orc)
    rng = np.random.default_rng(83)
    for a in (0.02, 1.0, 3.7e-3):
        sign = np.where(rng.random(256) < 0.5, -1.0, 1.0).astype(np.float32)
        s, t = L.quantize_group(256, (sign * np.float32(a)).astype(np.float32))
        assert s == _fp16(np.float32(a)) and np.array_equal(t, sign.astype(np.int8))
    for _ in range(10):
        ints = rng.integers(-64, 65, size=256)
        s, _ = L.quantize_group(256, (ints / 16.0).astype(np.float32))
        assert s == _fp16(np.float32(float(Fraction(int(np.sum(np.abs(ints))), 16 * 256))))
    # ties: probes at +-0.5 s, +-1.5 s, ... of the stored scale (round half to
    # even, clamp), the mean filled up to about s * 1.0003 over 256 weights
    for s0 in (1.0, 0.0234375):
        g128, expect, n = _tie_group(s0)
        probes = g128[:n]
        fill_total = 256 * s0 * 1.0003 - float(np.sum(np.abs(probes.astype(np.float64))))
        fill = np.full(256 - n, fill_total / (256 - n), dtype=np.float32)
        fill[1::2] *= -1
        s, t = L.quantize_group(256, np.concatenate([probes, fill]).astype(np.float32))
        assert s == _fp16(np.float32(s0)) and np.array_equal(t[:n], expect)
    for _ in range(20):
        w = (rng.standard_normal(128) * rng.uniform(1e-3, 10)).astype(np.float32)
        (sa, ta), (sb, tb) = L.quantize_group(128, w), orc.quantize_group(w)
        assert sa == sb and np.array_equal(ta, tb)
    found = 0
    for seed in range(4000):
        r = np.random.default_rng(9000 + seed)
        mag = np.exp(r.uniform(-6.0, 3.0, size=256)).astype(np.float32)
        others = sum(Fraction(float(v)) for v in mag[:-1])
        guess = np.float16(float(others + Fraction(float(mag[-1]))) / 256)
        lo = Fraction(float(guess))
        hi = Fraction(float(np.nextafter(guess, np.float16(np.inf))))
        need = 256 * (lo + hi) / 2 - others
        if need <= 0:
            continue
        mag[-1] = np.float32(float(need))
        sv = mag.astype(np.float32).copy()
        h = 128
        while h >= 1:
            sv[:h] = sv[:h] + sv[h:2 * h]
            h //= 2
        tree = _fp16(np.float32(sv[0] * np.float32(0.00390625)))
        acc = np.float32(0.0)
        for v in mag:
            acc = np.float32(acc + v)
        if tree == _fp16(np.float32(acc * np.float32(0.00390625))):
            continue
        s, _ = L.quantize_group(256, mag)
        assert s == tree, (hex(s), hex(tree))
        found += 1
        if found == 3:
            break
    assert found == 3


def check_layout_default_is_the_method(orc):
    """Block 128, group 128, no residual pass is the method itself: the layout
    quantiser equals the pinned one bit for bit, and so does its GEMV."""
    L = _lay(orc)
    rng = np.random.default_rng(84)
    W = (rng.standard_normal((9, 768)) * 0.02).astype(np.float32)
    T, S = L.quantize(W)
    T0, S0 = orc.quantize(W)
    assert np.array_equal(T, T0) and np.array_equal(S, S0)
    x = rng.standard_normal((2, 768)).astype(np.float32)
    assert np.max(np.abs(L.gemv(T, S, x) - orc.gemv(T0, S0, x))) <= 1e-12 * np.max(np.abs(orc.gemv(T0, S0, x)))


def check_residual_delta_row(orc):
    """[xxqk] sec. 3 (residual calibrator), a closed form.  A unit row e_j of W
    rotates to c * H[:, j] (all +-c), so pass 1 gives s1 = fp16(c) and
    t1 = H[:, j]; the residual is r = H[:, j] * d with d = c - fp32(s1)
    exactly; its rotation is 128 d c at position j (the sums of +-d are exact,
    one rounding in the multiply by c) and 0 elsewhere, so s2 =
    fp16(fp32(128 d c) / 128) and t2 = sign(d) at j, 0 elsewhere."""
    L = _lay(orc)
    H = scipy.linalg.hadamard(128)
    c = _f32(C_BITS)
    s1 = _fp16(c)
    d = np.float32(c - _fp16_val(s1))
    assert d != 0
    rj = np.float32(np.float32(np.float32(128.0) * d) * c)
    s2 = _fp16(np.float32(rj * np.float32(0.0078125)))
    for j in (0, 5, 127):
        W = np.zeros((1, 128), dtype=np.float32)
        W[0, j] = 1.0
        T, S = L.quantize(W, 128, 128, residual=True)
        assert list(S[0]) == [s1, s2]
        assert np.array_equal(T[0, :128], H[:, j])
        t2 = np.zeros(128, dtype=np.int8)
        t2[j] = 1 if d > 0 else -1
        assert np.array_equal(T[0, 128:], t2)


def check_residual_overflow_group(orc):
    """A group whose mean |w'| rounds to an infinite fp16 scale gets t1 = 0
    (w'/inf = 0); a zero trit dequantises to 0, so the residual is w' itself,
    whose rotation (W again) also overflows: s2 = inf, t2 = 0 -- and nothing
    becomes NaN."""
    L = _lay(orc)
    W = np.full((1, 128), 1.0e6, dtype=np.float32)
    T, S = L.quantize(W, 128, 128, residual=True)
    assert list(S[0]) == [0x7C00, 0x7C00]
    assert not T.any()


def check_residual_reduces_error(orc):
    """The residual pass brings the dequantised rotated weights closer to w'
    (what it is for): over random rows, ||w' - (s1 t1 + H_b s2 t2)|| is well
    below ||w' - s1 t1|| for every block and group size."""
    L = _lay(orc)
    rng = np.random.default_rng(85)
    W = (rng.standard_normal((6, 512)) * 0.02).astype(np.float32)
    for b in (64, 128, 256):
        for g in (128, 256):
            T, S = L.quantize(W, b, g, residual=True)
            K = 512
            wr = W.astype(np.float64) @ _block_h_n(K, b).T
            s = S.view(np.float16).astype(np.float64)
            d1 = T[:, :K] * np.repeat(s[:, :K // g], g, axis=1)
            d2 = T[:, K:] * np.repeat(s[:, K // g:], g, axis=1)
            approx = d1 + d2 @ _block_h_n(K, b).T
            e1 = np.linalg.norm(wr - d1)
            e2 = np.linalg.norm(wr - approx)
            assert e2 < 0.75 * e1, (b, g, e1, e2)


def check_layout_gemv_dense(orc):
    """The layout GEMV equals the dense fp64 product with scipy-built blocks:
    y = (t1 s1) . (H_b x) + (t2 s2) . (H_b H_b x); the second term is the
    residual against the unrotated x (H_b H_b = I)."""
    L = _lay(orc)
    rng = np.random.default_rng(86)
    K, N, M = 512, 7, 2
    x = rng.standard_normal((M, K)).astype(np.float32)
    for b in (64, 128, 256):
        for g in (128, 256):
            for res in (False, True):
                f = 2 if res else 1
                T = rng.integers(-1, 2, size=(N, f * K)).astype(np.int8)
                S = rng.uniform(0.001, 0.1, size=(N, f * (K // g))).astype(np.float16).view(np.uint16)
                s = S.view(np.float16).astype(np.float64)
                Bh = _block_h_n(K, b)
                xr = x.astype(np.float64) @ Bh.T
                ref = xr @ (T[:, :K] * np.repeat(s[:, :K // g], g, axis=1)).T
                if res:
                    ref = ref + x.astype(np.float64) @ (T[:, K:] * np.repeat(s[:, K // g:], g, axis=1)).T
                got = L.gemv(T, S, x, b, g, res)
                assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref))), (b, g, res)


def check_group256_bit_accounting(orc):
    """[mhpq] sec. 1.4: one fp16 scale per 256 weights costs 16/256 = 0.0625
    bit per weight; with the residual pass the layouts store twice the codes
    and scales (2 x 2.125 = 4.25 bit per weight in 2-bit codes at group 128)."""
    assert 16 / 256 == 0.0625
    L = _lay(orc)
    W = np.zeros((1, 512), dtype=np.float32)
    T, S = L.quantize(W, 128, 256, residual=False)
    assert S.shape[1] * 16 / 512 == 0.0625
    T, S = L.quantize(W, 128, 128, residual=True)
    assert (T.shape[1] * 2 + S.shape[1] * 16) / 512 == 4.25


# ------------------------------------------------------- 2:4 sparse format
# [mhpq] sec. 1.2: two of every four weights kept at regular positions, the
# kept ones ternarised.  Readings (documented in tq_oracle.h): the pattern is
# chosen on the rotated weights, per quad of consecutive k; the kept pair is
# the two largest |w'| (ties to the lower index); the absmean scale is taken
# over the 64 kept weights (halving tree over them in k order, times 2^-6).

_PAT24 = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


def _sp(orc):
    import oracle
    return oracle.Sparse24Oracle(orc)


def _keep_bruteforce(w: np.ndarray) -> np.ndarray:
    """Per quad: order the four positions by (-|w|, index) and keep the first two."""
    keep = np.zeros(w.size, dtype=np.uint8)
    for j in range(w.size // 4):
        q = np.abs(w[4 * j:4 * j + 4].astype(np.float64))
        order = sorted(range(4), key=lambda i: (-q[i], i))
        keep[4 * j + order[0]] = keep[4 * j + order[1]] = 1
    return keep


def check_sparse24_pattern_bruteforce(orc):
    """Exactly two kept per quad, and they are the two largest magnitudes
    (ties to the lower index), on random groups and on integer-valued groups
    with many ties (including all-equal quads and signed ties)."""
    sp = _sp(orc)
    rng = np.random.default_rng(61)
    for it in range(120):
        if it % 3 == 0:
            w = rng.integers(-2, 3, size=128).astype(np.float32)
        elif it % 3 == 1:
            w = (rng.standard_normal(128) * 0.02).astype(np.float32)
        else:
            w = rng.choice(np.array([-1.5, -0.5, 0.5, 1.5], dtype=np.float32), size=128)
        _, t, keep = sp.quantize_group(w)
        assert np.array_equal(keep, _keep_bruteforce(w)), it
        assert np.all(keep.reshape(32, 4).sum(1) == 2)
        assert not np.any(t[keep == 0]), "a pruned weight kept a trit"


def _code24(p: int, a: int, b: int) -> int:
    return 9 * p + 3 * (a + 1) + (b + 1)


def check_sparse24_codes_by_hand(orc):
    """Every one of the 54 (pattern, trit, trit) combinations, stored in quad
    j of a group, packs to code 9 p + 3 (t0 + 1) + (t1 + 1) with its low
    nibble in byte j // 2 (nibble j % 2) and its two high bits at bits
    2 (j % 4) of byte 16 + j // 4; unpacking gives the quad back.  Two
    whole-group byte images worked by hand: pattern (0,1) with trits (1, -1)
    everywhere is code 6 (bytes 0x66 x 16, then 0x00 x 8); pattern (2,3) with
    trits (1, 1) is code 53 = 0b110101 (bytes 0x55 x 16, then 0xFF x 8)."""
    sp = _sp(orc)
    combos = [(p, a, b) for p in range(6) for a in (-1, 0, 1) for b in (-1, 0, 1)]
    assert len(combos) == 54
    for start in range(0, 54, 32):
        T = np.zeros((1, 128), dtype=np.int8)
        KEEP = np.zeros((1, 128), dtype=np.uint8)
        expect = np.zeros(24, dtype=np.uint8)
        for j in range(32):
            p, a, b = combos[(start + j) % 54]
            i0, i1 = _PAT24[p]
            KEEP[0, 4 * j + i0] = KEEP[0, 4 * j + i1] = 1
            T[0, 4 * j + i0], T[0, 4 * j + i1] = a, b
            c = _code24(p, a, b)
            expect[j // 2] |= (c & 15) << (4 * (j % 2))
            expect[16 + j // 4] |= (c >> 4) << (2 * (j % 4))
        codes = sp.pack(T, KEEP)
        assert np.array_equal(codes[0], expect), (start, codes[0], expect)
        T2, K2, bad = sp.unpack(codes, 128)
        assert bad == 0 and np.array_equal(T2, T) and np.array_equal(K2, KEEP)
    for (p, a, b, img) in ((0, 1, -1, [0x66] * 16 + [0x00] * 8), (5, 1, 1, [0x55] * 16 + [0xFF] * 8)):
        i0, i1 = _PAT24[p]
        T = np.zeros((1, 128), dtype=np.int8)
        KEEP = np.zeros((1, 128), dtype=np.uint8)
        T[0, i0::4], T[0, i1::4] = a, b
        KEEP[0, i0::4] = KEEP[0, i1::4] = 1
        assert list(sp.pack(T, KEEP)[0]) == img
    # codes 54..63 are not valid: they unpack to zeros and are counted
    bad_codes = np.zeros((1, 24), dtype=np.uint8)
    bad_codes[0, 0] = 0x0F  # quad 0: low nibble 15 ...
    bad_codes[0, 16] = 0x03  # ... high bits 3: code 63
    T, KEEP, bad = sp.unpack(bad_codes, 128)
    assert bad == 1 and not T[0, :4].any() and not KEEP[0, :4].any()


def check_sparse24_scale_closed_forms(orc):
    """Kept magnitudes all equal to a (the pruned two of each quad smaller):
    the mean over the kept is a, the scale fp16(a), each kept weight maps to
    its sign.  An all-zero group keeps positions 0 and 1 of every quad (ties
    to the lower index), with scale 0 and all trits 0.  A group whose pruned
    weights are large would change a mean over all 128 but not this one."""
    sp = _sp(orc)
    rng = np.random.default_rng(62)
    for a in (0.02, 1.0, 3.7e-3, 1234.5):
        w = np.zeros(128, dtype=np.float32)
        keep = np.zeros(128, dtype=np.uint8)
        sign = np.where(rng.random(128) < 0.5, -1.0, 1.0).astype(np.float32)
        for j in range(32):
            i0, i1 = _PAT24[rng.integers(6)]
            small = np.float32(a) * np.float32(rng.uniform(0.0, 0.9, size=4))
            w[4 * j:4 * j + 4] = small * sign[4 * j:4 * j + 4]
            for i in (i0, i1):
                w[4 * j + i] = sign[4 * j + i] * np.float32(a)
                keep[4 * j + i] = 1
        s, t, kp = sp.quantize_group(w)
        assert s == _fp16(np.float32(a)), (a, hex(s))
        assert np.array_equal(kp, keep)
        assert np.array_equal(t[keep == 1], sign[keep == 1].astype(np.int8))
        assert not t[keep == 0].any()
    s, t, kp = sp.quantize_group(np.zeros(128, dtype=np.float32))
    assert s == 0 and not t.any()
    assert np.array_equal(kp, np.tile(np.array([1, 1, 0, 0], dtype=np.uint8), 32))


def _sum_halving_tree64_f32(a: np.ndarray) -> np.float32:
    s = a.astype(np.float32).copy()
    h = 32
    while h >= 1:
        s[:h] = s[:h] + s[h:2 * h]
        h //= 2
    return s[0]


def check_sparse24_sum_order(orc):
    """The kept weights' sum is the halving tree over the 64 kept values in
    k order.  Groups are built with two large kept values and two tiny pruned
    ones per quad, the kept magnitudes chosen so that their exact sum sits on
    an fp16 rounding midpoint of 64 * scale; kept only where the halving tree
    gives a different scale from a left-to-right sum and from a mean over all
    128 weights."""
    sp = _sp(orc)
    found = 0
    for seed in range(4000):
        rng = np.random.default_rng(7000 + seed)
        mag = np.exp(rng.uniform(-5.0, 3.0, size=64)).astype(np.float32)
        others = sum(Fraction(float(v)) for v in mag[:-1])
        guess = np.float16(float(others + Fraction(float(mag[-1]))) / 64)
        lo = Fraction(float(guess))
        hi = Fraction(float(np.nextafter(guess, np.float16(np.inf))))
        need = 64 * (lo + hi) / 2 - others
        if need <= 0:
            continue
        mag[-1] = np.float32(float(need))
        if float(mag.min()) < 1e-3:
            continue
        w = np.zeros(128, dtype=np.float32)
        pats = rng.integers(6, size=32)
        tiny = np.float32(1e-6)
        kept_pos = []
        for j in range(32):
            i0, i1 = _PAT24[pats[j]]
            w[4 * j:4 * j + 4] = tiny
            w[4 * j + i0] = mag[2 * j]
            w[4 * j + i1] = -mag[2 * j + 1]
            kept_pos += [4 * j + i0, 4 * j + i1]
        kept = np.abs(w[kept_pos])  # k order
        tree = _fp16(np.float32(_sum_halving_tree64_f32(kept) * np.float32(0.015625)))
        seq = _fp16(np.float32(_sum_sequential_f32(kept) * np.float32(0.015625)))
        all128 = _fp16(np.float32(_sum_halving_tree_f32(np.abs(w)) * np.float32(0.0078125)))
        if tree == seq or tree == all128:
            continue
        s, _, kp = sp.quantize_group(w)
        assert np.array_equal(np.nonzero(kp)[0], np.array(sorted(kept_pos)))
        assert s == tree, (hex(s), hex(tree))
        found += 1
        if found == 4:
            break
    assert found == 4, "too few order-sensitive sparse groups"


def check_sparse24_ties(orc):
    """Round half to even on the kept weights, against the stored scale:
    kept values at +-0.5 s, +-1.5 s, +-2.5 s and the fp32 neighbours of s/2
    (each kept beside a filler, the other two of its quad zero), the fillers
    making the mean of the 64 kept magnitudes s * 1.0003, which rounds to s
    in fp16.  Expected trits as in check_quantize_ties."""
    sp = _sp(orc)
    for s0 in (1.0, 0.01171875, 6.103515625e-05):
        s0 = np.float32(s0)
        probes = np.array([0.5, -0.5, 1.5, -1.5, 2.5, -2.5], dtype=np.float32) * s0
        up = np.nextafter(np.float32(0.5) * s0, np.float32(np.inf))
        dn = np.nextafter(np.float32(0.5) * s0, np.float32(0))
        probes = np.concatenate([probes, [up, dn, -up, -dn]]).astype(np.float32)
        expect = np.array([0, 0, 1, -1, 1, -1, 1, 0, -1, 0], dtype=np.int8)
        nfill = 64 - probes.size
        fill_total = 64 * float(s0) * 1.0003 - float(np.sum(np.abs(probes.astype(np.float64))))
        fill = np.float32(fill_total / nfill)  # (the other two of each quad are 0: both are kept)
        w = np.zeros(128, dtype=np.float32)
        for j in range(32):
            if j < probes.size:
                w[4 * j + 1], w[4 * j + 3] = probes[j], fill
            else:
                w[4 * j], w[4 * j + 2] = fill, -fill
        s, t, keep = sp.quantize_group(w)
        assert s == _fp16(s0), (s0, hex(s))
        assert np.array_equal(t[1:4 * probes.size:4], expect), (s0, t[1:4 * probes.size:4])


def check_sparse24_rule(orc):
    """Kept weights: clamp(rint(w / s), -1, 1) with the stored fp16 scale
    (numpy IEEE fp32 division and rint as the independent side); pruned: 0."""
    sp = _sp(orc)
    rng = np.random.default_rng(63)
    for _ in range(150):
        w = (rng.standard_normal(128) * rng.uniform(1e-4, 10)).astype(np.float32)
        s, t, keep = sp.quantize_group(w)
        sv = _fp16_val(s)
        ref = np.clip(np.rint(w / sv), -1, 1).astype(np.int8)
        ref[keep == 0] = 0
        assert np.array_equal(t, ref)


def check_sparse24_rows(orc):
    """Whole rows (fp32 and bf16 input) are the FWHT-128 of each group
    followed by the group rule: the rotation is checked against scipy's H
    (fp32 rounding aside, every group's pattern and trits agree with the
    group rule applied to the oracle's pinned fp32 rotation)."""
    sp = _sp(orc)
    rng = np.random.default_rng(64)
    W = (rng.standard_normal((5, 384)) * 0.02).astype(np.float32)
    T, KEEP, S = sp.quantize(W)
    Wb = W.view(np.uint32)
    Wb16 = ((Wb + 0x7FFF + ((Wb >> 16) & 1)) >> 16).astype(np.uint16)
    Tb, KEEPb, Sb = sp.quantize(Wb16)
    Wb32 = (Wb16.astype(np.uint32) << 16).view(np.float32)
    for (Wx, Tx, Kx, Sx) in ((W, T, KEEP, S), (Wb32, Tb, KEEPb, Sb)):
        for n in range(Wx.shape[0]):
            for g in range(3):
                rot = orc.fwht128_f32(Wx[n, 128 * g:128 * g + 128])
                ref = _block_h(128) @ Wx[n, 128 * g:128 * g + 128].astype(np.float64)
                assert np.max(np.abs(rot - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
                s, t, kp = sp.quantize_group(rot)
                assert s == Sx[n, g] and np.array_equal(t, Tx[n, 128 * g:128 * g + 128])
                assert np.array_equal(kp, Kx[n, 128 * g:128 * g + 128])


def check_sparse24_gemv_dense(orc):
    """y of the packed 2:4 weights equals the dense fp64 product of the
    expanded, dequantised trits (t * s) with the block-rotated activations
    (scipy H); the pruned weights contribute nothing."""
    sp = _sp(orc)
    rng = np.random.default_rng(65)
    for (N, K, M) in ((9, 128, 1), (21, 384, 3)):
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        T, KEEP, S = sp.quantize(W)
        codes = sp.pack(T, KEEP)
        x = rng.standard_normal((M, K)).astype(np.float32)
        ref = (x.astype(np.float64) @ _block_h(K).T) @ _dequant(T, S).T
        got = sp.gemv(codes, S, x, K)
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
        assert np.count_nonzero(T) <= N * K // 2


def check_sparse24_bit_accounting(orc):
    """24 bytes of codes per 128 weights (1.5 bit) plus a 2-byte scale
    (0.125 bit): 1.625 bits per weight.  The entropy bound of the stored
    information is log2(6 * 9) / 4 + 0.125 = 1.5637 bits: [mhpq] sec. 1.2's
    "about 1.29" is below what a mask that can name all six patterns and two
    free trits can reach (its accounting is not reproducible)."""
    sp = _sp(orc)
    for K in (128, 5120, 27648):
        assert sp.ld(K) == 24 * K // 128
        bits = (sp.ld(K) + 2 * (K // 128)) * 8 / K
        assert bits == 1.625
    assert abs(math.log2(54) / 4 + 0.125 - 1.5637) < 1e-4


ALL_CHECKS = [
    check_hadamard_definitions,
    check_hadamard_orthogonal,
    check_norm_const,
    check_fwht_dense_f64,
    check_fwht_f32_close,
    check_fwht_delta,
    check_fwht_stage_order,
    check_fwht_involution_energy,
    check_f16_conversion,
    check_quantize_constant_magnitude,
    check_quantize_zero_and_extremes,
    check_quantize_ties,
    check_quantize_rule_identity,
    check_quantize_mean_exact,
    check_quantize_sum_order,
    check_quantize_delta_rows,
    check_quantize_bf16_input,
    check_pack_golden,
    check_pack_roundtrip,
    check_bit_accounting,
    check_gemv_dense,
    check_gemv_delta_activation,
    check_rotation_invariance,
    check_fwht_n_definitions,
    check_fwht_n_stage_order,
    check_group256_quantiser,
    check_layout_default_is_the_method,
    check_residual_delta_row,
    check_residual_overflow_group,
    check_residual_reduces_error,
    check_layout_gemv_dense,
    check_group256_bit_accounting,
    check_sparse24_pattern_bruteforce,
    check_sparse24_codes_by_hand,
    check_sparse24_scale_closed_forms,
    check_sparse24_sum_order,
    check_sparse24_ties,
    check_sparse24_rule,
    check_sparse24_rows,
    check_sparse24_gemv_dense,
    check_sparse24_bit_accounting,
]
