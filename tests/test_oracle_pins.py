"""Pins for the CPU oracle, each against something other than the oracle itself.

The oracle (``oracle/``) is the yardstick for the CUDA path, so before it is trusted
every function is checked here against: the storage sizes the pages print, closed
forms, exact rational arithmetic, brute force over all codes, numpy's independent
binary16 conversion, scipy/mpmath softmax routines and attention invariants.  Each
check is chosen so that a plausible slip (a dropped term, a wrong sign or index, a
swapped nibble, a transposed operand) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BYTES_PER_BLOCK = {"f16": 64, "q8_0": 34, "q4_0": 18}  # derived below from the oracle, pinned by the pages


def f32(x):
    return np.float32(x)


def f16bits(x):
    return int(np.float16(np.float32(x)).view(np.uint16))


# ---------------------------------------------------------------------------------
# storage size: the pages' printed sizes ("HAL #582" section 1, 3b, 5 P1; qwisp #168)
# ---------------------------------------------------------------------------------

def _oracle_bytes_per_row(kv_type, D):
    x = np.zeros((1, D), np.float32)
    c, s = oracle.quantize(kv_type, x)
    return c.nbytes + s.nbytes


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "size_model.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            src, L, H, D, tk, tv, ctx, val, unit = [t.strip() for t in line.split("|")]
            rows.append((src, int(L), int(H), int(D), tk, tv, int(ctx), float(val), unit))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: f"{r[0]}-{r[4]}-{r[5]}-{r[6]}")
def test_oracle_storage_matches_pages(row):
    src, L, H, D, tk, tv, ctx, val, unit = row
    per_tok = L * H * (D // 32) * (oracle.BLOCK_BYTES[tk] + oracle.BLOCK_BYTES[tv])
    if unit == "KiB_per_token":
        assert per_tok / 1024 == val
    elif unit == "MiB":
        assert per_tok * ctx / 2**20 == val
    elif unit == "B_per_token":
        assert per_tok == val
    else:  # pragma: no cover
        raise AssertionError(unit)


def test_bytes_per_block():
    for t, nb in BYTES_PER_BLOCK.items():
        assert _oracle_bytes_per_row(t, 32) == nb
        # where the natural layout is already packed, the packed-storage formula agrees with it
        assert oracle.block_storage_bytes(t) == nb


def test_packed_storage_of_five_bit_codes():
    """q5_0 blocks: 32 five-bit codes (16 bytes of nibbles + 4 bytes of fifth bits) and one
    f16 scale = 22 bytes, which the q5_0/q5_0 row of the size model table (66 KiB per
    token) confirms; q5_1 adds the f16 minimum (24 bytes, the P1 ladder's floor)."""
    assert oracle.block_storage_bytes("q5_0") == 16 + 4 + 2
    assert oracle.block_storage_bytes("q5_1") == 16 + 4 + 2 + 2
    assert oracle.block_storage_bytes("q4_1") == 16 + 2 + 2
    # the oracle's natural q5_0 layout keeps one code per byte: the packed figure is smaller
    assert _oracle_bytes_per_row("q5_0", 32) == 32 + 2


# ---------------------------------------------------------------------------------
# q8_0
# ---------------------------------------------------------------------------------

def q8(x):
    c, s = oracle.quantize("q8_0", np.asarray(x, np.float32).reshape(1, 32))
    return c[0].astype(np.int64), int(s[0, 0])


def test_q8_zero_block():
    c, s = q8(np.zeros(32))
    assert (c == 0).all() and s == 0


@pytest.mark.parametrize("k,a", [(0, 1.0), (5, -3.25), (31, 1e-3), (17, 7e4)])
def test_q8_single_value(k, a):
    x = np.zeros(32, np.float32)
    x[k] = a
    c, s = q8(x)
    expect = np.zeros(32, np.int64)
    expect[k] = 127 if a > 0 else -127
    assert (c == expect).all()
    assert s == f16bits(f32(abs(a)) / f32(127))


@pytest.mark.parametrize("e", [-6, -1, 0, 3])
def test_q8_exact_multiples(e):
    rng = np.random.default_rng(7 + e)
    k = rng.integers(-127, 128, size=32)
    k[rng.integers(0, 32)] = -127  # amax = 127 * 2^e  ->  d = 2^e exactly
    x = (k * 2.0**e).astype(np.float32)
    c, s = q8(x)
    assert (c == k).all()
    assert s == f16bits(2.0**e)


def test_q8_half_rounds_away_from_zero():
    # d = 1 exactly (amax = 127); x = k + 1/2 lies exactly on a tie
    x = np.zeros(32, np.float32)
    x[0] = 127
    x[1], x[2], x[3], x[4] = 2.5, -2.5, 0.5, -0.5
    c, _ = q8(x)
    assert list(c[1:5]) == [3, -3, 1, -1]  # half-even would give 2, -2, 0, 0


def test_q8_brute_force_codes_minimise_error():
    """Each code is the integer nearest to x/d (exact rational arithmetic on the fp32
    d); away from exact ties only the true nearest integer is accepted."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-4, 4)
        x = (rng.standard_normal(32) * scale).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, 32, 4)] *= 10  # outlier channels
        c, s = q8(x)
        amax = max(abs(float(v)) for v in x)
        d = Fraction(float(f32(amax) / f32(127)))
        for j in range(32):
            t = Fraction(float(x[j])) / d
            lo = math.floor(t)
            frac = t - lo
            if abs(frac - Fraction(1, 2)) < Fraction(1, 2**20):
                assert c[j] in (lo, lo + 1)
            else:
                assert c[j] == (lo + 1 if frac > Fraction(1, 2) else lo)
            assert -127 <= c[j] <= 127
        assert s == f16bits(f32(amax) / f32(127))


def test_q8_round_trip_bounds():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((200, 32)) * 10.0 ** rng.uniform(-3, 3, (200, 1))).astype(np.float32)
    c, s = oracle.quantize("q8_0", x)
    d32 = np.abs(x).max(axis=1).astype(np.float32) / np.float32(127)
    d16 = oracle.f16_bits_to_f64(s[:, 0])
    # codes against the fp32 scale: |x - d q| <= d/2 (up to the rounding of 1/d)
    err32 = np.abs(x.astype(np.float64) - d32[:, None].astype(np.float64) * c)
    assert (err32 <= d32[:, None] / 2 * (1 + 2.0**-20)).all()
    # stored form: |x - x_hat| <= d/2 + |q| |d - f16(d)|
    xh = oracle.dequantize("q8_0", c, s, 32)
    bound = d32[:, None] / 2 * (1 + 2.0**-20) + np.abs(c) * np.abs(d32[:, None] - d16[:, None])
    assert (np.abs(x - xh) <= bound + 1e-30).all()


# ---------------------------------------------------------------------------------
# q4_0
# ---------------------------------------------------------------------------------

def q4(x):
    p, s = oracle.quantize("q4_0", np.asarray(x, np.float32).reshape(1, 32))
    p = p[0]
    codes = np.concatenate([p & 0x0F, p >> 4]).astype(np.int64)  # element i low, i+16 high
    return codes, p, int(s[0, 0])


def test_q4_zero_block():
    c, p, s = q4(np.zeros(32))
    # m = +0, d = 0 / -8 = -0 in IEEE arithmetic, so the stored scale is f16 -0 (0x8000)
    assert (c == 8).all() and (p == 0x88).all() and s == 0x8000


@pytest.mark.parametrize("a", [1.0, -2.0, 0.375, -96.0])
def test_q4_all_equal_block_is_exact(a):
    c, _, s = q4(np.full(32, a))
    assert (c == 0).all()  # x/d = -8 -> floor(-8 + 8.5) = 0
    xh = oracle.dequantize("q4_0", *oracle.quantize("q4_0", np.full((1, 32), a, np.float32)), 32)
    assert (xh == a).all()  # a/8 is f16-exact for these a
    assert s == f16bits(f32(a) / f32(-8))


def test_q4_known_codes_and_nibble_order():
    # d = 1 exactly: x0 = -8 is the (first) largest magnitude, so c_j = x_j + 8.
    want = np.array([0, 15, 3, 12, 7, 8, 1, 14, 2, 13, 4, 11, 5, 10, 6, 9,
                     9, 6, 10, 5, 11, 4, 12, 3, 13, 2, 14, 1, 15, 0, 8, 7])
    x = (want - 8).astype(np.float32)
    c, p, s = q4(x)
    assert (c == want).all()
    assert list(p) == [int(want[i] | (want[i + 16] << 4)) for i in range(16)]
    assert s == f16bits(1.0)


def test_q4_tie_first_index_wins_and_clips():
    x = np.zeros(32, np.float32)
    x[3], x[7] = 2.0, -2.0  # |x| tie: the first (+2) sets the sign of d
    c, _, s = q4(x)
    assert s == f16bits(-0.25)
    assert c[3] == 0 and c[7] == 15  # -2/-0.25 = 8 -> 16.5 -> clipped to 15
    x[3], x[7] = -2.0, 2.0
    c, _, s = q4(x)
    assert s == f16bits(0.25) and c[3] == 0 and c[7] == 15


def test_q4_brute_force_codes():
    """c = clip(floor(x/d + 1/2) + 8, 0, 15) in exact arithmetic, near-ties excepted."""
    rng = np.random.default_rng(3)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-4, 4)
        x = (rng.standard_normal(32) * scale).astype(np.float32)
        c, _, s = q4(x)
        k = int(np.argmax(np.abs(x)))  # numpy: first index of the maximum
        d32 = f32(x[k]) / f32(-8)
        d = Fraction(float(d32))
        for j in range(32):
            t = Fraction(float(x[j])) / d + Fraction(17, 2)
            fl = math.floor(t)
            if abs(t - round(t)) < Fraction(1, 2**19) and t != round(t):
                ok = {min(15, fl), min(15, fl - 1), min(15, fl + 1)}
                assert c[j] in ok
            else:
                assert c[j] == min(15, fl)
            assert 0 <= c[j] <= 15
        assert s == f16bits(d32)


def test_q4_round_trip_bounds():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((300, 32)) * 10.0 ** rng.uniform(-3, 3, (300, 1))).astype(np.float32)
    p, s = oracle.quantize("q4_0", x)
    codes = np.concatenate([p & 0x0F, p >> 4], axis=1).astype(np.int64)
    k = np.argmax(np.abs(x), axis=1)
    d32 = x[np.arange(300), k].astype(np.float32) / np.float32(-8)
    err = np.abs(x.astype(np.float64) - d32[:, None].astype(np.float64) * (codes - 8))
    ad = np.abs(d32[:, None]).astype(np.float64)
    clipped = codes == 15
    assert (err[~clipped] <= (ad / 2 * (1 + 2.0**-19) * np.ones_like(err))[~clipped]).all()
    assert (err[clipped] <= (ad * (1 + 2.0**-19) * np.ones_like(err))[clipped]).all()
    # the clip bound is reached: a value of opposite sign near |m| has error close to |d|
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 1.0, -0.999
    p, s = oracle.quantize("q4_0", x)
    xh = oracle.dequantize("q4_0", p, s, 32)
    assert (p[0, 1] & 0x0F) == 15 and abs(xh[0, 1] - x[0, 1]) > 0.1


# ---------------------------------------------------------------------------------
# f16 arm: numpy's binary16 conversion is an independent implementation
# ---------------------------------------------------------------------------------

def test_f16_matches_numpy():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.uniform(-9, 5, 20000).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65520.0, -70000.0, 6e-8, 2.98e-8, 1e-9, 0.1, 1 / 3], np.float32),
        # exact ties between two halves (round-half-even decides)
        (np.arange(1, 2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0**-10),
    ]).astype(np.float32)
    x = x[: (len(x) // 32) * 32].reshape(-1, 32)
    c, _ = oracle.quantize("f16", x)
    assert (c == x.astype(np.float16).view(np.uint16)).all()


# ---------------------------------------------------------------------------------
# attention (fp64 over the dequantised cache)
# ---------------------------------------------------------------------------------

def _cache(kv_type, x):
    """x [Hkv, n, D] fp32 -> (codes, scales) [Hkv, n, ...]."""
    return oracle.quantize(kv_type, x)


def _exact_attention_mp(q, k, v, scale):
    """mpmath at 50 digits: an exact-arithmetic reference for tiny cases."""
    import mpmath as mp
    mp.mp.dps = 50
    n, D = k.shape
    s = [mp.mpf(float(scale)) * mp.fsum(mp.mpf(float(q[d])) * mp.mpf(float(k[t, d])) for d in range(D))
         for t in range(n)]
    M = max(s)
    w = [mp.e ** (st - M) for st in s]
    L = mp.fsum(w)
    out = [mp.fsum(w[t] * mp.mpf(float(v[t, d])) for t in range(n)) / L for d in range(D)]
    return np.array([float(o) for o in out]), float(M + mp.log(L))


@pytest.mark.parametrize("tk,tv", [("q8_0", "q8_0"), ("q8_0", "q4_0"), ("q4_0", "q4_0"), ("f16", "f16"),
                                   ("f16", "q4_0")])
@pytest.mark.parametrize("G", [1, 2, 5, 8])
def test_attention_exact_tiny(tk, tv, G):
    rng = np.random.default_rng(100 + G)
    Hkv, n, D = 2, 7, 32
    Hq = Hkv * G
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    V = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    q = rng.standard_normal((Hq, D)).astype(np.float32) * 2
    scale = float(np.float32(1 / math.sqrt(D)))
    kc, ks = _cache(tk, K)
    vc, vs = _cache(tv, V)
    out, lse = oracle.attention(tk, kc, ks, tv, vc, vs, n, q, scale)
    Kh = oracle.dequantize(tk, kc, ks, D)
    Vh = oracle.dequantize(tv, vc, vs, D)
    for hq in range(Hq):
        h = hq // G
        ref, ref_lse = _exact_attention_mp(q[hq], Kh[h], Vh[h], scale)
        assert np.abs(out[hq] - ref).max() < 1e-13
        assert abs(lse[hq] - ref_lse) < 1e-13


def test_attention_matches_scipy_softmax():
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(4)
    Hkv, G, n, D = 2, 5, 300, 128
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    K[:, :, [3, 40, 77, 120]] *= 10
    V = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    q = rng.standard_normal((Hkv * G, D)).astype(np.float32)
    scale = float(np.float32(1 / math.sqrt(D)))
    kc, ks = _cache("q8_0", K)
    vc, vs = _cache("q4_0", V)
    out, lse = oracle.attention("q8_0", kc, ks, "q4_0", vc, vs, n, q, scale)
    Kh = oracle.dequantize("q8_0", kc, ks, D)
    Vh = oracle.dequantize("q4_0", vc, vs, D)
    for hq in range(Hkv * G):
        s = scale * (Kh[hq // G] @ q[hq].astype(np.float64))
        assert np.abs(out[hq] - softmax(s) @ Vh[hq // G]).max() < 1e-12
        assert abs(lse[hq] - logsumexp(s)) < 1e-12


def test_attention_invariants():
    rng = np.random.default_rng(8)
    Hkv, G, n, D = 2, 4, 64, 64
    Hq = Hkv * G
    q = rng.standard_normal((Hq, D)).astype(np.float32)
    scale = 0.125
    # identical keys -> mean of V_hat
    K = np.broadcast_to(rng.standard_normal((Hkv, 1, D)), (Hkv, n, D)).astype(np.float32)
    V = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    kc, ks = _cache("q8_0", K)
    vc, vs = _cache("q8_0", V)
    out, lse = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, n, q, scale)
    Vh = oracle.dequantize("q8_0", vc, vs, D)
    Kh = oracle.dequantize("q8_0", kc, ks, D)
    for hq in range(Hq):
        assert np.abs(out[hq] - Vh[hq // G].mean(axis=0)).max() < 1e-13
        s0 = scale * float(Kh[hq // G, 0] @ q[hq].astype(np.float64))
        assert abs(lse[hq] - (s0 + math.log(n))) < 1e-12
    # ctx = 1 -> V_hat[0], lse = s_0
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    kc, ks = _cache("q4_0", K)
    out, lse = oracle.attention("q4_0", kc, ks, "q8_0", vc, vs, 1, q, scale)
    Kh = oracle.dequantize("q4_0", kc, ks, D)
    for hq in range(Hq):
        assert np.abs(out[hq] - Vh[hq // G, 0]).max() == 0.0
        assert abs(lse[hq] - scale * float(Kh[hq // G, 0] @ q[hq].astype(np.float64))) < 1e-12
    # one dominant key -> its V row
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32) * 0.01
    K[:, 37] = np.sign(q[::G]) * 40  # aligned with the first query of each group only
    kc, ks = _cache("q8_0", K)
    out, _ = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, n, q, scale)
    for h in range(Hkv):
        assert np.abs(out[h * G] - Vh[h, 37]).max() < 1e-12
    # permuting the keys (with their values) changes nothing
    perm = rng.permutation(n)
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    kc, ks = _cache("q8_0", K)
    o1, l1 = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, n, q, scale)
    o2, l2 = oracle.attention("q8_0", kc[:, perm], ks[:, perm], "q8_0", vc[:, perm], vs[:, perm], n, q, scale)
    assert np.abs(o1 - o2).max() < 1e-13 and np.abs(l1 - l2).max() < 1e-12
    # grouped-query mapping: query head hq reads KV head hq // G
    V = np.stack([np.full((n, D), float(h + 1), np.float32) for h in range(Hkv)])
    vc2, vs2 = _cache("f16", V)
    out, _ = oracle.attention("q8_0", kc, ks, "f16", vc2, vs2, n, q, scale)
    for hq in range(Hq):
        assert np.abs(out[hq] - (hq // G + 1)).max() < 1e-14
    # empty context
    out, lse = oracle.attention("q8_0", kc, ks, "q8_0", vc, vs, 0, q, scale)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_f16_arm_close_to_unrounded_attention():
    """The f16 arm differs from attention on the raw fp32 inputs only by the binary16
    rounding of K and V: |out - out_exact| <= max|v| u + |s| u-derived term."""
    from scipy.special import softmax
    rng = np.random.default_rng(12)
    Hkv, n, D = 1, 500, 128
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    V = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    q = rng.standard_normal((1, D)).astype(np.float32)
    scale = float(np.float32(1 / math.sqrt(D)))
    kc, ks = _cache("f16", K)
    vc, vs = _cache("f16", V)
    out, _ = oracle.attention("f16", kc, ks, "f16", vc, vs, n, q, scale)
    s = scale * (K[0].astype(np.float64) @ q[0].astype(np.float64))
    exact = softmax(s) @ V[0].astype(np.float64)
    u = 2.0**-11
    ds = scale * np.abs(K[0]).astype(np.float64) @ np.abs(q[0]).astype(np.float64) * u
    bound = np.abs(V).max() * u + 2 * ds.max() * np.abs(V).max()
    assert np.abs(out[0] - exact).max() <= bound
    assert np.abs(out[0] - exact).max() > 0  # the rounding is really there


# ---------------------------------------------------------------------------------
# split triples and their merge
# ---------------------------------------------------------------------------------

def test_partials_and_combine():
    rng = np.random.default_rng(21)
    Hkv, G, n, D = 2, 3, 97, 64
    Hq = Hkv * G
    K = rng.standard_normal((Hkv, n, D)).astype(np.float32) * 2
    V = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    q = rng.standard_normal((Hq, D)).astype(np.float32)
    scale = 0.125
    kc, ks = _cache("q8_0", K)
    vc, vs = _cache("q4_0", V)
    ref, ref_lse = oracle.attention("q8_0", kc, ks, "q4_0", vc, vs, n, q, scale)
    for bounds in ([0, n], [0, 1, n], [0, 16, 32, 48, 64, 80, 96, n], [0, 40, 40, 90, n], [0, 0, n]):
        o, m, l = oracle.attention_partials("q8_0", kc, ks, "q4_0", vc, vs, bounds, q, scale)
        out, lse = oracle.combine(o, m, l)
        assert np.abs(out - ref).max() < 1e-13 and np.abs(lse - ref_lse).max() < 1e-12
        # order of the splits does not matter
        perm = rng.permutation(len(bounds) - 1)
        out2, lse2 = oracle.combine(o[:, perm], m[:, perm], l[:, perm])
        assert np.abs(out2 - ref).max() < 1e-13 and np.abs(lse2 - ref_lse).max() < 1e-12
    # a single split: combine only normalises
    o, m, l = oracle.attention_partials("q8_0", kc, ks, "q4_0", vc, vs, [0, n], q, scale)
    out, lse = oracle.combine(o, m, l)
    assert np.abs(out - o[:, 0] / l[:, :1]).max() < 1e-15
    assert np.abs(lse - (m[:, 0] + np.log(l[:, 0]))).max() < 1e-15
    # empty split triples are (m, l, o) = (-inf, 0, 0); all-empty merges to (0, -inf)
    o, m, l = oracle.attention_partials("q8_0", kc, ks, "q4_0", vc, vs, [5, 5, 5], q, scale)
    assert np.isneginf(m).all() and (l == 0).all() and (o == 0).all()
    out, lse = oracle.combine(o, m, l)
    assert (out == 0).all() and np.isneginf(lse).all()


# ---------------------------------------------------------------------------------------
# automatic KV tier ("HAL #582 -- per-layer KV compression study", section 5 P1)
# ---------------------------------------------------------------------------------------
def _tier_rows():
    rows = []
    with open(os.path.join(GOLDEN, "tier_ladder.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c = [x.strip() for x in line.split("|")]
                rows.append((int(c[0]), int(c[1]), int(c[2]), int(c[3]), int(c[4]), c[5], c[6], int(c[7])))
    return rows


@pytest.mark.parametrize("row", _tier_rows())
def test_tier_ladder_worked_example(row):
    """The page's validation: each budget picks the printed rung, at the printed size."""
    cells, L, H, D, budget_mib, tk, tv, kv_mib = row
    t = oracle.select_tier(cells, L, H, D, budget_mib << 20)
    assert (t["type_k"], t["type_v"]) == (tk, tv)
    assert t["fits"] and t["bytes"] == kv_mib << 20


def test_tier_ladder_properties():
    L, H, D, cells = 48, 8, 128, 32768
    sizes = [oracle.kv_cache_bytes(cells, L, H, D, tk, tv) for tk, tv in oracle.TIER_LADDER]
    assert sizes == sorted(sizes, reverse=True)            # each rung compresses more
    assert sizes[0] == 6144 << 20                           # f16: 192 KiB/token (section 1)
    # f16 whenever it fits, including exactly at the budget
    assert oracle.select_tier(cells, L, H, D, sizes[0])["rung"] == 0
    # one byte short of a rung moves one rung down
    for r in range(3):
        assert oracle.select_tier(cells, L, H, D, sizes[r] - 1)["rung"] == r + 1
    # nothing fits: the floor, flagged
    t = oracle.select_tier(cells, L, H, D, sizes[3] - 1)
    assert t["rung"] == 3 and not t["fits"]
    # monotone: a larger budget never picks a more compressing rung
    prev = 3
    for budget in range(0, sizes[0] + (64 << 20), 97 << 20):
        r = oracle.select_tier(cells, L, H, D, budget)["rung"]
        assert r <= prev
        prev = r
    # no cells cost nothing
    assert oracle.select_tier(0, L, H, D, 0) == {"rung": 0, "type_k": "f16", "type_v": "f16", "fits": True, "bytes": 0}


# ---------------------------------------------------------------------------------------
# q4_1 / q5_0 / q5_1 (the further scalar types; GGML-style reading, see kvq_oracle.c)
# ---------------------------------------------------------------------------------------
def qx(kv_type, x):
    c, s = oracle.quantize(kv_type, np.asarray(x, np.float32).reshape(1, 32))
    return c[0].astype(np.int64), [int(v) for v in s[0]]


def f16val(bits):
    return float(np.uint16(bits).view(np.float16))


@pytest.mark.parametrize("kv_type,levels", [("q4_1", 15), ("q5_1", 31)])
def test_min_types_zero_equal_and_ramp(kv_type, levels):
    c, s = qx(kv_type, np.zeros(32))
    assert (c == 0).all() and s == [0, 0]
    for a in (0.375, -2.5, 1000.0):                      # all equal: d = 0, x_hat = lo = a exactly
        c, s = qx(kv_type, np.full(32, a))
        assert (c == 0).all() and s == [0, f16bits(a)]
        assert (oracle.dequantize(kv_type, c[None].astype(np.uint8), np.array([s], np.uint16), 32) == a).all()
    lo, step = -1.0, 0.125                               # a ramp over every level: codes are the levels
    j = np.arange(32) % (levels + 1)
    x = (lo + step * j).astype(np.float32)
    c, s = qx(kv_type, x)
    assert (c == j).all() and s == [f16bits(step), f16bits(lo)]
    assert np.array_equal(oracle.dequantize(kv_type, c[None].astype(np.uint8), np.array([s], np.uint16), 32)[0], x)


@pytest.mark.parametrize("kv_type,levels", [("q4_1", 15), ("q5_1", 31)])
def test_min_types_brute_force_nearest(kv_type, levels):
    """c = min(levels, floor((x - lo)/d + 1/2)) in exact arithmetic, near-ties excepted; the
    code is the nearest level, so |x - (lo + d c)| <= d/2 on the fp32 d."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-4, 4)
        x = (rng.standard_normal(32) * scale + rng.uniform(-3, 3) * scale).astype(np.float32)
        c, s = qx(kv_type, x)
        lo, hi = f32(x.min()), f32(x.max())
        d32 = (hi - lo) / f32(levels)
        d = Fraction(float(d32))
        for j in range(32):
            t = (Fraction(float(x[j])) - Fraction(float(lo))) / d + Fraction(1, 2)
            fl = math.floor(t)
            if abs(t - round(t)) < Fraction(1, 2**18) and t != round(t):
                assert c[j] in {min(levels, fl), min(levels, fl - 1), min(levels, fl + 1)}
            else:
                assert c[j] == min(levels, fl)
            err = abs(Fraction(float(x[j])) - Fraction(float(lo)) - d * c[j])
            assert err <= d / 2 * (1 + Fraction(1, 2**18)) or c[j] == levels
        assert s == [f16bits(d32), f16bits(lo)]


def test_q5_0_zero_equal_tie_clip_and_brute_force():
    c, s = qx("q5_0", np.zeros(32))
    assert (c == 16).all() and s == [0x8000]             # d = 0 / -16 = -0
    c, s = qx("q5_0", np.full(32, 0.5))                  # all equal: code 0, x_hat = -16 d = a
    assert (c == 0).all() and f16val(s[0]) == -0.5 / 16
    x = np.zeros(32, np.float32)
    x[3], x[7] = 2.0, -2.0                               # tie: the first index sets the sign of d
    c, s = qx("q5_0", x)
    assert f16val(s[0]) == -0.125 and c[3] == 0 and c[7] == 31   # -2.0 would be 32: clipped
    rng = np.random.default_rng(12)
    for trial in range(300):
        xb = (rng.standard_normal(32) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32)
        c, s = qx("q5_0", xb)
        k = int(np.argmax(np.abs(xb)))
        d32 = f32(xb[k]) / f32(-16)
        d = Fraction(float(d32))
        for j in range(32):
            t = Fraction(float(xb[j])) / d + Fraction(33, 2)
            fl = math.floor(t)
            if abs(t - round(t)) < Fraction(1, 2**18) and t != round(t):
                assert c[j] in {min(31, fl), min(31, fl - 1), min(31, fl + 1)}
            else:
                assert c[j] == min(31, fl)
        assert s == [f16bits(d32)]


@pytest.mark.parametrize("tk,tv", [("q5_0", "q5_0"), ("q4_1", "q4_1"), ("q5_1", "q5_1"), ("q8_0", "q5_0"),
                                   ("q5_1", "q4_0")])
def test_new_types_attention_against_independent_decode(tk, tv):
    """Attention over the new types equals fp64 softmax attention on values decoded here,
    independently of the oracle's dequantiser, from its codes and scales."""
    rng = np.random.default_rng(13)
    H, n, D, G = 2, 37, 64, 3
    K = rng.standard_normal((H, n, D)).astype(np.float32)
    V = rng.standard_normal((H, n, D)).astype(np.float32)
    q = rng.standard_normal((H * G, D)).astype(np.float32)

    def decode(kv_type, c, s):
        d = np.vectorize(f16val)(s).astype(np.float64)
        if kv_type == "q8_0":
            return np.repeat(d, 32, -1) * c
        if kv_type == "q4_0":
            codes = np.concatenate([c.reshape(*c.shape[:-1], -1, 16) & 15, c.reshape(*c.shape[:-1], -1, 16) >> 4],
                                   -1).reshape(*c.shape[:-1], -1)
            return np.repeat(d, 32, -1) * (codes.astype(np.float64) - 8)
        if kv_type == "q5_0":
            return np.repeat(d, 32, -1) * (c.astype(np.float64) - 16)
        dd, lo = d[..., 0::2], d[..., 1::2]
        return np.repeat(dd, 32, -1) * c + np.repeat(lo, 32, -1)

    kc, ks = oracle.quantize(tk, K)
    vc, vs = oracle.quantize(tv, V)
    Kh, Vh = decode(tk, kc, ks), decode(tv, vc, vs)
    assert np.array_equal(Kh, oracle.dequantize(tk, kc, ks, D)) and np.array_equal(Vh, oracle.dequantize(tv, vc, vs, D))
    scale = float(np.float32(1 / math.sqrt(D)))
    out, lse = oracle.attention(tk, kc, ks, tv, vc, vs, n, q, scale)
    for hq in range(H * G):
        s_ = scale * (Kh[hq // G] @ q[hq].astype(np.float64))
        p = np.exp(s_ - s_.max())
        assert np.allclose(out[hq], p @ Vh[hq // G] / p.sum(), rtol=1e-12, atol=1e-12)
        assert abs(lse[hq] - (s_.max() + math.log(p.sum()))) < 1e-12
