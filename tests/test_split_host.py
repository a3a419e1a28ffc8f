"""The arithmetic the tensor-core paths rely on, checked on the host.

From 5 tokens both formats multiply small exact integers by x split into
three bf16 parts (hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid),
each rounded to nearest even).  These tests pin the two facts that make the
products exact and the Q4_K sums keep the per-weight accuracy:
  * the split is exact over the stated range |x| in [2^-100, 2^100]: every
    remainder is an fp32 value, lo equals the last remainder, and
    hi + mid + lo = x;
  * the Q4_K offset factoring (page 1 "Rewriting picoLM in Python",
    dequantize_q4_K, w = a*q - b with a = d*sc, b = dmin*mn) with c the
    integer in [0, 15] nearest b/a: where b/a <= 15.5 (c not clamped),
    r = b - a*c is exact in fp32 when c > 0, |r| <= a/2 and
    |a*(q - c)| <= 2|a*q - b| for q != c, so a*sum((q-c)*x) - r*sum(x) has
    every term bounded by its weight's |w*x|; where b/a > 15.5 (c = 15) r
    is rounded once, but a*(q - 15) and -r then share their sign, so every
    term is still bounded by |w*x|.
The same rounding is emulated here in numpy (bf16 = the upper 16 bits of
an fp32 after round-to-nearest-even), independent of the CUDA code.
"""
import numpy as np


def bf16_rn(x):
    """fp32 -> the nearest bf16 (ties to even), returned as fp32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def split3(x):
    x = np.asarray(x, dtype=np.float32)
    hi = bf16_rn(x)
    r1 = (x - hi).astype(np.float32)
    mid = bf16_rn(r1)
    r2 = (r1 - mid).astype(np.float32)
    lo = bf16_rn(r2)
    return hi, mid, lo, r1, r2


def test_three_bf16_parts_split_fp32_exactly():
    rng = np.random.default_rng(5)
    n = 200_000
    mant = rng.uniform(1.0, 2.0, n)
    expo = rng.integers(-100, 101, n)
    sign = rng.choice([-1.0, 1.0], n)
    x = (sign * mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    hi, mid, lo, r1, r2 = split3(x)
    # the remainders are exact (Sterbenz): computed in fp64 they agree
    assert np.array_equal(r1.astype(np.float64), x.astype(np.float64) - hi.astype(np.float64))
    assert np.array_equal(r2.astype(np.float64), r1.astype(np.float64) - mid.astype(np.float64))
    # the last part takes the rest whole, so the three sum to x exactly
    assert np.array_equal(lo, r2)
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(total, x.astype(np.float64))
    # and each part is a bf16 value (low 16 bits zero)
    for p in (hi, mid, lo):
        assert not (p.view(np.uint32) & 0xFFFF).any()


def test_split_of_integers_and_one_hot_values():
    """A one-hot x (a power of two) is its own hi part: mid = lo = 0."""
    x = np.float32(2.0) ** np.arange(-100, 101, dtype=np.float32)
    hi, mid, lo, _, _ = split3(x)
    assert np.array_equal(hi, x) and not mid.any() and not lo.any()


def q4k_offset(a, b):
    """The integer in [0, 15] nearest b/a (a = 0: the quotient is inf or NaN;
    NaN gives 0, inf the clamp)."""
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(np.float32(b) / np.float32(a))
    q = np.where(np.isnan(q), 0.0, q)
    return np.clip(q, 0.0, 15.0).astype(np.float32)


def test_q4k_offset_factoring_is_exact_and_bounded():
    rng = np.random.default_rng(6)
    n = 100_000
    # d and dmin as fp16 values (the block's fields), sc and mn 6-bit
    d = rng.uniform(2.0 ** -14, 2.0, n).astype(np.float16).astype(np.float32)
    dmin = rng.uniform(2.0 ** -14, 2.0, n).astype(np.float16).astype(np.float32)
    sc = rng.integers(1, 64, n).astype(np.float32)
    mn = rng.integers(0, 64, n).astype(np.float32)
    a = (d * sc).astype(np.float32)
    b = (dmin * mn).astype(np.float32)
    # a and b are exact products (fp16 x 6-bit fits fp32)
    assert np.array_equal(a.astype(np.float64), d.astype(np.float64) * sc.astype(np.float64))
    assert np.array_equal(b.astype(np.float64), dmin.astype(np.float64) * mn.astype(np.float64))
    c = q4k_offset(a, b)
    r = (b - a * c).astype(np.float32)
    exact = b.astype(np.float64) - a.astype(np.float64) * c.astype(np.float64)
    near = b <= 15.5 * a  # the nearest integer lies inside the clamp
    pos = (c > 0) & near
    assert pos.sum() > n // 4 and (~near).sum() > n // 50  # both cases occur
    assert np.array_equal(r[pos].astype(np.float64), exact[pos])
    # clamped: r rounded once, and every weight's two terms share a sign
    far = ~near
    assert (np.abs(r[far].astype(np.float64) - exact[far]) <= np.abs(exact[far]) * 2.0 ** -24).all()
    assert (exact[far] > 0).all()
    assert (np.abs(exact[near]) <= a[near].astype(np.float64) / 2 * (1 + 2.0 ** -20)).all()
    # every weight of the sub-block: |a*(q - c)| <= 2 |a*q - b| where q != c
    for q in range(16):
        w = a.astype(np.float64) * q - b.astype(np.float64)
        t = a.astype(np.float64) * (q - c.astype(np.float64))
        sel = near & (c != q)
        assert (np.abs(t[sel]) <= 2 * np.abs(w[sel]) * (1 + 2.0 ** -20)).all()


def test_q4k_factored_weights_reproduce_the_fp32_weight():
    """a*(q - c) - r, formed as the tensor-core path forms it for a one-hot
    x, is the page's fp32 weight RN(a*q - b) exactly where c is not clamped
    (b/a <= 15.5), and within one ulp of it where it is."""
    rng = np.random.default_rng(7)
    n = 100_000
    d = rng.uniform(2.0 ** -14, 2.0, n).astype(np.float16).astype(np.float32)
    dmin = rng.uniform(2.0 ** -14, 2.0, n).astype(np.float16).astype(np.float32)
    a = (d * rng.integers(0, 64, n).astype(np.float32)).astype(np.float32)
    b = (dmin * rng.integers(0, 64, n).astype(np.float32)).astype(np.float32)
    q = rng.integers(0, 16, n).astype(np.float32)
    c = q4k_offset(a, b)
    r = (b - a * c).astype(np.float32)
    got = (a * (q - c)).astype(np.float32)          # exact: 17-bit a times an integer below 16
    got = (got.astype(np.float64) - r.astype(np.float64)).astype(np.float32)  # one rounding
    want = (a * q - b).astype(np.float32)            # a*q exact, then one rounding
    near = b <= 15.5 * a
    assert np.array_equal(got[near], want[near])
    ulp = np.spacing(np.abs(want[~near]).astype(np.float32)).astype(np.float64)
    assert (np.abs(got[~near].astype(np.float64) - want[~near].astype(np.float64)) <= ulp).all()
