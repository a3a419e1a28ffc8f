"""Pins for the CPU oracle: each check ties it to something other than itself.

* hand-worked blocks from the pages' formulas (tests/golden/, each cited there),
* numpy's IEEE fp16 conversion over all 65536 bit patterns,
* the 96-bit bijection of the Q4_K 6-bit scale/min packing (page 1),
* exact closed forms (the dequantised value is a single rounding of an
  exactly representable fp64 expression),
* the IQ3 sign-parity invariant and an encode -> decode round trip (page 4),
* math.fsum for the fp64 dot product.
"""
import math

import numpy as np
import pytest

import oracle
from block_quantised_weight_gb300 import synth


# ------------------------------------------------------------------- sizes
def test_block_sizes_and_bpw():
    # page 1: 144 bytes -> 256 weights (4.5 bpw); page 4: 64 + 32 + 2 = 98 (3.0625 bpw)
    assert oracle.Q4K_BYTES == 144 and 144 * 8 / 256 == 4.5
    assert oracle.IQ3_BYTES == 256 // 4 + (256 // 32) * 4 + 2 == 98
    assert 98 * 8 / 256 == 3.0625
    W = synth.gen_q4k(3, 512, 0)
    assert W.shape == (3, 2 * 144)
    assert oracle.dequant_q4k(W, 512).shape == (3, 512)
    Wi, g = synth.gen_iq3(3, 768, 0)
    assert Wi.shape == (3, 3 * 98) and g.shape == (256, 4)
    assert oracle.dequant_iq3(Wi, g, 768).shape == (3, 768)


# ------------------------------------------------------------------- fp16
def test_f16_all_bit_patterns_match_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # spot values from the binary16 definition
    assert oracle.f16_to_f32(np.array([0x3C00, 0x0001, 0x7BFF, 0xFC00], np.uint16)).tolist() == [
        1.0, 2.0 ** -24, 65504.0, -math.inf]


# ------------------------------------------------------------------- Q4_K
def _q4k_golden(golden):
    rows = golden("q4k_block_handworked.txt")
    kv = {}
    ws, w2s = [], []
    for r in rows:
        if r[0] == "w":
            ws.append((int(r[1]), float(r[2])))
        elif r[0] == "w2":
            w2s.append((int(r[1]), float(r[2])))
        else:
            kv[r[0]] = r[1:]
    return kv, ws, w2s


def _q4k_golden_block(kv, header_key):
    qs = np.array([(l % 16) | ((15 - l % 16) << 4) for g in range(4) for l in range(32)], np.uint8)
    blk = np.concatenate([
        np.array([int(t, 16) for t in kv[header_key]], np.uint8),
        np.array([int(t, 16) for t in kv["scales"]], np.uint8),
        qs,
    ])
    assert blk.size == 144
    return blk, qs


def test_q4k_handworked_block(golden):
    kv, ws, w2s = _q4k_golden(golden)
    blk, qs = _q4k_golden_block(kv, "header")
    sc_ref = [int(t) for t in kv["sc"]]
    mn_ref = [int(t) for t in kv["mn"]]
    # the unpack gives the hand-chosen fields
    sc, mn = oracle.q4k_scale_min(blk[4:16])
    assert sc.tolist() == sc_ref and mn.tolist() == mn_ref
    # the block writer produces the hand-packed bytes
    assert np.array_equal(oracle.q4k_block(1.0, 0.5, sc_ref, mn_ref, qs), blk)
    w = oracle.dequant_q4k(blk[None, :], 256)[0]
    for i, v in ws:
        assert w[i] == np.float32(v), (i, w[i], v)
    blk2, _ = _q4k_golden_block(kv, "header2")
    w2 = oracle.dequant_q4k(blk2[None, :], 256)[0]
    for i, v in w2s:
        assert w2[i] == np.float32(v), (i, w2[i], v)


def test_q4k_scale_min_bit_bijection():
    """Each of the 96 packed bits lands in exactly one of the 16 six-bit fields,
    and every field bit is hit exactly once (page 1: j >= 4 straddles bytes)."""
    hit = set()
    for bit in range(96):
        p = np.zeros(12, np.uint8)
        p[bit // 8] = 1 << (bit % 8)
        sc, mn = oracle.q4k_scale_min(p)
        fields = np.concatenate([sc, mn]).astype(int)
        nz = np.nonzero(fields)[0]
        assert nz.size == 1, (bit, fields)
        f = int(nz[0])
        v = int(fields[f])
        assert v & (v - 1) == 0 and v < 64
        hit.add((f, v.bit_length() - 1))
    assert len(hit) == 96
    # the straddled field sc[4] takes bits 6-7 of byte 0 as its top bits
    p = np.zeros(12, np.uint8)
    p[0] = 0xC0
    sc, mn = oracle.q4k_scale_min(p)
    assert sc[4] == 48 and sc[0] == 0 and not mn.any()


def test_q4k_pack_unpack_roundtrip():
    rng = np.random.default_rng(11)
    for _ in range(200):
        p = rng.integers(0, 256, 12, dtype=np.uint8)
        sc, mn = oracle.q4k_scale_min(p)
        assert np.array_equal(oracle.pack_q4k_scale_min(sc, mn), p)
        sc2 = rng.integers(0, 64, 8)
        mn2 = rng.integers(0, 64, 8)
        s3, m3 = oracle.q4k_scale_min(oracle.pack_q4k_scale_min(sc2, mn2))
        assert s3.tolist() == sc2.tolist() and m3.tolist() == mn2.tolist()


def test_q4k_exact_single_rounding():
    """d*sc*q and dmin*mn are exact in fp32 and their difference is exact in
    fp64, so each weight is the fp64 expression rounded once to fp32."""
    K = 1024
    W = synth.gen_q4k(16, K, 5)
    got = oracle.dequant_q4k(W, K)
    blk = W.reshape(-1, 144)
    d = blk[:, 0:2].copy().view("<f2").astype(np.float64)[:, 0]
    dmin = blk[:, 2:4].copy().view("<f2").astype(np.float64)[:, 0]
    ref = np.empty((blk.shape[0], 256), np.float64)
    for b in range(blk.shape[0]):
        sc, mn = oracle.q4k_scale_min(blk[b, 4:16])
        qs = blk[b, 16:144].reshape(4, 32).astype(np.float64)
        for g in range(4):
            ref[b, 64 * g:64 * g + 32] = d[b] * sc[2 * g] * (qs[g] % 16) - dmin[b] * mn[2 * g]
            ref[b, 64 * g + 32:64 * g + 64] = d[b] * sc[2 * g + 1] * (qs[g] // 16) - dmin[b] * mn[2 * g + 1]
    assert np.array_equal(got.reshape(-1, 256), ref.astype(np.float32))


def test_q4k_weight_positions_distinct_per_nibble():
    """Setting one nibble at a time moves exactly the weight page 1 maps it to."""
    base = oracle.q4k_block(1.0, 0.0, [1] * 8, [0] * 8, np.zeros(128, np.uint8))
    for g in range(4):
        for l in (0, 7, 31):
            for hi in (0, 1):
                blk = base.copy()
                blk[16 + 32 * g + l] = (5 << 4) if hi else 5
                w = oracle.dequant_q4k(blk[None, :], 256)[0]
                nz = np.nonzero(w)[0].tolist()
                assert nz == [64 * g + 32 * hi + l] and w[nz[0]] == 5.0


# ------------------------------------------------------------------- IQ3
def _iq3_golden(golden, name="iq3_block_handworked.txt"):
    rows = golden(name)
    grid = np.full((256, 4), 4, np.uint8)
    subs, vals, d = {}, {}, None
    for r in rows:
        if r[0] == "grid_row":
            grid[int(r[1])] = [int(t) for t in r[2:6]]
        elif r[0] == "d":
            d = float(r[1])
        elif r[0] == "sub":
            ib = int(r[1])
            code = int(r[3])
            idx = [int(t) for t in r[5:13]]
            signs = [int(t) for t in r[14:18]]
            subs[ib] = (code, idx, signs)
        elif r[0] == "vals":
            vals[int(r[1])] = [float(t) for t in r[2:]]
    idx = sum((subs[ib][1] for ib in range(8)), [])
    words = [oracle.iq3_word(subs[ib][2], subs[ib][0]) for ib in range(8)]
    return grid, oracle.iq3_block(idx, words, d), vals


def test_iq3_handworked_block(golden):
    grid, blk, vals = _iq3_golden(golden)
    assert blk.size == 98
    assert blk[96:98].tolist() == [0x00, 0x3C]
    w = oracle.dequant_iq3(blk[None, :], grid, 256)[0]
    for ib, v in vals.items():
        assert w[32 * ib:32 * ib + 32].tolist() == v, ib
    for ib in range(4, 8):
        assert w[32 * ib:32 * ib + 32].tolist() == vals[3]
    # halving d halves every value (d is the fp16 at bytes 96-97)
    blk2 = blk.copy()
    blk2[96:98] = np.array([0.5], "<f2").view(np.uint8)
    w2 = oracle.dequant_iq3(blk2[None, :], grid, 256)[0]
    assert np.array_equal(w2, w * np.float32(0.5))


def test_iq3_sign_parity_invariant():
    """Decoded signs: the first seven of each 8-group are the stored bits and
    the count of negatives in every 8-group is even (page 4 decode)."""
    rng = np.random.default_rng(3)
    grid = np.full((256, 4), 8, np.uint8)
    for _ in range(50):
        idx = rng.integers(0, 256, 64)
        sevens = rng.integers(0, 128, (8, 4))
        words = [oracle.iq3_word(sevens[ib], rng.integers(0, 16)) for ib in range(8)]
        w = oracle.dequant_iq3(oracle.iq3_block(idx, words, 1.0)[None, :], grid, 256)[0]
        neg = (w < 0).reshape(8, 4, 8)
        assert (neg.sum(-1) % 2 == 0).all()
        for ib in range(8):
            for l in range(4):
                bits = [(int(sevens[ib, l]) >> j) & 1 for j in range(7)]
                assert neg[ib, l, :7].astype(int).tolist() == bits


def test_iq3_exact_any_order():
    """d*(0.5+code)*0.5*mag*sign needs at most 24 significant bits, so the fp32
    oracle value equals the fp64 product (no rounding at all)."""
    K = 512
    W, grid = synth.gen_iq3(8, K, 9)
    got = oracle.dequant_iq3(W, grid, K).astype(np.float64)
    blk = W.reshape(-1, 98)
    for b in range(blk.shape[0]):
        d = float(blk[b, 96:98].copy().view("<f2")[0])
        words = blk[b, 64:96].copy().view("<u4")
        for ib in range(8):
            code = int(words[ib]) >> 28
            for t in range(32):
                l, j = divmod(t, 8)
                seven = (int(words[ib]) >> (7 * l)) & 0x7F
                neg = ((seven >> j) & 1) if j < 7 else (bin(seven).count("1") & 1)
                mag = grid[blk[b, 8 * ib + t // 4], t % 4] / 2.0
                v = (-1.0 if neg else 1.0) * mag * d * (0.5 + code) * 0.5
                assert got.reshape(-1, 256)[b, 32 * ib + t] == v


def test_iq3_grid_row_and_position_map():
    """Weight t of sub-block ib reads grid row idx[8*ib + t//4], column t % 4."""
    grid = np.zeros((256, 4), np.uint8)
    grid[7] = [2, 4, 6, 8]
    for ib in (0, 5):
        for q in (0, 3, 7):
            idx = np.zeros(64, np.uint8)
            idx[8 * ib + q] = 7
            words = [oracle.iq3_word([0, 0, 0, 0], 1)] * 8
            w = oracle.dequant_iq3(oracle.iq3_block(idx, words, 1.0)[None, :], grid, 256)[0]
            nz = np.nonzero(w)[0].tolist()
            base = 32 * ib + 4 * q
            assert nz == [base, base + 1, base + 2, base + 3]
            # mag = byte/2, db = (0.5+1)*0.5 = 0.75
            assert w[base:base + 4].tolist() == [0.75, 1.5, 2.25, 3.0]


# ------------------------------------------------------------- IQ3 encoder
def test_iq3_encode_decode_roundtrip():
    rng = np.random.default_rng(21)
    grid = synth.gen_iq3_grid(4)
    x = rng.standard_normal((2, 512)).astype(np.float32) * 0.01
    enc = oracle.iq3_encode(x, grid)
    dec = oracle.dequant_iq3(enc, grid, 512)
    g = grid.astype(np.float64) * 0.5
    for r in range(2):
        for sb in range(2):
            xs = x[r, sb * 256:(sb + 1) * 256]
            ds = dec[r, sb * 256:(sb + 1) * 256]
            blk = enc[r, sb * 98:(sb + 1) * 98]
            # signs: equal to sign(x) except one flip at the smallest magnitude of odd groups
            for grp in range(32):
                xn = xs[grp * 8:(grp + 1) * 8] < 0
                dn = ds[grp * 8:(grp + 1) * 8] < 0
                diff = np.nonzero(xn != dn)[0]
                if xn.sum() % 2:
                    assert diff.tolist() == [int(np.argmin(np.abs(xs[grp * 8:(grp + 1) * 8])))]
                else:
                    assert diff.size == 0
            # d is the fp16 of the RMS anchor
            d = float(blk[96:98].copy().view("<f2")[0])
            rms = float(np.sqrt(np.mean(np.abs(xs).astype(np.float32) ** 2, dtype=np.float32)))
            assert d == float(np.float16(np.float32(rms / 20.0 + 1e-12)))
            # brute force: the stored (code, rows) minimise the sub-block error
            words = blk[64:96].copy().view("<u4")
            for ib in range(8):
                m = np.abs(xs[ib * 32:(ib + 1) * 32]).astype(np.float64)
                best = math.inf
                for code in range(16):
                    db = d * (0.5 + code) * 0.5
                    err = 0.0
                    for q in range(8):
                        seg = m[4 * q:4 * q + 4]
                        err += min(((g[i] * db - seg) ** 2).sum() for i in range(256))
                    best = min(best, err)
                code = int(words[ib]) >> 28
                db = d * (0.5 + code) * 0.5
                got = ((np.abs(ds[ib * 32:(ib + 1) * 32]).astype(np.float64) - m) ** 2).sum()
                assert got <= best * (1 + 1e-4) + 1e-18
    # decoding then re-encoding with the stored d reproduces the decoded values
    dstore = enc.reshape(2, 2, 98)[:, :, 96:98].copy().view("<f2").astype(np.float64)[..., 0]
    enc2 = oracle.iq3_encode(dec, grid, force_d=dstore)
    assert np.array_equal(oracle.dequant_iq3(enc2, grid, 512), dec)


# ------------------------------------------------------------------- GEMV
def test_gemv_matches_fsum():
    """fp32*fp32 products are exact in fp64, so fsum of them is the correctly
    rounded exact dot; the oracle's sequential fp64 sum is within K ulps."""
    K = 512
    W = synth.gen_q4k(5, K, 2)
    x = synth.gen_x(2, K, 3)
    Y, A = oracle.gemv_q4k(W, x)
    w = oracle.dequant_q4k(W, K).astype(np.float64)
    for m in range(2):
        for n in range(5):
            prods = w[n] * x[m].astype(np.float64)
            exact = math.fsum(prods)
            assert abs(Y[m, n] - exact) <= K * 2.0 ** -53 * A[m, n]
            assert abs(A[m, n] - math.fsum(np.abs(prods))) <= K * 2.0 ** -53 * A[m, n]
    Wi, grid = synth.gen_iq3(4, K, 6)
    Yi, Ai = oracle.gemv_iq3(Wi, grid, x)
    wi = oracle.dequant_iq3(Wi, grid, K).astype(np.float64)
    for m in range(2):
        for n in range(4):
            prods = wi[n] * x[m].astype(np.float64)
            assert abs(Yi[m, n] - math.fsum(prods)) <= K * 2.0 ** -53 * Ai[m, n]


def test_gemv_row_subset_and_threads():
    K = 768
    W = synth.gen_q4k(40, K, 8)
    x = synth.gen_x(3, K, 9)
    Y, A = oracle.gemv_q4k(W, x, nthreads=1)
    rows = np.array([39, 0, 17, 17, 5])
    Ys, As = oracle.gemv_q4k(W, x, rows=rows, nthreads=4)
    assert np.array_equal(Ys, Y[:, rows]) and np.array_equal(As, A[:, rows])
    # agrees with numpy's fp64 matmul of the dequantised rows (a library dot)
    ref = x.astype(np.float64) @ oracle.dequant_q4k(W, K).astype(np.float64).T
    assert np.allclose(Y, ref, rtol=0, atol=1e-12 * A.max())


def test_zero_rows_give_exact_zero():
    K = 512
    W = synth.gen_q4k(3, K, 1)
    W[1] = 0                      # d = dmin = 0 in every block
    x = synth.gen_x(1, K, 2)
    Y, A = oracle.gemv_q4k(W, x)
    assert Y[0, 1] == 0.0 and A[0, 1] == 0.0


# ------------------------------------------------- decode-step prologues
def test_rmsnorm_worked_example():
    """Page 2 "Candle", RmsNorm::forward on x = (3, 4): mean(x^2) = 12.5, so
    the outputs are 3/sqrt(12.5) and 4/sqrt(12.5) (worked by hand:
    0.8485281374238570, 1.1313708498984760), times the weight."""
    h = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 1.0]), 0.0)
    assert np.allclose(h, [0.8485281374238570, 1.1313708498984760], rtol=1e-15, atol=0)
    h2 = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([2.0, -0.5]), 0.0)
    assert np.allclose(h2, [1.6970562748477140, -0.5656854249492380], rtol=1e-15, atol=0)
    # eps enters under the root: x = (0, 0, 0, 2), eps = 1 -> 2 / sqrt(1 + 1)
    h3 = oracle.rmsnorm(np.array([0.0, 0.0, 0.0, 2.0]), np.ones(4), 1.0)
    assert np.allclose(h3, [0, 0, 0, 2 / math.sqrt(2.0)], rtol=1e-15, atol=0)


def test_rmsnorm_invariants():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((3, 64))
    w = np.ones(64)
    h = oracle.rmsnorm(x, w, 0.0)
    assert np.allclose(np.mean(h * h, axis=-1), 1.0, rtol=1e-13)          # unit mean square
    assert np.allclose(oracle.rmsnorm(7.5 * x, w, 0.0), h, rtol=1e-13)     # scale invariant
    assert np.allclose(oracle.rmsnorm(np.full(8, -3.0), np.ones(8), 0.0), -1.0, rtol=1e-15)
    g = rng.standard_normal(64)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), h * g, rtol=1e-13)       # weight is elementwise
    assert np.all(oracle.rmsnorm(np.zeros(16), np.ones(16), 1e-6) == 0.0)  # eps keeps zero finite


def test_silu_closed_forms():
    """silu(z) = z / (1 + exp(-z)): silu(0) = 0, silu(1) = e / (e + 1),
    silu(z) - silu(-z) = z, silu(z) -> z for large z and -> 0 for very
    negative z."""
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - math.e / (math.e + 1.0)) < 1e-16
    z = np.linspace(-30, 30, 121)
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=0, atol=1e-13)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-14
    assert oracle.silu(-800.0) == 0.0 and np.isfinite(oracle.silu(-800.0))
    assert np.allclose(oracle.swiglu(z, 2.0 * z), 2.0 * z * oracle.silu(z), rtol=1e-15)


def test_fused_gemv_reduces_to_the_plain_oracle():
    """No prologue: the fp64 matmul of the C-dequantised W equals the C GEMV;
    with a prologue, it equals the C GEMV of the fp32-rounded h within fp32
    rounding of h; the residual is added exactly."""
    K = 768
    W = synth.gen_q4k(33, K, 21)
    x = synth.gen_x(3, K, 22)
    Y0, A0 = oracle.fused_gemv_q4k(W, x)
    Yc, Ac = oracle.gemv_q4k(W, x)
    assert np.allclose(Y0, Yc, rtol=0, atol=1e-12 * A0.max()) and np.allclose(A0, Ac, rtol=1e-12)
    g = synth.gen_x(1, K, 23)[0]
    h = oracle.rmsnorm(x, g, 1e-5)
    Yn, An = oracle.fused_gemv_q4k(W, x, norm_weight=g, eps=1e-5)
    Yh, _ = oracle.gemv_q4k(W, h.astype(np.float32))
    assert np.all(np.abs(Yn - Yh) <= 2.0 ** -23 * An)
    up = synth.gen_x(3, K, 24)
    Ys, As = oracle.fused_gemv_q4k(W, x, up=up)
    Yh2, _ = oracle.gemv_q4k(W, oracle.swiglu(x, up).astype(np.float32))
    assert np.all(np.abs(Ys - Yh2) <= 2.0 ** -23 * As)
    R = synth.gen_x(3, 33, 25)
    Yr, _ = oracle.fused_gemv_q4k(W, x, up=up, residual=R)
    assert np.array_equal(Yr, Ys + R.astype(np.float64))


# ------------------------------------------------------------------ IQ3_XXS
def _iq3xxs_golden(golden):
    """The golden fields written in page 3's order: d, the 64 index bytes,
    the eight words (built by hand here, not by a converter)."""
    grid, p4blk, vals = _iq3_golden(golden, "iq3xxs_block_handworked.txt")
    d16 = p4blk[96:98]
    blk = np.concatenate([d16, p4blk[0:64], p4blk[64:96]]).astype(np.uint8)
    return grid, blk, vals


def test_iq3xxs_handworked_block(golden):
    grid, blk, vals = _iq3xxs_golden(golden)
    assert blk.size == 98 and blk[0:2].tolist() == [0x00, 0x3C]      # d first (page 3)
    w = oracle.dequant_iq3xxs(blk[None, :], grid, 256)[0]
    for ib, v in vals.items():
        assert w[32 * ib:32 * ib + 32].tolist() == v, ib
    for ib in range(4, 8):
        assert w[32 * ib:32 * ib + 32].tolist() == vals[3]


def test_iq3xxs_is_page4_reordered_and_doubled():
    """Page 3's eff = d*(0.5+s)*0.5 times the raw entry versus page 4's
    d*(0.5+code)*0.5 * entry*0.5: the same fields in the two byte orders
    give values in a ratio of exactly 2."""
    K = 768
    W, grid = synth.gen_iq3(9, K, 31)
    x3 = oracle.iq3_to_iq3xxs(W, K)
    assert not np.array_equal(x3, W)
    a = oracle.dequant_iq3(W, grid, K)
    b = oracle.dequant_iq3xxs(x3, grid, K)
    assert np.array_equal(b, 2.0 * a)
    x = synth.gen_x(2, K, 32)
    Ya, Aa = oracle.gemv_iq3(W, grid, x)
    Yb, Ab = oracle.gemv_iq3xxs(x3, grid, x)
    assert np.array_equal(Yb, 2.0 * Ya) and np.array_equal(Ab, 2.0 * Aa)


def test_iq3xxs_field_positions():
    """Bytes 0-1 scale the whole block; a byte in 2-65 moves one 4-weight
    group; the top byte of the word at 66+4*ib changes only sub-block ib."""
    K = 256
    W, grid = synth.gen_iq3(1, K, 33)
    W = oracle.iq3_to_iq3xxs(W, K)
    base = oracle.dequant_iq3xxs(W, grid, K)[0]
    v = W.copy()
    v[0, 0:2] = np.array([0x3C00], "<u2").view(np.uint8)              # d = 1
    v2 = v.copy()
    v2[0, 0:2] = np.array([0x4000], "<u2").view(np.uint8)             # d = 2
    assert np.array_equal(oracle.dequant_iq3xxs(v2, grid, K), 2.0 * oracle.dequant_iq3xxs(v, grid, K))
    for t in (2, 17, 65):
        w2 = W.copy()
        w2[0, t] ^= 0x5A
        diff = np.nonzero(oracle.dequant_iq3xxs(w2, grid, K)[0] != base)[0]
        assert diff.size and diff.min() >= 4 * (t - 2) and diff.max() < 4 * (t - 2) + 4
    for ib in (0, 5, 7):
        w3 = W.copy()
        w3[0, 66 + 4 * ib + 3] ^= 0x30                                  # bits 28-29: s
        diff = np.nonzero(oracle.dequant_iq3xxs(w3, grid, K)[0] != base)[0]
        assert diff.size and diff.min() >= 32 * ib and diff.max() < 32 * ib + 32


# ------------------------------------------------ page 3's codebook formats
def _cb_golden(golden):
    """{fmt: (W bytes [1, unit], table, {weight: value})} from the fixture."""
    out, cur = {}, None
    for r in golden("cb_blocks_handworked.txt"):
        if r[0] == "format":
            cur = r[1]
            if cur in ("iq4nl", "iq4xs"):
                tab = np.zeros(16, np.int8)
            elif cur == "iq3s":
                tab = np.ones((512, 4), np.uint8)
            else:
                tab = np.full((256, 8), 8, np.uint8)
            out[cur] = [None, tab, {}]
        elif r[0] == "table":
            out[cur][1][:] = [int(t) for t in r[1:]]
        elif r[0] == "gridrow":
            out[cur][1][int(r[1])] = [int(t) for t in r[2:]]
        elif r[0] == "bytes":
            out[cur][0] = np.array([int(t, 16) for t in r[1:]], np.uint8)
        elif r[0] == "val":
            out[cur][2][int(r[1])] = float(r[2])
    for fmt, e in out.items():   # pad IQ4_NL's two blocks to a 256-weight unit (d = 0 blocks)
        unit = synth.CB_UNIT_BYTES[fmt]
        e[0] = np.concatenate([e[0], np.zeros(unit - e[0].size, np.uint8)])[None, :]
    return out


@pytest.mark.parametrize("fmt", ["iq4nl", "iq4xs", "iq3s", "iq2xxs"])
def test_cb_handworked_blocks(golden, fmt):
    W, tab, vals = _cb_golden(golden)[fmt]
    w = oracle.dequant_cb(fmt, W, tab, 256)[0]
    for k, v in vals.items():
        assert w[k] == np.float32(v), (fmt, k, w[k], v)
    if fmt == "iq4nl":
        assert np.all(w[64:] == 0.0)      # the padding blocks have d = 0


@pytest.mark.parametrize("fmt", ["iq4nl", "iq4xs", "iq3s", "iq2xxs"])
def test_cb_exact_products_and_sizes(fmt):
    """Bytes per 256 weights from page 3's table (IQ4_NL 18 per 32); every
    value is eff * v exactly (an fp64 recomputation from the same fields
    agrees bit for bit); doubling d doubles every value of its block."""
    K = 512
    W, tab = synth.gen_cb(fmt, 4, K, 41)
    assert W.shape == (4, 2 * {"iq4nl": 144, "iq4xs": 136, "iq3s": 110, "iq2xxs": 66}[fmt])
    w = oracle.dequant_cb(fmt, W, tab, K)
    W2 = W.copy()
    if fmt == "iq4nl":
        d = W2.reshape(-1, 18)[:, 0:2].copy().view("<f2")
        W2.reshape(-1, 18)[:, 0:2] = (d.astype(np.float32) * 2).astype("<f2").view(np.uint8)
    else:
        u = synth.CB_UNIT_BYTES[fmt]
        d = W2.reshape(-1, u)[:, 0:2].copy().view("<f2")
        W2.reshape(-1, u)[:, 0:2] = (d.astype(np.float32) * 2).astype("<f2").view(np.uint8)
    assert np.array_equal(oracle.dequant_cb(fmt, W2, tab, K), 2 * w)


def test_iq4_table_sign_and_nibble_order():
    """IQ4_NL: negating the table negates every value; swapping the nibbles
    of every code byte swaps weights i and i+16 (page 3, encode)."""
    W, tab = synth.gen_cb("iq4nl", 2, 256, 42)
    w = oracle.dequant_cb("iq4nl", W, tab, 256)
    assert np.array_equal(oracle.dequant_cb("iq4nl", W, (-tab.astype(np.int16)).clip(-127, 127).astype(np.int8), 256), -w)
    Ws = W.copy().reshape(-1, 18)
    Ws[:, 2:] = (Ws[:, 2:] >> 4) | (Ws[:, 2:] << 4)
    ws = oracle.dequant_cb("iq4nl", Ws.reshape(W.shape), tab, 256).reshape(-1, 2, 16)
    assert np.array_equal(ws[:, 0], w.reshape(-1, 2, 16)[:, 1]) and np.array_equal(ws[:, 1], w.reshape(-1, 2, 16)[:, 0])


def test_cb_sign_parity_invariant():
    """IQ2_XXS: every 8-weight group has an even number of negative values
    (seven stored signs plus their parity); IQ3_S stores all 256 signs."""
    W, tab = synth.gen_cb("iq2xxs", 16, 256, 43)
    w = oracle.dequant_cb("iq2xxs", W, tab, 256).reshape(-1, 8)
    assert np.all((w < 0).sum(axis=1) % 2 == 0)
    W3, t3 = synth.gen_cb("iq3s", 16, 256, 44)
    w3 = oracle.dequant_cb("iq3s", W3, t3, 256)
    neg = np.unpackbits(W3.reshape(-1, 110)[:, 74:106], axis=1, bitorder="little").reshape(w3.shape)
    assert np.array_equal(neg == 1, w3 < 0)


@pytest.mark.parametrize("fmt", ["iq4nl", "iq4xs", "iq3s", "iq2xxs"])
def test_cb_gemv_matches_fsum(fmt):
    K = 512
    W, tab = synth.gen_cb(fmt, 3, K, 45)
    x = synth.gen_x(2, K, 46)
    Y, A = oracle.gemv_cb(fmt, W, tab, x)
    w = oracle.dequant_cb(fmt, W, tab, K).astype(np.float64)
    for m in range(2):
        for n in range(3):
            prods = w[n] * x[m].astype(np.float64)
            assert abs(Y[m, n] - math.fsum(prods)) <= K * 2.0 ** -53 * A[m, n]
