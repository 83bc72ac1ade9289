"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names the passage of the SharpInference issue pages (or the format
definition) it pins and the independent fact used: a closed form, brute
force, exact rational arithmetic, a library routine on a special case, or an
invariant.  Every plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, a wrong rounding rule, a wrong reduction
order) is meant to fail at least one of them.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle as O
from mixture_experts_ffn_top_gb300.workloads import (QK, Q3_K_BYTES, Q4_K_BYTES, Q8_0_BYTES, QK_K, pack_q3_k,
                                                     pack_q4_k, pack_q8_0)

F32_EPS = np.finfo(np.float32).eps


def dequant_q8_0(rows_bytes: np.ndarray) -> np.ndarray:
    """Q8_0 bytes [rows, nblk*34] -> float64 [rows, nblk*32] (format definition)."""
    rows = rows_bytes.shape[0]
    b = rows_bytes.reshape(rows, -1, Q8_0_BYTES)
    d = b[..., :2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = b[..., 2:].view(np.int8).astype(np.float64)
    return (q * d[..., None]).reshape(rows, -1)


def dequant_q4_k(rows_bytes: np.ndarray) -> np.ndarray:
    """Q4_K bytes [rows, nsb*144] -> float64 [rows, nsb*256] (the GGUF super-block definition:
    fp16 d, fp16 dmin, 12 bytes of 6-bit scales/mins, 4-bit quants; d*sc_j*q - dmin*m_j)."""
    rows = rows_bytes.shape[0]
    b = rows_bytes.reshape(rows, -1, Q4_K_BYTES).astype(np.int64)
    d = rows_bytes.reshape(rows, -1, Q4_K_BYTES)[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = rows_bytes.reshape(rows, -1, Q4_K_BYTES)[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    s12 = b[..., 4:16]
    sc = np.concatenate([s12[..., 0:4] & 63, (s12[..., 8:12] & 15) | ((s12[..., 0:4] >> 6) << 4)], axis=-1)
    mn = np.concatenate([s12[..., 4:8] & 63, (s12[..., 8:12] >> 4) | ((s12[..., 4:8] >> 6) << 4)], axis=-1)
    qs = b[..., 16:].reshape(rows, -1, 4, 32)
    q = np.stack([qs & 15, qs >> 4], axis=3).reshape(rows, -1, 8, 32)  # sub-block 2g low, 2g+1 high
    v = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None]
    return v.reshape(rows, -1)


def q3_k_fields(rows_bytes: np.ndarray):
    """Q3_K bytes [rows, nsb*110] -> (d [rows, nsb], s [rows, nsb, 16], q [rows, nsb, 256]) decoded field by
    field from the GGUF super-block definition: 32-byte high-bit mask, 64 bytes of 2-bit low parts,
    12 bytes of sixteen 6-bit scales (offset 32), fp16 d; q = low - 4*(1 - high)."""
    rows = rows_bytes.shape[0]
    b = rows_bytes.reshape(rows, -1, Q3_K_BYTES).astype(np.int64)
    d = rows_bytes.reshape(rows, -1, Q3_K_BYTES)[..., 108:110].copy().view(np.float16)[..., 0].astype(np.float64)
    high = (b[..., None, 0:32] >> np.arange(8)[:, None]) & 1  # [.., 8, 32]: bit k of byte l = value 32k + l
    qs = b[..., 32:96].reshape(rows, -1, 2, 1, 32)  # two 128-value halves
    low = ((qs >> (2 * np.arange(4))[:, None]) & 3).reshape(rows, -1, 8, 32)  # value 128h + 32g + l
    q = (low - 4 * (1 - high)).reshape(rows, -1, QK_K)
    s12 = b[..., 96:108]
    lo = np.concatenate([s12[..., 0:8] & 15, s12[..., 0:8] >> 4], axis=-1)  # scales 0..7, 8..15
    hi = np.concatenate([(s12[..., 8:12] >> (2 * g)) & 3 for g in range(4)], axis=-1)  # scale 4g + m
    return d, (lo | (hi << 4)) - 32, q


def dequant_q3_k(rows_bytes: np.ndarray) -> np.ndarray:
    """Q3_K bytes -> float64 [rows, nsb*256]: d*s_j*q_i, j = i/16."""
    d, sc, q = q3_k_fields(rows_bytes)
    v = d[..., None, None] * sc[..., None] * q.reshape(*q.shape[:-1], 16, 16)
    return v.reshape(rows_bytes.shape[0], -1)


def dequant_q8(q: np.ndarray, d16: np.ndarray) -> np.ndarray:
    d = d16.view(np.float16).astype(np.float64)
    return (q.astype(np.float64).reshape(*q.shape[:-1], -1, QK) * d[..., None]).reshape(q.shape)


# ----------------------------------------------------------------- fp16 ----
def test_half_conversions_match_numpy():
    """IEEE binary16 round trip: numpy's float16 conversion (a library routine) is the pin."""
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 5, 2000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -11), 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11, 0.1, 1 / 3.0], np.float32),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = O.float_to_half(vals)
    np.testing.assert_array_equal(got, ref)
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    bits = bits[(bits & 0x7C00) != 0x7C00]  # finite halves
    np.testing.assert_array_equal(O.half_to_float(bits), bits.view(np.float16).astype(np.float32))


# ------------------------------------------------------------ quantiser ----
def test_q8_1_ramp_block_closed_form():
    """x = 0..31: amax = 31, d = 31/127, q_i = round(127 i / 31) (no ties: 127 i mod 31 != 15.5)."""
    x = np.arange(32, dtype=np.float32)
    q, d16, s16 = O.quantize_q8_1(x)
    expect = [int((Fraction(127 * i, 31) + Fraction(1, 2)) // 1) for i in range(32)]
    assert q.tolist() == expect
    # fp16(31/127): 31/127 = 0.24409..., in [2^-3, 2^-2) -> fraction round(31/127 * 2^13) = 2000
    assert int(d16[0]) == ((12 << 10) + (2000 - 1024))
    assert float(np.uint16(d16[0]).view(np.float16)) == 2000 * 2.0 ** -13
    # Q8_1 sum field: fp16(d * sum q)
    assert int(s16[0]) == int(np.float16(np.float32(31.0 / 127.0) * np.float32(sum(expect))).view(np.uint16))


def test_q8_1_rounding_is_half_away_from_zero():
    """amax = 127 gives d = 1 exactly, so q = roundf(x): halves go away from zero, not to even."""
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -3.5, 0.49999997]
    q, d16, _ = O.quantize_q8_1(x)
    assert q[:9].tolist() == [127, 3, -3, 1, -1, 2, 127, -4, 0]
    assert float(np.uint16(d16[0]).view(np.float16)) == 1.0


def test_q8_1_quants_use_fp32_scale_not_fp16():
    """d = 1 + 2^-12 (fp16(d) = 1): q = roundf(63.5 * fp32(1/d)) = 63; with fp16 d it would be 64."""
    x = np.zeros(32, np.float32)
    x[0] = 127.0 * (1.0 + 2.0 ** -12)  # exact in fp32
    x[1] = 63.5
    q, d16, _ = O.quantize_q8_1(x)
    assert q[0] == 127 and q[1] == 63
    assert float(np.uint16(d16[0]).view(np.float16)) == 1.0


def test_q8_1_invariants_random():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((257, 64)) * np.exp(rng.uniform(-8, 8, (257, 1)))).astype(np.float32)
    x[3] = 0.0  # all-zero row: d = 0, q = 0
    q, d16, s16 = O.quantize_q8_1(x)
    assert np.abs(q.astype(np.int32)).max() <= 127
    xb = x.reshape(-1, 32)
    qb = q.reshape(-1, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=1)
    d32 = (amax / np.float32(127)).astype(np.float32)
    # the element of largest magnitude maps to +-127 (unless the block is zero)
    arg = np.abs(xb).argmax(axis=1)
    nz = amax > 0
    assert np.all(np.abs(qb[np.arange(len(qb)), arg])[nz] == 127)
    assert np.all(qb[~nz] == 0) and np.all(d16.reshape(-1)[~nz] == 0)
    # reconstruction error of every element is at most half a step (plus rounding slack)
    err = np.abs(xb.astype(np.float64) - qb * d32[:, None].astype(np.float64))
    assert np.all(err <= d32[:, None] * (0.5 + 4 * F32_EPS) + 1e-45)
    # the stored scale is the fp16 rounding of d
    np.testing.assert_array_equal(d16.reshape(-1), d32.astype(np.float16).view(np.uint16))
    # the sign of every nonzero quant is the sign of its input
    assert np.all(np.sign(qb) * np.sign(xb) >= 0)


# --------------------------------------------------------------- router ----
def test_router_unit_vectors_select_columns():
    """W_r rows = unit vectors e_j: logits[:, e] = x[:, j_e] exactly (#388 levers item 1)."""
    rng = np.random.default_rng(2)
    N, D, E = 5, 96, 7
    x = rng.standard_normal((N, D)).astype(np.float32)
    cols = rng.choice(D, E, replace=False)
    W = np.zeros((E, D), np.float32)
    W[np.arange(E), cols] = 1.0
    np.testing.assert_array_equal(O.router_logits(x, W), x[:, cols])


def test_router_matches_exactly_rounded_sum():
    """Non-square E != D: the exactly rounded fsum of x[t,d]*W[e,d] agrees to within the
    double-accumulation bound (gamma_D * sum|x w|), which is far below one fp32 ulp."""
    rng = np.random.default_rng(3)
    N, D, E = 6, 200, 9
    x = rng.standard_normal((N, D)).astype(np.float32)
    W = (rng.standard_normal((E, D)) / np.sqrt(D)).astype(np.float32)
    got = O.router_logits(x, W)
    for t in range(N):
        for e in range(E):
            prods = [float(x[t, d]) * float(W[e, d]) for d in range(D)]
            exact = math.fsum(prods)
            bound = D * 2.0 ** -53 * sum(abs(p) for p in prods) + abs(exact) * 2.0 ** -24
            assert abs(float(got[t, e]) - exact) <= bound


# -------------------------------------------------------- softmax / top-k ---
def test_softmax_equal_logits_uniform_and_lowest_indices():
    N, E, k = 3, 12, 4
    logits = np.full((N, E), 0.75, np.float32)
    idx, w, p = O.softmax_topk(logits, k, norm=False)
    np.testing.assert_allclose(p, 1.0 / E, rtol=2 * F32_EPS)
    assert idx.tolist() == [[0, 1, 2, 3]] * N
    np.testing.assert_allclose(w, 1.0 / E, rtol=2 * F32_EPS)
    _, wn, _ = O.softmax_topk(logits, k, norm=True)
    np.testing.assert_allclose(wn, 1.0 / k, rtol=2 * F32_EPS)


def test_topk_brute_force_tie_heavy():
    """Slots = experts sorted by (logit desc, index asc), first k; brute force by full sort."""
    rng = np.random.default_rng(4)
    for E, k in [(8, 2), (64, 8), (256, 8), (9, 9)]:
        logits = rng.integers(-3, 4, (200, E)).astype(np.float32)  # many ties
        idx, _, _ = O.softmax_topk(logits, k, norm=False)
        for t in range(200):
            ref = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert idx[t].tolist() == ref


def test_softmax_weights_against_python_math():
    """w = p_sel (norm off) or p_sel / sum_sel p (norm on), with p the softmax over ALL experts;
    reference computed with math.exp / math.fsum (a different exp and an exact sum)."""
    rng = np.random.default_rng(5)
    N, E, k = 40, 64, 8
    logits = (rng.standard_normal((N, E)) * 3).astype(np.float32)
    for norm in (False, True):
        idx, w, p = O.softmax_topk(logits, k, norm)
        for t in range(N):
            l = [float(v) for v in logits[t]]
            m = max(l)
            ex = [math.exp(v - m) for v in l]
            z = math.fsum(ex)
            pr = [v / z for v in ex]
            np.testing.assert_allclose(p[t], np.array(pr, np.float32), rtol=4 * F32_EPS, atol=1e-30)
            sel = [pr[e] for e in idx[t]]
            ref = [s / math.fsum(sel) for s in sel] if norm else sel
            np.testing.assert_allclose(w[t], np.array(ref, np.float32), rtol=4 * F32_EPS)
        if norm:
            np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=k * F32_EPS)
        else:
            # norm off: the selected weights are the full-softmax probabilities
            np.testing.assert_array_equal(w, np.take_along_axis(p, idx, axis=1))
            assert np.all(w.astype(np.float64).sum(axis=1) < 1.0 + k * F32_EPS)


def test_softmax_is_shift_invariant_at_large_logits():
    """softmax(l + c) = softmax(l): logits near 900 must not overflow exp (max-shifted form)."""
    base = np.array([[0.0, -0.5, -1.0, -50.0]], np.float32)
    idx, w, p = O.softmax_topk(base, 2, norm=False)
    idx2, w2, p2 = O.softmax_topk(base + np.float32(896.0), 2, norm=False)  # exact shift in fp32
    assert np.all(np.isfinite(p2))
    np.testing.assert_array_equal(p2, p)
    assert idx2.tolist() == idx.tolist() == [[0, 1]]
    # closed form: p_i = exp(l_i) / sum_j exp(l_j)
    ex = np.exp(np.array([0.0, -0.5, -1.0, -50.0]))
    np.testing.assert_allclose(p[0], ex / ex.sum(), rtol=4 * F32_EPS)


def test_sigmoid_special_values():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 5.0, -5.0], np.float32)
    s = O.sigmoid(g)
    assert s[0] == 0.5
    assert abs(float(s[1]) - 1 / (1 + math.exp(-1))) <= F32_EPS
    assert abs(float(s[1]) + float(s[2]) - 1.0) <= 2 * F32_EPS
    assert s[3] == 1.0 and 0 < s[4] < 1e-12
    assert abs(float(s[5]) + float(s[6]) - 1.0) <= 2 * F32_EPS


# ------------------------------------------------------------- bucketing ----
def _check_csr(idx, E, expStart, expTokI, expTokK):
    N, k = idx.shape
    assert expStart[0] == 0 and expStart[E] == N * k
    assert np.all(np.diff(expStart) >= 0)
    seen = np.zeros((N, k), np.int32)
    for e in range(E):
        seg = range(expStart[e], expStart[e + 1])
        ts = [int(expTokI[j]) for j in seg]
        assert ts == sorted(ts) and len(set(ts)) == len(ts)  # ascending t inside a segment
        for j in seg:
            t, s = int(expTokI[j]), int(expTokK[j])
            assert idx[t, s] == e
            seen[t, s] += 1
    assert np.all(seen == 1)  # every (token, slot) lands in exactly one bucket


def test_bucket_brute_force_and_invariants():
    """CSR (#388 levers item 1): stable counting sort by expert, checked against Python's
    stable sort of the flat (t, slot) pairs and against the CSR invariants."""
    rng = np.random.default_rng(6)
    for N, E, k in [(1, 8, 2), (64, 8, 2), (300, 64, 8), (50, 256, 8), (33, 9, 9), (17, 5, 1)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
        expStart, expTokI, expTokK = O.bucket(idx, E)
        _check_csr(idx, E, expStart, expTokI, expTokK)
        flat = sorted(range(N * k), key=lambda i: int(idx.flat[i]))  # stable in t, then slot
        assert expTokI.tolist() == [i // k for i in flat]
        assert expTokK.tolist() == [i % k for i in flat]
        np.testing.assert_array_equal(np.diff(expStart), np.bincount(idx.ravel(), minlength=E))


def test_bucket_rejects_bad_routing():
    with pytest.raises(ValueError):
        O.bucket(np.array([[0, 8]], np.int32), 8)
    with pytest.raises(ValueError):
        O.bucket(np.array([[3, 3]], np.int32), 8)
    with pytest.raises(ValueError):
        O.bucket(np.array([[-1, 2]], np.int32), 8)


# -------------------------------------------------------- int8 block dots ---
def test_block_dots_integer_brute_force():
    rng = np.random.default_rng(7)
    K = 256
    w = rng.standard_normal((1, K)).astype(np.float32)
    wb = pack_q8_0(w)
    aq = rng.integers(-127, 128, K).astype(np.int8)
    got = O.block_dots(wb[0], aq)
    qw = wb.reshape(-1, Q8_0_BYTES)[:, 2:].view(np.int8).astype(np.int64)
    ref = (qw * aq.reshape(-1, 32).astype(np.int64)).sum(axis=1)
    np.testing.assert_array_equal(got, ref)
    # extreme block: 32 * 127 * 127 (and the negative) are exact
    wmax = np.full((1, 64), 1.0, np.float32)
    wmax[0, 32:] = -1.0
    got = O.block_dots(pack_q8_0(wmax)[0], np.full(64, 127, np.int8))
    assert got.tolist() == [32 * 127 * 127, -32 * 127 * 127]


def test_block_dots_csr_integer_brute_force():
    """Every CSR entry x every weight row of its expert, one block, against pure-Python integer
    sums (token rows selected through expTokI, and activation rows in entry order)."""
    rng = np.random.default_rng(11)
    E, rows, K, N, k = 3, 5, 96, 7, 2
    W = pack_q8_0(rng.standard_normal((E * rows, K)).astype(np.float32)).reshape(E, rows, -1)
    qw = W.reshape(E, rows, K // 32, Q8_0_BYTES)[..., 2:].view(np.int8)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    es, ti, tk = O.bucket(idx, E)
    xq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    hq = rng.integers(-127, 128, (N * k, K)).astype(np.int8)
    for block in range(K // 32):
        got_x = O.block_dots_csr(W, xq, es, ti, block)
        got_h = O.block_dots_csr(W, hq, es, None, block)
        for j in range(N * k):
            e = max(i for i in range(E) if es[i] <= j)
            for r in range(rows):
                wq = [int(v) for v in qw[e, r, block]]
                xs = [int(v) for v in xq[ti[j], 32 * block:32 * block + 32]]
                hs = [int(v) for v in hq[j, 32 * block:32 * block + 32]]
                assert got_x[j, r] == sum(a * b for a, b in zip(wq, xs))
                assert got_h[j, r] == sum(a * b for a, b in zip(wq, hs))


def _hand_q4_k_block() -> np.ndarray:
    """One Q4_K super-block written byte by byte: d = 1, dmin = 0.5, sc = 1..7, 63 and
    m = 0..6, 40 (bytes below), every quant byte 0x2F (even sub-blocks q = 15, odd q = 2)."""
    blk = np.zeros(Q4_K_BYTES, np.uint8)
    blk[0:2] = [0x00, 0x3C]                 # fp16 1.0
    blk[2:4] = [0x00, 0x38]                 # fp16 0.5
    blk[4:8] = [1, 2, 3, 4 | (3 << 6)]      # sc_0..3, top bits of sc_7 = 63 >> 4 = 3
    blk[8:12] = [0, 1, 2, 3 | (2 << 6)]     # m_0..3, top bits of m_7 = 40 >> 4 = 2
    blk[12:16] = [5 | (4 << 4), 6 | (5 << 4), 7 | (6 << 4), 15 | (8 << 4)]  # low bits of sc_4..7 / m_4..7
    blk[16:] = 0x2F
    return blk


def test_q4_k_hand_block_decodes_to_the_format_values():
    """d*sc_j*q - dmin*m_j on the hand-written block, worked out by hand: sub-block 0: 1*1*15 - 0 = 15;
    1: 2*2 - 0.5 = 3.5; 2: 3*15 - 1 = 44; 3: 4*2 - 1.5 = 6.5; 4: 5*15 - 2 = 73; 5: 6*2 - 2.5 = 9.5;
    6: 7*15 - 3 = 102; 7: 63*2 - 20 = 106."""
    want = [15.0, 3.5, 44.0, 6.5, 73.0, 9.5, 102.0, 106.0]
    got = O.q4_k_dequant(_hand_q4_k_block(), QK_K).reshape(8, 32)
    for j in range(8):
        assert np.all(got[j] == want[j]), (j, got[j][:4])
    assert np.all(dequant_q4_k(_hand_q4_k_block()[None])[0].reshape(8, 32) == np.array(want)[:, None])


def test_q4_k_dequant_matches_format_definition():
    rng = np.random.default_rng(40)
    rows = pack_q4_k((rng.standard_normal((6, 512)) * 0.02).astype(np.float32))
    ref = dequant_q4_k(rows).astype(np.float32)
    got = np.stack([O.q4_k_dequant(r, 512) for r in rows])
    np.testing.assert_array_equal(got, ref)


def test_q4_k_block_dots_integer_brute_force():
    rng = np.random.default_rng(41)
    rows = pack_q4_k((rng.standard_normal((1, 512)) * 0.02).astype(np.float32))
    aq = rng.integers(-127, 128, 512).astype(np.int8)
    qs = rows[0].reshape(-1, Q4_K_BYTES)[:, 16:].astype(np.int64).reshape(-1, 4, 32)
    q = np.stack([qs & 15, qs >> 4], axis=2).reshape(-1, 32)  # sub-blocks in order
    ref = (q * aq.reshape(-1, 32).astype(np.int64)).sum(axis=1)
    np.testing.assert_array_equal(O.block_dots_q4_k(rows[0], aq), ref)
    # extreme block: 32 * 15 * 127 is exact
    hand = _hand_q4_k_block()
    assert O.block_dots_q4_k(hand, np.full(256, 127, np.int8))[0] == 32 * 15 * 127


@pytest.fixture(scope="module")
def small_expert_q4_k():
    rng = np.random.default_rng(42)
    D, F = 256, 256
    Wg = pack_q4_k((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wu = pack_q4_k((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wd = pack_q4_k((rng.standard_normal((D, F)) * 0.02).astype(np.float32))
    x = rng.standard_normal(D).astype(np.float32)
    xq, xd16, _ = O.quantize_q8_1(x)
    return D, F, Wg, Wu, Wd, xq, xd16


def test_q4_k_expert_matches_dequantised_matmul(small_expert_q4_k):
    """Q4_K gate/up and down against numpy float64 matmuls of the dequantised operands: the min
    term (dmin*m_j times the activation block's code sum) is part of the same number."""
    D, F, Wg, Wu, Wd, xq, xd16 = small_expert_q4_k
    h, hq, hd16, g, u = O.expert_gate_up(Wg, Wu, D, F, xq, xd16, fmt="q4_k")
    xdq = dequant_q8(xq, xd16)
    for got, W in ((g, Wg), (u, Wu)):
        Wdq = dequant_q4_k(W)
        assert np.all(np.abs(got - Wdq @ xdq) <= 1e-12 * (np.abs(Wdq) @ np.abs(xdq)))
    y = O.expert_down(Wd, D, F, hq, hd16, fmt="q4_k")
    Wdd = dequant_q4_k(Wd)
    hdq = dequant_q8(hq, hd16)
    assert np.all(np.abs(y - Wdd @ hdq) <= 1e-12 * (np.abs(Wdd) @ np.abs(hdq)))
    # the same bytes read as the wrong format do not give the same numbers
    assert not np.allclose(g, dequant_q4_k(Wg)[:, ::-1] @ xdq, rtol=1e-3)


def test_q4_k_single_expert_layer_is_dense_swiglu():
    rng = np.random.default_rng(43)
    N, D, F = 8, 256, 256
    hidden = rng.standard_normal((N, D)).astype(np.float32)
    routerW = (rng.standard_normal((1, D)) / np.sqrt(D)).astype(np.float32)
    pk = lambda r, c: pack_q4_k((rng.standard_normal((r, c)) * 0.02).astype(np.float32))  # noqa: E731
    inp = dict(hidden=hidden, routerW=routerW, gate=pk(F, D)[None], up=pk(F, D)[None], down=pk(D, F)[None],
               wfmt="q4_k")
    r = O.moe_ffn_inputs(inp, 1, True)
    assert np.all(r["topk_w"] == 1.0)
    xdq = dequant_q8(r["x_q"], r["x_d16"])
    g = xdq @ dequant_q4_k(inp["gate"][0]).T
    u = xdq @ dequant_q4_k(inp["up"][0]).T
    ref = (g / (1 + np.exp(-g)) * u) @ dequant_q4_k(inp["down"][0]).T
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-2
    ref_exact = dequant_q8(r["h_q"], r["h_d16"]) @ dequant_q4_k(inp["down"][0]).T
    np.testing.assert_allclose(r["out"][r["expTokI"]], ref_exact.astype(np.float32), rtol=1e-6, atol=1e-9)


_Q3_RAW = [0, 5, 9, 13, 17, 21, 25, 29, 34, 38, 42, 46, 50, 54, 58, 63]  # 6-bit scale fields; s_j = raw - 32


def _hand_q3_k_block() -> np.ndarray:
    """One Q3_K super-block written byte by byte: d = 0.5, scale fields _Q3_RAW (s_0 = -32, s_15 = 31),
    value i coded as q_i = (i % 8) - 4, so every quant byte repeats one 2-bit field and every
    hmask byte is all ones (l % 8 >= 4) or all zeros."""
    blk = np.zeros(Q3_K_BYTES, np.uint8)
    for l in range(32):
        blk[l] = 0xFF if l % 8 >= 4 else 0x00
        blk[32 + l] = blk[64 + l] = ((l % 8) & 3) * 0x55
    for j in range(8):
        blk[96 + j] = (_Q3_RAW[j] & 15) | ((_Q3_RAW[j + 8] & 15) << 4)
    for m in range(4):
        blk[104 + m] = sum((_Q3_RAW[4 * g + m] >> 4) << (2 * g) for g in range(4))
    blk[108:110] = [0x00, 0x38]  # fp16 0.5
    return blk


def test_q3_k_hand_block_decodes_to_the_format_values():
    """d*s_j*q on the hand-written block, by hand: value 0 = 0.5*(-32)*(-4) = 64; value 7 = 0.5*(-32)*3 = -48;
    value 16 = 0.5*(-27)*(-4) = 54; value 255 = 0.5*31*3 = 46.5; in general 0.5*(raw_(i/16) - 32)*((i % 8) - 4)."""
    got = O.q3_k_dequant(_hand_q3_k_block(), QK_K)
    assert (got[0], got[7], got[16], got[255]) == (64.0, -48.0, 54.0, 46.5)
    want = np.array([0.5 * (_Q3_RAW[i // 16] - 32) * ((i % 8) - 4) for i in range(QK_K)])
    assert np.all(got == want)
    assert np.all(dequant_q3_k(_hand_q3_k_block()[None])[0] == want)


def test_q3_k_dequant_matches_format_definition():
    rng = np.random.default_rng(50)
    rows = pack_q3_k((rng.standard_normal((6, 512)) * 0.02).astype(np.float32))
    ref = dequant_q3_k(rows).astype(np.float32)
    got = np.stack([O.q3_k_dequant(r, 512) for r in rows])
    np.testing.assert_array_equal(got, ref)
    # the generator reaches both ends of the code range, both signs of scale and s = -32 with q = -4
    _, sc, q = q3_k_fields(rows)
    assert q.min() == -4 and q.max() == 3 and (sc < 0).any() and (sc > 0).any()
    assert ((np.repeat(sc, 16, axis=-1) == -32) & (q == -4)).any()


def test_q3_k_block_dots_integer_brute_force():
    rng = np.random.default_rng(51)
    rows = pack_q3_k((rng.standard_normal((1, 512)) * 0.02).astype(np.float32))
    aq = rng.integers(-127, 128, 512).astype(np.int8)
    # integer codes s_j * q_i from the field-by-field decoder
    _, sc, q = q3_k_fields(rows)
    codes = (np.repeat(sc, 16, axis=-1) * q).reshape(-1, 32)
    ref = (codes * aq.reshape(-1, 32).astype(np.int64)).sum(axis=1)
    np.testing.assert_array_equal(O.block_dots_q3_k(rows[0], aq), ref)
    # hand block against all-127 codes: block 0 = 127 * (-32 * -8 + -27 * -8) = 59944
    assert O.block_dots_q3_k(_hand_q3_k_block(), np.full(256, 127, np.int8))[0] == 127 * 8 * (32 + 27)
    # extreme block: every q = -4 with s = -32 gives 2 * 16 * 128 * 127 per 32-wide block, exact
    ext = np.zeros(Q3_K_BYTES, np.uint8)
    ext[108:110] = [0x00, 0x3C]
    got = O.block_dots_q3_k(ext, np.full(256, 127, np.int8))
    assert got.tolist() == [32 * 128 * 127] * 8


@pytest.fixture(scope="module")
def small_expert_q3_k():
    rng = np.random.default_rng(52)
    D, F = 256, 512
    Wg = pack_q3_k((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wu = pack_q3_k((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wd = pack_q3_k((rng.standard_normal((D, F)) * 0.02).astype(np.float32))
    x = rng.standard_normal(D).astype(np.float32)
    xq, xd16, _ = O.quantize_q8_1(x)
    return D, F, Wg, Wu, Wd, xq, xd16


def test_q3_k_expert_matches_dequantised_matmul(small_expert_q3_k):
    """Q3_K gate/up and down against numpy float64 matmuls of the dequantised operands."""
    D, F, Wg, Wu, Wd, xq, xd16 = small_expert_q3_k
    h, hq, hd16, g, u = O.expert_gate_up(Wg, Wu, D, F, xq, xd16, fmt="q3_k")
    xdq = dequant_q8(xq, xd16)
    for got, W in ((g, Wg), (u, Wu)):
        Wdq = dequant_q3_k(W)
        assert np.all(np.abs(got - Wdq @ xdq) <= 1e-12 * (np.abs(Wdq) @ np.abs(xdq)))
    y = O.expert_down(Wd, D, F, hq, hd16, fmt="q3_k")
    Wdd = dequant_q3_k(Wd)
    hdq = dequant_q8(hq, hd16)
    assert np.all(np.abs(y - Wdd @ hdq) <= 1e-12 * (np.abs(Wdd) @ np.abs(hdq)))
    # an unknown format is refused, not guessed
    with pytest.raises(ValueError):
        O.expert_gate_up(Wg, Wu, D, F, xq, xd16, fmt="q5_k")


def test_q3_k_single_expert_layer_is_dense_swiglu():
    rng = np.random.default_rng(53)
    N, D, F = 8, 256, 256
    hidden = rng.standard_normal((N, D)).astype(np.float32)
    routerW = (rng.standard_normal((1, D)) / np.sqrt(D)).astype(np.float32)
    pk = lambda r, c: pack_q3_k((rng.standard_normal((r, c)) * 0.02).astype(np.float32))  # noqa: E731
    inp = dict(hidden=hidden, routerW=routerW, gate=pk(F, D)[None], up=pk(F, D)[None], down=pk(D, F)[None],
               wfmt="q3_k")
    r = O.moe_ffn_inputs(inp, 1, True)
    assert np.all(r["topk_w"] == 1.0)
    xdq = dequant_q8(r["x_q"], r["x_d16"])
    g = xdq @ dequant_q3_k(inp["gate"][0]).T
    u = xdq @ dequant_q3_k(inp["up"][0]).T
    ref = (g / (1 + np.exp(-g)) * u) @ dequant_q3_k(inp["down"][0]).T
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-2
    ref_exact = dequant_q8(r["h_q"], r["h_d16"]) @ dequant_q3_k(inp["down"][0]).T
    np.testing.assert_allclose(r["out"][r["expTokI"]], ref_exact.astype(np.float32), rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------- expert FFN -----
@pytest.fixture(scope="module")
def small_expert():
    rng = np.random.default_rng(8)
    D, F = 128, 96
    Wg = pack_q8_0((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wu = pack_q8_0((rng.standard_normal((F, D)) * 0.02).astype(np.float32))
    Wd = pack_q8_0((rng.standard_normal((D, F)) * 0.02).astype(np.float32))
    x = rng.standard_normal(D).astype(np.float32)
    xq, xd16, _ = O.quantize_q8_1(x)
    return D, F, Wg, Wu, Wd, xq, xd16


def test_gate_up_matches_dequantised_matmul(small_expert):
    """g = W_g x and u = W_u x on dequantised operands (numpy float64 matmul): the per-block
    sum of fp16(dw) * fp16(dx) * isum is the same number up to double rounding."""
    D, F, Wg, Wu, Wd, xq, xd16 = small_expert
    h, hq, hd16, g, u = O.expert_gate_up(Wg, Wu, D, F, xq, xd16)
    xdq = dequant_q8(xq, xd16)
    g_ref = dequant_q8_0(Wg) @ xdq
    u_ref = dequant_q8_0(Wu) @ xdq
    scale = np.abs(dequant_q8_0(Wg)) @ np.abs(xdq)
    assert np.all(np.abs(g - g_ref) <= 1e-13 * scale)
    assert np.all(np.abs(u - dequant_q8_0(Wu) @ xdq) <= 1e-13 * (np.abs(dequant_q8_0(Wu)) @ np.abs(xdq)))
    # SwiGLU: h = SiLU(g) * u, SiLU(z) = z * sigmoid(z) (textbook form), rounded to fp32
    h_ref = g_ref * (1.0 / (1.0 + np.exp(-g_ref))) * u_ref
    np.testing.assert_allclose(h, h_ref, rtol=2 * F32_EPS, atol=1e-12)
    # gate and up are not interchangeable (catches a swapped operand)
    h_swapped = u_ref * (1.0 / (1.0 + np.exp(-u_ref))) * g_ref
    assert not np.allclose(h, h_swapped, rtol=1e-3)
    # h is requantised with the Q8_1 rule
    q2, d2, _ = O.quantize_q8_1(h)
    np.testing.assert_array_equal(hq, q2)
    np.testing.assert_array_equal(hd16, d2)


def test_down_matches_dequantised_matmul(small_expert):
    D, F, Wg, Wu, Wd, xq, xd16 = small_expert
    _, hq, hd16, _, _ = O.expert_gate_up(Wg, Wu, D, F, xq, xd16)
    y = O.expert_down(Wd, D, F, hq, hd16)
    Wdd = dequant_q8_0(Wd)
    hdq = dequant_q8(hq, hd16)
    y_ref = Wdd @ hdq
    assert np.all(np.abs(y - y_ref) <= 1e-13 * (np.abs(Wdd) @ np.abs(hdq)))
    # linear in h: doubling every h scale doubles y exactly (power of two)
    hd2 = (hd16.view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.expert_down(Wd, D, F, hq, hd2), 2 * y)


def _layer(rng, N, D, E, k, F, norm, Fs=0, zero_hidden=False):
    hidden = np.zeros((N, D), np.float32) if zero_hidden else rng.standard_normal((N, D)).astype(np.float32)
    routerW = (rng.standard_normal((E, D)) / np.sqrt(D)).astype(np.float32)
    gate = np.stack([pack_q8_0((rng.standard_normal((F, D)) * 0.02).astype(np.float32)) for _ in range(E)])
    up = np.stack([pack_q8_0((rng.standard_normal((F, D)) * 0.02).astype(np.float32)) for _ in range(E)])
    down = np.stack([pack_q8_0((rng.standard_normal((D, F)) * 0.02).astype(np.float32)) for _ in range(E)])
    extra = {}
    if Fs:
        extra = dict(shexp_gate=(rng.standard_normal(D) / np.sqrt(D)).astype(np.float32),
                     sh_gate=pack_q8_0((rng.standard_normal((Fs, D)) * 0.02).astype(np.float32)),
                     sh_up=pack_q8_0((rng.standard_normal((Fs, D)) * 0.02).astype(np.float32)),
                     sh_down=pack_q8_0((rng.standard_normal((D, Fs)) * 0.02).astype(np.float32)))
    return dict(hidden=hidden, routerW=routerW, gate=gate, up=up, down=down, **extra)


def test_single_expert_layer_is_dense_swiglu():
    """E = 1, k = 1, norm on: w = 1, so the layer is one dense SwiGLU FFN.  The textbook FFN on
    dequantised weights (numpy float64, without requantising h) agrees to the Q8_1 error of h."""
    rng = np.random.default_rng(9)
    N, D, F = 12, 128, 64
    inp = _layer(rng, N, D, 1, 1, F, True)
    r = O.moe_ffn_inputs(inp, 1, True)
    assert np.all(r["topk_w"] == 1.0) and np.all(r["topk_idx"] == 0)
    xdq = dequant_q8(r["x_q"], r["x_d16"])
    g = xdq @ dequant_q8_0(inp["gate"][0]).T
    u = xdq @ dequant_q8_0(inp["up"][0]).T
    h = g / (1 + np.exp(-g)) * u
    ref = h @ dequant_q8_0(inp["down"][0]).T
    rel = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert rel < 1e-2  # Q8_1 requantisation of h: ~0.5/127 per element
    # exact down step on the oracle's own requantised h
    ref_exact = dequant_q8(r["h_q"], r["h_d16"]) @ dequant_q8_0(inp["down"][0]).T
    order = r["expTokI"]  # segment order -> token order
    np.testing.assert_allclose(r["out"][order], ref_exact.astype(np.float32), rtol=1e-6, atol=1e-9)


def test_zero_hidden_gives_zero_output():
    rng = np.random.default_rng(10)
    inp = _layer(rng, 4, 64, 4, 2, 32, False, Fs=32, zero_hidden=True)
    r = O.moe_ffn_inputs(inp, 2, False)
    assert np.all(r["out"] == 0.0)
    assert np.all(r["shexp_scale"] == 0.5)  # g = 0 -> sigmoid = 1/2
    np.testing.assert_allclose(r["topk_w"], 1.0 / 4, rtol=2 * F32_EPS)


def test_grouped_partials_land_in_token_slot_rows():
    """partials[t*k + s] is expert idx[t,s]'s unweighted output for token t (#129 'Scope'),
    recomputed row by row from the pinned single-row gate/up and down steps."""
    rng = np.random.default_rng(11)
    N, D, E, k, F = 10, 64, 6, 3, 32
    inp = _layer(rng, N, D, E, k, F, False)
    r = O.moe_ffn_inputs(inp, k, False)
    for t in range(N):
        for s in range(k):
            e = int(r["topk_idx"][t, s])
            _, hq, hd16, _, _ = O.expert_gate_up(inp["gate"][e], inp["up"][e], D, F, r["x_q"][t], r["x_d16"][t])
            y = O.expert_down(inp["down"][e], D, F, hq, hd16)
            np.testing.assert_array_equal(r["partials"][t * k + s], y.astype(np.float32))


def test_all_experts_selected():
    """k = E: every token lands in every bucket; with norm on the weights are the softmax."""
    rng = np.random.default_rng(12)
    N, D, E, F = 7, 64, 4, 32
    inp = _layer(rng, N, D, E, E, F, True)
    r = O.moe_ffn_inputs(inp, E, True)
    np.testing.assert_array_equal(np.diff(r["expStart"]), np.full(E, N))
    np.testing.assert_allclose(np.sort(r["topk_w"], axis=1), np.sort(r["probs"], axis=1), rtol=4 * F32_EPS)


def test_shared_expert_scaled_by_sigmoid_gate():
    """S = sigmoid(g) * y_shared, added after the routed slots (#129 'Scope': AddInPlace(shared))."""
    rng = np.random.default_rng(13)
    N, D, E, k, F, Fs = 6, 64, 4, 2, 32, 64
    inp = _layer(rng, N, D, E, k, F, True, Fs=Fs)
    r = O.moe_ffn_inputs(inp, k, True)
    g_ref = inp["hidden"].astype(np.float64) @ inp["shexp_gate"].astype(np.float64)
    np.testing.assert_allclose(r["shexp_scale"], 1 / (1 + np.exp(-g_ref)), rtol=1e-6)
    for t in range(N):
        _, hq, hd16, _, _ = O.expert_gate_up(inp["sh_gate"], inp["sh_up"], D, Fs, r["x_q"][t], r["x_d16"][t])
        y = O.expert_down(inp["sh_down"], D, Fs, hq, hd16)
        np.testing.assert_allclose(r["shared_out"][t], float(r["shexp_scale"][t]) * y, rtol=1e-6, atol=1e-12)
    no_shared = O.combine(r["partials"], r["topk_w"])
    np.testing.assert_array_equal(r["out"], (no_shared + r["shared_out"]).astype(np.float32))


# -------------------------------------------------------------- combine ----
def test_combine_single_slot_unit_weight_is_identity():
    rng = np.random.default_rng(14)
    p = rng.standard_normal((5, 40)).astype(np.float32)
    out = O.combine(p, np.ones((5, 1), np.float32))
    np.testing.assert_array_equal(out, p)


def test_combine_slot_order_is_load_bearing():
    """k = 0..na-1 order (#129 'Scope'): [2^24, 1, 1] sums to 2^24 in slot order (each +1 ties to
    even), while the reversed order would give 2^24 + 2."""
    p = np.array([[2.0 ** 24], [1.0], [1.0]], np.float32)
    w = np.ones((1, 3), np.float32)
    assert float(O.combine(p, w)[0, 0]) == 2.0 ** 24
    assert float(O.combine(p[::-1].copy(), w)[0, 0]) == 2.0 ** 24 + 2


def test_combine_uses_fused_multiply_add():
    """AddScaledInPlace read as one fma: (1+2^-12)^2 - 1 = 2^-11 + 2^-24 exactly; a separate
    multiply would round the product to 1 + 2^-11 first (a tie, to even) and give 2^-11."""
    a = 1.0 + 2.0 ** -12
    p = np.array([[-1.0], [a]], np.float32)
    w = np.array([[1.0, a]], np.float32)
    assert float(O.combine(p, w)[0, 0]) == 2.0 ** -11 + 2.0 ** -24


def test_combine_adds_shared_after_slots():
    """Clear -> slots -> AddInPlace(shared): 1 + 2^24 ties to even (2^24), then + 1 ties again,
    giving 2^24; adding the shared row first would give 1 + 1 + 2^24 = 2^24 + 2."""
    p = np.array([[1.0], [2.0 ** 24]], np.float32)
    w = np.ones((1, 2), np.float32)
    S = np.array([[1.0]], np.float32)
    assert float(O.combine(p, w, S)[0, 0]) == 2.0 ** 24


def test_combine_residual_zero_is_the_plain_combine():
    rng = np.random.default_rng(15)
    p = rng.standard_normal((3 * 4, 24)).astype(np.float32)
    w = rng.random((3, 4)).astype(np.float32)
    S = rng.standard_normal((3, 24)).astype(np.float32)
    np.testing.assert_array_equal(O.combine(p, w, S, R=np.zeros((3, 24), np.float32)), O.combine(p, w, S))


def test_combine_residual_single_slot_is_one_fp32_add():
    """k = 1, w = 1, no shared row: out = partial + residual, one IEEE fp32 addition."""
    rng = np.random.default_rng(16)
    p = (rng.standard_normal((6, 32)) * 10.0 ** rng.integers(-6, 6, (6, 1))).astype(np.float32)
    R = (rng.standard_normal((6, 32)) * 10.0 ** rng.integers(-6, 6, (6, 1))).astype(np.float32)
    np.testing.assert_array_equal(O.combine(p, np.ones((6, 1), np.float32), R=R), p + R)


def test_combine_residual_added_after_the_shared_row():
    """(routed + shared) + resid: 1 + 2^-24 ties to even (1), then + 2^-23 is exact; adding the
    residual first, or the two rows together first, ties the other way and gives 1 + 2^-22."""
    p = np.array([[1.0]], np.float32)
    w = np.ones((1, 1), np.float32)
    S = np.array([[2.0 ** -24]], np.float32)
    R = np.array([[2.0 ** -23]], np.float32)
    assert float(O.combine(p, w, S, R)[0, 0]) == 1.0 + 2.0 ** -23


def _single_slot(rows):
    """k = 1, w = 1, zero residual, no shared row: the combine's out is `rows` itself."""
    rows = np.asarray(rows, np.float32)
    return rows, np.ones((rows.shape[0], 1), np.float32), np.zeros_like(rows)


def test_rmsnorm_constant_rows_give_gamma():
    """A row of one value c (any sign, any size) has RMS |c|: with eps = 0 every normed value is
    sign(c) * gamma[c], exactly (c^2 and its square root are exact in double)."""
    rng = np.random.default_rng(17)
    D = 40
    rows = np.array([[3.0] * D, [-0.375] * D, [2.0 ** -60] * D, [1.5e30] * D], np.float32)
    gamma = (rng.standard_normal(D) * 3.0).astype(np.float32)
    p, w, R = _single_slot(rows)
    out, normed = O.combine_residual_rmsnorm(p, w, None, R, gamma, 0.0)
    np.testing.assert_array_equal(out, rows)
    np.testing.assert_array_equal(normed, np.sign(rows) * gamma[None, :])


def test_rmsnorm_epsilon_closed_form():
    """A constant row c with eps = 3 c^2: c / sqrt(c^2 + 3 c^2) = 1/2 exactly."""
    for c in (2.0, 0.25, -6.0):
        p, w, R = _single_slot(np.full((1, 24), c))
        _, normed = O.combine_residual_rmsnorm(p, w, None, R, np.ones(24, np.float32), 3.0 * c * c)
        np.testing.assert_array_equal(normed, np.full((1, 24), 0.5 * np.sign(c), np.float32))


def test_rmsnorm_rows_have_unit_rms():
    """gamma = 1, eps = 0: every normed row has mean square 1 (to fp32 rounding), whatever its scale."""
    rng = np.random.default_rng(18)
    rows = (rng.standard_normal((8, 256)) * 10.0 ** rng.integers(-8, 8, (8, 1))).astype(np.float32)
    p, w, R = _single_slot(rows)
    _, normed = O.combine_residual_rmsnorm(p, w, None, R, np.ones(256, np.float32), 0.0)
    ms = (normed.astype(np.float64) ** 2).mean(axis=1)
    np.testing.assert_allclose(ms, 1.0, rtol=2e-7)


def test_rmsnorm_power_of_two_scale_invariance_and_gamma_linearity():
    """With eps = 0, scaling a row by 2^j changes nothing (every step scales exactly), and doubling
    gamma doubles every normed value exactly."""
    rng = np.random.default_rng(19)
    rows = rng.standard_normal((5, 64)).astype(np.float32)
    gamma = rng.standard_normal(64).astype(np.float32)
    p, w, R = _single_slot(rows)
    _, n1 = O.combine_residual_rmsnorm(p, w, None, R, gamma, 0.0)
    p8, _, R8 = _single_slot(rows * np.float32(8.0))
    _, n8 = O.combine_residual_rmsnorm(p8, w, None, R8, gamma, 0.0)
    np.testing.assert_array_equal(n1, n8)
    _, n2 = O.combine_residual_rmsnorm(p, w, None, R, gamma * np.float32(2.0), 0.0)
    np.testing.assert_array_equal(n2, n1 * np.float32(2.0))


def test_rmsnorm_normalises_the_residual_combine_output():
    """out is the combine with residual bit for bit, and the norm is taken of out (not of the
    routed sum alone): each normed row is out * r * gamma with one r per row."""
    rng = np.random.default_rng(20)
    N, k, D = 4, 3, 48
    p = rng.standard_normal((N * k, D)).astype(np.float32)
    w = rng.random((N, k)).astype(np.float32)
    S = rng.standard_normal((N, D)).astype(np.float32)
    R = (rng.standard_normal((N, D)) * 4.0).astype(np.float32)
    gamma = (rng.random(D) + 0.5).astype(np.float32)
    out, normed = O.combine_residual_rmsnorm(p, w, S, R, gamma, 1e-6)
    np.testing.assert_array_equal(out, O.combine(p, w, S, R))
    ratio = normed.astype(np.float64) / (out.astype(np.float64) * gamma.astype(np.float64))
    want = 1.0 / np.sqrt((out.astype(np.float64) ** 2).mean(axis=1) + 1e-6)
    np.testing.assert_allclose(ratio, np.broadcast_to(want[:, None], ratio.shape), rtol=2e-7)


def test_rmsnorm_alone_constant_rows():
    """The norm of rows alone (no routed slot): a constant row c gives sign(c) * gamma exactly."""
    gamma = np.linspace(-2.0, 3.0, 16).astype(np.float32)
    x = np.array([[5.0] * 16, [-0.125] * 16], np.float32)
    np.testing.assert_array_equal(O.rmsnorm(x, gamma, 0.0), np.sign(x) * gamma[None, :])


# ---------------------------------------------------- regression fixture ---
@pytest.mark.parametrize("name,fixture", [("tiny", "tiny_layer.json"), ("tiny_q4k", "tiny_q4k_layer.json"),
                                          ("tiny_q3k", "tiny_q3k_layer.json")])
def test_tiny_layer_matches_recorded_fixture(name, fixture):
    """tests/golden/<fixture> (written by tests/golden/make_golden.py from this oracle):
    routing, CSR and quant codes exactly; floats to 1e-6 relative."""
    import json
    import os

    from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, make_inputs

    with open(os.path.join(os.path.dirname(__file__), "golden", fixture)) as f:
        fx = json.load(f)
    wl = WORKLOADS[name]
    assert fx["workload"] == wl.describe()
    r = O.moe_ffn_inputs(make_inputs(wl), wl.top_k, wl.norm_topk_prob)
    assert r["topk_idx"].tolist() == fx["topk_idx"]
    assert r["expStart"].tolist() == fx["expStart"]
    assert int(r["x_q"].astype(np.int64).sum()) == fx["x_q_int_sum"]
    assert int(np.abs(r["x_q"].astype(np.int64)).sum()) == fx["x_q_abs_sum"]
    assert r["x_d16"][0, :8].tolist() == fx["x_d16_first8"]
    assert abs(int(np.abs(r["h_q"].astype(np.int64)).sum()) - fx["h_q_abs_sum"]) <= 2
    np.testing.assert_allclose(r["topk_w"][:8], np.array(fx["topk_w_first8"]), rtol=1e-6)
    np.testing.assert_allclose(r["out"][0, :16], np.array(fx["out_row0_first16"]), rtol=1e-5, atol=1e-8)
    assert abs(float(np.linalg.norm(r["out"].astype(np.float64))) - fx["out_l2"]) <= 1e-6 * fx["out_l2"]
