"""Pins that tie the CPU oracle to what the pages and mathematics fix.

None of these re-types the oracle's own formula: each checks it against a
hand-derived value printed on (or derived from) the pages, a closed form,
an invariant, a textbook routine written independently here (float64
numpy attention), or brute force on tiny inputs.  The cases are chosen so
that a plausible slip in the oracle (a dropped scale, a transposed
operand, a wrong causal offset, a sign error in the smooth_k bias, a wrong
LSE base, a wrong page index) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def textbook_attention(q, k, v, sm_scale, causal=False, offset=0):
    """Plain float64 softmax(q k^T * sm_scale) v with natural-log LSE."""
    s = (q.astype(np.float64) @ k.astype(np.float64).T) * sm_scale
    if causal:
        i = np.arange(q.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= i + offset, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        # a row with every key masked has m = -inf: NaN output, -inf LSE
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        return (p / l) @ v.astype(np.float64), (m + np.log(l))[:, 0]


def integer_rows(rng, n, d, amax=127):
    """Integer rows whose absolute maximum is exactly ``amax`` (so s = amax/127)."""
    x = rng.integers(-amax, amax + 1, size=(n, d)).astype(np.float32)
    cols = rng.integers(0, d, size=n)
    sign = rng.choice([-1.0, 1.0], size=n)
    x[np.arange(n), cols] = sign * amax
    return x


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------

def _read_ties():
    rows = []
    for line in open(os.path.join(GOLDEN, "quant_ties.txt")):
        if line.startswith("#") or not line.strip():
            continue
        amax, xs, qs = [part.split() for part in line.split("|")]
        rows.append((float(amax[0]), np.array(xs, np.float32), np.array(qs, np.int64)))
    return rows


@pytest.mark.parametrize("case", range(4))
def test_quant_golden_ties(case):
    amax, xs, expect = _read_ties()[case]
    # every value is fp16-representable: the fp16 -> fp32 path is exact
    assert np.all(xs.astype(np.float16).astype(np.float32) == xs)
    q, s, _ = oracle.quant_int8(xs[None, None, :])
    assert s[0, 0] == np.float32(amax) / np.float32(127.0)
    assert q[0, 0].tolist() == expect.tolist()


def test_quant_bounds_and_error():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 37, 64)).astype(np.float16).astype(np.float32)
    for block in (1, 8, 16, 64):
        q, s, _ = oracle.quant_int8(x, block_tokens=block)
        assert q.dtype == np.int8 and np.abs(q.astype(np.int32)).max() <= 127
        G = (37 + block - 1) // block
        assert s.shape == (3, G)
        for b in range(3):
            for g in range(G):
                grp = x[b, g * block:(g + 1) * block]
                amax = np.abs(grp).max()
                assert s[b, g] == np.float32(amax) / np.float32(127)
                qq = q[b, g * block:(g + 1) * block].astype(np.float64)
                # reconstruction error at most half a step (plus fp32 slack)
                err = np.abs(qq * s[b, g] - grp)
                assert err.max() <= 0.5 * s[b, g] * (1 + 1e-5)
                # the element that sets amax lands on +-127
                idx = np.unravel_index(np.abs(grp).argmax(), grp.shape)
                assert abs(int(q[b, g * block + idx[0], idx[1]])) == 127
                # sign is preserved wherever the code is non-zero
                nz = qq != 0
                assert np.all(np.sign(qq[nz]) == np.sign(grp[nz]))


def test_quant_zero_group():
    x = np.zeros((1, 4, 16), np.float32)
    x[0, 2:] = 1.0
    q, s, _ = oracle.quant_int8(x, block_tokens=2)
    assert s[0, 0] == 0.0 and np.all(q[0, :2] == 0)
    assert s[0, 1] == np.float32(1) / np.float32(127) and np.all(q[0, 2:] == 127)


def test_quant_per_block_tail_group_closed_form():
    """S = 130 in 64-token groups: rows 0-127 hold even integers with amax
    254 (scale exactly 2, codes x / 2), the 2-row tail group integers with
    amax 127 (scale 1, codes x): a group boundary or tail taken wrong moves
    a scale or a code."""
    rng = np.random.default_rng(7)
    head = 2.0 * integer_rows(rng, 128, 32)            # every row reaches +-254
    tail = integer_rows(rng, 2, 32)                    # every row reaches +-127
    x = np.concatenate([head, tail])[None].astype(np.float32)
    q, s, _ = oracle.quant_int8(x, block_tokens=64)
    assert s.shape == (1, 3) and s[0].tolist() == [2.0, 2.0, 1.0]
    assert np.array_equal(q[0, :128].astype(np.float32), head / 2.0)
    assert np.array_equal(q[0, 128:].astype(np.float32), tail)


def test_quant_integer_identity():
    rng = np.random.default_rng(2)
    x = integer_rows(rng, 50, 128)
    q, s, _ = oracle.quant_int8(x[None])
    assert np.all(s == 1.0)
    assert np.array_equal(q[0].astype(np.float32), x)


def test_token_mean_closed_forms():
    S, D = 33, 16
    t = np.arange(S, dtype=np.float32)[:, None] * np.ones((1, D), np.float32)
    x = (t * 0.5 + np.arange(D, dtype=np.float32)[None, :])[None]
    mu = oracle.token_mean(x)
    # mean of 0.5*t + c over t = 0..S-1 is 0.25*(S-1) + c
    expect = 0.25 * (S - 1) + np.arange(D, dtype=np.float64)
    assert np.array_equal(mu[0], expect.astype(np.float32))
    const = np.full((2, 7, 4), 3.25, np.float32)
    assert np.all(oracle.token_mean(const) == 3.25)


def test_token_mean_wide_range_is_exact():
    """The mean is an exact sum rounded once: values 40 binades apart
    cancel exactly (a float32 running sum would lose the small terms and
    give 0), and a large offset plus a tiny mean comes back exactly."""
    x = np.array([2.0 ** 20, 2.0 ** -20, -(2.0 ** 20), 2.0 ** -20], np.float32)
    mu = oracle.token_mean(x[None, :, None])
    assert mu[0, 0] == np.float32(2.0 ** -21)
    big = np.array([3.0e4, 2.0 ** -18, -3.0e4, 0.0, 2.0 ** -18, 0.0, 0.0, 0.0], np.float32)
    assert oracle.token_mean(big[None, :, None])[0, 0] == np.float32(2.0 ** -20)


def test_smooth_subtracts_mean_before_quant():
    # K rows = mu + I with I integer (amax 127) and symmetric (+I, -I pairs)
    # so that the token mean is exactly mu and K - mu = I exactly.
    rng = np.random.default_rng(3)
    half = integer_rows(rng, 8, 32)
    I = np.concatenate([half, -half], 0)
    mu = (rng.integers(-64, 64, size=32) * 0.25).astype(np.float32)
    k = (I + mu[None, :]).astype(np.float32)
    q8, s, mu_o = oracle.quant_int8(k[None], smooth=True)
    assert np.array_equal(mu_o[0], mu)
    assert np.all(s == 1.0)
    assert np.array_equal(q8[0].astype(np.float32), I)


# --------------------------------------------------------------------------
# raw INT32 scores
# --------------------------------------------------------------------------

def test_int32_bound_golden():
    line = [l for l in open(os.path.join(GOLDEN, "int32_bound.txt")) if not l.startswith("#")][0]
    D, bound = map(int, line.split())
    ones = np.full((2, D), 127, np.int8)
    neg = np.full((2, D), -127, np.int8)
    assert oracle.qk_int32(ones, ones)[0, 0] == bound
    assert oracle.qk_int32(ones, neg)[0, 0] == -bound
    assert oracle.qk_int32(neg, neg)[1, 1] == bound


def test_qk_brute_force():
    rng = np.random.default_rng(4)
    q = rng.integers(-127, 128, size=(5, 48)).astype(np.int8)
    k = rng.integers(-127, 128, size=(7, 48)).astype(np.int8)
    acc = oracle.qk_int32(q, k)
    for i in range(5):
        for j in range(7):
            assert acc[i, j] == sum(int(q[i, c]) * int(k[j, c]) for c in range(48))


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def test_reduces_to_textbook_attention_when_quant_is_identity():
    rng = np.random.default_rng(5)
    Sq, Sk, D = 24, 40, 64
    q = integer_rows(rng, Sq, D)
    k = integer_rows(rng, Sk, D)
    v = rng.standard_normal((Sk, D))
    qi, sq, _ = oracle.quant_int8(q[None])
    ki, sk, _ = oracle.quant_int8(k[None])
    sm = 1.0 / 4096.0
    for causal in (False, True):
        o, lse = oracle.attend(qi[0], sq[0], ki[0], sk[0], v, sm_scale=sm, causal=causal,
                               causal_offset=Sk - Sq)
        o_ref, lse_ref = textbook_attention(q, k, v, sm, causal, Sk - Sq)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_scales_are_row_and_column_scales():
    # dequantised textbook: Qhat = q*sQ (per row), Khat = k*sK (per column);
    # per-token K scales are distinct powers of two, so any swap of the
    # row/column role or an off-by-one column shift changes the result.
    rng = np.random.default_rng(6)
    Sq, Sk, D = 9, 16, 32
    qi = rng.integers(-127, 128, (Sq, D)).astype(np.int8)
    ki = rng.integers(-127, 128, (Sk, D)).astype(np.int8)
    sq = (2.0 ** -rng.integers(8, 14, Sq)).astype(np.float32)
    sk = (2.0 ** -np.arange(6, 6 + Sk)).astype(np.float32)
    v = rng.standard_normal((Sk, D))
    o, lse = oracle.attend(qi, sq, ki, sk, v, sm_scale=0.125)
    o_ref, lse_ref = textbook_attention(qi * sq[:, None].astype(np.float64),
                                        ki * sk[:, None].astype(np.float64), v, 0.125)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_invariants_uniform_and_constant_values():
    rng = np.random.default_rng(7)
    Sq, Sk, D = 6, 33, 16
    qi = rng.integers(-127, 128, (Sq, D)).astype(np.int8)
    ki = rng.integers(-127, 128, (Sk, D)).astype(np.int8)
    sq = rng.uniform(0.01, 0.02, Sq).astype(np.float32)
    sk = rng.uniform(0.01, 0.02, Sk).astype(np.float32)
    # V == 1 -> O == 1 (softmax rows sum to one)
    o, _ = oracle.attend(qi, sq, ki, sk, np.ones((Sk, D)), sm_scale=0.3)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)
    # K == 0 -> uniform weights: O = mean(V), LSE = ln(Sk)
    v = rng.standard_normal((Sk, D))
    o, lse = oracle.attend(qi, sq, np.zeros((Sk, D), np.int8), sk, v, sm_scale=0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(Sk), rtol=0, atol=1e-14)


def test_causal_equals_truncated_key_set():
    rng = np.random.default_rng(8)
    Sq, Sk, D = 12, 20, 32
    qi = rng.integers(-127, 128, (Sq, D)).astype(np.int8)
    ki = rng.integers(-127, 128, (Sk, D)).astype(np.int8)
    sq = rng.uniform(0.005, 0.02, Sq).astype(np.float32)
    sk = rng.uniform(0.005, 0.02, Sk).astype(np.float32)
    v = rng.standard_normal((Sk, D))
    off = Sk - Sq
    o, lse = oracle.attend(qi, sq, ki, sk, v, sm_scale=0.2, causal=True, causal_offset=off)
    for i in range(Sq):
        n = i + off + 1
        oi, li = oracle.attend(qi[i:i + 1], sq[i:i + 1], ki[:n], sk[:n], v[:n], sm_scale=0.2)
        np.testing.assert_allclose(o[i], oi[0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[i], li[0], rtol=1e-13)
    # a row with no visible key: zero output, -inf LSE
    o2, l2 = oracle.attend(qi[:2], sq[:2], ki, sk, v, sm_scale=0.2, causal=True,
                           causal_offset=-1)
    assert np.all(o2[0] == 0) and l2[0] == -np.inf and np.isfinite(l2[1])


def test_smooth_k_bias_restores_unsmoothed_scores():
    # K = mu + I exactly (see test_smooth_subtracts_mean_before_quant), integer
    # Q with amax 127: with the smooth_k bias the method equals textbook
    # attention on the ORIGINAL K; without it the LSE is off by sm*(q.mu).
    rng = np.random.default_rng(9)
    D, Sq = 32, 10
    half = integer_rows(rng, 12, D)
    I = np.concatenate([half, -half], 0)
    mu = (rng.integers(-64, 64, size=D) * 0.25).astype(np.float32)
    k = (I + mu[None, :]).astype(np.float32)
    q = integer_rows(rng, Sq, D)
    v = rng.standard_normal((k.shape[0], D))
    sm = 1.0 / 8192.0
    ki, sk, mu_o = oracle.quant_int8(k[None, None], smooth=True)
    qi, sq, _ = oracle.quant_int8(q[None, None])
    bias = oracle.row_bias(q[None, None], mu_o)
    np.testing.assert_allclose(bias[0, 0], q.astype(np.float64) @ mu.astype(np.float64),
                               rtol=1e-15)
    o, lse = oracle.attend(qi[0, 0], sq[0, 0], ki[0, 0], sk[0, 0], v, sm_scale=sm,
                           qbias=bias[0, 0], smoothed=np.ones(k.shape[0], np.uint8))
    o_ref, lse_ref = textbook_attention(q, k, v, sm)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)
    o2, lse2 = oracle.attend(qi[0, 0], sq[0, 0], ki[0, 0], sk[0, 0], v, sm_scale=sm)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-11, atol=1e-12)  # row constant cancels in O
    np.testing.assert_allclose(lse2 + sm * bias[0, 0], lse_ref, rtol=1e-12, atol=1e-12)


def test_gqa_mapping():
    rng = np.random.default_rng(10)
    B, Hq, Hkv, S, D = 1, 6, 2, 16, 32
    q = rng.standard_normal((B, Hq, S, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, S, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, S, D))
    qi, sq, _ = oracle.quant_int8(q)
    ki, sk, _ = oracle.quant_int8(k)
    o, _ = oracle.prefill(qi, sq, 1, ki, sk, 1, v, causal=False, sm_scale=0.2, threads=1)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        oh, _ = oracle.attend(qi[0, h], sq[0, h], ki[0, g], sk[0, g], v[0, g], sm_scale=0.2)
        np.testing.assert_array_equal(o[0, h], oh)
        other, _ = oracle.attend(qi[0, h], sq[0, h], ki[0, 1 - g], sk[0, 1 - g], v[0, 1 - g],
                                 sm_scale=0.2)
        assert np.abs(o[0, h] - other).max() > 1e-3


# --------------------------------------------------------------------------
# paged cache, decode, split-K combine
# --------------------------------------------------------------------------

def _scatter_to_pages(k_logical, s_logical, table, nblk):
    """Write logical rows [Hkv][L][D] into pages of layout [blk][kvh][D/16][16][16]."""
    Hkv, L, D = k_logical.shape
    cache = np.zeros((nblk, Hkv, D // 16, 16, 16), np.int8)
    sc = np.zeros((nblk, Hkv, 16), np.float32)
    for g in range(Hkv):
        for t in range(L):
            blk = table[t // 16]
            for c in range(D):
                cache[blk, g, c // 16, t % 16, c % 16] = k_logical[g, t, c]
            sc[blk, g, t % 16] = s_logical[g, t]
    return cache, sc


def test_paged_decode_equals_dense_attention():
    rng = np.random.default_rng(11)
    Hq, Hkv, D, L = 4, 2, 32, 45       # ragged last page
    nblk = 7
    table = rng.permutation(nblk)[:3].astype(np.int32)
    kl = rng.integers(-127, 128, (Hkv, L, D)).astype(np.int8)
    vl = rng.integers(-127, 128, (Hkv, L, D)).astype(np.int8)
    ksl = rng.uniform(0.005, 0.02, (Hkv, L)).astype(np.float32)
    vsl = rng.uniform(0.005, 0.02, (Hkv, L)).astype(np.float32)
    kc, ks = _scatter_to_pages(kl, ksl, table, nblk)
    vc, vs = _scatter_to_pages(vl, vsl, table, nblk)
    qi = rng.integers(-127, 128, (1, Hq, D)).astype(np.int8)
    sq = rng.uniform(0.005, 0.02, (1, Hq)).astype(np.float32)
    o, lse = oracle.decode_paged(qi, sq, kc, vc, ks, vs, table[None], [L], sm_scale=0.25,
                                 threads=1)
    for h in range(Hq):
        g = h // 2
        vv = vl[g].astype(np.float64) * vsl[g][:, None].astype(np.float64)
        o_ref, l_ref = textbook_attention(qi[0, h:h + 1] * np.float64(sq[0, h]),
                                          kl[g] * ksl[g][:, None].astype(np.float64), vv, 0.25)
        np.testing.assert_allclose(o[0, h], o_ref[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[0, h], l_ref[0], rtol=1e-12)
    # a different physical placement of the same logical pages gives the
    # bitwise-same result
    table2 = rng.permutation(nblk)[:3].astype(np.int32)
    kc2, ks2 = _scatter_to_pages(kl, ksl, table2, nblk)
    vc2, vs2 = _scatter_to_pages(vl, vsl, table2, nblk)
    o2, lse2 = oracle.decode_paged(qi, sq, kc2, vc2, ks2, vs2, table2[None], [L], sm_scale=0.25,
                                   threads=1)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_splitk_combine_matches_unsplit():
    rng = np.random.default_rng(12)
    D, L = 16, 50
    qi = rng.integers(-127, 128, (3, D)).astype(np.int8)
    sq = rng.uniform(0.005, 0.02, 3).astype(np.float32)
    ki = rng.integers(-127, 128, (L, D)).astype(np.int8)
    sk = rng.uniform(0.005, 0.02, L).astype(np.float32)
    v = rng.standard_normal((L, D))
    o_full, l_full = oracle.attend(qi, sq, ki, sk, v, sm_scale=0.5)
    bounds = [0, 7, 7, 30, 50, 50]   # includes empty segments
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            o, l = oracle.attend(qi, sq, ki[a:b], sk[a:b], v[a:b], sm_scale=0.5)
        else:
            o, l = np.zeros((3, D)), np.full(3, -np.inf)
        parts_o.append(o)
        parts_l.append(l)
    op = np.stack(parts_o, 1)   # [3, S, D]
    lp = np.stack(parts_l, 1)   # [3, S]
    o, l = oracle.splitk_combine(op, lp)
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, l_full, rtol=1e-13)
    # one segment: identity
    o1, l1 = oracle.splitk_combine(op[:, 3:4], lp[:, 3:4])
    np.testing.assert_allclose(o1, op[:, 3], rtol=1e-15)
    assert np.array_equal(l1, lp[:, 3])
    # all segments empty
    oe, le = oracle.splitk_combine(np.zeros((2, 3, D)), np.full((2, 3), -np.inf))
    assert np.all(oe == 0) and np.all(le == -np.inf)


def test_prefill_with_paged_prefix_equals_concatenated_keys():
    rng = np.random.default_rng(13)
    Hq, Hkv, D, P, Sc = 2, 1, 32, 37, 20
    nblk = 5
    table = rng.permutation(nblk)[:3].astype(np.int32)
    kl = rng.integers(-127, 128, (Hkv, P, D)).astype(np.int8)
    vl = rng.integers(-127, 128, (Hkv, P, D)).astype(np.int8)
    ksl = rng.uniform(0.005, 0.02, (Hkv, P)).astype(np.float32)
    vsl = rng.uniform(0.005, 0.02, (Hkv, P)).astype(np.float32)
    kc, ks = _scatter_to_pages(kl, ksl, table, nblk)
    vc, vs = _scatter_to_pages(vl, vsl, table, nblk)
    qi = rng.integers(-127, 128, (1, Hq, Sc, D)).astype(np.int8)
    sq = rng.uniform(0.005, 0.02, (1, Hq, Sc)).astype(np.float32)
    kn = rng.integers(-127, 128, (1, Hkv, Sc, D)).astype(np.int8)
    skn = rng.uniform(0.005, 0.02, (1, Hkv, Sc)).astype(np.float32)
    vn = rng.standard_normal((1, Hkv, Sc, D))
    prefix = dict(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs, block_table=table[None],
                  lens=[P])
    o, lse = oracle.prefill(qi, sq, 1, kn, skn, 1, vn, causal=True, sm_scale=0.3,
                            prefix=prefix, threads=1)
    for h in range(Hq):
        kk = np.concatenate([kl[0] * ksl[0][:, None].astype(np.float64),
                             kn[0, 0] * skn[0, 0][:, None].astype(np.float64)], 0)
        vv = np.concatenate([vl[0] * vsl[0][:, None].astype(np.float64), vn[0, 0]], 0)
        o_ref, l_ref = textbook_attention(qi[0, h] * sq[0, h][:, None].astype(np.float64), kk, vv,
                                          0.3, causal=True, offset=P)
        np.testing.assert_allclose(o[0, h], o_ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[0, h], l_ref, rtol=1e-12)


def test_kv_append_identity_and_page_layout():
    """Rows of integers with amax exactly 127 quantise to themselves (s = 1);
    every element must land at [page][head][c/16][slot][c%16] of the page
    the block table names for its token ([P1] sections 3 and 4).  The
    expected cache is written here element by element, by hand."""
    rng = np.random.default_rng(21)
    B, H, n, D, nblk = 2, 3, 23, 64, 9
    x = rng.integers(-127, 128, (B, H, n, D)).astype(np.float32)
    x[..., 5] = np.where(rng.random((B, H, n)) < 0.5, 127.0, -127.0)
    table = np.stack([rng.permutation(nblk)[:4], rng.permutation(nblk)[:4]]).astype(np.int32)
    pos = np.array([3, 17], np.int32)
    cache0 = rng.integers(-127, 128, (nblk, H, D // 16, 16, 16)).astype(np.int8)
    scale0 = rng.uniform(0.005, 0.02, (nblk, H, 16)).astype(np.float32)
    cache, scale, skipped = oracle.kv_append(x, table, pos, cache0, scale0)
    assert skipped == 0
    want_c, want_s = cache0.copy(), scale0.copy()
    for b in range(B):
        for h in range(H):
            for t in range(n):
                p = pos[b] + t
                blk, slot = table[b, p // 16], p % 16
                want_s[blk, h, slot] = 1.0
                for c in range(D):
                    want_c[blk, h, c // 16, slot, c % 16] = x[b, h, t, c]
    assert np.array_equal(cache, want_c)
    assert np.array_equal(scale, want_s)


def test_kv_append_error_bound_and_bad_pages():
    """Each stored code times its scale is within half a quantisation step
    of the input, the scale is the row's amax / 127, and rows whose page
    index is out of range are skipped and leave the cache untouched."""
    rng = np.random.default_rng(22)
    B, H, n, D, nblk = 1, 2, 40, 128, 6
    x = rng.standard_normal((B, H, n, D)).astype(np.float32) * 3
    table = np.array([[2, 0, 99, 4]], np.int32)      # page index 99 does not exist
    pos = np.array([0], np.int32)
    cache0 = np.zeros((nblk, H, D // 16, 16, 16), np.int8)
    scale0 = np.zeros((nblk, H, 16), np.float32)
    cache, scale, skipped = oracle.kv_append(x, table, pos, cache0, scale0)
    assert skipped == H * 8                          # tokens 32..39 map to page 99
    for h in range(H):
        for t in range(32):
            blk, slot = table[0, t // 16], t % 16
            s = scale[blk, h, slot]
            assert s == np.float32(np.abs(x[0, h, t]).max() / np.float32(127))
            codes = cache[blk, h, :, slot, :].reshape(D).astype(np.float64)
            assert np.all(np.abs(codes * s - x[0, h, t]) <= s / 2 * (1 + 1e-6))
    untouched = [b for b in range(nblk) if b not in (2, 0)]
    assert not cache[untouched].any() and not scale[untouched].any()


# --------------------------------------------------------------------------
# variable-length packed batches: every sequence is its own problem
# --------------------------------------------------------------------------

def test_varlen_quant_groups_and_mean_are_per_sequence():
    # two sequences (70 and 50 tokens) packed back to back; per-64-token
    # groups.  Groups taken over the packed axis would put sequence 0's
    # tokens 64..69 in one group with sequence 1's first 58 tokens (amax 100).
    rng = np.random.default_rng(21)
    H, D = 2, 64
    cu = np.array([0, 70, 120])
    x = np.zeros((120, H, D), np.float32)
    x[0:64] = rng.uniform(-0.5, 0.5, (64, H, D))
    x[0:64, :, 3] = 1.0
    x[64:70] = rng.uniform(-0.25, 0.25, (6, H, D))
    x[64:70, :, 5] = -0.5
    x[70:120] = rng.uniform(-50, 50, (50, H, D))
    x[70:120, :, 7] = 100.0
    q, scales, _ = oracle.quant_int8_varlen(x, cu, block_tokens=64)
    f = np.float32
    assert scales[0].shape == (H, 2) and scales[1].shape == (H, 1)
    assert np.all(scales[0][:, 0] == f(1.0) / f(127.0))
    assert np.all(scales[0][:, 1] == f(0.5) / f(127.0))
    assert np.all(scales[1][:, 0] == f(100.0) / f(127.0))
    assert np.all(q[:, 0:64, 3] == 127) and np.all(q[:, 64:70, 5] == -127)
    assert np.all(q[:, 70:120, 7] == 127)
    # smooth: rows constant within a sequence -> the mean is that row, the
    # smoothed rows are zero, codes and scales are zero
    rows = np.array([0.25, -1.5, 3.0], np.float32)
    cu3 = np.array([0, 5, 5, 12])      # the middle sequence is empty
    x3 = np.zeros((12, 1, D), np.float32)
    x3[0:5] = rows[0]
    x3[5:12] = rows[2]
    q3, s3, mu3 = oracle.quant_int8_varlen(x3, cu3, block_tokens=1, smooth=True)
    assert np.all(mu3[0] == rows[0]) and np.all(mu3[1] == 0.0) and np.all(mu3[2] == rows[2])
    assert np.all(q3 == 0) and all(np.all(s == 0) for s in s3)
    assert s3[1].shape == (1, 0)


def _varlen_case(rng, lq, lk, Hq, Hkv, D):
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    q = np.stack([integer_rows(rng, cu_q[-1], D) for _ in range(Hq)])   # [Hq, tq, D]
    k = np.stack([integer_rows(rng, cu_k[-1], D) for _ in range(Hkv)])
    return cu_q, cu_k, q, k


def test_varlen_prefill_equals_textbook_per_sequence():
    # integer Q/K with per-token amax 127: quantisation is the identity, so
    # every sequence's rows equal exact float64 attention over its own keys
    rng = np.random.default_rng(22)
    lq, lk = [5, 0, 9, 3], [7, 4, 9, 1]
    Hq, Hkv, D = 4, 2, 64
    cu_q, cu_k, q, k = _varlen_case(rng, lq, lk, Hq, Hkv, D)
    v = rng.standard_normal((cu_k[-1], Hkv, D))
    sm = 1.0 / 4096
    qs = [np.ones((Hq, n), np.float32) for n in lq]
    ks = [np.ones((Hkv, n), np.float32) for n in lk]
    for causal in (False, True):
        o, lse = oracle.prefill_varlen(q.astype(np.int8), qs, 1, k.astype(np.int8), ks, 1, v,
                                       cu_q, cu_k, causal=causal, sm_scale=sm)
        for b in range(len(lq)):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                qq = q[h, cu_q[b]:cu_q[b + 1]]
                if len(qq) == 0:
                    continue
                ref_o, ref_l = textbook_attention(qq, k[g, cu_k[b]:cu_k[b + 1]],
                                                  v[cu_k[b]:cu_k[b + 1], g], sm, causal,
                                                  lk[b] - lq[b])
                got_o = o[cu_q[b]:cu_q[b + 1], h]
                got_l = lse[h, cu_q[b]:cu_q[b + 1]]
                fin = np.isfinite(ref_l)
                np.testing.assert_allclose(got_o[fin], ref_o[fin], rtol=1e-9, atol=1e-12)
                np.testing.assert_allclose(got_l[fin], ref_l[fin], rtol=1e-12)
                assert np.all(np.isneginf(got_l[~fin])) and np.all(got_o[~fin] == 0)


def test_varlen_causal_alignment_closed_form():
    # K codes 0: every visible key scores 0, so row i of sequence b averages
    # the visible keys' values v_j = j: o = (n - 1) / 2 and lse = ln n with
    # n = min(Sk_b, i + Sk_b - Sq_b + 1) (bottom-right alignment per sequence)
    lq, lk = [6, 4, 8], [3, 10, 8]
    Hq, Hkv, D = 2, 1, 64
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    rng = np.random.default_rng(23)
    q = rng.integers(-127, 128, (Hq, cu_q[-1], D)).astype(np.int8)
    k = np.zeros((Hkv, cu_k[-1], D), np.int8)
    v = np.zeros((cu_k[-1], Hkv, D))
    for b in range(3):
        v[cu_k[b]:cu_k[b + 1]] = np.arange(lk[b])[:, None, None]
    qs = [rng.uniform(0.01, 0.02, (Hq, n)).astype(np.float32) for n in lq]
    ks = [rng.uniform(0.01, 0.02, (Hkv, n)).astype(np.float32) for n in lk]
    o, lse = oracle.prefill_varlen(q, qs, 1, k, ks, 1, v, cu_q, cu_k, causal=True)
    for b in range(3):
        for i in range(lq[b]):
            n = min(lk[b], i + lk[b] - lq[b] + 1)
            t = cu_q[b] + i
            if n <= 0:
                assert np.all(o[t] == 0) and np.all(np.isneginf(lse[:, t]))
            else:
                np.testing.assert_allclose(o[t], (n - 1) / 2.0, rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[:, t], math.log(n), rtol=1e-14)


def test_varlen_values_never_leak_across_sequences():
    # V constant per sequence: softmax rows sum to 1, so every output row of
    # sequence b equals that sequence's constant, whatever the scores
    rng = np.random.default_rng(24)
    lq, lk = [33, 17, 50], [40, 17, 64]
    Hq, Hkv, D = 2, 2, 64
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    x_q = rng.standard_normal((cu_q[-1], Hq, D)).astype(np.float32)
    x_k = (rng.standard_normal((cu_k[-1], Hkv, D)) * 3).astype(np.float32)
    q, qs, _ = oracle.quant_int8_varlen(x_q, cu_q, block_tokens=1)
    k, ks, _ = oracle.quant_int8_varlen(x_k, cu_k, block_tokens=1)
    consts = [1.5, -2.0, 0.75]
    v = np.zeros((cu_k[-1], Hkv, D))
    for b in range(3):
        v[cu_k[b]:cu_k[b + 1]] = consts[b]
    for causal in (False, True):
        o, _ = oracle.prefill_varlen(q, qs, 1, k, ks, 1, v, cu_q, cu_k, causal=causal)
        for b in range(3):
            np.testing.assert_allclose(o[cu_q[b]:cu_q[b + 1]], consts[b], rtol=1e-13)


# --------------------------------------------------------------------------
# smooth_v: subtract the chunk's V mean from every value, add it back
# --------------------------------------------------------------------------

def test_smooth_v_is_exact_identity_with_prefix_and_empty_rows():
    # softmax rows sum to 1, so P (V - mu) + mu = P V: smoothing changes no
    # output in exact arithmetic, with or without a paged prefix, and a row
    # that sees no key stays 0 (a forgotten add-back, a wrong sign or a mean
    # taken off the chunk only would all show here: V has a large offset)
    rng = np.random.default_rng(31)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 40, 24, 64
    q = rng.integers(-127, 128, (B, Hq, Sq, D)).astype(np.int8)
    k = rng.integers(-127, 128, (B, Hkv, Sk, D)).astype(np.int8)
    qs = rng.uniform(0.001, 0.002, (B, Hq, Sq)).astype(np.float32)
    ks = rng.uniform(0.001, 0.002, (B, Hkv, Sk)).astype(np.float32)
    v = (rng.standard_normal((B, Hkv, Sk, D)) + 50.0).astype(np.float32)
    P = 32
    pre = dict(k_cache=rng.integers(-127, 128, (4, Hkv, D // 16, 16, 16)).astype(np.int8),
               v_cache=rng.integers(-127, 128, (4, Hkv, D // 16, 16, 16)).astype(np.int8),
               k_scale=rng.uniform(0.001, 0.002, (4, Hkv, 16)).astype(np.float32),
               v_scale=rng.uniform(0.005, 0.02, (4, Hkv, 16)).astype(np.float32),
               block_table=np.array([[2, 0, 3, 1]], np.int32), lens=np.array([P]))
    for prefix in (None, pre):
        # Sq > Sk + P: the first causal rows see no key at all
        o0, l0 = oracle.prefill(q, qs, 1, k, ks, 1, v, causal=True, prefix=prefix)
        o1, l1 = oracle.prefill(q, qs, 1, k, ks, 1, v, causal=True, prefix=prefix, smooth_v=True)
        assert np.array_equal(l0, l1)
        np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-11)
        empty = ~np.isfinite(l0)
        assert np.all(o1[empty] == 0)
        if prefix is None:
            assert empty.any()   # Sq > Sk: the first 16 rows see nothing


def test_smooth_v_mean_is_the_chunk_token_mean():
    # the subtracted mean is token_mean of the chunk values: with V constant
    # along tokens every smoothed value is 0, so only the add-back remains
    rng = np.random.default_rng(32)
    D = 64
    v = np.broadcast_to(rng.uniform(-3, 3, (1, 1, 1, D)), (1, 1, 20, D)).astype(np.float32)
    mu = oracle.token_mean(v)
    assert np.array_equal(mu[0, 0], v[0, 0, 0])
    q = rng.integers(-127, 128, (1, 1, 20, D)).astype(np.int8)
    k = rng.integers(-127, 128, (1, 1, 20, D)).astype(np.int8)
    s = np.full((1, 1, 20), 0.01, np.float32)
    o, _ = oracle.prefill(q, s, 1, k, s, 1, v, causal=False, smooth_v=True)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, 0], (20, D)), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# per-block scales, the mixed smoothed/unsmoothed key set, row sampling and
# the per-sequence row bias: the glue around the C functions
# --------------------------------------------------------------------------

def _grouped_rows(rng, n, d, block, exps):
    """Integer rows whose 'block'-token group g has amax exactly 127 * 2^exps[g]
    (every element a multiple of 2^exps[g]), so a per-block quantisation with
    that block has scale 2^exps[g] and is exact."""
    x = integer_rows(rng, n, d).astype(np.float64)
    for g in range((n + block - 1) // block):
        x[g * block:(g + 1) * block] *= 2.0 ** exps[g]
    return x.astype(np.float32)


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_per_block_scales_against_textbook(causal):
    """Q in 128-token groups and K in 64-token groups with a different
    power-of-two scale per group (ragged last groups): per-block quantisation
    is then exact, so the method equals float64 attention on the original
    values.  Swapping the two block sizes, or mapping rows to groups with
    anything but row // block, scales some scores by the wrong group and
    fails here."""
    rng = np.random.default_rng(41)
    Sq, Sk, D = 200, 300, 32                       # Q groups 128 + 72; K 4 x 64 + 44
    q = _grouped_rows(rng, Sq, D, 128, [-3, 2])
    k = _grouped_rows(rng, Sk, D, 64, [1, -2, 3, 0, -1])
    v = rng.standard_normal((Sk, D))
    qi, qs, _ = oracle.quant_int8(q[None, None], block_tokens=128)
    ki, ks, _ = oracle.quant_int8(k[None, None], block_tokens=64)
    assert qs[0, 0].tolist() == [2.0 ** -3, 2.0 ** 2]
    assert ks[0, 0].tolist() == [2.0, 2.0 ** -2, 2.0 ** 3, 1.0, 0.5]
    sm = 1.0 / (D * 127.0 * 127.0 * 8.0)
    o, lse = oracle.prefill(qi, qs, 128, ki, ks, 64, v[None, None], causal=causal, sm_scale=sm,
                            threads=1)
    o_ref, lse_ref = textbook_attention(q, k, v, sm, causal, Sk - Sq)
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=1e-12, atol=1e-12)


def test_prefill_bias_applies_to_the_chunk_not_the_prefix():
    """Chunked prefill with smooth_k over an unsmoothed paged prefix: the
    chunk keys are K_new = mu + I exactly (I integer, in +-pairs so the token
    mean is mu), the prefix keys are stored codes with power-of-two scales,
    Q is integer with amax 127.  With the row bias q.mu given, the result
    must equal float64 attention over [prefix keys as stored || chunk keys
    before smoothing]; the bias added to the prefix scores instead, or left
    off the chunk, fails."""
    rng = np.random.default_rng(42)
    Hq, Hkv, D, P, Sc, nblk = 2, 1, 32, 40, 24, 6
    half = integer_rows(rng, Sc // 2, D)
    I = np.concatenate([half, -half], 0)
    mu = (rng.integers(-200, 200, size=D) * 0.25).astype(np.float32)
    k_new = (I + mu[None, :]).astype(np.float32)
    q = np.stack([integer_rows(rng, Sc, D) for _ in range(Hq)])          # [Hq, Sc, D]
    v_new = rng.standard_normal((Sc, D))
    table = rng.permutation(nblk)[:3].astype(np.int32)
    kl = rng.integers(-127, 128, (Hkv, P, D)).astype(np.int8)
    vl = rng.integers(-127, 128, (Hkv, P, D)).astype(np.int8)
    ksl = (2.0 ** -rng.integers(-1, 3, (Hkv, P))).astype(np.float32)
    vsl = rng.uniform(0.005, 0.02, (Hkv, P)).astype(np.float32)
    kc, ks = _scatter_to_pages(kl, ksl, table, nblk)
    vc, vs = _scatter_to_pages(vl, vsl, table, nblk)
    prefix = dict(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs, block_table=table[None],
                  lens=[P])
    ki, ksn, mu_o = oracle.quant_int8(k_new[None, None], smooth=True)
    assert np.array_equal(mu_o[0, 0], mu) and np.all(ksn == 1.0)
    qi, qsc, _ = oracle.quant_int8(q[None])
    bias = oracle.row_bias(q[None], mu_o)
    sm = 1.0 / (D * 127.0 * 127.0 * 2.0)
    o, lse = oracle.prefill(qi, qsc, 1, ki, ksn, 1, v_new[None, None], causal=True, sm_scale=sm,
                            q_bias=bias, prefix=prefix, threads=1)
    keys = np.concatenate([kl[0] * ksl[0][:, None].astype(np.float64), k_new], 0)
    vals = np.concatenate([vl[0] * vsl[0][:, None].astype(np.float64), v_new], 0)
    for h in range(Hq):
        o_ref, l_ref = textbook_attention(q[h], keys, vals, sm, causal=True, offset=P)
        np.testing.assert_allclose(o[0, h], o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], l_ref, rtol=1e-12, atol=1e-12)


def test_prefill_row_sample_equals_full_rows():
    """Evaluating a subset of query rows (causal, over a paged prefix, per
    block Q and K) gives exactly those rows of the full evaluation: the row
    positions, not their order in the sample, decide what each row sees."""
    rng = np.random.default_rng(43)
    Hq, Hkv, D, P, Sq = 2, 1, 32, 37, 150
    table = rng.permutation(4)[:3].astype(np.int32)
    kc = rng.integers(-127, 128, (4, Hkv, D // 16, 16, 16)).astype(np.int8)
    vc = rng.integers(-127, 128, (4, Hkv, D // 16, 16, 16)).astype(np.int8)
    sc = rng.uniform(0.005, 0.02, (4, Hkv, 16)).astype(np.float32)
    prefix = dict(k_cache=kc, v_cache=vc, k_scale=sc, v_scale=sc[::-1].copy(),
                  block_table=table[None], lens=[P])
    x = rng.standard_normal((1, Hq, Sq, D)).astype(np.float32)
    kx = rng.standard_normal((1, Hkv, Sq, D)).astype(np.float32)
    qi, qs, _ = oracle.quant_int8(x, block_tokens=128)
    ki, ks, _ = oracle.quant_int8(kx, block_tokens=64)
    v = rng.standard_normal((1, Hkv, Sq, D))
    o, lse = oracle.prefill(qi, qs, 128, ki, ks, 64, v, causal=True, prefix=prefix, threads=1)
    rows = np.array([149, 0, 77, 128, 127, 5])
    o2, l2 = oracle.prefill(qi, qs, 128, ki, ks, 64, v, causal=True, prefix=prefix, rows=rows,
                            threads=1)
    assert np.array_equal(o2, o[:, :, rows]) and np.array_equal(l2, lse[:, :, rows])


def test_row_bias_varlen_hand_computed():
    """b[h, t] = sum_c x[t, h, c] mu[seq(t), h // (H / Hmu), c], written out
    with explicit loops over sequences, tokens, heads and channels; integer
    values make every sum exact, and each sequence's mean differs so a wrong
    sequence or GQA group changes the result."""
    rng = np.random.default_rng(44)
    H, Hmu, D = 4, 2, 8
    cu = np.array([0, 3, 3, 8, 9])                    # includes an empty sequence
    x = rng.integers(-5, 6, (cu[-1], H, D)).astype(np.float32)
    mu = rng.integers(-3, 4, (len(cu) - 1, Hmu, D)).astype(np.float32)
    got = oracle.row_bias_varlen(x, cu, mu)
    want = np.zeros((H, cu[-1]))
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1]):
            for h in range(H):
                acc = 0.0
                for c in range(D):
                    acc += float(x[t, h, c]) * float(mu[b, h // (H // Hmu), c])
                want[h, t] = acc
    assert np.array_equal(got, want)


def test_decode_pairs_and_varlen_rows_sample_the_full_result():
    """The sampled forms the full-size parity tests use: decode over a list
    of (sequence, KV head) pairs gives exactly those heads of the full
    decode (the others stay zero / -inf), and varlen prefill over per-
    sequence row lists gives exactly those rows (the others stay NaN)."""
    rng = np.random.default_rng(45)
    B, Hq, Hkv, D, nblk = 3, 4, 2, 32, 12
    lens = [40, 17, 64]
    table = rng.permutation(nblk).reshape(B, 4).astype(np.int32)
    kc = rng.integers(-127, 128, (nblk, Hkv, D // 16, 16, 16)).astype(np.int8)
    vc = rng.integers(-127, 128, (nblk, Hkv, D // 16, 16, 16)).astype(np.int8)
    ks = rng.uniform(0.005, 0.02, (nblk, Hkv, 16)).astype(np.float32)
    vs = rng.uniform(0.005, 0.02, (nblk, Hkv, 16)).astype(np.float32)
    qi = rng.integers(-127, 128, (B, Hq, D)).astype(np.int8)
    qs = rng.uniform(0.005, 0.02, (B, Hq)).astype(np.float32)
    o, lse = oracle.decode_paged(qi, qs, kc, vc, ks, vs, table, lens, threads=1)
    pairs = [(2, 0), (0, 1)]
    o2, l2 = oracle.decode_paged(qi, qs, kc, vc, ks, vs, table, lens, threads=1, pairs=pairs)
    for b in range(B):
        for g in range(Hkv):
            hs = slice(2 * g, 2 * g + 2)
            if (b, g) in pairs:
                assert np.array_equal(o2[b, hs], o[b, hs]) and np.array_equal(l2[b, hs], lse[b, hs])
            else:
                assert np.all(o2[b, hs] == 0) and np.all(np.isneginf(l2[b, hs]))
    lq, lk = [9, 30, 4], [12, 30, 20]
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    xq = rng.standard_normal((cu_q[-1], Hq, D)).astype(np.float32)
    xk = rng.standard_normal((cu_k[-1], Hkv, D)).astype(np.float32)
    q8, qsc, _ = oracle.quant_int8_varlen(xq, cu_q, block_tokens=1)
    k8, ksc, _ = oracle.quant_int8_varlen(xk, cu_k, block_tokens=1)
    v = rng.standard_normal((cu_k[-1], Hkv, D))
    of, lf = oracle.prefill_varlen(q8, qsc, 1, k8, ksc, 1, v, cu_q, cu_k, causal=True)
    rows = [np.array([8, 0]), np.array([29, 3, 17]), np.array([1])]
    os_, ls_ = oracle.prefill_varlen(q8, qsc, 1, k8, ksc, 1, v, cu_q, cu_k, causal=True,
                                     rows=rows)
    picked = np.zeros(cu_q[-1], bool)
    for b in range(3):
        t = cu_q[b] + rows[b]
        picked[t] = True
        assert np.array_equal(os_[t], of[t]) and np.array_equal(ls_[:, t], lf[:, t])
    assert np.all(np.isnan(os_[~picked])) and np.all(np.isnan(ls_[:, ~picked]))


# --------------------------------------------------------------------------
# INT8 P.V: V-scaled probabilities quantised per 16-key group
# --------------------------------------------------------------------------

def test_pv_int8_exact_when_codes_are_integers():
    """K = 0 makes every probability equal (p = 1 before normalising), so a
    group's w_j = sv_j; with sv_j = k_j 2^-10 (k_j integer) and one k_j = 127
    in every 16-key group (the last one short), the group scale is 2^-10 and
    the codes are the k_j themselves: INT8 P.V then equals float64 attention
    on v_j * sv_j exactly.  Groups not aligned at multiples of 16, a scale
    taken from p instead of p * sv, or a dropped group scale all fail."""
    rng = np.random.default_rng(51)
    nk, D = 45, 32
    kk = rng.integers(1, 127, nk)
    for g0 in range(0, nk, 16):
        kk[g0 + rng.integers(0, min(16, nk - g0))] = 127
    sv = (kk * 2.0 ** -10).astype(np.float32)
    v = rng.integers(-127, 128, (nk, D)).astype(np.int8)
    qi = rng.integers(-127, 128, (3, D)).astype(np.int8)
    sq = np.full(3, 0.01, np.float32)
    k = np.zeros((nk, D), np.int8)
    sk = np.full(nk, 0.02, np.float32)
    o, lse = oracle.attend_pv_int8(qi, sq, k, sk, v, sv, sm_scale=0.1)
    vhat = v.astype(np.float64) * sv.astype(np.float64)[:, None]
    o_ref, lse_ref = textbook_attention(np.zeros((3, D)), np.zeros((nk, D)), vhat, 0.1)
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-14)
    # the same values with the group boundaries moved by 8 keys change codes
    o8, _ = oracle.attend_pv_int8(qi, sq, k, sk, v[8:], sv[8:], sm_scale=0.1)
    o_ref8, _ = textbook_attention(np.zeros((3, D)), np.zeros((nk - 8, D)), vhat[8:], 0.1)
    assert np.abs(o8 - o_ref8).max() > 1e-6


def test_pv_int8_within_half_a_step_of_exact_attention():
    """Each code is within half a step of w_j / s_g, so INT8 P.V differs from
    exact attention (same scores, values v_j sv_j) by at most
    sum_j s_g(j) |v_j| / 2 / l per channel -- and it does differ."""
    rng = np.random.default_rng(52)
    nq, nk, D = 4, 70, 64
    qi = rng.integers(-127, 128, (nq, D)).astype(np.int8)
    ki = rng.integers(-127, 128, (nk, D)).astype(np.int8)
    sq = rng.uniform(0.005, 0.02, nq).astype(np.float32)
    sk = rng.uniform(0.005, 0.02, nk).astype(np.float32)
    v = rng.integers(-127, 128, (nk, D)).astype(np.int8)
    sv = rng.uniform(0.005, 0.02, nk).astype(np.float32)
    sm = 0.5
    o, lse = oracle.attend_pv_int8(qi, sq, ki, sk, v, sv, sm_scale=sm)
    vhat = v.astype(np.float64) * sv.astype(np.float64)[:, None]
    o_ex, lse_ex = oracle.attend(qi, sq, ki, sk, vhat, sm_scale=sm)
    np.testing.assert_allclose(lse, lse_ex, rtol=1e-14)
    z = (qi.astype(np.float64) @ ki.astype(np.float64).T) * sq[:, None] * sk[None, :] * sm
    p = np.exp(z - z.max(1, keepdims=True))
    w = p * sv[None, :]
    bound = np.zeros((nq, D))
    for g0 in range(0, nk, 16):
        s = w[:, g0:g0 + 16].max(1) / 127.0
        bound += (s[:, None, None] * 0.5 * np.abs(v[g0:g0 + 16].astype(np.float64))[None]).sum(1)
    bound /= p.sum(1)[:, None]
    err = np.abs(o - o_ex)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err.max() > 0


def test_pv_int8_single_dominant_key():
    """One key whose score dwarfs the rest (their probabilities underflow to
    0): its group's scale is its own w / 127, its code 127, every other code
    0, so the output is that key's value times its scale."""
    D = 16
    k = np.zeros((20, D), np.int8)
    k[13] = 127
    q = np.full((1, D), 127, np.int8)
    v = np.arange(20 * D).reshape(20, D).astype(np.int64) % 255 - 127
    v = v.astype(np.int8)
    sv = np.linspace(0.005, 0.02, 20).astype(np.float32)
    o, lse = oracle.attend_pv_int8(q, np.ones(1, np.float32), k, np.ones(20, np.float32), v, sv,
                                   sm_scale=1.0)
    np.testing.assert_allclose(o[0], v[13].astype(np.float64) * np.float64(sv[13]), rtol=1e-14)
    assert lse[0] == 16 * 127 * 127


def test_pv_int8_group_scales_and_rounding_by_hand():
    """Equal probabilities (K = 0) and hand-chosen v scales: group g of 16
    keys has its largest w at exactly 127 * 2^-(10+g), so its scale is
    2^-(10+g); inside a group w_j / s = x_j with x_j listed below (quarter
    and half steps), whose codes -- nearest integer, ties to even -- are
    written out by hand.  The output must equal the mean of code_j * s_g(j)
    * v_j.  Merged groups (a scale shared across 32 keys), truncation or
    ties away from zero all change it."""
    xs = [127.0, 3.25, 3.75, 4.5, 5.5, 0.5, 1.5, 0.25, 126.5, 2.0, 7.75, 10.5, 11.5, 0.0, 64.25,
          99.5]
    codes = [127, 3, 4, 4, 6, 0, 2, 0, 126, 2, 8, 10, 12, 0, 64, 100]
    D, G = 8, 3
    nk = 16 * G
    rng = np.random.default_rng(53)
    sv, code_all, scale_all = [], [], []
    for g in range(G):
        perm = rng.permutation(16)
        for t in perm:
            sv.append(xs[t] * 2.0 ** -(10 + g))
            code_all.append(codes[t])
            scale_all.append(2.0 ** -(10 + g))
    sv = np.array(sv, np.float32)
    assert np.array_equal(sv.astype(np.float64), np.array(sv, np.float64))
    v = rng.integers(-127, 128, (nk, D)).astype(np.int8)
    o, _ = oracle.attend_pv_int8(np.ones((1, D), np.int8), np.ones(1, np.float32),
                                 np.zeros((nk, D), np.int8), np.ones(nk, np.float32), v, sv,
                                 sm_scale=1.0)
    want = (np.array(code_all, np.float64)[:, None] * np.array(scale_all)[:, None]
            * v.astype(np.float64)).sum(0) / nk
    np.testing.assert_allclose(o[0], want, rtol=1e-14, atol=1e-18)
