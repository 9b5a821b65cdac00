"""GPU parity for packed variable-length batches.

Quantisation (codes, scales, the smooth_k mean) is checked bit for bit
against the oracle's per-sequence quantisation; raw INT32 scores bit for
bit; outputs and LSE within rel-L2 5e-3 / max-abs 2e-3 of the oracle's
per-sequence fp64 result.  The packed launch must also equal, bit for bit,
the dense kernel run on each sequence on its own.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _group0(cu_b, b, block):
    """First scale group of sequence b in the packed scale layout."""
    return cu_b if block == 1 else cu_b // block + b


def _seq_scales(scale, cu, block):
    """Per-sequence [H, ceil(len / block)] views of a packed scale array."""
    s = np_(scale)
    out = []
    for b in range(len(cu) - 1):
        n = (int(cu[b + 1]) - int(cu[b]) + block - 1) // block
        g0 = _group0(int(cu[b]), b, block)
        out.append(s[:, g0:g0 + n])
    return out


def _check_quant(sage, x, cu_t, max_len, block, smooth=False):
    q, s, mu, _ = sage.sage_quant_int8_varlen(x, cu_t, max_len, block_tokens=block, smooth=smooth)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    cu = np_(cu_t)
    xs = f32(x)
    mu_np = np_(mu) if smooth else None
    for b, (t0, t1) in enumerate(oracle.seq_bounds(cu)):
        if t1 == t0:
            if smooth:
                assert np.all(mu_np[b] == 0)
            continue
        xb = np.ascontiguousarray(xs[t0:t1].transpose(1, 0, 2))
        if smooth:
            # the mean is an exact sum rounded once: bit-exact
            assert np.array_equal(mu_np[b], oracle.token_mean(xb)), "mean of sequence %d" % b
        q_ref, s_ref, _ = oracle.quant_int8(xb, block_tokens=block, smooth=smooth,
                                            mu=mu_np[b] if smooth else None)
        assert np.array_equal(_seq_scales(s, cu, block)[b], s_ref), "scales of sequence %d" % b
        assert np.array_equal(np_(q)[:, t0:t1], q_ref), "codes of sequence %d" % b
    # and the whole batch through the oracle's own per-sequence loop
    q_all, s_all, _ = oracle.quant_int8_varlen(xs, cu, block_tokens=block, smooth=False) \
        if not smooth else (None, None, None)
    if q_all is not None:
        assert np.array_equal(np_(q), q_all)
        for a, r in zip(_seq_scales(s, cu, block), s_all):
            assert np.array_equal(a, r)
    return q, s, mu


LENS = [130, 0, 257, 1, 64, 700, 63]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("block", [1, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_varlen_quant_bit_exact(sage, D, block, dtype):
    x = W.varlen_qkv(LENS, LENS, 3, 3, D, seed=D + block, dtype=dtype, device="cuda",
                     k_offset_std=2.0)
    _check_quant(sage, x.q, x.cu_q, x.max_q, block)
    _check_quant(sage, x.k, x.cu_k, x.max_k, block, smooth=True)


def test_varlen_quant_strided_and_row_bias(sage):
    x = W.varlen_qkv(LENS, LENS, 6, 2, 128, seed=9, device="cuda", k_offset_std=2.0)
    # a strided view: Q packed inside a wider [total, 8, D] buffer
    wide = torch.zeros((x.q.shape[0], 8, 128), dtype=x.q.dtype, device="cuda")
    wide[:, 1:7] = x.q
    qv = wide[:, 1:7]
    q1, s1, _, _ = sage.sage_quant_int8_varlen(qv, x.cu_q, x.max_q)
    q2, s2, _, _ = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    _, _, mu, _ = sage.sage_quant_int8_varlen(x.k, x.cu_k, x.max_k, smooth=True)
    _, _, _, bias = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, mu_in=mu)
    torch.cuda.synchronize()
    ref = oracle.row_bias_varlen(f32(x.q), np_(x.cu_q), np_(mu))
    got = np_(bias)
    cu = np_(x.cu_q)
    for b, (t0, t1) in enumerate(oracle.seq_bounds(cu)):
        scale = np.abs(f32(x.q)[t0:t1]).sum(-1).T * np.abs(np_(mu)[b]).max()
        assert np.all(np.abs(got[:, t0:t1] - ref[:, t0:t1]) <= 1e-5 * scale + 1e-6)


def _quant_all(sage, x, q_block, k_block, smooth):
    qi, qs, _, _ = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, block_tokens=q_block)
    ki, ks, mu, _ = sage.sage_quant_int8_varlen(x.k, x.cu_k, x.max_k, block_tokens=k_block,
                                                smooth=smooth)
    bias = None
    if smooth:
        _, _, _, bias = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, block_tokens=q_block,
                                                    mu_in=mu)
    return qi, qs, ki, ks, bias


def _oracle(x, qi, qs, qb, ki, ks, kb, causal, bias=None, rows=None):
    cq, ck = np_(x.cu_q), np_(x.cu_k)
    return oracle.prefill_varlen(np_(qi), _seq_scales(qs, cq, qb), qb, np_(ki),
                                 _seq_scales(ks, ck, kb), kb, f32(x.v), cq, ck, causal=causal,
                                 q_bias=None if bias is None else np_(bias).astype(np.float64),
                                 rows=rows)


# query / key lengths per sequence: ragged tails, an empty sequence, a
# sequence with queries and no keys, more queries than keys (causal rows
# that see nothing), several key tiles
LQ = [200, 0, 129, 5, 64, 300, 17]
LK = [200, 9, 300, 0, 64, 100, 17]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("vdt", ["fp16", "bf16"])
def test_varlen_prefill_per_token(sage, D, causal, vdt):
    x = W.varlen_qkv(LQ, LK, 4, 2, D, seed=D + 3, device="cuda", v_dtype=vdt)
    qi, qs, ki, ks, _ = _quant_all(sage, x, 1, 1, False)
    out, lse = sage.sage_attn_prefill_varlen(qi, qs, 1, ki, ks, 1, x.v, x.cu_q, x.cu_k, x.max_q,
                                             x.max_k, causal=causal, out_dtype=torch.float16,
                                             return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    info = sage.last_launch_info()
    assert info["kernel"] == "prefill_varlen_kernel" and info["launches"] == 2
    o_ref, l_ref = _oracle(x, qi, qs, 1, ki, ks, 1, causal)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_varlen_prefill_per_block_smooth_k(sage, D):
    x = W.varlen_qkv(LQ, LK, 6, 3, D, seed=D + 11, device="cuda", k_offset_std=2.0)
    qi, qs, ki, ks, bias = _quant_all(sage, x, 128, 64, True)
    for causal in (False, True):
        out, lse = sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k,
                                                 x.max_q, x.max_k, causal=causal, q_bias=bias,
                                                 out_dtype=torch.float16, return_lse=True)
        torch.cuda.synchronize()
        assert sage.check_device_status()[0] == 0
        o_ref, l_ref = _oracle(x, qi, qs, 128, ki, ks, 64, causal, bias=bias)
        assert_close(f32(out), o_ref, "causal=%s" % causal)
        assert_close(np_(lse), l_ref, "lse causal=%s" % causal)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_varlen_raw_scores_bit_exact(sage, D):
    x = W.varlen_qkv(LQ, LK, 2, 1, D, seed=D + 5, device="cuda")
    qi, qs, ki, ks, _ = _quant_all(sage, x, 1, 1, False)
    tq = qi.shape[1]
    dbg = torch.full((2, tq, x.max_k), -(2 ** 31), dtype=torch.int32, device="cuda")
    sage.sage_attn_prefill_varlen(qi, qs, 1, ki, ks, 1, x.v, x.cu_q, x.cu_k, x.max_q, x.max_k,
                                  causal=True, debug_scores=dbg)
    torch.cuda.synchronize()
    d = np_(dbg)
    cq, ck = np_(x.cu_q), np_(x.cu_k)
    for b in range(len(LQ)):
        nq, nk = LQ[b], LK[b]
        if nq == 0:
            continue
        for h in range(2):
            blk = d[h, cq[b]:cq[b] + nq, :]
            if nk == 0:
                assert np.all(blk == -(2 ** 31))
                continue
            ref = oracle.qk_int32(np_(qi)[h, cq[b]:cq[b] + nq], np_(ki)[0, ck[b]:ck[b] + nk])
            vis = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
            assert np.array_equal(blk[:, :nk][vis], ref[vis])
            assert np.all(blk[:, :nk][~vis] == -(2 ** 31)) and np.all(blk[:, nk:] == -(2 ** 31))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("vdt", ["fp16", "bf16"])
@pytest.mark.parametrize("heads", [(4, 2), (3, 3)])
def test_varlen_equals_dense_per_sequence(sage, D, vdt, heads):
    """One packed launch gives, bit for bit, what the dense kernel gives on
    each sequence alone (the README's per-batch loop).  With an even GQA
    group a D <= 128 launch takes 128 rows of two heads per CTA, otherwise
    256 rows of one head: both layouts are covered."""
    lq, lk = [300, 77, 129], [300, 200, 129]
    x = W.varlen_qkv(lq, lk, heads[0], heads[1], D, seed=D + 17, device="cuda", v_dtype=vdt,
                     k_offset_std=2.0)
    qi, qs, ki, ks, bias = _quant_all(sage, x, 128, 64, True)
    out, lse = sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k,
                                             x.max_q, x.max_k, causal=True, q_bias=bias,
                                             return_lse=True)
    cq, ck = np_(x.cu_q), np_(x.cu_k)
    for b in range(3):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        gq0, gk0 = _group0(q0, b, 128), _group0(k0, b, 64)
        nq, nk = (q1 - q0 + 127) // 128, (k1 - k0 + 63) // 64
        o_b, l_b = sage.sage_attn_prefill(
            qi[:, q0:q1].unsqueeze(0).contiguous(), qs[:, gq0:gq0 + nq].unsqueeze(0).contiguous(),
            128, ki[:, k0:k1].unsqueeze(0).contiguous(),
            ks[:, gk0:gk0 + nk].unsqueeze(0).contiguous(), 64,
            x.v[k0:k1].transpose(0, 1).unsqueeze(0).contiguous(), causal=True,
            q_bias=bias[:, q0:q1].unsqueeze(0).contiguous(), return_lse=True, tail_split=False)
        torch.cuda.synchronize()
        assert torch.equal(out[q0:q1], o_b[0].transpose(0, 1)), "output of sequence %d" % b
        assert torch.equal(lse[:, q0:q1], l_b[0]), "lse of sequence %d" % b


def test_varlen_full_size_sampled(sage):
    """The varlen workload (24 sequences, log-uniform 256..8192 tokens, GQA
    32/8, D = 128, per-block Q/K with smooth_k, causal): every code exact
    and sampled rows of every sequence against the oracle."""
    P = W.WORKLOADS["varlen_prefill"].params
    lens = W.varlen_lengths(P["n"], P["lo"], P["hi"], P["seed"])
    x = W.varlen_qkv(lens, lens, P["Hq"], P["Hkv"], P["D"], seed=P["seed"], dtype=P["dtype"],
                     device="cuda", k_offset_std=P["k_offset_std"])
    qi, qs, ki, ks, bias = _quant_all(sage, x, P["q_block"], P["k_block"], True)
    out, lse = sage.sage_attn_prefill_varlen(qi, qs, P["q_block"], ki, ks, P["k_block"], x.v,
                                             x.cu_q, x.cu_k, x.max_q, x.max_k, causal=True,
                                             q_bias=bias, return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    rng = np.random.default_rng(0)
    rows = [np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 6)])) for n in lens]
    o_ref, l_ref = _oracle(x, qi, qs, P["q_block"], ki, ks, P["k_block"], True, bias=bias,
                           rows=rows)
    sel = np.concatenate([int(np_(x.cu_q)[b]) + r for b, r in enumerate(rows)])
    assert_close(f32(out)[sel], o_ref[sel])
    assert_close(np_(lse)[:, sel], l_ref[:, sel], "lse")


def test_varlen_bad_lengths_flag_and_skip(sage):
    x = W.varlen_qkv([64, 64], [64, 64], 2, 2, 64, seed=1, device="cuda")
    qi, qs, ki, ks, _ = _quant_all(sage, x, 1, 1, False)
    # sequence 1 claims 100 keys but max_seqlen_k says 64: flagged, treated empty
    bad_k = torch.tensor([0, 64, 164], dtype=torch.int32, device="cuda")
    out = sage.sage_attn_prefill_varlen(qi, qs, 1, ki, ks, 1, x.v, x.cu_q, bad_k, 64, 64,
                                        causal=False)
    st, word = sage.check_device_status()
    assert st == sage.SAGE_ERR_BAD_BLOCK
    good = sage.sage_attn_prefill_varlen(qi, qs, 1, ki, ks, 1, x.v, x.cu_q, x.cu_k, 64, 64,
                                         causal=False)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out[:64], good[:64])
    assert torch.all(out[64:] == 0)


@pytest.mark.parametrize("D", [128, 256])
def test_varlen_smooth_v(sage, D):
    """smooth_v per sequence: each sequence's own V mean (bit-exact), and the
    same outputs as the per-sequence oracle with smooth_v."""
    x = W.varlen_qkv(LQ, LK, 4, 2, D, seed=D + 81, device="cuda", v_dtype="bf16")
    x.v = (x.v.float() * 0.25 + 1.25).to(x.v.dtype)
    qi, qs, ki, ks, _ = _quant_all(sage, x, 1, 1, False)
    mu = torch.empty((len(LQ), 2, D), dtype=torch.float32, device="cuda")
    out, lse = sage.sage_attn_prefill_varlen(qi, qs, 1, ki, ks, 1, x.v, x.cu_q, x.cu_k, x.max_q,
                                             x.max_k, causal=True, out_dtype=torch.float16,
                                             return_lse=True, smooth_v=True, v_mean=mu)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    ck = np_(x.cu_k)
    for b, (t0, t1) in enumerate(oracle.seq_bounds(ck)):
        ref = oracle.token_mean(np.ascontiguousarray(f32(x.v)[t0:t1].transpose(1, 0, 2))) \
            if t1 > t0 else np.zeros((2, D), np.float32)
        assert np.array_equal(np_(mu)[b], ref), "mean of sequence %d" % b
    cq = np_(x.cu_q)
    o_ref, l_ref = oracle.prefill_varlen(np_(qi), _seq_scales(qs, cq, 1), 1, np_(ki),
                                         _seq_scales(ks, ck, 1), 1, f32(x.v), cq, ck,
                                         causal=True, smooth_v=True)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("nseq", [33, 70, 1100])
def test_varlen_many_sequences(sage, nseq):
    """Past 32 sequences a CTA's sequence search takes more than one round
    of warp-wide loads (two up to 1024, three beyond): every code, scale and
    mean stays exact and every output row (sampled for the largest batch)
    matches the oracle, empty and one-token sequences included."""
    g = np.random.default_rng(nseq)
    lens = [int(v) for v in g.integers(0, 300 if nseq < 1000 else 24, nseq)]
    lens[0], lens[nseq // 2], lens[-1] = 1, 0, 129
    x = W.varlen_qkv(lens, lens, 4, 2, 128, seed=nseq, device="cuda", k_offset_std=2.0)
    _check_quant(sage, x.q, x.cu_q, x.max_q, 128)
    _check_quant(sage, x.k, x.cu_k, x.max_k, 64, smooth=True)
    qi, qs, ki, ks, bias = _quant_all(sage, x, 128, 64, True)
    out, lse = sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k,
                                             x.max_q, x.max_k, causal=True, q_bias=bias,
                                             out_dtype=torch.float16, return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    rows = None
    if nseq > 100:
        rows = [np.unique(np.array([0, n - 1])) if n > 0 else np.zeros(0, np.int64) for n in lens]
    o_ref, l_ref = _oracle(x, qi, qs, 128, ki, ks, 64, True, bias=bias, rows=rows)
    if rows is None:
        assert_close(f32(out), o_ref)
        assert_close(np_(lse), l_ref, "lse")
    else:
        sel = np.concatenate([int(np_(x.cu_q)[b]) + r for b, r in enumerate(rows) if len(r)])
        assert_close(f32(out)[sel], o_ref[sel])
        assert_close(np_(lse)[:, sel], l_ref[:, sel], "lse")


def test_varlen_back_to_back_calls_share_workspace(sage):
    """Two packed calls on one workspace with no synchronisation between
    them: the second call's attention kernel, launched behind its staging
    pass, reads the staged copy only after that pass completed, so it gives
    what it gives alone on a fresh workspace, bit for bit."""
    lens = [1500, 300, 2600, 64, 900]
    calls = []
    for seed in (81, 82):
        x = W.varlen_qkv(lens, lens, 8, 2, 128, seed=seed, device="cuda", k_offset_std=2.0)
        qi, qs, ki, ks, bias = _quant_all(sage, x, 128, 64, True)
        calls.append((x, qi, qs, ki, ks, bias))
    torch.cuda.synchronize()
    ws = torch.empty(1 << 29, dtype=torch.uint8, device="cuda")

    def run(i, workspace):
        x, qi, qs, ki, ks, bias = calls[i]
        return sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k,
                                             x.max_q, x.max_k, causal=True, q_bias=bias,
                                             return_lse=True, workspace=workspace)

    run(0, ws)
    out, lse = run(1, ws)
    torch.cuda.synchronize()
    ref, ref_lse = run(1, torch.empty(1 << 29, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("heads", [(8, 2), (6, 6), (3, 1)])
def test_varlen_launch_layout(sage, heads):
    """D = 128 packed launches: with an even GQA group a CTA takes 128 query
    rows of two heads sharing a KV head, (total_q / 128 + B) * Hq / 2 CTAs;
    otherwise 256 rows of one head, (total_q / 256 + B) * Hq CTAs.  Both
    give the per-sequence dense result (tested above); this pins which one
    runs."""
    Hq, Hkv = heads
    lens = [300, 1000, 77]
    x = W.varlen_qkv(lens, lens, Hq, Hkv, 128, seed=Hq + 7 * Hkv, device="cuda")
    qi, qs, ki, ks, _ = _quant_all(sage, x, 128, 64, False)
    sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k, x.max_q, x.max_k,
                                  causal=True)
    info = sage.last_launch_info()
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    total, B = sum(lens), len(lens)
    want = (total // 128 + B) * (Hq // 2) if (Hq // Hkv) % 2 == 0 else (total // 256 + B) * Hq
    assert info["kernel"] == "prefill_varlen_kernel"
    assert info["grid"] == (want, 1, 1)
