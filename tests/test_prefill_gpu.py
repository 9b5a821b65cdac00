"""GPU parity: the tcgen05 prefill kernel against the oracle.

Raw INT32 scores (through the debug dump of the same tile path) must be
bit-exact; outputs and LSE within rel-L2 5e-3 / max-abs 2e-3 of the
oracle's fp64 quantized-math result.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _quant(sage, qkv, q_block, k_block, smooth):
    qi, qs, _, _ = sage.sage_quant_int8(qkv.q, block_tokens=q_block)
    ki, ks, mu, _ = sage.sage_quant_int8(qkv.k, block_tokens=k_block, smooth=smooth)
    bias = None
    if smooth:
        _, _, _, bias = sage.sage_quant_int8(qkv.q, block_tokens=q_block, mu_in=mu)
    return qi, qs, ki, ks, mu, bias


def _oracle(qi, qs, qb, ki, ks, kb, v, causal, bias=None, prefix=None, rows=None):
    pre = None
    if prefix is not None:
        pre = dict(k_cache=np_(prefix.k_cache), v_cache=np_(prefix.v_cache),
                   k_scale=np_(prefix.k_scale), v_scale=np_(prefix.v_scale),
                   block_table=np_(prefix.block_table), lens=np_(prefix.lens))
    return oracle.prefill(np_(qi), np_(qs), qb, np_(ki), np_(ks), kb, f32(v), causal=causal,
                          q_bias=None if bias is None else np_(bias).astype(np.float64),
                          prefix=pre, rows=rows)


def _prefix_dict(c, max_len):
    return dict(k_cache=c.k_cache, v_cache=c.v_cache, k_scale=c.k_scale, v_scale=c.v_scale,
                block_table=c.block_table, lens=c.lens, max_len=max_len)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_raw_scores_bit_exact(sage, D, causal):
    B, Hq, Hkv, S = 1, 2, 1, 200
    qkv = W.dense_qkv(B, Hq, Hkv, S, S, D, seed=D, device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    dbg = torch.full((B, Hq, S, S), -(2 ** 31), dtype=torch.int32, device="cuda")
    sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=causal, debug_scores=dbg)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    d = np_(dbg)
    for h in range(Hq):
        ref = oracle.qk_int32(np_(qi)[0, h], np_(ki)[0, h // 2])
        if causal:
            vis = np.tril(np.ones((S, S), bool))
            assert np.array_equal(d[0, h][vis], ref[vis])
            assert np.all(d[0, h][~vis] == -(2 ** 31))
        else:
            assert np.array_equal(d[0, h], ref)


def test_prefill_adversarial_int32_extremes(sage):
    """+-127 codes at D = 256: every raw score is +-4,129,024 exactly."""
    B, H, S, D = 1, 1, 128, 256
    qi = torch.full((B, H, S, D), 127, dtype=torch.int8, device="cuda")
    qi[:, :, 1::2] = -127
    ki = torch.full((B, H, S, D), 127, dtype=torch.int8, device="cuda")
    ki[:, :, 64:] = -127
    qs = torch.full((B, H, S), 1e-4, dtype=torch.float32, device="cuda")
    ks = torch.full((B, H, S), 1e-4, dtype=torch.float32, device="cuda")
    v = torch.randn((B, H, S, D), dtype=torch.float16, device="cuda")
    dbg = torch.zeros((B, H, S, S), dtype=torch.int32, device="cuda")
    sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, v, causal=False, debug_scores=dbg)
    torch.cuda.synchronize()
    ref = oracle.qk_int32(np_(qi)[0, 0], np_(ki)[0, 0])
    assert np.abs(ref).max() == 256 * 127 * 127
    assert np.array_equal(np_(dbg)[0, 0], ref)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S", [128, 200, 333])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("vdt", ["fp16", "bf16"])
def test_prefill_small_per_token(sage, D, S, causal, vdt):
    B, Hq, Hkv = 2, 4, 2
    qkv = W.dense_qkv(B, Hq, Hkv, S, S, D, seed=S + D, dtype="fp16", device="cuda", v_dtype=vdt)
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=causal,
                                      out_dtype=torch.float16, return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    o_ref, l_ref = _oracle(qi, qs, 1, ki, ks, 1, qkv.v, causal)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_per_block_smooth_k(sage, D):
    B, H, S = 1, 3, 700
    qkv = W.dense_qkv(B, H, H, S, S, D, seed=7, device="cuda", k_offset_std=2.0)
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
    for causal in (False, True):
        out, lse = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, causal=causal,
                                          q_bias=bias, out_dtype=torch.float16, return_lse=True)
        torch.cuda.synchronize()
        o_ref, l_ref = _oracle(qi, qs, 128, ki, ks, 64, qkv.v, causal, bias=bias)
        assert_close(f32(out), o_ref, "causal=%s" % causal)
        assert_close(np_(lse), l_ref, "lse causal=%s" % causal)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("P", [0, 100, 256])
def test_prefill_paged_prefix(sage, D, P):
    B, Hq, Hkv, Sc = 2, 6, 1, 150
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=P + D, dtype="bf16", device="cuda",
                      k_offset_std=2.0)
    lens = [P, max(P - 37, 0)]
    c = W.paged_cache(B, Hkv, D, [max(x, 1) for x in lens], seed=P + 1, device="cuda",
                      extra_blocks=3)
    c.lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 1, 1, True)
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True, q_bias=bias,
                                      prefix=_prefix_dict(c, max(max(lens), 1)),
                                      out_dtype=torch.float16, return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    o_ref, l_ref = _oracle(qi, qs, 1, ki, ks, 1, qkv.v, True, bias=bias, prefix=c)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_repeatable(sage, D):
    """Repeated calls give bit-identical outputs and LSE: the kernel has no
    order-dependent reduction, so any difference is a read that raced a
    tensor-core write (e.g. the epilogue reading O before the last P.V)."""
    B, Hq, Hkv, Sc, P = 1, 8, 2, 1024, 2048
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=D, dtype="bf16", device="cuda",
                      k_offset_std=1.0)
    c = W.paged_cache(B, Hkv, D, [P], seed=D + 1, device="cuda")
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
    outs = []
    for _ in range(6):
        outs.append(sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, causal=True,
                                           q_bias=bias, prefix=_prefix_dict(c, P),
                                           return_lse=True))
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0])
        assert torch.equal(l, outs[0][1])


def test_prefill_paged_prefix_raw_scores(sage):
    B, Hq, Hkv, Sc, D, P = 1, 2, 1, 64, 256, 77
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=3, dtype="bf16", device="cuda")
    c = W.paged_cache(B, Hkv, D, [P], seed=4, device="cuda", extra_blocks=2)
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    dbg = torch.full((B, Hq, Sc, P + Sc), -(2 ** 31), dtype=torch.int32, device="cuda")
    sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True,
                           prefix=_prefix_dict(c, P), debug_scores=dbg)
    torch.cuda.synchronize()
    keys = np.concatenate([oracle.gather_paged(np_(c.k_cache), np_(c.block_table)[0], P, 0),
                           np_(ki)[0, 0]], 0)
    for h in range(Hq):
        ref = oracle.qk_int32(np_(qi)[0, h], keys)
        vis = np.arange(P + Sc)[None, :] <= (np.arange(Sc)[:, None] + P)
        assert np.array_equal(np_(dbg)[0, h][vis], ref[vis])


def test_prefill_launch_record(sage):
    qkv = W.dense_qkv(1, 2, 2, 256, 256, 128, seed=1, device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True)
    info = sage.last_launch_info()
    # two 128-row query tiles per CTA at D = 128: one softmax warpgroup each,
    # plus a warpgroup holding the producer and MMA warps
    # (one linear index over query tiles x heads x batches)
    assert info["kernel"] == "prefill_kernel" and info["grid"] == (2, 1, 1)
    assert info["block"] == (384, 1, 1)


def test_tiny_prefill_full(sage):
    """The B1 H2 S128 D64 per-token non-causal workload, every output."""
    P = W.WORKLOADS["tiny_prefill"].params
    qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                      dtype=P["dtype"], device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=False,
                                      sm_scale=1 / 8, return_lse=True)
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(qi, qs, 1, ki, ks, 1, qkv.v, False)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


def test_dense_prefill_full_size_sampled(sage):
    """B2 H32 S16384 D128 causal per-block + smooth_k + LSE: sampled rows vs the oracle."""
    P = W.WORKLOADS["dense_prefill"].params
    qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                      dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
    out, lse = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, causal=True, q_bias=bias,
                                      return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, 1, 127, 128, 8191, 16383],
                                   rng.choice(P["S"], 58, replace=False)]))
    pairs = [(0, 0), (0, 17), (1, 5), (1, 31)]
    for b, h in pairs:
        sub = lambda t, hh=h: t[b:b + 1, hh:hh + 1]
        o_ref, l_ref = oracle.prefill(np_(sub(qi)), np_(sub(qs)), 128, np_(sub(ki)), np_(sub(ks)),
                                      64, f32(sub(qkv.v)), causal=True,
                                      q_bias=np_(sub(bias)).astype(np.float64), rows=rows)
        assert_close(f32(out)[b, h, rows], o_ref[0, 0], "b%d h%d" % (b, h))
        assert_close(np_(lse)[b, h, rows], l_ref[0, 0], "lse b%d h%d" % (b, h))


def test_chunked_prefill_full_size_sampled(sage):
    """B1 Hq24 Hkv4 D256: 2048 new tokens over a 16384-token paged INT8 prefix."""
    P = W.WORKLOADS["chunked_prefill"].params
    qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                      dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
    c = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["prefix"]], seed=P["seed"], device="cuda")
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 1, 1, True)
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True, q_bias=bias,
                                      prefix=_prefix_dict(c, P["prefix"]), return_lse=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([[0, 63, 64, 2047], rng.choice(P["S"], 28, replace=False)]))
    pre = dict(k_cache=np_(c.k_cache), v_cache=np_(c.v_cache), k_scale=np_(c.k_scale),
               v_scale=np_(c.v_scale), block_table=np_(c.block_table), lens=np_(c.lens))
    for h in (0, 5, 6, 23):
        g = h // 6
        o_ref, l_ref = oracle.prefill(np_(qi)[:, h:h + 1], np_(qs)[:, h:h + 1], 1,
                                      np_(ki)[:, g:g + 1], np_(ks)[:, g:g + 1], 1,
                                      f32(qkv.v)[:, g:g + 1], causal=True,
                                      q_bias=np_(bias)[:, h:h + 1].astype(np.float64),
                                      prefix=dict(pre, k_cache=pre["k_cache"][:, g:g + 1],
                                                  v_cache=pre["v_cache"][:, g:g + 1],
                                                  k_scale=pre["k_scale"][:, g:g + 1],
                                                  v_scale=pre["v_scale"][:, g:g + 1]),
                                      rows=rows)
        assert_close(f32(out)[0, h, rows], o_ref[0, 0], "h%d" % h)
        assert_close(np_(lse)[0, h, rows], l_ref[0, 0], "lse h%d" % h)


def test_prefill_bundled_order_covers_every_tile(sage):
    """Eight (batch, head) pairs of 16384 keys at D = 256 run in L2-sized
    bundles of three (3 + 3 + 2): every output row is written exactly by
    its own tile (rows pre-filled with NaN) and sampled rows of every pair
    match the oracle."""
    B, H, S, D = 1, 8, 16384, 256
    qkv = W.dense_qkv(B, H, H, S, S, D, seed=41, device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    out = torch.full((B, H, S, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = np.array([0, 127, 128, 5000, 16383])
    for h in range(H):
        o_ref, l_ref = oracle.prefill(np_(qi)[:, h:h + 1], np_(qs)[:, h:h + 1], 1,
                                      np_(ki)[:, h:h + 1], np_(ks)[:, h:h + 1], 1,
                                      f32(qkv.v)[:, h:h + 1], causal=True, rows=rows)
        assert_close(f32(out)[0, h, rows], o_ref[0, 0], "h%d" % h)
        assert_close(np_(lse)[0, h, rows], l_ref[0, 0], "lse h%d" % h)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("vdt", ["fp16", "bf16"])
def test_prefill_smooth_v(sage, D, vdt):
    """smooth_v: the V mean (bit-exact against the oracle's token mean) is
    subtracted before P.V and added back; outputs against the oracle's
    smooth_v result.  V carries a common offset (outputs stay below 2, so f16
    output rounding stays inside the tolerance)."""
    B, Hq, Hkv, S = 2, 4, 2, 333
    qkv = W.dense_qkv(B, Hq, Hkv, S, S, D, seed=D + 61, device="cuda", v_dtype=vdt)
    v = (qkv.v.float() * 0.25 + 1.25).to(qkv.v.dtype)
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    mu = torch.empty((B, Hkv, D), dtype=torch.float32, device="cuda")
    for causal in (False, True):
        out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, v, causal=causal,
                                          out_dtype=torch.float16, return_lse=True,
                                          smooth_v=True, v_mean=mu)
        torch.cuda.synchronize()
        assert sage.check_device_status()[0] == 0
        assert np.array_equal(np_(mu), oracle.token_mean(f32(v)))
        o_ref, l_ref = oracle.prefill(np_(qi), np_(qs), 1, np_(ki), np_(ks), 1, f32(v),
                                      causal=causal, smooth_v=True)
        assert_close(f32(out), o_ref, "causal=%s" % causal)
        assert_close(np_(lse), l_ref, "lse causal=%s" % causal)


def test_prefill_smooth_v_paged_prefix(sage):
    """smooth_v over a paged INT8 prefix: the chunk's V mean comes off the
    prefix values too, so the identity P (V - mu) + mu = P V still holds."""
    B, Hq, Hkv, Sc, D, P = 1, 6, 1, 150, 256, 200
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=71, dtype="bf16", device="cuda")
    v = (qkv.v.float() * 0.25 + 0.75).to(qkv.v.dtype)
    c = W.paged_cache(B, Hkv, D, [P], seed=72, device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    out = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, v, causal=True,
                                 prefix=_prefix_dict(c, P), out_dtype=torch.float16,
                                 smooth_v=True)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    pre = dict(k_cache=np_(c.k_cache), v_cache=np_(c.v_cache), k_scale=np_(c.k_scale),
               v_scale=np_(c.v_scale), block_table=np_(c.block_table), lens=np_(c.lens))
    o_ref, _ = oracle.prefill(np_(qi), np_(qs), 1, np_(ki), np_(ks), 1, f32(v), causal=True,
                              prefix=pre, smooth_v=True)
    assert_close(f32(out), o_ref)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("vdt", ["fp16", "bf16"])
@pytest.mark.parametrize("smooth_v", [False, True])
@pytest.mark.parametrize("with_prefix", [False, True])
def test_prefill_nhd_layout_equals_hnd(sage, D, vdt, smooth_v, with_prefix):
    """[P3]'s tensor_layout: V given as [B, Sk, Hkv, D] and the output written
    as [B, Sq, Hq, D] give, bit for bit, the HND result transposed -- f16 V
    read in place (a 4-D tensor map), bf16 V and smooth_v through the
    staging pass, with and without a paged prefix."""
    B, Hq, Hkv, S = 2, 4, 2, 300
    qkv = W.dense_qkv(B, Hq, Hkv, S, S, D, seed=D + 7, dtype=vdt, device="cuda", k_offset_std=2.0)
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 1, 64, True)
    prefix = None
    if with_prefix:
        c = W.paged_cache(B, Hkv, D, [100, 37], seed=D, device="cuda", extra_blocks=3)
        prefix = _prefix_dict(c, 100)
    v_nhd = qkv.v.transpose(1, 2).contiguous()
    out_h, lse_h = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 64, qkv.v, causal=True, q_bias=bias,
                                          prefix=prefix, return_lse=True, smooth_v=smooth_v)
    out_n, lse_n = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 64, v_nhd, causal=True, q_bias=bias,
                                          prefix=prefix, return_lse=True, smooth_v=smooth_v,
                                          layout="NHD")
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert tuple(out_n.shape) == (B, S, Hq, D)
    assert torch.equal(out_n, out_h.transpose(1, 2)) and torch.equal(lse_n, lse_h)


def test_prefill_nhd_dense_workload_shape_sampled(sage):
    """NHD at the dense-prefill shape class (f16 V read in place through the
    4-D map, per-block Q/K, smooth_k, causal, LSE): sampled rows against
    the oracle, and equal to the HND call."""
    B, Hq, Hkv, S, D = 1, 8, 8, 4096, 128
    qkv = W.dense_qkv(B, Hq, Hkv, S, S, D, seed=91, device="cuda", k_offset_std=2.0)
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
    v_nhd = qkv.v.transpose(1, 2).contiguous()
    out_n, lse_n = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, v_nhd, causal=True,
                                          q_bias=bias, return_lse=True, layout="NHD")
    out_h = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, causal=True, q_bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(out_n.transpose(1, 2), out_h)
    rows = np.array([0, 1, 127, 128, 2047, 4095])
    o_ref, l_ref = _oracle(qi, qs, 128, ki, ks, 64, qkv.v, True, bias=bias, rows=rows)
    assert_close(f32(out_n)[:, rows].transpose(0, 2, 1, 3), o_ref)
    assert_close(np_(lse_n)[:, :, rows], l_ref, "lse")


def _split_case(seed, causal, dtype="f16"):
    # 32 query tiles of 128 rows (1 x 8 heads x 512 rows) over 4096 keys at
    # D = 256: the whole grid is one partial wave on 152 SMs, so every tile
    # is split by key range (3 parts with the causal mask, 4 without) and
    # merged by the merge kernel
    return W.dense_qkv(1, 8, 2, 512, 4096, 256, seed=seed, dtype=dtype, device="cuda",
                       k_offset_std=2.0)


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_tail_split_matches_oracle(sage, causal):
    """The last wave's query tiles split by key range ("INT8 QK MMAC on gfx936
    DCU", section 4: split-K with an LSE combine) give the oracle's result on
    sampled rows of every head, stay within rounding of the unsplit launch,
    and dump the same raw INT32 scores."""
    qkv = _split_case(61, causal)
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
    kw = dict(causal=causal, q_bias=bias, out_dtype=torch.float16, return_lse=True)
    S, Sk = 512, 4096
    dbg_s = torch.full((1, 8, S, Sk), -(2 ** 31), dtype=torch.int32, device="cuda")
    out, lse = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, debug_scores=dbg_s, **kw)
    info = sage.last_launch_info()
    k = 3 if causal else 4
    assert info["kernel"] == "prefill_kernel" and info["grid"] == (32 * k, 1, 1)
    assert info["launches"] == 3  # staging, attention, merge
    dbg_u = torch.full_like(dbg_s, -(2 ** 31))
    out_u, lse_u = sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, debug_scores=dbg_u,
                                          tail_split=False, **kw)
    assert sage.last_launch_info()["grid"] == (32, 1, 1)
    assert sage.last_launch_info()["launches"] == 2
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(dbg_s, dbg_u)
    assert_close(f32(out), f32(out_u), "split vs unsplit", rel=1e-3, abs_=1e-3)
    assert_close(np_(lse), np_(lse_u), "lse split vs unsplit", rel=1e-5, abs_=1e-4)
    rows = np.array([0, 1, 127, 128, 255, 256, 383, 384, 511])
    o_ref, l_ref = _oracle(qi, qs, 128, ki, ks, 64, qkv.v, causal, bias=bias, rows=rows)
    assert_close(f32(out)[:, :, rows], o_ref)
    assert_close(np_(lse)[:, :, rows], l_ref, "lse")


@pytest.mark.parametrize("smooth_v", [False, True])
def test_prefill_tail_split_nhd_prefix_smooth_v(sage, smooth_v):
    """The merge kernel's other output paths: NHD output rows, bf16 output,
    the smooth_v mean added back, rows of a causal chunk over a paged
    prefix; equal within rounding to the unsplit launch."""
    B, Hq, Hkv, Sc, D, Pn = 1, 8, 2, 256, 256, 3840
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=63, dtype="bf16", device="cuda",
                      k_offset_std=2.0)
    c = W.paged_cache(B, Hkv, D, [Pn], seed=64, device="cuda")
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 1, 1, True)
    v_nhd = qkv.v.transpose(1, 2).contiguous()
    kw = dict(causal=True, q_bias=bias, prefix=_prefix_dict(c, Pn), return_lse=True,
              smooth_v=smooth_v, layout="NHD")
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, v_nhd, **kw)
    split_grid = sage.last_launch_info()["grid"][0]
    out_u, lse_u = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, v_nhd, tail_split=False, **kw)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert split_grid > 16  # 16 query tiles, each split
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (B, Sc, Hq, D)
    assert_close(f32(out), f32(out_u), "split vs unsplit", rel=2e-3, abs_=2e-3)
    assert_close(np_(lse), np_(lse_u), "lse split vs unsplit", rel=1e-5, abs_=1e-4)


def test_prefill_tail_split_ragged_prefix(sage):
    """Two sequences whose paged prefixes differ in length (3840 and 2200
    tokens): their query tiles have different key counts, so the split
    parts cover different key ranges; both sequences match the oracle on
    sampled rows and the unsplit launch within rounding."""
    B, Hq, Hkv, Sc, D = 2, 4, 1, 256, 256
    lens = [3840, 2200]
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=71, dtype="bf16", device="cuda",
                      k_offset_std=2.0)
    c = W.paged_cache(B, Hkv, D, lens, seed=72, device="cuda", extra_blocks=3)
    qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 1, 1, True)
    kw = dict(causal=True, q_bias=bias, prefix=_prefix_dict(c, max(lens)), return_lse=True,
              out_dtype=torch.float16)
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, **kw)
    grid = sage.last_launch_info()["grid"][0]
    out_u, lse_u = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, tail_split=False, **kw)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert grid > 16  # 16 query tiles, each split
    assert_close(f32(out), f32(out_u), "split vs unsplit", rel=1e-3, abs_=1e-3)
    assert_close(np_(lse), np_(lse_u), "lse split vs unsplit", rel=1e-5, abs_=1e-4)
    rows = np.array([0, 1, 127, 128, 200, 255])
    o_ref, l_ref = _oracle(qi, qs, 1, ki, ks, 1, qkv.v, True, bias=bias, prefix=c, rows=rows)
    assert_close(f32(out)[:, :, rows], o_ref)
    assert_close(np_(lse)[:, :, rows], l_ref, "lse")


@pytest.mark.parametrize("D", [128, 256])
def test_prefill_bad_prefix_page_sets_error_word(sage, D):
    """A block-table entry out of range inside a sequence's prefix is never
    read: the staging pass sets the error word's bad-block bit and stages
    zero rows for that page; the other sequence, whose table is valid,
    still matches the oracle."""
    B, Hq, Hkv, Sc = 2, 2, 1, 64
    lens = [200, 150]
    qkv = W.dense_qkv(B, Hq, Hkv, Sc, Sc, D, seed=D + 3, device="cuda")
    c = W.paged_cache(B, Hkv, D, lens, seed=D + 4, device="cuda", extra_blocks=2)
    c.lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qi, qs, ki, ks, _, _ = _quant(sage, qkv, 1, 1, False)
    bad = c.block_table.clone()
    bad[0, 3] = c.k_cache.shape[0] + 100
    c_bad = W.PagedCache(c.k_cache, c.v_cache, c.k_scale, c.v_scale, bad, c.lens)
    assert sage.check_device_status()[0] == 0
    out, lse = sage.sage_attn_prefill(qi, qs, 1, ki, ks, 1, qkv.v, causal=True,
                                      prefix=_prefix_dict(c_bad, max(lens)),
                                      out_dtype=torch.float16, return_lse=True)
    st, word = sage.check_device_status()
    assert st == sage.SAGE_ERR_BAD_BLOCK and word & 2
    o_ref, l_ref = _oracle(qi[1:], qs[1:], 1, ki[1:], ks[1:], 1, qkv.v[1:], True,
                           prefix=W.PagedCache(c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                               c.block_table[1:], c.lens[1:]))
    assert_close(f32(out)[1:], o_ref)
    assert_close(np_(lse)[1:], l_ref, "lse")


def _fuzz_case(i):
    """Seeded random prefill configuration i (shapes, head dim, GQA group,
    masks, scale granularity, smooth_k / smooth_v, layout, V dtype, paged
    prefix and ragged prefix lengths)."""
    rng = np.random.default_rng(1000 + i)
    D = int(rng.choice([64, 128, 256]))
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 3]))
    B = int(rng.integers(1, 3))
    Sq = int(rng.integers(1, 300))
    P = int(rng.choice([0, int(rng.integers(1, 400))]))
    Sc = int(rng.integers(0 if P > 0 else 1, 300))
    if i % 8 == 4:  # keys from the paged prefix only (Sk = 0)
        P, Sc = max(P, 100), 0
    return dict(D=D, Hkv=Hkv, Hq=Hq, B=B, Sq=Sq, Sc=Sc, P=P,
                causal=bool(rng.integers(0, 2)), qb=int(rng.choice([1, 128])),
                kb=int(rng.choice([1, 64])), smooth_k=bool(rng.integers(0, 2)) and Sc > 0,
                smooth_v=bool(rng.integers(0, 2)) and Sc > 0, nhd=bool(rng.integers(0, 2)),
                vdt=str(rng.choice(["fp16", "bf16"])), seed=2000 + i)


@pytest.mark.parametrize("i", range(24))
def test_prefill_random_configurations(sage, i):
    """Seeded random configurations against the oracle on every row:
    outputs and LSE within tolerance (empty rows: o = 0, lse = -inf)."""
    c = _fuzz_case(i)
    B, Hq, Hkv, Sq, Sc, D, P = c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sc"], c["D"], c["P"]
    qkv = W.dense_qkv(B, Hq, Hkv, Sq, max(Sc, 1), D, seed=c["seed"], dtype=c["vdt"],
                      device="cuda", k_offset_std=2.0)
    qi, qs, _, _ = sage.sage_quant_int8(qkv.q, block_tokens=c["qb"])
    bias = None
    if Sc > 0:
        k = qkv.k[:, :, :Sc].contiguous()
        v = qkv.v[:, :, :Sc].contiguous()
        ki, ks, mu, _ = sage.sage_quant_int8(k, block_tokens=c["kb"], smooth=c["smooth_k"])
        if c["smooth_k"]:
            _, _, _, bias = sage.sage_quant_int8(qkv.q, block_tokens=c["qb"], mu_in=mu)
    else:
        ki = torch.empty((B, Hkv, 0, D), dtype=torch.int8, device="cuda")
        ks = torch.empty((B, Hkv, 0), dtype=torch.float32, device="cuda")
        v = torch.empty((B, Hkv, 0, D), dtype=qkv.v.dtype, device="cuda")
    prefix, pc = None, None
    if P > 0:
        lens = [P] + [int(x) for x in np.random.default_rng(c["seed"]).integers(0, P + 1, B - 1)]
        pc = W.paged_cache(B, Hkv, D, [max(x, 1) for x in lens], seed=c["seed"] + 1,
                           device="cuda", extra_blocks=2)
        pc.lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
        prefix = _prefix_dict(pc, P)
    v_in = v.transpose(1, 2).contiguous() if c["nhd"] else v
    out, lse = sage.sage_attn_prefill(qi, qs, c["qb"], ki, ks, c["kb"], v_in, causal=c["causal"],
                                      q_bias=bias, prefix=prefix, out_dtype=torch.float16,
                                      return_lse=True, smooth_v=c["smooth_v"],
                                      layout="NHD" if c["nhd"] else "HND")
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    if c["nhd"]:
        out = out.transpose(1, 2)
    pre = None
    if pc is not None:
        pre = dict(k_cache=np_(pc.k_cache), v_cache=np_(pc.v_cache), k_scale=np_(pc.k_scale),
                   v_scale=np_(pc.v_scale), block_table=np_(pc.block_table), lens=np_(pc.lens))
    o_ref, l_ref = oracle.prefill(np_(qi), np_(qs), c["qb"], np_(ki), np_(ks), c["kb"], f32(v),
                                  causal=c["causal"],
                                  q_bias=None if bias is None else np_(bias).astype(np.float64),
                                  prefix=pre, smooth_v=c["smooth_v"])
    assert_close(f32(out), o_ref, "case %d %s" % (i, c))
    assert_close(np_(lse), l_ref, "lse case %d" % i)


@pytest.mark.parametrize("form", ["keys_only", "prefix_bf16", "tail_split"])
def test_prefill_back_to_back_calls_share_workspace(sage, form):
    """Two calls on one workspace, queued with no synchronisation between
    them: the second call's attention kernel starts while its staging pass
    may still run, and its merge while the attention kernel may still run.
    Each reads only after the grid ahead of it has completed, so the second
    call gives, bit for bit, what it gives alone on a fresh workspace."""
    D, S, Sk, Hq, Hkv, dt = {"keys_only": (128, 2048, 2048, 8, 8, "fp16"),
                             "prefix_bf16": (128, 1024, 1024, 8, 2, "bf16"),
                             "tail_split": (256, 512, 4096, 8, 2, "fp16")}[form]
    P = 3000 if form == "prefix_bf16" else 0
    calls = []
    for seed in (71, 72):
        qkv = W.dense_qkv(1, Hq, Hkv, S, Sk, D, seed=seed, dtype=dt, device="cuda",
                          k_offset_std=2.0)
        qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)
        kw = dict(causal=True, q_bias=bias, return_lse=True)
        if P:
            c = W.paged_cache(1, Hkv, D, [P], seed=seed + 10, device="cuda")
            kw["prefix"] = _prefix_dict(c, P)
        calls.append((qi, qs, ki, ks, qkv.v, kw))
    torch.cuda.synchronize()
    ws = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")

    def run(i, workspace):
        qi, qs, ki, ks, v, kw = calls[i]
        return sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, v, workspace=workspace, **kw)

    run(0, ws)
    out, lse = run(1, ws)
    if form == "tail_split":
        assert sage.last_launch_info()["launches"] == 3  # staging, attention, merge
    torch.cuda.synchronize()
    ref, ref_lse = run(1, torch.empty(1 << 30, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("form", ["dense", "tail_split", "varlen_pairs"])
def test_prefill_captured_in_a_cuda_graph(sage, form):
    """A prefill call captured into a CUDA graph and replayed gives, bit for
    bit, the eager call's output and LSE: the staging pass, the attention
    kernel launched as its programmatic dependent, and (tail split) the
    merge launched behind that, all inside one graph."""
    stream = torch.cuda.Stream()
    ws = torch.empty(1 << 29, dtype=torch.uint8, device="cuda")
    if form == "varlen_pairs":
        lens = [700, 130, 1500]
        x = W.varlen_qkv(lens, lens, 8, 2, 128, seed=91, device="cuda", k_offset_std=2.0)
        qi, qs, _, _ = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, block_tokens=128)
        ki, ks, mu, _ = sage.sage_quant_int8_varlen(x.k, x.cu_k, x.max_k, block_tokens=64,
                                                    smooth=True)
        _, _, _, bias = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, block_tokens=128,
                                                    mu_in=mu)

        def call():
            return sage.sage_attn_prefill_varlen(qi, qs, 128, ki, ks, 64, x.v, x.cu_q, x.cu_k,
                                                 x.max_q, x.max_k, causal=True, q_bias=bias,
                                                 return_lse=True, workspace=ws, stream=stream)
    else:
        D, S, Sk = (128, 1024, 1024) if form == "dense" else (256, 512, 4096)
        qkv = W.dense_qkv(1, 8, 2, S, Sk, D, seed=92, device="cuda", k_offset_std=2.0)
        qi, qs, ki, ks, mu, bias = _quant(sage, qkv, 128, 64, True)

        def call():
            return sage.sage_attn_prefill(qi, qs, 128, ki, ks, 64, qkv.v, causal=True,
                                          q_bias=bias, return_lse=True, workspace=ws,
                                          stream=stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ref, ref_lse = call()
        ref, ref_lse = ref.clone(), ref_lse.clone()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        out, lse = call()
    for _ in range(2):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)
