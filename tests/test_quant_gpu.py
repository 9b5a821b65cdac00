"""GPU parity: sage_quant_int8 against the oracle, bit-exact codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from helpers import f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_quant(sage, x, block, smooth=False, layout="HND"):
    q, s, mu, _ = sage.sage_quant_int8(x, block_tokens=block, smooth=smooth, layout=layout)
    torch.cuda.synchronize()
    xh = f32(x) if layout == "HND" else f32(x).transpose(0, 2, 1, 3)
    if smooth:
        mu_ref = oracle.token_mean(xh)
        # the mean is an exact sum rounded once: bit-exact on these inputs
        assert np.array_equal(np_(mu), mu_ref)
    q_ref, s_ref, _ = oracle.quant_int8(xh, block_tokens=block, smooth=smooth,
                                        mu=np_(mu) if smooth else None)
    assert np.array_equal(np_(s), s_ref), "scales differ"
    assert np.array_equal(np_(q), q_ref), "codes differ in %d places" % int((np_(q) != q_ref).sum())
    return q, s, mu


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("block", [1, 64, 128])
def test_quant_small_bit_exact(sage, D, dtype, block):
    qkv = W.dense_qkv(2, 3, 3, 200, 200, D, seed=D + block, dtype=dtype, device="cuda",
                      k_offset_std=2.0)
    _check_quant(sage, qkv.q, block)
    _check_quant(sage, qkv.k, block, smooth=True)


def test_quant_nhd_strided(sage):
    x = W.dense_qkv(1, 4, 4, 77, 77, 128, seed=5, device="cuda").q     # [B,H,S,D]
    nhd = x.transpose(1, 2).contiguous()                                  # [B,S,H,D]
    q1, s1, _ = _check_quant(sage, nhd, 1, layout="NHD")
    q2, s2, _, _ = sage.sage_quant_int8(x, block_tokens=1)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_quant_degenerate(sage):
    x = torch.zeros((1, 2, 130, 64), dtype=torch.float16, device="cuda")
    x[0, 1, 5:, 3] = 2.5
    q, s, _ = _check_quant(sage, x, 128)
    assert np_(s)[0, 0, 0] == 0.0 and np.all(np_(q)[0, 0] == 0)
    # empty input: nothing to do
    e = torch.zeros((1, 2, 0, 64), dtype=torch.float16, device="cuda")
    q, s, _, _ = sage.sage_quant_int8(e)
    assert q.numel() == 0


def test_quant_row_bias(sage):
    qkv = W.dense_qkv(1, 6, 2, 96, 96, 128, seed=11, device="cuda", k_offset_std=2.0)
    _, _, mu, _ = sage.sage_quant_int8(qkv.k, smooth=True)
    q, s, _, bias = sage.sage_quant_int8(qkv.q, mu_in=mu)
    torch.cuda.synchronize()
    ref = oracle.row_bias(f32(qkv.q), np_(mu))
    scale = np.abs(f32(qkv.q)).sum(-1) * np.abs(np_(mu)).max()
    assert np.all(np.abs(np_(bias) - ref) <= 1e-5 * scale + 1e-6)
    q_ref, s_ref, _ = oracle.quant_int8(f32(qkv.q))
    assert np.array_equal(np_(q), q_ref) and np.array_equal(np_(s), s_ref)


def test_quant_dense_prefill_full_size(sage):
    """Full-size dense-prefill inputs: per-block Q (128) and smoothed K (64), every bit."""
    P = W.WORKLOADS["dense_prefill"].params
    qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                      dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
    _check_quant(sage, qkv.k, 64, smooth=True)
    _check_quant(sage, qkv.q, 128)


def test_quant_chunked_prefill_full_size(sage):
    P = W.WORKLOADS["chunked_prefill"].params
    qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                      dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
    _check_quant(sage, qkv.k, 1, smooth=True)
    _check_quant(sage, qkv.q, 1)


def test_quant_decode_query_full_size(sage):
    P = W.WORKLOADS["paged_decode"].params
    q = W.decode_query(P["B"], P["Hq"], P["D"], seed=P["seed"], device="cuda")
    _check_quant(sage, q[:, :, None, :], 1)


def test_quant_exact_ties_with_non_power_of_two_scales(sage):
    """amax = 127 m gives s = m exactly; x = m (k + 1/2) makes x / s an exact
    tie, where x * fl32(1/m) lands a hair above or below it.  The codes must
    follow the correctly rounded quotient (ties to even), and so must values
    one f16 step either side of each tie."""
    D = 64
    rows = []
    # scales where x * fl32(1/s) misrounds up to 78 of the 254 ties
    for m in (0.4375, 0.9375, 1.625, 3.5, 7.0, 15.0):
        ties = np.array([m * (k + 0.5) for k in range(-127, 127)], np.float32)
        ties = ties[np.abs(ties) < 127 * m]
        vals = np.concatenate([ties, np.nextafter(ties.astype(np.float16), np.float16(np.inf)).astype(np.float32),
                               np.nextafter(ties.astype(np.float16), np.float16(-np.inf)).astype(np.float32)])
        vals = vals[np.abs(vals) < 127 * m]
        vals = vals[(vals.astype(np.float16).astype(np.float32) == vals)]
        for i in range(0, len(vals), D - 1):
            row = np.zeros(D, np.float32)
            chunk = vals[i:i + D - 1]
            row[0] = 127 * m
            row[1:1 + len(chunk)] = chunk
            rows.append(row)
    x = torch.tensor(np.stack(rows)[None, None], dtype=torch.float16, device="cuda")
    _check_quant(sage, x, 1)
    _check_quant(sage, x, 64)


@pytest.mark.parametrize("B,H,Hmu,S,D", [(7, 5, 5, 1, 64), (3, 6, 2, 3, 128), (2, 24, 4, 33, 256),
                                         (1, 9, 3, 2049, 64)])
def test_quant_rows_odd_shapes(sage, B, H, Hmu, S, D):
    """Per-token rows over (b, h, s) with sizes that are not powers of two:
    every row's sequence, head, token and GQA mean group lands in place."""
    x = W.dense_qkv(B, H, H, S, S, D, seed=S + H, device="cuda").q
    mu = torch.randn((B, Hmu, D), dtype=torch.float32, device="cuda",
                     generator=torch.Generator("cuda").manual_seed(B * H))
    q, s, _, bias = sage.sage_quant_int8(x, mu_in=mu)
    torch.cuda.synchronize()
    q_ref, s_ref, _ = oracle.quant_int8(f32(x))
    assert np.array_equal(np_(q), q_ref) and np.array_equal(np_(s), s_ref)
    ref = oracle.row_bias(f32(x), np_(mu))
    scale = np.abs(f32(x)).sum(-1) * np.abs(np_(mu)).max()
    assert np.all(np.abs(np_(bias) - ref) <= 1e-5 * scale + 1e-6)
    # the strided [B,S,H,D] view of the same tensor gives the same rows
    q2, s2, _, _ = sage.sage_quant_int8(x.transpose(1, 2).contiguous(), layout="NHD")
    assert torch.equal(q, q2) and torch.equal(s, s2)


def test_quant_bf16_mean_outside_exact_range(sage):
    """bf16 values the integer path cannot hold (finer than 2^-24, or of
    magnitude 2^16 and up) take the fp64 path; every value here is a
    multiple of 2^-26 and the sums stay below 2^25, so the mean is an exact
    sum rounded once on both sides, bit for bit."""
    g = np.random.default_rng(17)
    B, H, S, D = 1, 2, 256, 64
    x = g.standard_normal((B, H, S, D)).astype(np.float32)
    x = torch.tensor(x).to(torch.bfloat16).float().numpy()
    x[np.abs(x) < 2.0 ** -18] = 0.0                          # keep every unit >= 2^-26
    mant = 1.0 + g.integers(0, 128, size=(B, H, S, D)) / 128.0
    sign = np.where(g.random((B, H, S, D)) < 0.5, -1.0, 1.0)
    tiny = (sign * mant * 2.0 ** -19).astype(np.float32)      # unit 2^-26
    big = (sign * mant * 2.0 ** 16).astype(np.float32)        # 2^16 <= |x| < 2^17
    pick = g.random((B, H, S, D))
    x[..., 0:8] = np.where(pick[..., 0:8] < 0.1, tiny[..., 0:8], x[..., 0:8])
    x[..., 8:16] = np.where(pick[..., 8:16] < 0.1, big[..., 8:16], x[..., 8:16])
    x[..., 16] = tiny[..., 16]
    x[..., 17] = big[..., 17]
    x[..., 18] = np.where(pick[..., 18] < 0.5, tiny[..., 18], big[..., 18])
    xt = torch.tensor(x, dtype=torch.bfloat16, device="cuda")
    assert np.array_equal(f32(xt), x)                          # representable in bf16
    _check_quant(sage, xt, 1, smooth=True)
    _check_quant(sage, xt, 64, smooth=True)


def _tiny_bf16(rng, shape, group_axis_len, block, tiny_groups):
    """bf16 values, N(0,1), whose quantisation groups listed in tiny_groups
    (group index along the token axis, blocks of `block` tokens) are scaled
    so that the group's amax lies in [1e-40, 3.7e-37]: the scale amax / 127
    is then a subnormal float, whose reciprocal can overflow to infinity and
    whose few significand bits can put |x / s| above 127.5 (code 127 by the
    clamp).  Returns an fp32 array of values exactly representable in bf16."""
    x = rng.standard_normal(shape).astype(np.float32)
    for g in tiny_groups:
        t0, t1 = g * block, min((g + 1) * block, group_axis_len)
        sl = x[..., t0:t1, :]
        amax = np.abs(sl).max(axis=(-2, -1), keepdims=True)
        target = 10.0 ** rng.uniform(-40.0, np.log10(3.7e-37), size=amax.shape)
        x[..., t0:t1, :] = sl / amax * target
    return torch.tensor(x).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("block", [1, 64, 128])
def test_quant_bf16_subnormal_scales(sage, block):
    """Groups whose bf16 amax is below 3.7e-37 (subnormal scale): every code
    and scale bit-exact against the oracle, next to ordinary groups in the
    same tensor, per token and per block."""
    rng = np.random.default_rng(100 + block)
    B, H, S, D = 2, 3, 300, 128
    ngroups = (S + block - 1) // block
    tiny = [g for g in range(ngroups) if g % 3 != 1]          # some groups stay ordinary
    x = _tiny_bf16(rng, (B, H, S, D), S, block, tiny)
    xt = torch.tensor(x, dtype=torch.bfloat16, device="cuda")
    assert np.array_equal(f32(xt), x)
    q, s, _ = _check_quant(sage, xt, block)
    sub = np_(s)[np_(s) != 0]
    assert (sub < 1.17549435e-38).any() and (sub > 1e-3).any()


def test_quant_bf16_subnormal_scales_decode_query(sage):
    """A decode step's query (few rows: the small-CTA per-token path) with
    tiny bf16 heads, bit-exact; and the same query handed to the fused
    decode from pinned host memory, where the library quantises it once
    into the workspace (codes at the offsets the header declares)."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, ctx = 2, 24, 4, 256, 512
    x = _tiny_bf16(rng, (B, Hq, 1, D), 1, 1, [0])
    x[:, ::5] = rng.standard_normal((B, x[:, ::5].shape[1], 1, D))   # a few ordinary heads
    x = torch.tensor(x).to(torch.bfloat16).float().numpy()
    qd = torch.tensor(x, dtype=torch.bfloat16, device="cuda")
    _check_quant(sage, qd, 1)
    q_ref, s_ref, _ = oracle.quant_int8(x, block_tokens=1)
    cache = W.paged_cache(B, Hkv, D, [ctx] * B, seed=3, device="cuda")
    q_host = qd[:, :, 0].cpu().pin_memory()
    S = sage.decode_segments_used(ctx, 14)
    assert S > 8                                              # partials + combine
    # sized for the 14 segments asked for (the binding's check); the library
    # lays the workspace out for the S segments it actually uses
    ws = torch.zeros(sage.decode_workspace_size(B, Hq, D, 14), dtype=torch.uint8, device="cuda")
    sage.sage_attn_decode_paged_q16(q_host, cache.k_cache, cache.v_cache, cache.k_scale,
                                    cache.v_scale, cache.block_table, cache.lens, ctx,
                                    num_segments=14, workspace=ws)
    assert sage.last_launch_info()["launches"] == 3       # quant, decode, combine
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    up = lambda n: (n + 255) // 256 * 256
    rows = B * Hq * S
    qc_off = up(rows * D * 4) + up(rows * 4)                     # after partials and LSEs
    qs_off = qc_off + up(B * Hq * D)
    w = np_(ws)
    codes = w[qc_off:qc_off + B * Hq * D].view(np.int8).reshape(B, Hq, D)
    scales = w[qs_off:qs_off + B * Hq * 4].view(np.float32).reshape(B, Hq)
    assert np.array_equal(codes, q_ref[:, :, 0]) and np.array_equal(scales, s_ref[:, :, 0])


def test_quant_varlen_bf16_subnormal_scales(sage):
    """The packed-batch kernels with tiny bf16 groups: per-sequence codes and
    scales bit-exact, per token and per 64-token block."""
    rng = np.random.default_rng(9)
    lens = [70, 130, 1, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    H, D = 2, 128
    x = rng.standard_normal((cu[-1], H, D)).astype(np.float32)
    for b in range(len(lens)):            # in each sequence, the second half tiny
        t0, t1 = cu[b] + lens[b] // 2, cu[b + 1]
        if t1 > t0:
            sl = x[t0:t1]
            x[t0:t1] = sl / np.abs(sl).max() * 10.0 ** rng.uniform(-40, -36.5)
    x = torch.tensor(x).to(torch.bfloat16).float().numpy()
    xt = torch.tensor(x, dtype=torch.bfloat16, device="cuda")
    cu_t = torch.tensor(cu, device="cuda")
    for block in (1, 64):
        q, s, _, _ = sage.sage_quant_int8_varlen(xt, cu_t, max(lens), block_tokens=block)
        torch.cuda.synchronize()
        q_ref, s_ref, _ = oracle.quant_int8_varlen(x, cu, block_tokens=block)
        assert np.array_equal(np_(q), q_ref)
        sc = np_(s)
        for b in range(len(lens)):
            g0 = cu[b] if block == 1 else cu[b] // block + b
            assert np.array_equal(sc[:, g0:g0 + s_ref[b].shape[1]], s_ref[b])
