"""GPU parity: the KV-cache append (per-token, per-KV-head quantisation
scattered into the paged INT8 cache) against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _fresh_cache(nblk, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    kc = torch.randint(-127, 128, (nblk, H, D // 16, 16, 16), generator=g, dtype=torch.int8)
    vc = torch.randint(-127, 128, (nblk, H, D // 16, 16, 16), generator=g, dtype=torch.int8)
    ks = torch.rand((nblk, H, 16), generator=g) * 0.015 + 0.005
    vs = torch.rand((nblk, H, 16), generator=g) * 0.015 + 0.005
    return [t.cuda() for t in (kc, vc, ks, vs)]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 37])
def test_kv_append_bit_exact(sage, D, dtype, n):
    B, H, nblk = 3, 4, 40
    g = torch.Generator().manual_seed(D + n)
    k_new = (torch.randn((B, H, n, D), generator=g) * 2).to(dtype).cuda()
    v_new = torch.randn((B, H, n, D), generator=g).to(dtype).cuda()
    v_new[0, 1, 0] = 0                                   # an all-zero row: s = 0, codes 0
    perm = torch.randperm(nblk, generator=g)[: B * 10].view(B, 10).to(torch.int32).cuda()
    pos = torch.tensor([0, 15, 100], dtype=torch.int32).cuda()
    kc, vc, ks, vs = _fresh_cache(nblk, H, D, seed=D)
    want_k = oracle.kv_append(f32(k_new), np_(perm), np_(pos), np_(kc), np_(ks))
    want_v = oracle.kv_append(f32(v_new), np_(perm), np_(pos), np_(vc), np_(vs))
    sage.sage_kv_cache_append(k_new, v_new, kc, vc, ks, vs, perm, pos)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert np.array_equal(np_(kc), want_k[0]) and np.array_equal(np_(ks), want_k[1])
    assert np.array_equal(np_(vc), want_v[0]) and np.array_equal(np_(vs), want_v[1])


def test_kv_append_bad_page_sets_error_and_skips(sage):
    B, H, n, D, nblk = 1, 2, 20, 128, 8
    k_new = torch.randn((B, H, n, D), dtype=torch.bfloat16).cuda()
    v_new = torch.randn((B, H, n, D), dtype=torch.bfloat16).cuda()
    table = torch.tensor([[3, 77]], dtype=torch.int32).cuda()   # page 77 does not exist
    pos = torch.tensor([4], dtype=torch.int32).cuda()            # tokens 4..23 -> pages 3, 77
    kc, vc, ks, vs = _fresh_cache(nblk, H, D, seed=5)
    want_k = oracle.kv_append(f32(k_new), np_(table), np_(pos), np_(kc), np_(ks))
    assert want_k[2] == H * 8
    sage.sage_kv_cache_append(k_new, v_new, kc, vc, ks, vs, table, pos)
    st, word = sage.check_device_status()
    assert st != 0 and word & 2                                  # bad-block bit
    assert np.array_equal(np_(kc), want_k[0]) and np.array_equal(np_(ks), want_k[1])


def test_decode_after_append_matches_oracle(sage):
    """Append a decode step's new token to every sequence, then decode over
    the grown context: the result equals the oracle decode of the cache the
    oracle's own append produced."""
    B, Hq, Hkv, D = 4, 24, 4, 256
    lens = [100, 257, 1, 640]
    c = W.paged_cache(B, Hkv, D, [x + 1 for x in lens], seed=9, device="cuda")
    g = torch.Generator().manual_seed(10)
    k_new = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).cuda()
    pos = torch.tensor(lens, dtype=torch.int32).cuda()
    kc_o, ks_o, _ = oracle.kv_append(f32(k_new), np_(c.block_table), np_(pos), np_(c.k_cache),
                                     np_(c.k_scale))
    vc_o, vs_o, _ = oracle.kv_append(f32(v_new), np_(c.block_table), np_(pos), np_(c.v_cache),
                                     np_(c.v_scale))
    sage.sage_kv_cache_append(k_new, v_new, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                              c.block_table, pos)
    c.lens = (pos + 1).to(torch.int32)
    q = W.decode_query(B, Hq, D, seed=11, device="cuda")
    out, lse = sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                               c.block_table, c.lens, max(lens) + 1,
                                               return_lse=True, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    qi, qs, _ = oracle.quant_int8(f32(q)[:, :, None, :])
    o_ref, l_ref = oracle.decode_paged(qi[:, :, 0], qs[:, :, 0], kc_o, vc_o, ks_o, vs_o,
                                       np_(c.block_table), np_(c.lens))
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 19])
def test_kv_producer_bit_exact(sage, D, dtype, n):
    """One launch appends the step's K/V rows to the cache and quantises its
    query rows ([P1] section 4): cache bytes and scales equal the oracle's
    append, query codes and scales the oracle's per-token quantisation."""
    B, Hq, Hkv, nblk = 3, 12, 4, 40
    g = torch.Generator().manual_seed(D + n + 1)
    q_new = torch.randn((B, Hq, n, D), generator=g).to(dtype).cuda()
    k_new = (torch.randn((B, Hkv, n, D), generator=g) * 2).to(dtype).cuda()
    v_new = torch.randn((B, Hkv, n, D), generator=g).to(dtype).cuda()
    q_new[1, 3, 0] = 0                                   # an all-zero query row
    perm = torch.randperm(nblk, generator=g)[: B * 10].view(B, 10).to(torch.int32).cuda()
    pos = torch.tensor([0, 15, 100], dtype=torch.int32).cuda()
    kc, vc, ks, vs = _fresh_cache(nblk, Hkv, D, seed=D + 1)
    want_k = oracle.kv_append(f32(k_new), np_(perm), np_(pos), np_(kc), np_(ks))
    want_v = oracle.kv_append(f32(v_new), np_(perm), np_(pos), np_(vc), np_(vs))
    want_q, want_qs, _ = oracle.quant_int8(f32(q_new), block_tokens=1)
    qi, qs = sage.sage_kv_producer(q_new, k_new, v_new, kc, vc, ks, vs, perm, pos)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    info = sage.last_launch_info()
    assert info["kernel"] == "kv_producer_kernel" and info["launches"] == 1
    assert np.array_equal(np_(kc), want_k[0]) and np.array_equal(np_(ks), want_k[1])
    assert np.array_equal(np_(vc), want_v[0]) and np.array_equal(np_(vs), want_v[1])
    assert np.array_equal(np_(qi), want_q) and np.array_equal(np_(qs), want_qs)


def test_kv_producer_then_decode(sage):
    """A decode step the way [P1] section 4 runs it: the producer appends the
    new token and quantises the query once, then the split-K decode reads
    those codes -- bit for bit the decode with the query quantised inside
    the kernel, and within tolerance of the oracle."""
    B, Hq, Hkv, D = 4, 24, 4, 256
    lens = [700, 4095, 31, 2000]
    c = W.paged_cache(B, Hkv, D, [n + 1 for n in lens], seed=71, device="cuda")
    g = torch.Generator().manual_seed(72)
    q = torch.randn((B, Hq, 1, D), generator=g).to(torch.bfloat16).cuda()
    k_new = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn((B, Hkv, 1, D), generator=g).to(torch.bfloat16).cuda()
    pos = torch.tensor(lens, dtype=torch.int32).cuda()
    qi, qs = sage.sage_kv_producer(q, k_new, v_new, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                   c.block_table, pos)
    L = max(lens) + 1
    out = sage.sage_attn_decode_paged(qi[:, :, 0].contiguous(), qs[:, :, 0].contiguous(),
                                      c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.block_table,
                                      c.lens, L, num_segments=12, out_dtype=torch.float16)
    ref = sage.sage_attn_decode_paged_q16(q[:, :, 0].contiguous(), c.k_cache, c.v_cache,
                                          c.k_scale, c.v_scale, c.block_table, c.lens, L,
                                          num_segments=12, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out, ref)
    o_ref, _ = oracle.decode_paged(np_(qi)[:, :, 0], np_(qs)[:, :, 0], np_(c.k_cache),
                                   np_(c.v_cache), np_(c.k_scale), np_(c.v_scale),
                                   np_(c.block_table), np_(c.lens))
    assert_close(f32(out), o_ref)


def test_kv_producer_bad_page_skips_cache_rows_not_query_rows(sage):
    """A page outside the cache skips only the K/V rows that would land there
    (error word's bad-block bit set, the rest of the cache as the oracle's
    append leaves it); the query rows, which never touch the cache, are
    quantised all the same."""
    B, Hq, Hkv, n, D, nblk = 1, 4, 2, 20, 128, 8
    q_new = torch.randn((B, Hq, n, D), dtype=torch.bfloat16).cuda()
    k_new = torch.randn((B, Hkv, n, D), dtype=torch.bfloat16).cuda()
    v_new = torch.randn((B, Hkv, n, D), dtype=torch.bfloat16).cuda()
    table = torch.tensor([[3, 77]], dtype=torch.int32).cuda()   # page 77 does not exist
    pos = torch.tensor([4], dtype=torch.int32).cuda()            # tokens 4..23 -> pages 3, 77
    kc, vc, ks, vs = _fresh_cache(nblk, Hkv, D, seed=6)
    want_k = oracle.kv_append(f32(k_new), np_(table), np_(pos), np_(kc), np_(ks))
    want_q, want_qs, _ = oracle.quant_int8(f32(q_new), block_tokens=1)
    qi, qs = sage.sage_kv_producer(q_new, k_new, v_new, kc, vc, ks, vs, table, pos)
    st, word = sage.check_device_status()
    assert st != 0 and word & 2                                  # bad-block bit
    assert np.array_equal(np_(kc), want_k[0]) and np.array_equal(np_(ks), want_k[1])
    assert np.array_equal(np_(qi), want_q) and np.array_equal(np_(qs), want_qs)
