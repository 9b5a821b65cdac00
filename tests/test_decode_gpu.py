"""GPU parity: split-K paged decode + LSE combine against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _quant_query(sage, B, Hq, D, seed):
    q = W.decode_query(B, Hq, D, seed=seed, device="cuda")
    qi, qs, _, _ = sage.sage_quant_int8(q[:, :, None, :])
    return qi[:, :, 0].contiguous(), qs[:, :, 0].contiguous()


def _run(sage, qi, qs, c, max_len, **kw):
    return sage.sage_attn_decode_paged(qi, qs, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                       c.block_table, c.lens, max_len, **kw)


def _oracle(qi, qs, c, pairs=None):
    return oracle.decode_paged(np_(qi), np_(qs), np_(c.k_cache), np_(c.v_cache), np_(c.k_scale),
                               np_(c.v_scale), np_(c.block_table), np_(c.lens), pairs=pairs)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (4, 4), (16, 2), (24, 4)])
@pytest.mark.parametrize("segments", [1, 3, 12, 24, 0])
def test_decode_small(sage, D, Hq, Hkv, segments):
    B = 3
    lens = [37, 300, 129]                     # ragged last pages
    c = W.paged_cache(B, Hkv, D, lens, seed=D + Hq, device="cuda", extra_blocks=5)
    qi, qs = _quant_query(sage, B, Hq, D, seed=Hq)
    # short contexts give |O| ~ 0.5: f16 output keeps output rounding well inside tolerance
    out, lse = _run(sage, qi, qs, c, max(lens), num_segments=segments, return_lse=True,
                    out_dtype=torch.float16)
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(qi, qs, c)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")
    st, word = sage.check_device_status()
    assert st == 0, word


def test_decode_raw_scores_bit_exact(sage):
    B, Hq, Hkv, D = 2, 12, 2, 256
    lens = [45, 200]
    c = W.paged_cache(B, Hkv, D, lens, seed=7, device="cuda", extra_blocks=3)
    qi, qs = _quant_query(sage, B, Hq, D, seed=8)
    dbg = torch.full((B, Hq, max(lens)), -(2 ** 31), dtype=torch.int32, device="cuda")
    _run(sage, qi, qs, c, max(lens), num_segments=2, debug_scores=dbg)
    torch.cuda.synchronize()
    d = np_(dbg)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            keys = oracle.gather_paged(np_(c.k_cache), np_(c.block_table)[b], lens[b], g)
            ref = oracle.qk_int32(np_(qi)[b, h][None], keys)[0]
            assert np.array_equal(d[b, h, :lens[b]], ref), (b, h)
            assert np.all(d[b, h, lens[b]:] == -(2 ** 31))


def test_decode_adversarial_int32_bound(sage):
    """All-+-127 codes at D=256: raw scores hit the 256*127*127 bound exactly."""
    B, Hq, Hkv, D = 1, 6, 1, 256
    c = W.paged_cache(B, Hkv, D, [32], seed=1, device="cuda")
    c.k_cache.fill_(127)
    c.k_cache[:, :, :, 8:, :] = -127          # slots 8..15 negative
    qi = torch.full((B, Hq, D), 127, dtype=torch.int8, device="cuda")
    qi[0, 3] = -127
    qs = torch.full((B, Hq), 0.01, dtype=torch.float32, device="cuda")
    dbg = torch.zeros((B, Hq, 32), dtype=torch.int32, device="cuda")
    _run(sage, qi, qs, c, 32, num_segments=1, debug_scores=dbg)
    torch.cuda.synchronize()
    d = np_(dbg)
    bound = 256 * 127 * 127
    assert d[0, 0, 0] == bound and d[0, 0, 8] == -bound and d[0, 3, 0] == -bound


def test_decode_permuted_block_table_bitwise(sage):
    B, Hq, Hkv, D = 2, 24, 4, 256
    lens = [1000, 777]
    c = W.paged_cache(B, Hkv, D, lens, seed=21, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=22)
    out1 = _run(sage, qi, qs, c, max(lens), num_segments=4)
    # move every page to a new physical slot and remap the table
    nblk = c.k_cache.shape[0]
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(3)).to("cuda")
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nblk, device="cuda")
    c2 = W.PagedCache(c.k_cache[inv], c.v_cache[inv], c.k_scale[inv], c.v_scale[inv],
                      perm[c.block_table.long()].to(torch.int32), c.lens)
    out2 = _run(sage, qi, qs, c2, max(lens), num_segments=4)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_decode_split_invariance(sage):
    B, Hq, Hkv, D = 2, 24, 4, 128
    lens = [2048, 1500]
    c = W.paged_cache(B, Hkv, D, lens, seed=5, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=6)
    ref, lref = _run(sage, qi, qs, c, max(lens), num_segments=1, return_lse=True,
                     out_dtype=torch.float16)
    for S in (2, 7, 32):
        out, lse = _run(sage, qi, qs, c, max(lens), num_segments=S, return_lse=True,
                        out_dtype=torch.float16)
        torch.cuda.synchronize()
        assert_close(f32(out), f32(ref), "split %d" % S, rel=2e-3, abs_=1e-3)
        assert_close(np_(lse), np_(lref), "lse split %d" % S, rel=1e-5, abs_=1e-4)


def test_decode_empty_context(sage):
    B, Hq, Hkv, D = 3, 8, 1, 64
    lens = [0, 20, 0]
    c = W.paged_cache(B, Hkv, D, [max(x, 1) for x in lens], seed=9, device="cuda")
    c.lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=10)
    out, lse = _run(sage, qi, qs, c, 20, num_segments=0, return_lse=True,
                    out_dtype=torch.float16)
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(qi, qs, c)
    assert np.all(f32(out)[[0, 2]] == 0) and np.all(np.isneginf(np_(lse)[[0, 2]]))
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


def test_decode_bad_block_sets_error_word(sage):
    B, Hq, Hkv, D = 1, 6, 1, 128
    c = W.paged_cache(B, Hkv, D, [64], seed=2, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=3)
    sage.check_device_status()
    bad = c.block_table.clone()
    bad[0, 1] = c.k_cache.shape[0] + 100       # out of range: must not be read
    c_bad = W.PagedCache(c.k_cache, c.v_cache, c.k_scale, c.v_scale, bad, c.lens)
    _run(sage, qi, qs, c_bad, 64, num_segments=1, out_dtype=torch.float16)
    st, word = sage.check_device_status()
    assert st == sage.SAGE_ERR_BAD_BLOCK and word & 2
    # the context is still usable
    out = _run(sage, qi, qs, c, 64, num_segments=1, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert_close(f32(out), _oracle(qi, qs, c)[0])


def test_bounded_wait_times_out_and_context_survives(sage):
    sage.check_device_status()
    sage.debug_timeout_probe(20000)            # 20 ms wait nobody ends
    st, word = sage.check_device_status()
    assert st == sage.SAGE_ERR_TIMEOUT and word & 1
    x = torch.randn(1, 1, 16, 64, device="cuda", dtype=torch.float16)
    q, s, _, _ = sage.sage_quant_int8(x)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0


def test_decode_launch_record(sage):
    c = W.paged_cache(2, 4, 256, [4096, 4096], seed=1, device="cuda")
    qi, qs = _quant_query(sage, 2, 24, 256, seed=1)
    # up to 8 segments: one launch, the segments of a (sequence, kv head)
    # form a cluster and combine in distributed shared memory
    _run(sage, qi, qs, c, 4096, num_segments=8)
    info = sage.last_launch_info()
    assert info["kernel"] == "decode_kernel" and info["num_segments"] == 8
    assert info["launches"] == 1 and info["grid"] == (8, 4, 2) and info["cluster"] == (8, 1, 1)
    # more segments: partials in the workspace, then the combine kernel
    _run(sage, qi, qs, c, 4096, num_segments=32)
    info = sage.last_launch_info()
    assert info["kernel"] == "decode_kernel" and info["num_segments"] == 32
    assert info["launches"] == 2 and info["grid"] == (32, 4, 2) and info["cluster"] == (1, 1, 1)


def test_decode_paged_decode_full_size(sage):
    """The B8 / 24:4 GQA / D256 / 8192-token workload, every output vs the oracle."""
    P = W.WORKLOADS["paged_decode"].params
    c = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["ctx"]] * P["B"], seed=P["seed"],
                      device="cuda")
    qi, qs = _quant_query(sage, P["B"], P["Hq"], P["D"], seed=P["seed"])
    out, lse = _run(sage, qi, qs, c, P["ctx"], return_lse=True)
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(qi, qs, c)
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("L", [8192, 16384, 32768])
@pytest.mark.parametrize("B", [1, 16, 64])
def test_decode_sweep(sage, L, B):
    P = W.WORKLOADS["decode_sweep"].params
    c = W.paged_cache(B, P["Hkv"], P["D"], [L] * B, seed=P["seed"] + L + B, device="cuda")
    qi, qs = _quant_query(sage, B, P["Hq"], P["D"], seed=P["seed"])
    out, lse = _run(sage, qi, qs, c, L, return_lse=True)
    torch.cuda.synchronize()
    # all (b, kv head) pairs up to 16 sequences; a seeded sample beyond
    pairs = [(b, g) for b in range(B) for g in range(P["Hkv"])]
    if B > 16:
        rng = np.random.default_rng(L)
        pairs = [pairs[i] for i in rng.choice(len(pairs), 24, replace=False)]
    o_ref, l_ref = _oracle(qi, qs, c, pairs=pairs)
    grp = P["Hq"] // P["Hkv"]
    rows = [(b, h) for (b, g) in pairs for h in range(g * grp, (g + 1) * grp)]
    bi, hi = np.array(rows).T
    assert_close(f32(out)[bi, hi], o_ref[bi, hi])
    assert_close(np_(lse)[bi, hi], l_ref[bi, hi], "lse")


def test_decode_partials_then_combine(sage):
    B, Hq, Hkv, D = 2, 24, 4, 256
    lens = [3000, 1234]
    c = W.paged_cache(B, Hkv, D, lens, seed=31, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=32)
    op, lp = sage.sage_attn_decode_paged_partials(qi, qs, c.k_cache, c.v_cache, c.k_scale,
                                                  c.v_scale, c.block_table, c.lens, max(lens), 5)
    out, lse = sage.sage_splitk_combine(op, lp, out_dtype=torch.float16, return_lse=True)
    full, lfull = _run(sage, qi, qs, c, max(lens), num_segments=5, return_lse=True,
                       out_dtype=torch.float16)
    torch.cuda.synchronize()
    # up to 8 segments the full decode combines inside a thread-block cluster
    # (base-2 arithmetic), the standalone kernel in natural log: equal up to
    # fp32 rounding order, i.e. within an ulp of the f16 output
    assert_close(f32(out), f32(full), "combine vs fused", rel=1e-3, abs_=1e-3)
    assert_close(np_(lse), np_(lfull), "lse combine vs fused", rel=1e-6, abs_=1e-5)
    # each segment partial is itself the attention over its own key range:
    # segment s covers pages [s * P / S, (s + 1) * P / S) of the longest
    # context (P pages), so the segments differ by one page at most
    P = (max(lens) + 15) // 16
    seg = 1
    lo, hi = seg * P // 5 * 16, min((seg + 1) * P // 5 * 16, lens[1])
    keys = oracle.gather_paged(np_(c.k_cache), np_(c.block_table)[1], lens[1], 0)[lo:hi]
    ks = oracle.gather_paged_scale(np_(c.k_scale), np_(c.block_table)[1], lens[1], 0)[lo:hi]
    vals = oracle.gather_paged(np_(c.v_cache), np_(c.block_table)[1], lens[1], 0)[lo:hi]
    vs = oracle.gather_paged_scale(np_(c.v_scale), np_(c.block_table)[1], lens[1], 0)[lo:hi]
    o1, l1 = oracle.attend(np_(qi)[1, :6], np_(qs)[1, :6], keys, ks,
                           vals.astype(np.float64) * vs[:, None].astype(np.float64),
                           sm_scale=1 / 16)
    assert_close(np_(op)[1, :6, seg], o1, "segment partial")
    assert_close(np_(lp)[1, :6, seg], l1, "segment lse")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(24, 4), (4, 4), (16, 2)])
@pytest.mark.parametrize("segments", [1, 3, 12])
@pytest.mark.parametrize("qdt", [torch.bfloat16, torch.float16])
def test_decode_fused_query_quant_bitwise(sage, D, Hq, Hkv, segments, qdt):
    """Quantising the query inside the decode kernel gives the same codes and
    scales as sage_quant_int8, hence bit-identical outputs and LSE."""
    B = 3
    lens = [37, 300, 129]
    c = W.paged_cache(B, Hkv, D, lens, seed=D + Hq + 7, device="cuda", extra_blocks=5)
    q = W.decode_query(B, Hq, D, seed=Hq + 3, device="cuda").to(qdt).contiguous()
    qi, qs, _, _ = sage.sage_quant_int8(q[:, :, None, :])
    ref, lref = _run(sage, qi.view(B, Hq, D), qs.view(B, Hq), c, max(lens), num_segments=segments,
                     return_lse=True, out_dtype=torch.float16)
    out, lse = sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                               c.block_table, c.lens, max(lens),
                                               num_segments=segments, return_lse=True,
                                               out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert torch.equal(out, ref) and torch.equal(lse, lref)


def test_decode_pinned_host_io_bitwise(sage):
    """Per-step inputs and outputs in pinned host memory (read and written by
    the kernel in place) give exactly the device-memory result; pageable
    host memory is refused before anything is launched."""
    B, Hq, Hkv, D, ctx = 4, 12, 2, 128, 700
    c = W.paged_cache(B, Hkv, D, [ctx, 5, 333, 0], seed=91, device="cuda")
    q = W.decode_query(B, Hq, D, seed=91, device="cuda")
    ref, ref_lse = sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                                   c.block_table, c.lens, ctx, return_lse=True)
    out_h = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    got = sage.sage_attn_decode_paged_q16(q.cpu().pin_memory(), c.k_cache, c.v_cache, c.k_scale,
                                          c.v_scale, c.block_table.cpu().pin_memory(),
                                          c.lens.cpu().pin_memory(), ctx, out=out_h)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    assert got.data_ptr() == out_h.data_ptr()
    assert torch.equal(out_h, ref.cpu())
    # the INT8 entry point with pinned query codes and scales
    qi, qs, _, _ = sage.sage_quant_int8(q[:, :, None, :])
    r2 = sage.sage_attn_decode_paged(qi[:, :, 0], qs[:, :, 0], c.k_cache, c.v_cache, c.k_scale,
                                     c.v_scale, c.block_table, c.lens, ctx)
    o2 = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    sage.sage_attn_decode_paged(qi[:, :, 0].cpu().pin_memory(), qs[:, :, 0].cpu().pin_memory(),
                                c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                c.block_table.cpu().pin_memory(), c.lens.cpu().pin_memory(), ctx,
                                out=o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, r2.cpu())
    # pageable host memory: rejected on the host, nothing launched
    a = sage._decode_args(None, None, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.block_table,
                          c.lens, ctx, None, 0, ref, None, shape=(B, Hq, D))
    pageable = np.zeros(B * Hq * D, np.float32)
    st = sage.lib().sage_attn_decode_paged_q16(ctypes.byref(a), pageable.ctypes.data_as(ctypes.c_void_p),
                                               sage.SAGE_BF16, None, 0, None)
    assert st == sage.SAGE_ERR_INVALID_ARG
    assert b"pinned host memory" in sage.lib().sage_get_last_error_message()


def test_auto_segments_fill_one_wave(sage):
    """Past one cluster's 8 segments the library's choice is one full wave:
    decode_kernel<256> holds 3 CTAs per SM (160 threads x 128 registers,
    ~71 KB of shared memory), and the (sequence, KV head) units times the
    segments fill the SMs to that without a second wave.  Pinned host I/O
    takes the same choice for this shape."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hq, Hkv, D, ctx = 8, 24, 4, 256, 8192
    S = sage.decode_num_segments(B, Hq, Hkv, D, ctx)
    units = B * Hkv
    assert S > 8 and S * units <= 3 * sms < (S + 1) * units, (S, sms)
    c = W.paged_cache(B, Hkv, D, [ctx] * B, seed=7, device="cuda")
    q = W.decode_query(B, Hq, D, seed=7, device="cuda")
    dev = sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                          c.block_table, c.lens, ctx)
    torch.cuda.synchronize()
    assert sage.last_launch_info()["num_segments"] == S
    qh, bth, lh = q.cpu().pin_memory(), c.block_table.cpu().pin_memory(), c.lens.cpu().pin_memory()
    out_h = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    sage.sage_attn_decode_paged_q16(qh, c.k_cache, c.v_cache, c.k_scale, c.v_scale, bth, lh, ctx,
                                    out=out_h)
    torch.cuda.synchronize()
    assert sage.last_launch_info()["num_segments"] == S
    assert torch.equal(out_h, dev.cpu())


def test_decode_output_only_8_byte_aligned(sage):
    """An output that is only 8-byte aligned (what the interface requires)
    gets the same bits as a 16-byte aligned one."""
    B, Hq, Hkv, D = 2, 24, 4, 256
    c = W.paged_cache(B, Hkv, D, [4096, 3000], seed=51, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=52)
    ref = _run(sage, qi, qs, c, 4096, num_segments=20)
    buf = torch.zeros(B * Hq * D + 4, dtype=torch.bfloat16, device="cuda")
    out = buf[4:].view(B, Hq, D)                      # 8 bytes past a 16-byte boundary
    assert out.data_ptr() % 16 == 8
    _run(sage, qi, qs, c, 4096, num_segments=20, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_decode_host_query_quantised_once(sage):
    """A query in pinned host memory is quantised once into the workspace
    by the per-token kernel, and the decode launched behind it reads the
    codes: the same bits as the fused path on a device query, with one more
    launch (quantisation, decode, combine at 14 segments)."""
    B, Hq, Hkv, D, ctx = 8, 24, 4, 256, 8192
    c = W.paged_cache(B, Hkv, D, [ctx, 8000, 4097, 16, 8192, 3000, 1, 7777], seed=93,
                      device="cuda")
    q = W.decode_query(B, Hq, D, seed=93, device="cuda")
    ref, ref_lse = sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                                   c.block_table, c.lens, ctx, num_segments=14,
                                                   return_lse=True)
    torch.cuda.synchronize()
    assert sage.last_launch_info()["launches"] == 2
    got, lse = sage.sage_attn_decode_paged_q16(q.cpu().pin_memory(), c.k_cache, c.v_cache,
                                               c.k_scale, c.v_scale, c.block_table, c.lens, ctx,
                                               num_segments=14, return_lse=True)
    torch.cuda.synchronize()
    info = sage.last_launch_info()
    assert info["kernel"] == "decode_kernel" and info["launches"] == 3
    assert sage.check_device_status()[0] == 0
    assert torch.equal(got, ref) and torch.equal(lse, ref_lse)


def test_decode_permuted_pages_bitwise_partials_path(sage):
    """Past one cluster (14 segments: partials in the workspace, then the
    combine kernel) the same logical cache on permuted physical pages still
    gives the same bits, with contexts of different lengths."""
    B, Hq, Hkv, D = 4, 24, 4, 256
    lens = [8192, 8000, 5000, 8192]
    c = W.paged_cache(B, Hkv, D, lens, seed=61, device="cuda")
    qi, qs = _quant_query(sage, B, Hq, D, seed=62)
    out1 = _run(sage, qi, qs, c, max(lens), num_segments=14)
    assert sage.last_launch_info()["launches"] == 2
    nblk = c.k_cache.shape[0]
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(5)).to("cuda")
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nblk, device="cuda")
    c2 = W.PagedCache(c.k_cache[inv], c.v_cache[inv], c.k_scale[inv], c.v_scale[inv],
                      perm[c.block_table.long()].to(torch.int32), c.lens)
    out2 = _run(sage, qi, qs, c2, max(lens), num_segments=14)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("pv", ["int8", "fp16+fp32", "fp16"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("segments", [1, 5, 12])
def test_decode_pv_modes(sage, pv, D, segments):
    """The P.V variants against the oracle: INT8 P.V against the oracle's
    INT8 P.V (V-scaled probabilities quantised per 16-key page), the f16
    accumulators against exact attention; ragged contexts, GQA 6:1, one
    segment, an in-cluster merge and the combine kernel."""
    B, Hq, Hkv = 3, 24, 4
    lens = [37, 300, 1029]
    c = W.paged_cache(B, Hkv, D, lens, seed=D + segments, device="cuda", extra_blocks=3)
    qi, qs = _quant_query(sage, B, Hq, D, seed=segments)
    out, lse = _run(sage, qi, qs, c, max(lens), num_segments=segments, return_lse=True,
                    out_dtype=torch.float16, pv_mode=pv)
    torch.cuda.synchronize()
    assert sage.check_device_status()[0] == 0
    o_ref, l_ref = oracle.decode_paged(np_(qi), np_(qs), np_(c.k_cache), np_(c.v_cache),
                                       np_(c.k_scale), np_(c.v_scale), np_(c.block_table),
                                       np_(c.lens), pv_int8=pv == "int8")
    assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")


@pytest.mark.parametrize("pv", ["int8", "fp16+fp32", "fp16"])
def test_decode_pv_modes_full_size(sage, pv):
    """The paged-decode workload (B8, 24:4, D256, 8192 tokens, 14 segments,
    bf16 output) in each P.V variant, every output against the oracle."""
    P = W.WORKLOADS["paged_decode"].params
    c = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["ctx"]] * P["B"], seed=P["seed"],
                      device="cuda")
    qi, qs = _quant_query(sage, P["B"], P["Hq"], P["D"], seed=P["seed"])
    out, lse = _run(sage, qi, qs, c, P["ctx"], return_lse=True, pv_mode=pv)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode_paged(np_(qi), np_(qs), np_(c.k_cache), np_(c.v_cache),
                                       np_(c.k_scale), np_(c.v_scale), np_(c.block_table),
                                       np_(c.lens), pv_int8=pv == "int8")
    r, m = assert_close(f32(out), o_ref)
    assert_close(np_(lse), l_ref, "lse")
    print("pv %s: rel-L2 %.3g max-abs %.3g" % (pv, r, m))
