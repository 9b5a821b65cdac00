"""CPU oracle for INT8-QK quantized attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it; the only thing both sides share is the
seeded input generator, which holds none of the method's arithmetic.

The arithmetic lives in ``sage_oracle.c`` (plain C, fp32 quantisation
decisions, exact integer dot products, fp64 softmax).  This module only
marshals numpy arrays, performs the paged-cache gather (a pure index
lookup) and runs independent (batch, head) problems on a thread pool.

Sources, by page title and section:
  [P1] "INT8 QK MMAC on gfx936 DCU: paged access, fragment mapping and GQA"
  [P3] "SageAttention -- MetaX MXMACA port" README
"""
from __future__ import annotations

import ctypes
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_LIB = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(_build.build())
        lib.oracle_quant_int8.argtypes = [_vp, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]
        lib.oracle_quant_int8.restype = None
        lib.oracle_token_mean.argtypes = [_vp, _i64, _i64, ctypes.c_int, _vp]
        lib.oracle_token_mean.restype = None
        lib.oracle_row_bias.argtypes = [_vp, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp]
        lib.oracle_row_bias.restype = None
        lib.oracle_qk_int32.argtypes = [_vp, _i64, _vp, _i64, ctypes.c_int, _vp]
        lib.oracle_qk_int32.restype = _i64
        lib.oracle_attend.argtypes = [_i64, ctypes.c_int, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp,
                                      _vp, ctypes.c_int, _i64, ctypes.c_double, _vp, _vp]
        lib.oracle_attend.restype = _i64
        lib.oracle_attend_pv_int8.argtypes = [_i64, ctypes.c_int, _vp, _vp, _i64, _vp, _vp, _vp,
                                              _vp, ctypes.c_int, ctypes.c_double, _vp, _vp]
        lib.oracle_attend_pv_int8.restype = _i64
        lib.oracle_splitk_combine.argtypes = [_vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp]
        lib.oracle_splitk_combine.restype = None
        lib.oracle_kv_append.argtypes = [_vp, _i64, _i64, _i64, ctypes.c_int, _vp, _i64, _vp, _i64,
                                         _vp, _vp]
        lib.oracle_kv_append.restype = _i64
        _LIB = lib
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(_vp)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    return os.cpu_count() or 1


# --------------------------------------------------------------------------
# Quantisation ([P1] section 4; [P3] quant kernel table and advanced config)
# --------------------------------------------------------------------------

def token_mean(x):
    """Per-(sequence, channel) mean over tokens, fp64 token-order sum -> fp32.

    x: [..., S, D] float32.  Returns float32 [..., D].
    """
    x = _c(x, np.float32)
    *lead, S, D = x.shape
    BH = int(np.prod(lead)) if lead else 1
    mu = np.empty((BH, D), np.float32)
    _lib().oracle_token_mean(_p(x), BH, S, D, _p(mu))
    return mu.reshape(*lead, D)


def quant_int8(x, block_tokens: int = 1, smooth: bool = False, mu=None):
    """Symmetric INT8 quantisation, s = amax/127, q = rne(x/s) in fp32.

    x: float32 [..., S, D] (fp16/bf16 inputs converted exactly to fp32).
    block_tokens: 1 = per token, else tokens per block (128 Q, 64 K).
    smooth: subtract the token mean first (computed here unless ``mu``
    is given, in which case that mean is used as is).
    Returns (q int8 [..., S, D], scale fp32 [..., ceil(S/block)], mu or None).
    """
    x = _c(x, np.float32)
    *lead, S, D = x.shape
    BH = int(np.prod(lead)) if lead else 1
    if smooth and mu is None:
        mu = token_mean(x)
    mu_c = None if (not smooth) else _c(mu, np.float32).reshape(BH, D)
    G = (S + block_tokens - 1) // block_tokens
    q = np.empty((BH, S, D), np.int8)
    s = np.empty((BH, G), np.float32)
    _lib().oracle_quant_int8(_p(x), BH, S, D, int(block_tokens), _p(mu_c), _p(q), _p(s))
    mu_out = None if mu_c is None else mu_c.reshape(*lead, D)
    return q.reshape(*lead, S, D), s.reshape(*lead, G), mu_out


def row_bias(x, mu):
    """b_i = sum_c x_ic mu_c in fp64.  x: [B,H,S,D]; mu: [B,Hmu,D] (GQA groups)."""
    x = _c(x, np.float32)
    mu = _c(mu, np.float32)
    B, H, S, D = x.shape
    Hmu = mu.shape[1]
    out = np.empty((B, H, S), np.float64)
    _lib().oracle_row_bias(_p(x), B, H, S, D, _p(mu), Hmu, _p(out))
    return out


def qk_int32(q, k):
    """Raw INT32 scores of one head ([P1] 2.1): q [Sq,D] int8, k [Sk,D] int8."""
    q = _c(q, np.int8)
    k = _c(k, np.int8)
    Sq, D = q.shape
    Sk = k.shape[0]
    acc = np.empty((Sq, Sk), np.int32)
    bad = _lib().oracle_qk_int32(_p(q), Sq, _p(k), Sk, D, _p(acc))
    if bad:
        raise ValueError("raw score outside the INT32 bound D*127^2")
    return acc


def expand_scale(scale, n: int, block: int):
    """Per-row scale of rows 0..n-1 from per-group scales ([..., G])."""
    idx = np.arange(n) // block
    return np.asarray(scale)[..., idx]


# --------------------------------------------------------------------------
# Paged cache lookup ([P1] section 3, steps 1-5)
# cache layout [block, kv_head, head_dim/16, block_size=16, 16];
# scale layout [block, kv_head, 16]
# --------------------------------------------------------------------------

PAGE = 16


def gather_paged(cache, block_row, n_tokens: int, kv_head: int):
    """Logical [n_tokens, D] int8 rows of one (sequence, kv head).

    Token t lives in physical block block_row[t // 16], slot t % 16;
    channel c in sub-block c // 16 at position c % 16.
    """
    cache = np.asarray(cache)
    D = cache.shape[2] * 16
    t = np.arange(n_tokens)
    blk = np.asarray(block_row)[t // PAGE].astype(np.int64)
    # advanced indices (blk, kv_head, slot) -> [n_tokens, D/16, 16]
    rows = cache[blk, kv_head, :, t % PAGE, :]
    return np.ascontiguousarray(rows.reshape(n_tokens, D))


def gather_paged_scale(scale, block_row, n_tokens: int, kv_head: int):
    """Per-token fp32 scale [n_tokens] of one (sequence, kv head)."""
    t = np.arange(n_tokens)
    blk = np.asarray(block_row)[t // PAGE].astype(np.int64)
    return np.ascontiguousarray(np.asarray(scale)[blk, kv_head, t % PAGE], dtype=np.float32)


# --------------------------------------------------------------------------
# Attention ([P1] section 1; [P3] attention pipeline)
# --------------------------------------------------------------------------

def attend(q, sq, k, sk, v, *, sm_scale, causal=False, causal_offset=0, qpos=None,
           qbias=None, smoothed=None):
    """One query-row batch against one key set; returns (o fp64, lse fp64)."""
    q = _c(q, np.int8)
    sq = _c(sq, np.float32)
    k = _c(k, np.int8)
    sk = _c(sk, np.float32)
    v = _c(v, np.float64)
    nq, D = q.shape
    nk = k.shape[0]
    qb = None if qbias is None else _c(qbias, np.float64)
    sm = None if smoothed is None else _c(smoothed, np.uint8)
    qp = None
    if causal:
        qp = _c(np.arange(nq) if qpos is None else qpos, np.int64)
    o = np.empty((nq, D), np.float64)
    lse = np.empty((nq,), np.float64)
    bad = _lib().oracle_attend(nq, D, _p(q), _p(sq), _p(qb), _p(qp), nk, _p(k), _p(sk), _p(sm),
                               _p(v), int(bool(causal)), int(causal_offset), float(sm_scale),
                               _p(o), _p(lse))
    if bad:
        raise ValueError("raw score outside the INT32 bound D*127^2")
    return o, lse


def attend_pv_int8(q, sq, k, sk, v, sv, *, sm_scale, block=PAGE):
    """One query-row batch against one key set with INT8 P.V ([P1] sections
    6 and 8): v int8 [nk, D] codes and sv fp32 [nk] their per-token scales;
    the V-scaled probabilities are quantised per group of `block` keys.
    Returns (o fp64, lse fp64)."""
    q = _c(q, np.int8)
    sq = _c(sq, np.float32)
    k = _c(k, np.int8)
    sk = _c(sk, np.float32)
    v = _c(v, np.int8)
    sv = _c(sv, np.float32)
    nq, D = q.shape
    nk = k.shape[0]
    o = np.empty((nq, D), np.float64)
    lse = np.empty((nq,), np.float64)
    bad = _lib().oracle_attend_pv_int8(nq, D, _p(q), _p(sq), nk, _p(k), _p(sk), _p(v), _p(sv),
                                       int(block), float(sm_scale), _p(o), _p(lse))
    if bad:
        raise ValueError("raw score outside the INT32 bound D*127^2")
    return o, lse


def _run(jobs, threads):
    threads = threads or default_threads()
    if threads <= 1 or len(jobs) <= 1:
        return [j() for j in jobs]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda f: f(), jobs))


def prefill(q_i8, q_scale, q_block, k_i8, k_scale, k_block, v, *, causal, sm_scale=None,
            q_bias=None, prefix=None, rows=None, threads=None, smooth_v=False):
    """Prefill attention, optionally over a paged INT8 prefix.

    q_i8 [B,Hq,Sq,D] int8, q_scale [B,Hq,ceil(Sq/q_block)] fp32;
    k_i8 [B,Hkv,Sc,D] int8 (the contiguous chunk), k_scale [B,Hkv,ceil(Sc/k_block)];
    v [B,Hkv,Sc,D] float values (fp16/bf16 as given);
    q_bias [B,Hq,Sq] fp64 or None: when given the chunk keys are smoothed
    and their scores get q_bias back (the smooth_k correction);
    prefix: None or dict(k_cache, v_cache [nblk,Hkv,D/16,16,16] int8,
    k_scale, v_scale [nblk,Hkv,16] fp32, block_table [B,maxblk] int32,
    lens [B]) -- prefix keys come first, then the chunk.
    Causal alignment is bottom-right: key j is visible to query i iff
    j <= i + (Sk - Sq), Sk = prefix + chunk length.
    rows: optional query-row indices to evaluate (same for every b, h).
    smooth_v ([P3] "V mean fusion"): mu = the chunk's per-(b, kv head,
    channel) mean of V (token_mean, rounded to fp32) is subtracted from every
    value the rows attend to (prefix included) and added back to the output;
    a row that sees no key keeps o = 0.  In exact arithmetic the result is
    unchanged (each softmax row sums to 1); the kernels gain precision.
    Returns (o fp64 [B,Hq,R,D], lse fp64 [B,Hq,R]).
    """
    q_i8 = np.asarray(q_i8)
    B, Hq, Sq, D = q_i8.shape
    Hkv, Sc = k_i8.shape[1], k_i8.shape[2]
    group = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    rows = np.arange(Sq) if rows is None else np.asarray(rows, np.int64)
    R = len(rows)
    o = np.zeros((B, Hq, R, D), np.float64)
    lse = np.zeros((B, Hq, R), np.float64)
    v = np.asarray(v, np.float64)
    sq_full = expand_scale(q_scale, Sq, q_block)
    sk_full = expand_scale(k_scale, Sc, k_block)
    mu_v = token_mean(np.asarray(v, np.float32)).astype(np.float64) if smooth_v else None
    jobs = []
    for b in range(B):
        P = 0 if prefix is None else int(prefix["lens"][b])
        for g in range(Hkv):
            if P:
                bt = prefix["block_table"][b]
                kp = gather_paged(prefix["k_cache"], bt, P, g)
                vp = gather_paged(prefix["v_cache"], bt, P, g).astype(np.float64)
                skp = gather_paged_scale(prefix["k_scale"], bt, P, g)
                svp = gather_paged_scale(prefix["v_scale"], bt, P, g).astype(np.float64)
                vp = vp * svp[:, None]
                keys = np.concatenate([kp, k_i8[b, g]], 0)
                sks = np.concatenate([skp, sk_full[b, g]], 0)
                vals = np.concatenate([vp, v[b, g]], 0)
            else:
                keys, sks, vals = np.asarray(k_i8[b, g]), sk_full[b, g], v[b, g]
            smoothed = None
            if q_bias is not None:
                smoothed = np.concatenate([np.zeros(P, np.uint8), np.ones(Sc, np.uint8)])
            mu = None if mu_v is None else mu_v[b, g]
            if mu is not None:
                vals = vals - mu[None, :]
            for h in range(g * group, (g + 1) * group):
                def job(b=b, h=h, keys=keys, sks=sks, vals=vals, smoothed=smoothed, P=P, mu=mu):
                    qb = None if q_bias is None else np.asarray(q_bias)[b, h, rows]
                    ob, lb = attend(q_i8[b, h, rows], sq_full[b, h, rows], keys, sks, vals,
                                    sm_scale=sm_scale, causal=causal,
                                    causal_offset=P + Sc - Sq, qpos=rows, qbias=qb,
                                    smoothed=smoothed)
                    if mu is not None:
                        seen = np.isfinite(lb)
                        ob = np.where(seen[:, None], ob + mu[None, :], 0.0)
                    o[b, h] = ob
                    lse[b, h] = lb
                jobs.append(job)
    _run(jobs, threads)
    return o, lse


def decode_paged(q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
                 context_lens, *, sm_scale=None, threads=None, pairs=None, pv_int8=False):
    """Single-token decode over a paged INT8 K/V cache ([P1] sections 3-5).

    q_i8 [B,Hq,D] int8, q_scale [B,Hq] fp32; caches [nblk,Hkv,D/16,16,16]
    int8; scales [nblk,Hkv,16] fp32; block_table [B,maxblk] int32;
    context_lens [B].  Query head h reads kv head h // (Hq/Hkv).
    pairs: optional list of (b, kv_head) to evaluate (others stay zero).
    pv_int8: INT8 P.V (attend_pv_int8), quantisation groups = cache pages.
    Returns (o fp64 [B,Hq,D], lse fp64 [B,Hq]).
    """
    q_i8 = np.asarray(q_i8)
    B, Hq, D = q_i8.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    o = np.zeros((B, Hq, D), np.float64)
    lse = np.full((B, Hq), -np.inf, np.float64)
    if pairs is None:
        pairs = [(b, g) for b in range(B) for g in range(Hkv)]
    jobs = []
    for (b, g) in pairs:
        def job(b=b, g=g):
            n = int(context_lens[b])
            bt = block_table[b]
            keys = gather_paged(k_cache, bt, n, g)
            sk = gather_paged_scale(k_scale, bt, n, g)
            hs = slice(g * group, (g + 1) * group)
            if pv_int8:
                ob, lb = attend_pv_int8(q_i8[b, hs], np.asarray(q_scale)[b, hs], keys, sk,
                                        gather_paged(v_cache, bt, n, g),
                                        gather_paged_scale(v_scale, bt, n, g), sm_scale=sm_scale)
            else:
                vals = gather_paged(v_cache, bt, n, g).astype(np.float64)
                vals *= gather_paged_scale(v_scale, bt, n, g).astype(np.float64)[:, None]
                ob, lb = attend(q_i8[b, hs], np.asarray(q_scale)[b, hs], keys, sk, vals,
                                sm_scale=sm_scale)
            o[b, hs] = ob
            lse[b, hs] = lb
        jobs.append(job)
    _run(jobs, threads)
    return o, lse


def splitk_combine(o_part, lse_part):
    """LSE-weighted combine of split-K partials: o_part [..., S, D], lse_part [..., S]."""
    o_part = _c(o_part, np.float64)
    lse_part = _c(lse_part, np.float64)
    *lead, S, D = o_part.shape
    R = int(np.prod(lead)) if lead else 1
    o = np.empty((R, D), np.float64)
    lse = np.empty((R,), np.float64)
    _lib().oracle_splitk_combine(_p(o_part), _p(lse_part), R, S, D, _p(o), _p(lse))
    return o.reshape(*lead, D), lse.reshape(*lead)


def kv_append(x, block_table, positions, cache, scale):
    """Quantise new rows per (token, KV head) and write them into a paged cache.

    x float32 [B,H,n,D] (exact fp32 copies of the fp16/bf16 rows);
    block_table int32 [B,max_blocks]; positions int32 [B] (row 0's token
    index); cache int8 [num_blocks,H,D/16,16,16] and scale float32
    [num_blocks,H,16] are copied, updated and returned with the count of
    rows whose page index was out of range (those are left untouched).
    ([P1] sections 3 and 4.)
    """
    x = _c(x, np.float32)
    B, H, n, D = x.shape
    bt = _c(block_table, np.int32)
    pos = _c(positions, np.int32)
    cache = np.array(cache, dtype=np.int8, copy=True, order="C")
    scale = np.array(scale, dtype=np.float32, copy=True, order="C")
    skipped = _lib().oracle_kv_append(_p(x), B, H, n, D, _p(bt), bt.shape[1], _p(pos),
                                      cache.shape[0], _p(cache), _p(scale))
    return cache, scale, int(skipped)


# --------------------------------------------------------------------------
# Variable-length packed batches ([P3] "Varlen per-batch loop" and the
# batched varlen kernel its roadmap plans): sequence b occupies packed
# tokens cu_seqlens[b] .. cu_seqlens[b+1]-1; it is sliced out and processed
# as one single-sequence call, so quantisation groups, the smooth_k mean and
# the causal alignment are all per sequence.
# --------------------------------------------------------------------------

def seq_bounds(cu_seqlens):
    cu = np.asarray(cu_seqlens, np.int64)
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]


def quant_int8_varlen(x, cu_seqlens, block_tokens: int = 1, smooth: bool = False):
    """Per-sequence INT8 quantisation of a packed batch.

    x: float32 [total, H, D] (token-major, as packed batches are stored).
    Returns (q int8 [H, total, D], scales: list over sequences of fp32
    [H, ceil(len_b / block_tokens)], mu fp32 [B, H, D] or None).  An empty
    sequence has no groups and a zero mean.
    """
    x = _c(x, np.float32)
    total, H, D = x.shape
    bounds = seq_bounds(cu_seqlens)
    q = np.zeros((H, total, D), np.int8)
    scales = []
    mu = np.zeros((len(bounds), H, D), np.float32) if smooth else None
    for b, (t0, t1) in enumerate(bounds):
        if t1 == t0:
            scales.append(np.zeros((H, 0), np.float32))
            continue
        xb = np.ascontiguousarray(x[t0:t1].transpose(1, 0, 2))   # [H, len, D]
        qb, sb, mb = quant_int8(xb, block_tokens=block_tokens, smooth=smooth)
        q[:, t0:t1] = qb
        scales.append(sb)
        if smooth:
            mu[b] = mb
    return q, scales, mu


def row_bias_varlen(x, cu_seqlens, mu):
    """b[h, t] = sum_c x[t, h, c] mu[b(t), h / (H / Hmu), c] in fp64.

    x: [total, H, D]; mu: [B, Hmu, D].  Returns fp64 [H, total].
    """
    x = _c(x, np.float32)
    mu = _c(mu, np.float32)
    total, H, _ = x.shape
    out = np.zeros((H, total), np.float64)
    for b, (t0, t1) in enumerate(seq_bounds(cu_seqlens)):
        if t1 > t0:
            xb = np.ascontiguousarray(x[t0:t1].transpose(1, 0, 2))[None]
            out[:, t0:t1] = row_bias(xb, mu[b:b + 1])[0]
    return out


def prefill_varlen(q_i8, q_scales, q_block, k_i8, k_scales, k_block, v, cu_seqlens_q,
                   cu_seqlens_k, *, causal, sm_scale=None, q_bias=None, rows=None,
                   threads=None, smooth_v=False):
    """Prefill attention over a packed batch, one single-sequence call each.

    q_i8 int8 [Hq, total_q, D]; q_scales list of fp32 [Hq, ceil(len_q_b / q_block)];
    k_i8 int8 [Hkv, total_k, D]; k_scales list of fp32 [Hkv, ceil(len_k_b / k_block)];
    v float [total_k, Hkv, D]; q_bias fp64 [Hq, total_q] or None (the
    sequence's keys are smoothed); causal alignment bottom-right within
    each sequence.  rows: optional list over sequences of row indices
    (within the sequence) to evaluate; other rows stay NaN.
    Returns (o fp64 [total_q, Hq, D], lse fp64 [Hq, total_q]).
    """
    q_i8 = np.asarray(q_i8)
    Hq, total_q, D = q_i8.shape
    o = np.full((total_q, Hq, D), np.nan)
    lse = np.full((Hq, total_q), np.nan)
    bq, bk = seq_bounds(cu_seqlens_q), seq_bounds(cu_seqlens_k)
    for b, ((q0, q1), (k0, k1)) in enumerate(zip(bq, bk)):
        if q1 == q0:
            continue
        if k1 == k0:
            # no keys: nothing to attend to (zero output, empty sum)
            sel = np.arange(q1 - q0) if rows is None else np.asarray(rows[b], np.int64)
            o[q0 + sel] = 0.0
            lse[:, q0 + sel] = -np.inf
            continue
        sel = None if rows is None else rows[b]
        qb = None if q_bias is None else np.asarray(q_bias)[None, :, q0:q1]
        ob, lb = prefill(q_i8[None, :, q0:q1], np.asarray(q_scales[b])[None], q_block,
                         np.asarray(k_i8)[None, :, k0:k1], np.asarray(k_scales[b])[None], k_block,
                         np.asarray(v)[k0:k1].transpose(1, 0, 2)[None], causal=causal,
                         sm_scale=sm_scale, q_bias=qb, rows=sel, threads=threads,
                         smooth_v=smooth_v)
        idx = np.arange(q1 - q0) if sel is None else np.asarray(sel, np.int64)
        o[q0 + idx] = ob[0].transpose(1, 0, 2)
        lse[:, q0 + idx] = lb[0]
    return o, lse
