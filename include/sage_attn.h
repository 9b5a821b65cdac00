/*
 * sage_attn.h -- C ABI of libsageattn.so: INT8-QK quantized attention for
 * GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [P1] "INT8 QK MMAC on gfx936 DCU: paged access, fragment mapping and
 *        GQA" (forum.sourcefind.cn) -- quantisation rule (section 4), score
 *        recovery (section 1), INT32 bound (section 2.1), paged K cache
 *        layout and lookup (section 3), split-K decode and GQA (sections
 *        4-5), reject-don't-guess applicability checks (section 7).
 *   [P3] "SageAttention -- MetaX MXMACA port" README (gitlink.org.cn) --
 *        per-block granularity CTA_Q=128 / CTA_K=64, smooth_k with LSE
 *        correction, causal masking, base-2 online softmax, FP16 P.V with
 *        FP32 accumulation, LSE return (feature matrix, attention kernel
 *        pipeline, advanced configuration).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller unless
 *     the comment says "host".  The library never allocates, frees or
 *     keeps a pointer beyond the call.
 *   - Work is enqueued on the caller's CUDA stream (`stream`, a
 *     cudaStream_t passed as void*; NULL = legacy default stream).  No call
 *     synchronises except sage_check_device_status().
 *   - Tensors are dense row-major unless strides are given; "[B,H,S,D]"
 *     lists dimensions outermost first.
 *   - Every call returns a sage_status_t and never throws or aborts.  On
 *     failure nothing has been enqueued (argument errors) or the launch
 *     failed (SAGE_ERR_CUDA); sage_get_last_error_message() tells why.
 *   - Kernels never trap.  Every wait inside a kernel is bounded; a wait
 *     that runs out, a block-table entry outside [0, num_blocks) or a
 *     context length outside [0, max_context_len] sets a per-device error
 *     word that sage_check_device_status() reads; the offending page is
 *     not read (its keys are masked) and the length is clamped.
 */
#ifndef SAGE_ATTN_H
#define SAGE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sage_status {
    SAGE_OK = 0,
    SAGE_ERR_INVALID_ARG = 1,   /* null pointer, bad shape/stride/alignment, GQA mismatch */
    SAGE_ERR_UNSUPPORTED = 2,   /* valid request outside what this build implements */
    SAGE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    SAGE_ERR_TIMEOUT = 4,       /* device error word: a bounded wait ran out */
    SAGE_ERR_BAD_BLOCK = 5      /* device error word: block-table entry or length out of range */
} sage_status_t;

typedef enum sage_dtype {
    SAGE_F16 = 0,
    SAGE_BF16 = 1
} sage_dtype_t;

/* Message of the last failing call on the calling host thread. */
const char *sage_get_last_error_message(void);

/* Library ABI version (increments on any signature change). */
int sage_version(void);   /* 6 */

/* --------------------------------------------------------------------------
 * Quantisation  ([P1] section 4; [P3] quant kernel table, feature matrix)
 *
 * Symmetric dynamic INT8 quantisation of x [B,H,S,D]:
 *   group = one token row (block_tokens == 1) or block_tokens consecutive
 *   tokens of one (b, h) (per-block granularity, 128 for Q and 64 for K);
 *   s = amax / 127 in fp32 (amax = max |x| over the group; s = 0 when
 *   amax = 0);  q = round-to-nearest-even(fp32(x / s)) in [-127, 127].
 * smooth != 0: first computes mu[b,h,c] = mean over the S tokens of
 *   x[b,h,:,c] (exact sum, rounded once to fp32) and quantises x - mu
 *   (smooth_k).
 * mu_in != NULL: also writes the row bias bias[b,h,s] = sum_c x[b,h,s,c] *
 *   mu_in[b, h / (H / mu_heads), c] (fp32), the term smooth_k removes from
 *   the scores of Q against smoothed K.
 *
 * x        : f16/bf16, element strides (stride_b, stride_h, stride_s) with the
 *            channel dimension contiguous; the base address and every row
 *            must be 16-byte aligned (strides multiples of 8 elements).  HND
 *            and NHD layouts are both expressed through the strides.
 * D        : 64, 128 or 256.   block_tokens: 1..1024.
 * x_int8   : int8 [B,H,S,D] dense (HND).
 * scale    : fp32 [B,H,ceil(S/block_tokens)].
 * mu_out   : fp32 [B,H,D], required iff smooth; 16-byte aligned.
 * mu_in    : fp32 [B,mu_heads,D], 16-byte aligned.
 * bias_out : fp32 [B,H,S], required iff mu_in.
 * ------------------------------------------------------------------------ */
sage_status_t sage_quant_int8(const void *x, sage_dtype_t dtype, int B, int H, int S, int D,
                              int64_t stride_b, int64_t stride_h, int64_t stride_s,
                              int block_tokens, int smooth, const float *mu_in, int mu_heads,
                              int8_t *x_int8, float *scale, float *mu_out, float *bias_out,
                              void *stream);

/* --------------------------------------------------------------------------
 * Variable-length packed batches  ([P3] "Varlen per-batch loop": each
 * sequence of a packed batch is sliced out and processed as one
 * single-sequence call; the roadmap's batched varlen kernel is what the
 * calls below provide, one launch for the whole batch)
 *
 * Sequence b holds packed tokens cu_seqlens[b] .. cu_seqlens[b+1]-1
 * (cu_seqlens: int32 [B+1] device array, cu_seqlens[0] >= 0,
 * non-decreasing, cu_seqlens[B] <= total, each length <= the caller's
 * max_seqlen).  Packed tokens outside every sequence are not read or
 * written.  A sequence that breaks these rules sets the bad-block bit of
 * the device error word and is treated as empty; where cu_seqlens
 * decreases, the kernels' searches over it may misplace the other
 * sequences' tiles too, so their results are then unspecified (nothing is
 * read or written outside the tensors).
 *
 * Scale groups: per token (block_tokens == 1) group = packed token; per
 * block, sequence b's groups start at cu_seqlens[b] / block_tokens + b and
 * cover its own tokens only (ceil(len / block_tokens) groups; one unused
 * slot per sequence at most, holding 0).  sage_varlen_scale_groups() gives
 * the groups per head: total (per token) or total / block_tokens + B.
 *
 * sage_quant_int8_varlen: the rule of sage_quant_int8, per sequence.
 *   x        : f16/bf16 [total, H, D] through element strides (stride_t
 *              between tokens, stride_h between heads), channels contiguous,
 *              16-byte aligned, strides multiples of 8.
 *   x_int8   : int8 [H, total, D].   scale: fp32 [H, groups].
 *   smooth   : mu_out fp32 [B, H, D] = each sequence's own token mean (0 for
 *              an empty sequence), subtracted before quantising; 16-byte
 *              aligned.
 *   mu_in    : optional fp32 [B, mu_heads, D], 16-byte aligned; bias_out fp32 [H, total] =
 *              sum_c x[t,h,c] * mu_in[b(t), h / (H / mu_heads), c].
 * ------------------------------------------------------------------------ */
int64_t sage_varlen_scale_groups(int64_t total, int B, int block_tokens);

sage_status_t sage_quant_int8_varlen(const void *x, sage_dtype_t dtype, int B, int H,
                                     int64_t total, int D, int64_t stride_h, int64_t stride_t,
                                     const int32_t *cu_seqlens, int max_seqlen, int block_tokens,
                                     int smooth, const float *mu_in, int mu_heads,
                                     int8_t *x_int8, float *scale, float *mu_out,
                                     float *bias_out, void *stream);

/* --------------------------------------------------------------------------
 * Paged INT8 K/V cache  ([P1] section 3)
 *   k_cache, v_cache : int8 [num_blocks, Hkv, D/16, 16, 16]; token t of a
 *                      sequence sits in physical block block_table[b][t/16],
 *                      slot t % 16; channel c at [c/16][slot][c%16].
 *   k_scale, v_scale : fp32 [num_blocks, Hkv, 16], per token and KV head.
 *   block_table      : int32 [B, max_blocks].
 * ------------------------------------------------------------------------ */

/* --------------------------------------------------------------------------
 * KV producer: append new tokens to the paged INT8 cache  ([P1] sections 3, 4)
 *
 * k_new, v_new: f16/bf16 [B, Hkv, n_new, D] contiguous, 16-byte aligned.
 * Row t of sequence b is token positions[b] + t: it is quantised per token
 * and KV head (s = max|x| / 127 in fp32, codes rne(x / s) clamped to
 * [-127, 127]; an all-zero row gives s = 0 and codes 0, the rule of
 * sage_quant_int8) and written to page block_table[b][pos / 16], slot
 * pos % 16, in the cache layout above, with its scale at
 * k_scale/v_scale[page][kv_head][slot].  positions (int32 [B]) and
 * block_table are device arrays read on the GPU: a position outside the
 * table or a page outside [0, num_blocks) skips that row and sets the
 * bad-block bit of the device error word (sage_check_device_status).
 * Rows of different sequences must not share a page slot.
 * ------------------------------------------------------------------------ */
sage_status_t sage_kv_cache_append(const void *k_new, const void *v_new, sage_dtype_t dtype,
                                   int B, int Hkv, int n_new, int D,
                                   const int32_t *block_table, int max_blocks,
                                   const int32_t *positions, int num_blocks, int8_t *k_cache,
                                   int8_t *v_cache, float *k_scale, float *v_scale, void *stream);

/* The KV producer of a decode or prefill step ([P1] section 4: the query
 * is quantised once, in the producer that writes the step's K/V, and every
 * split-K segment reuses its codes): sage_kv_cache_append's K/V rows plus
 * the step's query rows in ONE launch.  q_new f16/bf16 [B, Hq, n_new, D]
 * (same dtype as k_new/v_new, 16-byte aligned) is quantised per (token,
 * head) with the rule of sage_quant_int8 into q_int8 [B, Hq, n_new, D]
 * (8-byte aligned) and q_scale [B, Hq, n_new] fp32 -- for a decode step
 * (n_new = 1) exactly the q / q_scale that sage_attn_decode_paged reads.
 * Errors and bad pages as sage_kv_cache_append; query rows never touch
 * the cache.  All pointers are device memory. */
sage_status_t sage_kv_producer(const void *q_new, const void *k_new, const void *v_new,
                               sage_dtype_t dtype, int B, int Hq, int Hkv, int n_new, int D,
                               const int32_t *block_table, int max_blocks,
                               const int32_t *positions, int num_blocks, int8_t *k_cache,
                               int8_t *v_cache, float *k_scale, float *v_scale, int8_t *q_int8,
                               float *q_scale, void *stream);

/* --------------------------------------------------------------------------
 * Split-K paged decode  ([P1] sections 1, 3, 4, 5)
 *
 * One new query token per sequence.  Query head h reads KV head
 * h / (Hq / Hkv) (GQA).  For each (b, h):
 *   acc_j = sum_c q[b,h,c] * k_j[c]                      (exact INT32)
 *   t_j   = acc_j * q_scale[b,h] * k_scale_j * sm_scale   (per score)
 *   o     = sum_j softmax(t)_j * v_scale_j * v_j          (FP32 accumulation)
 *   lse   = ln sum_j exp(t_j)
 * The context is cut into num_segments contiguous runs of pages; each is
 * reduced on its own and the partials are merged by the LSE combine
 * (sage_splitk_combine).  With 2..8 segments the segments of one (sequence,
 * KV head) run as one thread-block cluster and the combine happens in
 * distributed shared memory inside the same kernel (one launch, no partials
 * in device memory); with more segments the partials go through the
 * workspace and the combine kernel.
 * Per-step inputs and outputs -- q (or the f16/bf16 query of the _q16 form),
 * q_scale, block_table, context_lens, out and lse -- may be device memory
 * or pinned host memory that the GPU addresses at the same pointer (as on
 * GB300, whose kernels then read and write it over NVLink-C2C with no
 * copy-engine transfer); any other pointer is rejected with
 * SAGE_ERR_INVALID_ARG.  The caches, scales and workspace must be device
 * memory.
 * ------------------------------------------------------------------------ */
typedef struct sage_decode_args {
    const int8_t *q;            /* [B, Hq, D] int8 (sage_quant_int8 output) */
    const float *q_scale;       /* [B, Hq] fp32 */
    const int8_t *k_cache;      /* paged layout above */
    const int8_t *v_cache;
    const float *k_scale;       /* [num_blocks, Hkv, 16] */
    const float *v_scale;
    const int32_t *block_table; /* [B, max_blocks] */
    const int32_t *context_lens;/* [B], each in [0, max_context_len] */
    int B, Hq, Hkv, D;          /* D = 64, 128 or 256; Hq % Hkv == 0 */
    int num_blocks, max_blocks;
    int max_context_len;        /* host-side bound on context_lens, <= 16 * max_blocks */
    float sm_scale;             /* <= 0 selects 1/sqrt(D) */
    int num_segments;           /* 0 selects sage_decode_num_segments() */
    void *out;                  /* [B, Hq, D], 8-byte aligned */
    sage_dtype_t out_dtype;
    float *lse;                 /* optional [B, Hq] natural-log LSE (-inf for empty context) */
    int pv_mode;                /* SAGE_PV_* below; 0 = SAGE_PV_F32 */
} sage_decode_args_t;

/* P.V of the decode ([P3] advanced configuration, pv_accum_dtype "fp32" /
 * "fp16" / "fp16+fp16"; [P1] sections 6 and 8: INT8 P.V with the V scale
 * fused into P).  The INT8 values of a page enter the product exactly in
 * every mode; P' = p_j * v_scale_j (p = 2^(t_j - m), m a running row max).
 *   SAGE_PV_F32      P' rounded to f16, fp32 accumulation (default)
 *   SAGE_PV_F16      P' rounded to f16, f16 accumulation throughout
 *   SAGE_PV_F16_F32  each 16-key page's product accumulated in f16, then
 *                    added into fp32 accumulators (two-level accumulation)
 *   SAGE_PV_INT8     P' quantised per (query head, 16-key page):
 *                    s = max_j P' / 127, codes rne(P' / s) in [0, 127]
 *                    (the rounding of sage_quant_int8); the page adds
 *                    s * sum_j code_j * v_j, the sum exact, to fp32
 *                    accumulators; the softmax denominator uses unquantised p.
 * On this GPU the four run at the same tensor rate; F32 is the most precise. */
enum {
    SAGE_PV_F32 = 0,
    SAGE_PV_F16 = 1,
    SAGE_PV_F16_F32 = 2,
    SAGE_PV_INT8 = 3
};

/* Segment count the library picks for num_segments == 0 (host only).  With
 * U = B * Hkv * ceil(Hq/Hkv/8) (sequence, KV head, 8-head tile) units and
 * P = ceil(max_context_len/16) pages: S = 2.5 SMs / U rounded (one wave of
 * about 2.5 CTAs per SM), or, when that is below 2, S = 5 SMs / U rounded
 * (several waves of shorter CTAs); when floor(R SMs / U) is above 8 (R the
 * decode kernel's CTAs per SM for this D, the segments then merged by the
 * combine kernel rather than in a cluster) and not below that choice, S is
 * that one full wave instead; at least 8 pages per segment, at most 64
 * segments.  This is the choice for device-resident per-step inputs; a call
 * with num_segments == 0 whose query, block table or output is pinned host
 * memory starts from about 1.7 CTAs per SM instead of 2.5 (each segment's
 * CTA reads its inputs across the CPU-GPU link), the full-wave clause
 * alike.  The rule is empirical, measured on GB300. */
int sage_decode_num_segments(int B, int Hq, int Hkv, int D, int max_context_len);

/* The segment count a decode call with args->num_segments == 0 will use,
 * taking into account where its per-step inputs and output live (q: the
 * f16/bf16 query of the _q16 form, or NULL for args->q).  Host only; use it
 * to size the workspace. */
int sage_decode_auto_segments(const sage_decode_args_t *args, const void *q);

/* Bytes of workspace sage_attn_decode_paged may need (0 when S == 1): fp32
 * partial outputs [B,Hq,S,D], fp32 partial LSEs [B,Hq,S], then int8 query
 * codes [B,Hq,D] and fp32 scales [B,Hq], each region 256-byte aligned.  A
 * call with 2..8 segments normally combines in-cluster and leaves the
 * partials untouched (it uses them only if the cluster launch is refused);
 * the query regions serve sage_attn_decode_paged_q16 with a query in pinned
 * host memory. */
size_t sage_attn_decode_workspace_size(int B, int Hq, int D, int num_segments);

/* workspace: device buffer of at least sage_attn_decode_workspace_size()
 * bytes, 16-byte aligned; may be NULL when the segment count is 1.  Its
 * contents are scratch and are overwritten. */
sage_status_t sage_attn_decode_paged(const sage_decode_args_t *args, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Same decode with the query quantisation fused in: q is the f16/bf16 query
 * [B, Hq, D] (8-byte aligned); args->q and args->q_scale are ignored.  Each
 * CTA quantises the query rows of its heads per (token, head) with the
 * arithmetic of sage_quant_int8 ([P1] section 4: s = max|q| / 127, codes
 * round(q / s)), so the codes and the result equal sage_quant_int8 followed
 * by sage_attn_decode_paged bit for bit; the split-K segments recompute the
 * same codes instead of reading them from a separate launch.  Exception:
 * with a query in pinned host memory and more than one segment, the query
 * is quantised once into the workspace (by the sage_quant_int8 kernel, one
 * extra launch) and the decode, launched behind it, reads the codes -- every
 * segment reading the query across the CPU-GPU link cost more. */
sage_status_t sage_attn_decode_paged_q16(const sage_decode_args_t *args, const void *q,
                                         sage_dtype_t q_dtype, void *workspace,
                                         size_t workspace_bytes, void *stream);

/* Same decode, without the combine: writes each segment's normalised output
 * o_part [B*Hq, S, D] and natural-log LSE lse_part [B*Hq, S] (fp32, caller
 * buffers, o_part 16-byte aligned; 0 / -inf for a segment with no keys).
 * num_segments must be >= 1; segments that would start past the longest
 * context are dropped, so S = ceil(P / ceil(P / num_segments)) with
 * P = ceil(max_context_len / 16) (S = 1 when P = 0); S is also returned in
 * *segments_used (host, optional).  sage_splitk_combine over these
 * partials gives the sage_attn_decode_paged result. */
sage_status_t sage_attn_decode_paged_partials(const sage_decode_args_t *args, float *o_part,
                                              float *lse_part, int *segments_used, void *stream);

/* --------------------------------------------------------------------------
 * Allocation-free decode (no counterpart on the source pages: a deployment
 * convenience of this library).
 *
 * Same computation and result as sage_attn_decode_paged, for callers that
 * cannot hand the library a workspace: code inside a CUDA graph captured
 * with a fixed memory plan, plugins whose host framework owns every device
 * allocation, or embedders that must not re-enter their allocator from the
 * attention call.  The split-K partials live in one device array built into
 * the library, of sage_attn_decode_noalloc_max_bytes() bytes (8 MiB) per
 * GPU that loads the library, held until the process exits.  The call
 * allocates and frees nothing.
 *   - Arguments are checked exactly as by sage_attn_decode_paged (shapes,
 *     alignment, per-step buffers in device or mapped pinned host memory)
 *     before anything is launched.
 *   - num_segments 0: the library's own choice (sage_decode_auto_segments),
 *     lowered to the largest count whose partials fit the array.  An
 *     explicit count whose partials exceed it (B*Hq*S*(D+1)*4 bytes, S the
 *     segment count actually used) is rejected with SAGE_ERR_INVALID_ARG and
 *     a message saying how many bytes were needed; with one segment no
 *     scratch is used at all.  The segments always merge in the combine
 *     kernel (two launches), never in a thread-block cluster.
 *   - The first call on a device looks the array's address up
 *     (cudaGetSymbolAddress); make that first call outside any stream
 *     capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; each call overwrites every slot it reads, so nothing needs
 *     clearing, but calls that overlap on the GPU (different streams, no
 *     ordering between them) race on the array: serialise them.
 * ------------------------------------------------------------------------ */
size_t sage_attn_decode_noalloc_max_bytes(void);
sage_status_t sage_attn_decode_paged_noalloc(const sage_decode_args_t *args, void *stream);

/* --------------------------------------------------------------------------
 * Split-K LSE combine  ([P1] section 4 split-K; [P3] LSE returned "for
 * concatenation").  For every row r:
 *   M = max_s lse_part[r,s],  L = M + ln sum_s exp(lse_part[r,s] - M)
 *   out[r] = sum_s exp(lse_part[r,s] - L) * o_part[r,s]
 * Segments with lse = -inf are skipped; a row with no live segment gets
 * out = 0 and lse = -inf.
 * o_part : fp32 [R, S, D] (each segment's output, already normalised)
 * lse_part: fp32 [R, S] natural log.  out: [R, D] of out_dtype.
 * lse_out : optional fp32 [R].  D = 64, 128 or 256; 1 <= S <= 1024.
 * ------------------------------------------------------------------------ */
sage_status_t sage_splitk_combine(const float *o_part, const float *lse_part, int R, int S, int D,
                                  void *out, sage_dtype_t out_dtype, float *lse_out,
                                  void *stream);

/* --------------------------------------------------------------------------
 * Prefill  ([P3] attention kernel pipeline and advanced configuration;
 * [P1] sections 5.2 and 7 for chunked prefill over a paged INT8 history)
 *
 * Queries [B,Hq,Sq,D] attend to Sp paged prefix keys (optional) followed by
 * Sk contiguous chunk keys.  Query head h reads KV head h / (Hq/Hkv).
 *   acc_ij = sum_c q_ic k_jc                         (exact INT32)
 *   z_ij   = sm_scale * (acc_ij * sq_i * sk_j + [j in chunk and q_bias] * q_bias_i)
 *   causal: key j (index over prefix + chunk) is visible to query i iff
 *           j <= i + (Sp + Sk - Sq)  (bottom-right alignment)
 *   o_i    = sum_j softmax(z)_ij v_j,  v_j = v_scale_j * v_int8_j (prefix) or
 *            the f16/bf16 value (chunk);  P.V in 16-bit with FP32 accumulation
 *   lse_i  = ln sum_j exp(z_ij)
 * q_bias (from sage_quant_int8's bias_out with the K mean) restores the
 * scores of smoothed chunk keys; with no prefix it only shifts the LSE
 * ([P3]'s LSE correction).
 * smooth_v ([P3] feature matrix "V mean fusion", SubMean kernel, output
 * stage "V mean added back"): mu[b,kvh,c] = mean over the chunk's Sk
 * tokens of v[b,kvh,:,c] (exact sum rounded once to fp32, as smooth_k's
 * mean) is subtracted from every value the rows attend to (prefix included,
 * rounded to f16 after an fp32 subtraction) and added to o_i; a row that
 * sees no key keeps o_i = 0.  The result equals the unsmoothed one in exact
 * arithmetic; the f16 P.V operand carries (v - mu) instead of v.  v_mean
 * (optional, [B, Hkv, D] fp32) receives mu.
 * ------------------------------------------------------------------------ */
typedef struct sage_prefill_args {
    int B, Hq, Hkv, Sq, Sk, D;      /* D = 64, 128 or 256; Sk may be 0 with a prefix */
    const int8_t *q;                /* [B, Hq, Sq, D] int8 */
    const float *q_scale;           /* [B, Hq, ceil(Sq / q_block)] */
    int q_block;                    /* 1 (per token) or a multiple of 128 */
    const int8_t *k;                /* [B, Hkv, Sk, D] int8 (chunk keys) */
    const float *k_scale;           /* [B, Hkv, ceil(Sk / k_block)] */
    int k_block;                    /* 1 (per token) or a multiple of 64 */
    const void *v;                  /* [B, Hkv, Sk, D] chunk values */
    sage_dtype_t v_dtype;           /* P.V runs in this 16-bit type */
    const float *q_bias;            /* optional [B, Hq, Sq]: chunk keys are smoothed */
    /* optional paged INT8 prefix (all NULL / 0 when absent) */
    const int8_t *k_cache, *v_cache;
    const float *k_cache_scale, *v_cache_scale;
    const int32_t *block_table;     /* [B, max_blocks] */
    const int32_t *prefix_lens;     /* [B] device; each <= max_prefix_len */
    int num_blocks, max_blocks, max_prefix_len;
    int causal;
    float sm_scale;                 /* <= 0 selects 1/sqrt(D) */
    void *out;                      /* [B, Hq, Sq, D] */
    sage_dtype_t out_dtype;
    float *lse;                     /* optional [B, Hq, Sq] */
    int smooth_v;                   /* subtract the chunk's V mean, add it back to o */
    float *v_mean;                  /* optional out [B, Hkv, D] fp32 (smooth_v) */
    int layout;                     /* SAGE_LAYOUT_HND (0) or SAGE_LAYOUT_NHD (1), below */
    int tail_split;                 /* SAGE_TAIL_SPLIT_AUTO (0) or SAGE_TAIL_SPLIT_OFF (1), below */
} sage_prefill_args_t;

/* Layout of the prefill's f16/bf16 tensors ([P3] tensor_layout): HND keeps
 * v [B, Hkv, Sk, D] and out [B, Hq, Sq, D]; NHD takes v [B, Sk, Hkv, D] and
 * writes out [B, Sq, Hq, D].  The INT8 codes, scales, q_bias and lse are
 * head-major in both (the layout sage_quant_int8 writes). */
enum { SAGE_LAYOUT_HND = 0, SAGE_LAYOUT_NHD = 1 };

/* Split of the last wave (head_dim 256).  A CTA there takes one 128-row query
 * tile.  When the tiles leave the last wave of CTAs partly empty and carry
 * about equal work (no causal mask, or a chunk over much longer history),
 * AUTO splits that wave's tiles by key range into up to 8 parts of at least
 * 16 key tiles.  Each part is one CTA.
 * A second kernel merges the parts with the split-K combine ("INT8 QK MMAC
 * on gfx936 DCU", section 4).  The parts' results are normalised outputs and
 * their base-2 LSEs, kept in the workspace.  The result is the same attention
 * to within rounding, but not bit-for-bit the unsplit computation.  OFF never
 * splits.  The choice changes the workspace size, so pass the same args to
 * sage_attn_prefill_workspace_size. */
enum { SAGE_TAIL_SPLIT_AUTO = 0, SAGE_TAIL_SPLIT_OFF = 1 };

/* Workspace of sage_attn_prefill (host only).  The tensor cores of sm_103a
 * have no INT8 mode, so each call first expands the INT8 codes it reads
 * into an exact f16 copy, together with per-key scales.  Those codes are
 * chunk K, and the paged prefix's K and V gathered through the block table.
 * bf16 chunk V is rounded to f16 there too.  With a tail split (above) the
 * workspace also holds the split tiles' partial results.  Returns the bytes
 * needed; 0 only for an invalid request.  The stored representation stays
 * INT8; the copy is scratch of the call.  The size depends on the current
 * device's SM count through the tail split. */
size_t sage_attn_prefill_workspace_size(const sage_prefill_args_t *args);

/* workspace: device buffer of at least sage_attn_prefill_workspace_size()
 * bytes, 256-byte aligned; overwritten by the call. */
sage_status_t sage_attn_prefill(const sage_prefill_args_t *args, void *workspace,
                                size_t workspace_bytes, void *stream);

/* --------------------------------------------------------------------------
 * Varlen prefill  ([P3] "Varlen per-batch loop" and roadmap; the attention
 * itself is sage_attn_prefill's, per sequence)
 *
 * For every sequence b: its queries (cu_seqlens_q) attend to its keys
 * (cu_seqlens_k) exactly as sage_attn_prefill with B = 1 and no prefix
 * would, including the per-score scale recovery, the smooth_k bias and the
 * bottom-right causal alignment j <= i + (Sk_b - Sq_b).  A sequence with
 * queries and no keys gets out = 0 and lse = -inf.  One staging launch and
 * one attention launch cover the whole batch.
 *   q       : int8 [Hq, total_q, D] (sage_quant_int8_varlen),
 *   q_scale : fp32 [Hq, sage_varlen_scale_groups(total_q, B, q_block)],
 *   k       : int8 [Hkv, total_k, D], k_scale likewise with k_block,
 *   v       : f16/bf16 [total_k, Hkv, D] through element strides
 *             (v_stride_t, v_stride_h; 0 selects the dense packing),
 *             multiples of 8, 16-byte aligned,
 *   q_bias  : optional fp32 [Hq, total_q] (the sequences' keys are smoothed),
 *   out     : [total_q, Hq, D] (16-byte aligned), lse: optional fp32 [Hq, total_q].
 * B <= 65535.  D, q_block, k_block, dtypes and sm_scale as in sage_attn_prefill.
 * ------------------------------------------------------------------------ */
typedef struct sage_prefill_varlen_args {
    int B, Hq, Hkv, D;
    int64_t total_q, total_k;       /* packed query / key tokens */
    int max_seqlen_q, max_seqlen_k; /* host bounds on the sequences' lengths */
    const int32_t *cu_seqlens_q;    /* [B + 1] device */
    const int32_t *cu_seqlens_k;    /* [B + 1] device */
    const int8_t *q;
    const float *q_scale;
    int q_block;
    const int8_t *k;
    const float *k_scale;
    int k_block;
    const void *v;
    sage_dtype_t v_dtype;
    int64_t v_stride_t, v_stride_h;
    const float *q_bias;
    int causal;
    float sm_scale;                 /* <= 0 selects 1/sqrt(D) */
    void *out;
    sage_dtype_t out_dtype;
    float *lse;
    int smooth_v;                   /* per-sequence V mean, as sage_attn_prefill's */
    float *v_mean;                  /* optional out [B, Hkv, D] fp32 (smooth_v) */
} sage_prefill_varlen_args_t;

/* Workspace bytes of sage_attn_prefill_varlen (host only): the f16 copy of
 * every sequence's keys and values, each padded to whole key tiles. */
size_t sage_attn_prefill_varlen_workspace_size(const sage_prefill_varlen_args_t *args);

/* workspace: at least sage_attn_prefill_varlen_workspace_size() bytes,
 * 256-byte aligned; overwritten by the call. */
sage_status_t sage_attn_prefill_varlen(const sage_prefill_varlen_args_t *args, void *workspace,
                                       size_t workspace_bytes, void *stream);

/* --------------------------------------------------------------------------
 * Test hooks: raw INT32 scores through the same device tile paths
 * ([P1] section 7, layer 1: check the lane/fragment mapping of the raw
 * accumulators).
 * sage_debug_prefill_qk_int32: runs sage_attn_prefill and also writes
 *   scores[b,h,i,j] = acc_ij for every visible (i, j); masked entries are
 *   left untouched.  scores: int32 [B, Hq, Sq, max_prefix_len + Sk].
 * sage_debug_decode_qk_int32: runs sage_attn_decode_paged and writes
 *   scores[b,h,j] for j < context_lens[b]; scores: int32 [B, Hq, max_context_len].
 * ------------------------------------------------------------------------ */
sage_status_t sage_debug_prefill_qk_int32(const sage_prefill_args_t *args, void *workspace,
                                          size_t workspace_bytes, int32_t *scores,
                                          void *stream);
/* sage_debug_prefill_varlen_qk_int32: the same for a packed batch;
 *   scores[h, t, j] (int32 [Hq, total_q, max_seqlen_k]) for query token t
 *   and key j of t's sequence. */
sage_status_t sage_debug_prefill_varlen_qk_int32(const sage_prefill_varlen_args_t *args,
                                                 void *workspace, size_t workspace_bytes,
                                                 int32_t *scores, void *stream);
sage_status_t sage_debug_decode_qk_int32(const sage_decode_args_t *args, void *workspace,
                                         size_t workspace_bytes, int32_t *scores, void *stream);

/* --------------------------------------------------------------------------
 * Runtime-path evidence ([P1] section 7, layer 4: prove the target kernel
 * ran).  Describes the last kernel launched by the calling host thread.
 * ------------------------------------------------------------------------ */
typedef struct sage_launch_info {
    char kernel[64];
    int grid[3];
    int block[3];
    int cluster[3];
    int smem_bytes;
    int num_segments;
    int launches;               /* kernels enqueued by the last API call */
} sage_launch_info_t;

sage_status_t sage_last_launch_info(sage_launch_info_t *info /* host */);

/* Synchronises `stream`, reads and clears the current device's error word.
 * Returns SAGE_OK, SAGE_ERR_TIMEOUT or SAGE_ERR_BAD_BLOCK (or SAGE_ERR_CUDA).
 * `detail` (host, optional) receives the raw word. */
sage_status_t sage_check_device_status(void *stream, int *detail);

/* Test hook for the bounded-wait path: launches a kernel that waits on an
 * mbarrier nothing arrives on, with a limit of `timeout_us` microseconds
 * (1..5,000,000); the kernel gives up, sets SAGE_ERR_TIMEOUT in the error
 * word and returns.  Used to show the context stays usable. */
sage_status_t sage_debug_timeout_probe(int timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_ATTN_H */
