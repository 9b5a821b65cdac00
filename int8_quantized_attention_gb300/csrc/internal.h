// Internal (non-exported) interface between the C-ABI host layer and the
// kernel translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "sage_attn.h"

namespace sage {

// Record of the kernels one API call enqueued (runtime-path evidence).
struct LaunchLog {
    char kernel[64] = {0};
    dim3 grid, block, cluster;
    int smem = 0;
    int segments = 0;
    int count = 0;
    void add(const char *name, dim3 g, dim3 b, dim3 c, int sm) {
        strncpy(kernel, name, sizeof(kernel) - 1);
        grid = g;
        block = b;
        cluster = c;
        smem = sm;
        ++count;
    }
};

// Division of 32-bit n < 2^31 by an invariant divisor d (1 <= d < 2^31)
// as a multiply-high and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (mulhi(n, m) + n) >> l; mulhi(n, m) <= n keeps the sum in 32 bits.
struct FastDiv {
    uint32_t d = 1, m = 1;
    int l = 0;
    FastDiv() = default;
    explicit FastDiv(uint32_t div) : d(div) {
        l = 0;
        while ((1ull << l) < d) ++l;
        m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    }
#ifdef __CUDACC__
    __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> l; }
#endif
};

struct QuantParams {
    const void *x;
    int bf16;
    int B, H, S, D;
    int64_t sb, sh, ss;
    int block;                // tokens per group (1 = per token)
    int smooth;
    const float *mu_sub;      // set internally to mu_out after the mean pass
    const float *mu_bias;     // optional mean for the row bias
    int mu_heads;
    int8_t *q;
    float *scale;
    float *mu_out;
    float *bias;
    // packed variable-length batch (cu == null: the dense [B,H,S,D] form):
    // sequence b is tokens [cu[b], cu[b+1]) of x [total, H, D] (strides sh,
    // ss); S is the caller's bound on a sequence's length; codes [H, total, D],
    // scales [H, groups], mu [B, H, D], bias [H, total]
    const int32_t *cu;
    int64_t total;
    int64_t groups;
    int *err;
    // per-token kernels: rows are (outer, inner) pairs, outer = b * H + h and
    // inner = s (dense) or outer = h and inner = t (packed); one launch takes
    // outers [outer0, outer0 + n_outer) with n_outer * inner < 2^31
    int64_t outer0;
    uint32_t n_outer;
    FastDiv div_inner, div_h, div_grp;
    // dense per-block kernel: CTA x prefetches into L2 the group of CTA
    // x + ahead (half the CTAs resident at once; 0 = no prefetch)
    uint32_t ahead;
};

cudaError_t launch_quant(const QuantParams &p, cudaStream_t st, LaunchLog &log);
// The smooth_k mean pass alone: mu_out[b, h, :] over x's tokens.
cudaError_t launch_token_mean(const QuantParams &p, cudaStream_t st, LaunchLog &log);

struct CombineParams {
    const float *o_part;      // [R, S, D]
    const float *lse_part;    // [R, S]
    int R, S, D;
    void *out;
    int out_bf16;
    float *lse_out;
    // launched right behind the decode kernel that writes the partials: the
    // combine may start while that grid runs (programmatic dependent launch)
    // and waits on the device for its completion before reading them
    int after_decode;
};

cudaError_t launch_combine(const CombineParams &p, cudaStream_t st, LaunchLog &log);

struct DecodeParams {
    const int8_t *q;
    const float *q_scale;
    const void *q_fp;         // optional [B, Hq, D] f16/bf16 query quantised in the kernel
    int q_fp_bf16;
    const int8_t *k_cache, *v_cache;
    const float *k_scale, *v_scale;
    const int32_t *block_table, *context_lens;
    int B, Hq, Hkv, D, group, head_tiles;
    int num_blocks, max_blocks;
    int num_segments, pages_per_seg;
    int max_pages;            // ceil(max_ctx / 16): segment s covers pages
                              // [s * max_pages / S, (s + 1) * max_pages / S)
    int max_ctx;              // host bound on context_lens (<= 16 * max_blocks)
    float qk_scale_log2;      // sm_scale * log2(e)
    float *o_part;            // [B*Hq, S, D] when num_segments > 1
    float *lse_part;          // [B*Hq, S]
    void *out;                // [B*Hq, D] when num_segments == 1
    int out_bf16;
    float *lse;               // optional [B*Hq] when num_segments == 1
    int32_t *dbg;             // optional raw score dump [B*Hq, dbg_stride]
    int dbg_stride;
    int force_partials;       // write o_part/lse_part even with one segment
    int cluster;              // 1: the segments of a (sequence, kv head, head tile) form one
                              // thread-block cluster and merge through distributed shared memory
    int after_quant;          // 1: launched right behind the kernel that writes q / q_scale
                              // (programmatic dependent launch; consumers wait on the device)
    int pv_mode;              // SAGE_PV_* (P.V operands and accumulation)
    int *err;
};

constexpr int kDecodeMaxCluster = 8;   // segments merged in-cluster (portable cluster size;
                                       // larger, non-portable clusters measured slower)

int decode_ctas_per_sm(int D);
int decode_max_segment_pages();   // longest segment (in 16-token pages) one CTA takes
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t st, LaunchLog &log);

struct KvAppendParams {
    const void *k, *v;        // [B, H, n, D] f16/bf16 new rows
    int bf16;
    int B, H, n, D;
    const int32_t *block_table, *pos;  // [B, max_blocks], [B]
    int max_blocks, num_blocks;
    int8_t *k_cache, *v_cache;         // [num_blocks, H, D/16, 16, 16]
    float *k_scale, *v_scale;          // [num_blocks, H, 16]
    // optional query rows quantised in the same launch (the KV producer
    // form): q [B, Hq, n, D] f16/bf16 -> q_int8 [B, Hq, n, D], q_scale [B, Hq, n]
    const void *q;
    int Hq;
    int8_t *q_int8;
    float *q_scale;
    FastDiv div_n, div_h;     // set by the launcher
    int *err;
};

cudaError_t launch_kv_append(const KvAppendParams &p, cudaStream_t st, LaunchLog &log);

struct PrefillParams {
    int B, Hq, Hkv, Sq, Sk, D, group;
    const int8_t *q;
    const float *q_scale;
    int q_shift;              // log2(q_block): 0 per token, 7 per 128-token block
    int q_groups;             // ceil(Sq / q_block)
    const int8_t *k;
    const float *k_scale;
    int k_shift;
    int k_groups;
    const void *v;
    int v_bf16;
    const float *q_bias;
    const int8_t *k_cache, *v_cache;
    const float *k_cache_scale, *v_cache_scale;
    const int32_t *block_table, *prefix_lens;
    int num_blocks, max_blocks, max_prefix_len;
    int causal;
    float qk_scale_log2;      // sm_scale * log2(e)
    void *out;
    int out_bf16;
    float *lse;
    int32_t *dbg;             // optional [B,Hq,Sq,dbg_stride]
    int dbg_stride;           // max_prefix_len + Sk
    int *err;
    // ---- workspace (exact f16 expansion of the keys/values a call reads)
    int BN;                   // key tile of the kernel (128, or 64 at D = 256)
    int Ppad;                 // prefix rows per (b, kv head), a multiple of BN
    int Lpad;                 // Ppad + Sk rounded up to BN
    int Vrows;                // rows of v_ws: Lpad for bf16 V, else Ppad (f16 chunk V read in place)
    __half *k_ws;             // [B*Hkv][Lpad][D] exact f16 key codes
    __half *v_ws;             // [B*Hkv][Vrows][D] f16 prefix values (code * v_scale; + bf16 chunk V)
    float *ksc_ws;            // [B*Hkv][Lpad] per-key K scale (0 on padding rows)
    // ---- packed variable-length batch (cu_q == null: the dense form).
    // Sq / Sk are then the bounds max_seqlen_q / max_seqlen_k; q [Hq, total_q, D],
    // q_scale [Hq, q_groups], k [Hkv, total_k, D], k_scale [Hkv, k_groups],
    // v [total_k, Hkv, D] (strides v_st, v_sh), q_bias / lse [Hq, total_q],
    // out [total_q, Hq, D]; the workspace holds [Hkv][Lpad] rows with
    // sequence b's keys from varlen_key_row0(); no paged prefix.
    const int32_t *cu_q, *cu_k;
    int64_t total_q, total_k;
    int64_t v_st, v_sh;
    // dense form, [P3] tensor_layout NHD: v is [B, Sk, Hkv, D] (element
    // strides v_sb, v_sh, v_st per batch, head, token; HND otherwise) and out
    // is [B, Sq, Hq, D]
    int nhd;
    int64_t v_sb;
    // dense form: (batch, head) pairs per scheduling bundle (1 .. B * Hq)
    int bundle;
    // smooth_v: per (batch or sequence, kv head) V mean [B * Hkv][D], subtracted
    // from the staged values and added back to the output; null when off
    const float *v_mean;
    // dense form, D = 256: the last, partly filled wave's query tiles split by
    // key range (split_k parts each; 0 = no split).  CTAs [0, split_f) take
    // whole query tiles; CTA split_f + u * split_k + j takes part j of tile
    // split_f + u (u < split_tail) and writes its normalised O and base-2 LSE
    // to part_o [slot][128][D] / part_lse [slot][128] (slot = u * split_k + j),
    // which the merge kernel combines into out and lse.
    int split_f, split_k, split_tail;
    float *part_o, *part_lse;
    // D <= 128: CTA x prefetches into L2 the query tile of CTA x + q_ahead
    // (one wave of one-CTA-per-SM launches ahead; 0 = no prefetch)
    int q_ahead;
    // packed form, D <= 128, even GQA group: a CTA takes 128 query rows of
    // two heads sharing a KV head (query tile t = head 2u + t) instead of
    // 256 rows of one head; the grid has (total_q / 128 + B) * Hq / 2 CTAs
    int vl_pairs;
};

// How the dense prefill splits its last wave: `full` whole query tiles, then
// `tail` tiles split into `parts` key ranges each (parts == 0: no split).
struct PrefillSplit {
    int full, tail, parts;
};
// keys: a query tile's largest key count (prefix + chunk); sms: the device's SMs
PrefillSplit prefill_split(int B, int Hq, int Sq, int D, int keys, bool causal, int sms);

// Pairs per bundle of the dense prefill's CTA order: as many KV heads'
// staged keys and values (f16, rows each) as fit in a share of L2, times
// the GQA group, so that the heads of one KV head stay together.
int prefill_bundle(int B, int Hq, int group, int rows, int D);

struct PrefillLayout {
    int BN, Ppad, Lpad, Vrows;
    // off_vmean: smooth_v's mean [B*Hkv][D]; off_part_o / off_part_lse: the
    // split tail's partial results
    size_t off_k, off_v, off_ksc, off_vmean, off_part_o, off_part_lse, bytes;
};

PrefillLayout prefill_layout(int B, int Hkv, int Sk, int D, int max_prefix_len, bool v_bf16,
                             bool smooth_v, const PrefillSplit &split);
PrefillLayout prefill_layout_varlen(int B, int Hkv, int64_t total_k, int D, bool smooth_v);
cudaError_t launch_prefill_stage(const PrefillParams &p, cudaStream_t st, LaunchLog &log);
cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t st, LaunchLog &log);

cudaError_t launch_timeout_probe(int timeout_us, int *err, cudaStream_t st, LaunchLog &log);

// Host-layer services shared by entry points defined outside api.cu.
int report_error(int status, const char *fmt, ...);   // sets the thread's last message
int device_error_word(int **out);                      // this device's error word
void record_launch(const LaunchLog &log);              // updates sage_last_launch_info

// Argument checks every decode entry point makes before it launches
// anything: head_dim and output dtype supported, Hq a multiple of Hkv,
// max_context_len within the block table, pointers present and aligned
// (q 4 bytes, or 8 for the f16/bf16 query q_fp of the fused form; out 8;
// caches and scales 16), and the per-step inputs and outputs in device
// memory or mapped pinned host memory.  Returns 0 (SAGE_OK) or the status
// with the thread's last message set; with B == 0 only the shape checks run.
int check_decode_args(const sage_decode_args_t *args, const void *q_fp);

}  // namespace sage
