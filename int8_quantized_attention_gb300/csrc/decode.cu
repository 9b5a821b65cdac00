// Split-K paged INT8 decode ("INT8 QK MMAC on gfx936 DCU", sections 1, 3-5).
//
// Work decomposition: one CTA per (segment, kv head x head tile, sequence).
// A segment is a contiguous run of 16-token pages of one sequence; the
// per-segment results are merged by the LSE combine (combine.cu).
//
// Data path, per page:
//   * a producer warp issues 1-D bulk async copies (cp.async.bulk) of the
//     page's contiguous K slab, V slab (D*16 bytes each: the cache layout
//     [block, kv_head, D/16, 16, 16] keeps one (block, kv head) contiguous)
//     and its two 64-byte scale rows into a ring of shared-memory stages,
//     completing on mbarriers (bounded waits everywhere);
//   * four consumer warps take pages round-robin.  QK^T runs as native
//     INT8 tensor-core MMA (m16n8k32, exact INT32) with the 16 keys of the
//     page in the M dimension and up to 8 query heads of the GQA group in
//     N (6 of 8 columns useful at 6:1, against 6 of 16 rows when heads fill
//     the M rows);
//   * each score is rescaled by q_scale[head] * k_scale[key] *
//     sm_scale * log2(e) in registers and enters a base-2 online softmax;
//   * P^T (times v_scale[key], rounded to f16) is transposed in registers
//     (movmatrix) into the B operand of an f16 MMA whose A operand is V^T,
//     converted exactly from int8 to f16 in a per-warp staging buffer;
//     FP32 accumulation.
// At the end the four warps merge (m, l, O) through shared memory and the
// CTA writes either the segment partial (O normalised, LSE) or, with one
// segment, the final output.  When the segments of a (sequence, kv head,
// head tile) are launched as one thread-block cluster (at most 8), the LSE
// combine ("INT8 QK MMAC on gfx936 DCU", section 4: split-K) happens here
// instead: each CTA leaves its normalised segment output and base-2 LSE in
// its shared memory, and after a cluster barrier every CTA reduces a slice
// of the outputs by reading all segments through distributed shared memory,
// so no partial touches HBM and no second kernel is launched.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace sage {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

constexpr int kMaxSegPages = 1024;  // block-table entries staged per CTA (segment length cap)

template <int D>
struct DecodeCfg {
    static constexpr int kSlab = D * 16;                 // bytes of one page slab
    static constexpr int kStageBytes = 2 * kSlab + 128;  // K, V, K scales, V scales
    static constexpr int kStages = D == 256 ? 8 : (D == 128 ? 12 : 16);
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kOffBar = kRingBytes;
    // after the loop the ring holds the warp merge and the cluster combine
    static_assert(kRingBytes >= (2 * kConsumerWarps * 8 + kConsumerWarps * 8 * D + 8 * D + 8) * 4,
                  "merge area fits in the ring");
    static constexpr int kOffBt = kOffBar + kStages * 16 + 64;
    static constexpr int kSmem = kOffBt + kMaxSegPages * 4;
    static constexpr int kCtasPerSm = 227 * 1024 / (kSmem + 1024);
    // Page i goes to stage i % kStages and to consumer warp i % kConsumerWarps.
    // Every stage must always be read by the same warp: mbarrier parity waits
    // cannot tell phase k from phase k-2, so a stage shared by two warps
    // would let one of them pass a full-barrier wait a phase early.
    static_assert(kStages % kConsumerWarps == 0, "each stage belongs to one consumer warp");
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(DecodeParams p) {
    using Cfg = DecodeCfg<D>;
    constexpr int NST = Cfg::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint64_t *empty = full + NST;
    int *stage_ok = reinterpret_cast<int *>(empty + NST);
    int *bt_s = reinterpret_cast<int *>(smem + Cfg::kOffBt);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x;
    const int kvh = blockIdx.y / p.head_tiles;
    const int ht = blockIdx.y % p.head_tiles;
    const int b = blockIdx.z;
    const int head0 = kvh * p.group + ht * 8;
    const int nheads = min(8, p.group - ht * 8);
    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_ctx) {  // never read past the table row
        if (threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
        ctx = ctx < 0 ? 0 : p.max_ctx;
    }
    const int npages = (ctx + 15) >> 4;
    const int pg0 = seg * p.pages_per_seg;
    int np = max(0, min(pg0 + p.pages_per_seg, npages) - pg0);
    if (np > kMaxSegPages) {  // the host never asks for longer segments
        if (threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
        np = kMaxSegPages;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        fence_barrier_init();
    }
    {
        const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks + pg0;
        for (int i = threadIdx.x; i < np; i += kThreads) bt_s[i] = bt[i];
    }
    __syncthreads();

    // online-softmax state of a consumer thread: columns (heads) 2*q4, 2*q4+1
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.0f, 0.0f};
    float o[D / 16][4];  // O^T fragments: rows = channels, cols = heads
#pragma unroll
    for (int t = 0; t < D / 16; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.0f;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int i = 0; i < np; ++i) {
                const int s = i % NST;
                const uint32_t ph = (uint32_t)(i / NST) & 1u;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.err)) break;
                const int blk = bt_s[i];
                const uint32_t fb = smem_u32(&full[s]);
                if ((unsigned)blk >= (unsigned)p.num_blocks) {
                    atomicOr(p.err, kErrBadBlock);
                    stage_ok[s] = 0;
                    mbar_arrive(fb);
                    ++issued;
                    continue;
                }
                stage_ok[s] = 1;
                const int64_t pg = (int64_t)blk * p.Hkv + kvh;
                const uint32_t dst = smem_u32(ring + s * Cfg::kStageBytes);
                mbar_arrive_expect_tx(fb, 2 * Cfg::kSlab + 128);
                bulk_g2s_evict_first(dst, p.k_cache + pg * Cfg::kSlab, Cfg::kSlab, fb, pol);
                bulk_g2s_evict_first(dst + Cfg::kSlab, p.v_cache + pg * Cfg::kSlab, Cfg::kSlab, fb,
                                     pol);
                bulk_g2s(dst + 2 * Cfg::kSlab, p.k_scale + pg * 16, 64, fb);
                bulk_g2s(dst + 2 * Cfg::kSlab + 64, p.v_scale + pg * 16, 64, fb);
                ++issued;
            }
            // Do not retire while copies may still be landing: wait (bounded)
            // for the last phase armed on each stage.
            for (int i = max(0, issued - NST); i < issued; ++i)
                mbar_wait(smem_u32(&full[i % NST]), (uint32_t)(i / NST) & 1u, p.err);
        }
    } else {
        // ------------------------------------------------------ consumers
        const int g = lane >> 2, q4 = lane & 3;
        // B operand (Q^T): column n = head g of this tile, 4 bytes per k-quad.
        uint32_t qf[D / 32][2];
        {
            const bool hv = g < nheads;
            const int8_t *qrow = p.q + ((int64_t)b * p.Hq + head0 + (hv ? g : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < D / 32; ++ks) {
                qf[ks][0] = hv ? *reinterpret_cast<const uint32_t *>(qrow + ks * 32 + 4 * q4) : 0u;
                qf[ks][1] =
                    hv ? *reinterpret_cast<const uint32_t *>(qrow + ks * 32 + 16 + 4 * q4) : 0u;
            }
        }
        // Column heads of the accumulator fragments: 2*q4 and 2*q4+1.
        float colscale[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int hc = 2 * q4 + j;
            colscale[j] = hc < nheads ? p.q_scale[(int64_t)b * p.Hq + head0 + hc] * p.qk_scale_log2
                                      : 0.0f;
        }
        // ldmatrix row address of this lane for the transposed V loads:
        // matrix (lane / 8) = (16-channel block 2*dp + lane/16, keys 0-7 or 8-15)
        const uint32_t v_off = (lane >> 4) * 256 + ((lane >> 3) & 1) * 128 + (lane & 7) * 16;
        for (int i = warp; i < np; i += kConsumerWarps) {
            const int s = i % NST;
            const bool got = mbar_wait(smem_u32(&full[s]), (uint32_t)(i / NST) & 1u, p.err);
            if (!__all_sync(0xffffffffu, got)) break;  // keep the warp converged
            const uint8_t *stg = ring + s * Cfg::kStageBytes;
            const bool ok = stage_ok[s] != 0;
            const uint32_t stg_a = smem_u32(stg);
            // ---- QK^T: rows = 16 keys of the page, cols = 8 heads; two
            // independent accumulation chains (integer sums, exact)
            int c[4] = {0, 0, 0, 0}, c2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int ks = 0; ks < D / 32; ks += 2) {
                uint32_t a[4];
                ldsm_x4(stg_a + ks * 512 + lane * 16, a);
                mma_s8(c, a, qf[ks][0], qf[ks][1]);
                if (ks + 1 < D / 32) {
                    ldsm_x4(stg_a + (ks + 1) * 512 + lane * 16, a);
                    mma_s8(c2, a, qf[ks + 1][0], qf[ks + 1][1]);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] += c2[e];
            const float *ksc = reinterpret_cast<const float *>(stg + 2 * Cfg::kSlab);
            const float *vsc = ksc + 16;
            const float sk0 = ksc[g], sk1 = ksc[g + 8];
            const float sv0 = vsc[g], sv1 = vsc[g + 8];
            // ---- scores, mask, online softmax (base 2)
            const int tok0 = (pg0 + i) * 16;
            const bool v0 = ok && (tok0 + g) < ctx, v1 = ok && (tok0 + g + 8) < ctx;
            if (p.dbg) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hc = 2 * q4 + j;
                    if (hc < nheads) {
                        int32_t *dr = p.dbg + ((int64_t)b * p.Hq + head0 + hc) * p.dbg_stride;
                        if (v0) dr[tok0 + g] = c[j];
                        if (v1) dr[tok0 + g + 8] = c[2 + j];
                    }
                }
            }
            float t[2][2];  // [key row r][col j]
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                t[0][j] = v0 ? (float)c[j] * sk0 * colscale[j] : -INFINITY;
                t[1][j] = v1 ? (float)c[2 + j] * sk1 * colscale[j] : -INFINITY;
            }
            // Lazy rescaling: the running max m moves only when a page's max
            // exceeds it by more than 2^8, so most pages leave O untouched
            // (P then stays below 2^8; f16 P and fp32 O/l hold that easily).
            float alpha[2], pr[2][2];
            bool need = false;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(t[0][j], t[1][j]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                alpha[j] = 1.0f;
                if (mx != -INFINITY && (m[j] == -INFINITY || mx > m[j] + 8.0f)) {
                    alpha[j] = m[j] == -INFINITY ? 0.0f : fast_exp2(m[j] - mx);
                    m[j] = mx;
                    need = true;
                }
                const float ms = m[j] == -INFINITY ? 0.0f : m[j];  // all masked so far
                pr[0][j] = fast_exp2(t[0][j] - ms);
                pr[1][j] = fast_exp2(t[1][j] - ms);
                l[j] = l[j] * alpha[j] + pr[0][j] + pr[1][j];
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int dt = 0; dt < D / 16; ++dt) {
                    o[dt][0] *= alpha[0];
                    o[dt][1] *= alpha[1];
                    o[dt][2] *= alpha[0];
                    o[dt][3] *= alpha[1];
                }
            }
            // ---- P^T (x v_scale) -> B operand via in-register transpose
            const uint32_t pb0 = movmatrix_trans(pack_f16x2(pr[0][0] * sv0, pr[0][1] * sv0));
            const uint32_t pb1 = movmatrix_trans(pack_f16x2(pr[1][0] * sv1, pr[1][1] * sv1));
            // ---- O^T += V^T P^T.  A = V^T straight from the INT8 slab: a
            // transposed ldmatrix gives each lane keys (2q4, 2q4+1) of the
            // channel pair (2g, 2g+1); the even channel fills A row g, the odd
            // one row g + 8, so accumulator rows g / g+8 hold channels 2g / 2g+1
            // of the 16-channel block.  Exact int8 -> f16 in registers.
            const uint32_t vstg = stg_a + Cfg::kSlab + v_off;
#pragma unroll
            for (int dp = 0; dp < D / 32; ++dp) {
                uint32_t r[4], a[4];
                ldsm_x4_trans(vstg + dp * 512, r);
                i8x4_to_f16x2_even_odd(r[0], a[0], a[1]);
                i8x4_to_f16x2_even_odd(r[1], a[2], a[3]);
                mma_f16(o[2 * dp], a, pb0, pb1);
                i8x4_to_f16x2_even_odd(r[2], a[0], a[1]);
                i8x4_to_f16x2_even_odd(r[3], a[2], a[3]);
                mma_f16(o[2 * dp + 1], a, pb0, pb1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // stage fully read
        }
        // ---- per-warp totals of l over the 8 key rows sharing a column
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l[j] += __shfl_xor_sync(0xffffffffu, l[j], 4);
            l[j] += __shfl_xor_sync(0xffffffffu, l[j], 8);
            l[j] += __shfl_xor_sync(0xffffffffu, l[j], 16);
        }
    }
    __syncthreads();  // ring and staging are free from here on

    // ------------------------------------------------------- warp merge
    // merge area (the ring is free now): mm/ml [w][head], mo [w][head][D]
    float *mm = reinterpret_cast<float *>(ring);
    float *ml = mm + kConsumerWarps * 8;
    float *mo = ml + kConsumerWarps * 8;
    if (warp < kConsumerWarps) {
        const int g = lane >> 2, q4 = lane & 3;
        if (lane < 4) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mm[warp * 8 + 2 * q4 + j] = m[j];
                ml[warp * 8 + 2 * q4 + j] = l[j];
            }
        }
        // accumulator rows g / g + 8 of block dt are channels 2g / 2g + 1
        float *mw = mo + warp * 8 * D;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
            mw[(2 * q4) * D + dt * 16 + 2 * g] = o[dt][0];
            mw[(2 * q4 + 1) * D + dt * 16 + 2 * g] = o[dt][1];
            mw[(2 * q4) * D + dt * 16 + 2 * g + 1] = o[dt][2];
            mw[(2 * q4 + 1) * D + dt * 16 + 2 * g + 1] = o[dt][3];
        }
    }
    __syncthreads();
    if (p.cluster) {
        // ------------------------------------------- in-cluster LSE combine
        // this CTA's segment result: co[head][D] normalised, cl[head] base-2 LSE
        float *co = mo + kConsumerWarps * 8 * D;
        float *cl = co + 8 * D;
        for (int idx = threadIdx.x; idx < nheads * D; idx += kThreads) {
            const int j = idx / D, d = idx - j * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + j]);
            float val = 0.0f;
            if (M != -INFINITY) {
                float L = 0.0f, acc = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float f = exp2f(mm[w * 8 + j] - M);
                    L = fmaf(f, ml[w * 8 + j], L);
                    acc = fmaf(f, mo[(w * 8 + j) * D + d], acc);
                }
                val = acc / L;
            }
            co[j * D + d] = val;
        }
        if (threadIdx.x < nheads) {
            const int j = threadIdx.x;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + j]);
            float lse2 = -INFINITY;
            if (M != -INFINITY) {
                float L = 0.0f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    L = fmaf(exp2f(mm[w * 8 + j] - M), ml[w * 8 + j], L);
                lse2 = M + log2f(L);
            }
            cl[j] = lse2;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int S = p.num_segments;
        for (int idx = seg * kThreads + threadIdx.x; idx < nheads * D; idx += S * kThreads) {
            const int j = idx / D, d = idx - j * D;
            float ls[kDecodeMaxCluster];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kDecodeMaxCluster; ++r) {
                ls[r] = r < S ? cluster.map_shared_rank(cl, r)[j] : -INFINITY;
                M = fmaxf(M, ls[r]);
            }
            float val = 0.0f, L = 0.0f;
            if (M != -INFINITY) {
                float acc = 0.0f;
#pragma unroll
                for (int r = 0; r < kDecodeMaxCluster; ++r) {
                    if (r < S && ls[r] != -INFINITY) {
                        const float w = exp2f(ls[r] - M);
                        L += w;
                        acc = fmaf(w, cluster.map_shared_rank(co, r)[j * D + d], acc);
                    }
                }
                val = acc / L;
            }
            const int64_t row = (int64_t)b * p.Hq + head0 + j;
            if (p.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(val);
            else
                reinterpret_cast<__half *>(p.out)[row * D + d] = __float2half_rn(val);
            if (d == 0 && p.lse)
                p.lse[row] = M == -INFINITY ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
        }
        cluster.sync();  // every CTA's shared memory stays alive until all have read it
        return;
    }
    const bool direct = p.num_segments == 1 && !p.force_partials;
    for (int idx = threadIdx.x; idx < nheads * D; idx += kThreads) {
        const int j = idx / D, d = idx - j * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + j]);
        float val = 0.0f;
        if (M != -INFINITY) {
            float L = 0.0f, acc = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = exp2f(mm[w * 8 + j] - M);
                L = fmaf(f, ml[w * 8 + j], L);
                acc = fmaf(f, mo[(w * 8 + j) * D + d], acc);
            }
            val = acc / L;
        }
        const int64_t row = (int64_t)b * p.Hq + head0 + j;
        if (direct) {
            if (p.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(val);
            else
                reinterpret_cast<__half *>(p.out)[row * D + d] = __float2half_rn(val);
        } else {
            p.o_part[(row * p.num_segments + seg) * D + d] = val;
        }
    }
    if (threadIdx.x < nheads) {
        const int j = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + j]);
        float lse = -INFINITY;
        if (M != -INFINITY) {
            float L = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) L = fmaf(exp2f(mm[w * 8 + j] - M), ml[w * 8 + j], L);
            lse = (M + log2f(L)) * 0.69314718055994530942f;
        }
        const int64_t row = (int64_t)b * p.Hq + head0 + j;
        if (direct) {
            if (p.lse) p.lse[row] = lse;
        } else {
            p.lse_part[row * p.num_segments + seg] = lse;
        }
    }
}

template <int D>
cudaError_t launch_d(const DecodeParams &p, cudaStream_t st, LaunchLog &log) {
    using Cfg = DecodeCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid(p.num_segments, p.Hkv * p.head_tiles, p.B);
    if (p.cluster) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Cfg::kSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = p.num_segments;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_kernel<D>, p);
        if (e != cudaSuccess) return e;
        log.add("decode_kernel", grid, dim3(kThreads), dim3(p.num_segments, 1, 1), Cfg::kSmem);
    } else {
        decode_kernel<D><<<grid, kThreads, Cfg::kSmem, st>>>(p);
        log.add("decode_kernel", grid, dim3(kThreads), dim3(1, 1, 1), Cfg::kSmem);
    }
    log.segments = p.num_segments;
    return cudaGetLastError();
}

}  // namespace

int decode_max_segment_pages() { return kMaxSegPages; }

int decode_ctas_per_sm(int D) {
    int n = 0;
    cudaError_t e = cudaSuccess;
    switch (D) {
        case 64:
            e = cudaFuncSetAttribute(decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<64>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<64>, kThreads,
                                                                  DecodeCfg<64>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<64>::kCtasPerSm;
            break;
        case 128:
            e = cudaFuncSetAttribute(decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<128>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<128>, kThreads,
                                                                  DecodeCfg<128>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<128>::kCtasPerSm;
            break;
        default:
            e = cudaFuncSetAttribute(decode_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<256>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<256>, kThreads,
                                                                  DecodeCfg<256>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<256>::kCtasPerSm;
            break;
    }
    return n;
}

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.D) {
        case 64: return launch_d<64>(p, st, log);
        case 128: return launch_d<128>(p, st, log);
        case 256: return launch_d<256>(p, st, log);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sage
