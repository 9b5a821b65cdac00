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
constexpr int kPvF32 = 0, kPvF16 = 1, kPvF16F32 = 2, kPvInt8 = 3;  // sage_decode_args_t::pv_mode
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
    static_assert(kRingBytes >= (3 * kConsumerWarps * 8 + kConsumerWarps * 8 * (D + 4) + 8 + 8 * D +
                                 kDecodeMaxCluster * 8 + 8) * 4,
                  "merge area fits in the ring");
    static constexpr int kOffBt = kOffBar + kStages * 16 + 64;
    static constexpr int kOffQ = kOffBt + kMaxSegPages * 4;     // int8 query codes [8][D]
    static constexpr int kOffQs = kOffQ + 8 * D;               // their scales [8]
    static constexpr int kSmem = kOffQs + 8 * 4;
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

// Same MMA with f16 accumulators: d/c = {row g, row g + 8} x columns
// (2 q4, 2 q4 + 1), each an f16x2 word.
__device__ __forceinline__ void mma_f16_f16acc(uint32_t (&c)[2], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f16.f16.f16.f16 {%0,%1}, {%2,%3,%4,%5}, {%6,%7}, "
        "{%0,%1};"
        : "+r"(c[0]), "+r"(c[1])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
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

// P.V variants (SageAttention MXMACA README, advanced configuration:
// pv_accum_dtype; "INT8 QK MMAC on gfx936 DCU", sections 6 and 8: INT8 P.V
// with the V scale fused into P).
//   kPvF32     f16 P x V, fp32 accumulators (the default)
//   kPvF16     f16 P x V, f16 accumulators throughout
//   kPvF16F32  each page's product in f16 accumulators, added to fp32 ones
//              (the README's two-level "InstBuf" accumulation)
//   kPvInt8    P' = p * v_scale quantised to INT8 per head over the page's 16
//              keys (s = max P' / 127, codes rne(P' / s)); codes times INT8
//              values summed exactly, then scaled by s into fp32
template <int D, int PV>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(DecodeParams p) {
    using Cfg = DecodeCfg<D>;
    constexpr int NST = Cfg::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint64_t *empty = full + NST;
    int *stage_ok = reinterpret_cast<int *>(empty + NST);
    int *bt_s = reinterpret_cast<int *>(smem + Cfg::kOffBt);
    int8_t *q_s = reinterpret_cast<int8_t *>(smem + Cfg::kOffQ);
    float *qsc_s = reinterpret_cast<float *>(smem + Cfg::kOffQs);

    // a combine kernel launched behind this grid may be scheduled once every
    // CTA has started; it waits on the device for this grid to complete
    asm volatile("griddepcontrol.launch_dependents;");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x;
    const int kvh = blockIdx.y / p.head_tiles;
    const int ht = blockIdx.y % p.head_tiles;
    const int b = blockIdx.z;
    const int head0 = kvh * p.group + ht * 8;
    const int nheads = min(8, p.group - ht * 8);
    // The consumers of the fused-query form load their query channels first
    // thing: the loads land during the barrier set-up and the block-table
    // round trip.  Issued after those, a query in pinned host memory (read
    // over NVLink-C2C by every segment's CTA) delayed the first page by ~4 us.
    constexpr int kQPieces = D / 64;  // 8-byte pieces (4 channels) per lane
    uint2 qraw[kQPieces];
    {
        const int hh = 2 * warp + (lane >> 4);
        const bool ld = p.q_fp && warp < kConsumerWarps && hh < nheads;
        const uint16_t *src = ld ? static_cast<const uint16_t *>(p.q_fp) +
                                       ((int64_t)b * p.Hq + head0 + hh) * D + (lane & 15) * (D / 16)
                                 : nullptr;
#pragma unroll
        for (int k = 0; k < kQPieces; ++k)
            qraw[k] = ld ? *reinterpret_cast<const uint2 *>(src + 4 * k) : make_uint2(0u, 0u);
    }
    // Segment seg covers pages [seg * P / S, (seg + 1) * P / S) of the
    // longest context (P pages): the segments differ by one page at most.
    const int pg0 = (int)((int64_t)seg * p.max_pages / p.num_segments);
    const int pg1 = (int)((int64_t)(seg + 1) * p.max_pages / p.num_segments);
    // The segment's block-table entries are loaded together with the context
    // length (one DRAM round trip for both, not two in a row); pg1 <=
    // max_pages <= max_blocks keeps them inside the table row, and entries
    // past the context are never used.
    constexpr int kBtRegs = 2;
    const int32_t *bt = p.block_table + (int64_t)b * p.max_blocks + pg0;
    int btr[kBtRegs];
#pragma unroll
    for (int k = 0; k < kBtRegs; ++k) {
        const int i = threadIdx.x + k * kThreads;
        btr[k] = i < pg1 - pg0 ? bt[i] : 0;
    }
    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_ctx) {  // never read past the table row
        if (threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
        ctx = ctx < 0 ? 0 : p.max_ctx;
    }
    const int npages = (ctx + 15) >> 4;
    int np = max(0, min(pg1, npages) - pg0);
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
#pragma unroll
    for (int k = 0; k < kBtRegs; ++k) {
        const int i = threadIdx.x + k * kThreads;
        if (i < np) bt_s[i] = btr[k];
    }
    for (int i = threadIdx.x + kBtRegs * kThreads; i < np; i += kThreads) bt_s[i] = bt[i];
    __syncthreads();

    // online-softmax state of a consumer thread: columns (heads) 2*q4, 2*q4+1
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.0f, 0.0f};
    float o[D / 16][4];  // O^T fragments: rows = channels, cols = heads
#pragma unroll
    for (int t = 0; t < D / 16; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.0f;
    uint32_t oh[PV == kPvF16 ? D / 16 : 1][2];  // the same fragments in f16 (kPvF16)
#pragma unroll
    for (int t = 0; t < (PV == kPvF16 ? D / 16 : 1); ++t) oh[t][0] = oh[t][1] = 0u;
    // With f16 accumulators the running max moves with every larger page
    // max, so p <= 1 and the accumulated P'.V stays far inside the f16 range.
    constexpr float kLazy = PV == kPvF16 ? 0.0f : 8.0f;

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
        float colscale[2];
        const bool hv = g < nheads;
        if (p.q_fp) {
            // The query quantised here, per (token, head), with the same
            // arithmetic as the quant kernel (bit-identical codes and scale).
            // Warp w quantises heads 2w, 2w+1 (16 lanes per head, D/16
            // channels per lane) into shared memory; the consumer warps then
            // meet at a named barrier (the producer is already copying).
            {
                const int hh = 2 * warp + (lane >> 4);  // head of this half-warp
                const int cpl = D / 16;                 // channels per lane
                const int c0 = (lane & 15) * cpl;
                float f[cpl];
                if (hh < nheads) {
#pragma unroll
                    for (int e = 0; e < cpl; e += 4) {
                        const uint2 u = qraw[e / 4];  // loaded at kernel start
                        const uint32_t w2[2] = {u.x, u.y};
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            float2 t;
                            if (p.q_fp_bf16)
                                t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w2[k]));
                            else
                                t = __half22float2(*reinterpret_cast<const __half2 *>(&w2[k]));
                            f[e + 2 * k] = t.x;
                            f[e + 2 * k + 1] = t.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < cpl; ++e) f[e] = 0.0f;
                }
                float amax = 0.0f;
#pragma unroll
                for (int e = 0; e < cpl; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sq = __fdiv_rn(amax, 127.0f);
                const float rq = quant_recip(sq);
                if (hh < 8) {
#pragma unroll
                    for (int e = 0; e < cpl; e += 4) {
                        uint32_t w = 0;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w |= (uint32_t)(uint8_t)quant_code(f[e + k], sq, rq) << (8 * k);
                        *reinterpret_cast<uint32_t *>(q_s + hh * D + c0 + e) = w;
                    }
                    if ((lane & 15) == 0) qsc_s[hh] = sq;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
#pragma unroll
            for (int ks = 0; ks < D / 32; ++ks) {
                qf[ks][0] = hv ? *reinterpret_cast<const uint32_t *>(q_s + g * D + ks * 32 + 4 * q4) : 0u;
                qf[ks][1] =
                    hv ? *reinterpret_cast<const uint32_t *>(q_s + g * D + ks * 32 + 16 + 4 * q4) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                colscale[j] = 2 * q4 + j < nheads ? qsc_s[2 * q4 + j] * p.qk_scale_log2 : 0.0f;
        } else {
            // launched behind the kernel that quantises the query: wait here
            // (the producer is already copying pages) until its codes are
            // visible; a no-op otherwise
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const int8_t *qrow = p.q + ((int64_t)b * p.Hq + head0 + (hv ? g : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < D / 32; ++ks) {
                qf[ks][0] = hv ? *reinterpret_cast<const uint32_t *>(qrow + ks * 32 + 4 * q4) : 0u;
                qf[ks][1] =
                    hv ? *reinterpret_cast<const uint32_t *>(qrow + ks * 32 + 16 + 4 * q4) : 0u;
            }
            // Column heads of the accumulator fragments: 2*q4 and 2*q4+1.
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int hc = 2 * q4 + j;
                colscale[j] = hc < nheads
                                  ? p.q_scale[(int64_t)b * p.Hq + head0 + hc] * p.qk_scale_log2
                                  : 0.0f;
            }
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
            // ---- QK^T: rows = 16 keys of the page, cols = 8 heads; up to
            // four independent accumulation chains (integer sums, exact)
            constexpr int KS = D / 32, NC = KS < 4 ? KS : 4;
            int cc[NC][4];
#pragma unroll
            for (int h = 0; h < NC; ++h) cc[h][0] = cc[h][1] = cc[h][2] = cc[h][3] = 0;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(stg_a + ks * 512 + lane * 16, a);
                mma_s8(cc[ks % NC], a, qf[ks][0], qf[ks][1]);
            }
            int c[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                c[e] = cc[0][e];
#pragma unroll
                for (int h = 1; h < NC; ++h) c[e] += cc[h][e];
            }
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
                if (mx != -INFINITY && (m[j] == -INFINITY || mx > m[j] + kLazy)) {
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
                if constexpr (PV == kPvF16) {
                    const uint32_t al = pack_f16x2(alpha[0], alpha[1]);
#pragma unroll
                    for (int dt = 0; dt < D / 16; ++dt) {
                        __half2 *h = reinterpret_cast<__half2 *>(oh[dt]);
                        h[0] = __hmul2(h[0], *reinterpret_cast<const __half2 *>(&al));
                        h[1] = __hmul2(h[1], *reinterpret_cast<const __half2 *>(&al));
                    }
                } else {
#pragma unroll
                    for (int dt = 0; dt < D / 16; ++dt) {
                        o[dt][0] *= alpha[0];
                        o[dt][1] *= alpha[1];
                        o[dt][2] *= alpha[0];
                        o[dt][3] *= alpha[1];
                    }
                }
            }
            // ---- P^T (x v_scale) -> B operand via in-register transpose;
            // for INT8 P the operand holds the page's codes and sp the
            // per-head scale that multiplies the page's exact product
            float sp[2] = {1.0f, 1.0f};
            uint32_t pb0, pb1;
            if constexpr (PV == kPvInt8) {
                float w[2][2], cd[2][2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    w[0][j] = pr[0][j] * sv0;
                    w[1][j] = pr[1][j] * sv1;
                    float mx = fmaxf(w[0][j], w[1][j]);  // over the page's 16 keys
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    sp[j] = __fdiv_rn(mx, 127.0f);
                    const float rp = quant_recip(sp[j]);
                    cd[0][j] = (float)quant_code(w[0][j], sp[j], rp);
                    cd[1][j] = (float)quant_code(w[1][j], sp[j], rp);
                }
                pb0 = movmatrix_trans(pack_f16x2(cd[0][0], cd[0][1]));  // integers: exact in f16
                pb1 = movmatrix_trans(pack_f16x2(cd[1][0], cd[1][1]));
            } else {
                pb0 = movmatrix_trans(pack_f16x2(pr[0][0] * sv0, pr[0][1] * sv0));
                pb1 = movmatrix_trans(pack_f16x2(pr[1][0] * sv1, pr[1][1] * sv1));
            }
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
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int dt = 2 * dp + hf;
                    i8x4_to_f16x2_even_odd(r[2 * hf], a[0], a[1]);
                    i8x4_to_f16x2_even_odd(r[2 * hf + 1], a[2], a[3]);
                    if constexpr (PV == kPvF32) {
                        mma_f16(o[dt], a, pb0, pb1);
                    } else if constexpr (PV == kPvF16) {
                        mma_f16_f16acc(oh[dt], a, pb0, pb1);
                    } else if constexpr (PV == kPvF16F32) {
                        uint32_t h[2] = {0u, 0u};  // this page's product, f16
                        mma_f16_f16acc(h, a, pb0, pb1);
                        const float2 lo = unpack_f16x2(h[0]), hi = unpack_f16x2(h[1]);
                        o[dt][0] += lo.x;
                        o[dt][1] += lo.y;
                        o[dt][2] += hi.x;
                        o[dt][3] += hi.y;
                    } else {
                        // codes x values: products <= 127 * 128, sums over 16
                        // keys below 2^24 -- exact in the fp32 accumulator
                        float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        mma_f16(t, a, pb0, pb1);
                        o[dt][0] = fmaf(sp[0], t[0], o[dt][0]);
                        o[dt][1] = fmaf(sp[1], t[1], o[dt][1]);
                        o[dt][2] = fmaf(sp[0], t[2], o[dt][2]);
                        o[dt][3] = fmaf(sp[1], t[3], o[dt][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // stage fully read
        }
        if constexpr (PV == kPvF16) {
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                const float2 lo = unpack_f16x2(oh[dt][0]), hi = unpack_f16x2(oh[dt][1]);
                o[dt][0] = lo.x;
                o[dt][1] = lo.y;
                o[dt][2] = hi.x;
                o[dt][3] = hi.y;
            }
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
    // merge area (the ring is free now): mm/ml [w][head], mo [w][head][D (+4)]
    constexpr int kMoStride = D + 4;
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
        // accumulator rows g / g + 8 of block dt are channels 2g / 2g + 1:
        // (o0, o2) and (o1, o3) are channel pairs of heads 2q4 and 2q4 + 1.
        // Rows of kMoStride = D + 4 floats keep these 8-byte stores at the
        // minimum two wavefronts per warp.
        float *mw = mo + warp * 8 * kMoStride;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
            *reinterpret_cast<float2 *>(mw + (2 * q4) * kMoStride + dt * 16 + 2 * g) =
                make_float2(o[dt][0], o[dt][2]);
            *reinterpret_cast<float2 *>(mw + (2 * q4 + 1) * kMoStride + dt * 16 + 2 * g) =
                make_float2(o[dt][1], o[dt][3]);
        }
    }
    __syncthreads();
    // per-head merge weights, once: fw[w][j] = 2^(m_wj - M_j) / L_j and the
    // segment's base-2 LSE hl[j] = M_j + log2 L_j (-inf with no visible key)
    float *fw = mo + kConsumerWarps * 8 * kMoStride;
    float *hl = fw + kConsumerWarps * 8;
    if (threadIdx.x < nheads) {
        const int j = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + j]);
        if (M == -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) fw[w * 8 + j] = 0.0f;
            hl[j] = -INFINITY;
        } else {
            float f[kConsumerWarps], L = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                f[w] = fast_exp2(mm[w * 8 + j] - M);
                L = fmaf(f[w], ml[w * 8 + j], L);
            }
            const float inv = 1.0f / L;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) fw[w * 8 + j] = f[w] * inv;
            hl[j] = M + log2f(L);
        }
    }
    __syncthreads();
    // the segment's normalised output, 4 channels per thread
    auto seg_out = [&](int j, int d) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = fw[w * 8 + j];
            const float4 v = *reinterpret_cast<const float4 *>(mo + (w * 8 + j) * kMoStride + d);
            acc.x = fmaf(f, v.x, acc.x);
            acc.y = fmaf(f, v.y, acc.y);
            acc.z = fmaf(f, v.z, acc.z);
            acc.w = fmaf(f, v.w, acc.w);
        }
        return acc;
    };
    auto store_out = [&](int64_t row, int d, float4 v) {
        if (p.out_bf16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 u = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + row * D + d) = u;
        } else {
            __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
            uint2 u = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(p.out) + row * D + d) = u;
        }
    };
    constexpr float kLn2 = 0.69314718055994530942f;
    if (p.cluster) {
        // ------------------------------------------- in-cluster LSE combine
        // this CTA's segment result co[head][D]; its base-2 LSE is hl[head]
        float *co = hl + 8;
        float *cw = co + 8 * D;                  // [rank][head] combine weights
        float *gl = cw + kDecodeMaxCluster * 8;  // [head] combined base-2 LSE
        for (int idx = 4 * threadIdx.x; idx < nheads * D; idx += 4 * kThreads) {
            const int j = idx / D, d = idx - j * D;
            *reinterpret_cast<float4 *>(co + j * D + d) = seg_out(j, d);
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int S = p.num_segments;
        if (threadIdx.x < nheads) {
            const int j = threadIdx.x;
            float ls[kDecodeMaxCluster];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kDecodeMaxCluster; ++r) {
                ls[r] = r < S ? cluster.map_shared_rank(hl, r)[j] : -INFINITY;
                M = fmaxf(M, ls[r]);
            }
            float L = 0.0f;
            float f[kDecodeMaxCluster];
#pragma unroll
            for (int r = 0; r < kDecodeMaxCluster; ++r) {
                f[r] = (M != -INFINITY && ls[r] != -INFINITY) ? fast_exp2(ls[r] - M) : 0.0f;
                L += f[r];
            }
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
            for (int r = 0; r < kDecodeMaxCluster; ++r) cw[r * 8 + j] = f[r] * inv;
            gl[j] = M == -INFINITY ? -INFINITY : M + log2f(L);
        }
        __syncthreads();
        // this CTA reduces a slice of the outputs, 4 channels per thread
        for (int idx = 4 * (seg * kThreads + threadIdx.x); idx < nheads * D; idx += 4 * S * kThreads) {
            const int j = idx / D, d = idx - j * D;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int r = 0; r < kDecodeMaxCluster; ++r) {
                if (r < S) {
                    const float w = cw[r * 8 + j];
                    const float4 v = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(co, r) + j * D + d);
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
                }
            }
            const int64_t row = (int64_t)b * p.Hq + head0 + j;
            store_out(row, d, acc);
            if (d == 0 && p.lse) p.lse[row] = gl[j] * kLn2;
        }
        cluster.sync();  // every CTA's shared memory stays alive until all have read it
        return;
    }
    const bool direct = p.num_segments == 1 && !p.force_partials;
    for (int idx = 4 * threadIdx.x; idx < nheads * D; idx += 4 * kThreads) {
        const int j = idx / D, d = idx - j * D;
        const float4 v = seg_out(j, d);
        const int64_t row = (int64_t)b * p.Hq + head0 + j;
        if (direct)
            store_out(row, d, v);
        else
            *reinterpret_cast<float4 *>(p.o_part + (row * p.num_segments + seg) * D + d) = v;
    }
    if (threadIdx.x < nheads) {
        const int j = threadIdx.x;
        const float lse = hl[j] * kLn2;  // -inf * ln2 stays -inf
        const int64_t row = (int64_t)b * p.Hq + head0 + j;
        if (direct) {
            if (p.lse) p.lse[row] = lse;
        } else {
            p.lse_part[row * p.num_segments + seg] = lse;
        }
    }
}

template <int D, int PV>
cudaError_t launch_d(const DecodeParams &p, cudaStream_t st, LaunchLog &log) {
    using Cfg = DecodeCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D, PV>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid(p.num_segments, p.Hkv * p.head_tiles, p.B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.cluster) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.num_segments;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (p.after_quant) {
        // may start while the query's quantisation runs (programmatic
        // dependent launch); the consumers wait for it on the device
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, decode_kernel<D, PV>, p);
    if (e != cudaSuccess) return e;
    log.add("decode_kernel", grid, dim3(kThreads), dim3(p.cluster ? p.num_segments : 1, 1, 1),
            Cfg::kSmem);
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
            e = cudaFuncSetAttribute(decode_kernel<64, kPvF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<64>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<64, kPvF32>, kThreads,
                                                                  DecodeCfg<64>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<64>::kCtasPerSm;
            break;
        case 128:
            e = cudaFuncSetAttribute(decode_kernel<128, kPvF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<128>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<128, kPvF32>, kThreads,
                                                                  DecodeCfg<128>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<128>::kCtasPerSm;
            break;
        default:
            e = cudaFuncSetAttribute(decode_kernel<256, kPvF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DecodeCfg<256>::kSmem);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<256, kPvF32>, kThreads,
                                                                  DecodeCfg<256>::kSmem);
            if (e != cudaSuccess || n < 1) n = DecodeCfg<256>::kCtasPerSm;
            break;
    }
    return n;
}

template <int D>
cudaError_t launch_pv(const DecodeParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.pv_mode) {
        case kPvF32: return launch_d<D, kPvF32>(p, st, log);
        case kPvF16: return launch_d<D, kPvF16>(p, st, log);
        case kPvF16F32: return launch_d<D, kPvF16F32>(p, st, log);
        case kPvInt8: return launch_d<D, kPvInt8>(p, st, log);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.D) {
        case 64: return launch_pv<64>(p, st, log);
        case 128: return launch_pv<128>(p, st, log);
        case 256: return launch_pv<256>(p, st, log);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sage
