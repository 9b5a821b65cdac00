// Split-K LSE combine: merges the per-segment outputs of the paged decode
// (the split-K segments of "INT8 QK MMAC on gfx936 DCU", section 4) using
// the log-sum-exp each segment returns (the SageAttention MXMACA README
// returns the LSE "for concatenation"):
//   M = max_s lse_s,  L = M + ln sum_s exp(lse_s - M),
//   out = sum_s exp(lse_s - L) * o_s.
// One CTA per output row; its W warps (one per segment, at most 8) take
// every W-th segment.  Each warp first issues the loads of its segments'
// partial outputs and LSEs (up to kSegChunk per round, all independent),
// then scans the row's S LSEs itself for M and L (no barrier), weights and
// adds its segments, and the W partial rows add up in shared memory, each
// thread summing and storing its own channels: one memory round trip and
// one barrier per row.  With few rows (batch-1 decode
// has a handful of (sequence, head) rows and up to 64 segments) the
// segments, not the rows, carry the parallelism.  HBM/L2-bound.
#include "common.cuh"
#include "internal.h"

namespace sage {

namespace {

constexpr int kMaxCombineWarps = 8;
constexpr int kSegChunk = 8;  // segments a warp holds in registers per round

template <int D, typename TO>
__global__ void __launch_bounds__(32 * kMaxCombineWarps) combine_kernel(CombineParams p) {
    constexpr int V = D / 32;  // channels per lane: 2, 4 or 8
    __shared__ float part[kMaxCombineWarps][D];
    const int W = (int)blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = blockIdx.x;
    const float *lp = p.lse_part + r * p.S;
    const float *op = p.o_part + r * (int64_t)p.S * D + lane * V;
    // launched behind the decode kernel: wait here (not at the launch) until
    // that grid has completed and its partials are visible; a no-op otherwise
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    float L = -INFINITY;
    for (int s0 = warp; s0 < p.S; s0 += W * kSegChunk) {
        // this round's segments: loads first, all independent of M and L
        float lv[kSegChunk], ov[kSegChunk][V];
#pragma unroll
        for (int k = 0; k < kSegChunk; ++k) {
            const int s = s0 + k * W;
            lv[k] = s < p.S ? lp[s] : -INFINITY;
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                float2 o2 = make_float2(0.0f, 0.0f);
                if (s < p.S) o2 = *reinterpret_cast<const float2 *>(op + (int64_t)s * D + i);
                ov[k][i] = o2.x;
                ov[k][i + 1] = o2.y;
            }
        }
        if (s0 == warp) {
            // the row's M and L, scanned by every warp (no barrier)
            float M = -INFINITY;
            for (int s = lane; s < p.S; s += 32) M = fmaxf(M, lp[s]);
            M = warp_max(M);
            if (M != -INFINITY) {
                float sum = 0.0f;
                for (int s = lane; s < p.S; s += 32) {
                    const float l = lp[s];
                    if (l != -INFINITY) sum += expf(l - M);
                }
                sum = warp_sum(sum);
                L = M + logf(sum);
            }
        }
        if (L == -INFINITY) break;  // no segment saw a key: the row stays 0
#pragma unroll
        for (int k = 0; k < kSegChunk; ++k) {
            const float w = lv[k] == -INFINITY ? 0.0f : expf(lv[k] - L);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = fmaf(w, ov[k][i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < V; ++i) part[warp][lane * V + i] = acc[i];
    __syncthreads();
    // every thread adds the W warp rows of its channels and stores them
    TO *out = reinterpret_cast<TO *>(p.out) + r * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float v = part[0][c];
        for (int k = 1; k < W; ++k) v += part[k][c];
        out[c] = DT<TO>::from_f(v);
    }
    // every warp, warp 0 included, found L in its first round (W <= S)
    if (p.lse_out && threadIdx.x == 0) p.lse_out[r] = L;
}

template <int D>
cudaError_t launch_d(const CombineParams &p, cudaStream_t st, LaunchLog &log) {
    const unsigned grid = (unsigned)p.R;
    if (grid == 0) return cudaSuccess;
    int W = p.S;  // one warp per segment, at most kMaxCombineWarps
    W = W < 1 ? 1 : (W > kMaxCombineWarps ? kMaxCombineWarps : W);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(32 * W, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.after_decode ? 1 : 0;
    const cudaError_t e = p.out_bf16 ? cudaLaunchKernelEx(&cfg, combine_kernel<D, __nv_bfloat16>, p)
                                     : cudaLaunchKernelEx(&cfg, combine_kernel<D, __half>, p);
    log.add("combine_kernel", cfg.gridDim, cfg.blockDim, dim3(1, 1, 1), 0);
    return e;
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.D) {
        case 64: return launch_d<64>(p, st, log);
        case 128: return launch_d<128>(p, st, log);
        case 256: return launch_d<256>(p, st, log);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sage
