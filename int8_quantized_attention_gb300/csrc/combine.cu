// Split-K LSE combine: merges the per-segment outputs of the paged decode
// (the split-K segments of "INT8 QK MMAC on gfx936 DCU", section 4) using
// the log-sum-exp each segment returns (the SageAttention MXMACA README
// returns the LSE "for concatenation"):
//   M = max_s lse_s,  L = M + ln sum_s exp(lse_s - M),
//   out = sum_s exp(lse_s - L) * o_s.
// One CTA per output row; its W warps (up to 8, about one per 8 segments)
// each take every W-th segment and accumulate all D channels (D/32 per
// lane, coalesced float4 loads, independent across segments), then the W
// partial rows add up in shared memory.  With few rows (batch-1 decode has
// a handful of (sequence, head) rows and up to 64 segments) the segments,
// not the rows, carry the parallelism.  HBM/L2-bound.
#include "common.cuh"
#include "internal.h"

namespace sage {

namespace {

constexpr int kMaxCombineWarps = 8;

template <int D, typename TO>
__global__ void __launch_bounds__(32 * kMaxCombineWarps) combine_kernel(CombineParams p) {
    constexpr int V = D / 32;  // channels per lane: 2, 4 or 8
    __shared__ float part[kMaxCombineWarps][D];
    __shared__ float sh_L;
    const int W = (int)blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = blockIdx.x;
    const float *lp = p.lse_part + r * p.S;
    // launched behind the decode kernel: wait here (not at the launch) until
    // that grid has completed and its partials are visible; a no-op otherwise
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == 0) {
        float M = -INFINITY;
        for (int s = lane; s < p.S; s += 32) M = fmaxf(M, lp[s]);
        M = warp_max(M);
        float L = -INFINITY;
        if (M != -INFINITY) {
            float sum = 0.0f;
            for (int s = lane; s < p.S; s += 32) {
                const float l = lp[s];
                if (l != -INFINITY) sum += expf(l - M);
            }
            sum = warp_sum(sum);
            L = M + logf(sum);
        }
        if (lane == 0) sh_L = L;
    }
    __syncthreads();
    const float L = sh_L;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    if (L != -INFINITY) {
        const float *op = p.o_part + r * (int64_t)p.S * D + lane * V;
#pragma unroll 4
        for (int s = warp; s < p.S; s += W) {
            const float l = lp[s];
            const float w = l == -INFINITY ? 0.0f : expf(l - L);
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const float2 o2 = *reinterpret_cast<const float2 *>(op + (int64_t)s * D + i);
                acc[i] = fmaf(w, o2.x, acc[i]);
                acc[i + 1] = fmaf(w, o2.y, acc[i + 1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < V; ++i) part[warp][lane * V + i] = acc[i];
    __syncthreads();
    if (warp == 0) {
        TO *out = reinterpret_cast<TO *>(p.out) + r * D + lane * V;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float v = part[0][lane * V + i];
            for (int k = 1; k < W; ++k) v += part[k][lane * V + i];
            out[i] = DT<TO>::from_f(v);
        }
        if (p.lse_out && lane == 0) p.lse_out[r] = L;
    }
}

template <int D>
cudaError_t launch_d(const CombineParams &p, cudaStream_t st, LaunchLog &log) {
    const unsigned grid = (unsigned)p.R;
    if (grid == 0) return cudaSuccess;
    int W = (p.S + 7) / 8;
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
