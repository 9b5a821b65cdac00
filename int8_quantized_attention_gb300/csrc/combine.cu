// Split-K LSE combine: merges the per-segment outputs of the paged decode
// (the split-K segments of "INT8 QK MMAC on gfx936 DCU", section 4) using
// the log-sum-exp each segment returns (the SageAttention MXMACA README
// returns the LSE "for concatenation"):
//   M = max_s lse_s,  L = M + ln sum_s exp(lse_s - M),
//   out = sum_s exp(lse_s - L) * o_s.
// One warp per output row; each lane owns D/32 contiguous channels.  The
// partials are read once (coalesced float4 loads); HBM/L2-bound.
#include "common.cuh"
#include "internal.h"

namespace sage {

namespace {

constexpr int kRowsPerCta = 4;

template <int D, typename TO>
__global__ void __launch_bounds__(32 * kRowsPerCta) combine_kernel(CombineParams p) {
    constexpr int V = D / 32;  // channels per lane: 2, 4 or 8
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (r >= p.R) return;  // whole warp leaves together
    const float *lp = p.lse_part + r * p.S;
    float M = -INFINITY;
    for (int s = lane; s < p.S; s += 32) M = fmaxf(M, lp[s]);
    M = warp_max(M);
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.0f;
    float L = -INFINITY;
    if (M != -INFINITY) {
        float sum = 0.0f;
        for (int s = lane; s < p.S; s += 32) {
            const float l = lp[s];
            if (l != -INFINITY) sum += expf(l - M);
        }
        sum = warp_sum(sum);
        L = M + logf(sum);
        const float *op = p.o_part + r * (int64_t)p.S * D + lane * V;
        // 32 segments at a time: lane k computes segment k's weight once, the
        // weights are broadcast by shuffle and the partial loads of the 32
        // segments are independent (no serial L2 round trip per segment)
        for (int s0 = 0; s0 < p.S; s0 += 32) {
            const int sl = s0 + lane;
            const float l = sl < p.S ? lp[sl] : -INFINITY;
            const float wl = l == -INFINITY ? 0.0f : expf(l - L);
            const int n = min(32, p.S - s0);
#pragma unroll 8
            for (int k = 0; k < n; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
#pragma unroll
                for (int i = 0; i < V; i += 2) {
                    const float2 o2 = *reinterpret_cast<const float2 *>(op + (int64_t)(s0 + k) * D + i);
                    acc[i] = fmaf(w, o2.x, acc[i]);
                    acc[i + 1] = fmaf(w, o2.y, acc[i + 1]);
                }
            }
        }
    }
    TO *out = reinterpret_cast<TO *>(p.out) + r * D + lane * V;
#pragma unroll
    for (int i = 0; i < V; ++i) out[i] = DT<TO>::from_f(acc[i]);
    if (p.lse_out && lane == 0) p.lse_out[r] = L;
}

template <int D>
cudaError_t launch_d(const CombineParams &p, cudaStream_t st, LaunchLog &log) {
    const unsigned grid = (unsigned)((p.R + kRowsPerCta - 1) / kRowsPerCta);
    if (grid == 0) return cudaSuccess;
    if (p.out_bf16)
        combine_kernel<D, __nv_bfloat16><<<grid, 32 * kRowsPerCta, 0, st>>>(p);
    else
        combine_kernel<D, __half><<<grid, 32 * kRowsPerCta, 0, st>>>(p);
    log.add("combine_kernel", dim3(grid), dim3(32 * kRowsPerCta), dim3(1, 1, 1), 0);
    return cudaGetLastError();
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
