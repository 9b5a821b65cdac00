// Symmetric dynamic INT8 quantisation of Q / K and the smooth_k mean.
//
// Rule ("INT8 QK MMAC on gfx936 DCU", section 4): s = amax / 127 and
// q = round(x / s), with the division taken as one correctly rounded fp32
// division and round-to-nearest-even; groups are one token row or a block
// of consecutive tokens (SageAttention MXMACA README, quant kernel table:
// block size 128 for Q, 64 for K).  smooth_k (same README, feature matrix)
// subtracts the per-channel mean over tokens before quantising.
//
// Memory layout: x is read through (b, h, s) strides with the channel
// dimension contiguous, 16 bytes (8 elements) per thread per load; the
// int8 output is dense [B,H,S,D].  A packed variable-length batch (the
// README's varlen path: sequence b is packed tokens cu[b] .. cu[b+1]-1 of
// x [total, H, D]) is quantised sequence by sequence: groups start at each
// sequence's first token and smooth_k takes each sequence's own mean; the
// int8 output is [H, total, D] and the scales [H, groups] with sequence
// b's groups from varlen_group0().  These kernels are HBM-bound.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace sage {

namespace {

template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&v)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(p);
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = DT<T>::to_f(e[i]);
}

__device__ __forceinline__ int8_t quant1(float v, float s) { return quant_code(v, s); }

__device__ __forceinline__ void store8_i8(int8_t *dst, const float (&v)[8], float s) {
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) w0 |= (uint32_t)(uint8_t)quant1(v[i], s) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) w1 |= (uint32_t)(uint8_t)quant1(v[i + 4], s) << (8 * i);
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w0, w1);
}

// Reduce across the `tpr` consecutive lanes that share one row.
__device__ __forceinline__ float row_max(float v, int tpr) {
    for (int o = tpr >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float row_sum(float v, int tpr) {
    for (int o = tpr >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Per-token quantisation: each row of D elements is handled by D/8 lanes.
// ---------------------------------------------------------------------------
// One row: src its first element (this lane's 8 channels), msub / mbias the
// mean rows (or null), orow its output row (codes, bias), sidx its scale.
template <typename T>
__device__ __forceinline__ void quant_row(const QuantParams &p, bool valid, const T *src,
                                          const float *msub, const float *mbias, int64_t orow,
                                          int64_t sidx, int c0, int tpr) {
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float amax = 0.0f, dot = 0.0f;
    if (valid) {
        load8(src, v);
        if (mbias) {
#pragma unroll
            for (int i = 0; i < 8; ++i) dot = fmaf(v[i], mbias[i], dot);
        }
        if (msub) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = v[i] - msub[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = row_max(amax, tpr);
    dot = row_sum(dot, tpr);
    if (!valid) return;
    const float s = __fdiv_rn(amax, 127.0f);
    store8_i8(p.q + orow * p.D + c0, v, s);
    if (threadIdx.x % tpr == 0) {
        p.scale[sidx] = s;
        if (p.bias) p.bias[orow] = dot;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) quant_rows_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int rows_per_cta = 256 / tpr;
    const int64_t nrows = (int64_t)p.B * p.H * p.S;
    const int64_t r = (int64_t)blockIdx.x * rows_per_cta + threadIdx.x / tpr;
    const int c0 = (threadIdx.x % tpr) * 8;
    const bool valid = r < nrows;
    const T *src = nullptr;
    const float *msub = nullptr, *mbias = nullptr;
    if (valid) {
        const int64_t s = r % p.S;
        const int64_t bh = r / p.S;
        const int64_t b = bh / p.H, h = bh % p.H;
        src = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + s * p.ss + c0;
        if (p.mu_bias) mbias = p.mu_bias + (b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0;
        if (p.mu_sub) msub = p.mu_sub + bh * p.D + c0;
    }
    quant_row<T>(p, valid, src, msub, mbias, r, r, c0, tpr);
}

// Packed batch: row r = (head h, packed token t); t's sequence by bisection.
// Tokens outside every valid sequence are left untouched.
template <typename T>
__global__ void __launch_bounds__(256) quant_rows_varlen_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int rows_per_cta = 256 / tpr;
    const int64_t nrows = (int64_t)p.H * p.total;
    const int64_t r = (int64_t)blockIdx.x * rows_per_cta + threadIdx.x / tpr;
    const int c0 = (threadIdx.x % tpr) * 8;
    bool valid = r < nrows;
    const T *src = nullptr;
    const float *msub = nullptr, *mbias = nullptr;
    if (r < p.B && c0 == 0) {
        // the first B rows also check one sequence each for the error word
        int64_t start = 0;
        varlen_seq(p.cu, (int)r, p.S, p.total, p.err, &start);
    }
    if (valid) {
        const int64_t h = r / p.total, t = r % p.total;
        const int b = varlen_bisect(p.B, t, [&](int i) { return (int64_t)p.cu[i]; });
        int64_t start = 0;
        const int len = varlen_seq(p.cu, b, p.S, p.total, nullptr, &start);
        valid = t >= start && t < start + len;
        src = reinterpret_cast<const T *>(p.x) + h * p.sh + t * p.ss + c0;
        if (p.mu_bias)
            mbias = p.mu_bias + ((int64_t)b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0;
        if (p.mu_sub) msub = p.mu_sub + ((int64_t)b * p.H + h) * p.D + c0;
    }
    quant_row<T>(p, valid, src, msub, mbias, r, r, c0, tpr);
}

// ---------------------------------------------------------------------------
// Per-block quantisation: one CTA per (b, h, block of `block` tokens).
// Pass 1 finds the block's amax (and per-row biases); pass 2 re-reads the
// block (L1/L2 resident) and writes the codes.
// ---------------------------------------------------------------------------
// Tokens [t0, t1) of one (sequence, head): token t at base + t * p.ss (this
// lane's channels), output row orow0 + t, scale at sidx.
template <typename T>
__device__ __forceinline__ void quant_block(const QuantParams &p, const T *base,
                                            const float *msub, const float *mbias, int64_t t0,
                                            int64_t t1, int64_t orow0, int64_t sidx) {
    __shared__ float red[8];
    const int tpr = p.D / 8;
    const int rows_per_pass = 256 / tpr;
    const int c0 = (threadIdx.x % tpr) * 8;
    float amax = 0.0f;
    for (int64_t t = t0 + threadIdx.x / tpr; t - (threadIdx.x / tpr) < t1; t += rows_per_pass) {
        const bool valid = t < t1;
        float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float dot = 0.0f;
        if (valid) {
            load8(base + t * p.ss, v);
            if (mbias) {
#pragma unroll
                for (int i = 0; i < 8; ++i) dot = fmaf(v[i], mbias[i], dot);
            }
            if (msub) {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = v[i] - msub[i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        if (mbias) {
            dot = row_sum(dot, tpr);
            if (valid && threadIdx.x % tpr == 0) p.bias[orow0 + t] = dot;
        }
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float a = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
        a = warp_max(a);
        if (threadIdx.x == 0) red[0] = a;
    }
    __syncthreads();
    const float s = __fdiv_rn(red[0], 127.0f);
    if (threadIdx.x == 0) p.scale[sidx] = s;
    for (int64_t t = t0 + threadIdx.x / tpr; t < t1; t += rows_per_pass) {
        float v[8];
        load8(base + t * p.ss, v);
        if (msub) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = v[i] - msub[i];
        }
        store8_i8(p.q + (orow0 + t) * p.D + c0, v, s);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) quant_blocks_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int64_t ngroups = (p.S + p.block - 1) / p.block;
    const int64_t g = blockIdx.x % ngroups;
    const int64_t bh = blockIdx.x / ngroups;
    const int64_t b = bh / p.H, h = bh % p.H;
    const int64_t t0 = g * p.block;
    const int64_t t1 = (t0 + p.block < (int64_t)p.S) ? t0 + p.block : (int64_t)p.S;
    const int c0 = (threadIdx.x % tpr) * 8;
    const T *base = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + c0;
    const float *msub = p.mu_sub ? p.mu_sub + bh * p.D + c0 : nullptr;
    const float *mbias =
        p.mu_bias ? p.mu_bias + (b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0 : nullptr;
    quant_block<T>(p, base, msub, mbias, t0, t1, bh * p.S, bh * ngroups + g);
}

// Packed batch: one CTA per (head, scale group); the group's sequence by
// bisection over the sequences' first groups.  A group slot past its
// sequence's end (the layout reserves up to one per sequence) gets scale 0.
template <typename T>
__global__ void __launch_bounds__(256) quant_blocks_varlen_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int64_t g = blockIdx.x % p.groups;
    const int64_t h = blockIdx.x / p.groups;
    const int b = varlen_bisect(p.B, g, [&](int i) {
        return varlen_group0(p.cu[i] < 0 ? 0 : p.cu[i], i, p.block);
    });
    int64_t start = 0;
    const int len = varlen_seq(p.cu, b, p.S, p.total, threadIdx.x == 0 ? p.err : nullptr, &start);
    const int64_t j = g - varlen_group0(start, b, p.block);
    const int64_t t0 = j * p.block;
    if (len == 0 || j < 0 || t0 >= len) {
        if (threadIdx.x == 0) p.scale[h * p.groups + g] = 0.0f;
        return;
    }
    const int64_t t1 = (t0 + p.block < (int64_t)len) ? t0 + p.block : (int64_t)len;
    const int c0 = (threadIdx.x % tpr) * 8;
    const T *base = reinterpret_cast<const T *>(p.x) + h * p.sh + start * p.ss + c0;
    const float *msub = p.mu_sub ? p.mu_sub + ((int64_t)b * p.H + h) * p.D + c0 : nullptr;
    const float *mbias =
        p.mu_bias ? p.mu_bias + ((int64_t)b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0
                  : nullptr;
    quant_block<T>(p, base, msub, mbias, t0, t1, h * p.total + start, h * p.groups + g);
}

// ---------------------------------------------------------------------------
// smooth_k mean: mu[b,h,c] = (sum_t x[b,h,t,c]) / S rounded once to fp32.
// A cluster of kMeanCluster CTAs shares one (b, h): each CTA sums a slice
// of tokens, rank 0 adds the slices through distributed shared memory.
// f16: every f16 value is an integer multiple of 2^-24 below 2^16, so the
// sum is accumulated EXACTLY as an int64 count of 2^-24 units; bf16 sums
// in fp64 (exact whenever the fp64 sum is).
// ---------------------------------------------------------------------------
constexpr int kMeanCluster = 8;

template <typename T>
struct MeanAcc {
    using type = double;
    static __device__ __forceinline__ double conv(float x) { return (double)x; }
    static __device__ __forceinline__ double finish(double s) { return s; }
};
template <>
struct MeanAcc<__half> {
    using type = long long;
    static __device__ __forceinline__ long long conv(float x) {
        return __float2ll_rn(x * 16777216.0f);  // exact: x * 2^24 is an integer
    }
    static __device__ __forceinline__ double finish(long long s) {
        return (double)s * (1.0 / 16777216.0);
    }
};

template <typename T>
__global__ void __launch_bounds__(256) token_mean_kernel(QuantParams p) {
    using Acc = typename MeanAcc<T>::type;
    __shared__ Acc part[2048];     // [token lanes][D]: (256 / (D/8)) * D = 2048
    __shared__ Acc cta_sum[256];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int tpr = p.D / 8;
    const int lanes_t = 256 / tpr;
    const int64_t bh = blockIdx.y;
    const int64_t b = bh / p.H, h = bh % p.H;
    // tokens of this (sequence, head): dense S rows, or one packed sequence
    int64_t n = p.S;
    const T *base = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh;
    if (p.cu) {
        int64_t start = 0;
        n = varlen_seq(p.cu, (int)b, p.S, p.total, nullptr, &start);
        base = reinterpret_cast<const T *>(p.x) + start * p.ss + h * p.sh;
    }
    const int64_t chunk = (n + kMeanCluster - 1) / kMeanCluster;
    const int64_t t0 = rank * chunk;
    const int64_t t1 = (t0 + chunk < n) ? t0 + chunk : n;
    const int c0 = (threadIdx.x % tpr) * 8;
    const int lt = threadIdx.x / tpr;
    base += c0;
    Acc acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    for (int64_t t = t0 + lt; t < t1; t += lanes_t) {
        float v[8];
        load8(base + t * p.ss, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += MeanAcc<T>::conv(v[i]);
    }
    // reduce over the token lanes
#pragma unroll
    for (int i = 0; i < 8; ++i) part[lt * p.D + c0 + i] = acc[i];
    __syncthreads();
    if (threadIdx.x < p.D) {
        Acc sum = 0;
        for (int l = 0; l < lanes_t; ++l) sum += part[l * p.D + threadIdx.x];
        cta_sum[threadIdx.x] = sum;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x < p.D) {
        Acc tot = 0;
        for (int r = 0; r < kMeanCluster; ++r) tot += cluster.map_shared_rank(cta_sum, r)[threadIdx.x];
        // an empty sequence has no mean; 0 keeps its (unused) row defined
        const double mean = n > 0 ? MeanAcc<T>::finish(tot) / (double)n : 0.0;
        p.mu_out[bh * p.D + threadIdx.x] = (float)mean;
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

template <typename T>
cudaError_t launch_quant_t(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    cudaError_t e = cudaSuccess;
    QuantParams q = p;
    if (p.smooth) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kMeanCluster, (unsigned)(p.B * p.H), 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kMeanCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, token_mean_kernel<T>, q);
        log.add("token_mean_kernel", cfg.gridDim, cfg.blockDim, dim3(kMeanCluster, 1, 1), 0);
        if (e != cudaSuccess) return e;
        q.mu_sub = p.mu_out;
    }
    if (p.cu) {
        if (p.block == 1) {
            const int rows_per_cta = 256 / (p.D / 8);
            const int64_t nrows = (int64_t)p.H * p.total;
            const unsigned grid = (unsigned)((nrows + rows_per_cta - 1) / rows_per_cta);
            if (grid > 0) {
                quant_rows_varlen_kernel<T><<<grid, 256, 0, st>>>(q);
                log.add("quant_rows_varlen_kernel", dim3(grid), dim3(256), dim3(1, 1, 1), 0);
            }
        } else {
            const unsigned grid = (unsigned)((int64_t)p.H * p.groups);
            if (grid > 0) {
                quant_blocks_varlen_kernel<T><<<grid, 256, 0, st>>>(q);
                log.add("quant_blocks_varlen_kernel", dim3(grid), dim3(256), dim3(1, 1, 1), 0);
            }
        }
    } else if (p.block == 1) {
        const int rows_per_cta = 256 / (p.D / 8);
        const int64_t nrows = (int64_t)p.B * p.H * p.S;
        const unsigned grid = (unsigned)((nrows + rows_per_cta - 1) / rows_per_cta);
        if (grid > 0) {
            quant_rows_kernel<T><<<grid, 256, 0, st>>>(q);
            log.add("quant_rows_kernel", dim3(grid), dim3(256), dim3(1, 1, 1), 0);
        }
    } else {
        const int64_t ngroups = (p.S + p.block - 1) / p.block;
        const unsigned grid = (unsigned)((int64_t)p.B * p.H * ngroups);
        if (grid > 0) {
            quant_blocks_kernel<T><<<grid, 256, 0, st>>>(q);
            log.add("quant_blocks_kernel", dim3(grid), dim3(256), dim3(1, 1, 1), 0);
        }
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    if (p.bf16) return launch_quant_t<__nv_bfloat16>(p, st, log);
    return launch_quant_t<__half>(p, st, log);
}

}  // namespace sage
