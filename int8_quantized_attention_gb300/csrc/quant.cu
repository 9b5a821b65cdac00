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
__device__ __forceinline__ void cvt8(const uint4 &raw, float (&v)[8]) {
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = DT<T>::to_f(e[i]);
}

template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&v)[8]) {
    cvt8<T>(*reinterpret_cast<const uint4 *>(p), v);
}

// 16-byte load through the read-only path (inputs are never written here)
__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void store8_i8(int8_t *dst, const float (&v)[8], float s) {
    uint32_t w0, w1;
    quant8(v, s, quant_recip(s), w0, w1);
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
// Each thread takes kRowsPerThread rows (its 8 channels of each), issuing
// all their loads before any arithmetic so that several 16-byte loads per
// thread are in flight (one at a time left the kernel latency-bound).
constexpr int kRowsPerThread = 4;

// One row of a thread: src its 8 channels, msub / mbias the mean rows (or
// null), orow its output row (codes, bias; also its scale index).
template <typename T>
struct RowJob {
    const T *src;
    const float *msub, *mbias;
    int64_t orow;
    bool valid;
};

template <typename T>
__device__ __forceinline__ void quant_rows(const QuantParams &p, const RowJob<T> (&job)[kRowsPerThread],
                                           int c0, int tpr) {
    uint4 raw[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k)
        raw[k] = job[k].valid ? ldg16(job[k].src) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        float v[8];
        cvt8<T>(raw[k], v);
        float amax = 0.0f, dot = 0.0f;
        if (job[k].valid) {
            if (job[k].mbias) {
#pragma unroll
                for (int i = 0; i < 8; ++i) dot = fmaf(v[i], job[k].mbias[i], dot);
            }
            if (job[k].msub) {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = v[i] - job[k].msub[i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        // every lane of the row takes part (valid is uniform over a row)
        amax = row_max(amax, tpr);
        dot = row_sum(dot, tpr);
        if (!job[k].valid) continue;
        const float sc = __fdiv_rn(amax, 127.0f);
        store8_i8(p.q + job[k].orow * p.D + c0, v, sc);
        if (threadIdx.x % tpr == 0) {
            p.scale[job[k].orow] = sc;
            if (p.bias) p.bias[job[k].orow] = dot;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) quant_rows_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int rows_per_slab = 256 / tpr;
    const int64_t nrows = (int64_t)p.B * p.H * p.S;
    const int c0 = (threadIdx.x % tpr) * 8;
    RowJob<T> job[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const int64_t r =
            ((int64_t)blockIdx.x * kRowsPerThread + k) * rows_per_slab + threadIdx.x / tpr;
        job[k] = RowJob<T>{nullptr, nullptr, nullptr, r, r < nrows};
        if (r < nrows) {
            const int64_t s = r % p.S;
            const int64_t bh = r / p.S;
            const int64_t b = bh / p.H, h = bh % p.H;
            job[k].src = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + s * p.ss + c0;
            if (p.mu_bias)
                job[k].mbias = p.mu_bias + (b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0;
            if (p.mu_sub) job[k].msub = p.mu_sub + bh * p.D + c0;
        }
    }
    quant_rows<T>(p, job, c0, tpr);
}

// Packed batch: row r = (head h, packed token t); t's sequence by bisection.
// Tokens outside every valid sequence are left untouched.
template <typename T>
__global__ void __launch_bounds__(256) quant_rows_varlen_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const int rows_per_slab = 256 / tpr;
    const int64_t nrows = (int64_t)p.H * p.total;
    const int c0 = (threadIdx.x % tpr) * 8;
    {
        // the first B threads of the grid also check one sequence each for
        // the error word
        const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        if (g < p.B) {
            int64_t start = 0;
            varlen_seq(p.cu, (int)g, p.S, p.total, p.err, &start);
        }
    }
    RowJob<T> job[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const int64_t r =
            ((int64_t)blockIdx.x * kRowsPerThread + k) * rows_per_slab + threadIdx.x / tpr;
        job[k] = RowJob<T>{nullptr, nullptr, nullptr, r, false};
        if (r < nrows) {
            const int64_t h = r / p.total, t = r % p.total;
            const int b = varlen_bisect(p.B, t, [&](int i) { return (int64_t)p.cu[i]; });
            int64_t start = 0;
            const int len = varlen_seq(p.cu, b, p.S, p.total, nullptr, &start);
            job[k].valid = t >= start && t < start + len;
            job[k].src = reinterpret_cast<const T *>(p.x) + h * p.sh + t * p.ss + c0;
            if (p.mu_bias)
                job[k].mbias =
                    p.mu_bias + ((int64_t)b * p.mu_heads + h / (p.H / p.mu_heads)) * p.D + c0;
            if (p.mu_sub) job[k].msub = p.mu_sub + ((int64_t)b * p.H + h) * p.D + c0;
        }
    }
    quant_rows<T>(p, job, c0, tpr);
}

// ---------------------------------------------------------------------------
// Per-block quantisation: one CTA per (b, h, block of `block` tokens).
// The CTA is sized to the block (block * D / 32 threads, at most 1024), so
// each thread holds at most kBlockRows rows of 8 channels in registers: every
// load of the block is issued at once and the codes are written from the
// registers.  Larger blocks take two passes with 256 threads (the second
// re-reads the block from L1/L2).
// ---------------------------------------------------------------------------
constexpr int kBlockRows = 4;

__device__ __forceinline__ float block_max(float amax) {
    __shared__ float red[32];
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float a = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        a = warp_max(a);
        if (threadIdx.x == 0) red[0] = a;
    }
    __syncthreads();
    return red[0];
}

// Tokens [t0, t1) of one (sequence, head): token t at base + t * p.ss (this
// lane's channels), output row orow0 + t, scale at sidx.
template <typename T, int IT>
__device__ __forceinline__ void quant_block_regs(const QuantParams &p, const T *base,
                                                 const float *msub, const float *mbias,
                                                 int64_t t0, int64_t t1, int64_t orow0,
                                                 int64_t sidx) {
    const int tpr = p.D / 8;
    const int rpp = blockDim.x / tpr;
    const int lt = threadIdx.x / tpr;
    const int c0 = (threadIdx.x % tpr) * 8;
    uint4 raw[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int64_t t = t0 + lt + (int64_t)it * rpp;
        raw[it] = t < t1 ? ldg16(base + t * p.ss) : make_uint4(0, 0, 0, 0);
    }
    float ms[8], mb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ms[i] = msub ? msub[i] : 0.0f;
        mb[i] = mbias ? mbias[i] : 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int64_t t = t0 + lt + (int64_t)it * rpp;
        float v[8];
        cvt8<T>(raw[it], v);
        if (mbias) {
            float dot = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) dot = fmaf(v[i], mb[i], dot);
            dot = row_sum(dot, tpr);
            if (t < t1 && threadIdx.x % tpr == 0) p.bias[orow0 + t] = dot;
        }
        if (t < t1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(msub ? v[i] - ms[i] : v[i]));
        }
    }
    const float s = __fdiv_rn(block_max(amax), 127.0f);
    if (threadIdx.x == 0) p.scale[sidx] = s;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int64_t t = t0 + lt + (int64_t)it * rpp;
        if (t < t1) {
            float v[8];
            cvt8<T>(raw[it], v);
            if (msub) {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = v[i] - ms[i];
            }
            store8_i8(p.q + (orow0 + t) * p.D + c0, v, s);
        }
    }
}

template <typename T>
__device__ __forceinline__ void quant_block(const QuantParams &p, const T *base,
                                            const float *msub, const float *mbias, int64_t t0,
                                            int64_t t1, int64_t orow0, int64_t sidx) {
    const int tpr = p.D / 8;
    const int rows_per_pass = blockDim.x / tpr;
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
    const float s = __fdiv_rn(block_max(amax), 127.0f);
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

template <typename T, int IT>
__device__ __forceinline__ void quant_block_any(const QuantParams &p, const T *base,
                                                const float *msub, const float *mbias,
                                                int64_t t0, int64_t t1, int64_t orow0,
                                                int64_t sidx) {
    if constexpr (IT > 0)
        quant_block_regs<T, IT>(p, base, msub, mbias, t0, t1, orow0, sidx);
    else
        quant_block<T>(p, base, msub, mbias, t0, t1, orow0, sidx);
}

template <typename T, int IT>
__global__ void __launch_bounds__(1024) quant_blocks_kernel(QuantParams p) {
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
    quant_block_any<T, IT>(p, base, msub, mbias, t0, t1, bh * p.S, bh * ngroups + g);
}

// Packed batch: one CTA per (head, scale group); the group's sequence by
// bisection over the sequences' first groups.  A group slot past its
// sequence's end (the layout reserves up to one per sequence) gets scale 0.
template <typename T, int IT>
__global__ void __launch_bounds__(1024) quant_blocks_varlen_kernel(QuantParams p) {
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
    quant_block_any<T, IT>(p, base, msub, mbias, t0, t1, h * p.total + start, h * p.groups + g);
}

// ---------------------------------------------------------------------------
// smooth_k mean: mu[b,h,c] = (sum_t x[b,h,t,c]) / S rounded once to fp32.
// A cluster of kMeanCluster CTAs shares one (b, h): each CTA sums a slice
// of tokens, rank 0 adds the slices through distributed shared memory.
// f16: every f16 value is an integer multiple of 2^-24 below 2^16, so the
// sum is kept EXACTLY as an integer count of 2^-24 units.  Without a
// 64-bit float-to-integer conversion per element (that unit saturated
// first): x * 2^24 = hi * 2^20 + lo with integers |hi| <= 2^20 and
// |lo| <= 2^19, both obtained on the FMA pipe from the bits of
// t = x * 2^4 + 1.5 * 2^23 (rounded once to the integer hi, held in the
// low mantissa bits of t) and of lo + 1.5 * 2^23; the raw bit patterns are
// summed in 32 bits (their constant 1.5 * 2^23 part is taken off once per
// count) and folded into 64 bits every kMeanFold tokens.  bf16 sums in
// fp64 (exact whenever the fp64 sum is).
// ---------------------------------------------------------------------------
constexpr int kMeanCluster = 8;
constexpr int kMeanUnroll = 8;
constexpr int kMeanFold = 1024;  // tokens per thread between 64-bit folds

template <typename T>
struct MeanAcc {  // bf16: fp64 sums
    struct Part {
        double s[8];
        __device__ __forceinline__ void zero() {
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i] = 0.0;
        }
        __device__ __forceinline__ void add(const float (&v)[8]) {
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i] += (double)v[i];
        }
    };
    using type = double;
    static __device__ __forceinline__ void fold(Part &p, type (&acc)[8], int) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += p.s[i];
        p.zero();
    }
    static __device__ __forceinline__ double finish(double s) { return s; }
};

template <>
struct MeanAcc<__half> {
    static constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    struct Part {
        uint32_t hi[8], lo[8];
        __device__ __forceinline__ void zero() {
#pragma unroll
            for (int i = 0; i < 8; ++i) hi[i] = lo[i] = 0u;
        }
        __device__ __forceinline__ void add(const float (&v)[8]) {
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 x = make_float2(v[i], v[i + 1]);
                // t = rne(x * 2^4) + 1.5 * 2^23 (|x * 2^4| < 2^20: one rounding)
                const float2 t = ffma2(x, make_float2(16.0f, 16.0f), make_float2(kMagic, kMagic));
                const float2 h = fadd2(t, make_float2(-kMagic, -kMagic));  // hi, exact
                // lo = x * 2^24 - hi * 2^20: an integer of magnitude <= 2^19, exact
                const float2 xl = fmul2(x, make_float2(16777216.0f, 16777216.0f));
                const float2 l = ffma2(h, make_float2(-1048576.0f, -1048576.0f), xl);
                const float2 tl = fadd2(l, make_float2(kMagic, kMagic));
                hi[i] += __float_as_uint(t.x);
                hi[i + 1] += __float_as_uint(t.y);
                lo[i] += __float_as_uint(tl.x);
                lo[i + 1] += __float_as_uint(tl.y);
            }
        }
    };
    using type = long long;
    // n: values added since the last fold (each carried 1.5 * 2^23 in its bits)
    static __device__ __forceinline__ void fold(Part &p, type (&acc)[8], int n) {
        const uint32_t off = (uint32_t)n * (uint32_t)__float_as_uint(kMagic);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long h = (int32_t)(p.hi[i] - off), l = (int32_t)(p.lo[i] - off);
            acc[i] += h * 1048576ll + l;
        }
        p.zero();
    }
    static __device__ __forceinline__ double finish(long long s) {
        return (double)s * (1.0 / 16777216.0);
    }
};

template <typename T>
__global__ void __launch_bounds__(256) token_mean_kernel(QuantParams p) {
    using M = MeanAcc<T>;
    using Acc = typename M::type;
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
    typename M::Part part32;
    part32.zero();
    int since_fold = 0;
    // kMeanUnroll loads in flight per thread; rows past the slice load as
    // zeros, which add nothing (and are counted like the rest)
    for (int64_t t = t0 + lt; t < t1; t += (int64_t)lanes_t * kMeanUnroll) {
        uint4 raw[kMeanUnroll];
#pragma unroll
        for (int u = 0; u < kMeanUnroll; ++u) {
            const int64_t tt = t + (int64_t)u * lanes_t;
            raw[u] = tt < t1 ? ldg16(base + tt * p.ss) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kMeanUnroll; ++u) {
            float v[8];
            cvt8<T>(raw[u], v);
            part32.add(v);
        }
        since_fold += kMeanUnroll;
        if (since_fold >= kMeanFold) {
            M::fold(part32, acc, since_fold);
            since_fold = 0;
        }
    }
    M::fold(part32, acc, since_fold);
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

// Per-block kernels, instantiated by the block's rows per thread (IT, the
// register-resident path) or 0 (two passes, blocks too large for registers).
template <typename T, int IT>
void launch_blocks_it(const QuantParams &q, unsigned grid, unsigned threads, cudaStream_t st,
                      bool varlen) {
    if (varlen)
        quant_blocks_varlen_kernel<T, IT><<<grid, threads, 0, st>>>(q);
    else
        quant_blocks_kernel<T, IT><<<grid, threads, 0, st>>>(q);
}

// Threads per block CTA: kBlockRows rows of 8 channels per thread (a whole
// number of warps, which is a whole number of rows since D / 8 <= 32);
// 0 when the block needs more than 1024 threads.
inline unsigned block_threads(int block, int D) {
    const long long elems = (long long)block * D;
    const long long t = (elems / (8 * kBlockRows) + 31) / 32 * 32;
    return t <= 1024 ? (unsigned)(t < 32 ? 32 : t) : 0u;
}

template <typename T>
unsigned launch_blocks(const QuantParams &q, unsigned grid, cudaStream_t st, bool varlen) {
    const unsigned threads = block_threads(q.block, q.D);
    if (threads)
        launch_blocks_it<T, kBlockRows>(q, grid, threads, st, varlen);
    else
        launch_blocks_it<T, 0>(q, grid, 256, st, varlen);
    return threads ? threads : 256;
}

template <typename T>
cudaError_t launch_mean_t(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
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
    const cudaError_t e = cudaLaunchKernelEx(&cfg, token_mean_kernel<T>, p);
    log.add("token_mean_kernel", cfg.gridDim, cfg.blockDim, dim3(kMeanCluster, 1, 1), 0);
    return e;
}

template <typename T>
cudaError_t launch_quant_t(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    cudaError_t e = cudaSuccess;
    QuantParams q = p;
    if (p.smooth) {
        e = launch_mean_t<T>(q, st, log);
        if (e != cudaSuccess) return e;
        q.mu_sub = p.mu_out;
    }
    if (p.cu) {
        if (p.block == 1) {
            const int rows_per_cta = 256 / (p.D / 8) * kRowsPerThread;
            const int64_t nrows = (int64_t)p.H * p.total;
            const int64_t checks = ((int64_t)p.B + 255) / 256;   // error-word checks
            int64_t g = (nrows + rows_per_cta - 1) / rows_per_cta;
            const unsigned grid = (unsigned)(g > checks ? g : checks);
            if (grid > 0) {
                quant_rows_varlen_kernel<T><<<grid, 256, 0, st>>>(q);
                log.add("quant_rows_varlen_kernel", dim3(grid), dim3(256), dim3(1, 1, 1), 0);
            }
        } else {
            const unsigned grid = (unsigned)((int64_t)p.H * p.groups);
            if (grid > 0) {
                const unsigned th = launch_blocks<T>(q, grid, st, true);
                log.add("quant_blocks_varlen_kernel", dim3(grid), dim3(th), dim3(1, 1, 1), 0);
            }
        }
    } else if (p.block == 1) {
        const int rows_per_cta = 256 / (p.D / 8) * kRowsPerThread;
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
            const unsigned th = launch_blocks<T>(q, grid, st, false);
            log.add("quant_blocks_kernel", dim3(grid), dim3(th), dim3(1, 1, 1), 0);
        }
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    if (p.bf16) return launch_quant_t<__nv_bfloat16>(p, st, log);
    return launch_quant_t<__half>(p, st, log);
}

cudaError_t launch_token_mean(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    if ((int64_t)p.B * p.H == 0) return cudaSuccess;
    if (p.bf16) return launch_mean_t<__nv_bfloat16>(p, st, log);
    return launch_mean_t<__half>(p, st, log);
}

}  // namespace sage
