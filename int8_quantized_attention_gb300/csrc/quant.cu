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

#include <type_traits>

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
// Per-token quantisation: each row of D elements is handled by
// D / (8 * kRowChunks) lanes, each holding kRowChunks 16-byte chunks of it,
// interleaved so that one load instruction of a row's lanes reads
// contiguous bytes.  The per-row work (the lane reductions, the scale's
// division and reciprocal, the row's addresses) is shared by 32 channels of
// a lane (with 8 per lane it was most of the instructions).  Each thread
// takes kRowsPerThread rows, issuing all their loads before any arithmetic.
// ---------------------------------------------------------------------------
constexpr int kRowChunks = 4;
constexpr int kRowsPerThread = 1;

// One row of a thread: src its first chunk, msub / mbias the mean rows at
// that chunk (or null), orow its output row (codes, bias; also its scale).
template <typename T>
struct RowJob {
    const T *src;
    const float *msub, *mbias;
    int64_t orow;
    bool valid;
};

__device__ __forceinline__ void sub8(float (&v)[8], const float *m) {
    const float4 a = *reinterpret_cast<const float4 *>(m);
    const float4 b = *reinterpret_cast<const float4 *>(m + 4);
    v[0] -= a.x, v[1] -= a.y, v[2] -= a.z, v[3] -= a.w;
    v[4] -= b.x, v[5] -= b.y, v[6] -= b.z, v[7] -= b.w;
}

__device__ __forceinline__ float dot8(const float (&v)[8], const float *m, float acc) {
    const float4 a = *reinterpret_cast<const float4 *>(m);
    const float4 b = *reinterpret_cast<const float4 *>(m + 4);
    acc = fmaf(v[0], a.x, acc), acc = fmaf(v[1], a.y, acc);
    acc = fmaf(v[2], a.z, acc), acc = fmaf(v[3], a.w, acc);
    acc = fmaf(v[4], b.x, acc), acc = fmaf(v[5], b.y, acc);
    acc = fmaf(v[6], b.z, acc), acc = fmaf(v[7], b.w, acc);
    return acc;
}

// cs: elements between a lane's chunks (tpr * 8); c0: this lane's first
// channel.  Lanes of one row are consecutive and `valid` is uniform over them.
template <typename T>
__device__ __forceinline__ void quant_rows(const QuantParams &p, const RowJob<T> (&job)[kRowsPerThread],
                                           int c0, int tpr) {
    const int cs = tpr * 8;
    uint4 raw[kRowsPerThread][kRowChunks];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k)
#pragma unroll
        for (int c = 0; c < kRowChunks; ++c)
            raw[k][c] = job[k].valid ? ldg16(job[k].src + c * cs) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        float amax = 0.0f, dot = 0.0f;
        if (job[k].valid) {
#pragma unroll
            for (int c = 0; c < kRowChunks; ++c) {
                float v[8];
                cvt8<T>(raw[k][c], v);
                if (job[k].mbias) dot = dot8(v, job[k].mbias + c * cs, dot);
                if (job[k].msub) sub8(v, job[k].msub + c * cs);
                amax = fmax3(amax, fmax3(fabsf(v[0]), fabsf(v[1]), fabsf(v[2])),
                             fmax3(fabsf(v[3]), fabsf(v[4]), fmaxf(fabsf(v[5]),
                                   fmaxf(fabsf(v[6]), fabsf(v[7])))));
            }
        }
        amax = row_max(amax, tpr);
        dot = row_sum(dot, tpr);
        if (!job[k].valid) continue;
        const float sc = __fdiv_rn(amax, 127.0f);
        const float rc = quant_recip(sc);
        int8_t *dst = p.q + job[k].orow * p.D + c0;
#pragma unroll
        for (int c = 0; c < kRowChunks; ++c) {
            float v[8];
            cvt8<T>(raw[k][c], v);
            if (job[k].msub) sub8(v, job[k].msub + c * cs);
            uint32_t w0, w1;
            quant8(v, sc, rc, w0, w1);
            *reinterpret_cast<uint2 *>(dst + c * cs) = make_uint2(w0, w1);
        }
        if (threadIdx.x % tpr == 0) {
            p.scale[job[k].orow] = sc;
            if (p.bias) p.bias[job[k].orow] = dot;
        }
    }
}

// Row r of a launch (r < n_outer * inner) is (outer0 + r / inner, r % inner);
// the divisions are multiplications by invariant-divisor constants (64-bit
// division per row left these kernels instruction-bound).
template <typename T>
__global__ void __launch_bounds__(256) quant_rows_kernel(QuantParams p) {
    // a decode launched behind this kernel may start now; it waits on the
    // device before reading the codes
    asm volatile("griddepcontrol.launch_dependents;");
    const int tpr = p.D / (8 * kRowChunks);
    const int rows_per_slab = (int)blockDim.x / tpr;
    const uint32_t nrows = p.n_outer * (uint32_t)p.S;
    const int c0 = (threadIdx.x % tpr) * 8;
    RowJob<T> job[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const uint32_t r =
            (blockIdx.x * kRowsPerThread + k) * rows_per_slab + threadIdx.x / tpr;
        job[k] = RowJob<T>{nullptr, nullptr, nullptr, 0, r < nrows};
        if (r < nrows) {
            const uint32_t ol = p.div_inner.div(r);
            const uint32_t s = r - ol * (uint32_t)p.S;
            const int64_t bh = p.outer0 + ol;
            const uint32_t b = p.div_h.div((uint32_t)bh);
            const uint32_t h = (uint32_t)bh - b * (uint32_t)p.H;
            job[k].orow = bh * p.S + s;
            job[k].src = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + s * p.ss + c0;
            if (p.mu_bias)
                job[k].mbias =
                    p.mu_bias + ((int64_t)b * p.mu_heads + p.div_grp.div(h)) * p.D + c0;
            if (p.mu_sub) job[k].msub = p.mu_sub + bh * p.D + c0;
        }
    }
    quant_rows<T>(p, job, c0, tpr);
}

// Packed batch: row r = (head h, packed token t); t's sequence by bisection.
// Tokens outside every valid sequence are left untouched.
template <typename T>
__global__ void __launch_bounds__(256) quant_rows_varlen_kernel(QuantParams p) {
    const int tpr = p.D / (8 * kRowChunks);
    const int rows_per_slab = (int)blockDim.x / tpr;
    const uint32_t nrows = p.n_outer * (uint32_t)p.total;
    const int c0 = (threadIdx.x % tpr) * 8;
    if (p.outer0 == 0) {
        // the first B threads of the first launch also check one sequence
        // each for the error word
        const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        if (g < p.B) {
            int64_t start = 0;
            varlen_seq(p.cu, (int)g, p.S, p.total, p.err, &start);
        }
    }
    RowJob<T> job[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const uint32_t r =
            (blockIdx.x * kRowsPerThread + k) * rows_per_slab + threadIdx.x / tpr;
        job[k] = RowJob<T>{nullptr, nullptr, nullptr, 0, false};
        if (r < nrows) {
            const uint32_t hl = p.div_inner.div(r);
            const int64_t t = r - hl * (uint32_t)p.total;
            const int64_t h = p.outer0 + hl;
            const int b = varlen_bisect(p.B, t, [&](int i) { return (int64_t)p.cu[i]; });
            int64_t start = 0;
            const int len = varlen_seq(p.cu, b, p.S, p.total, nullptr, &start);
            job[k].orow = h * p.total + t;
            job[k].valid = t >= start && t < start + len;
            job[k].src = reinterpret_cast<const T *>(p.x) + h * p.sh + t * p.ss + c0;
            if (p.mu_bias)
                job[k].mbias = p.mu_bias +
                               ((int64_t)b * p.mu_heads + p.div_grp.div((uint32_t)h)) * p.D + c0;
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
    // the mean rows are read per use (L1 hits), not held in registers
    float amax = 0.0f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int64_t t = t0 + lt + (int64_t)it * rpp;
        float v[8];
        cvt8<T>(raw[it], v);
        if (mbias) {
            float dot = dot8(v, mbias, 0.0f);
            dot = row_sum(dot, tpr);
            if (t < t1 && threadIdx.x % tpr == 0) p.bias[orow0 + t] = dot;
        }
        if (t < t1) {
            if (msub) sub8(v, msub);
            amax = fmax3(amax, fmax3(fabsf(v[0]), fabsf(v[1]), fabsf(v[2])),
                         fmax3(fabsf(v[3]), fabsf(v[4]), fmaxf(fabsf(v[5]),
                               fmaxf(fabsf(v[6]), fabsf(v[7])))));
        }
    }
    const float s = __fdiv_rn(block_max(amax), 127.0f);
    const float rc = quant_recip(s);
    if (threadIdx.x == 0) p.scale[sidx] = s;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int64_t t = t0 + lt + (int64_t)it * rpp;
        if (t < t1) {
            float v[8];
            cvt8<T>(raw[it], v);
            if (msub) sub8(v, msub);
            uint32_t w0, w1;
            quant8(v, s, rc, w0, w1);
            *reinterpret_cast<uint2 *>(p.q + (orow0 + t) * p.D + c0) = make_uint2(w0, w1);
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

// Group of CTA x of the dense per-block launch into L2 (rows contiguous:
// one bulk request; strided rows are not prefetched).  Each CTA loads its
// group at its start; asking L2 for the group of the CTA half a wave of
// resident CTAs ahead turns those later loads from DRAM misses into L2
// hits (half a wave measured best: Q 109 to 101 us, K mean + quantisation
// 178 to 175 us on 268 MB tensors; one and two waves gained less).
template <typename T>
__device__ __forceinline__ void prefetch_group(const QuantParams &p, uint32_t x) {
    if (x >= gridDim.x || p.ss != p.D) return;
    const uint32_t bh = p.div_inner.div(x);
    const uint32_t g = x - bh * p.div_inner.d;
    const uint32_t b = p.div_h.div(bh);
    const uint32_t h = bh - b * (uint32_t)p.H;
    const int64_t t0 = (int64_t)g * p.block;
    const int64_t t1 = (t0 + p.block < (int64_t)p.S) ? t0 + p.block : (int64_t)p.S;
    const T *src = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + t0 * p.D;
    const uint32_t bytes = (uint32_t)((t1 - t0) * p.D * (int64_t)sizeof(T));
    if (t1 > t0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <typename T, int IT>
__global__ void __launch_bounds__(1024) quant_blocks_kernel(QuantParams p) {
    if (threadIdx.x == 0 && p.ahead > 0) prefetch_group<T>(p, blockIdx.x + p.ahead);
    const int tpr = p.D / 8;
    // CTA = (b * H + h) * ngroups + g, split by invariant-divisor constants
    const uint32_t ngroups = p.div_inner.d;
    const uint32_t bh = p.div_inner.div(blockIdx.x);
    const uint32_t g = blockIdx.x - bh * ngroups;
    const uint32_t b = p.div_h.div(bh);
    const uint32_t h = bh - b * (uint32_t)p.H;
    const int64_t t0 = (int64_t)g * p.block;
    const int64_t t1 = (t0 + p.block < (int64_t)p.S) ? t0 + p.block : (int64_t)p.S;
    const int c0 = (threadIdx.x % tpr) * 8;
    const T *base = reinterpret_cast<const T *>(p.x) + b * p.sb + h * p.sh + c0;
    const float *msub = p.mu_sub ? p.mu_sub + (int64_t)bh * p.D + c0 : nullptr;
    const float *mbias =
        p.mu_bias ? p.mu_bias + ((int64_t)b * p.mu_heads + p.div_grp.div(h)) * p.D + c0 : nullptr;
    quant_block_any<T, IT>(p, base, msub, mbias, t0, t1, (int64_t)bh * p.S,
                           (int64_t)bh * ngroups + g);
}

// Packed batch: one CTA per (head, scale group); the group's sequence by
// bisection over the sequences' first groups.  A group slot past its
// sequence's end (the layout reserves up to one per sequence) gets scale 0.
template <typename T, int IT>
__global__ void __launch_bounds__(1024) quant_blocks_varlen_kernel(QuantParams p) {
    const int tpr = p.D / 8;
    const uint32_t hh = p.div_inner.div(blockIdx.x);  // CTA = h * groups + g
    const int64_t g = blockIdx.x - hh * (uint32_t)p.groups;
    const int64_t h = hh;
    const int b = varlen_find_warp(p.B, g, [&](int i) {
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
        p.mu_bias ? p.mu_bias + ((int64_t)b * p.mu_heads + p.div_grp.div(hh)) * p.D + c0
                  : nullptr;
    quant_block_any<T, IT>(p, base, msub, mbias, t0, t1, h * p.total + start, h * p.groups + g);
}

// ---------------------------------------------------------------------------
// smooth_k mean: mu[b,h,c] = (sum_t x[b,h,t,c]) / S rounded once to fp32.
// A cluster of kMeanCluster CTAs shares one (b, h) and kMeanSlice channels:
// each CTA sums a slice of tokens, rank 0 adds the slices through
// distributed shared memory (channel slices keep few (b, h) pairs from
// leaving most SMs idle).
// A value |x| < 2^16 that is an integer multiple of 2^-24 (every f16 value;
// a bf16 value of exponent -17 .. 15) is summed EXACTLY as an integer count
// of 2^-24 units.  Without a 64-bit float-to-integer conversion per element
// (that unit saturated first): x * 2^24 = hi * 2^20 + lo with integers
// |hi| <= 2^20 and |lo| <= 2^19, both obtained on the FMA pipe from the bits
// of t = x * 2^4 + 1.5 * 2^23 (rounded once to the integer hi, held in the
// low mantissa bits of t) and of lo + 1.5 * 2^23; the raw bit patterns are
// summed in 32 bits (their constant 1.5 * 2^23 part is taken off once per
// count) and folded into 64 bits every kMeanFold tokens.  Other bf16 values
// (tiny, large or not finite) are summed in fp64 on a rarely taken branch
// (the fp64 pipe is narrow: summing every bf16 value there was the
// bottleneck).  The total, count * 2^-24 plus the fp64 part, is exact
// whenever the values' binary span fits fp64's 53 bits.
// ---------------------------------------------------------------------------
constexpr int kMeanCluster = 8;
constexpr int kMeanSlice = 64;   // channels per CTA (8 lanes of 8)
constexpr int kMeanUnroll = 4;   // rows per thread per batch (two batches in flight)
constexpr int kMeanFold = 1024;  // tokens per thread between 64-bit folds
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// One thread's running sums over its 8 channels; kCheck: values may fall
// outside the exact range (bf16).
template <bool kCheck>
struct MeanPart {
    uint32_t hi[8], lo[8];
    double fb[8];  // values outside the exact range (kCheck only)
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hi[i] = lo[i] = 0u;
            fb[i] = 0.0;
        }
    }
    // the split of x (one pair of channels); ok: x lies in the exact range
    static __device__ __forceinline__ void split(float2 x, float2 &t, float2 &tl, bool &ok0,
                                                 bool &ok1) {
        // t = rne(x * 2^4) + 1.5 * 2^23 (|x * 2^4| < 2^20: one rounding)
        t = ffma2(x, make_float2(16.0f, 16.0f), make_float2(kMagic, kMagic));
        const float2 h = fadd2(t, make_float2(-kMagic, -kMagic));  // hi, exact
        // lo = x * 2^24 - hi * 2^20: an integer of magnitude <= 2^19 when x
        // is a multiple of 2^-24 (exact), else a fraction that tl rounds
        const float2 xl = fmul2(x, make_float2(16777216.0f, 16777216.0f));
        const float2 l = ffma2(h, make_float2(-1048576.0f, -1048576.0f), xl);
        tl = fadd2(l, make_float2(kMagic, kMagic));
        ok0 = ok1 = true;
        if (kCheck) {
            const float2 back = fadd2(tl, make_float2(-kMagic, -kMagic));
            ok0 = fabsf(x.x) < 65536.0f && back.x == l.x;
            ok1 = fabsf(x.y) < 65536.0f && back.y == l.y;
        }
    }
    __device__ __forceinline__ void add(const float (&v)[8]) {
        uint32_t bad = 0;  // bit i: channel i's value lies outside the range
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            float2 t, tl;
            bool ok0, ok1;
            split(make_float2(v[i], v[i + 1]), t, tl, ok0, ok1);
            // a value outside the range adds the magic alone (integer 0)
            hi[i] += ok0 ? __float_as_uint(t.x) : __float_as_uint(kMagic);
            hi[i + 1] += ok1 ? __float_as_uint(t.y) : __float_as_uint(kMagic);
            lo[i] += ok0 ? __float_as_uint(tl.x) : __float_as_uint(kMagic);
            lo[i + 1] += ok1 ? __float_as_uint(tl.y) : __float_as_uint(kMagic);
            bad |= (ok0 ? 0u : 1u << i) | (ok1 ? 0u : 2u << i);
        }
        if (kCheck && bad) add_outside(fb, v, bad);
    }
    // out of line: the rare fp64 path keeps its sums in local memory, off
    // the registers of the streaming loop
    static __device__ __noinline__ void add_outside(double *fb, const float (&v)[8], uint32_t bad) {
        for (int i = 0; i < 8; ++i)
            if (bad >> i & 1u) fb[i] += (double)v[i];
    }
    // n: values added since the last fold (each carried 1.5 * 2^23 in its bits)
    __device__ __forceinline__ void fold(long long (&acc)[8], int n) {
        const uint32_t off = (uint32_t)n * (uint32_t)__float_as_uint(kMagic);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const long long h = (int32_t)(hi[i] - off), l = (int32_t)(lo[i] - off);
            acc[i] += h * 1048576ll + l;
            hi[i] = lo[i] = 0u;
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(256) token_mean_kernel(QuantParams p) {
    constexpr bool kCheck = !std::is_same<T, __half>::value;
    constexpr int kTpr = kMeanSlice / 8;   // lanes per token row
    constexpr int kLanesT = 256 / kTpr;    // token lanes
    __shared__ long long part[kLanesT * kMeanSlice];
    __shared__ long long cta_sum[kMeanSlice];
    __shared__ double fpart[kCheck ? kLanesT * kMeanSlice : 1];
    __shared__ double fcta[kCheck ? kMeanSlice : 1];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
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
    const int cl = (threadIdx.x % kTpr) * 8;      // channel within the slice
    const int ch0 = blockIdx.z * kMeanSlice;      // the slice's first channel
    const int lt = threadIdx.x / kTpr;
    base += ch0 + cl;
    long long acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    MeanPart<kCheck> part32;
    part32.zero();
    int since_fold = 0;
    // Software pipelined: the next batch of kMeanUnroll rows is loaded
    // before the current one is summed, so a thread always has loads in
    // flight (loading, then summing, left HBM idle during the sums); rows
    // past the slice load as zeros, which add nothing (and are counted like
    // the rest).
    const int64_t step = (int64_t)kLanesT * kMeanUnroll;
    auto load_batch = [&](int64_t t, uint4 (&raw)[kMeanUnroll]) {
#pragma unroll
        for (int u = 0; u < kMeanUnroll; ++u) {
            const int64_t tt = t + (int64_t)u * kLanesT;
            raw[u] = tt < t1 ? ldg16(base + tt * p.ss) : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 cur[kMeanUnroll];
    load_batch(t0 + lt, cur);
    for (int64_t t = t0 + lt; t < t1; t += step) {
        uint4 nxt[kMeanUnroll];
        load_batch(t + step, nxt);
#pragma unroll
        for (int u = 0; u < kMeanUnroll; ++u) {
            float v[8];
            cvt8<T>(cur[u], v);
            part32.add(v);
        }
        since_fold += kMeanUnroll;
        if (since_fold >= kMeanFold) {
            part32.fold(acc, since_fold);
            since_fold = 0;
        }
#pragma unroll
        for (int u = 0; u < kMeanUnroll; ++u) cur[u] = nxt[u];
    }
    part32.fold(acc, since_fold);
    // reduce over the token lanes
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        part[lt * kMeanSlice + cl + i] = acc[i];
        if (kCheck) fpart[lt * kMeanSlice + cl + i] = part32.fb[i];
    }
    __syncthreads();
    if (threadIdx.x < kMeanSlice) {
        long long sum = 0;
        double fsum = 0.0;
        for (int l = 0; l < kLanesT; ++l) {
            sum += part[l * kMeanSlice + threadIdx.x];
            if (kCheck) fsum += fpart[l * kMeanSlice + threadIdx.x];
        }
        cta_sum[threadIdx.x] = sum;
        if (kCheck) fcta[threadIdx.x] = fsum;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x < kMeanSlice) {
        long long tot = 0;
        double ftot = 0.0;
        for (int r = 0; r < kMeanCluster; ++r) {
            tot += cluster.map_shared_rank(cta_sum, r)[threadIdx.x];
            if (kCheck) ftot += cluster.map_shared_rank(fcta, r)[threadIdx.x];
        }
        // an empty sequence has no mean; 0 keeps its (unused) row defined
        const double mean = n > 0 ? ((double)tot * (1.0 / 16777216.0) + ftot) / (double)n : 0.0;
        p.mu_out[bh * p.D + ch0 + threadIdx.x] = (float)mean;
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

// CTAs of `kernel` resident on the whole device at `threads` per CTA (0 if
// the query fails)
template <typename K>
uint32_t resident_ctas(K kernel, unsigned threads) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, (int)threads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return (uint32_t)(sms * per_sm);
}

template <typename T>
unsigned launch_blocks(const QuantParams &p, unsigned grid, cudaStream_t st, bool varlen) {
    QuantParams q = p;
    const unsigned threads = block_threads(q.block, q.D);
    if (threads) {
        if (!varlen) q.ahead = resident_ctas(quant_blocks_kernel<T, kBlockRows>, threads) / 2;
        launch_blocks_it<T, kBlockRows>(q, grid, threads, st, varlen);
    } else {
        if (!varlen) q.ahead = resident_ctas(quant_blocks_kernel<T, 0>, 256) / 2;
        launch_blocks_it<T, 0>(q, grid, 256, st, varlen);
    }
    return threads ? threads : 256;
}

template <typename T>
cudaError_t launch_mean_t(const QuantParams &p, cudaStream_t st, LaunchLog &log) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMeanCluster, (unsigned)(p.B * p.H), (unsigned)(p.D / kMeanSlice));
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
    q.div_h = FastDiv((uint32_t)(p.H > 0 ? p.H : 1));
    q.div_grp = FastDiv((uint32_t)(p.H / p.mu_heads > 0 ? p.H / p.mu_heads : 1));
    if (p.block == 1) {
        // per-token rows, in launches of whole outers below 2^31 rows each
        const int64_t inner = p.cu ? p.total : (int64_t)p.S;
        const int64_t outers = p.cu ? (int64_t)p.H : (int64_t)p.B * p.H;
        // few rows (a decode step's query): 64-thread CTAs spread the loads
        // over 4x the SMs (the rows' latency, not bandwidth, is the cost there)
        const int64_t all_rows = inner * outers;
        const int threads = all_rows <= 4096 ? 64 : 256;
        const int rows_per_cta = threads / (p.D / (8 * kRowChunks)) * kRowsPerThread;
        const int64_t limit = (1ll << 31) - 1 - rows_per_cta;
        const int64_t per = inner > 0 ? limit / inner : outers;  // outers per launch
        if ((inner > 0 && per < 1) || outers >= (1ll << 31))
            return cudaErrorInvalidValue;  // one outer of 2^31 rows, or 2^31 outers
        const int64_t chunk = per < outers ? per : outers;
        q.div_inner = FastDiv((uint32_t)(inner > 0 ? inner : 1));
        const int64_t checks = p.cu ? ((int64_t)p.B + threads - 1) / threads : 0;  // error-word checks
        int64_t o0 = 0, n = 0;
        do {
            n = outers - o0 < chunk ? outers - o0 : chunk;
            q.outer0 = o0;
            q.n_outer = (uint32_t)n;
            int64_t g = (n * inner + rows_per_cta - 1) / rows_per_cta;
            if (o0 == 0 && g < checks) g = checks;
            if (g > 0) {
                if (p.cu) {
                    quant_rows_varlen_kernel<T><<<(unsigned)g, threads, 0, st>>>(q);
                    log.add("quant_rows_varlen_kernel", dim3((unsigned)g), dim3(threads),
                            dim3(1, 1, 1), 0);
                } else {
                    quant_rows_kernel<T><<<(unsigned)g, threads, 0, st>>>(q);
                    log.add("quant_rows_kernel", dim3((unsigned)g), dim3(threads), dim3(1, 1, 1), 0);
                }
            }
            o0 += n;
        } while (o0 < outers && n > 0);
    } else if (p.cu) {
        const unsigned grid = (unsigned)((int64_t)p.H * p.groups);
        q.div_inner = FastDiv((uint32_t)(p.groups > 0 ? p.groups : 1));
        if (grid > 0) {
            const unsigned th = launch_blocks<T>(q, grid, st, true);
            log.add("quant_blocks_varlen_kernel", dim3(grid), dim3(th), dim3(1, 1, 1), 0);
        }
    } else {
        const int64_t ngroups = (p.S + p.block - 1) / p.block;
        const int64_t cta = (int64_t)p.B * p.H * ngroups;
        if (cta >= (1ll << 31)) return cudaErrorInvalidValue;  // 2^31 groups or more
        const unsigned grid = (unsigned)cta;
        q.div_inner = FastDiv((uint32_t)(ngroups > 0 ? ngroups : 1));
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
