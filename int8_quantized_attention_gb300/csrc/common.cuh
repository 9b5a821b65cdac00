// Device primitives shared by the sm_103a kernels: bounded mbarrier waits,
// bulk async copies, exact int8 -> f16 conversion, small math helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sage {

// Bits of the per-device error word (see sage_check_device_status).
constexpr int kErrTimeout = 1;
constexpr int kErrBadBlock = 2;

// ------------------------------------------------ variable-length batches
// Sequence b of a packed batch holds packed tokens [cu[b], cu[b+1]).  A
// range outside [0, total], running backwards or longer than the caller's
// bound max_len sets the bad-block bit of *err (when err is given) and is
// treated as an empty sequence.
// The same from the two offsets a = cu[b], e = cu[b+1] already loaded.
__device__ __forceinline__ int varlen_seq_of(int64_t a, int64_t e, int max_len, int64_t total,
                                             int *err, int64_t *start) {
    if (a < 0 || e < a || e > total || e - a > max_len) {
        if (err) atomicOr(err, kErrBadBlock);
        *start = 0;
        return 0;
    }
    *start = a;
    return (int)(e - a);
}

__device__ __forceinline__ int varlen_seq(const int32_t *cu, int b, int max_len, int64_t total,
                                          int *err, int64_t *start) {
    return varlen_seq_of(cu[b], cu[b + 1], max_len, total, err, start);
}

// First scale group of sequence b: per token (block 1) its first packed
// token; per block cu[b] / block + b, which leaves every sequence
// ceil(len / block) groups of its own (at most total / block + B in all).
__host__ __device__ __forceinline__ int64_t varlen_group0(int64_t cu_b, int b, int block) {
    return block == 1 ? cu_b : cu_b / block + b;
}

// First workspace row of sequence b's keys in the prefill's staged copy
// of a packed batch: its first packed key plus b * (bn + 4) rows, rounded up
// to a multiple of 4.  Each sequence's tiles of bn rows stay clear of the
// next sequence, the per-key scale rows stay 16-byte aligned, and all rows
// fit below total_k + B * (bn + 4).
__host__ __device__ __forceinline__ int64_t varlen_key_row0(int64_t cu_b, int b, int bn) {
    return (cu_b + (int64_t)b * (bn + 4) + 3) & ~(int64_t)3;
}

// The same answer found by a whole warp at once (every lane passes the
// same B and x): each step the 32 lanes test 32 evenly spaced candidates
// of the remaining range -- one round of independent loads -- and keep the
// stretch after the last one that passes, so B <= 32 takes one step and
// B <= 1024 two, where a bisection makes log2(B) dependent loads (each an
// L2 round trip once streaming data has pushed the offsets out of L1).
// For keys that are not non-decreasing it still returns some b in [0, B).
template <typename Key>
__device__ __forceinline__ int varlen_find_warp(int B, int64_t x, Key key) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int step = (hi - lo + 32) / 32;  // ceil((hi - lo + 1) / 32) >= 1
        const int c = lo + lane * step;
        const unsigned m = __ballot_sync(0xffffffffu, c <= hi && key(c) <= x);
        if (m == 0u) return lo;  // only at the first step: no key <= x, as the bisection
        const int nlo = lo + (31 - __clz(m)) * step;
        hi = min(hi, nlo + step - 1);
        lo = nlo;
    }
    return lo;
}

// Largest b in [0, B) whose key(b) <= x, by bisection (key non-decreasing
// for a valid packed batch; any input terminates).
template <typename Key>
__device__ __forceinline__ int varlen_bisect(int B, int64_t x, Key key) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (key(mid) <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Upper bound on any single wait inside a kernel (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA / bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete.  Gives up after kWaitLimitNs,
// sets the timeout bit of *err and returns false; never spins forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// ------------------------------------------------------- bulk async copies
// 1-D global -> shared copy completing on an mbarrier (transaction bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_evict_first(uint32_t dst, const void *src, uint32_t bytes,
                                                     uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ------------------------------------------------ exact int8 -> f16 / bf16
// For a signed byte b, (b ^ 0x80) = b + 128 =: u in [0, 255].  The f16 with
// bit pattern 0x6400 | u equals 1024 + u exactly, so subtracting 1152 gives
// b exactly (all integers below 2048 are f16-representable).
// Input: four int8 packed in a 32-bit word; output: two f16x2 words holding
// bytes (0,1) and (2,3).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    // __byte_perm: result byte k = byte (selector nibble k) of {u (0..3), 0x64646464 (4..7)}
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // halves: 0x64|u0, 0x64|u1
    uint32_t c = __byte_perm(u, 0x64646464u, 0x4342);  // halves: 0x64|u2, 0x64|u3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 l = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&c), bias);
    lo = *reinterpret_cast<uint32_t *>(&l);
    hi = *reinterpret_cast<uint32_t *>(&h);
}

// Symmetric INT8 code of v with scale s = fl32(amax / 127): one correctly
// rounded fp32 division, round to nearest even, clamped to [-127, 127]; an
// all-zero row (s == 0) gives code 0.  ("INT8 QK MMAC on gfx936 DCU",
// section 4: q = round(x / s), s = max|x| / 127.)
// Packed FP32 pair arithmetic (fma / mul / add .f32x2 on sm_100-family
// parts): one instruction updates two values, which halves the FP32 issue
// slots the softmax spends per score.  Same rounding as the scalar forms.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 u2f2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// three-input maximum (one instruction on sm_100-family parts)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Reciprocal of a group scale for quant_code (0 for s = 0).
__device__ __forceinline__ float quant_recip(float s) { return s != 0.0f ? __frcp_rn(s) : 0.0f; }

// rne(fl32(v / s)) clamped to [-127, 127], with r = quant_recip(s).  The
// correctly rounded quotient is only needed near a rounding boundary:
// y = fl32(v * r) differs from fl32(v / s) by at most 3 * 2^-24 * |v / s|,
// and |v / s| <= 127.00001 because |v| <= amax and s = fl32(amax / 127), so
// y is within 2.3e-5 of it.  When y lies farther than kTieBand from every
// k + 0.5, both round to the same integer; otherwise (and for a non-finite
// or out-of-range y) the division is taken.
constexpr float kTieBand = 3.0e-5f;
__device__ __forceinline__ int8_t quant_code(float v, float s, float r) {
    if (s == 0.0f) return 0;
    const float y = v * r;
    const float yr = rintf(y);
    int q;
    if (fabsf(y) < 128.0f && fabsf(y - yr) < 0.5f - kTieBand)
        q = (int)yr;
    else
        q = __float2int_rn(__fdiv_rn(v, s));
    q = max(-127, min(127, q));
    return static_cast<int8_t>(q);
}

// Three-input maximum that returns NaN when any input is NaN.
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Eight values at once, the same codes as quant_code, as two little-endian
// words of int8.  With |y| < 2^22, t = y + 1.5 * 2^23 holds rne(y) in the
// low bits of its mantissa, so the low byte of t's bits is the two's
// complement code itself and t - 1.5 * 2^23 is rne(y) as a float.  That
// shortcut is taken only when s is a normal float (then r = 1/s is finite
// and |y| <= 127.00002, so no code needs the clamp) or s = 0 (every y is
// 0), and every y lies farther than kTieBand from a rounding boundary.
// Otherwise the group is redone through quant_code: a subnormal s (a bf16
// group with amax below about 1.5e-36) can make r infinite -- y then is
// +-inf or NaN -- or, with its few significand bits, put |v / s| above
// 127.5, where the code is the clamp's 127.
__device__ __forceinline__ void quant8(const float (&v)[8], float s, float r, uint32_t &w0,
                                       uint32_t &w1) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    constexpr float kMinNormal = 1.17549435e-38f;
    uint32_t tb[8];
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 y = fmul2(make_float2(v[i], v[i + 1]), make_float2(r, r));
        const float2 t = fadd2(y, make_float2(kMagic, kMagic));
        const float2 yr = fadd2(t, make_float2(-kMagic, -kMagic));
        const float2 d = fadd2(y, make_float2(-yr.x, -yr.y));
        dmax = fmax3_nan(dmax, fabsf(d.x), fabsf(d.y));  // a NaN d makes dmax NaN
        tb[i] = __float_as_uint(t.x);
        tb[i + 1] = __float_as_uint(t.y);
    }
    // the comparison is false when dmax is NaN
    if (dmax < 0.5f - kTieBand && (s >= kMinNormal || s == 0.0f)) {
        w0 = __byte_perm(__byte_perm(tb[0], tb[1], 0x0040), __byte_perm(tb[2], tb[3], 0x0040), 0x5410);
        w1 = __byte_perm(__byte_perm(tb[4], tb[5], 0x0040), __byte_perm(tb[6], tb[7], 0x0040), 0x5410);
        return;
    }
    w0 = w1 = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) w0 |= (uint32_t)(uint8_t)quant_code(v[i], s, r) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) w1 |= (uint32_t)(uint8_t)quant_code(v[i + 4], s, r) << (8 * i);
}

// Same exact conversion, pairing bytes (0, 2) and (1, 3): for a register
// holding two 16-bit elements of two rows (a transposed ldmatrix of int8 data),
// `even` gets the low byte of each element and `odd` the high byte.
__device__ __forceinline__ void i8x4_to_f16x2_even_odd(uint32_t w, uint32_t &even, uint32_t &odd) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4240);  // halves: 0x64|u0, 0x64|u2
    uint32_t c = __byte_perm(u, 0x64646464u, 0x4341);  // halves: 0x64|u1, 0x64|u3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 l = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&c), bias);
    even = *reinterpret_cast<uint32_t *>(&l);
    odd = *reinterpret_cast<uint32_t *>(&h);
}

// bf16 variant: the fp32 with bits 0x4B000000 | u equals 2^23 + u exactly;
// subtracting 2^23 + 128 gives b exactly, and every |b| <= 128 is exact in
// bf16 (8 significand bits), so the final rounding is exact too.
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const float k = 8388736.0f;  // 2^23 + 128
    const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - k;
    const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - k;
    const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - k;
    const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - k;
    __nv_bfloat162 l = __floats2bfloat162_rn(f0, f1);
    __nv_bfloat162 h = __floats2bfloat162_rn(f2, f3);
    lo = *reinterpret_cast<uint32_t *>(&l);
    hi = *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
struct DT;
template <>
struct DT<__half> {
    static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
    static __device__ __forceinline__ float2 to_f2(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <>
struct DT<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ float2 to_f2(uint32_t w) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) {
        return __float2bfloat16_rn(x);
    }
};

}  // namespace sage
