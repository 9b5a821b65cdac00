// Staging pass of the prefill: expands, once per call, the INT8 key codes
// (and the paged prefix's INT8 value codes, and bf16 chunk values) into an
// exact f16 copy in the caller's workspace, with one per-key scale array, so
// that the attention kernel's tiles arrive by TMA in the layout the tensor
// cores read and every query tile re-reads them from L2 without converting.
//
// Prefix values are stored as f16(code * v_scale) (one rounding, as the P.V
// operand); K codes stay exact.
// Workspace rows per (batch, kv head), in key order: [0, Ppad) the paged
// prefix (key r at row r; rows past the batch's prefix length are zero),
// [Ppad, Ppad + Sk) the contiguous chunk, then zero rows up to Lpad.  With
// smooth_v every staged value is f16(value - V mean of its channel), the
// chunk's f16 values included.  The
// INT8 -> f16 expansion is exact (|code| <= 127), so S = Q K^T computed on
// the copy equals the INT32 product of the codes ("INT8 QK MMAC on gfx936
// DCU", sections 2.1 and 5.2: the scores are exact integer dot products,
// rescaled afterwards by the per-token / per-block scales).
#include "common.cuh"
#include "internal.h"

namespace sage {

namespace {

__device__ __forceinline__ void store_f16x16(__half *dst, uint4 w) {
    uint4 h0, h1;
    i8x4_to_f16x4(w.x, h0.x, h0.y);
    i8x4_to_f16x4(w.y, h0.z, h0.w);
    i8x4_to_f16x4(w.z, h1.x, h1.y);
    i8x4_to_f16x4(w.w, h1.z, h1.w);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[0] = h0;
    d[1] = h1;
}

// 16 int8 codes times one scale -> 16 f16 (round to nearest, finite range)
__device__ __forceinline__ void store_f16x16_scaled(__half *dst, uint4 w, float sc) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int8_t *b = reinterpret_cast<const int8_t *>(&u[e]);
        const float f0 = fminf(fmaxf((float)b[0] * sc, -65504.0f), 65504.0f);
        const float f1 = fminf(fmaxf((float)b[1] * sc, -65504.0f), 65504.0f);
        const float f2 = fminf(fmaxf((float)b[2] * sc, -65504.0f), 65504.0f);
        const float f3 = fminf(fmaxf((float)b[3] * sc, -65504.0f), 65504.0f);
        __half2 lo = __floats2half2_rn(f0, f1), hi = __floats2half2_rn(f2, f3);
        h[2 * e] = *reinterpret_cast<uint32_t *>(&lo);
        h[2 * e + 1] = *reinterpret_cast<uint32_t *>(&hi);
    }
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 values minus the V mean of their channels -> f16 (round to nearest,
// saturating); mu points at the 16 channels' means
__device__ __forceinline__ void store_f16x16_minus(__half *dst, const float (&v)[16],
                                                   const float *mu) {
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float a = fminf(fmaxf(v[2 * e] - mu[2 * e], -65504.0f), 65504.0f);
        const float b = fminf(fmaxf(v[2 * e + 1] - mu[2 * e + 1], -65504.0f), 65504.0f);
        __half2 x = __floats2half2_rn(a, b);
        h[e] = *reinterpret_cast<uint32_t *>(&x);
    }
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 consecutive f16 or bf16 values as floats
__device__ __forceinline__ void load16f(const void *src, bool bf16, float (&v)[16]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    const uint4 w[2] = {s[0], s[1]};
    const uint32_t *u = reinterpret_cast<const uint32_t *>(w);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float2 f;
        if (bf16)
            f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u[e]));
        else
            f = __half22float2(*reinterpret_cast<const __half2 *>(&u[e]));
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

// 8 bf16 -> 8 f16, round to nearest, saturating to the finite f16 range
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x) {
    uint32_t *u = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u[e]));
        __half2 h = __floats2half2_rn(fminf(fmaxf(f.x, -65504.0f), 65504.0f),
                                      fminf(fmaxf(f.y, -65504.0f), 65504.0f));
        u[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return x;
}

// One thread per 16-channel piece of a key row; a block of 256 threads
// covers 256 / D groups of 16 rows.  Prefix groups read page slabs laid out
// [D/16][16 tokens][16 bytes] with the token index varying fastest across
// threads (256 contiguous bytes per 16 threads); chunk groups read rows with
// the channel piece varying fastest.
__global__ void __launch_bounds__(256) prefill_stage_kernel(const __grid_constant__ PrefillParams p) {
    // the attention kernel launched behind this pass may be scheduled once
    // every CTA has started; it waits on the device before reading the copy
    asm volatile("griddepcontrol.launch_dependents;");
    const int D = p.D;
    const int per_block = 256 / D;
    const int t = threadIdx.x % D;
    const int64_t g = (int64_t)blockIdx.x * per_block + threadIdx.x / D;
    const int gpb = p.Lpad >> 4;
    const int64_t BH = (int64_t)p.B * p.Hkv;
    if (g >= BH * gpb) return;
    const int bh = (int)(g / gpb);
    const int row0 = (int)(g % gpb) * 16;
    const int b = bh / p.Hkv, kvh = bh % p.Hkv;
    const int Vrows = p.Vrows;

    if (row0 < p.Ppad) {
        int P = p.prefix_lens[b];
        if (P < 0 || P > p.max_prefix_len) P = P < 0 ? 0 : p.max_prefix_len;
        const int slot = t & 15, dc = t >> 4;
        const int row = row0 + slot;
        uint4 wk = make_uint4(0, 0, 0, 0), wv = make_uint4(0, 0, 0, 0);
        float ks = 0.0f, vs = 0.0f;
        if (row < P) {
            const int blk = p.block_table[(int64_t)b * p.max_blocks + (row >> 4)];
            if ((unsigned)blk < (unsigned)p.num_blocks) {
                const int64_t pg = (int64_t)blk * p.Hkv + kvh;
                wk = *reinterpret_cast<const uint4 *>(p.k_cache + pg * D * 16 + dc * 256 + slot * 16);
                wv = *reinterpret_cast<const uint4 *>(p.v_cache + pg * D * 16 + dc * 256 + slot * 16);
                ks = p.k_cache_scale[pg * 16 + slot];
                vs = p.v_cache_scale[pg * 16 + slot];
            } else if (t == 0) {
                atomicOr(p.err, kErrBadBlock);
            }
        }
        store_f16x16(p.k_ws + ((int64_t)bh * p.Lpad + row) * D + dc * 16, wk);
        // prefix values: the per-token V scale is applied here, once, so the
        // attention kernel treats prefix and chunk values alike
        __half *vd = p.v_ws + ((int64_t)bh * Vrows + row) * D + dc * 16;
        if (p.v_mean && row < P) {
            const int8_t *c = reinterpret_cast<const int8_t *>(&wv);
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = (float)c[e] * vs;
            store_f16x16_minus(vd, v, p.v_mean + (int64_t)bh * D + dc * 16);
        } else {
            store_f16x16_scaled(vd, wv, vs);
        }
        if (dc == 0) p.ksc_ws[(int64_t)bh * p.Lpad + row] = ks;
    } else {
        const int np = D >> 4;
        const int slot = t / np, dc = t % np;
        const int row = row0 + slot;
        const int c = row - p.Ppad;
        const bool ok = c < p.Sk;
        uint4 wk = make_uint4(0, 0, 0, 0);
        float ks = 0.0f;
        if (ok) {
            wk = *reinterpret_cast<const uint4 *>(p.k + ((int64_t)bh * p.Sk + c) * D + dc * 16);
            ks = p.k_scale[(int64_t)bh * p.k_groups + (c >> p.k_shift)];
        }
        store_f16x16(p.k_ws + ((int64_t)bh * p.Lpad + row) * D + dc * 16, wk);
        if (dc == 0) p.ksc_ws[(int64_t)bh * p.Lpad + row] = ks;
        __half *vd = p.v_ws + ((int64_t)bh * Vrows + row) * D + dc * 16;
        // element (b, kv head, token c, channel) of the chunk's V (HND or NHD)
        const int64_t vo = (int64_t)(bh / p.Hkv) * p.v_sb + (int64_t)(bh % p.Hkv) * p.v_sh +
                           (int64_t)c * p.v_st + dc * 16;
        if (p.v_mean) {
            if (ok) {
                float v[16];
                load16f(static_cast<const char *>(p.v) + vo * 2, p.v_bf16 != 0, v);
                store_f16x16_minus(vd, v, p.v_mean + (int64_t)bh * D + dc * 16);
            } else {
                uint4 *d = reinterpret_cast<uint4 *>(vd);
                d[0] = d[1] = make_uint4(0, 0, 0, 0);
            }
        } else if (p.v_bf16) {
            uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
            if (ok) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const __nv_bfloat16 *>(p.v) + vo);
                v0 = bf16x8_to_f16x8(src[0]);
                v1 = bf16x8_to_f16x8(src[1]);
            }
            uint4 *d = reinterpret_cast<uint4 *>(vd);
            d[0] = v0;
            d[1] = v1;
        }
    }
}

// K codes alone with no paged prefix (f16 V read in place, no smooth_v):
// every workspace row is a chunk row, and each thread takes kStageG 16-row
// groups, the block's 256 / D groups apart, issuing all of their loads
// before the first conversion and store (46 registers, five CTAs per SM),
// and asks L2 for the key codes of the CTA half a wave of resident CTAs
// ahead (capping the registers for a sixth CTA per SM spilled and gained
// less).
// One group per thread left this pass latency-bound; the other forms keep
// it, because their registers (the paged prefix's table and page loads, or
// V as well) would cost more CTAs per SM than the batching gains.
constexpr int kStageG = 4;

__global__ void __launch_bounds__(256) prefill_stage_keys_kernel(const __grid_constant__ PrefillParams p,
                                                                 uint32_t ahead) {
    // the attention kernel launched behind this pass may be scheduled once
    // every CTA has started; it waits on the device before reading the copy
    asm volatile("griddepcontrol.launch_dependents;");
    const int D = p.D;
    const int per_block = 256 / D;
    const int np = D >> 4;
    const int t = threadIdx.x % D;
    const int slot = t / np, dc = t % np;
    const uint32_t gpb = (uint32_t)p.Lpad >> 4;   // 16-row groups per (b, kv head)
    const uint32_t groups = (uint32_t)(p.B * p.Hkv) * gpb;
    const uint32_t g0 = blockIdx.x * (uint32_t)(kStageG * per_block) + threadIdx.x / D;
    if (threadIdx.x == 0 && ahead > 0) {
        // the key codes of the CTA `ahead` CTAs on (within its first
        // (b, kv head)) into L2, so that its loads at its start hit L2
        const uint32_t x = blockIdx.x + ahead;
        const uint32_t gx = x * (uint32_t)(kStageG * per_block);
        if (x < gridDim.x && gx < groups) {
            const uint32_t bh = gx / gpb;
            const int c0 = (int)(gx % gpb) * 16;
            const int c1 = min(c0 + kStageG * 256 / (D >> 4), p.Sk);
            if (c1 > c0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 p.k + ((int64_t)bh * p.Sk + c0) * D),
                             "r"((uint32_t)((c1 - c0) * D))
                             : "memory");
        }
    }
    uint4 wk[kStageG];
    float ks[kStageG];
#pragma unroll
    for (int u = 0; u < kStageG; ++u) {
        wk[u] = make_uint4(0, 0, 0, 0);
        ks[u] = 0.0f;
        const uint32_t g = g0 + u * per_block;
        if (g >= groups) continue;
        const int bh = (int)(g / gpb);
        const int c = (int)(g % gpb) * 16 + slot;   // key row = token of the chunk
        if (c >= p.Sk) continue;
        wk[u] = *reinterpret_cast<const uint4 *>(p.k + ((int64_t)bh * p.Sk + c) * D + dc * 16);
        ks[u] = p.k_scale[(int64_t)bh * p.k_groups + (c >> p.k_shift)];
    }
#pragma unroll
    for (int u = 0; u < kStageG; ++u) {
        const uint32_t g = g0 + u * per_block;
        if (g >= groups) break;
        const int64_t row = (int64_t)(g / gpb) * p.Lpad + (g % gpb) * 16 + slot;
        store_f16x16(p.k_ws + row * D + dc * 16, wk[u]);
        if (dc == 0) p.ksc_ws[row] = ks[u];
    }
}

// Packed variable-length batch: sequence b's keys go to workspace rows
// [r0, r0 + ceil(len / BN) * BN) of each KV head, r0 = varlen_key_row0(),
// with zero rows after its last key up to the tile boundary.  K codes ->
// exact f16, V (f16 copied, bf16 rounded) -> f16, one K scale per key.  One
// thread per 16-channel piece, the piece varying fastest along a row.
__global__ void __launch_bounds__(256)
    prefill_stage_varlen_kernel(const __grid_constant__ PrefillParams p, uint32_t nslot) {
    // the attention kernel launched behind this pass may be scheduled once
    // every CTA has started; it waits on the device before reading the copy
    asm volatile("griddepcontrol.launch_dependents;");
    const int D = p.D;
    const int per_block = 256 / D;
    const int t = threadIdx.x % D;
    // compact 16-row group slots per kv head: sequence b owns the slots from
    // cu_k[b] / 16 + b * (BN / 16 + 1) on, at least ceil(len_b / BN) * BN / 16
    // of them (a grid of B x the longest sequence's groups left most CTAs
    // empty).  A warp lies inside one group (D >= 64 threads per group), so
    // its lanes find the group's sequence together.
    const uint32_t g = blockIdx.x * (uint32_t)per_block + threadIdx.x / D;
    if (g >= (uint32_t)p.Hkv * nslot) return;
    const int kvh = (int)(g / nslot);
    const int64_t gs = g - (uint32_t)kvh * nslot;   // the group's slot
    const int spare = p.BN / 16 + 1;
    const int b = varlen_find_warp(p.B, gs, [&](int k) {
        const int c = p.cu_k[k];
        return (int64_t)(c < 0 ? 0 : c) / 16 + (int64_t)k * spare;
    });
    int64_t ks = 0;
    const int len = varlen_seq(p.cu_k, b, p.Sk, p.total_k, nullptr, &ks);
    const int64_t j = gs - (ks / 16 + (int64_t)b * spare);
    if (len == 0 || j < 0 || j * 16 >= (len + p.BN - 1) / p.BN * p.BN) return;
    const int row0 = (int)j * 16;
    const int np = D >> 4;
    const int slot = t / np, dc = t % np;
    const int row = row0 + slot;
    const bool ok = row < len;
    const int64_t wrow = (int64_t)kvh * p.Lpad + varlen_key_row0(ks, b, p.BN) + row;
    uint4 wk = make_uint4(0, 0, 0, 0);
    uint4 vv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    float ksc = 0.0f;
    if (ok) {
        wk = *reinterpret_cast<const uint4 *>(p.k + ((int64_t)kvh * p.total_k + ks + row) * D +
                                              dc * 16);
        ksc = p.k_scale[(int64_t)kvh * p.k_groups + varlen_group0(ks, b, 1 << p.k_shift) +
                        (row >> p.k_shift)];
        const int64_t vo = (ks + row) * p.v_st + kvh * p.v_sh + dc * 16;
        if (p.v_mean) {
            float v[16];
            load16f(static_cast<const char *>(p.v) + vo * 2, p.v_bf16 != 0, v);
            store_f16x16_minus(reinterpret_cast<__half *>(vv), v,
                               p.v_mean + ((int64_t)b * p.Hkv + kvh) * D + dc * 16);
        } else if (p.v_bf16) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(p.v) + vo);
            vv[0] = bf16x8_to_f16x8(src[0]);
            vv[1] = bf16x8_to_f16x8(src[1]);
        } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __half *>(p.v) + vo);
            vv[0] = src[0];
            vv[1] = src[1];
        }
    }
    store_f16x16(p.k_ws + wrow * D + dc * 16, wk);
    if (dc == 0) p.ksc_ws[wrow] = ksc;
    uint4 *d = reinterpret_cast<uint4 *>(p.v_ws + wrow * D + dc * 16);
    d[0] = vv[0];
    d[1] = vv[1];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

PrefillLayout prefill_layout(int B, int Hkv, int Sk, int D, int max_prefix_len, bool v_bf16,
                             bool smooth_v, const PrefillSplit &split) {
    PrefillLayout L = {};
    L.BN = D == 256 ? 64 : 128;
    L.Ppad = (max_prefix_len + L.BN - 1) / L.BN * L.BN;
    L.Lpad = L.Ppad + (Sk + L.BN - 1) / L.BN * L.BN;
    L.Vrows = (v_bf16 || smooth_v) ? L.Lpad : L.Ppad;
    const size_t BH = (size_t)B * Hkv;
    L.off_k = 0;
    L.off_v = align256(L.off_k + BH * L.Lpad * D * 2);
    L.off_ksc = align256(L.off_v + BH * L.Vrows * D * 2);
    L.off_vmean = align256(L.off_ksc + BH * L.Lpad * 4);
    const size_t slots = split.parts > 0 ? (size_t)split.tail * split.parts : 0;
    L.off_part_o = align256(L.off_vmean + (smooth_v ? BH * D * 4 : 0));
    L.off_part_lse = align256(L.off_part_o + slots * 128 * D * 4);
    L.bytes = align256(L.off_part_lse + slots * 128 * 4);
    return L;
}

PrefillLayout prefill_layout_varlen(int B, int Hkv, int64_t total_k, int D, bool smooth_v) {
    PrefillLayout L = {};
    L.BN = D == 256 ? 64 : 128;
    L.Ppad = 0;
    const int64_t rows = (total_k + (int64_t)B * (L.BN + 4) + 15) / 16 * 16;
    L.Lpad = (int)rows;
    L.Vrows = L.Lpad;
    const size_t H = (size_t)Hkv;
    L.off_k = 0;
    L.off_v = align256(L.off_k + H * rows * D * 2);
    L.off_ksc = align256(L.off_v + H * rows * D * 2);
    L.off_vmean = align256(L.off_ksc + H * rows * 4);
    L.off_part_o = L.off_part_lse = L.bytes =
        align256(L.off_vmean + (smooth_v ? (size_t)B * Hkv * D * 4 : 0));
    return L;
}

cudaError_t launch_prefill_stage(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    if (p.cu_q) {
        // group slots per kv head: total_k / 16, plus BN / 16 + 1 per sequence
        const int64_t nslot = p.total_k / 16 + (int64_t)p.B * (p.BN / 16 + 1);
        const int64_t groups = (int64_t)p.Hkv * nslot;
        const int per_block = 256 / p.D;
        const int64_t blocks = (groups + per_block - 1) / per_block;
        if (blocks == 0) return cudaSuccess;
        if (groups > 0x7fffffff) return cudaErrorInvalidValue;
        prefill_stage_varlen_kernel<<<(unsigned)blocks, 256, 0, st>>>(p, (uint32_t)nslot);
        log.add("prefill_stage_varlen_kernel", dim3((unsigned)blocks), dim3(256), dim3(1, 1, 1), 0);
        return cudaGetLastError();
    }
    const int64_t groups = (int64_t)p.B * p.Hkv * (p.Lpad >> 4);
    const int per_block = 256 / p.D;
    if (p.Ppad == 0 && !p.v_mean && !p.v_bf16) {
        // group indices are 32-bit there (2^31 groups of 16 f16 rows would
        // exceed any device's memory many times over)
        if (groups > 0x7fffffff) return cudaErrorInvalidValue;
        const int64_t blocks = (groups + kStageG * per_block - 1) / (kStageG * per_block);
        if (blocks == 0) return cudaSuccess;
        // prefetch distance: half the CTAs resident at once
        int dev = 0, sms = 0, per_sm = 0;
        uint32_t ahead = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_stage_keys_kernel, 256, 0) ==
                cudaSuccess)
            ahead = (uint32_t)(sms * per_sm / 2);
        else
            cudaGetLastError();
        prefill_stage_keys_kernel<<<(unsigned)blocks, 256, 0, st>>>(p, ahead);
        log.add("prefill_stage_keys_kernel", dim3((unsigned)blocks), dim3(256), dim3(1, 1, 1), 0);
        return cudaGetLastError();
    }
    const int64_t blocks = (groups + per_block - 1) / per_block;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    prefill_stage_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
    log.add("prefill_stage_kernel", dim3((unsigned)blocks), dim3(256), dim3(1, 1, 1), 0);
    return cudaGetLastError();
}

}  // namespace sage
