// KV producer step: quantise new key/value rows per (token, KV head) and
// write them into the paged INT8 cache ("INT8 QK MMAC on gfx936 DCU",
// section 4: s = max|x| / 127, codes round(x / s); section 3: token t of
// sequence b sits in page block_table[b][t / 16], slot t % 16, channel c at
// [page][kv_head][c / 16][slot][c % 16], its scale at [page][kv_head][slot]).
//
// One warp per row (K rows, V rows and, in the producer form, the step's
// query rows in one launch): each lane loads D/32 consecutive channels (one
// 4-16 byte vector) -- issued first, so that the row's data and its page
// index (position, then block-table entry) travel at the same time -- the
// row's amax comes from a warp max-reduction, and each lane stores its codes
// as one vector into the 16-channel group of the page slot.  Query rows go
// to a dense [B, Hq, n, D] array with their scales ("INT8 QK MMAC on gfx936
// DCU", section 4: the query is quantised once, in the producer, and every
// split-K segment reuses the codes).  Pages outside [0, num_blocks) and
// positions outside the block table set the error word's bad-block bit and
// the row is skipped.
#include "common.cuh"
#include "internal.h"

namespace sage {

namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) kv_append_kernel(KvAppendParams p) {
    constexpr int CPL = D / 32;  // channels per lane: 2, 4 or 8
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t rows = (int64_t)p.B * p.H * p.n;
    const int64_t qrows = p.q ? (int64_t)p.B * p.Hq * p.n : 0;
    if (row >= 2 * rows + qrows) return;  // whole warp leaves together
    const bool is_q = row >= 2 * rows;
    const bool is_v = !is_q && row >= rows;
    const int64_t r = is_q ? row - 2 * rows : (is_v ? row - rows : row);
    const T *src = static_cast<const T *>(is_q ? p.q : (is_v ? p.v : p.k)) + r * D + lane * CPL;
    float f[CPL];
    if constexpr (CPL == 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(src);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 v = DT<T>::to_f2(w[e]);
            f[2 * e] = v.x, f[2 * e + 1] = v.y;
        }
    } else if constexpr (CPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        const float2 a = DT<T>::to_f2(u.x), c = DT<T>::to_f2(u.y);
        f[0] = a.x, f[1] = a.y, f[2] = c.x, f[3] = c.y;
    } else {
        const float2 a = DT<T>::to_f2(*reinterpret_cast<const uint32_t *>(src));
        f[0] = a.x, f[1] = a.y;
    }
    int64_t page = 0, slot = 0;
    if (!is_q) {
        // row r = (b * H + h) * n + t: divisions by invariant-divisor
        // constants (r < 2^31, checked on the host)
        const uint32_t bh = p.div_n.div((uint32_t)r);
        const uint32_t t = (uint32_t)r - bh * (uint32_t)p.n;
        const uint32_t b = p.div_h.div(bh);
        const uint32_t h = bh - b * (uint32_t)p.H;
        const int64_t pos = (int64_t)p.pos[b] + t;
        const int64_t pi = pos >> 4;
        int blk = -1;
        if (pos >= 0 && pi < p.max_blocks) blk = p.block_table[(int64_t)b * p.max_blocks + pi];
        if ((unsigned)blk >= (unsigned)p.num_blocks) {
            if (lane == 0) atomicOr(p.err, kErrBadBlock);
            return;
        }
        page = (int64_t)blk * p.H + h;
        slot = pos & 15;
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) amax = fmaxf(amax, fabsf(f[e]));
    amax = warp_max(amax);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = quant_recip(s);
    uint32_t w[2] = {0u, 0u};
    if constexpr (CPL == 8) {
        quant8(f, s, rs, w[0], w[1]);  // the same codes, eight at a time
    } else {
#pragma unroll
        for (int e = 0; e < CPL; ++e)
            w[e >> 2] |= (uint32_t)(uint8_t)quant_code(f[e], s, rs) << (8 * (e & 3));
    }
    const int c0 = lane * CPL;
    int8_t *dst;
    if (is_q) {
        dst = p.q_int8 + r * D + c0;
        if (lane == 0) p.q_scale[r] = s;
    } else {
        dst = (is_v ? p.v_cache : p.k_cache) + page * D * 16 + (c0 >> 4) * 256 + slot * 16 + (c0 & 15);
        if (lane == 0) (is_v ? p.v_scale : p.k_scale)[page * 16 + slot] = s;
    }
    if constexpr (CPL == 8)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    else if constexpr (CPL == 4)
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    else
        *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w[0];
}

template <typename T>
cudaError_t launch_t(const KvAppendParams &p, cudaStream_t st, LaunchLog &log) {
    const int64_t rows = 2 * (int64_t)p.B * p.H * p.n + (p.q ? (int64_t)p.B * p.Hq * p.n : 0);
    const int64_t grid = (rows + 7) / 8;
    if (grid == 0) return cudaSuccess;
    if (rows >= 0x7fffffff) return cudaErrorInvalidValue;  // row indices are 32-bit
    KvAppendParams q = p;
    q.div_n = FastDiv((uint32_t)p.n);
    q.div_h = FastDiv((uint32_t)p.H);
    switch (p.D) {
        case 64: kv_append_kernel<T, 64><<<(unsigned)grid, 256, 0, st>>>(q); break;
        case 128: kv_append_kernel<T, 128><<<(unsigned)grid, 256, 0, st>>>(q); break;
        case 256: kv_append_kernel<T, 256><<<(unsigned)grid, 256, 0, st>>>(q); break;
        default: return cudaErrorInvalidValue;
    }
    log.add(p.q ? "kv_producer_kernel" : "kv_append_kernel", dim3((unsigned)grid), dim3(256),
            dim3(1, 1, 1), 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendParams &p, cudaStream_t st, LaunchLog &log) {
    return p.bf16 ? launch_t<__nv_bfloat16>(p, st, log) : launch_t<__half>(p, st, log);
}

}  // namespace sage
