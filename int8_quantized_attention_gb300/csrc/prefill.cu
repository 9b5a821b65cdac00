// INT8-QK prefill attention on the 5th-generation tensor cores (tcgen05).
//
// What it computes (SageAttention MXMACA README: attention kernel pipeline,
// feature matrix; "INT8 QK MMAC on gfx936 DCU", sections 1, 2.1, 3, 5.2):
//   S = Q_int8 K_int8^T exactly, each score rescaled by
//   q_scale[row] * k_scale[col] * sm_scale * log2(e) (+ the smooth_k row bias
//   on smoothed keys) before a base-2 online softmax; P.V in f16 with FP32
//   accumulation (bf16 V is rounded to f16 in shared memory first, as the
//   README's port converts bf16 V to f16 before its kernel); O / l and LSE
//   in the epilogue.  Keys come from an
//   optional paged INT8 prefix followed by the contiguous chunk.
//
// GB300 design.  sm_103a has no integer tcgen05 MMA, so QK^T runs on
// kind::f16 with the INT8 codes converted EXACTLY to f16 (|q|,|k| <= 127;
// every partial sum of D <= 256 products is an integer below 2^24, which
// the FP32 accumulator holds exactly).  One CTA owns 128 query rows of one
// (batch, head); keys stream in tiles of BN (128, or 64 at D = 256).
//   warps 0-3  softmax: one thread per query row (TMEM lane); tcgen05.ld of
//              the S row, per-column K-scale recovery in registers, online
//              softmax with lazy rescaling (O is rescaled only when the row
//              max grows by more than 2^8), P written back over S in TMEM.
//   warps 4-7  converters: Q int8 -> f16 straight into TMEM (once); per tile
//              K int8 -> f16 into the 128-byte-swizzled shared layout the MMA
//              reads, INT8 prefix V -> 16-bit likewise, column scales.
//   warp 8     producer: 1-D bulk copies of raw INT8 K (and paged V) tiles,
//              TMA tensor loads of 16-bit chunk V straight into the swizzled
//              layout (out-of-range rows zero-filled).
//   warp 9     TMEM owner and MMA issuer (one thread): S = Q K^T with Q from
//              TMEM, then O += P V with P from TMEM; completion through
//              tcgen05.commit on mbarriers.  S is double-buffered so the next
//              QK^T overlaps the current softmax.
// Tensor memory (512 columns): O [0, D), S0/S1 [D, D+2BN), Q [D+2BN, +D/2).
// Every mbarrier wait is bounded; a timeout raises a CTA-wide abort flag
// that makes every other wait give up at once, in-flight copies and MMAs
// are drained (bounded), TMEM is freed and the error word is set.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace sage {

namespace {

constexpr int kThreads = 320;
constexpr int kLaneTmemWarps = 4;

template <int D>
struct PCfg {
    static constexpr int BN = D == 256 ? 64 : 128;
    static constexpr int KF = BN * D * 2;   // f16 K tile, swizzled
    static constexpr int VF = BN * D * 2;   // 16-bit V tile, swizzled
    static constexpr int KR = BN * D;       // raw int8 K tile
    static constexpr int VR = BN * D;       // raw int8 V tile (paged prefix)
    static constexpr int SR = BN * 4;       // raw per-token scales of the tile's pages
    static constexpr int OFF_KF = 0;
    static constexpr int OFF_VF = OFF_KF + 2 * KF;
    static constexpr int OFF_KR = OFF_VF + 2 * VF;
    static constexpr int OFF_VR = OFF_KR + 2 * KR;
    static constexpr int OFF_KSR = OFF_VR + 2 * VR;
    static constexpr int OFF_VSR = OFF_KSR + 2 * SR;
    static constexpr int OFF_KSC = OFF_VSR + 2 * SR;
    static constexpr int OFF_VSC = OFF_KSC + 2 * BN * 4;
    static constexpr int OFF_BAR = OFF_VSC + 2 * BN * 4;
    static constexpr int NBAR = 16;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int USED = OFF_MISC + 64;
    // at least ~120 KB so that a single CTA (which owns all 512 TMEM
    // columns) is resident per SM
    static constexpr int SMEM = (USED + 1024 > 122880 ? USED + 1024 : 122880);
    static constexpr uint32_t COL_O = 0, COL_S = D, COL_Q = D + 2 * BN;
};

// barrier slots
enum {
    B_RAW_FULL = 0,   // [2] producer: raw int8 K (+ paged V, scales) landed
    B_V_FULL = 2,     // [2] producer: 16-bit V tile landed (or prefix: nothing to wait for)
    B_KV_FULL = 4,    // [2] converters: f16 K (+ prefix V) and column scales ready
    B_RAW_EMPTY = 6,  // [2] converters: raw stage may be refilled
    B_KV_EMPTY = 8,   // [2] MMA: P.V of the tile done (K/V buffers free, O updated)
    B_S_FULL = 10,    // [2] MMA: S = Q K^T done
    B_P_FULL = 12,    // [2] softmax: P written to TMEM (and O rescaled)
    B_Q_READY = 14,   // converters: Q in TMEM
    B_DRAIN = 15      // MMA: every issued MMA retired
};

struct Tile {
    int pre;   // from the paged prefix
    int key0;  // first key within its source
    int n;     // valid keys
    int kg0;   // first key's index over prefix + chunk
};

__device__ __forceinline__ Tile tile_at(int j, int n_pre, int P, int Sk, int BN) {
    Tile t;
    if (j < n_pre) {
        t.pre = 1;
        t.key0 = j * BN;
        t.n = min(BN, P - t.key0);
        t.kg0 = t.key0;
    } else {
        t.pre = 0;
        t.key0 = (j - n_pre) * BN;
        t.n = min(BN, Sk - t.key0);
        t.kg0 = P + t.key0;
    }
    return t;
}

// Bounded wait that also gives up as soon as another role raised `abort`.
__device__ __forceinline__ bool wait_ab(uint32_t bar, uint32_t parity, int *err,
                                        volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 16 int8 channels [16*dc, 16*dc+16) of key r -> exact f16, stored as the
// two 16-byte chunks 2*dc, 2*dc+1 of row r in a 128-byte-swizzled tile
// (64-channel atom columns BN*128 bytes apart, chunk c of row r at c ^ (r%8)).
template <int BN>
__device__ __forceinline__ void store_piece(uint8_t *tile, int r, int dc, uint4 w) {
    uint4 h0, h1;
    i8x4_to_f16x4(w.x, h0.x, h0.y);
    i8x4_to_f16x4(w.y, h0.z, h0.w);
    i8x4_to_f16x4(w.z, h1.x, h1.y);
    i8x4_to_f16x4(w.w, h1.z, h1.w);
    const int c8 = 2 * dc;
    uint8_t *row = tile + (c8 >> 3) * (BN * 128) + (r >> 3) * 1024 + (r & 7) * 128;
    *reinterpret_cast<uint4 *>(row + (((c8 & 7) ^ (r & 7)) << 4)) = h0;
    *reinterpret_cast<uint4 *>(row + ((((c8 + 1) & 7) ^ (r & 7)) << 4)) = h1;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p,
                   const __grid_constant__ CUtensorMap tmap_v) {
    using C = PCfg<D>;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sm_a = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);
    float *ksc_all = reinterpret_cast<float *>(sm + C::OFF_KSC);
    float *vsc_all = reinterpret_cast<float *>(sm + C::OFF_VSC);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqt = (p.Sq + 127) >> 7;
    const int qt = nqt - 1 - (int)blockIdx.x;  // heaviest (causal) tiles first
    const int hq = blockIdx.y, b = blockIdx.z;
    const int kvh = hq / p.group;
    const int i0 = qt * 128;

    // ------------------------------------------------------ tile schedule
    int P = 0;
    if (p.prefix_lens) {
        P = p.prefix_lens[b];
        if (P < 0 || P > p.max_prefix_len) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
            P = P < 0 ? 0 : p.max_prefix_len;
        }
    }
    const int off = P + p.Sk - p.Sq;  // key j visible to row i iff j <= i + off (causal)
    const int row_last = min(i0 + 127, p.Sq - 1);
    const int kmax = p.causal ? row_last + off : P + p.Sk - 1;
    int n_pre = 0, n_ch = 0;
    if (kmax >= 0) {
        n_pre = min((P + BN - 1) / BN, kmax / BN + 1);
        if (kmax >= P) n_ch = min((p.Sk + BN - 1) / BN, (kmax - P) / BN + 1);
    }
    const int T = n_pre + n_ch;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_RAW_FULL + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_KV_FULL + s), 128);
            mbar_init(bar(B_RAW_EMPTY + s), 128);
            mbar_init(bar(B_KV_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 128);
        }
        mbar_init(bar(B_Q_READY), 128);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tc::alloc(smem_u32(tmem_slot), 512);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ============================================================ producer
        if (lane == 0) {
            if (n_ch > 0) tc::prefetch_tmap(&tmap_v);
            const int32_t *bt = p.block_table ? p.block_table + (int64_t)b * p.max_blocks : nullptr;
            const int8_t *kchunk = p.k ? p.k + (int64_t)(b * p.Hkv + kvh) * p.Sk * D : nullptr;
            int raw_issued = 0, v_issued = 0;
            for (int j = 0; j < T; ++j) {
                const int buf = j & 1;
                const uint32_t prev = (uint32_t)((j >> 1) - 1) & 1u;
                const Tile t = tile_at(j, n_pre, P, p.Sk, BN);
                if (j >= 2 && !wait_ab(bar(B_RAW_EMPTY + buf), prev, p.err, abort_flag)) break;
                uint8_t *kr = sm + C::OFF_KR + buf * C::KR;
                if (t.pre) {
                    const int npg = (t.n + 15) >> 4;
                    mbar_arrive_expect_tx(bar(B_RAW_FULL + buf), npg * (2 * D * 16 + 128));
                    for (int q = 0; q < npg; ++q) {
                        int blk = bt[(t.key0 >> 4) + q];
                        if ((unsigned)blk >= (unsigned)p.num_blocks) {
                            atomicOr(p.err, kErrBadBlock);
                            blk = 0;
                        }
                        const int64_t pg = (int64_t)blk * p.Hkv + kvh;
                        bulk_g2s(smem_u32(kr + q * D * 16), p.k_cache + pg * D * 16, D * 16,
                                 bar(B_RAW_FULL + buf));
                        bulk_g2s(smem_u32(sm + C::OFF_VR + buf * C::VR + q * D * 16),
                                 p.v_cache + pg * D * 16, D * 16, bar(B_RAW_FULL + buf));
                        bulk_g2s(smem_u32(sm + C::OFF_KSR + buf * C::SR + q * 64),
                                 p.k_cache_scale + pg * 16, 64, bar(B_RAW_FULL + buf));
                        bulk_g2s(smem_u32(sm + C::OFF_VSR + buf * C::SR + q * 64),
                                 p.v_cache_scale + pg * 16, 64, bar(B_RAW_FULL + buf));
                    }
                } else {
                    mbar_arrive_expect_tx(bar(B_RAW_FULL + buf), t.n * D);
                    bulk_g2s(smem_u32(kr), kchunk + (int64_t)t.key0 * D, t.n * D,
                             bar(B_RAW_FULL + buf));
                }
                ++raw_issued;
                if (j >= 2 && !wait_ab(bar(B_KV_EMPTY + buf), prev, p.err, abort_flag)) break;
                if (t.pre) {
                    mbar_arrive(bar(B_V_FULL + buf));
                } else {
                    mbar_arrive_expect_tx(bar(B_V_FULL + buf), BN * D * 2);
                    for (int a = 0; a < D / 64; ++a)
                        tc::tma_load_3d(sm_a + C::OFF_VF + buf * C::VF + a * BN * 128, &tmap_v,
                                        a * 64, t.key0, b * p.Hkv + kvh, bar(B_V_FULL + buf));
                }
                ++v_issued;
            }
            // never retire with copies in flight
            for (int j = max(0, raw_issued - 2); j < raw_issued; ++j)
                mbar_wait(bar(B_RAW_FULL + (j & 1)), (uint32_t)(j >> 1) & 1u, p.err);
            for (int j = max(0, v_issued - 2); j < v_issued; ++j)
                mbar_wait(bar(B_V_FULL + (j & 1)), (uint32_t)(j >> 1) & 1u, p.err);
        }
    } else if (warp == 9) {
        // ============================================================ MMA issuer
        if (lane == 0 && T > 0) {
            const uint32_t idq = tc::idesc_f16(128, BN, false, false);
            const uint32_t idp = tc::idesc_f16(128, D, false, true);  // P.V always in f16
            auto issue_qk = [&](int j) -> bool {
                const int buf = j & 1;
                if (!wait_ab(bar(B_KV_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag))
                    return false;
                tc::fence_after();
                const uint32_t kf = sm_a + C::OFF_KF + buf * C::KF;
                const uint32_t s_t = tmem + C::COL_S + buf * BN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t bd =
                        tc::sdesc_sw128(kf + (ks >> 2) * (BN * 128) + (ks & 3) * 32, 16, 1024);
                    tc::mma_ts(s_t, tmem + C::COL_Q + ks * 8, bd, idq, ks > 0 ? 1u : 0u);
                }
                tc::commit(bar(B_S_FULL + buf));
                return true;
            };
            bool ok = wait_ab(bar(B_Q_READY), 0, p.err, abort_flag);
            if (ok) {
                tc::fence_after();
                ok = issue_qk(0);
            }
            for (int j = 0; ok && j < T; ++j) {
                const int buf = j & 1;
                if (j + 1 < T && !issue_qk(j + 1)) break;
                if (!wait_ab(bar(B_P_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag)) break;
                if (!wait_ab(bar(B_V_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag)) break;
                tc::fence_after();
                const uint32_t vf = sm_a + C::OFF_VF + buf * C::VF;
                const uint32_t p_t = tmem + C::COL_S + buf * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bd = tc::sdesc_sw128(vf + kk * 2048, BN * 128, 1024);
                    tc::mma_ts(tmem + C::COL_O, p_t + kk * 8, bd, idp, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(bar(B_KV_EMPTY + buf));
            }
            tc::commit(bar(B_DRAIN));
            mbar_wait(bar(B_DRAIN), 0, p.err);  // every issued MMA has retired
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============================================================ converters
        const int ct = threadIdx.x - 128;  // 0..127 = TMEM lane of the Q row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        {
            const int i = i0 + ct;
            const int8_t *qrow = p.q + (((int64_t)b * p.Hq + hq) * p.Sq + i) * D;
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t v[32];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (i < p.Sq) w = *reinterpret_cast<const uint4 *>(qrow + c * 64 + u * 16);
                    i8x4_to_f16x4(w.x, v[u * 8 + 0], v[u * 8 + 1]);
                    i8x4_to_f16x4(w.y, v[u * 8 + 2], v[u * 8 + 3]);
                    i8x4_to_f16x4(w.z, v[u * 8 + 4], v[u * 8 + 5]);
                    i8x4_to_f16x4(w.w, v[u * 8 + 6], v[u * 8 + 7]);
                }
                tc::st32(tmem + lane_base + C::COL_Q + c * 32, v);
            }
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bar(B_Q_READY));
        }
        for (int j = 0; j < T; ++j) {
            const int buf = j & 1;
            const Tile t = tile_at(j, n_pre, P, p.Sk, BN);
            bool ok = true;
            if (j >= 2)
                ok = wait_ab(bar(B_KV_EMPTY + buf), (uint32_t)((j >> 1) - 1) & 1u, p.err, abort_flag);
            ok = ok && wait_ab(bar(B_RAW_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint8_t *kr = sm + C::OFF_KR + buf * C::KR;
            uint8_t *kf = sm + C::OFF_KF + buf * C::KF;
            // 16-byte pieces (16 channels of one key) -> two swizzled f16
            // chunks.  Contiguous rows: channel pieces vary fastest across
            // threads; page slabs ([D/16][16 keys][16]): keys vary fastest.
            // Both mappings keep the shared-memory reads conflict-free.
            constexpr int PIECES = BN * D / 16;
            if (t.pre) {
                const uint8_t *vr = sm + C::OFF_VR + buf * C::VR;
                uint8_t *vf = sm + C::OFF_VF + buf * C::VF;
#pragma unroll 4
                for (int it = ct; it < PIECES; it += 128) {
                    const int r = it % BN, dc = it / BN;
                    const int src = (r >> 4) * (D * 16) + dc * 256 + (r & 15) * 16;
                    uint4 wk = make_uint4(0, 0, 0, 0), wv = make_uint4(0, 0, 0, 0);
                    if (r < t.n) {
                        wk = *reinterpret_cast<const uint4 *>(kr + src);
                        wv = *reinterpret_cast<const uint4 *>(vr + src);
                    }
                    store_piece<BN>(kf, r, dc, wk);
                    store_piece<BN>(vf, r, dc, wv);
                }
            } else {
#pragma unroll 4
                for (int it = ct; it < PIECES; it += 128) {
                    const int r = it / (D / 16), dc = it % (D / 16);
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (r < t.n) w = *reinterpret_cast<const uint4 *>(kr + r * D + dc * 16);
                    store_piece<BN>(kf, r, dc, w);
                }
            }
            if (!t.pre && p.v_bf16) {
                // bf16 chunk V landed by TMA: round it to f16 in place (same
                // swizzled position), finite-saturating, so P.V runs in f16
                const bool w = wait_ab(bar(B_V_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag);
                if (!__all_sync(0xffffffffu, w)) break;
                uint4 *vf = reinterpret_cast<uint4 *>(sm + C::OFF_VF + buf * C::VF);
#pragma unroll 4
                for (int it = ct; it < BN * D / 8; it += 128) {
                    uint4 x = vf[it];
                    uint32_t *u = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u[e]));
                        __half2 h = __floats2half2_rn(fminf(fmaxf(f.x, -65504.0f), 65504.0f),
                                                      fminf(fmaxf(f.y, -65504.0f), 65504.0f));
                        u[e] = *reinterpret_cast<uint32_t *>(&h);
                    }
                    vf[it] = x;
                }
            }
            if (ct < BN) {
                float ks = 0.0f, vs = 1.0f;
                if (ct < t.n) {
                    if (t.pre) {
                        ks = reinterpret_cast<const float *>(sm + C::OFF_KSR + buf * C::SR)[ct];
                        vs = reinterpret_cast<const float *>(sm + C::OFF_VSR + buf * C::SR)[ct];
                    } else {
                        ks = p.k_scale[(int64_t)(b * p.Hkv + kvh) * p.k_groups +
                                       ((t.key0 + ct) >> p.k_shift)];
                    }
                }
                ksc_all[buf * BN + ct] = ks;
                vsc_all[buf * BN + ct] = vs;
            }
            tc::fence_proxy_async();  // st.shared -> visible to the tensor core
            mbar_arrive(bar(B_RAW_EMPTY + buf));
            mbar_arrive(bar(B_KV_FULL + buf));
        }
    } else {
        // ============================================================ softmax
        const int r = threadIdx.x;  // query row within the tile = TMEM lane
        const int i = i0 + r;
        const bool row_ok = i < p.Sq;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        // kept strictly positive so that a masked (-inf) score stays -inf; an
        // all-zero Q row (scale 0) then scores ~1e-30 * acc = 0 as it should
        const float rq = fmaxf(row_ok ? p.q_scale[((int64_t)b * p.Hq + hq) * p.q_groups +
                                                  (i >> p.q_shift)] * p.qk_scale_log2
                                      : 0.0f,
                               1e-30f);
        const float bc =
            (row_ok && p.q_bias) ? p.q_bias[((int64_t)b * p.Hq + hq) * p.Sq + i] * p.qk_scale_log2
                                 : 0.0f;
        const int lim = i + off;
        float m_run = -INFINITY, l = 0.0f;
        int done = 0;
        for (int j = 0; j < T; ++j) {
            const int buf = j & 1;
            const Tile t = tile_at(j, n_pre, P, p.Sk, BN);
            bool ok = wait_ab(bar(B_S_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag);
            ok = ok && wait_ab(bar(B_KV_FULL + buf), (uint32_t)(j >> 1) & 1u, p.err, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after();
            const uint32_t s_t = tmem + lane_base + C::COL_S + buf * BN;
            const float *ksc = ksc_all + buf * BN;
            const float *vsc = vsc_all + buf * BN;
            const bool masked = (t.n < BN) || (p.causal && (t.kg0 + BN - 1 > i0 + off));
            // ---- pass 1: row max of the scaled scores (S stays in TMEM)
            float mx = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rr[32];
                tc::ld32(s_t + c * 32, rr);
                tc::wait_ld();
                if (p.dbg && row_ok) {
                    int32_t *dr = p.dbg + (((int64_t)b * p.Hq + hq) * p.Sq + i) * p.dbg_stride;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int cc = c * 32 + e, kg = t.kg0 + cc;
                        if (cc < t.n && (!p.causal || kg <= lim))
                            dr[kg] = __float2int_rn(__uint_as_float(rr[e]));
                    }
                }
                if (masked) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int cc = c * 32 + e;
                        const float u = (cc >= t.n || (p.causal && t.kg0 + cc > lim))
                                            ? -INFINITY
                                            : __uint_as_float(rr[e]) * ksc[cc];
                        mx = fmaxf(mx, u);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(rr[e]) * ksc[c * 32 + e]);
                }
            }
            const float tb = t.pre ? 0.0f : bc;
            const float tmax = fmaf(mx, rq, tb);  // -inf when every key is masked (rq > 0)
            const float cand = fmaxf(m_run, tmax);
            const bool move = cand != -INFINITY && (m_run == -INFINITY || cand > m_run + 8.0f);
            float alpha = 1.0f;
            if (move) {
                alpha = m_run == -INFINITY ? 0.0f : exp2f(m_run - cand);
                l *= alpha;
                m_run = cand;
            }
            const bool fix = move && j > 0 && alpha != 1.0f;
            if (__any_sync(0xffffffffu, fix)) {
                // O holds P.V of earlier tiles scaled to the old max: wait for
                // the last P.V to land, then rescale this warp's rows in TMEM
                const bool w = wait_ab(bar(B_KV_EMPTY + ((j - 1) & 1)),
                                       (uint32_t)((j - 1) >> 1) & 1u, p.err, abort_flag);
                if (!__all_sync(0xffffffffu, w)) break;
                tc::fence_after();
                const float f = fix ? alpha : 1.0f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tc::ld32(tmem + lane_base + C::COL_O + c * 32, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tc::st32(tmem + lane_base + C::COL_O + c * 32, o);
                }
                tc::wait_st();
            }
            const float nb = tb - (m_run == -INFINITY ? 0.0f : m_run);
            // ---- pass 2: P = 2^(s*ksc*rq + tb - m) in 32-key chunks; the 16
            // packed f16x2 words of chunk c overwrite S columns [16c, 16c+16),
            // which were read in this pass already
            float lsum = 0.0f;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rr[32];
                tc::ld32(s_t + c * 32, rr);
                tc::wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c0 = c * 32 + 2 * e;
                    float u0 = __uint_as_float(rr[2 * e]) * ksc[c0];
                    float u1 = __uint_as_float(rr[2 * e + 1]) * ksc[c0 + 1];
                    if (masked) {
                        if (c0 >= t.n || (p.causal && t.kg0 + c0 > lim)) u0 = -INFINITY;
                        if (c0 + 1 >= t.n || (p.causal && t.kg0 + c0 + 1 > lim)) u1 = -INFINITY;
                    }
                    float p0 = fast_exp2(fmaf(u0, rq, nb));
                    float p1 = fast_exp2(fmaf(u1, rq, nb));
                    lsum += p0 + p1;
                    if (t.pre) {
                        p0 *= vsc[c0];
                        p1 *= vsc[c0 + 1];
                    }
                    pk[e] = pack2(p0, p1, false);
                }
                tc::st16(s_t + c * 16, pk);
            }
            l += lsum;
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bar(B_P_FULL + buf));
            done = j + 1;
        }
        // ------------------------------------------------ epilogue
        bool have = done == T && T > 0;
        if (have) {
            const bool w = wait_ab(bar(B_KV_EMPTY + ((T - 1) & 1)), (uint32_t)((T - 1) >> 1) & 1u,
                                   p.err, abort_flag);
            have = __all_sync(0xffffffffu, w);
            tc::fence_after();
        }
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const int64_t orow = ((int64_t)b * p.Hq + hq) * p.Sq + i;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (have) {
                tc::ld32(tmem + lane_base + C::COL_O + c * 32, o);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv,
                                  p.out_bf16 != 0);
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) +
                                                       orow * D + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
        }
        if (row_ok && p.lse)
            p.lse[orow] = l > 0.0f ? (m_run + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 9) {
        tc::fence_after();
        tc::dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

template <int D>
cudaError_t launch_d(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    using C = PCfg<D>;
    CUtensorMap tm;
    memset(&tm, 0, sizeof(tm));
    if (p.Sk > 0) {
        auto enc = encode_fn();
        if (!enc) return cudaErrorNotSupported;
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Sk, (cuuint64_t)p.B * p.Hkv};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Sk * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)C::BN, 1};
        cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&tm, p.v_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         3, const_cast<void *>(p.v), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((p.Sq + 127) / 128, p.Hq, p.B);
    prefill_kernel<D><<<grid, kThreads, C::SMEM, st>>>(p, tm);
    log.add("prefill_kernel", grid, dim3(kThreads), dim3(1, 1, 1), C::SMEM);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.D) {
        case 64: return launch_d<64>(p, st, log);
        case 128: return launch_d<128>(p, st, log);
        case 256: return launch_d<256>(p, st, log);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace sage
