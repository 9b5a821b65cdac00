// INT8-QK prefill attention on the 5th-generation tensor cores (tcgen05).
//
// What it computes (SageAttention MXMACA README: attention kernel pipeline,
// feature matrix; "INT8 QK MMAC on gfx936 DCU", sections 1, 2.1, 3, 5.2):
//   S = Q_int8 K_int8^T exactly, each score rescaled by
//   q_scale[row] * k_scale[col] * sm_scale * log2(e) (+ the smooth_k row bias
//   on smoothed keys) before a base-2 online softmax; P.V in f16 with FP32
//   accumulation (bf16 V is rounded to f16 first, as the README's port
//   converts bf16 V to f16 before its kernel); O / l and LSE in the
//   epilogue.  Keys come from an optional paged INT8 prefix followed by the
//   contiguous chunk.  A packed variable-length batch (the README's varlen
//   path, there one launch per sequence) runs as one launch: every CTA
//   finds its sequence's query rows and keys through cu_seqlens and the
//   result is the single-sequence attention of each sequence.
//
// GB300 design.  sm_103a has no integer tcgen05 MMA, so QK^T runs on
// kind::f16 over the INT8 codes expanded EXACTLY to f16 (|q|,|k| <= 127;
// every partial sum of D <= 256 products is an integer below 2^24, which
// the FP32 accumulator holds exactly).  A staging kernel has already written
// the f16 key codes (and the prefix's value codes, and bf16 values as f16)
// plus one per-key scale array to the workspace, so here every K/V tile
// arrives by TMA straight into the 128-byte-swizzled layout the MMA reads.
// One CTA owns NQ query tiles of 128 rows (NQ = 2 for D <= 128, 1 for
// D = 256) of one (batch, head); keys stream in tiles of BN (128, or 64 at
// D = 256) through an NST-deep ring.
//   warps 0..4NQ*SPLIT-1  softmax: per query tile one warpgroup (one thread
//              per query row = TMEM lane), or at D = 256 two warpgroups
//              sharing each row's columns; Q int8 -> f16 once, into shared
//              memory (at D = 256 channels 0-127 into TMEM);
//              per key tile one tcgen05.ld of the whole S row into
//              registers, per-column K-scale recovery, online softmax with
//              lazy rescaling (O is rescaled only when the row max grows by
//              more than 2^8), P written back over S in TMEM.
//   next warp  producer (one thread): per key tile the K and V tiles (TMA
//              tensor loads) and the per-key K scales (1-D bulk copy) into
//              one stage of an NST-deep ring (D = 256: the K tiles only).
//   next warp  TMEM owner and MMA issuer (one thread): S_t = Q_t K^T, then
//              O_t += P_t V with P from TMEM.  With two query tiles the two
//              warpgroups ping-pong: the tensor core works on one tile's
//              MMAs while the other tile's softmax runs (one issuer keeps
//              each tile's MMAs together; two issuers interleaving them
//              measured slower).  With one tile (D = 256) S has three slots
//              instead, this warp issues only O += P V, and
//   next warp  issues S = Q K^T, and
//   next warp  streams the V tiles with the per-key K scales through a ring
//              of their own.
// Tensor memory (512 columns): O_t at [t*D, t*D+D), S slots from NQ*D.
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

constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per CTA

template <int D>
struct PCfg {
    static constexpr int BN = D == 256 ? 64 : 128;
    static constexpr int NQ = D == 256 ? 1 : 2;  // 128-row query tiles per CTA
    // Wide heads (D = 256): one query tile and three S slots in TMEM (P
    // written back over S), Q split between TMEM (channels 0-127) and
    // shared memory (128-255), K and V streamed through separate rings (a K
    // stage is released when its QK^T retires, a V stage -- V tile and the
    // per-key K scales -- when its P.V retires) and QK^T and P.V issued by
    // two threads.  With two S slots (all of Q in TMEM) QK^T(j) had to wait
    // for P.V(j-2) to retire, a chain of two MMAs and three hand-offs
    // longer than a key tile's softmax; with three it waits for P.V(j-3).
    static constexpr bool WIDE = D == 256;
    static constexpr int NS = WIDE ? 3 : 1;      // S slots per query tile
    static constexpr int NPH = BN / 64;          // P handed to the MMA in 64-key parts
    // softmax warpgroups per query tile: at D = 256 two, each taking half of
    // a row's 64 columns (one warpgroup alone is the critical path there)
    static constexpr int SPLIT = D == 256 ? 2 : 1;
    static constexpr int CW = BN / SPLIT;        // S columns per softmax thread
    static constexpr int NSW = NQ * SPLIT;       // softmax warpgroups
    // softmax warpgroups + one warpgroup holding the producer and MMA warps
    // (and, unless WIDE, two idle warps, so that register reallocation works
    // per warpgroup)
    static constexpr int THREADS = NSW * 128 + 128;
    // registers: 2 x 128 x 208 + 128 x 88 = 384 x 168, the launch budget
    static constexpr int REG_SOFTMAX = 208, REG_OTHER = 88;
    static_assert(NSW == 1 || NSW * 128 * REG_SOFTMAX + 128 * REG_OTHER <= THREADS * 168,
                  "register split exceeds the launch budget");
    static_assert(SPLIT == 1 || NPH == 1, "split rows hand P over as one part");
    // Q as the A operand of QK^T: in shared memory (two query tiles fill
    // TMEM with O and S), or (WIDE) channels 0-127 in TMEM and the rest in
    // shared memory
    static constexpr int QB = WIDE ? 128 * 128 * 2 : 128 * D * 2;  // f16 Q (part) in smem, swizzled
    static constexpr int KB = BN * D * 2;      // f16 K (or V) tile, swizzled
    static constexpr int NSV = 2;                                   // V ring depth (WIDE)
    static constexpr int VSB = (KB + BN * 4 + 1023) / 1024 * 1024;  // V stage (WIDE)
    // stage: K tile | V tile | per-key K scales (or, WIDE, the K tile alone)
    static constexpr int SB = (2 * KB + BN * 4 + 1023) / 1024 * 1024;
    static constexpr int KSB = WIDE ? KB : SB;   // ring stride of the K stages
    static constexpr int OFF_ST = NQ * QB;
    static constexpr int NST_FIT = (kSmemLimit - 1024 - OFF_ST - 512) / SB;
    static constexpr int NST = WIDE ? 3 : (NST_FIT > 4 ? 4 : NST_FIT);
    static constexpr int OFF_V = OFF_ST + NST * KSB;                // WIDE: V ring
    static constexpr int OFF_BAR = OFF_V + (WIDE ? NSV * VSB : 0);
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    // split rows: partial row max / sum of each half, double-buffered
    static constexpr int OFF_RED = OFF_MISC + 64;
    static constexpr int SMEM = OFF_RED + (SPLIT > 1 ? 2 * NSW * 128 * 4 : 0) + 1024;
    static constexpr uint32_t COL_S = NQ * D;
    static constexpr uint32_t COL_Q = NQ * D + NQ * NS * BN;  // WIDE: Q channels 0-127
    static_assert(NST >= 2, "the key ring needs two stages");
    static_assert(NQ * D + NQ * NS * BN + (WIDE ? 64 : 0) <= 512, "tensor memory holds 512 columns");
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    // epilogue staging: 4 KB per softmax warp, in its tile's Q tile or, with
    // one query tile, in the key ring
    static_assert(NQ == 1 ? NST * KSB >= NSW * 4 * 4096 : QB >= 4 * 4096, "epilogue staging fits");
    static_assert(!WIDE || (NQ == 1 && SPLIT == 2 && NPH == 1), "wide-head layout");
};

// barrier slots
enum {
    B_KV_FULL = 0,    // [NST] producer: K tile, V tile and per-key scales landed (WIDE: K tile)
    B_KV_EMPTY = 4,   // [NST] MMA: every QK^T and P.V reading the stage retired (WIDE: its QK^T)
    B_S_FREE = 8,     // [NS] WIDE, P.V issuer: the P.V reading an S slot retired
    B_V_FULL = 11,    // [NSV] WIDE, V producer: V tile and per-key scales landed
    B_V_EMPTY = 13,   // [NSV] WIDE, P.V issuer: the P.V reading the V stage retired
    B_DRAIN_QK = 15,  // WIDE, QK^T issuer: every QK^T it issued retired
    B_S_FULL = 16,    // [NQ*NS] MMA: S = Q K^T done
    B_P_FULL = 20,    // [NQ*NS*NPH] softmax warps: a 64-key part of P in TMEM (O rescaled)
    B_O_FINAL = 26,   // [NQ] MMA: the last O_t += P_t V done (one phase)
    B_Q_READY = 28,   // softmax: Q in shared memory / TMEM
    B_DRAIN = 29      // MMA: every issued MMA retired
};

struct PrefillMaps {
    CUtensorMap k;      // f16 key codes [B*Hkv][Lpad][D]
    CUtensorMap v_pre;  // f16 value codes of the prefix [B*Hkv][Vrows][D]
    CUtensorMap v_ch;   // chunk values: the caller's f16 V [B*Hkv][Sk][D] or v_pre; with the
                        // caller's NHD V [B][Sk][Hkv][D] a 4-D map (channel, head, token, batch)
    int v_ch_4d;        // 1: v_ch is that 4-D map
};

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

// 16 int8 channels [16*dc, 16*dc+16) of row r -> exact f16, stored as the
// two 16-byte chunks 2*dc, 2*dc+1 of row r in a 128-byte-swizzled tile of
// ROWS rows (64-channel atom columns ROWS*128 bytes apart, chunk c of row r
// at c ^ (r%8)).
template <int ROWS>
__device__ __forceinline__ void store_piece(uint8_t *tile, int r, int dc, uint4 w) {
    uint4 h0, h1;
    i8x4_to_f16x4(w.x, h0.x, h0.y);
    i8x4_to_f16x4(w.y, h0.z, h0.w);
    i8x4_to_f16x4(w.z, h1.x, h1.y);
    i8x4_to_f16x4(w.w, h1.z, h1.w);
    const int c8 = 2 * dc;
    uint8_t *row = tile + (c8 >> 3) * (ROWS * 128) + (r >> 3) * 1024 + (r & 7) * 128;
    *reinterpret_cast<uint4 *>(row + (((c8 & 7) ^ (r & 7)) << 4)) = h0;
    *reinterpret_cast<uint4 *>(row + ((((c8 + 1) & 7) ^ (r & 7)) << 4)) = h1;
}

// Dense form: query tile index -> (batch, head, query tile).  One linear
// index over (batch, head) pairs taken in bundles of p.bundle (whose staged
// keys fit in L2 together); within a bundle the heaviest (causal) query
// tiles of all its pairs come first, so that no heavy tile is left to run
// alone at the end of the grid.  Returns the pair index b * Hq + hq.  (The
// attention kernel writes the same decode out in place.)
__device__ __forceinline__ int dense_tile(const PrefillParams &p, int QR, int item, int &ct) {
    const int nct = (p.Sq + QR - 1) / QR;
    const int per = nct * p.bundle;
    const int bun = item / per;
    const int nb = min(p.bundle, p.B * p.Hq - bun * p.bundle);
    const int r = item - bun * per;
    ct = nct - 1 - r / nb;
    return bun * p.bundle + r % nb;
}

// Dense form: CTA index -> query tile index; part = the CTA's key range of a
// split tail tile, or -1 for a whole tile.
__device__ __forceinline__ int split_item(const PrefillParams &p, int L, int &part) {
    part = -1;
    if (p.split_k > 0 && L >= p.split_f) {
        const int v = L - p.split_f;
        part = v % p.split_k;
        return p.split_f + v / p.split_k;
    }
    return L;
}

// VL: a packed variable-length batch (rows and keys located through
// cu_seqlens); the dense instantiation keeps its addressing in closed form.
template <int D, bool VL, bool PR = false>
__global__ void __launch_bounds__(PCfg<D>::THREADS, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p,
                   const __grid_constant__ PrefillMaps maps) {
    using C = PCfg<D>;
    constexpr int BN = C::BN, NQ = C::NQ, NS = C::NS, NST = C::NST;
    constexpr int kProducer = C::NSW * 4, kMma = C::NSW * 4 + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sm_a = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int QR = 128 * NQ;  // query rows per CTA
    int b, hq, ct;
    int part = -1;  // dense form, D = 256: this CTA's part of a split query tile
    int cq0 = 0, cq1 = 0, ck0 = 0, ck1 = 0;  // packed batch: this sequence's offsets
    // PR (packed form, even GQA group): a CTA takes 128 query rows of two
    // heads that share a KV head -- query tile t is head hq + t -- instead
    // of 256 rows of one head, so a sequence's last CTA is not half empty
    // and the first tile does not sweep the second tile's diagonal key tile
    // fully masked.  Every other instantiation keeps the code below as is.
    static_assert(!PR || (VL && NQ == 2), "head pairs: packed form, two query tiles");
    if constexpr (PR) {
        const int g = (int)(blockIdx.x / (unsigned)(p.Hq / 2));
        hq = 2 * (int)(blockIdx.x - (unsigned)g * (unsigned)(p.Hq / 2));
        b = varlen_find_warp(p.B, g, [&](int k) {
            const int c = p.cu_q[k];
            return varlen_group0(c < 0 ? 0 : c, k, 128);
        });
        cq0 = p.cu_q[b], cq1 = p.cu_q[b + 1], ck0 = p.cu_k[b], ck1 = p.cu_k[b + 1];
        ct = g - (int)varlen_group0(cq0 < 0 ? 0 : cq0, b, 128);  // reversed below
    } else if constexpr (VL) {
        // one linear index, heads fastest: the CTAs of a tile slot for every
        // head start together, and the grid ends on the light (first) tiles
        // of the last sequence instead of on one head's heaviest tiles
        const int g = (int)(blockIdx.x / (unsigned)p.Hq);
        hq = (int)(blockIdx.x - (unsigned)g * (unsigned)p.Hq);
        // compact tile index: sequence b owns tiles [cu_q[b] / QR + b, ...),
        // ceil(len_b / QR) of them (at most one spare slot per sequence)
        b = varlen_find_warp(p.B, g, [&](int k) {
            const int c = p.cu_q[k];
            return varlen_group0(c < 0 ? 0 : c, k, QR);
        });
        // the sequence's query and key bounds, loaded together
        cq0 = p.cu_q[b], cq1 = p.cu_q[b + 1], ck0 = p.cu_k[b], ck1 = p.cu_k[b + 1];
        ct = g - (int)varlen_group0(cq0 < 0 ? 0 : cq0, b, QR);  // reversed below
    } else {
        // (the tile decode is written out here and in late_pair(): through
        // the shared helper the D = 128 kernel spilled more)
        int item = blockIdx.x;
        if constexpr (C::WIDE) item = split_item(p, item, part);
        const int nct = (p.Sq + QR - 1) / QR;
        const int per = nct * p.bundle;
        const int bun = item / per;
        const int nb = min(p.bundle, p.B * p.Hq - bun * p.bundle);
        const int rr = item - bun * per;
        ct = nct - 1 - rr / nb;
        const int u = bun * p.bundle + rr % nb;
        b = u / p.Hq;
        hq = u % p.Hq;
    }
    const int kvh = hq / p.group;

    // ------------------------------------------------ where this CTA's rows live
    // Sq(), Sk(): this sequence's query and chunk-key counts (the dense form
    // reads the kernel parameters at each use, which keeps them out of the
    // registers); kz, krow0: the staged keys' (head, first row) coordinates.
    int vsq = 0, vsk = 0;
    int64_t qs = 0, vq_row0 = 0, vsc0 = 0, vmu_vl = 0;
    int kz = b * p.Hkv + kvh, krow0 = 0;
    auto Sq = [&]() -> int {
        if constexpr (VL) return vsq;
        return p.Sq;
    };
    auto Sk = [&]() -> int {
        if constexpr (VL) return vsk;
        return p.Sk;
    };
    if constexpr (VL) {
        int *e = threadIdx.x == 0 ? p.err : nullptr;  // each CTA checks its sequence
        int64_t ks = 0;
        vsq = varlen_seq_of(cq0, cq1, p.Sq, p.total_q, e, &qs);
        vsk = varlen_seq_of(ck0, ck1, p.Sk, p.total_k, e, &ks);
        const int ntile = (vsq + (PR ? 128 : QR) - 1) / (PR ? 128 : QR);
        // a spare slot, a slot before the first sequence, or an empty or
        // invalid sequence: nothing to do (the whole CTA returns)
        if (ct < 0 || ct >= ntile) return;
        ct = ntile - 1 - ct;      // heaviest (causal) tiles of the sequence first
        vq_row0 = (int64_t)hq * p.total_q + qs;
        vsc0 = (int64_t)hq * p.q_groups + varlen_group0(qs, b, 1 << p.q_shift);
        kz = kvh;
        krow0 = (int)varlen_key_row0(ks, b, BN);
        vmu_vl = ((int64_t)b * p.Hkv + kvh) * D;
    }
    // row of query i in q, q_bias, lse and the debug dump ([Hq, total_q]
    // packed, [B, Hq, Sq] dense); its output row (packed output is
    // token-major [total_q, Hq, D]); its scale group
    auto q_row = [&](int i) -> int64_t {
        if constexpr (VL) return vq_row0 + i;
        return ((int64_t)b * p.Hq + hq) * p.Sq + i;
    };
    auto out_row = [&](int i) -> int64_t {
        if constexpr (VL) return (qs + i) * p.Hq + hq;
        return ((int64_t)b * p.Hq + hq) * p.Sq + i;
    };
    auto q_group = [&](int i) -> int64_t {
        if constexpr (VL) return vsc0 + (i >> p.q_shift);
        return ((int64_t)b * p.Hq + hq) * p.q_groups + (i >> p.q_shift);
    };
    // The same rows for use after the key loop.  Dense: (b, hq) come from
    // the linear CTA index, so the pair index b * Hq + hq is recomputed from
    // a fresh read of it rather than kept live through the softmax loop.
    auto late_pair = [&]() -> int64_t {
        int L;
        asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(L));
        if constexpr (C::WIDE) {
            int pt;
            L = split_item(p, L, pt);
        }
        const int per = (p.Sq + QR - 1) / QR * p.bundle;
        const int bun = L / per;
        const int nb = min(p.bundle, p.B * p.Hq - bun * p.bundle);
        return (int64_t)bun * p.bundle + (L - bun * per) % nb;
    };
    auto q_row_late = [&](int i) -> int64_t {
        if constexpr (VL) return vq_row0 + i;
        return late_pair() * p.Sq + i;
    };
    auto out_row_late = [&](int i) -> int64_t {
        if constexpr (VL) return (qs + i) * p.Hq + hq;
        const int64_t u = late_pair();
        if (p.nhd) return ((u / p.Hq) * p.Sq + i) * p.Hq + u % p.Hq;  // [B, Sq, Hq, D]
        return u * p.Sq + i;
    };
    // smooth_v: this (batch or sequence, kv head)'s V mean row
    auto v_mean_late = [&]() -> const float * {
        if constexpr (VL) return p.v_mean + vmu_vl;
        const int64_t u = late_pair();
        const int64_t bb = u / p.Hq, kv = (u % p.Hq) / p.group;
        return p.v_mean + (bb * p.Hkv + kv) * D;
    };
    const int i0 = ct * (PR ? 128 : QR);

    // ------------------------------------------------------ tile schedule
    int P = 0;
    if (p.prefix_lens) {
        P = p.prefix_lens[b];
        if (P < 0 || P > p.max_prefix_len) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBadBlock);
            P = P < 0 ? 0 : p.max_prefix_len;
        }
    }
    const int off = P + Sk() - Sq();  // key j visible to row i iff j <= i + off (causal)
    const int row_last = min(i0 + (PR ? 128 : 128 * NQ) - 1, Sq() - 1);
    const int kmax = p.causal ? row_last + off : P + Sk() - 1;
    int n_pre = 0, n_ch = 0;
    if (kmax >= 0) {
        n_pre = min((P + BN - 1) / BN, kmax / BN + 1);
        if (kmax >= P) n_ch = min((Sk() + BN - 1) / BN, (kmax - P) / BN + 1);
    }
    int T = n_pre + n_ch;
    // a part of a split query tile takes key tiles [j0, j0 + T) of it
    int j0 = 0;
    if constexpr (C::WIDE && !VL) {
        if (part >= 0) {
            j0 = (int)((int64_t)part * T / p.split_k);
            T = (int)((int64_t)(part + 1) * T / p.split_k) - j0;
        }
    }
    const int wpre = p.Ppad / BN;  // first chunk tile in the workspace

    // The softmax threads issue their query loads now: they land while the
    // barriers and tensor memory are set up (issued after that, each
    // 16-byte piece between shared-memory stores, the query took ~3 us of
    // every CTA's start-up).  A query tile's rows are consecutive in memory,
    // so with Q headed for shared memory each warpgroup reads its tile
    // coalesced, piece u = thread + 128 m (row u / (D / 16)); reading one
    // row per thread made every load instruction gather 32 rows, and the
    // CTA's ~2000 scattered misses held up its tensor-memory allocation by
    // a microsecond.  With Q headed for tensor memory each thread needs its
    // own row's channels (its TMEM lane).
    constexpr int QLD = D / (16 * C::SPLIT);  // 16-byte pieces per thread
    uint4 qw[QLD];
    // dense form: the softmax thread's query scale and row bias, loaded
    // with the query (after the query staging they held up the first key
    // tile's softmax; the packed form loads them there, which spills less)
    float q_sc0 = 0.0f, q_b0 = 0.0f;
    {
        const int wq = warp >> 2;
        const int ti = threadIdx.x & 127;
        if constexpr (!VL) {
            const int irow = i0 + (wq / C::SPLIT) * 128 + ti;
            if (warp < kProducer && irow < Sq()) {
                q_sc0 = __ldg(p.q_scale + q_group(irow));
                if (p.q_bias) q_b0 = __ldg(p.q_bias + q_row(irow));
            }
        }
        if constexpr (C::WIDE) {
            const int iq = i0 + (wq / C::SPLIT) * 128 + ti;
            const bool ok = warp < kProducer && iq < Sq();
            const int8_t *src = p.q + (ok ? q_row(iq) * D : 0) + (wq % C::SPLIT) * (D / C::SPLIT);
#pragma unroll
            for (int k = 0; k < QLD; ++k)
                qw[k] = ok ? __ldg(reinterpret_cast<const uint4 *>(src) + k) : make_uint4(0, 0, 0, 0);
        } else {
            static_assert(C::WIDE || C::SPLIT == 1, "a shared-memory Q tile belongs to one warpgroup");
            const int row0 = i0 + (PR ? 0 : wq * 128);
            const bool sm_thread = warp < kProducer;
            const int64_t qoff = PR ? (int64_t)wq * p.total_q : 0;  // PR: tile wq is head hq + wq
            const int8_t *src = p.q + (sm_thread && row0 < Sq() ? (q_row(row0) + qoff) * D : 0);
#pragma unroll
            for (int m = 0; m < QLD; ++m) {
                const int u = ti + 128 * m;
                const bool ok = sm_thread && row0 + u / (D / 16) < Sq();
                qw[m] = ok ? __ldg(reinterpret_cast<const uint4 *>(src) + u) : make_uint4(0, 0, 0, 0);
            }
        }
    }

    // barriers set up by the producer warp's first thread, which holds no
    // query loads: the initialising thread's fence waits for its own
    // outstanding loads, and with those in flight it held the whole CTA
    // (and the first key copies) back by about a microsecond
    if (threadIdx.x == kProducer * 32) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), 1);
        }
        for (int s = 0; s < NQ * NS; ++s) mbar_init(bar(B_S_FULL + s), 1);
        // WIDE: one arrival per softmax warp (its lanes' stores ordered by
        // the warp's own synchronisation), 0.2 % faster on the chunked
        // workload; per thread at D <= 128, where per warp measured 0.5 %
        // slower on the dense workload
        for (int s = 0; s < NQ * NS * C::NPH; ++s)
            mbar_init(bar(B_P_FULL + s), C::WIDE ? 4 * C::SPLIT : 128 * C::SPLIT);
        for (int t = 0; t < NQ; ++t) {
            mbar_init(bar(B_O_FINAL + t), 1);
        }
        mbar_init(bar(B_Q_READY), C::NSW * 128);
        mbar_init(bar(B_DRAIN), 1);
        if constexpr (C::WIDE) {
            for (int s = 0; s < NS; ++s) mbar_init(bar(B_S_FREE + s), 1);
            for (int s = 0; s < C::NSV; ++s) {
                mbar_init(bar(B_V_FULL + s), 1);
                mbar_init(bar(B_V_EMPTY + s), 1);
            }
            mbar_init(bar(B_DRAIN_QK), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMma) {
        tc::alloc(smem_u32(tmem_slot), 512);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp >= kProducer) {
        if constexpr (C::NSW == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if (warp == kProducer || (C::WIDE && warp == kMma + 2)) {
        // ============================================================ producers
        if (lane == 0 && T > 0) {
            // one stage per key tile, refilled once the MMAs reading it
            // retired: K, V and the per-key K scales on one barrier, or (WIDE)
            // the K tile from this warp and V with the scales from warp
            // kMma + 2, each through its own ring
            const bool load_k = !C::WIDE || warp == kProducer;
            const bool load_v = !C::WIDE || warp != kProducer;
            // this grid is launched behind the staging pass and may start
            // before it ends: the staged keys, values and per-key scales are
            // read only after that grid has completed (no-op otherwise).
            // Everything else this kernel reads was written before the
            // staging pass began.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (load_k) tc::prefetch_tmap(&maps.k);
            if (load_v && n_pre > 0) tc::prefetch_tmap(&maps.v_pre);
            if (load_v && n_ch > 0) tc::prefetch_tmap(&maps.v_ch);
            // chunk values staged after the prefix (bf16 or smoothed V), or
            // read in place from the caller's f16 V
            const int vch_off = (p.v_bf16 || p.v_mean) ? p.Ppad : 0;
            const int ns = load_k ? NST : C::NSV;
            const int full0 = C::WIDE && !load_k ? B_V_FULL : B_KV_FULL;
            const int empty0 = C::WIDE && !load_k ? B_V_EMPTY : B_KV_EMPTY;
            int issued = 0;
            for (int jj = 0; jj < T; ++jj) {
                const int s = jj % ns;
                if (jj >= ns &&
                    !wait_ab(bar(empty0 + s), (uint32_t)(jj / ns - 1) & 1u, p.err, abort_flag))
                    break;
                const int kt = j0 + jj;  // key tile
                const bool pre = kt < n_pre;
                const int w = pre ? kt : wpre + (kt - n_pre);
                const uint32_t fb = bar(full0 + s);
                // K tile at kst; V tile at vst, its per-key scales after it
                const uint32_t kst = sm_a + C::OFF_ST + s * C::KSB;
                const uint32_t vst = C::WIDE ? sm_a + C::OFF_V + s * C::VSB : kst + C::KB;
                mbar_arrive_expect_tx(fb, (load_k ? C::KB : 0) + (load_v ? C::KB + BN * 4 : 0));
                if (load_k) {
#pragma unroll
                    for (int a = 0; a < D / 64; ++a)
                        tc::tma_load_3d(kst + a * BN * 128, &maps.k, a * 64, krow0 + w * BN, kz, fb);
                }
                if (load_v) {
                    const CUtensorMap *vm = pre ? &maps.v_pre : &maps.v_ch;
                    const int vrow = krow0 + (pre ? w * BN : (w - wpre) * BN + vch_off);
                    if (!pre && maps.v_ch_4d) {
#pragma unroll
                        for (int a = 0; a < D / 64; ++a)
                            tc::tma_load_4d(vst + a * BN * 128, vm, a * 64, kvh, vrow, b, fb);
                    } else {
#pragma unroll
                        for (int a = 0; a < D / 64; ++a)
                            tc::tma_load_3d(vst + a * BN * 128, vm, a * 64, vrow, kz, fb);
                    }
                    bulk_g2s(vst + C::KB, p.ksc_ws + (int64_t)kz * p.Lpad + krow0 + w * BN, BN * 4,
                             fb);
                }
                ++issued;
            }
            // wait for the copies still in flight before the CTA may exit
            for (int jj = max(0, issued - ns); jj < issued; ++jj)
                mbar_wait(bar(full0 + jj % ns), (uint32_t)(jj / ns) & 1u, p.err);
        }
        __syncwarp();
    } else if (warp == kMma || (C::WIDE && warp == kMma + 1)) {
        // ============================================================ MMA issuers
        // WIDE: two threads issue, warp kMma + 1 the QK^T of each key tile and
        // warp kMma the P.V.  The tensor core takes only a couple of MMAs
        // ahead of execution, so every barrier wait of a single issuer (a few
        // hundred cycles per key tile) left it idle; with two issuers one
        // thread's waits overlap the other's MMAs.
        if (lane == 0 && T > 0) {
            const uint32_t idq = tc::idesc_f16(128, BN, false, false);
            const uint32_t idp = tc::idesc_f16(128, D, false, true);  // P.V in f16
            // descriptors built once; a k-step adds its byte offset >> 4
            const uint64_t qd0 = tc::sdesc_sw128(sm_a, 16, 1024);
            const uint64_t kd0 = tc::sdesc_sw128(sm_a + C::OFF_ST, 16, 1024);
            const uint64_t vd0 = tc::sdesc_sw128(sm_a + (C::WIDE ? C::OFF_V : C::OFF_ST + C::KB),
                                                 BN * 128, 1024);
            auto qk = [&](int jj, int t) {
                const int slot = t * NS + jj % NS;
                const uint64_t qd = qd0 + (uint64_t)((t * C::QB) >> 4);
                const uint64_t kd = kd0 + (uint64_t)(((jj % NST) * C::KSB) >> 4);
                const uint32_t d = tmem + C::COL_S + slot * BN;
                if constexpr (C::WIDE) {
                    // channels 0-127: A = Q from TMEM (column c of lane r holds
                    // f16 channels 2c, 2c+1); 128-255: A = Q from shared memory
                    const uint32_t qa = tmem + C::COL_Q;
                    tc::mma_ts(d, qa, kd, idq, 0u);
#pragma unroll
                    for (int ks = 1; ks < 8; ++ks)
                        tc::mma_ts_acc(d, qa + ks * 8,
                                       kd + (((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4), idq);
#pragma unroll
                    for (int ks = 8; ks < D / 16; ++ks)
                        tc::mma_ss_acc(d, qd + ((((ks - 8) >> 2) * (128 * 128) + (ks & 3) * 32) >> 4),
                                       kd + (((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4), idq);
                } else {
                    tc::mma_ss(d, qd, kd, idq, 0u);
#pragma unroll
                    for (int ks = 1; ks < D / 16; ++ks)
                        tc::mma_ss_acc(d, qd + (((ks >> 2) * (128 * 128) + (ks & 3) * 32) >> 4),
                                       kd + (((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4), idq);
                }
                tc::commit(bar(B_S_FULL + slot));
            };
            // O_t += P_t V_j in 64-key parts, each issued as soon as the
            // softmax has stored that part of P (the first part also needs V)
            auto pv = [&](int jj, int t) -> bool {
                const int slot = t * NS + jj % NS;
                const uint32_t sp = (uint32_t)(jj / NS) & 1u;
                const uint64_t vd = C::WIDE ? vd0 + (uint64_t)(((jj % C::NSV) * C::VSB) >> 4)
                                            : vd0 + (uint64_t)(((jj % NST) * C::SB) >> 4);
                const uint32_t pt = tmem + C::COL_S + slot * BN;
                const uint32_t o = tmem + t * D;
#pragma unroll
                for (int h = 0; h < C::NPH; ++h) {
                    // (the stage's V landed with its K, waited before QK^T;
                    // WIDE: the P.V issuer waited for the V stage)
                    const bool ok = wait_ab(bar(B_P_FULL + slot * C::NPH + h), sp, p.err, abort_flag);
                    if (!ok) return false;
                    tc::fence_after();
#pragma unroll
                    for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {
                        if (kk == 0)
                            tc::mma_ts(o, pt, vd, idp, jj > 0 ? 1u : 0u);
                        else
                            tc::mma_ts_acc(o, pt + kk * 8, vd + ((kk * 2048) >> 4), idp);
                    }
                }
                if (jj == T - 1) tc::commit(bar(B_O_FINAL + t));
                return true;
            };
            auto k_ready = [&](int jj) {
                const bool ok = wait_ab(bar(B_KV_FULL + jj % NST), (uint32_t)(jj / NST) & 1u, p.err,
                                        abort_flag);
                tc::fence_after();
                return ok;
            };
            if constexpr (C::WIDE) {
                if (warp == kMma + 1) {
                    // S_j = Q K_j^T into slot j % 3 once K_j landed and the
                    // P.V of key tile j - 3 (the slot's last reader) retired;
                    // the K stage is free when this QK^T retires
                    bool ok = wait_ab(bar(B_Q_READY), 0, p.err, abort_flag);
                    for (int jj = 0; ok && jj < T; ++jj) {
                        if (!(ok = k_ready(jj))) break;
                        if (jj >= NS && !(ok = wait_ab(bar(B_S_FREE + jj % NS),
                                                       (uint32_t)(jj / NS - 1) & 1u, p.err, abort_flag)))
                            break;
                        tc::fence_after();
                        qk(jj, 0);
                        tc::commit(bar(B_KV_EMPTY + jj % NST));
                    }
                    tc::commit(bar(B_DRAIN_QK));
                    mbar_wait(bar(B_DRAIN_QK), 0, p.err);
                } else {
                    // O += P_j V_j once V_j landed and P_j is in TMEM; then V
                    // stage j and S slot j % 3 are free
                    bool ok = true;
                    for (int jj = 0; ok && jj < T; ++jj) {
                        if (!(ok = wait_ab(bar(B_V_FULL + jj % C::NSV), (uint32_t)(jj / C::NSV) & 1u,
                                           p.err, abort_flag)))
                            break;
                        if (!(ok = pv(jj, 0))) break;
                        tc::commit(bar(B_V_EMPTY + jj % C::NSV));
                        tc::commit(bar(B_S_FREE + jj % NS));
                    }
                    tc::commit(bar(B_DRAIN));
                    mbar_wait(bar(B_DRAIN), 0, p.err);
                }
            } else {
                // one issuer; per query tile: O_t += P_t V_j, then S_t = Q_t K_{j+1}
                bool ok = wait_ab(bar(B_Q_READY), 0, p.err, abort_flag) && k_ready(0);
                if (ok) {
#pragma unroll
                    for (int t = 0; t < NQ; ++t) qk(0, t);
                }
                for (int jj = 0; ok && jj < T; ++jj) {
                    for (int t = 0; t < NQ; ++t) {
                        if (!(ok = pv(jj, t))) break;
                        if (t == NQ - 1) tc::commit(bar(B_KV_EMPTY + jj % NST));
                        if (jj + 1 < T) {
                            if (t == 0 && !(ok = k_ready(jj + 1))) break;
                            qk(jj + 1, t);
                        }
                    }
                }
                tc::commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0, p.err);  // every issued MMA has retired
            }
        }
        __syncwarp();
    } else if (!C::WIDE && warp == kMma + 1 && p.q_ahead > 0) {
        // ============================================================ query prefetch
        // An otherwise idle warp asks L2 for the query tile of the CTA one
        // wave ahead, so that CTA's query loads at its start hit L2.
        const unsigned x = blockIdx.x + (unsigned)p.q_ahead;
        if (x < gridDim.x) {
            int pb, ph, pct, r0 = 0, nr = 0;
            int64_t prow = 0;
            if constexpr (VL) {
                constexpr int QV = PR ? 128 : QR;    // rows per CTA
                constexpr unsigned HC = PR ? 2 : 1;  // heads per CTA
                const int g = (int)(x / ((unsigned)p.Hq / HC));
                ph = (int)(x - (unsigned)g * ((unsigned)p.Hq / HC)) * HC;
                pb = varlen_find_warp(p.B, g, [&](int k) {
                    const int c = p.cu_q[k];
                    return varlen_group0(c < 0 ? 0 : c, k, QV);
                });
                int64_t pqs = 0;
                const int len = varlen_seq_of(p.cu_q[pb], p.cu_q[pb + 1], p.Sq, p.total_q, nullptr, &pqs);
                const int ntile = (len + QV - 1) / QV;
                pct = g - (int)varlen_group0(pqs, pb, QV);
                if (pct >= 0 && pct < ntile) {
                    r0 = (ntile - 1 - pct) * QV;
                    nr = min(QV, len - r0);
                    prow = (int64_t)ph * p.total_q + pqs + r0;
                }
            } else {
                const int nct = (p.Sq + QR - 1) / QR;
                const int per = nct * p.bundle;
                const int bun = (int)x / per;
                const int nb = min(p.bundle, p.B * p.Hq - bun * p.bundle);
                const int rr = (int)x - bun * per;
                pct = nct - 1 - rr / nb;
                const int u = bun * p.bundle + rr % nb;
                pb = u / p.Hq;
                ph = u % p.Hq;
                r0 = pct * QR;
                nr = min(QR, p.Sq - r0);
                prow = ((int64_t)pb * p.Hq + ph) * p.Sq + r0;
            }
            if (lane == 0 && nr > 0) {
                // rows of a query tile are consecutive: one bulk prefetch
                // (16-byte aligned, a multiple of 16 bytes: D is)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.q + prow * D),
                             "r"((uint32_t)(nr * D))
                             : "memory");
            }
            if constexpr (PR) {
                // the pair's second head
                if (lane == 1 && nr > 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                     p.q + (prow + p.total_q) * D),
                                 "r"((uint32_t)(nr * D))
                                 : "memory");
            }
            // dense form: the tile's row biases and scales too, one 128-byte
            // line per lane, every address inside the rows' range (in the
            // packed form the extra code made the softmax spill more and
            // the varlen launch 2.6 % slower)
            if constexpr (!VL) {
                auto lines = [&](const float *a, int n) {
                    if (n > 0 && lane <= (n + 31) / 32) {
                        const float *x = a + min(32 * lane, n - 1);
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(x) : "memory");
                    }
                };
                if (nr > 0) {
                    if (p.q_bias) lines(p.q_bias + prow, nr);
                    const int g0 = r0 >> p.q_shift, g1 = (r0 + nr - 1) >> p.q_shift;
                    lines(p.q_scale + ((int64_t)pb * p.Hq + ph) * p.q_groups + g0, g1 - g0 + 1);
                }
            }
        }
        __syncwarp();
    }
    } else {
        if constexpr (C::NSW == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
        // ============================================================ softmax
        constexpr int SPLIT = C::SPLIT, CW = C::CW;
        const int wg = warp >> 2;              // softmax warpgroup
        const int t = wg / SPLIT;              // query tile of this warpgroup
        const int hc = wg % SPLIT;             // which part of the row's columns
        const int c0 = hc * CW;                // first S column of this thread
        const int r = threadIdx.x & 127;       // row within the tile = TMEM lane
        const int i_first = i0 + (PR ? 0 : t * 128);
        if constexpr (PR) {
            // this warpgroup's head: every row address below follows it
            hq += t;
            vq_row0 += (int64_t)t * p.total_q;
            vsc0 += (int64_t)t * p.q_groups;
        }
        const int i = i_first + r;
        const bool row_ok = i < Sq();
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        // split rows: the two threads of a row swap partial maxima / sums
        float *red = reinterpret_cast<float *>(sm + C::OFF_RED);
        auto pair_sync = [&]() {
            asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(SPLIT * 128) : "memory");
        };
        auto pair_max = [&](float v, int ph) {
            if constexpr (SPLIT == 1) {
                return v;
            } else {
                float *rb = red + ((ph & 1) * C::NSW + wg) * 128;
                rb[r] = v;
                pair_sync();
                return fmaxf(v, red[((ph & 1) * C::NSW + (wg ^ 1)) * 128 + r]);
            }
        };
        {
            if constexpr (C::WIDE) {
                if (hc == 0) {
                    // channels 0-127 -> exact f16 pairs in this thread's TMEM lane
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t v[32];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint4 w = qw[c * 4 + u];
                            i8x4_to_f16x4(w.x, v[u * 8 + 0], v[u * 8 + 1]);
                            i8x4_to_f16x4(w.y, v[u * 8 + 2], v[u * 8 + 3]);
                            i8x4_to_f16x4(w.z, v[u * 8 + 4], v[u * 8 + 5]);
                            i8x4_to_f16x4(w.w, v[u * 8 + 6], v[u * 8 + 7]);
                        }
                        tc::st32(tmem + lane_base + C::COL_Q + c * 32, v);
                    }
                    tc::wait_st();
                    tc::fence_before();
                } else {
                    // channels 128-255 -> f16 in the swizzled K-major
                    // shared-memory tile (two 64-channel atom columns)
#pragma unroll
                    for (int m = 0; m < QLD; ++m) store_piece<128>(sm, r, m, qw[m]);
                    tc::fence_proxy_async();  // st.shared -> visible to the tensor core
                }
            } else {
                // Q row int8 -> f16 in the swizzled K-major layout of the A operand
                uint8_t *qt = sm + t * C::QB;
#pragma unroll
                for (int m = 0; m < QLD; ++m) {
                    const int u = r + 128 * m;
                    store_piece<128>(qt, u / (D / 16), u % (D / 16), qw[m]);
                }
                tc::fence_proxy_async();  // st.shared -> visible to the tensor core
            }
            mbar_arrive(bar(B_Q_READY));
        }
        // kept strictly positive so that a masked (-inf) score stays -inf; an
        // all-zero Q row (scale 0) then scores ~1e-30 * acc = 0 as it should
        if constexpr (VL) {
            if (row_ok) {
                q_sc0 = p.q_scale[q_group(i)];
                if (p.q_bias) q_b0 = p.q_bias[q_row(i)];
            }
        }
        const float rq = fmaxf(row_ok ? q_sc0 * p.qk_scale_log2 : 0.0f, 1e-30f);
        const float bc = (row_ok && p.q_bias) ? q_b0 * p.qk_scale_log2 : 0.0f;
        const int lim = i + off;
        // K scales constant over 64-key groups (k_block >= 64, chunk keys):
        // the max runs on the raw integer scores and the scale folds into
        // the exponent's FMA, one value per group
        const bool kuni = p.k_shift >= 6;
        constexpr int NG = CW >= 64 ? CW / 64 : 1;   // 64-key groups this thread touches
        constexpr int GW = CW >= 64 ? 64 : CW;       // its columns per group
        float m_run = -INFINITY, l = 0.0f;
        int done = 0;
        // After an abort (a bounded wait gave up) a split row's two threads
        // still pass the same pair barriers, tile by tile, so neither waits
        // for a partner that left; with whole rows the loop simply ends.
        bool alive = true;
        for (int jj = 0; jj < T; ++jj) {
            if (!alive) {
                pair_max(0.0f, jj);
                continue;
            }
            const int s = jj % NST;
            const int slot = t * NS + jj % NS;
            const uint32_t sp = (uint32_t)(jj / NS) & 1u;
            const int kt = j0 + jj;  // key tile
            const bool pre = kt < n_pre;
            const int key0 = pre ? kt * BN : (kt - n_pre) * BN;  // within its source
            const int nvalid = min(BN, (pre ? P : Sk()) - key0);
            const int kg0 = pre ? key0 : P + key0;  // over prefix + chunk
            // S, and the stage holding this tile's per-key K scales.  At D <= 128
            // that stage (with K) landed before its QK^T could run, so it is
            // waited first, while S is still being computed: a wait on a
            // completed barrier still costs ~100 cycles, kept off the path
            // from S to the softmax.
            bool ok;
            if constexpr (C::WIDE) {
                ok = wait_ab(bar(B_S_FULL + slot), sp, p.err, abort_flag);
                ok = ok && wait_ab(bar(B_V_FULL + jj % C::NSV), (uint32_t)(jj / C::NSV) & 1u, p.err,
                                   abort_flag);
            } else {
                ok = wait_ab(bar(B_KV_FULL + s), (uint32_t)(jj / NST) & 1u, p.err, abort_flag);
                ok = ok && wait_ab(bar(B_S_FULL + slot), sp, p.err, abort_flag);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if constexpr (SPLIT == 1) break;
                alive = false;
                pair_max(0.0f, jj);
                continue;
            }
            tc::fence_after();
            const uint32_t s_t = tmem + lane_base + C::COL_S + slot * BN;
            const uint8_t *ksc = C::WIDE ? sm + C::OFF_V + (jj % C::NSV) * C::VSB + C::KB
                                         : sm + C::OFF_ST + s * C::SB + 2 * C::KB;
            const float4 *ksc4 = reinterpret_cast<const float4 *>(ksc) + c0 / 4;
            uint32_t x[CW];
            if constexpr (CW >= 32) {
#pragma unroll
                for (int c = 0; c < CW / 32; ++c)
                    tc::ld32(s_t + c0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
            }
            tc::wait_ld();
            if (p.dbg) {
                // debug dump of the raw INT32 scores, re-read from TMEM in
                // 8-column pieces so that it adds no live registers here
                int32_t *dr = p.dbg + q_row_late(i) * p.dbg_stride;
#pragma unroll 1
                for (int c8 = 0; c8 < CW / 8; ++c8) {
                    uint32_t v[8];
                    tc::ld8(s_t + c0 + c8 * 8, v);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int c = c0 + c8 * 8 + e;
                        if (row_ok && c < nvalid && (!p.causal || kg0 + c <= lim))
                            dr[kg0 + c] = __float2int_rn(__uint_as_float(v[e]));
                    }
                }
            }
            // ---- the row max of the scaled scores
            const bool tmask = nvalid < BN || (p.causal && kg0 + BN - 1 > i_first + off);
            const bool uni = kuni && !pre && !tmask;
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            float kg[NG];
            if (uni) {
                // scale >= 0, so max(s) * k == max(s * k)
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    kg[g] = ksc4[16 * g].x;
                    float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                    for (int q = 0; q < GW / 8; ++q) {
                        const int c = GW * g + 8 * q;
                        a0 = fmax3(a0, __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
                        a1 = fmax3(a1, __uint_as_float(x[c + 2]), __uint_as_float(x[c + 3]));
                        a2 = fmax3(a2, __uint_as_float(x[c + 4]), __uint_as_float(x[c + 5]));
                        a3 = fmax3(a3, __uint_as_float(x[c + 6]), __uint_as_float(x[c + 7]));
                    }
                    m4[g] = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * kg[g];
                }
            } else if (!tmask) {
                // per-key scales: x <- s * k_scale in place
#pragma unroll
                for (int c4 = 0; c4 < CW / 4; ++c4) {
                    const float4 k = ksc4[c4];
                    const float2 z01 = fmul2(u2f2(x[4 * c4], x[4 * c4 + 1]), make_float2(k.x, k.y));
                    const float2 z23 = fmul2(u2f2(x[4 * c4 + 2], x[4 * c4 + 3]), make_float2(k.z, k.w));
                    x[4 * c4] = __float_as_uint(z01.x);
                    x[4 * c4 + 1] = __float_as_uint(z01.y);
                    x[4 * c4 + 2] = __float_as_uint(z23.x);
                    x[4 * c4 + 3] = __float_as_uint(z23.y);
                    m4[c4 & 1] = fmax3(m4[c4 & 1], z01.x, z01.y);
                    m4[2 + (c4 & 1)] = fmax3(m4[2 + (c4 & 1)], z23.x, z23.y);
                }
            } else {
                // keys [0, cl) of the tile count
                const int cl = (p.causal ? min(nvalid, lim - kg0 + 1) : nvalid) - c0;
#pragma unroll
                for (int c4 = 0; c4 < CW / 4; ++c4) {
                    const float4 k = ksc4[c4];
                    const float kk[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * c4 + e;
                        const float z = c < cl ? __uint_as_float(x[c]) * kk[e] : -INFINITY;
                        x[c] = __float_as_uint(z);
                        m4[e] = fmaxf(m4[e], z);
                    }
                }
            }
            const float mx = pair_max(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), jj);
            const float tb = pre ? 0.0f : bc;
            const float tmax = fmaf(mx, rq, tb);  // -inf when every key is masked (rq > 0)
            const float cand = fmaxf(m_run, tmax);
            const bool move = cand != -INFINITY && (m_run == -INFINITY || cand > m_run + 8.0f);
            float alpha = 1.0f;
            if (move) {
                alpha = m_run == -INFINITY ? 0.0f : exp2f(m_run - cand);
                l *= alpha;
                m_run = cand;
            }
            const bool fix = move && jj > 0 && alpha != 1.0f;
            if (__any_sync(0xffffffffu, fix)) {
                // O holds P.V of earlier tiles scaled to the old max: once the
                // last P.V retired, rescale this thread's columns of the row
                if constexpr (C::WIDE) {
                    // P.V(jj-1) frees its S slot when it retires; S(jj) alone
                    // does not imply it (QK(jj) did not wait for P.V(jj-1))
                    const bool w = wait_ab(bar(B_S_FREE + (jj - 1) % NS),
                                           (uint32_t)((jj - 1) / NS) & 1u, p.err, abort_flag);
                    if (!__all_sync(0xffffffffu, w)) {
                        if constexpr (SPLIT == 1) break;
                        alive = false;  // this tile's pair barrier is behind us
                        continue;
                    }
                }
                tc::fence_after();
                const float f = fix ? alpha : 1.0f;
                // 8-column pieces: the S row is live in registers here
#pragma unroll 1
                for (int c = hc * (D / 8 / SPLIT); c < (hc + 1) * (D / 8 / SPLIT); ++c) {
                    uint32_t o[8];
                    tc::ld8(tmem + lane_base + t * D + c * 8, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float2 v = fmul2(u2f2(o[e], o[e + 1]), make_float2(f, f));
                        o[e] = __float_as_uint(v.x);
                        o[e + 1] = __float_as_uint(v.y);
                    }
                    tc::st8(tmem + lane_base + t * D + c * 8, o);
                }
                tc::wait_st();
            }
            const float nb = tb - (m_run == -INFINITY ? 0.0f : m_run);
            // ---- P = 2^(z*rq + tb - m), packed f16 pairs over the S columns;
            // a 64-key part goes to the MMA as soon as it is stored
            float2 ls01 = make_float2(0.0f, 0.0f), ls23 = make_float2(0.0f, 0.0f);
            const float2 nb2 = make_float2(nb, nb);
            const float2 rq2 = make_float2(rq, rq);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const float2 kr2 = uni ? make_float2(kg[g] * rq, kg[g] * rq) : rq2;
                uint32_t pk[GW / 2];
#pragma unroll
                for (int q4 = 0; q4 < GW / 4; ++q4) {
                    const int c = GW * g + 4 * q4;
                    const float2 a01 = ffma2(u2f2(x[c], x[c + 1]), kr2, nb2);
                    const float2 a23 = ffma2(u2f2(x[c + 2], x[c + 3]), kr2, nb2);
                    const float2 p01 = make_float2(fast_exp2(a01.x), fast_exp2(a01.y));
                    const float2 p23 = make_float2(fast_exp2(a23.x), fast_exp2(a23.y));
                    ls01 = fadd2(ls01, p01);
                    ls23 = fadd2(ls23, p23);
                    pk[2 * q4] = pack2(p01.x, p01.y, false);
                    pk[2 * q4 + 1] = pack2(p23.x, p23.y, false);
                }
                const uint32_t pcol = s_t + (c0 + GW * g) / 2;
                if constexpr (GW == 64)
                    tc::st32(pcol, pk);
                else
                    tc::st16(pcol, *reinterpret_cast<uint32_t(*)[16]>(pk));
                tc::wait_st();
                tc::fence_before();
                if constexpr (C::WIDE) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_P_FULL + slot * C::NPH + (c0 + GW * g) / 64));
                } else {
                    mbar_arrive(bar(B_P_FULL + slot * C::NPH + (c0 + GW * g) / 64));
                }
            }
            l += (ls01.x + ls01.y) + (ls23.x + ls23.y);
            done = jj + 1;
        }
        // ------------------------------------------------ epilogue
        if constexpr (SPLIT > 1) {
            // the row's sum is the two halves' sums (same running max)
            float *rb = red + ((T & 1) * C::NSW + wg) * 128;
            rb[r] = l;
            pair_sync();
            l += red[((T & 1) * C::NSW + (wg ^ 1)) * 128 + r];
        }
        // with several S slots the last P.V may be in flight together with
        // earlier ones, and a parity wait on a per-tile barrier cannot tell
        // its last phase from two phases back, so the epilogue waits on a
        // barrier that completes exactly once
        bool have = done == T && T > 0;
        if (have) {
            const bool w = wait_ab(bar(B_O_FINAL + t), 0u, p.err, abort_flag);
            have = __all_sync(0xffffffffu, w);
            tc::fence_after();
        }
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        if (part >= 0) {
            // a part of a split query tile: its normalised O (f32, without
            // the smooth_v mean) and base-2 LSE, for the merge kernel; each
            // thread writes its row's channels straight from TMEM
            const int64_t slot = (int64_t)blockIdx.x - p.split_f;
            constexpr int NPC = D / 32 / SPLIT;  // 32-channel pieces of this thread
            float *po = p.part_o + (slot * 128 + r) * D + hc * NPC * 32;
#pragma unroll 1
            for (int c = 0; c < NPC; ++c) {
                uint32_t o[32];
                if (have) {
                    tc::ld32(tmem + lane_base + t * D + (hc * NPC + c) * 32, o);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                float4 *d4 = reinterpret_cast<float4 *>(po + c * 32);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    d4[q] = make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                        __uint_as_float(o[4 * q + 2]) * inv,
                                        __uint_as_float(o[4 * q + 3]) * inv);
            }
            if (hc == 0) p.part_lse[slot * 128 + r] = l > 0.0f ? m_run + log2f(l) : -INFINITY;
        } else {
            const int64_t orow = q_row_late(i);
            // smooth_v: the V mean goes back onto rows that saw a key
            const float *vmu = (p.v_mean && l > 0.0f) ? v_mean_late() : nullptr;
            // The O rows go out through shared memory: each warp stages its 32
            // rows, 64 channels at a time, then stores 4 rows' 128-byte pieces
            // per instruction (one row per thread made every store instruction
            // touch 32 rows, most of the epilogue's time).  The staging space is
            // this tile's Q tile (not read since its last QK^T, which retired
            // before the last P.V) or, with one query tile, the key ring (every
            // MMA has retired by now); 16-byte pieces XOR-swizzled by row.
            const int i_w0 = i - lane;  // this warp's first row (rows are consecutive)
            const int64_t ostride = (VL || p.nhd) ? (int64_t)p.Hq * D : (int64_t)D;  // between rows
            uint16_t *obase0 = reinterpret_cast<uint16_t *>(p.out) + out_row_late(i_w0) * D;
            uint8_t *ost = (NQ > 1 ? sm + t * C::QB + (warp & 3) * 4096 : sm + C::OFF_ST + warp * 4096);
            const int nrow_w = min(32, Sq() - i_w0);  // rows of this warp inside the sequence
            // two 32-column pieces of O per tensor-memory round trip
            constexpr int NCH = D / 32 / SPLIT;
            static_assert(NCH % 2 == 0, "O pieces go in pairs");
#pragma unroll 1
            for (int c2 = 0; c2 < NCH; c2 += 2) {
                uint32_t oo[2][32];
                if (have) {
                    tc::ld32(tmem + lane_base + t * D + (hc * NCH + c2) * 32, oo[0]);
                    tc::ld32(tmem + lane_base + t * D + (hc * NCH + c2 + 1) * 32, oo[1]);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) oo[0][e] = oo[1][e] = 0u;
                }
                uint32_t pk[32];  // this row's 64 channels, f16 / bf16 pairs
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint32_t(&o)[32] = oo[h2];
                    if (vmu) {
                        const float4 *m4 = reinterpret_cast<const float4 *>(vmu + (hc * NCH + c2 + h2) * 32);
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float4 m = m4[e / 2];
                            const float2 v0 = ffma2(u2f2(o[2 * e], o[2 * e + 1]), make_float2(inv, inv),
                                                    make_float2(m.x, m.y));
                            const float2 v1 = ffma2(u2f2(o[2 * e + 2], o[2 * e + 3]),
                                                    make_float2(inv, inv), make_float2(m.z, m.w));
                            pk[h2 * 16 + e] = pack2(v0.x, v0.y, p.out_bf16 != 0);
                            pk[h2 * 16 + e + 1] = pack2(v1.x, v1.y, p.out_bf16 != 0);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 v = fmul2(u2f2(o[2 * e], o[2 * e + 1]), make_float2(inv, inv));
                            pk[h2 * 16 + e] = pack2(v.x, v.y, p.out_bf16 != 0);
                        }
                    }
                }
                __syncwarp();  // the previous pair's staged rows have been read
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4 *>(ost + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                __syncwarp();
                const int j = lane & 7;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = (lane >> 3) + 4 * k;
                    if (rr < nrow_w) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(ost + rr * 128 + ((j ^ (rr & 7)) << 4));
                        *reinterpret_cast<uint4 *>(obase0 + rr * ostride + (hc * NCH + c2) * 32 + j * 8) = v;
                    }
                }
            }
            if (row_ok && p.lse && hc == 0)
                p.lse[orow] = l > 0.0f ? (m_run + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == kMma) {
        tc::fence_after();
        tc::dealloc(tmem, 512);
    }
}

// Merge of a split query tile's parts (dense form, D = 256): one warp per
// row, CPL channels per lane.  With lse_j the parts' base-2 LSEs and M their
// maximum, o = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M) (the parts' O
// are normalised by their own sums), plus the smooth_v mean on rows that saw
// a key, and lse = (M + log2 sum_j 2^(lse_j - M)) ln 2: the attention over
// the union of the parts' keys (the split-K combine of "INT8 QK MMAC on
// gfx936 DCU", section 4, over key ranges of a prefill tile).
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int CPL = D / 32;
    static_assert(CPL == 8, "one 16-byte output store per lane");
    // launched behind the attention kernel: its partial results are read
    // only after that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * 8 + warp;  // (split tile, row)
    if (g >= (int64_t)p.split_tail * 128) return;
    const int u = (int)(g >> 7), r = (int)(g & 127);
    int ct;
    const int pair = dense_tile(p, 128, p.split_f + u, ct);
    const int i = ct * 128 + r;
    if (i >= p.Sq) return;
    const int64_t slot0 = (int64_t)u * p.split_k;
    float M = -INFINITY;
    for (int j = 0; j < p.split_k; ++j) M = fmaxf(M, p.part_lse[(slot0 + j) * 128 + r]);
    float acc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = 0.0f;
    float W = 0.0f;
    if (M != -INFINITY) {
        for (int j = 0; j < p.split_k; ++j) {
            const float lj = p.part_lse[(slot0 + j) * 128 + r];
            if (lj == -INFINITY) continue;  // no key of this part visible to the row
            const float w = exp2f(lj - M);
            W += w;
            const float4 *src =
                reinterpret_cast<const float4 *>(p.part_o + ((slot0 + j) * 128 + r) * D + lane * CPL);
#pragma unroll
            for (int q = 0; q < CPL / 4; ++q) {
                const float4 v = src[q];
                acc[4 * q] = fmaf(w, v.x, acc[4 * q]);
                acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
            }
        }
    }
    const float inv = W > 0.0f ? 1.0f / W : 0.0f;
    const int b = pair / p.Hq, hq = pair - b * p.Hq;
    const float *vmu = (p.v_mean && W > 0.0f)
                           ? p.v_mean + ((int64_t)b * p.Hkv + hq / p.group) * D + lane * CPL
                           : nullptr;
    uint32_t pk[CPL / 2];
#pragma unroll
    for (int e = 0; e < CPL / 2; ++e) {
        const float m0 = vmu ? vmu[2 * e] : 0.0f, m1 = vmu ? vmu[2 * e + 1] : 0.0f;
        pk[e] = pack2(fmaf(acc[2 * e], inv, m0), fmaf(acc[2 * e + 1], inv, m1), p.out_bf16 != 0);
    }
    const int64_t orow = p.nhd ? ((int64_t)b * p.Sq + i) * p.Hq + hq : (int64_t)pair * p.Sq + i;
    *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) + orow * D + lane * CPL) =
        make_uint4(pk[0], pk[1], pk[2], pk[3]);
    if (p.lse && lane == 0)
        p.lse[(int64_t)pair * p.Sq + i] = W > 0.0f ? (M + log2f(W)) * 0.69314718055994530942f : -INFINITY;
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

// [B][Sk][Hkv][D] f16 (NHD) as dims (channel, kv head, token, batch) with
// increasing strides, boxes of 64 channels x 1 head x BN tokens (the same
// shared-memory tile as the 3-D map's), 128-byte swizzle; tokens past Sk
// read as zero.
template <int D>
bool make_map_nhd(CUtensorMap *tm, const void *base, uint64_t sk, uint64_t hkv, uint64_t batch) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)sk, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2,
                             (cuuint64_t)sk * hkv * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)PCfg<D>::BN, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*Hkv][rows][D] f16, boxes of 64 channels x BN rows, 128-byte swizzle;
// rows past `rows` read as zero.
template <int D>
bool make_map(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t bh) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)PCfg<D>::BN, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool VL, bool PR = false>
cudaError_t launch_dv(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    using C = PCfg<D>;
    if (p.BN != C::BN) return cudaErrorInvalidValue;
    if (!encode_fn()) return cudaErrorNotSupported;
    PrefillMaps m;
    memset(&m, 0, sizeof(m));
    // staged keys per (batch, kv head), or per kv head for a packed batch
    const uint64_t bh = p.cu_q ? (uint64_t)p.Hkv : (uint64_t)p.B * p.Hkv;
    if (!make_map<D>(&m.k, p.k_ws, p.Lpad, bh)) return cudaErrorInvalidValue;
    if (p.Vrows > 0 && !make_map<D>(&m.v_pre, p.v_ws, p.Vrows, bh)) return cudaErrorInvalidValue;
    if (p.Sk > 0) {
        if (p.v_bf16 || p.cu_q || p.v_mean) {
            m.v_ch = m.v_pre;
        } else if (p.nhd) {
            if (!make_map_nhd<D>(&m.v_ch, p.v, p.Sk, p.Hkv, p.B)) return cudaErrorInvalidValue;
            m.v_ch_4d = 1;
        } else if (!make_map<D>(&m.v_ch, p.v, p.Sk, bh)) {
            return cudaErrorInvalidValue;
        }
    }
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, VL, PR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // packed batches: one CTA per (compact tile slot, head) -- ceil(len_b /
    // QR) slots per sequence, at most total_q / QR + B -- heads fastest
    constexpr int QR = 128 * C::NQ;
    // PR: 128 rows of two heads (sharing a KV head) per CTA
    if (PR && (p.group % 2 != 0 || p.Hq % 2 != 0)) return cudaErrorInvalidValue;
    const int64_t vl_ctas =
        VL ? (p.total_q / (PR ? 128 : QR) + p.B) * (int64_t)(PR ? p.Hq / 2 : p.Hq) : 0;
    if (vl_ctas > 0x7fffffff) return cudaErrorInvalidValue;
    // dense form at D = 256: CTAs of whole query tiles, then the split tail's parts
    const int64_t dense_ctas = (int64_t)(p.Sq + QR - 1) / QR * p.Hq * p.B;
    const bool split = !VL && C::WIDE && p.split_k > 0;
    if (!split && p.split_k != 0) return cudaErrorInvalidValue;
    if (split && (p.split_k > 64 || p.split_tail < 1 ||
                  (int64_t)p.split_f + p.split_tail != dense_ctas || !p.part_o || !p.part_lse))
        return cudaErrorInvalidValue;
    const int64_t ctas = VL ? vl_ctas : split ? p.split_f + (int64_t)p.split_tail * p.split_k : dense_ctas;
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)ctas, 1, 1);
    if (!VL && (p.bundle < 1 || p.bundle > p.B * p.Hq)) return cudaErrorInvalidValue;
    // programmatic dependent launches: the attention kernel behind the
    // staging pass, the merge behind the attention kernel; each waits on the
    // device before reading what the grid ahead of it wrote.  The staging
    // pass lets its dependent start once every staging CTA has started; the
    // attention kernel does not signal early (a trigger at CTA start made
    // the dense launch 0.7 % slower), so the merge is released when the
    // attention grid completes and only its launch overlaps.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_kernel<D, VL, PR>, p, m);
    log.add(VL ? "prefill_varlen_kernel" : "prefill_kernel", grid, dim3(C::THREADS), dim3(1, 1, 1),
            C::SMEM);
    if constexpr (!VL && C::WIDE) {
        if (split && e == cudaSuccess) {
            cfg.gridDim = dim3((unsigned)(((int64_t)p.split_tail * 128 + 7) / 8), 1, 1);
            cfg.blockDim = dim3(256, 1, 1);
            cfg.dynamicSmemBytes = 0;
            e = cudaLaunchKernelEx(&cfg, prefill_merge_kernel<D>, p);
            ++log.count;  // the attention kernel stays the recorded launch
        }
    }
    return e;
}

template <int D>
cudaError_t launch_d(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    if (!p.cu_q) return launch_dv<D, false>(p, st, log);
    if constexpr (PCfg<D>::NQ == 2) {
        if (p.vl_pairs) return launch_dv<D, true, true>(p, st, log);
    }
    return p.vl_pairs ? cudaErrorInvalidValue : launch_dv<D, true>(p, st, log);
}

}  // namespace

PrefillSplit prefill_split(int B, int Hq, int Sq, int D, int keys, bool causal, int sms) {
    PrefillSplit s = {0, 0, 0};
    if (D != 256 || sms < 1 || keys < 1 || Sq < 1) return s;
    const int64_t tiles = (int64_t)((Sq + 127) / 128) * B * Hq;  // one 128-row query tile per CTA
    const int64_t tail = tiles % sms;                             // CTAs of the last, partial wave
    if (tail == 0 || tiles > 0x3fffffff) return s;
    // key tiles of a query tile: at most T; causal rows see fewer, the first
    // query tile at least Tmin.  The model below assumes tiles of about
    // equal work (a chunk over a long prefix, or no mask).
    const int T = (keys + 63) / 64;
    const int Tmin = causal ? (keys - Sq + 128 > 0 ? (keys - Sq + 128) / 64 : 0) : T;
    if (4 * Tmin < 3 * T) return s;
    // In units of one query tile's time: k parts of a tail tile run in
    // ceil(tail * k / sms) rounds, each costing 1/k of a tile plus a fixed
    // start-up and drain of about 8 key tiles' time; parts of at least 16
    // key tiles; a split must save 5 %.
    const double fixed = 8.0 / Tmin;
    double best = 1.0 + fixed;
    int bk = 1;
    for (int k = 2; k <= 8 && Tmin / k >= 16; ++k) {
        const double c = (double)((tail * k + sms - 1) / sms) * (1.0 / k + fixed);
        if (c < 0.95 * best) best = c, bk = k;
    }
    if (bk > 1) s = {(int)(tiles - tail), (int)tail, bk};
    return s;
}

int prefill_bundle(int B, int Hq, int group, int rows, int D) {
    constexpr double kL2Share = 32.0 * 1024 * 1024;  // of the 126 MB L2 (16-96 MB swept)
    const double kv = (double)rows * D * 2 * 2;       // f16 K and V of one KV head
    int kvh = kv > 0 ? (int)(kL2Share / kv) : 1;
    kvh = kvh < 1 ? 1 : kvh;
    const long long n = (long long)kvh * group;
    const long long pairs = (long long)B * Hq;
    return (int)(n < pairs ? n : pairs);
}

cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t st, LaunchLog &log) {
    switch (p.D) {
        case 64: return launch_d<64>(p, st, log);
        case 128: return launch_d<128>(p, st, log);
        case 256: return launch_d<256>(p, st, log);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace sage
