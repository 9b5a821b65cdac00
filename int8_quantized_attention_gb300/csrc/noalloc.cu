// sage_attn_decode_paged_noalloc: the split-K paged decode for callers that
// cannot allocate device memory themselves -- code running inside a CUDA
// graph that is being captured with a fixed memory plan, plugins whose host
// framework owns every allocation, or embedders whose allocator must not be
// re-entered from the attention call.  The regular entry point needs a
// caller-provided workspace for the per-segment partial results; this
// variant keeps them in one statically sized device array that lives in the
// library image instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library reserves kNoallocScratchBytes for it until the process exits.
// Host code cannot use the array's name as a device address; its address is
// looked up once per device with cudaGetSymbolAddress and handed to the
// kernels as a plain pointer.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sage_attn.h"

#define SAGE_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;  // 8 MiB of fp32 partials
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array; the first call on a device
// performs the lookup (that call should therefore not be made while the
// stream is being captured).
sage_status_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return (sage_status_t)sage::report_error(SAGE_ERR_CUDA, "cudaGetDevice: %s",
                                                 cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return (sage_status_t)sage::report_error(SAGE_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return (sage_status_t)sage::report_error(
                SAGE_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SAGE_OK;
}

}  // namespace

SAGE_API size_t sage_attn_decode_noalloc_max_bytes(void) { return kNoallocScratchBytes; }

SAGE_API sage_status_t sage_attn_decode_paged_noalloc(const sage_decode_args_t *a, void *stream) {
    using sage::report_error;
    if (!a) return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG, "args is NULL");
    if (a->D != 64 && a->D != 128 && a->D != 256)
        return (sage_status_t)report_error(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}",
                                           a->D);
    if (a->out_dtype != SAGE_F16 && a->out_dtype != SAGE_BF16)
        return (sage_status_t)report_error(SAGE_ERR_UNSUPPORTED, "out dtype must be f16 or bf16");
    if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv)
        return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG,
                                           "need Hq a positive multiple of Hkv (Hq=%d Hkv=%d)",
                                           a->Hq, a->Hkv);
    if (a->max_context_len < 0 || a->max_blocks < 0 ||
        (int64_t)a->max_context_len > 16ll * a->max_blocks)
        return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG,
                                           "max_context_len %d exceeds 16 * max_blocks (%d)",
                                           a->max_context_len, a->max_blocks);
    if (a->num_segments < 0 || a->num_segments > 1024)
        return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG, "num_segments outside [0, 1024]");
    if (a->B == 0) return SAGE_OK;
    if (!a->q || !a->q_scale || !a->context_lens || !a->out)
        return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG,
                                           "q, q_scale, context_lens and out are required");
    if (a->max_context_len > 0) {
        if (!a->k_cache || !a->v_cache || !a->k_scale || !a->v_scale || !a->block_table)
            return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG,
                                               "cache, scales and block_table are required");
        if (a->num_blocks < 1)
            return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG, "num_blocks must be >= 1");
        if ((reinterpret_cast<uintptr_t>(a->k_cache) | reinterpret_cast<uintptr_t>(a->v_cache) |
             reinterpret_cast<uintptr_t>(a->k_scale) | reinterpret_cast<uintptr_t>(a->v_scale)) & 15)
            return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG,
                                               "caches and scales must be 16-byte aligned");
    }
    if (reinterpret_cast<uintptr_t>(a->q) & 3)
        return (sage_status_t)report_error(SAGE_ERR_INVALID_ARG, "q must be 4-byte aligned");

    int S = a->num_segments ? a->num_segments
                            : sage_decode_num_segments(a->B, a->Hq, a->Hkv, a->D,
                                                       a->max_context_len);
    const int pages = (a->max_context_len + 15) / 16;
    {   // a segment is at most decode_max_segment_pages() pages long
        const int cap = sage::decode_max_segment_pages();
        if ((int64_t)S * cap < pages) S = (pages + cap - 1) / cap;
    }
    const int pps = pages > 0 ? (pages + S - 1) / S : 1;
    S = pages > 0 ? (pages + pps - 1) / pps : 1;
    const size_t rows = (size_t)a->B * a->Hq * S;
    const size_t o_bytes = (rows * a->D * sizeof(float) + 255) & ~(size_t)255;
    const size_t need = S > 1 ? o_bytes + rows * sizeof(float) : 0;
    if (need > kNoallocScratchBytes)
        return (sage_status_t)report_error(
            SAGE_ERR_INVALID_ARG,
            "decode partials need %zu bytes (B=%d Hq=%d D=%d segments=%d) but the built-in "
            "scratch holds %zu; pass fewer segments or use sage_attn_decode_paged",
            need, a->B, a->Hq, a->D, S, kNoallocScratchBytes);

    int *ew = nullptr;
    sage_status_t st = (sage_status_t)sage::device_error_word(&ew);
    if (st != SAGE_OK) return st;
    void *scratch = nullptr;
    if (S > 1) {
        st = scratch_address(&scratch);
        if (st != SAGE_OK) return st;
    }
    sage::DecodeParams p = {};
    p.q = a->q, p.q_scale = a->q_scale;
    p.k_cache = a->k_cache, p.v_cache = a->v_cache, p.k_scale = a->k_scale, p.v_scale = a->v_scale;
    p.block_table = a->block_table, p.context_lens = a->context_lens;
    p.B = a->B, p.Hq = a->Hq, p.Hkv = a->Hkv, p.D = a->D, p.group = a->Hq / a->Hkv;
    p.head_tiles = (p.group + 7) / 8;
    p.num_blocks = a->num_blocks, p.max_blocks = a->max_blocks;
    p.num_segments = S, p.pages_per_seg = pps;
    p.max_ctx = a->max_context_len;
    const float sm = a->sm_scale > 0.0f ? a->sm_scale : 1.0f / sqrtf((float)a->D);
    p.qk_scale_log2 = sm * 1.4426950408889634f;
    p.out = a->out, p.out_bf16 = a->out_dtype == SAGE_BF16, p.lse = a->lse;
    p.err = ew;
    if (S > 1) {
        // every (row, segment) slot of both arrays is written by the decode
        // kernel before the combine reads it: nothing needs clearing
        p.o_part = static_cast<float *>(scratch);
        p.lse_part = reinterpret_cast<float *>(static_cast<char *>(scratch) + o_bytes);
    }
    sage::LaunchLog log;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = sage::launch_decode(p, cs, log);
    if (e != cudaSuccess)
        return (sage_status_t)report_error(SAGE_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    if (S > 1) {
        sage::LaunchLog tmp = log;
        sage::CombineParams c = {p.o_part, p.lse_part, a->B * a->Hq, S, a->D, a->out, p.out_bf16,
                                 a->lse, 1};
        e = sage::launch_combine(c, cs, tmp);
        if (e != cudaSuccess)
            return (sage_status_t)report_error(SAGE_ERR_CUDA, "combine launch: %s",
                                               cudaGetErrorString(e));
        log.count = tmp.count;
    }
    sage::record_launch(log);
    return SAGE_OK;
}
