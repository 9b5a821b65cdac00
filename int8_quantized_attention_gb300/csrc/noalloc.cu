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

// Bytes of built-in scratch a call with S segments uses: the fp32 partial
// outputs [B*Hq, S, D] (256-byte aligned end) and partial LSEs [B*Hq, S].
static size_t scratch_bytes(const sage_decode_args_t *a, int S) {
    if (S <= 1) return 0;
    const size_t rows = (size_t)a->B * a->Hq * S;
    return ((rows * a->D * sizeof(float) + 255) & ~(size_t)255) + rows * sizeof(float);
}

SAGE_API sage_status_t sage_attn_decode_paged_noalloc(const sage_decode_args_t *a, void *stream) {
    using sage::report_error;
    sage::record_launch(sage::LaunchLog());  // nothing launched by this call yet
    // the same checks as the workspace entry point (shapes, alignment, and
    // q / q_scale / block_table / context_lens / out / lse reachable by the GPU)
    const sage_status_t chk = (sage_status_t)sage::check_decode_args(a, nullptr);
    if (chk != SAGE_OK || a->B == 0) return chk;

    const int pages = (a->max_context_len + 15) / 16;
    const int cap = sage::decode_max_segment_pages();
    const int s_min = pages > cap ? (pages + cap - 1) / cap : 1;  // segments of <= cap pages
    int S = a->num_segments;
    if (S == 0) {
        // the library's choice for these buffers, lowered to the largest
        // count whose partials fit the scratch (never below s_min)
        S = sage_decode_auto_segments(a, nullptr);
        while (S > s_min && scratch_bytes(a, S) > kNoallocScratchBytes) --S;
    }
    if (S < s_min) S = s_min;
    const int pps = pages > 0 ? (pages + S - 1) / S : 1;
    S = pages > 0 ? (pages + pps - 1) / pps : 1;
    const size_t need = scratch_bytes(a, S);
    const size_t o_bytes = S > 1 ? ((size_t)a->B * a->Hq * S * a->D * sizeof(float) + 255) &
                                       ~(size_t)255
                                 : 0;
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
    p.max_pages = pages;
    p.max_ctx = a->max_context_len;
    p.pv_mode = a->pv_mode;
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
