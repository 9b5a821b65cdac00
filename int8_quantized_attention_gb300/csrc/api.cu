// C-ABI host layer of libsageattn.so: argument validation, launch
// configuration, the per-device error word and the launch record.
// Every entry point is declared (and documented) in include/sage_attn.h.
#include <math.h>

#include <cmath>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "sage_attn.h"

#define SAGE_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_msg;
thread_local sage::LaunchLog g_last;

// Error word of the device (bit set of sage::kErrTimeout / kErrBadBlock).
__device__ int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_err_ptr[kMaxDevices] = {};

sage_status_t fail(sage_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_msg = buf;
    return s;
}

sage_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(SAGE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device address of this device's error word (looked up once per device).
sage_status_t error_word(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SAGE_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        g_err_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_err_ptr[dev];
    return SAGE_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A per-step input or output of decode may live in device memory or in
// pinned host memory that the GPU reaches at the same address (GB300: the
// kernels read and write it over NVLink-C2C, no copy-engine transfer).
// Anything else (pageable host memory, a foreign pointer) is rejected here
// rather than faulting on the device.
sage_status_t check_reachable(const void *ptr, const char *name) {
    if (!ptr) return SAGE_OK;
    cudaPointerAttributes at = {};
    const cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SAGE_ERR_INVALID_ARG, "%s: not memory the GPU can reach (%s)", name,
                    cudaGetErrorString(e));
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return SAGE_OK;
    if (at.type == cudaMemoryTypeHost && at.devicePointer == ptr) return SAGE_OK;
    return fail(SAGE_ERR_INVALID_ARG, "%s: must be device memory or mapped pinned host memory",
                name);
}
// True when `ptr` is pinned host memory (checked reachable beforehand).
bool is_host_memory(const void *ptr) {
    if (!ptr) return false;
    cudaPointerAttributes at = {};
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

int ilog2_exact(int x) {
    int s = 0;
    while ((1 << s) < x) ++s;
    return (1 << s) == x ? s : -1;
}

__global__ void timeout_probe_kernel(long long limit_ns, int *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        sage::mbar_init(sage::smem_u32(&bar), 1);
        sage::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    // Nothing ever arrives on `bar`: the wait must give up on its own.
    const unsigned long long t0 = sage::global_timer_ns();
    while (!sage::mbar_try_wait(sage::smem_u32(&bar), 0)) {
        if ((long long)(sage::global_timer_ns() - t0) > limit_ns) {
            atomicOr(err, sage::kErrTimeout);
            return;
        }
    }
}

}  // namespace

namespace sage {
int report_error(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_msg = buf;
    return status;
}
int device_error_word(int **out) { return (int)error_word(out); }
void record_launch(const LaunchLog &log) { g_last = log; }
}  // namespace sage

// ---------------------------------------------------------------------------

SAGE_API const char *sage_get_last_error_message(void) { return g_msg.c_str(); }

SAGE_API int sage_version(void) { return 7; }

SAGE_API sage_status_t sage_last_launch_info(sage_launch_info_t *info) {
    if (!info) return fail(SAGE_ERR_INVALID_ARG, "info is NULL");
    memset(info, 0, sizeof(*info));
    strncpy(info->kernel, g_last.kernel, sizeof(info->kernel) - 1);
    info->grid[0] = g_last.grid.x, info->grid[1] = g_last.grid.y, info->grid[2] = g_last.grid.z;
    info->block[0] = g_last.block.x, info->block[1] = g_last.block.y,
    info->block[2] = g_last.block.z;
    info->cluster[0] = g_last.cluster.x, info->cluster[1] = g_last.cluster.y,
    info->cluster[2] = g_last.cluster.z;
    info->smem_bytes = g_last.smem;
    info->num_segments = g_last.segments;
    info->launches = g_last.count;
    return SAGE_OK;
}

SAGE_API sage_status_t sage_check_device_status(void *stream, int *detail) {
    int *ew = nullptr;
    sage_status_t s = error_word(&ew);
    if (s != SAGE_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int word = 0;
    e = cudaMemcpy(&word, ew, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    e = cudaMemset(ew, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
    if (detail) *detail = word;
    if (word & sage::kErrBadBlock)
        return fail(SAGE_ERR_BAD_BLOCK, "a block-table entry or context length was out of range");
    if (word & sage::kErrTimeout) return fail(SAGE_ERR_TIMEOUT, "a bounded device wait ran out");
    return SAGE_OK;
}

SAGE_API sage_status_t sage_debug_timeout_probe(int timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 5000000)
        return fail(SAGE_ERR_INVALID_ARG, "timeout_us must be in [1, 5e6]");
    int *ew = nullptr;
    sage_status_t s = error_word(&ew);
    if (s != SAGE_OK) return s;
    g_last = sage::LaunchLog();
    timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (long long)timeout_us * 1000ll, ew);
    g_last.add("timeout_probe_kernel", dim3(1), dim3(32), dim3(1, 1, 1), 0);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "timeout probe launch");
}

// ------------------------------------------------------------------ quant

SAGE_API sage_status_t sage_quant_int8(const void *x, sage_dtype_t dtype, int B, int H, int S,
                                       int D, int64_t stride_b, int64_t stride_h,
                                       int64_t stride_s, int block_tokens, int smooth,
                                       const float *mu_in, int mu_heads, int8_t *x_int8,
                                       float *scale, float *mu_out, float *bias_out,
                                       void *stream) {
    if (dtype != SAGE_F16 && dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "x dtype must be f16 or bf16");
    if (!head_dim_ok(D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", D);
    if (B < 0 || H < 0 || S < 0) return fail(SAGE_ERR_INVALID_ARG, "negative shape");
    if (block_tokens < 1 || block_tokens > 1024)
        return fail(SAGE_ERR_INVALID_ARG, "block_tokens %d outside [1, 1024]", block_tokens);
    g_last = sage::LaunchLog();
    if ((int64_t)B * H * S == 0) return SAGE_OK;
    if (!x || !x_int8 || !scale) return fail(SAGE_ERR_INVALID_ARG, "x, x_int8 and scale are required");
    if (!aligned(x, 16)) return fail(SAGE_ERR_INVALID_ARG, "x must be 16-byte aligned");
    if (!aligned(x_int8, 8)) return fail(SAGE_ERR_INVALID_ARG, "x_int8 must be 8-byte aligned");
    if (stride_b % 8 || stride_h % 8 || stride_s % 8)
        return fail(SAGE_ERR_INVALID_ARG, "strides must be multiples of 8 elements");
    if (smooth && !mu_out) return fail(SAGE_ERR_INVALID_ARG, "smooth needs mu_out");
    if ((smooth && !aligned(mu_out, 16)) || (mu_in && !aligned(mu_in, 16)))
        return fail(SAGE_ERR_INVALID_ARG, "mu_out and mu_in must be 16-byte aligned");
    if (smooth && (int64_t)B * H > 65535)
        return fail(SAGE_ERR_UNSUPPORTED, "smooth supports at most 65535 (batch, head) pairs");
    if (mu_in) {
        if (!bias_out) return fail(SAGE_ERR_INVALID_ARG, "mu_in needs bias_out");
        if (mu_heads < 1 || H % mu_heads)
            return fail(SAGE_ERR_INVALID_ARG, "H (%d) must be a multiple of mu_heads (%d)", H,
                        mu_heads);
    }
    sage::QuantParams p = {};
    p.x = x;
    p.bf16 = dtype == SAGE_BF16;
    p.B = B, p.H = H, p.S = S, p.D = D;
    p.sb = stride_b, p.sh = stride_h, p.ss = stride_s;
    p.block = block_tokens;
    p.smooth = smooth;
    p.mu_bias = mu_in;
    p.mu_heads = mu_in ? mu_heads : 1;
    p.q = x_int8;
    p.scale = scale;
    p.mu_out = mu_out;
    p.bias = mu_in ? bias_out : nullptr;
    cudaError_t e = sage::launch_quant(p, static_cast<cudaStream_t>(stream), g_last);
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "quant launch");
}

SAGE_API int64_t sage_varlen_scale_groups(int64_t total, int B, int block_tokens) {
    if (total < 0 || B < 0 || block_tokens < 1) return 0;
    return block_tokens == 1 ? total : total / block_tokens + B;
}

SAGE_API sage_status_t sage_quant_int8_varlen(const void *x, sage_dtype_t dtype, int B, int H,
                                              int64_t total, int D, int64_t stride_h,
                                              int64_t stride_t, const int32_t *cu_seqlens,
                                              int max_seqlen, int block_tokens, int smooth,
                                              const float *mu_in, int mu_heads, int8_t *x_int8,
                                              float *scale, float *mu_out, float *bias_out,
                                              void *stream) {
    if (dtype != SAGE_F16 && dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "x dtype must be f16 or bf16");
    if (!head_dim_ok(D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", D);
    if (B < 0 || H < 0 || total < 0 || max_seqlen < 0)
        return fail(SAGE_ERR_INVALID_ARG, "negative shape");
    if (block_tokens < 1 || block_tokens > 1024)
        return fail(SAGE_ERR_INVALID_ARG, "block_tokens %d outside [1, 1024]", block_tokens);
    g_last = sage::LaunchLog();
    if ((int64_t)B * H == 0 || total == 0) return SAGE_OK;
    if (!x || !x_int8 || !scale || !cu_seqlens)
        return fail(SAGE_ERR_INVALID_ARG, "x, x_int8, scale and cu_seqlens are required");
    if (!aligned(x, 16)) return fail(SAGE_ERR_INVALID_ARG, "x must be 16-byte aligned");
    if (!aligned(x_int8, 8)) return fail(SAGE_ERR_INVALID_ARG, "x_int8 must be 8-byte aligned");
    if (stride_h % 8 || stride_t % 8)
        return fail(SAGE_ERR_INVALID_ARG, "strides must be multiples of 8 elements");
    if (smooth && !mu_out) return fail(SAGE_ERR_INVALID_ARG, "smooth needs mu_out");
    if ((smooth && !aligned(mu_out, 16)) || (mu_in && !aligned(mu_in, 16)))
        return fail(SAGE_ERR_INVALID_ARG, "mu_out and mu_in must be 16-byte aligned");
    if (smooth && (int64_t)B * H > 65535)
        return fail(SAGE_ERR_UNSUPPORTED, "smooth supports at most 65535 (sequence, head) pairs");
    if (mu_in) {
        if (!bias_out) return fail(SAGE_ERR_INVALID_ARG, "mu_in needs bias_out");
        if (mu_heads < 1 || H % mu_heads)
            return fail(SAGE_ERR_INVALID_ARG, "H (%d) must be a multiple of mu_heads (%d)", H,
                        mu_heads);
    }
    const int64_t groups = sage_varlen_scale_groups(total, B, block_tokens);
    if ((int64_t)H * groups > 0x7fffffffll)
        return fail(SAGE_ERR_UNSUPPORTED, "too many scale groups");
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::QuantParams p = {};
    p.x = x;
    p.bf16 = dtype == SAGE_BF16;
    p.B = B, p.H = H, p.S = max_seqlen, p.D = D;
    p.sb = 0, p.sh = stride_h, p.ss = stride_t;
    p.block = block_tokens;
    p.smooth = smooth;
    p.mu_bias = mu_in;
    p.mu_heads = mu_in ? mu_heads : 1;
    p.q = x_int8;
    p.scale = scale;
    p.mu_out = mu_out;
    p.bias = mu_in ? bias_out : nullptr;
    p.cu = cu_seqlens;
    p.total = total;
    p.groups = groups;
    p.err = ew;
    cudaError_t e = sage::launch_quant(p, static_cast<cudaStream_t>(stream), g_last);
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "varlen quant launch");
}

// ---------------------------------------------------------------- combine

static sage_status_t check_combine(const float *o_part, const float *lse_part, int R, int S, int D,
                                   const void *out, sage_dtype_t out_dtype) {
    if (!head_dim_ok(D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", D);
    if (out_dtype != SAGE_F16 && out_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "out dtype must be f16 or bf16");
    if (R < 0 || S < 1 || S > 1024) return fail(SAGE_ERR_INVALID_ARG, "need R >= 0, 1 <= S <= 1024");
    if (R > 0 && (!o_part || !lse_part || !out))
        return fail(SAGE_ERR_INVALID_ARG, "o_part, lse_part and out are required");
    if (!aligned(o_part, 8)) return fail(SAGE_ERR_INVALID_ARG, "o_part must be 8-byte aligned");
    return SAGE_OK;
}

SAGE_API sage_status_t sage_splitk_combine(const float *o_part, const float *lse_part, int R,
                                           int S, int D, void *out, sage_dtype_t out_dtype,
                                           float *lse_out, void *stream) {
    sage_status_t s = check_combine(o_part, lse_part, R, S, D, out, out_dtype);
    if (s != SAGE_OK) return s;
    g_last = sage::LaunchLog();
    sage::CombineParams p = {o_part, lse_part, R, S, D, out, out_dtype == SAGE_BF16, lse_out};
    cudaError_t e = sage::launch_combine(p, static_cast<cudaStream_t>(stream), g_last);
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "combine launch");
}

// ----------------------------------------------------------------- decode

// Segment count for a decode call.  `per_sm_x16` is 16 times the CTAs per
// SM the single-wave choice aims at: 40 (2.5 per SM) when the per-step
// inputs and outputs are in device memory, 27 (about 1.7) when they are in
// pinned host memory -- there every segment's CTA reads its query and table
// slice across NVLink-C2C at start-up, and fewer CTAs measured faster.
static int decode_segments(int B, int Hq, int Hkv, int D, int max_context_len, int per_sm_x16) {
    if (B <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv || max_context_len <= 0) return 1;
    const int group = Hq / Hkv;
    const int64_t units = (int64_t)B * Hkv * ((group + 7) / 8);
    const int64_t sms = sm_count();
    const int pages = (max_context_len + 15) / 16;
    // at least 8 pages per segment (shorter ones cost more in start-up and
    // combine than they gain in parallelism, measured), at most 64 segments
    int64_t smax = pages / 8 > 1 ? pages / 8 : 1;
    if (smax > 64) smax = 64;
    // Measured on GB300 (D = 256; every segment count 2..16, 20..64 on the
    // batch 1 / 8 / 16 / 64 shapes): when the units are few, the fastest grid
    // is one wave of about 2.5 CTAs per SM with device-resident inputs (a
    // fuller wave of ~3 per SM measured slower, clusters of 7 much slower);
    // when even two segments per unit would overfill that, about 5 CTAs per
    // SM in several waves (shorter CTAs even out the tail).
    int64_t best = (sms * per_sm_x16 / 16 + units / 2) / units;
    if (best < 2) best = (sms * 5 + units / 2) / units;
    if (best < 1) best = 1;
    // With more segments than one cluster takes (the partials then merge in
    // the combine kernel), one wave that fills every SM to the kernel's
    // residency beats it: CTAs on an SM that holds fewer of them finish
    // early and leave HBM idle at the end (batch 8: 448 CTAs at 3 per SM,
    // 33.4 us per call; 384 at the 2.5-per-SM choice, 36.5; with pinned host
    // I/O 38.3 us against 40.1 for 8 segments in one cluster).
    {
        const int64_t full = sms * sage::decode_ctas_per_sm(D) / units;
        if (full > sage::kDecodeMaxCluster && full >= best) best = full;
    }
    if (best > smax) best = smax;
    const int64_t cap = sage::decode_max_segment_pages();
    if (best * cap < pages) best = (pages + cap - 1) / cap;
    const int64_t pps = (pages + best - 1) / best;
    best = (pages + pps - 1) / pps;
    return (int)best;
}

SAGE_API int sage_decode_num_segments(int B, int Hq, int Hkv, int D, int max_context_len) {
    return decode_segments(B, Hq, Hkv, D, max_context_len, 40);
}

SAGE_API int sage_decode_auto_segments(const sage_decode_args_t *a, const void *q) {
    if (!a) return 1;
    const bool host_io = is_host_memory(q ? q : (const void *)a->q) ||
                         is_host_memory(a->block_table) || is_host_memory(a->out);
    return decode_segments(a->B, a->Hq, a->Hkv, a->D, a->max_context_len, host_io ? 27 : 40);
}

// Decode workspace (S > 1): fp32 partial outputs [B*Hq, S, D], fp32 partial
// LSEs [B*Hq, S], then the int8 query codes [B*Hq, D] and their scales
// [B*Hq] of a query that sits in pinned host memory, each region 256-byte
// aligned.
struct DecodeWorkspace {
    size_t l_off, qc_off, qs_off, bytes;
};
static DecodeWorkspace decode_workspace(int B, int Hq, int D, int S) {
    DecodeWorkspace w = {0, 0, 0, 0};
    if (S <= 1 || B <= 0 || Hq <= 0 || D <= 0) return w;
    const size_t rows = (size_t)B * Hq * S, qrows = (size_t)B * Hq;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    w.l_off = up(rows * D * sizeof(float));
    w.qc_off = w.l_off + up(rows * sizeof(float));
    w.qs_off = w.qc_off + up(qrows * D);
    w.bytes = w.qs_off + qrows * sizeof(float);
    return w;
}

SAGE_API size_t sage_attn_decode_workspace_size(int B, int Hq, int D, int num_segments) {
    return decode_workspace(B, Hq, D, num_segments).bytes;
}

namespace sage {

int check_decode_args(const sage_decode_args_t *a, const void *q_fp) {
    if (!a) return fail(SAGE_ERR_INVALID_ARG, "args is NULL");
    if (!head_dim_ok(a->D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", a->D);
    if (a->out_dtype != SAGE_F16 && a->out_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "out dtype must be f16 or bf16");
    if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv)
        return fail(SAGE_ERR_INVALID_ARG, "need Hq a positive multiple of Hkv (Hq=%d Hkv=%d)",
                    a->Hq, a->Hkv);
    if (a->max_context_len < 0 || a->max_blocks < 0 ||
        (int64_t)a->max_context_len > 16ll * a->max_blocks)
        return fail(SAGE_ERR_INVALID_ARG, "max_context_len %d exceeds 16 * max_blocks (%d)",
                    a->max_context_len, a->max_blocks);
    if (a->num_segments < 0 || a->num_segments > 1024)
        return fail(SAGE_ERR_INVALID_ARG, "num_segments outside [0, 1024]");
    if (a->pv_mode < SAGE_PV_F32 || a->pv_mode > SAGE_PV_INT8)
        return fail(SAGE_ERR_UNSUPPORTED, "pv_mode %d is not one of SAGE_PV_*", a->pv_mode);
    if (a->B == 0) return SAGE_OK;
    if ((!q_fp && (!a->q || !a->q_scale)) || !a->context_lens || !a->out)
        return fail(SAGE_ERR_INVALID_ARG, "q, q_scale, context_lens and out are required");
    if (q_fp && !aligned(q_fp, 8)) return fail(SAGE_ERR_INVALID_ARG, "q must be 8-byte aligned");
    if (a->max_context_len > 0) {
        if (!a->k_cache || !a->v_cache || !a->k_scale || !a->v_scale || !a->block_table)
            return fail(SAGE_ERR_INVALID_ARG, "cache, scales and block_table are required");
        if (a->num_blocks < 1) return fail(SAGE_ERR_INVALID_ARG, "num_blocks must be >= 1");
        if (!aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->k_scale, 16) ||
            !aligned(a->v_scale, 16))
            return fail(SAGE_ERR_INVALID_ARG, "caches and scales must be 16-byte aligned");
    }
    if (!q_fp && !aligned(a->q, 4)) return fail(SAGE_ERR_INVALID_ARG, "q must be 4-byte aligned");
    if (!aligned(a->out, 8)) return fail(SAGE_ERR_INVALID_ARG, "out must be 8-byte aligned");
    {   // the per-step inputs and outputs: device or mapped pinned host memory
        const struct { const void *p; const char *n; } io[] = {
            {q_fp ? q_fp : (const void *)a->q, "q"}, {q_fp ? nullptr : (const void *)a->q_scale, "q_scale"},
            {a->max_context_len > 0 ? a->block_table : nullptr, "block_table"},
            {a->context_lens, "context_lens"}, {a->out, "out"}, {a->lse, "lse"}};
        for (const auto &x : io) {
            const sage_status_t r = check_reachable(x.p, x.n);
            if (r != SAGE_OK) return r;
        }
    }
    return SAGE_OK;
}

}  // namespace sage

// partials_o / partials_l (optional): write the segment partials there and
// skip the combine (num_segments must be given).
static sage_status_t run_decode(const sage_decode_args_t *a, void *workspace,
                                size_t workspace_bytes, int32_t *dbg, void *stream,
                                float *partials_o = nullptr, float *partials_l = nullptr,
                                int *segments_used = nullptr, const void *q_fp = nullptr,
                                int q_fp_bf16 = 0) {
    g_last = sage::LaunchLog();
    const sage_status_t chk = (sage_status_t)sage::check_decode_args(a, q_fp);
    if (chk != SAGE_OK || a->B == 0) return chk;
    int S = a->num_segments ? a->num_segments : sage_decode_auto_segments(a, q_fp);
    const int pages = (a->max_context_len + 15) / 16;
    {   // a segment is at most decode_max_segment_pages() pages long
        const int cap = sage::decode_max_segment_pages();
        if ((int64_t)S * cap < pages) S = (pages + cap - 1) / cap;
    }
    int pps = pages > 0 ? (pages + S - 1) / S : 1;
    if (pages > 0) S = (pages + pps - 1) / pps;
    else S = 1;
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::DecodeParams p = {};
    p.q = a->q, p.q_scale = a->q_scale;
    p.q_fp = q_fp, p.q_fp_bf16 = q_fp_bf16;
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
    p.dbg = dbg, p.dbg_stride = a->max_context_len;
    p.err = ew;
    if (segments_used) *segments_used = S;
    if (partials_o) {
        if (!aligned(partials_o, 16) || !partials_l)
            return fail(SAGE_ERR_INVALID_ARG, "o_part (16-byte aligned) and lse_part are required");
        p.o_part = partials_o;
        p.lse_part = partials_l;
        p.force_partials = 1;
        cudaError_t e = sage::launch_decode(p, static_cast<cudaStream_t>(stream), g_last);
        return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "decode launch");
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const DecodeWorkspace w = decode_workspace(a->B, a->Hq, a->D, S);
    if (S > 1) {
        if (!workspace || workspace_bytes < w.bytes)
            return fail(SAGE_ERR_INVALID_ARG, "workspace too small: need %zu bytes for %d segments",
                        w.bytes, S);
        if (!aligned(workspace, 16)) return fail(SAGE_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    }
    if (q_fp && S > 1 && !dbg && is_host_memory(q_fp)) {
        // A query in pinned host memory is quantised once, by the per-token
        // kernel reading it across NVLink-C2C, into the workspace (the same
        // codes and scales, bit for bit); every segment's CTA then reads the
        // codes from device memory instead of the query from the host (14
        // segments per (sequence, kv head) read it 14 times).  The decode is
        // launched right behind it and overlaps its start-up with it.
        char *ws = static_cast<char *>(workspace);
        sage::QuantParams qp = {};
        qp.x = q_fp;
        qp.bf16 = q_fp_bf16;
        qp.B = a->B, qp.H = a->Hq, qp.S = 1, qp.D = a->D;
        qp.sb = (int64_t)a->Hq * a->D, qp.sh = a->D, qp.ss = a->D;
        qp.block = 1;
        qp.mu_heads = 1;
        qp.q = reinterpret_cast<int8_t *>(ws + w.qc_off);
        qp.scale = reinterpret_cast<float *>(ws + w.qs_off);
        sage::LaunchLog qlog;
        cudaError_t e = sage::launch_quant(qp, cs, qlog);
        if (e != cudaSuccess) return cuda_fail(e, "query quantisation launch");
        p.q = qp.q, p.q_scale = qp.scale;
        p.q_fp = nullptr;
        p.after_quant = 1;
        g_last.count = qlog.count;
    }
    if (S > 1 && S <= sage::kDecodeMaxCluster) {
        // the segments of each (sequence, kv head, head tile) form one
        // cluster and combine in distributed shared memory
        p.cluster = 1;
        cudaError_t e = sage::launch_decode(p, cs, g_last);
        if (e == cudaSuccess) return SAGE_OK;
        if (e != cudaErrorInvalidClusterSize && e != cudaErrorNotSupported &&
            e != cudaErrorLaunchOutOfResources)
            return cuda_fail(e, "decode launch (cluster)");
        cudaGetLastError();  // clear, then take the partials + combine path below
        p.cluster = 0;
        const int n = g_last.count;
        g_last = sage::LaunchLog();
        g_last.count = n > 0 ? n - 1 : 0;  // the query's quantisation, when it ran
    }
    if (S > 1) {
        p.o_part = static_cast<float *>(workspace);
        p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + w.l_off);
    }
    cudaError_t e = sage::launch_decode(p, cs, g_last);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    if (S > 1) {
        sage::LaunchLog tmp = g_last;
        sage::CombineParams c = {p.o_part, p.lse_part, a->B * a->Hq, S, a->D, a->out,
                                 p.out_bf16, a->lse, 1};
        e = sage::launch_combine(c, cs, tmp);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
        // keep the decode kernel as the recorded kernel; count both launches
        g_last.count = tmp.count;
    }
    return SAGE_OK;
}

SAGE_API sage_status_t sage_attn_decode_paged(const sage_decode_args_t *args, void *workspace,
                                              size_t workspace_bytes, void *stream) {
    return run_decode(args, workspace, workspace_bytes, nullptr, stream);
}

SAGE_API sage_status_t sage_attn_decode_paged_q16(const sage_decode_args_t *args, const void *q,
                                                  sage_dtype_t q_dtype, void *workspace,
                                                  size_t workspace_bytes, void *stream) {
    if (!q) return fail(SAGE_ERR_INVALID_ARG, "q is NULL");
    if (q_dtype != SAGE_F16 && q_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "q dtype must be f16 or bf16");
    return run_decode(args, workspace, workspace_bytes, nullptr, stream, nullptr, nullptr, nullptr,
                      q, q_dtype == SAGE_BF16);
}

SAGE_API sage_status_t sage_attn_decode_paged_partials(const sage_decode_args_t *args,
                                                       float *o_part, float *lse_part,
                                                       int *segments_used, void *stream) {
    if (!args) return fail(SAGE_ERR_INVALID_ARG, "args is NULL");
    if (args->num_segments < 1)
        return fail(SAGE_ERR_INVALID_ARG, "num_segments must be given (>= 1) for partials");
    if (!o_part) return fail(SAGE_ERR_INVALID_ARG, "o_part is NULL");
    return run_decode(args, nullptr, 0, nullptr, stream, o_part, lse_part, segments_used);
}

SAGE_API sage_status_t sage_debug_decode_qk_int32(const sage_decode_args_t *args, void *workspace,
                                                  size_t workspace_bytes, int32_t *scores,
                                                  void *stream) {
    if (!scores) return fail(SAGE_ERR_INVALID_ARG, "scores is NULL");
    return run_decode(args, workspace, workspace_bytes, scores, stream);
}

// ---------------------------------------------------------------- prefill

static sage_status_t check_prefill(const sage_prefill_args_t *a, int *qs_out, int *ks_out) {
    if (!a) return fail(SAGE_ERR_INVALID_ARG, "args is NULL");
    if (!head_dim_ok(a->D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", a->D);
    if (a->out_dtype != SAGE_F16 && a->out_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "out dtype must be f16 or bf16");
    if (a->v_dtype != SAGE_F16 && a->v_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "v dtype must be f16 or bf16");
    if (a->B < 0 || a->Sq < 0 || a->Sk < 0 || a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv)
        return fail(SAGE_ERR_INVALID_ARG, "bad shape (B=%d Hq=%d Hkv=%d Sq=%d Sk=%d)", a->B, a->Hq,
                    a->Hkv, a->Sq, a->Sk);
    const int qs = a->q_block == 1 ? 0 : ilog2_exact(a->q_block);
    const int ks = a->k_block == 1 ? 0 : ilog2_exact(a->k_block);
    if (qs < 0 || (a->q_block != 1 && a->q_block < 128))
        return fail(SAGE_ERR_UNSUPPORTED, "q_block must be 1 or a power of two >= 128");
    if (ks < 0 || (a->k_block != 1 && a->k_block < 64))
        return fail(SAGE_ERR_UNSUPPORTED, "k_block must be 1 or a power of two >= 64");
    if (a->max_prefix_len < 0 ||
        (a->max_prefix_len > 0 && (int64_t)a->max_prefix_len > 16ll * a->max_blocks))
        return fail(SAGE_ERR_INVALID_ARG, "max_prefix_len exceeds 16 * max_blocks");
    if (a->layout != SAGE_LAYOUT_HND && a->layout != SAGE_LAYOUT_NHD)
        return fail(SAGE_ERR_UNSUPPORTED, "layout %d is not SAGE_LAYOUT_HND or SAGE_LAYOUT_NHD",
                    a->layout);
    if (a->tail_split != SAGE_TAIL_SPLIT_AUTO && a->tail_split != SAGE_TAIL_SPLIT_OFF)
        return fail(SAGE_ERR_INVALID_ARG, "tail_split %d is not SAGE_TAIL_SPLIT_AUTO or _OFF",
                    a->tail_split);
    *qs_out = qs;
    *ks_out = ks;
    return SAGE_OK;
}

// The tail split of a (checked) request on the current device.
static sage::PrefillSplit prefill_split_of(const sage_prefill_args_t *a) {
    if (a->tail_split == SAGE_TAIL_SPLIT_OFF) return sage::PrefillSplit{0, 0, 0};
    return sage::prefill_split(a->B, a->Hq, a->Sq, a->D, a->max_prefix_len + a->Sk,
                               a->causal != 0, sm_count());
}

SAGE_API size_t sage_attn_prefill_workspace_size(const sage_prefill_args_t *a) {
    int qs = 0, ks = 0;
    if (check_prefill(a, &qs, &ks) != SAGE_OK) return 0;
    return sage::prefill_layout(a->B, a->Hkv, a->Sk, a->D, a->max_prefix_len,
                                a->v_dtype == SAGE_BF16, a->smooth_v != 0, prefill_split_of(a))
        .bytes;
}

static sage_status_t run_prefill(const sage_prefill_args_t *a, void *workspace,
                                 size_t workspace_bytes, int32_t *dbg, void *stream) {
    int qs = 0, ks = 0;
    sage_status_t cs = check_prefill(a, &qs, &ks);
    if (cs != SAGE_OK) return cs;
    const bool has_prefix = a->max_prefix_len > 0;
    g_last = sage::LaunchLog();
    if ((int64_t)a->B * a->Sq == 0) return SAGE_OK;
    if (!a->q || !a->q_scale || !a->out) return fail(SAGE_ERR_INVALID_ARG, "q, q_scale, out required");
    if (a->Sk > 0 && (!a->k || !a->k_scale || !a->v))
        return fail(SAGE_ERR_INVALID_ARG, "k, k_scale and v are required when Sk > 0");
    if (has_prefix) {
        if (!a->k_cache || !a->v_cache || !a->k_cache_scale || !a->v_cache_scale ||
            !a->block_table || !a->prefix_lens || a->num_blocks < 1)
            return fail(SAGE_ERR_INVALID_ARG, "paged prefix needs caches, scales, table, lens");
        if (!aligned(a->k_cache, 16) || !aligned(a->v_cache, 16))
            return fail(SAGE_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    }
    if (a->Sk + a->max_prefix_len == 0) return fail(SAGE_ERR_INVALID_ARG, "no keys");
    if (!aligned(a->q, 16) || (a->k && !aligned(a->k, 16)) || (a->v && !aligned(a->v, 16)) ||
        !aligned(a->out, 16))
        return fail(SAGE_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (a->smooth_v && (int64_t)a->B * a->Hkv > 65535)
        return fail(SAGE_ERR_UNSUPPORTED, "smooth_v supports at most 65535 (batch, kv head) pairs");
    if (a->v_mean && !aligned(a->v_mean, 16))
        return fail(SAGE_ERR_INVALID_ARG, "v_mean must be 16-byte aligned");
    const sage::PrefillSplit split = prefill_split_of(a);
    const sage::PrefillLayout L = sage::prefill_layout(a->B, a->Hkv, a->Sk, a->D,
                                                       a->max_prefix_len, a->v_dtype == SAGE_BF16,
                                                       a->smooth_v != 0, split);
    if (!workspace || workspace_bytes < L.bytes)
        return fail(SAGE_ERR_INVALID_ARG, "workspace too small: need %zu bytes", L.bytes);
    if (!aligned(workspace, 256)) return fail(SAGE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::PrefillParams p = {};
    p.B = a->B, p.Hq = a->Hq, p.Hkv = a->Hkv, p.Sq = a->Sq, p.Sk = a->Sk, p.D = a->D;
    p.group = a->Hq / a->Hkv;
    p.q = a->q, p.q_scale = a->q_scale, p.q_shift = qs;
    p.q_groups = (a->Sq + a->q_block - 1) / a->q_block;
    p.k = a->k, p.k_scale = a->k_scale, p.k_shift = ks;
    p.k_groups = (a->Sk + a->k_block - 1) / a->k_block;
    p.v = a->v, p.v_bf16 = a->v_dtype == SAGE_BF16;
    p.nhd = a->layout == SAGE_LAYOUT_NHD;
    // element strides of the chunk's V per batch, kv head and token
    p.v_sb = (int64_t)a->Hkv * a->Sk * a->D;
    p.v_sh = p.nhd ? (int64_t)a->D : (int64_t)a->Sk * a->D;
    p.v_st = p.nhd ? (int64_t)a->Hkv * a->D : (int64_t)a->D;
    p.q_bias = a->q_bias;
    if (has_prefix) {
        p.k_cache = a->k_cache, p.v_cache = a->v_cache;
        p.k_cache_scale = a->k_cache_scale, p.v_cache_scale = a->v_cache_scale;
        p.block_table = a->block_table, p.prefix_lens = a->prefix_lens;
        p.num_blocks = a->num_blocks, p.max_blocks = a->max_blocks;
        p.max_prefix_len = a->max_prefix_len;
    }
    p.causal = a->causal != 0;
    const float sm = a->sm_scale > 0.0f ? a->sm_scale : 1.0f / sqrtf((float)a->D);
    p.qk_scale_log2 = sm * 1.4426950408889634f;
    p.out = a->out, p.out_bf16 = a->out_dtype == SAGE_BF16, p.lse = a->lse;
    p.dbg = dbg;
    p.dbg_stride = a->max_prefix_len + a->Sk;
    p.err = ew;
    char *w = static_cast<char *>(workspace);
    p.BN = L.BN, p.Ppad = L.Ppad, p.Lpad = L.Lpad, p.Vrows = L.Vrows;
    p.bundle = sage::prefill_bundle(a->B, a->Hq, p.group, L.Lpad, a->D);
    p.q_ahead = sm_count();
    p.k_ws = reinterpret_cast<__half *>(w + L.off_k);
    p.v_ws = L.Vrows ? reinterpret_cast<__half *>(w + L.off_v) : nullptr;
    p.ksc_ws = reinterpret_cast<float *>(w + L.off_ksc);
    if (split.parts > 0) {
        p.split_f = split.full, p.split_k = split.parts, p.split_tail = split.tail;
        p.part_o = reinterpret_cast<float *>(w + L.off_part_o);
        p.part_lse = reinterpret_cast<float *>(w + L.off_part_lse);
    }
    cudaStream_t cst = static_cast<cudaStream_t>(stream);
    sage::LaunchLog stage_log;
    cudaError_t e = cudaSuccess;
    if (a->smooth_v) {
        // the chunk's V mean per (batch, kv head), the smooth_k mean kernel's
        float *mu = a->v_mean ? a->v_mean : reinterpret_cast<float *>(w + L.off_vmean);
        sage::QuantParams mp = {};
        mp.x = a->v;
        mp.bf16 = a->v_dtype == SAGE_BF16;
        mp.B = a->B, mp.H = a->Hkv, mp.S = a->Sk, mp.D = a->D;
        mp.sb = p.v_sb, mp.sh = p.v_sh, mp.ss = p.v_st;
        mp.smooth = 1;
        mp.mu_out = mu;
        e = sage::launch_token_mean(mp, cst, stage_log);
        if (e != cudaSuccess) return cuda_fail(e, "V mean launch");
        p.v_mean = mu;
    }
    e = sage::launch_prefill_stage(p, cst, stage_log);
    if (e != cudaSuccess) return cuda_fail(e, "prefill staging launch");
    e = sage::launch_prefill(p, cst, g_last);
    g_last.count += stage_log.count;
    if (e == cudaErrorNotSupported)
        return fail(SAGE_ERR_UNSUPPORTED, "prefill configuration not supported by this build");
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "prefill launch");
}

SAGE_API sage_status_t sage_attn_prefill(const sage_prefill_args_t *args, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    return run_prefill(args, workspace, workspace_bytes, nullptr, stream);
}

SAGE_API sage_status_t sage_debug_prefill_qk_int32(const sage_prefill_args_t *args,
                                                   void *workspace, size_t workspace_bytes,
                                                   int32_t *scores, void *stream) {
    if (!scores) return fail(SAGE_ERR_INVALID_ARG, "scores is NULL");
    return run_prefill(args, workspace, workspace_bytes, scores, stream);
}

// --------------------------------------------------------- varlen prefill

static sage_status_t check_prefill_varlen(const sage_prefill_varlen_args_t *a, int *qs_out,
                                          int *ks_out) {
    if (!a) return fail(SAGE_ERR_INVALID_ARG, "args is NULL");
    if (!head_dim_ok(a->D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", a->D);
    if (a->out_dtype != SAGE_F16 && a->out_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "out dtype must be f16 or bf16");
    if (a->v_dtype != SAGE_F16 && a->v_dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "v dtype must be f16 or bf16");
    if (a->B < 0 || a->B > 65535 || a->Hq < 1 || a->Hq > 65535 || a->Hkv < 1 ||
        a->Hq % a->Hkv || a->total_q < 0 || a->total_k < 0 || a->max_seqlen_q < 0 ||
        a->max_seqlen_k < 0)
        return fail(SAGE_ERR_INVALID_ARG, "bad shape (B=%d Hq=%d Hkv=%d total_q=%lld total_k=%lld)",
                    a->B, a->Hq, a->Hkv, (long long)a->total_q, (long long)a->total_k);
    const int qs = a->q_block == 1 ? 0 : ilog2_exact(a->q_block);
    const int ks = a->k_block == 1 ? 0 : ilog2_exact(a->k_block);
    if (qs < 0 || (a->q_block != 1 && a->q_block < 128))
        return fail(SAGE_ERR_UNSUPPORTED, "q_block must be 1 or a power of two >= 128");
    if (ks < 0 || (a->k_block != 1 && a->k_block < 64))
        return fail(SAGE_ERR_UNSUPPORTED, "k_block must be 1 or a power of two >= 64");
    const int BN = a->D == 256 ? 64 : 128;
    if (a->total_k + (int64_t)a->B * (BN + 4) + 16 > 0x7fffffffll ||
        (int64_t)a->Hkv * a->total_k > 0x7fffffffffffll)
        return fail(SAGE_ERR_UNSUPPORTED, "packed key count too large");
    *qs_out = qs;
    *ks_out = ks;
    return SAGE_OK;
}

SAGE_API size_t sage_attn_prefill_varlen_workspace_size(const sage_prefill_varlen_args_t *a) {
    int qs = 0, ks = 0;
    if (check_prefill_varlen(a, &qs, &ks) != SAGE_OK) return 0;
    return sage::prefill_layout_varlen(a->B, a->Hkv, a->total_k, a->D, a->smooth_v != 0).bytes;
}

static sage_status_t run_prefill_varlen(const sage_prefill_varlen_args_t *a, void *workspace,
                                        size_t workspace_bytes, int32_t *dbg, void *stream) {
    int qs = 0, ks = 0;
    sage_status_t cs = check_prefill_varlen(a, &qs, &ks);
    if (cs != SAGE_OK) return cs;
    g_last = sage::LaunchLog();
    if ((int64_t)a->B * a->total_q * a->max_seqlen_q == 0) return SAGE_OK;
    if (!a->cu_seqlens_q || !a->cu_seqlens_k)
        return fail(SAGE_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k are required");
    if (!a->q || !a->q_scale || !a->out) return fail(SAGE_ERR_INVALID_ARG, "q, q_scale, out required");
    if (a->total_k > 0 && (!a->k || !a->k_scale || !a->v))
        return fail(SAGE_ERR_INVALID_ARG, "k, k_scale and v are required when total_k > 0");
    const int64_t vst = a->v_stride_t ? a->v_stride_t : (int64_t)a->Hkv * a->D;
    const int64_t vsh = a->v_stride_h ? a->v_stride_h : a->D;
    if (vst % 8 || vsh % 8) return fail(SAGE_ERR_INVALID_ARG, "v strides must be multiples of 8");
    if (!aligned(a->q, 16) || (a->k && !aligned(a->k, 16)) || (a->v && !aligned(a->v, 16)) ||
        !aligned(a->out, 16))
        return fail(SAGE_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (a->smooth_v && (int64_t)a->B * a->Hkv > 65535)
        return fail(SAGE_ERR_UNSUPPORTED, "smooth_v supports at most 65535 (sequence, kv head) pairs");
    if (a->v_mean && !aligned(a->v_mean, 16))
        return fail(SAGE_ERR_INVALID_ARG, "v_mean must be 16-byte aligned");
    const sage::PrefillLayout L =
        sage::prefill_layout_varlen(a->B, a->Hkv, a->total_k, a->D, a->smooth_v != 0);
    if (!workspace || workspace_bytes < L.bytes)
        return fail(SAGE_ERR_INVALID_ARG, "workspace too small: need %zu bytes", L.bytes);
    if (!aligned(workspace, 256)) return fail(SAGE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::PrefillParams p = {};
    p.B = a->B, p.Hq = a->Hq, p.Hkv = a->Hkv, p.D = a->D;
    p.Sq = a->max_seqlen_q, p.Sk = a->max_seqlen_k;
    p.group = a->Hq / a->Hkv;
    p.q = a->q, p.q_scale = a->q_scale, p.q_shift = qs;
    p.q_groups = (int)sage_varlen_scale_groups(a->total_q, a->B, a->q_block);
    p.k = a->k, p.k_scale = a->k_scale, p.k_shift = ks;
    p.k_groups = (int)sage_varlen_scale_groups(a->total_k, a->B, a->k_block);
    p.v = a->v, p.v_bf16 = a->v_dtype == SAGE_BF16;
    p.q_bias = a->q_bias;
    p.causal = a->causal != 0;
    const float sm = a->sm_scale > 0.0f ? a->sm_scale : 1.0f / sqrtf((float)a->D);
    p.qk_scale_log2 = sm * 1.4426950408889634f;
    p.out = a->out, p.out_bf16 = a->out_dtype == SAGE_BF16, p.lse = a->lse;
    p.dbg = dbg;
    p.dbg_stride = a->max_seqlen_k;
    p.err = ew;
    p.cu_q = a->cu_seqlens_q, p.cu_k = a->cu_seqlens_k;
    p.total_q = a->total_q, p.total_k = a->total_k;
    p.v_st = vst, p.v_sh = vsh;
    char *w = static_cast<char *>(workspace);
    p.BN = L.BN, p.Ppad = 0, p.Lpad = L.Lpad, p.Vrows = L.Vrows;
    p.q_ahead = sm_count();
    p.vl_pairs = a->D <= 128 && p.group % 2 == 0;
    p.k_ws = reinterpret_cast<__half *>(w + L.off_k);
    p.v_ws = reinterpret_cast<__half *>(w + L.off_v);
    p.ksc_ws = reinterpret_cast<float *>(w + L.off_ksc);
    cudaStream_t cst = static_cast<cudaStream_t>(stream);
    sage::LaunchLog stage_log;
    cudaError_t e = cudaSuccess;
    if (a->smooth_v) {
        // each sequence's V mean per kv head
        float *mu = a->v_mean ? a->v_mean : reinterpret_cast<float *>(w + L.off_vmean);
        sage::QuantParams mp = {};
        mp.x = a->v;
        mp.bf16 = a->v_dtype == SAGE_BF16;
        mp.B = a->B, mp.H = a->Hkv, mp.S = a->max_seqlen_k, mp.D = a->D;
        mp.sh = vsh, mp.ss = vst;
        mp.smooth = 1;
        mp.mu_out = mu;
        mp.cu = a->cu_seqlens_k, mp.total = a->total_k, mp.err = ew;
        e = sage::launch_token_mean(mp, cst, stage_log);
        if (e != cudaSuccess) return cuda_fail(e, "varlen V mean launch");
        p.v_mean = mu;
    }
    e = sage::launch_prefill_stage(p, cst, stage_log);
    if (e != cudaSuccess) return cuda_fail(e, "varlen prefill staging launch");
    e = sage::launch_prefill(p, cst, g_last);
    g_last.count += stage_log.count;
    if (e == cudaErrorNotSupported)
        return fail(SAGE_ERR_UNSUPPORTED, "prefill configuration not supported by this build");
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "varlen prefill launch");
}

SAGE_API sage_status_t sage_attn_prefill_varlen(const sage_prefill_varlen_args_t *args,
                                                void *workspace, size_t workspace_bytes,
                                                void *stream) {
    return run_prefill_varlen(args, workspace, workspace_bytes, nullptr, stream);
}

SAGE_API sage_status_t sage_debug_prefill_varlen_qk_int32(const sage_prefill_varlen_args_t *args,
                                                          void *workspace, size_t workspace_bytes,
                                                          int32_t *scores, void *stream) {
    if (!scores) return fail(SAGE_ERR_INVALID_ARG, "scores is NULL");
    return run_prefill_varlen(args, workspace, workspace_bytes, scores, stream);
}

// ---------------------------------------------------------------- kv append

SAGE_API sage_status_t sage_kv_cache_append(const void *k_new, const void *v_new,
                                            sage_dtype_t dtype, int B, int Hkv, int n_new, int D,
                                            const int32_t *block_table, int max_blocks,
                                            const int32_t *positions, int num_blocks,
                                            int8_t *k_cache, int8_t *v_cache, float *k_scale,
                                            float *v_scale, void *stream) {
    if (!head_dim_ok(D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", D);
    if (dtype != SAGE_F16 && dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "k/v dtype must be f16 or bf16");
    if (B < 0 || Hkv < 1 || n_new < 0 || max_blocks < 1 || num_blocks < 1)
        return fail(SAGE_ERR_INVALID_ARG, "bad shape (B=%d Hkv=%d n=%d max_blocks=%d num_blocks=%d)",
                    B, Hkv, n_new, max_blocks, num_blocks);
    g_last = sage::LaunchLog();
    if ((int64_t)B * n_new == 0) return SAGE_OK;
    if (!k_new || !v_new || !block_table || !positions || !k_cache || !v_cache || !k_scale ||
        !v_scale)
        return fail(SAGE_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16))
        return fail(SAGE_ERR_INVALID_ARG, "k_new, v_new and the caches must be 16-byte aligned");
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::KvAppendParams p = {};
    p.k = k_new, p.v = v_new, p.bf16 = dtype == SAGE_BF16;
    p.B = B, p.H = Hkv, p.n = n_new, p.D = D;
    p.block_table = block_table, p.pos = positions;
    p.max_blocks = max_blocks, p.num_blocks = num_blocks;
    p.k_cache = k_cache, p.v_cache = v_cache, p.k_scale = k_scale, p.v_scale = v_scale;
    p.err = ew;
    cudaError_t e = sage::launch_kv_append(p, static_cast<cudaStream_t>(stream), g_last);
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "kv append launch");
}

SAGE_API sage_status_t sage_kv_producer(const void *q_new, const void *k_new, const void *v_new,
                                        sage_dtype_t dtype, int B, int Hq, int Hkv, int n_new,
                                        int D, const int32_t *block_table, int max_blocks,
                                        const int32_t *positions, int num_blocks, int8_t *k_cache,
                                        int8_t *v_cache, float *k_scale, float *v_scale,
                                        int8_t *q_int8, float *q_scale, void *stream) {
    if (!head_dim_ok(D)) return fail(SAGE_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", D);
    if (dtype != SAGE_F16 && dtype != SAGE_BF16)
        return fail(SAGE_ERR_UNSUPPORTED, "q/k/v dtype must be f16 or bf16");
    if (B < 0 || Hq < 1 || Hkv < 1 || n_new < 0 || max_blocks < 1 || num_blocks < 1)
        return fail(SAGE_ERR_INVALID_ARG,
                    "bad shape (B=%d Hq=%d Hkv=%d n=%d max_blocks=%d num_blocks=%d)", B, Hq, Hkv,
                    n_new, max_blocks, num_blocks);
    g_last = sage::LaunchLog();
    if ((int64_t)B * n_new == 0) return SAGE_OK;
    if (!q_new || !k_new || !v_new || !block_table || !positions || !k_cache || !v_cache ||
        !k_scale || !v_scale || !q_int8 || !q_scale)
        return fail(SAGE_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(q_new, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q_int8, 8))
        return fail(SAGE_ERR_INVALID_ARG,
                    "q_new, k_new, v_new and the caches must be 16-byte aligned, q_int8 8-byte");
    int *ew = nullptr;
    sage_status_t st = error_word(&ew);
    if (st != SAGE_OK) return st;
    sage::KvAppendParams p = {};
    p.k = k_new, p.v = v_new, p.bf16 = dtype == SAGE_BF16;
    p.B = B, p.H = Hkv, p.n = n_new, p.D = D;
    p.block_table = block_table, p.pos = positions;
    p.max_blocks = max_blocks, p.num_blocks = num_blocks;
    p.k_cache = k_cache, p.v_cache = v_cache, p.k_scale = k_scale, p.v_scale = v_scale;
    p.q = q_new, p.Hq = Hq, p.q_int8 = q_int8, p.q_scale = q_scale;
    p.err = ew;
    cudaError_t e = sage::launch_kv_append(p, static_cast<cudaStream_t>(stream), g_last);
    return e == cudaSuccess ? SAGE_OK : cuda_fail(e, "kv producer launch");
}
