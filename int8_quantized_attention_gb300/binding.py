"""Thin ctypes binding of libsageattn.so (the C ABI in include/sage_attn.h).

Argument marshalling only: torch tensors are checked for device, dtype and
layout, outputs are allocated with torch, and raw device pointers plus the
current CUDA stream are handed to the library.  Every step of the
attention path runs in the library's kernels; there is no fallback: if the
library is missing or the tensors are not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

SAGE_OK = 0
SAGE_ERR_INVALID_ARG = 1
SAGE_ERR_UNSUPPORTED = 2
SAGE_ERR_CUDA = 3
SAGE_ERR_TIMEOUT = 4
SAGE_ERR_BAD_BLOCK = 5

SAGE_F16 = 0
SAGE_BF16 = 1

_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float


class SageError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("sage status %d: %s" % (status, message))
        self.status = status


class DecodeArgs(ctypes.Structure):
    _fields_ = [("q", _vp), ("q_scale", _vp), ("k_cache", _vp), ("v_cache", _vp),
                ("k_scale", _vp), ("v_scale", _vp), ("block_table", _vp), ("context_lens", _vp),
                ("B", _i), ("Hq", _i), ("Hkv", _i), ("D", _i), ("num_blocks", _i),
                ("max_blocks", _i), ("max_context_len", _i), ("sm_scale", _f),
                ("num_segments", _i), ("out", _vp), ("out_dtype", _i), ("lse", _vp),
                ("pv_mode", _i)]


class PrefillArgs(ctypes.Structure):
    _fields_ = [("B", _i), ("Hq", _i), ("Hkv", _i), ("Sq", _i), ("Sk", _i), ("D", _i),
                ("q", _vp), ("q_scale", _vp), ("q_block", _i),
                ("k", _vp), ("k_scale", _vp), ("k_block", _i),
                ("v", _vp), ("v_dtype", _i), ("q_bias", _vp),
                ("k_cache", _vp), ("v_cache", _vp), ("k_cache_scale", _vp), ("v_cache_scale", _vp),
                ("block_table", _vp), ("prefix_lens", _vp),
                ("num_blocks", _i), ("max_blocks", _i), ("max_prefix_len", _i),
                ("causal", _i), ("sm_scale", _f), ("out", _vp), ("out_dtype", _i), ("lse", _vp),
                ("smooth_v", _i), ("v_mean", _vp), ("layout", _i), ("tail_split", _i)]


class PrefillVarlenArgs(ctypes.Structure):
    _fields_ = [("B", _i), ("Hq", _i), ("Hkv", _i), ("D", _i), ("total_q", _i64), ("total_k", _i64),
                ("max_seqlen_q", _i), ("max_seqlen_k", _i),
                ("cu_seqlens_q", _vp), ("cu_seqlens_k", _vp),
                ("q", _vp), ("q_scale", _vp), ("q_block", _i),
                ("k", _vp), ("k_scale", _vp), ("k_block", _i),
                ("v", _vp), ("v_dtype", _i), ("v_stride_t", _i64), ("v_stride_h", _i64),
                ("q_bias", _vp), ("causal", _i), ("sm_scale", _f), ("out", _vp), ("out_dtype", _i),
                ("lse", _vp), ("smooth_v", _i), ("v_mean", _vp)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char * 64), ("grid", _i * 3), ("block", _i * 3),
                ("cluster", _i * 3), ("smem_bytes", _i), ("num_segments", _i), ("launches", _i)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libsageattn.so (built in-tree by build.py); raise if it is absent."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError("libsageattn.so is not built (%s); run "
                               "int8_quantized_attention_gb300.build.build()" % path)
        L = ctypes.CDLL(path)
        L.sage_get_last_error_message.restype = ctypes.c_char_p
        L.sage_version.restype = _i
        L.sage_quant_int8.argtypes = [_vp, _i, _i, _i, _i, _i, _i64, _i64, _i64, _i, _i, _vp, _i,
                                      _vp, _vp, _vp, _vp, _vp]
        L.sage_quant_int8.restype = _i
        L.sage_varlen_scale_groups.argtypes = [_i64, _i, _i]
        L.sage_varlen_scale_groups.restype = _i64
        L.sage_quant_int8_varlen.argtypes = [_vp, _i, _i, _i, _i64, _i, _i64, _i64, _vp, _i, _i,
                                             _i, _vp, _i, _vp, _vp, _vp, _vp, _vp]
        L.sage_quant_int8_varlen.restype = _i
        L.sage_attn_prefill_varlen_workspace_size.argtypes = [ctypes.POINTER(PrefillVarlenArgs)]
        L.sage_attn_prefill_varlen_workspace_size.restype = ctypes.c_size_t
        L.sage_attn_prefill_varlen.argtypes = [ctypes.POINTER(PrefillVarlenArgs), _vp,
                                               ctypes.c_size_t, _vp]
        L.sage_attn_prefill_varlen.restype = _i
        L.sage_debug_prefill_varlen_qk_int32.argtypes = [ctypes.POINTER(PrefillVarlenArgs), _vp,
                                                         ctypes.c_size_t, _vp, _vp]
        L.sage_debug_prefill_varlen_qk_int32.restype = _i
        L.sage_decode_num_segments.argtypes = [_i, _i, _i, _i, _i]
        L.sage_decode_num_segments.restype = _i
        L.sage_decode_auto_segments.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
        L.sage_decode_auto_segments.restype = _i
        L.sage_attn_decode_workspace_size.argtypes = [_i, _i, _i, _i]
        L.sage_attn_decode_workspace_size.restype = ctypes.c_size_t
        L.sage_attn_decode_paged.argtypes = [ctypes.POINTER(DecodeArgs), _vp, ctypes.c_size_t, _vp]
        L.sage_attn_decode_paged.restype = _i
        L.sage_attn_decode_paged_q16.argtypes = [ctypes.POINTER(DecodeArgs), _vp, _i, _vp,
                                                 ctypes.c_size_t, _vp]
        L.sage_attn_decode_paged_q16.restype = _i
        L.sage_kv_cache_append.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp, _i, _vp,
                                           _vp, _vp, _vp, _vp]
        L.sage_kv_cache_append.restype = _i
        L.sage_kv_producer.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i, _vp, _i,
                                       _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.sage_kv_producer.restype = _i
        L.sage_attn_decode_paged_partials.argtypes = [ctypes.POINTER(DecodeArgs), _vp, _vp,
                                                      ctypes.POINTER(_i), _vp]
        L.sage_attn_decode_paged_partials.restype = _i
        L.sage_attn_decode_noalloc_max_bytes.argtypes = []
        L.sage_attn_decode_noalloc_max_bytes.restype = ctypes.c_size_t
        L.sage_attn_decode_paged_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
        L.sage_attn_decode_paged_noalloc.restype = _i
        L.sage_debug_decode_qk_int32.argtypes = [ctypes.POINTER(DecodeArgs), _vp, ctypes.c_size_t,
                                                 _vp, _vp]
        L.sage_debug_decode_qk_int32.restype = _i
        L.sage_splitk_combine.argtypes = [_vp, _vp, _i, _i, _i, _vp, _i, _vp, _vp]
        L.sage_splitk_combine.restype = _i
        L.sage_attn_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
        L.sage_attn_prefill_workspace_size.restype = ctypes.c_size_t
        L.sage_attn_prefill.argtypes = [ctypes.POINTER(PrefillArgs), _vp, ctypes.c_size_t, _vp]
        L.sage_attn_prefill.restype = _i
        L.sage_debug_prefill_qk_int32.argtypes = [ctypes.POINTER(PrefillArgs), _vp,
                                                  ctypes.c_size_t, _vp, _vp]
        L.sage_debug_prefill_qk_int32.restype = _i
        L.sage_last_launch_info.argtypes = [ctypes.POINTER(LaunchInfo)]
        L.sage_last_launch_info.restype = _i
        L.sage_check_device_status.argtypes = [_vp, ctypes.POINTER(_i)]
        L.sage_check_device_status.restype = _i
        L.sage_debug_timeout_probe.argtypes = [_i, _vp]
        L.sage_debug_timeout_probe.restype = _i
        _LIB = L
    return _LIB


def _check(status: int):
    if status != SAGE_OK:
        raise SageError(status, lib().sage_get_last_error_message().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_io(t: Optional[torch.Tensor]):
    """A per-step decode input/output: a CUDA tensor or a pinned host tensor
    (which the kernels reach directly; the library checks the mapping)."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("tensor must be on a CUDA device or in pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(dtype) -> int:
    if dtype == torch.float16:
        return SAGE_F16
    if dtype == torch.bfloat16:
        return SAGE_BF16
    raise ValueError("dtype must be float16 or bfloat16, got %s" % dtype)


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


# --------------------------------------------------------------------------
# Entry points
# --------------------------------------------------------------------------

def sage_quant_int8(x: torch.Tensor, block_tokens: int = 1, smooth: bool = False,
                    mu_in: Optional[torch.Tensor] = None, layout: str = "HND", stream=None):
    """Quantise x to INT8 (s = amax/127, round-to-nearest-even).

    x: [B,H,S,D] (layout "HND") or [B,S,H,D] ("NHD"), f16/bf16, channel
    dimension contiguous.  Returns (x_int8 [B,H,S,D], scale, mu, bias):
    scale [B,H,ceil(S/block_tokens)]; mu [B,H,D] when smooth; bias [B,H,S]
    (= x . mu_in, GQA-broadcast) when mu_in [B,Hmu,D] is given.
    """
    if layout == "HND":
        B, H, S, D = x.shape
        sb, sh, ss = x.stride(0), x.stride(1), x.stride(2)
    elif layout == "NHD":
        B, S, H, D = x.shape
        sb, ss, sh = x.stride(0), x.stride(1), x.stride(2)
    else:
        raise ValueError("layout must be HND or NHD")
    if x.stride(3) != 1:
        raise ValueError("channel dimension must be contiguous")
    dev = x.device
    G = (S + block_tokens - 1) // block_tokens
    q = torch.empty((B, H, S, D), dtype=torch.int8, device=dev)
    scale = torch.empty((B, H, G), dtype=torch.float32, device=dev)
    mu = torch.empty((B, H, D), dtype=torch.float32, device=dev) if smooth else None
    bias = None
    mu_heads = 0
    if mu_in is not None:
        _need(mu_in, torch.float32, "mu_in")
        mu_heads = mu_in.shape[1]
        bias = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    _check(lib().sage_quant_int8(_ptr(x), _dt(x.dtype), B, H, S, D, sb, sh, ss, block_tokens,
                                 int(bool(smooth)), _ptr(mu_in), mu_heads, _ptr(q), _ptr(scale),
                                 _ptr(mu), _ptr(bias), _stream(stream)))
    return q, scale, mu, bias


def decode_num_segments(B: int, Hq: int, Hkv: int, D: int, max_context_len: int) -> int:
    return int(lib().sage_decode_num_segments(B, Hq, Hkv, D, max_context_len))


def decode_workspace_size(B: int, Hq: int, D: int, num_segments: int) -> int:
    return int(lib().sage_attn_decode_workspace_size(B, Hq, D, num_segments))


PV_MODES = {"fp32": 0, "fp16": 1, "fp16+fp32": 2, "int8": 3}


def _pv(pv_mode) -> int:
    if pv_mode not in PV_MODES:
        raise ValueError("pv_mode must be one of %s" % sorted(PV_MODES))
    return PV_MODES[pv_mode]


def _decode_args(q_int8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                 max_context_len, sm_scale, num_segments, out, lse, shape=None, pv_mode="fp32"):
    if shape is None:
        _need(q_int8, torch.int8, "q_int8")
        _need(q_scale, torch.float32, "q_scale")
    _need(k_cache, torch.int8, "k_cache")
    _need(v_cache, torch.int8, "v_cache")
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    B, Hq, D = q_int8.shape if shape is None else shape
    a = DecodeArgs()
    a.q, a.q_scale = _ptr_io(q_int8), _ptr_io(q_scale)
    a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
    a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
    a.block_table, a.context_lens = _ptr_io(block_table), _ptr_io(context_lens)
    a.B, a.Hq, a.Hkv, a.D = B, Hq, k_cache.shape[1], D
    a.num_blocks, a.max_blocks = k_cache.shape[0], block_table.shape[1]
    a.max_context_len = int(max_context_len)
    a.sm_scale = float(sm_scale) if sm_scale else 0.0
    a.num_segments = int(num_segments)
    a.out, a.out_dtype = _ptr_io(out), _dt(out.dtype)
    a.lse = _ptr_io(lse)
    a.pv_mode = _pv(pv_mode)
    return a


def sage_attn_decode_paged(q_int8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
                           context_lens, max_context_len: int, *, sm_scale=None,
                           num_segments: int = 0, out_dtype=torch.bfloat16,
                           return_lse: bool = False, workspace: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, debug_scores=None,
                           pv_mode: str = "fp32", stream=None):
    """Split-K paged INT8 decode + LSE combine.  Returns out [B,Hq,D] (and lse).

    pv_mode: "fp32" (default), "fp16", "fp16+fp32" or "int8" -- the P.V
    operands and accumulation (SAGE_PV_* in the header).
    """
    B, Hq, D = q_int8.shape
    Hkv = k_cache.shape[1]
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=k_cache.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=k_cache.device) if return_lse else None
    a = _decode_args(q_int8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
                     context_lens, max_context_len, sm_scale, num_segments, out, lse,
                     pv_mode=pv_mode)
    # the library's choice for these buffers (it depends on where they live)
    S = num_segments or int(lib().sage_decode_auto_segments(ctypes.byref(a), None))
    a.num_segments = S
    need = decode_workspace_size(B, Hq, D, S)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty((need,), dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if debug_scores is not None:
        _need(debug_scores, torch.int32, "debug_scores")
        _check(lib().sage_debug_decode_qk_int32(ctypes.byref(a), _ptr(workspace), ws_bytes,
                                                _ptr(debug_scores), _stream(stream)))
    else:
        _check(lib().sage_attn_decode_paged(ctypes.byref(a), _ptr(workspace), ws_bytes,
                                            _stream(stream)))
    return (out, lse) if return_lse else out


def sage_attn_decode_paged_q16(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                               max_context_len: int, *, sm_scale=None, num_segments: int = 0,
                               out_dtype=torch.bfloat16, return_lse: bool = False,
                               workspace: Optional[torch.Tensor] = None,
                               out: Optional[torch.Tensor] = None, pv_mode: str = "fp32",
                               stream=None):
    """Paged decode with the per-token query quantisation fused into the kernel.

    q [B,Hq,D] f16/bf16.  Same result as sage_quant_int8 + sage_attn_decode_paged.
    q, block_table, context_lens and out may be pinned host tensors: the
    kernel reads and writes them in place (NVLink-C2C on GB300).
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if q.dtype not in (torch.float16, torch.bfloat16) or not q.is_contiguous():
        raise ValueError("q must be a contiguous f16/bf16 tensor")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=k_cache.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=k_cache.device) if return_lse else None
    a = _decode_args(None, None, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                     max_context_len, sm_scale, num_segments, out, lse, shape=(B, Hq, D),
                     pv_mode=pv_mode)
    # the library's choice for these buffers (it depends on where they live)
    S = num_segments or int(lib().sage_decode_auto_segments(ctypes.byref(a), _ptr_io(q)))
    a.num_segments = S
    need = decode_workspace_size(B, Hq, D, S)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty((need,), dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().sage_attn_decode_paged_q16(ctypes.byref(a), _ptr_io(q), _dt(q.dtype), _ptr(workspace),
                                            ws_bytes, _stream(stream)))
    return (out, lse) if return_lse else out


def sage_kv_cache_append(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table,
                         positions, stream=None):
    """Quantise new K/V rows per (token, KV head) into the paged INT8 cache, in place.

    k_new, v_new [B,Hkv,n,D] f16/bf16; block_table int32 [B,max_blocks];
    positions int32 [B] (token index of row 0 of each sequence).
    """
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if t.dtype not in (torch.float16, torch.bfloat16) or not t.is_contiguous():
            raise ValueError(name + " must be a contiguous f16/bf16 tensor")
    if v_new.dtype != k_new.dtype or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must match in dtype and shape")
    _need(k_cache, torch.int8, "k_cache")
    _need(v_cache, torch.int8, "v_cache")
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need(block_table, torch.int32, "block_table")
    _need(positions, torch.int32, "positions")
    B, H, n, D = k_new.shape
    _check(lib().sage_kv_cache_append(_ptr(k_new), _ptr(v_new), _dt(k_new.dtype), B, H, n, D,
                                      _ptr(block_table), block_table.shape[1], _ptr(positions),
                                      k_cache.shape[0], _ptr(k_cache), _ptr(v_cache),
                                      _ptr(k_scale), _ptr(v_scale), _stream(stream)))


def sage_kv_producer(q_new, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table,
                     positions, stream=None):
    """The step's KV producer in one launch: append k_new/v_new [B,Hkv,n,D] to
    the paged cache (as sage_kv_cache_append) and quantise q_new [B,Hq,n,D]
    per (token, head).  Returns (q_int8 [B,Hq,n,D], q_scale [B,Hq,n])."""
    for t, name in ((q_new, "q_new"), (k_new, "k_new"), (v_new, "v_new")):
        if t.dtype not in (torch.float16, torch.bfloat16) or not t.is_contiguous():
            raise ValueError(name + " must be a contiguous f16/bf16 tensor")
    if len({q_new.dtype, k_new.dtype, v_new.dtype}) != 1 or v_new.shape != k_new.shape:
        raise ValueError("q_new, k_new and v_new must share a dtype; k_new and v_new a shape")
    _need(k_cache, torch.int8, "k_cache")
    _need(v_cache, torch.int8, "v_cache")
    _need(k_scale, torch.float32, "k_scale")
    _need(v_scale, torch.float32, "v_scale")
    _need(block_table, torch.int32, "block_table")
    _need(positions, torch.int32, "positions")
    B, Hkv, n, D = k_new.shape
    Hq = q_new.shape[1]
    if q_new.shape != (B, Hq, n, D):
        raise ValueError("q_new must be [B, Hq, n, D] with k_new's B, n and D")
    q_int8 = torch.empty((B, Hq, n, D), dtype=torch.int8, device=q_new.device)
    q_scale = torch.empty((B, Hq, n), dtype=torch.float32, device=q_new.device)
    _check(lib().sage_kv_producer(_ptr(q_new), _ptr(k_new), _ptr(v_new), _dt(k_new.dtype), B, Hq,
                                  Hkv, n, D, _ptr(block_table), block_table.shape[1],
                                  _ptr(positions), k_cache.shape[0], _ptr(k_cache), _ptr(v_cache),
                                  _ptr(k_scale), _ptr(v_scale), _ptr(q_int8), _ptr(q_scale),
                                  _stream(stream)))
    return q_int8, q_scale


def decode_segments_used(max_context_len: int, num_segments: int) -> int:
    """Segment count the partials layout uses (see sage_attn_decode_paged_partials)."""
    pages = (int(max_context_len) + 15) // 16
    if pages == 0:
        return 1
    cap = 1024  # longest segment in pages (decode_max_segment_pages)
    if num_segments * cap < pages:
        num_segments = (pages + cap - 1) // cap
    pps = (pages + num_segments - 1) // num_segments
    return (pages + pps - 1) // pps


def sage_attn_decode_paged_partials(q_int8, q_scale, k_cache, v_cache, k_scale, v_scale,
                                    block_table, context_lens, max_context_len: int,
                                    num_segments: int, *, sm_scale=None, pv_mode: str = "fp32",
                                    stream=None):
    """Decode without the combine: returns (o_part [B,Hq,S,D], lse_part [B,Hq,S])."""
    B, Hq, D = q_int8.shape
    S = decode_segments_used(max_context_len, num_segments)
    o_part = torch.empty((B, Hq, S, D), dtype=torch.float32, device=k_cache.device)
    lse_part = torch.empty((B, Hq, S), dtype=torch.float32, device=k_cache.device)
    dummy = torch.empty((1,), dtype=torch.float16, device=k_cache.device)
    a = _decode_args(q_int8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
                     context_lens, max_context_len, sm_scale, num_segments, dummy, None,
                     pv_mode=pv_mode)
    used = _i(0)
    _check(lib().sage_attn_decode_paged_partials(ctypes.byref(a), _ptr(o_part), _ptr(lse_part),
                                                 ctypes.byref(used), _stream(stream)))
    assert used.value == S, (used.value, S)
    return o_part, lse_part


def sage_splitk_combine(o_part: torch.Tensor, lse_part: torch.Tensor, out_dtype=torch.bfloat16,
                        return_lse: bool = False, stream=None):
    """LSE combine of split-K partials: o_part [..., S, D] fp32, lse_part [..., S] fp32."""
    _need(o_part, torch.float32, "o_part")
    _need(lse_part, torch.float32, "lse_part")
    *lead, S, D = o_part.shape
    R = int(math.prod(lead)) if lead else 1
    out = torch.empty((*lead, D), dtype=out_dtype, device=o_part.device)
    lse = torch.empty(tuple(lead), dtype=torch.float32, device=o_part.device) if return_lse else None
    _check(lib().sage_splitk_combine(_ptr(o_part), _ptr(lse_part), R, S, D, _ptr(out),
                                     _dt(out_dtype), _ptr(lse), _stream(stream)))
    return (out, lse) if return_lse else out


def sage_attn_prefill(q_int8, q_scale, q_block: int, k_int8, k_scale, k_block: int, v, *,
                      causal: bool, sm_scale=None, q_bias=None, prefix: Optional[dict] = None,
                      out_dtype=None, return_lse: bool = False, debug_scores=None,
                      workspace: Optional[torch.Tensor] = None, out=None, lse=None,
                      smooth_v: bool = False, v_mean: Optional[torch.Tensor] = None,
                      layout: str = "HND", tail_split: bool = True, stream=None):
    """INT8-QK prefill attention over an optional paged INT8 prefix + a chunk.

    q_int8 [B,Hq,Sq,D]; q_scale [B,Hq,ceil(Sq/q_block)]; k_int8 [B,Hkv,Sk,D];
    k_scale [B,Hkv,ceil(Sk/k_block)]; v [B,Hkv,Sk,D] f16/bf16; q_bias [B,Hq,Sq]
    (smooth_k correction) or None; prefix = dict(k_cache, v_cache, k_scale,
    v_scale, block_table, lens, max_len) or None.  smooth_v subtracts the
    chunk's V mean from every value and adds it back to the output; v_mean
    ([B, Hkv, D] fp32, optional) receives that mean.  layout "NHD" takes v
    as [B,Sk,Hkv,D] and returns out as [B,Sq,Hq,D] (the INT8 codes, scales,
    q_bias and lse stay head-major).  tail_split=False keeps every query tile
    in one CTA (SAGE_TAIL_SPLIT_OFF); by default the library may split the
    last wave's tiles by key range (head_dim 256), equal to within rounding.
    """
    B, Hq, Sq, D = q_int8.shape
    Hkv, Sk = k_int8.shape[1], k_int8.shape[2]
    if layout not in ("HND", "NHD"):
        raise ValueError("layout must be HND or NHD")
    nhd = layout == "NHD"
    vshape = (B, Sk, Hkv, D) if nhd else (B, Hkv, Sk, D)
    oshape = (B, Sq, Hq, D) if nhd else (B, Hq, Sq, D)
    if tuple(v.shape) != vshape:
        raise ValueError("v must be %s for layout %s, got %s" % (vshape, layout, tuple(v.shape)))
    _need(q_int8, torch.int8, "q_int8")
    _need(k_int8, torch.int8, "k_int8")
    _need(q_scale, torch.float32, "q_scale")
    _need(k_scale, torch.float32, "k_scale")
    if not v.is_contiguous():
        raise ValueError("v must be contiguous")
    out_dtype = out.dtype if out is not None else (out_dtype or v.dtype)
    if out is None:
        out = torch.empty(oshape, dtype=out_dtype, device=q_int8.device)
    elif tuple(out.shape) != oshape or not out.is_contiguous():
        raise ValueError("out must be a contiguous %s tensor" % (oshape,))
    if lse is not None:
        _need(lse, torch.float32, "lse")
        return_lse = True
    elif return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q_int8.device)
    a = PrefillArgs()
    a.B, a.Hq, a.Hkv, a.Sq, a.Sk, a.D = B, Hq, Hkv, Sq, Sk, D
    a.q, a.q_scale, a.q_block = _ptr(q_int8), _ptr(q_scale), q_block
    a.k, a.k_scale, a.k_block = _ptr(k_int8), _ptr(k_scale), k_block
    a.v, a.v_dtype = _ptr(v), _dt(v.dtype)
    if q_bias is not None:
        _need(q_bias, torch.float32, "q_bias")
    a.q_bias = _ptr(q_bias)
    if prefix is not None:
        for key in ("k_cache", "v_cache"):
            _need(prefix[key], torch.int8, key)
        for key in ("k_scale", "v_scale"):
            _need(prefix[key], torch.float32, key)
        _need(prefix["block_table"], torch.int32, "block_table")
        _need(prefix["lens"], torch.int32, "lens")
        a.k_cache, a.v_cache = _ptr(prefix["k_cache"]), _ptr(prefix["v_cache"])
        a.k_cache_scale, a.v_cache_scale = _ptr(prefix["k_scale"]), _ptr(prefix["v_scale"])
        a.block_table, a.prefix_lens = _ptr(prefix["block_table"]), _ptr(prefix["lens"])
        a.num_blocks = prefix["k_cache"].shape[0]
        a.max_blocks = prefix["block_table"].shape[1]
        a.max_prefix_len = int(prefix["max_len"])
    a.causal = int(bool(causal))
    a.sm_scale = float(sm_scale) if sm_scale else 0.0
    a.out, a.out_dtype, a.lse = _ptr(out), _dt(out_dtype), _ptr(lse)
    if v_mean is not None:
        _need(v_mean, torch.float32, "v_mean")
    a.smooth_v, a.v_mean = int(bool(smooth_v)), _ptr(v_mean)
    a.layout = 1 if nhd else 0
    a.tail_split = 0 if tail_split else 1
    need = int(lib().sage_attn_prefill_workspace_size(ctypes.byref(a)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q_int8.device)
    wsb = workspace.numel() * workspace.element_size()
    if debug_scores is not None:
        _need(debug_scores, torch.int32, "debug_scores")
        _check(lib().sage_debug_prefill_qk_int32(ctypes.byref(a), _ptr(workspace), wsb,
                                                 _ptr(debug_scores), _stream(stream)))
    else:
        _check(lib().sage_attn_prefill(ctypes.byref(a), _ptr(workspace), wsb, _stream(stream)))
    return (out, lse) if return_lse else out


# --------------------------------------------------------------------------
# Variable-length packed batches (sequence b = packed tokens
# cu_seqlens[b] .. cu_seqlens[b+1]-1)
# --------------------------------------------------------------------------

def varlen_scale_groups(total: int, B: int, block_tokens: int) -> int:
    """Scale groups per head of a packed batch (see sage_quant_int8_varlen)."""
    return int(lib().sage_varlen_scale_groups(int(total), int(B), int(block_tokens)))


def sage_quant_int8_varlen(x: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
                           block_tokens: int = 1, smooth: bool = False,
                           mu_in: Optional[torch.Tensor] = None, stream=None):
    """Per-sequence INT8 quantisation of a packed batch x [total, H, D].

    Returns (x_int8 [H, total, D], scale [H, groups], mu [B, H, D] when
    smooth, bias [H, total] when mu_in [B, Hmu, D] is given).
    """
    total, H, D = x.shape
    if x.stride(2) != 1:
        raise ValueError("channel dimension must be contiguous")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    B = cu_seqlens.numel() - 1
    dev = x.device
    G = varlen_scale_groups(total, B, block_tokens)
    q = torch.empty((H, total, D), dtype=torch.int8, device=dev)
    scale = torch.empty((H, G), dtype=torch.float32, device=dev)
    mu = torch.empty((B, H, D), dtype=torch.float32, device=dev) if smooth else None
    bias = None
    mu_heads = 0
    if mu_in is not None:
        _need(mu_in, torch.float32, "mu_in")
        mu_heads = mu_in.shape[1]
        bias = torch.empty((H, total), dtype=torch.float32, device=dev)
    _check(lib().sage_quant_int8_varlen(_ptr(x), _dt(x.dtype), B, H, total, D, x.stride(1),
                                        x.stride(0), _ptr(cu_seqlens), int(max_seqlen),
                                        block_tokens, int(bool(smooth)), _ptr(mu_in), mu_heads,
                                        _ptr(q), _ptr(scale), _ptr(mu), _ptr(bias),
                                        _stream(stream)))
    return q, scale, mu, bias


def prefill_varlen_workspace_size(B: int, Hq: int, Hkv: int, D: int, total_q: int, total_k: int,
                                  max_seqlen_q: int, max_seqlen_k: int,
                                  smooth_v: bool = False) -> int:
    """Workspace bytes sage_attn_prefill_varlen needs for these sizes."""
    a = PrefillVarlenArgs()
    a.smooth_v = int(bool(smooth_v))
    a.B, a.Hq, a.Hkv, a.D = B, Hq, Hkv, D
    a.total_q, a.total_k = total_q, total_k
    a.max_seqlen_q, a.max_seqlen_k = max_seqlen_q, max_seqlen_k
    a.q_block = a.k_block = 1
    a.v_dtype = a.out_dtype = SAGE_F16
    return int(lib().sage_attn_prefill_varlen_workspace_size(ctypes.byref(a)))


def sage_attn_prefill_varlen(q_int8, q_scale, q_block: int, k_int8, k_scale, k_block: int, v,
                             cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, *,
                             causal: bool, sm_scale=None, q_bias=None, out_dtype=None,
                             return_lse: bool = False, debug_scores=None,
                             workspace: Optional[torch.Tensor] = None, smooth_v: bool = False,
                             v_mean: Optional[torch.Tensor] = None, stream=None):
    """INT8-QK prefill attention over a packed variable-length batch.

    q_int8 [Hq, total_q, D]; q_scale [Hq, groups_q]; k_int8 [Hkv, total_k, D];
    k_scale [Hkv, groups_k] (sage_quant_int8_varlen layouts); v [total_k, Hkv, D]
    f16/bf16 (channels contiguous); q_bias [Hq, total_q] or None.
    Returns out [total_q, Hq, D] (and lse [Hq, total_q]).
    """
    Hq, total_q, D = q_int8.shape
    Hkv, total_k = k_int8.shape[0], k_int8.shape[1]
    _need(q_int8, torch.int8, "q_int8")
    _need(k_int8, torch.int8, "k_int8")
    _need(q_scale, torch.float32, "q_scale")
    _need(k_scale, torch.float32, "k_scale")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    if v.stride(2) != 1:
        raise ValueError("v channel dimension must be contiguous")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different batch sizes")
    out_dtype = out_dtype or v.dtype
    dev = q_int8.device
    out = torch.empty((total_q, Hq, D), dtype=out_dtype, device=dev)
    lse = torch.empty((Hq, total_q), dtype=torch.float32, device=dev) if return_lse else None
    a = PrefillVarlenArgs()
    a.B, a.Hq, a.Hkv, a.D = B, Hq, Hkv, D
    a.total_q, a.total_k = total_q, total_k
    a.max_seqlen_q, a.max_seqlen_k = int(max_seqlen_q), int(max_seqlen_k)
    a.cu_seqlens_q, a.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    a.q, a.q_scale, a.q_block = _ptr(q_int8), _ptr(q_scale), q_block
    a.k, a.k_scale, a.k_block = _ptr(k_int8), _ptr(k_scale), k_block
    a.v, a.v_dtype = _ptr(v), _dt(v.dtype)
    a.v_stride_t, a.v_stride_h = v.stride(0), v.stride(1)
    if q_bias is not None:
        _need(q_bias, torch.float32, "q_bias")
    a.q_bias = _ptr(q_bias)
    a.causal = int(bool(causal))
    a.sm_scale = float(sm_scale) if sm_scale else 0.0
    a.out, a.out_dtype, a.lse = _ptr(out), _dt(out_dtype), _ptr(lse)
    if v_mean is not None:
        _need(v_mean, torch.float32, "v_mean")
    a.smooth_v, a.v_mean = int(bool(smooth_v)), _ptr(v_mean)
    need = int(lib().sage_attn_prefill_varlen_workspace_size(ctypes.byref(a)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    wsb = workspace.numel() * workspace.element_size()
    if debug_scores is not None:
        _need(debug_scores, torch.int32, "debug_scores")
        _check(lib().sage_debug_prefill_varlen_qk_int32(ctypes.byref(a), _ptr(workspace), wsb,
                                                        _ptr(debug_scores), _stream(stream)))
    else:
        _check(lib().sage_attn_prefill_varlen(ctypes.byref(a), _ptr(workspace), wsb,
                                              _stream(stream)))
    return (out, lse) if return_lse else out


def last_launch_info() -> dict:
    info = LaunchInfo()
    _check(lib().sage_last_launch_info(ctypes.byref(info)))
    return dict(kernel=info.kernel.decode(), grid=tuple(info.grid), block=tuple(info.block),
                cluster=tuple(info.cluster), smem_bytes=info.smem_bytes,
                num_segments=info.num_segments, launches=info.launches)


def check_device_status(stream=None):
    """Synchronise and read/clear the device error word: (status, raw word)."""
    word = _i(0)
    st = lib().sage_check_device_status(_stream(stream), ctypes.byref(word))
    return st, word.value


def debug_timeout_probe(timeout_us: int, stream=None):
    _check(lib().sage_debug_timeout_probe(int(timeout_us), _stream(stream)))
