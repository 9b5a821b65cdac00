"""The allocation-free decode entry point (sage_attn_decode_paged_noalloc).

It exists for callers that cannot allocate device memory for a workspace
(captured graphs with a fixed memory plan, plugins whose host owns every
allocation, embedders that must not re-enter their allocator).  It must give
the same output as sage_attn_decode_paged, which uses a caller workspace, on
consecutive calls that share its built-in scratch array.  This file is named
so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from helpers import assert_close, f32, np_
from int8_quantized_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _args(sage, qi, qs, c, max_len, out, lse, segments=0):
    return sage._decode_args(qi, qs, c.k_cache, c.v_cache, c.k_scale, c.v_scale, c.block_table,
                             c.lens, max_len, None, segments, out, lse)


def _query(sage, B, Hq, D, seed):
    q = W.decode_query(B, Hq, D, seed=seed, device="cuda")
    qi, qs, _, _ = sage.sage_quant_int8(q[:, :, None, :])
    return qi[:, :, 0].contiguous(), qs[:, :, 0].contiguous()


@pytest.mark.parametrize("segments", [0, 5])
def test_noalloc_decode_matches_workspace_decode_twice(sage, segments):
    """segments 0: the library's choice (more than 8 here, partials + combine
    on both paths); 5: the workspace entry point merges the 5 segments inside
    a thread-block cluster, this one through its scratch and the combine
    kernel, so the two merge paths are compared."""
    L = sage.lib()
    B, Hq, Hkv, D = 4, 24, 4, 256
    lens = [8192, 5000, 333, 4096]
    c = W.paged_cache(B, Hkv, D, lens, seed=41, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((42, 43)):          # two calls in a row share the scratch
        qi, qs = _query(sage, B, Hq, D, seed)
        ref, lref = sage.sage_attn_decode_paged(qi, qs, c.k_cache, c.v_cache, c.k_scale,
                                                c.v_scale, c.block_table, c.lens, max(lens),
                                                out_dtype=torch.float16, return_lse=True,
                                                num_segments=segments)
        if segments:
            assert sage.last_launch_info()["launches"] == 1      # in-cluster combine
        out = torch.empty((B, Hq, D), dtype=torch.float16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        a = _args(sage, qi, qs, c, max(lens), out, lse, segments=segments)
        assert L.sage_attn_decode_paged_noalloc(ctypes.byref(a), stream) == 0, \
            L.sage_get_last_error_message()
        torch.cuda.synchronize()
        assert sage.check_device_status()[0] == 0
        info = sage.last_launch_info()
        assert info["kernel"] == "decode_kernel" and info["launches"] == 2
        assert_close(f32(out), f32(ref), "call %d output" % call)
        assert_close(np_(lse), np_(lref), "call %d lse" % call)


def test_noalloc_rejects_requests_beyond_its_scratch(sage):
    L = sage.lib()
    cap = L.sage_attn_decode_noalloc_max_bytes()
    assert cap == 8 << 20
    B, Hq, Hkv, D = 64, 24, 4, 256
    c = W.paged_cache(B, Hkv, D, [1024] * B, seed=5, device="cuda")
    qi, qs = _query(sage, B, Hq, D, 6)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    # 64*24*16 segments*(256+1)*4 bytes > 8 MiB
    a = _args(sage, qi, qs, c, 1024, out, None, segments=16)
    st = L.sage_attn_decode_paged_noalloc(ctypes.byref(a), None)
    assert st == sage.SAGE_ERR_INVALID_ARG
    assert b"scratch" in L.sage_get_last_error_message()


def test_noalloc_rejects_pageable_output_before_launch(sage):
    """An output in ordinary (pageable) host memory is not memory the GPU
    can write: the call refuses it, as the workspace entry point does,
    instead of launching a kernel that would fault."""
    L = sage.lib()
    B, Hq, Hkv, D = 2, 8, 2, 128
    c = W.paged_cache(B, Hkv, D, [64, 64], seed=7, device="cuda")
    qi, qs = _query(sage, B, Hq, D, 8)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16)        # pageable, not pinned
    a = _args(sage, qi, qs, c, 64, torch.empty(1, dtype=torch.bfloat16, device="cuda"), None)
    a.out = ctypes.c_void_p(out.data_ptr())
    st = L.sage_attn_decode_paged_noalloc(ctypes.byref(a), None)
    assert st == sage.SAGE_ERR_INVALID_ARG
    assert b"out" in L.sage_get_last_error_message()
    assert sage.last_launch_info()["launches"] == 0
