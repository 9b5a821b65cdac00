"""Host-side checks of the C ABI that need no GPU: the library builds,
loads, exports every function the header declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

from int8_quantized_attention_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "sage_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sage_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("sage_quant_int8", "sage_attn_prefill", "sage_attn_decode_paged",
                 "sage_splitk_combine"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True).stdout
    ours = sorted(l.split()[-1] for l in out.splitlines() if " T sage_" in l)
    assert ours == declared_functions()


def test_rejects_bad_arguments_on_host(lib):
    # unsupported head dim / dtype and bad strides are refused before any launch
    st = lib.sage_quant_int8(None, 0, 1, 1, 1, 48, 0, 0, 0, 1, 0, None, 0, None, None, None,
                             None, None)
    assert st == binding.SAGE_ERR_UNSUPPORTED
    assert b"head_dim" in lib.sage_get_last_error_message()
    st = lib.sage_quant_int8(None, 7, 1, 1, 1, 64, 0, 0, 0, 1, 0, None, 0, None, None, None,
                             None, None)
    assert st == binding.SAGE_ERR_UNSUPPORTED
    st = lib.sage_quant_int8(ctypes.c_void_p(16), 0, 1, 1, 1, 64, 64, 64, 3, 1, 0, None, 0,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), None, None, None)
    assert st == binding.SAGE_ERR_INVALID_ARG
    st = lib.sage_splitk_combine(None, None, 1, 0, 64, None, 0, None, None)
    assert st == binding.SAGE_ERR_INVALID_ARG
    a = binding.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D = 1, 6, 4, 128
    assert lib.sage_attn_decode_paged(ctypes.byref(a), None, 0, None) == binding.SAGE_ERR_INVALID_ARG
    a.Hkv, a.D = 2, 96
    assert lib.sage_attn_decode_paged(ctypes.byref(a), None, 0, None) == binding.SAGE_ERR_UNSUPPORTED
    assert lib.sage_attn_decode_paged_q16(ctypes.byref(a), None, binding.SAGE_BF16, None, 0,
                                          None) == binding.SAGE_ERR_INVALID_ARG
    p = binding.PrefillArgs()
    p.B, p.Hq, p.Hkv, p.Sq, p.Sk, p.D = 1, 2, 2, 8, 8, 64
    p.q_block, p.k_block = 100, 1
    assert lib.sage_attn_prefill(ctypes.byref(p), None, 0, None) == binding.SAGE_ERR_UNSUPPORTED
    assert lib.sage_attn_prefill(None, None, 0, None) == binding.SAGE_ERR_INVALID_ARG
    assert lib.sage_attn_prefill_workspace_size(None) == 0


def test_workspace_arithmetic(lib):
    assert lib.sage_attn_decode_workspace_size(8, 24, 256, 1) == 0
    n = lib.sage_attn_decode_workspace_size(8, 24, 256, 10)
    rows = 8 * 24 * 10
    assert n >= rows * 256 * 4 + rows * 4


def test_launch_info_struct(lib):
    info = binding.LaunchInfo()
    assert lib.sage_last_launch_info(ctypes.byref(info)) == binding.SAGE_OK
