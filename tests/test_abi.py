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


def test_varlen_scale_group_layout(lib):
    # per token: one group per packed token; per block: total / block + B
    assert lib.sage_varlen_scale_groups(1000, 7, 1) == 1000
    assert lib.sage_varlen_scale_groups(1000, 7, 64) == 1000 // 64 + 7
    # the documented first groups (cu[b] / block + b) leave every sequence
    # ceil(len / block) slots of its own inside that count
    rng = __import__("numpy").random.default_rng(3)
    for block in (64, 128, 256):
        for _ in range(200):
            lens = rng.integers(0, 700, size=rng.integers(1, 12))
            cu = [0]
            for n in lens:
                cu.append(cu[-1] + int(n))
            G = lib.sage_varlen_scale_groups(cu[-1], len(lens), block)
            ends = []
            for b, n in enumerate(lens):
                g0 = cu[b] // block + b
                ends.append((g0, g0 + (int(n) + block - 1) // block))
            for (a0, a1), (b0, _) in zip(ends, ends[1:]):
                assert a1 <= b0
            assert ends[-1][1] <= G


def test_varlen_rejects_bad_arguments_on_host(lib):
    st = lib.sage_quant_int8_varlen(None, 0, 1, 1, 10, 96, 0, 0, None, 10, 1, 0, None, 0, None,
                                    None, None, None, None)
    assert st == binding.SAGE_ERR_UNSUPPORTED
    st = lib.sage_quant_int8_varlen(ctypes.c_void_p(16), 0, 1, 1, 10, 64, 64, 64, None, 10, 1, 0,
                                    None, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                                    None, None)
    assert st == binding.SAGE_ERR_INVALID_ARG     # cu_seqlens missing
    a = binding.PrefillVarlenArgs()
    a.B, a.Hq, a.Hkv, a.D = 2, 6, 4, 128
    a.total_q = a.total_k = 100
    a.max_seqlen_q = a.max_seqlen_k = 60
    a.q_block = a.k_block = 1
    assert lib.sage_attn_prefill_varlen(ctypes.byref(a), None, 0, None) == \
        binding.SAGE_ERR_INVALID_ARG              # Hq % Hkv != 0
    a.Hkv = 2
    a.q_block = 96
    assert lib.sage_attn_prefill_varlen(ctypes.byref(a), None, 0, None) == \
        binding.SAGE_ERR_UNSUPPORTED
    a.q_block = 1
    assert lib.sage_attn_prefill_varlen(ctypes.byref(a), None, 0, None) == \
        binding.SAGE_ERR_INVALID_ARG              # no cu_seqlens
    assert lib.sage_attn_prefill_varlen_workspace_size(None) == 0
    # workspace: K and V f16 copies plus scales over total_k + B * (BN + 4) rows
    need = lib.sage_attn_prefill_varlen_workspace_size(ctypes.byref(a))
    rows = 100 + 2 * (128 + 4)
    assert need >= 2 * (2 * rows * 128 * 2) + 2 * rows * 4


@pytest.mark.parametrize("entry", ["sage_attn_decode_paged", "sage_attn_decode_paged_noalloc"])
def test_decode_rejects_unaligned_out_before_any_launch(lib, entry):
    """An output two bytes off an 8-byte boundary (the single-segment decode
    writes it 8 bytes at a time) is refused by the host checks, which run
    before any CUDA call: the fake pointers here are never dereferenced."""
    a = binding.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D = 1, 4, 4, 128
    a.max_context_len, a.max_blocks, a.num_blocks = 0, 1, 1
    a.q, a.q_scale = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    a.context_lens = ctypes.c_void_p(0x30000)
    a.out, a.out_dtype = ctypes.c_void_p(0x40002), binding.SAGE_BF16
    fn = getattr(lib, entry)
    st = fn(ctypes.byref(a), None, 0, None) if entry == "sage_attn_decode_paged" else \
        fn(ctypes.byref(a), None)
    assert st == binding.SAGE_ERR_INVALID_ARG
    assert b"out must be 8-byte aligned" in lib.sage_get_last_error_message()


def test_prefill_tail_split_workspace_and_check(lib):
    """The tail split's partial results are part of the prefill workspace
    (D = 256, 32 query tiles over 4096 keys: one partial wave), OFF drops
    them, and an unknown tail_split value is rejected before any launch."""
    a = binding.PrefillArgs()
    a.B, a.Hq, a.Hkv, a.Sq, a.Sk, a.D = 1, 8, 2, 512, 4096, 256
    a.q_block, a.k_block, a.v_dtype, a.out_dtype = 128, 64, 0, 0
    a.causal = 0
    with_split = lib.sage_attn_prefill_workspace_size(ctypes.byref(a))
    a.tail_split = 1
    without = lib.sage_attn_prefill_workspace_size(ctypes.byref(a))
    # 32 tiles x 4 parts x 128 rows x (256 + 1) fp32
    assert with_split >= without + 32 * 4 * 128 * 257 * 4
    a.tail_split = 2
    assert lib.sage_attn_prefill_workspace_size(ctypes.byref(a)) == 0
    ws = ctypes.c_void_p(0)
    assert lib.sage_attn_prefill(ctypes.byref(a), ws, 0, None) == binding.SAGE_ERR_INVALID_ARG


def _prefill_ws(lib, **kw):
    a = binding.PrefillArgs()
    a.B, a.Hq, a.Hkv, a.D = kw.get("B", 1), kw["Hq"], kw.get("Hkv", 1), kw["D"]
    a.Sq, a.Sk = kw["Sq"], kw["Sk"]
    a.q_block, a.k_block, a.v_dtype, a.out_dtype = 1, 1, 0, 0
    a.causal = int(kw.get("causal", 0))
    if kw.get("prefix", 0):
        a.max_prefix_len, a.max_blocks = kw["prefix"], (kw["prefix"] + 15) // 16
    a.tail_split = 0
    auto = lib.sage_attn_prefill_workspace_size(ctypes.byref(a))
    a.tail_split = 1
    off = lib.sage_attn_prefill_workspace_size(ctypes.byref(a))
    return auto, off


def test_prefill_tail_split_plan(lib):
    """Host side of the tail split (152 SMs without a GPU): a causal chunk
    over a long prefix at D = 256 with a partial last wave splits (its
    workspace grows by the parts' partial results); causal self-attention,
    a grid of whole waves and D <= 128 do not."""
    # 2048 new tokens over a 16384-token prefix, 24 heads: 384 tiles, 80 in
    # the last wave, split into 3 parts each
    auto, off = _prefill_ws(lib, Hq=24, Hkv=4, D=256, Sq=2048, Sk=2048, prefix=16384, causal=1)
    assert auto - off >= 80 * 3 * 128 * 257 * 4
    # causal self-attention: the tiles' work differs too much
    auto, off = _prefill_ws(lib, Hq=24, D=256, Sq=16384, Sk=16384, causal=1)
    assert auto == off
    # 152 tiles (one full wave): nothing to balance
    auto, off = _prefill_ws(lib, Hq=19, D=256, Sq=1024, Sk=8192)
    assert auto == off
    # head dim 128: never split
    auto, off = _prefill_ws(lib, Hq=24, D=128, Sq=2048, Sk=2048, prefix=16384, causal=1)
    assert auto == off
