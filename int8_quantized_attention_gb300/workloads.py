"""Seeded synthetic inputs for INT8-QK attention.

This module only draws random tensors (it holds none of the method's
arithmetic), so both the CUDA path and the CPU oracle may consume what it
produces.  Shapes and distributions follow the workloads the pages
describe:

* dense prefill: Q/K/V ~ N(0, 1) in fp16/bf16, HND layout, with an
  optional per-(head, channel) K offset ~ N(0, 4) that smooth_k removes;
* packed variable-length batches: the same distributions, token-major
  [total, H, D] with sequence lengths drawn log-uniformly (many short
  sequences and a few long ones, the mix a varlen batch serves);
* paged decode / paged prefix: INT8 cache values uniform in [-127, 127],
  per-token per-KV-head fp32 scales ~ U(0.005, 0.02), cache layout
  [block, kv_head, head_dim/16, 16, 16], block table a random
  permutation of the physical pages.

Every generator takes a seed and a device; the same seed and device give
the same tensors.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

PAGE = 16

_DT = {"fp16": torch.float16, "bf16": torch.bfloat16, "f16": torch.float16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, dtype, std=1.0, offset_shape=None, offset_std=0.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if offset_shape is not None and offset_std > 0:
        x += torch.randn(offset_shape, generator=g, device=device, dtype=torch.float32) * offset_std
    return x.to(dtype)


@dataclass
class PagedCache:
    k_cache: torch.Tensor      # int8 [nblk, Hkv, D/16, 16, 16]
    v_cache: torch.Tensor      # int8 [nblk, Hkv, D/16, 16, 16]
    k_scale: torch.Tensor      # fp32 [nblk, Hkv, 16]
    v_scale: torch.Tensor      # fp32 [nblk, Hkv, 16]
    block_table: torch.Tensor  # int32 [B, maxblk]
    lens: torch.Tensor         # int32 [B]


def paged_cache(B: int, Hkv: int, D: int, lens, seed: int, device="cpu",
                extra_blocks: int = 0, max_blocks: Optional[int] = None) -> PagedCache:
    """Random INT8 paged K/V cache holding ``lens[b]`` tokens for sequence b.

    Physical pages are a random permutation; ``extra_blocks`` unused pages
    are added to the pool so that the table does not cover it exactly.
    """
    g = _gen(seed, device)
    lens = [int(x) for x in lens]
    need = [(n + PAGE - 1) // PAGE for n in lens]
    maxblk = max(max(need) if need else 0, 1) if max_blocks is None else max_blocks
    nblk = sum(need) + extra_blocks
    nblk = max(nblk, 1)
    kc = torch.randint(-127, 128, (nblk, Hkv, D // 16, PAGE, 16), generator=g, device=device,
                       dtype=torch.int8)
    vc = torch.randint(-127, 128, (nblk, Hkv, D // 16, PAGE, 16), generator=g, device=device,
                       dtype=torch.int8)
    ks = torch.rand((nblk, Hkv, PAGE), generator=g, device=device) * 0.015 + 0.005
    vs = torch.rand((nblk, Hkv, PAGE), generator=g, device=device) * 0.015 + 0.005
    perm = torch.randperm(nblk, generator=g, device=device).to(torch.int32)
    bt = torch.zeros((B, maxblk), dtype=torch.int32, device=device)
    pos = 0
    for b in range(B):
        bt[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    return PagedCache(kc, vc, ks, vs, bt, torch.tensor(lens, dtype=torch.int32, device=device))


@dataclass
class DenseQKV:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor


def dense_qkv(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, seed: int, dtype="fp16",
              device="cpu", k_offset_std: float = 0.0, v_dtype=None) -> DenseQKV:
    """Q [B,Hq,Sq,D], K/V [B,Hkv,Sk,D] ~ N(0,1); K gets a per-(head, channel)
    offset ~ N(0, k_offset_std^2) shared by all tokens and batches."""
    g = _gen(seed, device)
    dt = _DT[dtype]
    vdt = _DT[v_dtype] if v_dtype else dt
    q = _normal((B, Hq, Sq, D), g, device, dt)
    k = _normal((B, Hkv, Sk, D), g, device, dt, offset_shape=(1, Hkv, 1, D),
                offset_std=k_offset_std)
    v = _normal((B, Hkv, Sk, D), g, device, vdt)
    return DenseQKV(q, k, v)


@dataclass
class VarlenQKV:
    q: torch.Tensor            # [total_q, Hq, D]
    k: torch.Tensor            # [total_k, Hkv, D]
    v: torch.Tensor            # [total_k, Hkv, D]
    cu_q: torch.Tensor         # int32 [B + 1]
    cu_k: torch.Tensor         # int32 [B + 1]
    max_q: int
    max_k: int


def varlen_lengths(n: int, lo: int, hi: int, seed: int):
    """n sequence lengths, log-uniform in [lo, hi] (seeded, CPU)."""
    g = _gen(seed, "cpu")
    u = torch.rand((n,), generator=g, dtype=torch.float64)
    return [int(round(lo * (hi / lo) ** float(x))) for x in u]


def varlen_qkv(lens_q, lens_k, Hq: int, Hkv: int, D: int, seed: int, dtype="fp16", device="cpu",
               k_offset_std: float = 0.0, v_dtype=None) -> VarlenQKV:
    """Packed token-major Q/K/V ~ N(0,1); K gets a per-(head, channel) offset
    ~ N(0, k_offset_std^2) shared by every token of the batch."""
    g = _gen(seed, device)
    dt = _DT[dtype]
    vdt = _DT[v_dtype] if v_dtype else dt
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = _normal((tq, Hq, D), g, device, dt)
    k = _normal((tk, Hkv, D), g, device, dt, offset_shape=(1, Hkv, D), offset_std=k_offset_std)
    v = _normal((tk, Hkv, D), g, device, vdt)

    def cu(lens):
        c = [0]
        for n in lens:
            c.append(c[-1] + int(n))
        return torch.tensor(c, dtype=torch.int32, device=device)

    return VarlenQKV(q, k, v, cu(lens_q), cu(lens_k), max(lens_q, default=0),
                     max(lens_k, default=0))


def decode_query(B: int, Hq: int, D: int, seed: int, dtype="bf16", device="cpu") -> torch.Tensor:
    """One new query token per sequence: [B, Hq, D] ~ N(0, 1)."""
    g = _gen(seed, device)
    return _normal((B, Hq, D), g, device, _DT[dtype])


# ----------------------------------------------------------------------------
# The named workloads (sizes as the pages' configurations state them)
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    params: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny_prefill": Workload("tiny_prefill", dict(B=1, Hq=2, Hkv=2, S=128, D=64, dtype="fp16",
                                                  seed=0, q_block=1, k_block=1, smooth_k=False,
                                                  causal=False)),
    "paged_decode": Workload("paged_decode", dict(B=8, Hq=24, Hkv=4, D=256, ctx=8192,
                                                  dtype="bf16", seed=1)),
    "chunked_prefill": Workload("chunked_prefill", dict(B=1, Hq=24, Hkv=4, S=2048, prefix=16384,
                                                        D=256, dtype="bf16", seed=2, q_block=1,
                                                        k_block=1, smooth_k=True, causal=True,
                                                        k_offset_std=2.0)),
    "dense_prefill": Workload("dense_prefill", dict(B=2, Hq=32, Hkv=32, S=16384, D=128,
                                                    dtype="fp16", seed=3, q_block=128,
                                                    k_block=64, smooth_k=True, causal=True,
                                                    k_offset_std=2.0, return_lse=True)),
    "varlen_prefill": Workload("varlen_prefill", dict(n=24, lo=256, hi=8192, Hq=32, Hkv=8,
                                                      D=128, dtype="fp16", seed=5, q_block=128,
                                                      k_block=64, smooth_k=True, causal=True,
                                                      k_offset_std=2.0)),
    "decode_sweep": Workload("decode_sweep", dict(Hq=24, Hkv=4, D=256, dtype="bf16", seed=4,
                                                  ctx=(8192, 16384, 32768), batch=(1, 16, 64))),
}
