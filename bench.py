"""Benchmark of the INT8-QK attention hot path on GB300.

One step = one pass of the decode hot path over one batch of the paged
decode workload (batch 8, 24 query / 4 KV heads, head_dim 256, 8192-token
INT8 paged context): quantise the bf16 query (INT8, per token/head), run
the split-K paged decode kernel, merge the segments with the LSE combine.

Prints ONE JSON line (rank 0).  `value` is the decode workload's
algorithmic bytes (INT8 K/V pages + their scales + block table + context
lengths + bf16 query in + bf16 output) per second of device time, inputs
resident in HBM, L2 flushed between steps.  `e2e` is the same metric
through the public API with the per-step inputs (query, block table,
context lengths) and the output in pinned host memory: the kernels read
and write them in place across NVLink-C2C inside every timed step (no
copy-engine transfer); the KV cache is device-resident state, as in
serving.  `roofline` describes the decode kernel launched on its own
(events around that one launch).  The dense and chunked prefill workloads
are measured under `prefill`, each with its own `roofline` (the prefill
kernel against the tensor peak) and `cpu_baseline` (the oracle on a row
sample, scaled by work).

--impl reference times the CPU oracle (the plain C reference of the
method) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT8-QK attention prefill TFLOP/s and paged-decode KV GB/s on 1 GB300 (% roofline)"
WORKLOAD = "paged_decode"
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2


def l2_flush(buf):
    """Evict L2 by READING a buffer 4x its size (clean lines: no write-back of
    the flush itself lands inside the next timed region)."""
    buf.max()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest of every rank's value (the slowest replica's time); the
    value itself with one process."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput of N replicas: every rank's units over the
    slowest rank's time (weak scaling), in units per second."""
    return units_per_rank * world * steps / (max_ms * 1e-3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def decode_bytes(B, Hq, Hkv, D, ctx, max_blocks):
    """Algorithmic bytes of one decode step (what the method must move) and
    of the decode kernel launched alone in the partials form (INT8 query
    codes and scales in; the split-K partials it writes are not algorithmic
    bytes)."""
    kv = 2 * B * ctx * Hkv * D            # INT8 K and V pages
    scales = 2 * B * ctx * Hkv * 4        # fp32 per-token K and V scales
    table = B * max_blocks * 4 + B * 4    # block table + context lengths
    q_bf16 = B * Hq * D * 2               # query in (quantised inside the decode kernel)
    out = B * Hq * D * 2                  # bf16 output
    step = kv + scales + table + q_bf16 + out
    kernel = kv + scales + table + B * Hq * (D + 4)
    return kernel, step


def run_ours(args):
    import torch

    from int8_quantized_attention_gb300 import binding as sage
    from int8_quantized_attention_gb300 import build
    from int8_quantized_attention_gb300 import workloads as W

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    build.build()
    P = W.WORKLOADS[WORKLOAD].params
    B, Hq, Hkv, D, ctx = P["B"], P["Hq"], P["Hkv"], P["D"], P["ctx"]
    # every rank runs its own replica of the workload (independent batches)
    cache = W.paged_cache(B, Hkv, D, [ctx] * B, seed=P["seed"] + rank, device="cuda")
    q = W.decode_query(B, Hq, D, seed=P["seed"] + rank, device="cuda")
    max_blocks = cache.block_table.shape[1]
    S = args.segments or sage.decode_num_segments(B, Hq, Hkv, D, ctx)
    kbytes, sbytes = decode_bytes(B, Hq, Hkv, D, ctx, max_blocks)
    stream = torch.cuda.current_stream()
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    ws_step = torch.empty(max(1, sage.decode_workspace_size(B, Hq, D, S)), dtype=torch.uint8,
                          device="cuda")
    out_step = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    launches = {"n": 0}

    def step(ev=None):
        # one launch: per-token query quantisation, split-K paged decode and
        # (up to 8 segments) the LSE combine all run in the decode kernel
        if ev is not None:
            ev[0].record(stream)
        out = sage.sage_attn_decode_paged_q16(q, cache.k_cache, cache.v_cache, cache.k_scale,
                                              cache.v_scale, cache.block_table, cache.lens, ctx,
                                              num_segments=S, workspace=ws_step, out=out_step)
        if ev is not None:
            ev[1].record(stream)
        launches["n"] = sage.last_launch_info()["launches"]
        return out

    clk = ClockSampler(local).__enter__()   # samples from warm-up through the timed steps
    for _ in range(args.warmup):
        step()
        l2_flush(flush)
    torch.cuda.synchronize()
    st, word = sage.check_device_status()
    if st != 0:
        raise RuntimeError("device error word %d after warm-up" % word)

    # the step (quantise the query + decode with the in-cluster combine) is
    # captured once as a CUDA graph and replayed: host launch overhead stays
    # out of the device-timed step, as in a serving loop
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        l2_flush(flush)               # L2 flush outside the timed window
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    barrier()
    # The decode kernel on its own: the partials form launches the same
    # decode_kernel<256> grid (same segments, same pages) without the
    # combine behind it, with the query codes quantised beforehand; events
    # bracket that one launch, L2 flushed before each.
    qi, qs, _, _ = sage.sage_quant_int8(q[:, :, None, :])
    qi, qs = qi[:, :, 0].contiguous(), qs[:, :, 0].contiguous()
    for i in range(args.steps):
        l2_flush(flush)
        kev[i][0].record(stream)
        sage.sage_attn_decode_paged_partials(qi, qs, cache.k_cache, cache.v_cache, cache.k_scale,
                                             cache.v_scale, cache.block_table, cache.lens, ctx, S)
        kev[i][1].record(stream)
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    t_ms = max_over_ranks(sum(step_ms), device="cuda")
    value = whole_job_rate(sbytes, ws, args.steps, t_ms) / 1e9

    # ---- end to end through the public API, host buffers: the step's
    # inputs (query, block table, context lengths) and its output live in
    # pinned host memory and are handed to the API as they are; the decode
    # kernel reads them and writes the result across NVLink-C2C inside the
    # step (GB300's CPU-GPU link; no copy-engine transfer).  L2 is flushed
    # between steps, so every step moves its inputs from the host again.
    e2e = None
    if rank == 0 or ws > 1:
        q_host = q.cpu().pin_memory()
        bt_host = cache.block_table.cpu().pin_memory()
        lens_host = cache.lens.cpu().pin_memory()
        out_host = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
        # segment count: the library's own choice for host-resident I/O
        S_e2e = args.segments
        ws_buf = torch.empty(max(1, sage.decode_workspace_size(B, Hq, D, 64)), dtype=torch.uint8,
                             device="cuda")

        def e2e_step():
            sage.sage_attn_decode_paged_q16(q_host, cache.k_cache, cache.v_cache, cache.k_scale,
                                            cache.v_scale, bt_host, lens_host, ctx,
                                            num_segments=S_e2e, workspace=ws_buf, out=out_host)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            l2_flush(flush)
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize()
        e_ms = sum(a.elapsed_time(b) for a, b in zip(es, ee))
        h2d = q_host.numel() * 2 + bt_host.numel() * 4 + lens_host.numel() * 4
        d2h = out_host.numel() * 2
        e2e = {"value": round(sbytes * args.steps / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms / args.steps, 5),
               "method": "per step: sage_attn_decode_paged_q16 called on pinned host "
                         "buffers (query, block table, context lengths in; bf16 output out), "
                         "read and written over NVLink-C2C (the query quantised once by the "
                         "library's quantisation kernel, the decode launched behind it); "
                         "eager call, no graph"}
    torch.cuda.synchronize()
    st, word = sage.check_device_status()
    if st != 0:
        raise RuntimeError("device error word %d after the timed region" % word)

    peaks, kind = _peaks()
    k_avg = statistics.mean(kern_ms)
    achieved = kbytes / (k_avg * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": "decode_kernel", "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_kind": kind, "traffic": _profile_traffic("decode_kernel"),
            "algorithmic_bytes": kbytes, "avg_launch_ms": round(k_avg, 5),
            "launch": "decode_kernel alone (partials form: %d segments, no combine), CUDA events "
                      "around the launch, L2 flushed before each" % S,
            "step_frac": round(value / peaks["hbm_gbs"], 4)}
    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8",
        "data": "synthetic (seeded; uniform INT8 cache, U(0.005,0.02) scales, N(0,1) bf16 query)",
        "config": {"workload": "paged_decode B8 Hq24 Hkv4 D256 ctx8192 block16",
                   "segments": S, "l2": "flushed between steps (read of a 512 MB buffer)",
                   "step": "query quant + split-K paged decode + in-cluster LSE combine, one kernel"
                           if 1 < S <= 8 else "query quant + split-K paged decode (one kernel) + LSE combine",
                   "launch": "CUDA graph replay per step",
                   "parallelism": "replicas" if ws > 1 else "single"},
        "roofline": roof, "e2e": e2e, "gpu_launches": launches["n"] * args.steps,
        "clocks": clk.summary(),
    }
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(args.cpu_seconds)
    if args.prefill:
        line["prefill"] = prefill_measure(args)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return line


def _profile_traffic(kernel):
    """dram bytes per launch from the committed ncu summary of the workload, if any."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    return d.get(kernel)


def cpu_baseline_decode(seconds: float):
    """The oracle timed on the host cores on a bounded sample of the workload."""
    import numpy as np

    import oracle
    from int8_quantized_attention_gb300 import workloads as W

    P = W.WORKLOADS[WORKLOAD].params
    B, Hq, Hkv, D, ctx = P["B"], P["Hq"], P["Hkv"], P["D"], P["ctx"]
    cache = W.paged_cache(B, Hkv, D, [ctx] * B, seed=P["seed"], device="cpu")
    q = W.decode_query(B, Hq, D, seed=P["seed"], device="cpu").float().numpy()
    qi, qs, _ = oracle.quant_int8(q[:, :, None, :])
    qi, qs = qi[:, :, 0], qs[:, :, 0]
    args = [cache.k_cache.numpy(), cache.v_cache.numpy(), cache.k_scale.numpy(),
            cache.v_scale.numpy(), cache.block_table.numpy(), cache.lens.numpy()]
    threads = oracle.default_threads()
    _, sbytes = decode_bytes(B, Hq, Hkv, D, ctx, cache.block_table.shape[1])
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_paged(qi, qs, *args, threads=threads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds or passes >= 1000:
            break
    return {"value": round(sbytes * passes / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d full pass(es) of the paged_decode workload (all 8x4 sequence/kv-head "
                      "pairs), %.1f s" % (passes, el)}


def prefill_flops(B, Hq, Sq, prefix, Sk, D, causal):
    """4*D FLOP per unmasked (query, key) pair (QK^T and P.V)."""
    if not causal:
        pairs = Sq * (prefix + Sk)
    else:
        off = prefix + Sk - Sq
        pairs = sum(max(0, min(prefix + Sk, i + off + 1)) for i in range(Sq))
    return 4 * D * B * Hq * pairs


def _oracle_prefill_sample(name, qi, qs, ki, ks, v, bias, prefix_cache, plen, P, threads):
    """The oracle on one (batch, head) and 16 evenly spaced query rows of a
    prefill workload; returns (seconds, FLOP of that sample)."""
    import numpy as np

    import oracle

    Sq, D = P["S"], P["D"]
    rows = np.arange(Sq) if Sq <= 128 else np.linspace(0, Sq - 1, 16).astype(np.int64)
    sub = lambda t: t[0:1, 0:1].cpu().numpy()
    pre = None
    if prefix_cache is not None:
        c = prefix_cache
        pre = dict(k_cache=c.k_cache.cpu().numpy(), v_cache=c.v_cache.cpu().numpy(),
                   k_scale=c.k_scale.cpu().numpy(), v_scale=c.v_scale.cpu().numpy(),
                   block_table=c.block_table.cpu().numpy(), lens=c.lens.cpu().numpy())
    t0 = time.perf_counter()
    oracle.prefill(sub(qi), sub(qs), P["q_block"], sub(ki), sub(ks), P["k_block"],
                   sub(v.float()), causal=P["causal"],
                   q_bias=None if bias is None else sub(bias).astype(np.float64), prefix=pre,
                   rows=rows, threads=threads)
    el = time.perf_counter() - t0
    vis = lambda i: min(plen + Sq, int(i) + plen + 1) if P["causal"] else plen + Sq
    return el, 4 * D * sum(vis(i) for i in rows)


def prefill_measure(args):
    """Prefill throughput on the dense and chunked prefill workloads: the
    prefill call (staging pass + prefill_kernel) timed with CUDA events, its
    roofline against the measured dense tensor peak, the call with the Q/K
    quantisation in front of it, and the oracle on a row sample as the CPU
    baseline (scaled by FLOP, marked extrapolated)."""
    import torch

    import oracle
    from int8_quantized_attention_gb300 import binding as sage
    from int8_quantized_attention_gb300 import workloads as W

    peaks, kind = _peaks()
    peak = peaks["bf16_tflops"]   # f16 dense tensor rate = bf16 rate (nominal ratio 1)
    stream = torch.cuda.current_stream()
    threads = oracle.default_threads()
    res = {}
    for name in ("dense_prefill", "chunked_prefill"):
        P = W.WORKLOADS[name].params
        qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                          dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
        prefix, plen, pc = None, 0, None
        if name == "chunked_prefill":
            pc = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["prefix"]], seed=P["seed"],
                               device="cuda")
            plen = P["prefix"]
            prefix = dict(k_cache=pc.k_cache, v_cache=pc.v_cache, k_scale=pc.k_scale,
                          v_scale=pc.v_scale, block_table=pc.block_table, lens=pc.lens,
                          max_len=plen)
        qb, kb = P["q_block"], P["k_block"]

        def quant():
            ki, ks, mu, _ = sage.sage_quant_int8(qkv.k, block_tokens=kb, smooth=True)
            qi, qs, _, bias = sage.sage_quant_int8(qkv.q, block_tokens=qb, mu_in=mu)
            return qi, qs, ki, ks, bias

        qi, qs, ki, ks, bias = quant()

        def attn():
            return sage.sage_attn_prefill(qi, qs, qb, ki, ks, kb, qkv.v, causal=P["causal"],
                                          q_bias=bias, prefix=prefix,
                                          return_lse=P.get("return_lse", False))

        for _ in range(args.warmup):
            attn()
        torch.cuda.synchronize()
        n = max(3, min(args.steps, 10))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            attn()
            b.record(stream)
        torch.cuda.synchronize()
        k_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        launches = sage.last_launch_info()["launches"]
        sv = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in sv:
            a.record(stream)
            qi, qs, ki, ks, bias = quant()
            attn()
            b.record(stream)
        torch.cuda.synchronize()
        s_ms = statistics.mean(a.elapsed_time(b) for a, b in sv)
        st, word = sage.check_device_status()
        if st != 0:
            raise RuntimeError("device error word %d in %s" % (word, name))
        fl = prefill_flops(P["B"], P["Hq"], P["S"], plen, P["S"], P["D"], P["causal"])
        tf = fl / (k_ms * 1e-3) / 1e12
        cpu = None
        if args.cpu_baseline:
            el, fl_s = _oracle_prefill_sample(name, qi, qs, ki, ks, qkv.v, bias, pc, plen, P,
                                              threads)
            cpu = {"value": round(fl_s / el / 1e12, 8), "unit": "TFLOP/s", "cores": threads,
                   "kind": "oracle",
                   "sample": "1 (batch, head) x 16 evenly spaced query rows (%.2f s, %.3g FLOP); "
                             "extrapolated: the full workload would take %.0f s" %
                             (el, fl_s, el * fl / fl_s)}
        res[name] = {
            "tflops": round(tf, 1), "kernel_ms": round(k_ms, 4), "launches_per_call": launches,
            "step_ms_with_quant": round(s_ms, 4),
            "step_tflops_with_quant": round(fl / (s_ms * 1e-3) / 1e12, 1), "flop": fl,
            "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": round(tf, 1),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                         "peak_kind": kind + " bf16 dense (f16 runs at the same nominal rate)",
                         "traffic": _profile_traffic("prefill_kernel:" + name),
                         "algorithmic_flop": fl, "avg_launch_ms": round(k_ms, 4),
                         "launch": "the prefill call (staging pass + prefill_kernel), CUDA "
                                   "events around it, %d calls" % n},
            "cpu_baseline": cpu}
        del qkv, qi, qs, ki, ks, bias, prefix, pc
        torch.cuda.empty_cache()
    return res


def run_profile(args):
    """Launch one kernel of a named workload a few times (for ncu captures).

    --profile dense_prefill|chunked_prefill|varlen_prefill|paged_decode,
    --heads H shrinks the query heads (and KV heads in proportion) to keep a
    capture small.
    """
    import torch

    from int8_quantized_attention_gb300 import binding as sage
    from int8_quantized_attention_gb300 import build
    from int8_quantized_attention_gb300 import workloads as W

    build.build()
    P = dict(W.WORKLOADS["paged_decode" if args.profile == "kv_producer" else args.profile].params)
    if args.heads:
        ratio = P["Hq"] // P["Hkv"]
        P["Hq"] = args.heads
        P["Hkv"] = max(1, args.heads // ratio)
    if args.profile == "paged_decode":
        c = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["ctx"]] * P["B"], seed=P["seed"],
                          device="cuda")
        q = W.decode_query(P["B"], P["Hq"], P["D"], seed=P["seed"], device="cuda")
        run = lambda: sage.sage_attn_decode_paged_q16(q, c.k_cache, c.v_cache, c.k_scale,
                                                      c.v_scale, c.block_table, c.lens, P["ctx"],
                                                      pv_mode=args.pv_mode)
    elif args.profile == "kv_producer":
        # the KV producer of a 2048-token chunk of the chunked-prefill shape
        # (24 query / 4 KV heads, D 256) appended after a 16384-token context
        n, ctx = 2048, 16384
        c = W.paged_cache(1, P["Hkv"], P["D"], [ctx + n], seed=9, device="cuda")
        g = torch.Generator("cuda").manual_seed(10)
        kn = torch.randn((1, P["Hkv"], n, P["D"]), generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn((1, P["Hkv"], n, P["D"]), generator=g, device="cuda").to(torch.bfloat16)
        qn = torch.randn((1, P["Hq"], n, P["D"]), generator=g, device="cuda").to(torch.bfloat16)
        pos = torch.full((1,), ctx, dtype=torch.int32, device="cuda")
        run = lambda: sage.sage_kv_producer(qn, kn, vn, c.k_cache, c.v_cache, c.k_scale,
                                            c.v_scale, c.block_table, pos)
    elif args.profile == "varlen_prefill":
        lens = W.varlen_lengths(P["n"], P["lo"], P["hi"], P["seed"])
        x = W.varlen_qkv(lens, lens, P["Hq"], P["Hkv"], P["D"], seed=P["seed"], dtype=P["dtype"],
                         device="cuda", k_offset_std=P["k_offset_std"])
        ki, ks, mu, _ = sage.sage_quant_int8_varlen(x.k, x.cu_k, x.max_k,
                                                    block_tokens=P["k_block"], smooth=True)
        qi, qs, _, bias = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q,
                                                      block_tokens=P["q_block"], mu_in=mu)
        run = lambda: sage.sage_attn_prefill_varlen(qi, qs, P["q_block"], ki, ks, P["k_block"],
                                                    x.v, x.cu_q, x.cu_k, x.max_q, x.max_k,
                                                    causal=P["causal"], q_bias=bias,
                                                    return_lse=True)
    else:
        qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], P["S"], P["S"], P["D"], seed=P["seed"],
                          dtype=P["dtype"], device="cuda", k_offset_std=P["k_offset_std"])
        prefix = None
        if args.profile == "chunked_prefill":
            c = W.paged_cache(P["B"], P["Hkv"], P["D"], [P["prefix"]], seed=P["seed"],
                              device="cuda")
            prefix = dict(k_cache=c.k_cache, v_cache=c.v_cache, k_scale=c.k_scale,
                          v_scale=c.v_scale, block_table=c.block_table, lens=c.lens,
                          max_len=P["prefix"])
        ki, ks, mu, _ = sage.sage_quant_int8(qkv.k, block_tokens=P["k_block"], smooth=True)
        qi, qs, _, bias = sage.sage_quant_int8(qkv.q, block_tokens=P["q_block"], mu_in=mu)
        run = lambda: sage.sage_attn_prefill(qi, qs, P["q_block"], ki, ks, P["k_block"], qkv.v,
                                             causal=P["causal"], q_bias=bias, prefix=prefix)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    st, word = sage.check_device_status()
    print(json.dumps({"profile": args.profile, "params": P, "launches": args.warmup + args.steps,
                      "status": st}))
    return None


def run_configs(args):
    """Every configuration of the workload table, one JSON line each: GPU time
    (CUDA events, L2 flushed before each timed call), throughput, fraction of
    the measured peak, and the CPU oracle's time on the host cores (full for
    the small configurations, a row/pair sample scaled by work otherwise)."""
    import numpy as np
    import torch

    import oracle
    from int8_quantized_attention_gb300 import binding as sage
    from int8_quantized_attention_gb300 import workloads as W

    sage.lib()
    peaks, kind = _peaks()
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    threads = oracle.default_threads()

    def gpu_ms(fn, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ts.sort()
        return statistics.median(ts)

    def emit(d):
        print(json.dumps(d), flush=True)

    # ---- prefill configurations
    for name in ("tiny_prefill", "chunked_prefill", "dense_prefill"):
        P = W.WORKLOADS[name].params
        Sq = P["S"]
        prefix_len = P.get("prefix", 0)
        qkv = W.dense_qkv(P["B"], P["Hq"], P["Hkv"], Sq, Sq, P["D"], seed=P["seed"],
                          dtype=P["dtype"], device="cuda", k_offset_std=P.get("k_offset_std", 0.0))
        prefix, pc = None, None
        if prefix_len:
            pc = W.paged_cache(P["B"], P["Hkv"], P["D"], [prefix_len], seed=P["seed"], device="cuda")
            prefix = dict(k_cache=pc.k_cache, v_cache=pc.v_cache, k_scale=pc.k_scale,
                          v_scale=pc.v_scale, block_table=pc.block_table, lens=pc.lens,
                          max_len=prefix_len)
        qb, kb = P["q_block"], P["k_block"]
        ki, ks, mu, _ = sage.sage_quant_int8(qkv.k, block_tokens=kb, smooth=P["smooth_k"])
        qi, qs, _, bias = sage.sage_quant_int8(qkv.q, block_tokens=qb,
                                               mu_in=mu if P["smooth_k"] else None)
        sm = 1.0 / 8.0 if name == "tiny_prefill" else None
        ws = torch.empty(1, dtype=torch.uint8, device="cuda")
        out = sage.sage_attn_prefill(qi, qs, qb, ki, ks, kb, qkv.v, causal=P["causal"],
                                     q_bias=bias, prefix=prefix, sm_scale=sm)
        fn = lambda: sage.sage_attn_prefill(qi, qs, qb, ki, ks, kb, qkv.v, causal=P["causal"],
                                            q_bias=bias, prefix=prefix, sm_scale=sm)
        ms = gpu_ms(fn)
        flop = prefill_flops(P["B"], P["Hq"], Sq, prefix_len, Sq, P["D"], P["causal"])
        tf = flop / (ms * 1e-3) / 1e12
        # oracle: one (batch, head) on a row sample, scaled by visible pairs
        rows = np.arange(Sq) if Sq <= 128 else np.linspace(0, Sq - 1, 16).astype(np.int64)
        sub = lambda t: t[0:1, 0:1].cpu().numpy()
        pre = None
        if pc is not None:
            pre = dict(k_cache=pc.k_cache.cpu().numpy(), v_cache=pc.v_cache.cpu().numpy(),
                       k_scale=pc.k_scale.cpu().numpy(), v_scale=pc.v_scale.cpu().numpy(),
                       block_table=pc.block_table.cpu().numpy(), lens=pc.lens.cpu().numpy())
        t0 = time.perf_counter()
        oracle.prefill(sub(qi), sub(qs), qb, sub(ki), sub(ks), kb, sub(qkv.v.float()),
                       causal=P["causal"], sm_scale=sm,
                       q_bias=None if bias is None else sub(bias).astype(np.float64),
                       prefix=pre, rows=rows, threads=threads)
        t_or = time.perf_counter() - t0
        off = prefix_len + Sq - Sq
        vis = lambda i: (min(prefix_len + Sq, i + off + 1) if P["causal"] else prefix_len + Sq)
        pairs_s = sum(vis(int(i)) for i in rows)
        scale = flop / (4 * P["D"]) / pairs_s
        emit({"config": name, "gpu_ms": round(ms, 4), "tflops": round(tf, 1),
              "frac_of_measured_f16_peak": round(tf / peaks["bf16_tflops"], 4),
              "oracle_s": round(t_or * scale, 2), "oracle_cores": threads,
              "oracle_sample": "full" if scale == 1 else "1 (batch, head), %d rows, scaled x%.0f" % (len(rows), scale)})
        del qkv, qi, ki, out

    # ---- packed variable-length prefill (one launch over every sequence)
    P = W.WORKLOADS["varlen_prefill"].params
    lens = W.varlen_lengths(P["n"], P["lo"], P["hi"], P["seed"])
    x = W.varlen_qkv(lens, lens, P["Hq"], P["Hkv"], P["D"], seed=P["seed"], dtype=P["dtype"],
                     device="cuda", k_offset_std=P["k_offset_std"])
    qb, kb = P["q_block"], P["k_block"]
    ki, ks, mu, _ = sage.sage_quant_int8_varlen(x.k, x.cu_k, x.max_k, block_tokens=kb, smooth=True)
    qi, qs, _, bias = sage.sage_quant_int8_varlen(x.q, x.cu_q, x.max_q, block_tokens=qb, mu_in=mu)
    vws = torch.empty(sage.prefill_varlen_workspace_size(len(lens), P["Hq"], P["Hkv"], P["D"],
                                                        x.q.shape[0], x.k.shape[0], x.max_q,
                                                        x.max_k),
                      dtype=torch.uint8, device="cuda")
    fn = lambda: sage.sage_attn_prefill_varlen(qi, qs, qb, ki, ks, kb, x.v, x.cu_q, x.cu_k,
                                               x.max_q, x.max_k, causal=P["causal"], q_bias=bias,
                                               return_lse=True, workspace=vws)
    ms = gpu_ms(fn)
    flop = sum(4 * P["D"] * P["Hq"] * (n * (n + 1) // 2 if P["causal"] else n * n) for n in lens)
    tf = flop / (ms * 1e-3) / 1e12
    # oracle: the longest sequence, one head, 16 rows, scaled by visible pairs
    bl = int(np.argmax(lens))
    cq = x.cu_q.cpu().numpy()
    n = lens[bl]
    t0s, t1s = int(cq[bl]), int(cq[bl + 1])
    g0q, g0k = t0s // qb + bl, t0s // kb + bl
    rows = np.linspace(0, n - 1, 16).astype(np.int64)
    t0 = time.perf_counter()
    oracle.prefill(qi[0:1, t0s:t1s][None].cpu().numpy(),
                   qs[0:1, g0q:g0q + (n + qb - 1) // qb][None].cpu().numpy(), qb,
                   ki[0:1, t0s:t1s][None].cpu().numpy(),
                   ks[0:1, g0k:g0k + (n + kb - 1) // kb][None].cpu().numpy(), kb,
                   x.v[t0s:t1s, 0:1].float().transpose(0, 1)[None].cpu().numpy(),
                   causal=P["causal"], q_bias=bias[0:1, t0s:t1s][None].cpu().numpy().astype(np.float64),
                   rows=rows, threads=threads)
    t_or = time.perf_counter() - t0
    pairs_s = sum(int(i) + 1 for i in rows) if P["causal"] else len(rows) * n
    scale = flop / (4 * P["D"]) / pairs_s
    emit({"config": "varlen_prefill", "sequences": len(lens), "tokens": int(sum(lens)),
          "gpu_ms": round(ms, 4), "tflops": round(tf, 1),
          "frac_of_measured_f16_peak": round(tf / peaks["bf16_tflops"], 4),
          "oracle_s": round(t_or * scale, 2), "oracle_cores": threads,
          "oracle_sample": "1 sequence x 1 head, %d rows, scaled x%.0f" % (len(rows), scale)})
    del x, qi, ki

    # ---- decode configurations
    P = W.WORKLOADS["paged_decode"].params
    shapes = [("paged_decode", P["B"], P["ctx"])]
    SW = W.WORKLOADS["decode_sweep"].params
    shapes += [("decode_sweep", b, c) for c in SW["ctx"] for b in SW["batch"]]
    for name, B, ctx in shapes:
        Hq, Hkv, D = P["Hq"], P["Hkv"], P["D"]
        cache = W.paged_cache(B, Hkv, D, [ctx] * B, seed=P["seed"], device="cuda")
        q = W.decode_query(B, Hq, D, seed=P["seed"], device="cuda")
        S = sage.decode_num_segments(B, Hq, Hkv, D, ctx)
        ws = torch.empty(max(1, sage.decode_workspace_size(B, Hq, D, S)), dtype=torch.uint8,
                         device="cuda")
        fn = lambda: sage.sage_attn_decode_paged_q16(q, cache.k_cache, cache.v_cache,
                                                     cache.k_scale, cache.v_scale,
                                                     cache.block_table, cache.lens, ctx,
                                                     num_segments=S, workspace=ws)
        ms = gpu_ms(fn)
        _, sbytes = decode_bytes(B, Hq, Hkv, D, ctx, cache.block_table.shape[1])
        gbs = sbytes / (ms * 1e-3) / 1e9
        # oracle: one (sequence, kv head) pair, scaled by the pair count
        cc = [cache.k_cache.cpu().numpy(), cache.v_cache.cpu().numpy(), cache.k_scale.cpu().numpy(),
              cache.v_scale.cpu().numpy(), cache.block_table.cpu().numpy(), cache.lens.cpu().numpy()]
        qq = q.float().cpu().numpy()
        t0 = time.perf_counter()
        qi, qs, _ = oracle.quant_int8(qq[:, :, None, :])
        oracle.decode_paged(qi[:, :, 0], qs[:, :, 0], *cc, threads=threads, pairs=[(0, 0)])
        t_or = (time.perf_counter() - t0) * B * Hkv
        emit({"config": name, "B": B, "ctx": ctx, "segments": S, "gpu_ms": round(ms, 4),
              "GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
              "oracle_s": round(t_or, 3), "oracle_cores": threads,
              "oracle_sample": "1 of %d (sequence, kv head) pairs, scaled" % (B * Hkv)})
        del cache

    _configs_kv_append(emit, gpu_ms, peaks)


def _configs_kv_append(emit, gpu_ms, peaks):
    """The KV producer (sage_kv_cache_append): a decode step's new token for
    every sequence of the paged-decode workload, and a 2048-token chunk of
    the chunked-prefill workload, quantised and scattered into the cache."""
    import torch

    from int8_quantized_attention_gb300 import binding as sage
    from int8_quantized_attention_gb300 import workloads as W

    P = W.WORKLOADS["paged_decode"].params
    for label, B, n, ctx in (("decode step", P["B"], 1, P["ctx"]), ("prefill chunk", 1, 2048, 16384)):
        Hkv, D = P["Hkv"], P["D"]
        c = W.paged_cache(B, Hkv, D, [ctx + n] * B, seed=9, device="cuda")
        g = torch.Generator("cuda").manual_seed(10)
        k = torch.randn((B, Hkv, n, D), generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn((B, Hkv, n, D), generator=g, device="cuda").to(torch.bfloat16)
        pos = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
        fn = lambda: sage.sage_kv_cache_append(k, v, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                               c.block_table, pos)
        ms = gpu_ms(fn)
        rows = 2 * B * Hkv * n
        nbytes = rows * (2 * D + D + 4) + B * (c.block_table.shape[1] + 1) * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        emit({"config": "kv_append", "case": label, "B": B, "new_tokens": n, "Hkv": Hkv, "D": D,
              "gpu_ms": round(ms, 4), "GBps": round(gbs, 1),
              "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
              "bytes": nbytes})
        # the producer form: the same append plus the step's query quantised
        # (Hq rows per token) in one launch
        Hq = P["Hq"]
        q = torch.randn((B, Hq, n, D), generator=g, device="cuda").to(torch.bfloat16)
        fp = lambda: sage.sage_kv_producer(q, k, v, c.k_cache, c.v_cache, c.k_scale, c.v_scale,
                                           c.block_table, pos)
        ms = gpu_ms(fp)
        pbytes = nbytes + B * Hq * n * (2 * D + D + 4)
        gbs = pbytes / (ms * 1e-3) / 1e9
        emit({"config": "kv_producer", "case": label, "B": B, "new_tokens": n, "Hq": Hq,
              "Hkv": Hkv, "D": D, "gpu_ms": round(ms, 4), "GBps": round(gbs, 1),
              "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4), "bytes": pbytes})
        del c


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    import numpy as np  # noqa: F401

    from int8_quantized_attention_gb300 import workloads as W
    import oracle

    P = W.WORKLOADS[WORKLOAD].params
    B, Hq, Hkv, D, ctx = P["B"], P["Hq"], P["Hkv"], P["D"], P["ctx"]
    cache = W.paged_cache(B, Hkv, D, [ctx] * B, seed=P["seed"], device="cpu")
    q = W.decode_query(B, Hq, D, seed=P["seed"], device="cpu").float().numpy()
    threads = oracle.default_threads()
    _, sbytes = decode_bytes(B, Hq, Hkv, D, ctx, cache.block_table.shape[1])
    # each step: the whole workload (all 32 (sequence, kv head) pairs), ~0.3 s on 8+ cores
    pairs = [(b, g) for b in range(B) for g in range(Hkv)]
    frac = len(pairs) / (B * Hkv)
    cargs = [cache.k_cache.numpy(), cache.v_cache.numpy(), cache.k_scale.numpy(),
             cache.v_scale.numpy(), cache.block_table.numpy(), cache.lens.numpy()]

    def one():
        qi, qs, _ = oracle.quant_int8(q[:, :, None, :])
        oracle.decode_paged(qi[:, :, 0], qs[:, :, 0], *cargs, threads=threads, pairs=pairs)

    for _ in range(args.warmup):
        one()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        times.append(time.perf_counter() - t0)
    t = sum(times)
    value = sbytes * frac * args.steps / t / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8", "data": "synthetic",
            "config": {"workload": "paged_decode B8 Hq24 Hkv4 D256 ctx8192 block16",
                       "step": "quant(Q) + paged decode, CPU oracle"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": "per step: the full paged_decode workload (32 sequence/"
                                       "kv-head pairs)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--profile", default=None,
                    choices=["paged_decode", "dense_prefill", "chunked_prefill",
                             "varlen_prefill", "kv_producer"])
    ap.add_argument("--pv-mode", default="fp32", choices=["fp32", "fp16", "fp16+fp32", "int8"],
                    help="decode P.V variant for --profile paged_decode")
    ap.add_argument("--heads", type=int, default=0)
    ap.add_argument("--segments", type=int, default=0,
                    help="decode segment count (0: the library's choice)")
    ap.add_argument("--configs", action="store_true",
                    help="time every configuration of the workload table (one JSON line each)")
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.configs:
        run_configs(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
