#!/usr/bin/env python3
"""Benchmark of the paged decode-attention step on GB300.

One step = the whole hot path over one batch: fused per-head RMSNorm + neox
RoPE on q/k with the k/v append (pkvqk_norm_rope_append), split-KV paged
decode attention (pkvqk_paged_decode / _partials) and, when the split count
is above 1, the LSE combine (pkvqk_lse_combine) — all through the C ABI.

Default workload: Qwen3-0.6B decode, 16 q / 8 kv heads, head_dim 128, bf16,
block_size 16, batch 64 x context 8192, shuffled block ids (2.15 GB of K/V
per step, larger than L2, so no flush is needed between steps).  Workloads
under 4x L2 start every step from a cold, clean L2: 2x L2 written, then 2x L2
read (the written lines go back to HBM before the step, not inside it).

Timing: pass 1 times K steps issued back to back with no event between the
calls of a step (the `value`); pass 2 times the same K steps with events
around each call (the per-call durations of `roofline`); the `e2e` pass adds
every step's host-to-device input copy and device-to-host output copy,
pipelined on their own streams.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle as reference arm

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica (replicas only: the step has no exchange between GPUs).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attn achieved HBM GB/s (% of GB300 peak) and seq-steps/s vs batch×ctx"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    # name: (builder, kwargs, description)
    "decode_64x8192": ("decode_uniform", {"batch": 64, "ctx": 8192},
                       "Qwen3-0.6B decode 16q/8kv D128 bf16 bs16, batch 64 x ctx 8192"),
    "decode_32x8192": ("decode_uniform", {"batch": 32, "ctx": 8192},
                       "Qwen3-0.6B decode 16q/8kv D128 bf16 bs16, batch 32 x ctx 8192"),
    "decode_long_8x32768": ("decode_long", {},
                            "Qwen3-1.7B long-context decode 16q/8kv D128 bs16, batch 8 x ctx 32768"),
    "decode_gqa8_64": ("decode_gqa8", {},
                       "Qwen3-30B-A3B-like decode 32q/4kv D128 bs16, batch 64, ctx log-U[256,16384]"),
    "verify_32x5": ("verify_causal", {},
                    "speculative verify 16q/8kv D128 bs16, batch 32, 5 query tokens, prior U[2048,8192]"),
}
WORKLOADS["decode_gqa8_64x4096"] = ("make_problem_uniform_gqa8", {},
                                    "GQA-8 decode 32q/4kv D128 bs16, batch 64 x ctx 4096 (uniform)")
WORKLOADS["decode_gqa4_32x8192"] = ("make_problem_uniform_gqa4", {},
                                    "Qwen3-8B decode 32q/8kv D128 bs16, batch 32 x ctx 8192 (uniform)")
# the tensor-core multi-query kernel (pkvqk_paged_prefill): chunked prefill,
# and the verify shape through the same kernel
PREFILL_WORKLOADS = {
    "prefill_8x512": ("chunked_prefill", {},
                      "chunked prefill 16q/8kv D128 bs16, batch 8 x 512-token chunk, "
                      "prior context U[0, 6144]"),
    "prefill_4x2048": ("chunked_prefill", {"batch": 4, "chunk": 2048, "lo": 0, "hi": 8192},
                       "chunked prefill 16q/8kv D128 bs16, batch 4 x 2048-token chunk, "
                       "prior context U[0, 8192]"),
    "prefill_gqa8_8x512": ("chunked_prefill", {"Hq": 32, "Hkv": 4},
                           "chunked prefill 32q/4kv D128 bs16, batch 8 x 512-token chunk, "
                           "prior context U[0, 6144]"),
    "prefill_varlen_16": ("varlen_prefill", {},
                          "varlen prefill 16q/8kv D128 bs16, 16 fresh prompts of U[128, 2048] "
                          "tokens, packed"),
    "verify_32x5_tc": ("verify_causal", {},
                       "speculative verify 16q/8kv D128 bs16, batch 32, 5 query tokens, prior "
                       "U[2048,8192], on the tensor-core multi-query kernel"),
}
WORKLOADS.update(PREFILL_WORKLOADS)
PREFILL_METRIC = "causal multi-query paged attention achieved TFLOP/s (% of measured bf16 peak)"
for _b in (1, 8, 32, 64):
    for _c in (512, 2048, 8192):
        WORKLOADS.setdefault(f"decode_{_b}x{_c}", ("decode_uniform", {"batch": _b, "ctx": _c},
                             f"Qwen3-0.6B decode 16q/8kv D128 bf16 bs16, batch {_b} x ctx {_c}"))


# dram__bytes_read.sum + dram__bytes_write.sum of one decode-kernel launch,
# mean of two launches from the 1-pass ncu capture recorded in
# profiles/paged_decode_kernel_decode_64x8192.md.  A capture describes the
# kernel sources it was taken with: when the sources hash differently, the
# bench reports traffic as null.
MEASURED_TRAFFIC = {
    "decode_64x8192": {"src": "86eac2e7161a8320", "bytes": 2149813120, "num_splits": 2},
}


def kernel_src_hash():
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_cache_qk_gb300", "csrc")
    parts = []
    for f in ("decode.cu", "device_common.cuh", "kernels.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            parts.append(hashlib.sha256(fh.read()).hexdigest())
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def load_peaks(key="hbm_gbs", fallback=FALLBACK_HBM_GBS):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return fallback, "fallback"


def attention_flops(p):
    """Algorithmic FLOPs of the causal attention: per visible (query token,
    key) pair and q head, 2*D for q.k and 2*D for p*v."""
    q_lens = p.q_lens_host if p.q_lens_host is not None else [p.q_len] * p.B
    n = 0
    for L, T in zip(p.seq_lens_host, q_lens):
        L, T = int(L), int(T)
        # token t sees L - T + t + 1 keys (clipped at 0)
        n += sum(max(0, L - T + t + 1) for t in range(T))
    return 4 * p.D * p.Hq * n


def step_bytes(p):
    """Algorithmic HBM bytes of one step (what the step must move at least).

    decode: every visible K and V row once (seq_len * Hkv * D * 2 B * 2),
            q (B*q_len*Hq*D*2), the bf16 output (same), 4 B per block-table
            entry read; split partials are overhead and not counted.
    append: q read + written, k and v read, k and v rows written to the cache.
    """
    D, Hq, Hkv = p.D, p.Hq, p.Hkv
    kv = int(p.seq_lens_host.sum()) * Hkv * D * 2 * 2
    qo = 2 * p.T * Hq * D * 2
    pages = int(sum(-(-int(n) // p.block_size) for n in p.seq_lens_host))
    decode = kv + qo + 4 * pages
    append = 2 * p.T * Hq * D * 2 + 2 * p.T * Hkv * D * 2 + 2 * p.T * Hkv * D * 2
    return decode, append


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, path):
        self.path = path
        self.proc = None
        self.gpu = gpu_index
        try:
            self.fh = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline_sample(seconds=10.0, max_seqs=64, ctx=8192, seed=2024):
    """Time the fp64 oracle on sequences of the benchmark workload's shape.

    Runs in this process with whatever threads numpy uses; called from a
    child process pinned to one BLAS thread so the core count is known.
    """
    import numpy as np

    import oracle
    from paged_kv_cache_qk_gb300 import workloads

    import torch

    chunk = 8
    p = workloads.decode_uniform(chunk, ctx, device="cpu", seed=seed)
    q = p.q.view(torch.int16).numpy().view(np.uint16).reshape(chunk, 1, p.Hq, p.D)
    kb = p.k_cache.view(torch.int16).numpy().view(np.uint16)
    vb = p.v_cache.view(torch.int16).numpy().view(np.uint16)
    done_seqs, done_bytes, elapsed = 0, 0, 0.0
    while done_seqs < max_seqs and elapsed < seconds:
        t0 = time.perf_counter()
        oracle.paged_attention(q, kb, vb, p.block_tables_host, p.seq_lens_host, p.block_size)
        elapsed += time.perf_counter() - t0
        done_seqs += chunk
        done_bytes += step_bytes(p)[0]
    return {"seqs": done_seqs, "ctx": ctx, "bytes": done_bytes, "seconds": elapsed}


def run_cpu_baseline_child(seconds, max_seqs, ctx):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
           "--cpu-seconds", str(seconds), "--cpu-max-seqs", str(max_seqs), "--cpu-ctx", str(ctx)]
    r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.decode(errors="replace")[-300:]}
    return json.loads(r.stdout.decode().strip().splitlines()[-1])


def max_over_ranks(values, device):
    """Element-wise max of per-rank values (every rank calls it; the result
    is the same on all).  Single process: the values unchanged."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_rate(world, units_per_rank_step, ms_per_step):
    """Whole-job rate of `world` replicas that each process
    units_per_rank_step per step, timed by the slowest rank (units / s)."""
    return world * units_per_rank_step / (ms_per_step * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(args):
    """Reference arm: the fp64 CPU oracle timed on the host cores.

    Decode workloads: the oracle over one sequence of the workload's context
    per step (GB/s).  Multi-query (prefill) workloads: the oracle over the
    last tokens of one sequence's chunk, each with its whole causal context,
    per step (TFLOP/s, the same algorithmic flop count as the GPU arm)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    name = args.workload
    builder, kw, desc = WORKLOADS[name]
    import numpy as np
    import torch

    import oracle
    from paged_kv_cache_qk_gb300 import workloads

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    if name in PREFILL_WORKLOADS:
        # one sequence of the workload, the last `tail` tokens of its chunk
        p = getattr(workloads, builder)(device="cpu", **kw)
        b = int(np.argmax(p.seq_lens_host))
        q_lens = p.q_lens_host if p.q_lens_host is not None else np.full(p.B, p.q_len)
        cu = np.concatenate([[0], np.cumsum(q_lens)])
        tail = int(min(8, q_lens[b]))
        L = int(p.seq_lens_host[b])
        rows = u16(p.q)[cu[b] + q_lens[b] - tail: cu[b] + q_lens[b]].reshape(1, tail, p.Hq, p.D)
        kb, vb = u16(p.k_cache), u16(p.v_cache)
        table = p.block_tables_host[b:b + 1]
        lens = np.array([L])

        def once():
            oracle.paged_attention(rows, kb, vb, table, lens, p.block_size, q_len=tail)
        flops = 4 * p.D * p.Hq * sum(L - tail + t + 1 for t in range(tail))
        sample = (f"sequence {b}: its last {tail} new tokens with {L - tail + 1}..{L} visible "
                  f"keys each ({p.Hq}q/{p.Hkv}kv, D128) per step; numpy default threads")
        metric, unit, scale = PREFILL_METRIC, "TFLOP/s", 1e12
        work = flops
    else:
        ctx = kw.get("ctx", 8192)
        seqs_per_step = 1
        p = workloads.decode_uniform(seqs_per_step, ctx, device="cpu", seed=4242)
        rows = u16(p.q).reshape(seqs_per_step, 1, p.Hq, p.D)
        kb, vb = u16(p.k_cache), u16(p.v_cache)

        def once():
            oracle.paged_attention(rows, kb, vb, p.block_tables_host, p.seq_lens_host,
                                   p.block_size)
        sample = f"{seqs_per_step} sequence x ctx {ctx} (16q/8kv, D128) per step; numpy default threads"
        metric, unit, scale = METRIC, "GB/s", 1e9
        work = step_bytes(p)[0]
    for _ in range(args.warmup):
        once()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        once()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    rate = work / dt / scale
    line = {
        "impl": "reference", "metric": metric, "value": rate, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "sample": sample},
        "cpu_baseline": {"value": rate, "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkvqk", choices=["pkvqk", "reference"])
    ap.add_argument("--workload", default="decode_64x8192", choices=sorted(WORKLOADS))
    ap.add_argument("--num-splits", type=int, default=-1,
                    help="0: balanced persistent schedule; -1: split heuristic; >0: fixed splits")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-max-seqs", type=int, default=4096)
    ap.add_argument("--cpu-ctx", type=int, default=8192)
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()

    if args.cpu_baseline_child:
        print(json.dumps(cpu_baseline_sample(args.cpu_seconds, args.cpu_max_seqs, args.cpu_ctx)))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import numpy as np
    import torch

    from paged_kv_cache_qk_gb300 import binding as lib
    from paged_kv_cache_qk_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    builder, kw, desc = WORKLOADS[args.workload]
    if builder == "make_problem_uniform_gqa8":
        import numpy as _np
        p = workloads.make_problem("gqa8_uniform", 32, 4, 128, 16, _np.full(64, 4096), 1,
                                   64 * 256, workloads.BASE_SEED + 3, device=dev)
    elif builder == "make_problem_uniform_gqa4":
        import numpy as _np
        p = workloads.make_problem("gqa4_uniform", 32, 8, 128, 16, _np.full(32, 8192), 1,
                                   32 * 512, workloads.BASE_SEED + 7, device=dev)
    else:
        p = getattr(workloads, builder)(device=dev, **kw)
    decode_bytes, append_bytes = step_bytes(p)
    rows_per_kv = p.q_len * p.Hq // p.Hkv
    prefill = args.workload in PREFILL_WORKLOADS
    if prefill:
        S = args.num_splits if args.num_splits >= 1 else lib.choose_prefill_splits(
            p.B, p.Hkv, p.q_len, p.Hq // p.Hkv, p.max_seq_len)
        ws_bytes = lib.prefill_workspace_bytes(1, p.T, p.Hq, p.D, S)
    else:
        S = args.num_splits if args.num_splits >= 0 else lib.choose_num_splits(
            p.B, p.Hkv, rows_per_kv, p.max_seq_len, p.total_tokens, p.block_size)
        ws_bytes = lib.decode_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev) if ws_bytes else None
    varlen = p.cu_seqlens is not None
    out = (torch.empty(p.T, p.Hq, p.D, dtype=torch.bfloat16, device=dev) if varlen else
           torch.empty(p.B, p.q_len, p.Hq, p.D, dtype=torch.bfloat16, device=dev))
    q = p.q.clone()
    stream = torch.cuda.current_stream()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    big_inputs = decode_bytes > 4 * l2_bytes
    flush = None if big_inputs else torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    flush_clean = None if big_inputs else torch.empty(2 * l2_bytes, dtype=torch.uint8,
                                                      device=dev)

    def cold_l2():
        # write 2x L2 (evicts every input line), then read another 2x L2 so
        # the written lines go back to HBM here and not inside the next step
        flush.zero_()
        flush_clean.max()

    def decode_call(qq, bt, sl, cu=None, o=None):
        o = out if o is None else o
        if varlen:
            lib.paged_prefill_varlen(qq, p.cu_seqlens if cu is None else cu, p.q_len,
                                     p.k_cache, p.v_cache, bt, sl, o, num_splits=S,
                                     max_seq_len_hint=p.max_seq_len, workspace=ws, stream=stream)
        elif prefill:
            lib.paged_prefill(qq, p.k_cache, p.v_cache, bt, sl, o, q_len=p.q_len,
                              num_splits=S, max_seq_len_hint=p.max_seq_len, workspace=ws,
                              stream=stream)
        else:
            lib.paged_decode(qq, p.k_cache, p.v_cache, bt, sl, o, q_len=p.q_len,
                             num_splits=S, max_seq_len_hint=p.max_seq_len, workspace=ws,
                             stream=stream)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        lib.norm_rope_append(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q, p.gamma_k,
                             p.theta, p.eps, p.k_cache, p.v_cache, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        decode_call(q, p.block_tables, p.seq_lens)
        if ev is not None:
            ev[2].record(stream)

    if prefill:   # append, prefill (+ lse combine when split)
        launches_per_step = 2 + (1 if S > 1 else 0)
    else:         # append, decode (+ the combine of the split or balanced partials)
        launches_per_step = 2 + (1 if S != 1 else 0)

    # the clock sampler starts (and settles) before the warm-up, so that the
    # warm-up, not an idle pause, is what directly precedes the timed steps
    clocks = ClockSampler(local, os.path.join(tempfile.gettempdir(),
                                              f"pkvqk_bench_clocks_r{rank}.csv"))
    time.sleep(0.3)

    for _ in range(args.warmup):
        if not big_inputs:
            cold_l2()
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    K = args.steps
    # Pass 1, the step value: K steps as a caller issues them, with no event
    # between the calls of a step (an event recorded between two kernels ends
    # the programmatic-dependent overlap of the second one's launch and
    # prologue with the first one's tail).
    if big_inputs:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)
    else:
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K)]
        for i in range(K):
            cold_l2()
            step_ev[i][0].record(stream)
            step()
            step_ev[i][1].record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    if world > 1:
        torch.distributed.barrier()
    # Pass 2, the per-call durations for the roofline: the same K steps with an
    # event before and after each call on the launching stream.
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    for i in range(K):
        if not big_inputs:
            cold_l2()
        step(evs[i])
    torch.cuda.synchronize()
    append_ms = [e[0].elapsed_time(e[1]) for e in evs]
    decode_ms = [e[1].elapsed_time(e[2]) for e in evs]

    # end to end: host (pinned) inputs in, host output back, every step
    # the step's inputs packed into one pinned host buffer (16-byte aligned
    # fields), one host->device copy, typed device views into the copy
    names = ("q", "k", "v", "positions", "slot_mapping", "block_tables", "seq_lens")
    if varlen:
        names = names + ("cu_seqlens",)
    fields, off = {}, 0
    for n in names:
        t = getattr(p, n)
        nbytes = t.numel() * t.element_size()
        fields[n] = (off, nbytes, t.dtype, tuple(t.shape))
        off += (nbytes + 15) // 16 * 16
    host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(off, dtype=torch.uint8, device=dev)
    dev_in = {}
    for n, (o, nb, dt, shp) in fields.items():
        src = getattr(p, n).contiguous().view(torch.uint8).reshape(-1).cpu()
        host_buf[o:o + nb].copy_(src)
        dev_in[n] = dev_buf[o:o + nb].view(dt).view(shp)
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = off
    d2h = host_out.numel() * host_out.element_size()
    K_e2e = max(3, min(K, 500))

    # Pipelined as a serving loop runs it: step i's inputs go up on an upload
    # stream and its output comes back on a readback stream while the compute
    # stream works on the neighbouring steps; two input and two output buffers
    # alternate, and events order every reuse.  Each step still moves its own
    # inputs and output inside the timed region.
    dev_bufs = [dev_buf, torch.empty_like(dev_buf)]
    dev_ins = [dev_in, {n: dev_bufs[1][o:o + nb].view(dt).view(shp)
                        for n, (o, nb, dt, shp) in fields.items()}]
    outs = [out, torch.empty_like(out)]
    host_outs = [host_out, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]
    for ev in computed + read_back:
        ev.record(stream)

    def e2e_step(i):
        k = i & 1
        with torch.cuda.stream(up):
            up.wait_event(computed[k])           # step i - 2 is done reading buffer k
            dev_bufs[k].copy_(host_buf, non_blocking=True)
            uploaded[k].record(up)
        stream.wait_event(uploaded[k])
        stream.wait_event(read_back[k])          # step i - 2's output has left outs[k]
        d = dev_ins[k]
        lib.norm_rope_append(d["q"], d["k"], d["v"], d["positions"], d["slot_mapping"],
                             p.gamma_q, p.gamma_k, p.theta, p.eps, p.k_cache, p.v_cache,
                             stream=stream)
        decode_call(d["q"], d["block_tables"], d["seq_lens"], d.get("cu_seqlens"), outs[k])
        computed[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[k])
            host_outs[k].copy_(outs[k], non_blocking=True)
            read_back[k].record(down)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K_e2e):
        e2e_step(i)
    for ev in read_back:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K_e2e
    clk = clocks.stop()

    ms = total_ms / K
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dev)
    bytes_step = decode_bytes + append_bytes
    value = aggregate_rate(world, bytes_step, ms) / 1e9
    e2e_value = aggregate_rate(world, bytes_step, e2e_ms) / 1e9

    peak, peak_kind = load_peaks()
    rec = MEASURED_TRAFFIC.get(args.workload)
    traffic = (rec["bytes"] if rec and rec["src"] == kernel_src_hash() and rec["num_splits"] == S
               else None)
    dec_avg_ms = statistics.fmean(decode_ms)
    achieved = decode_bytes / (dec_avg_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": desc,
            "batch": p.B, "ctx_max": p.max_seq_len, "total_tokens": p.total_tokens,
            "q_len": p.q_len, "heads_q": p.Hq, "heads_kv": p.Hkv, "head_dim": p.D,
            "block_size": p.block_size,
            "schedule": "balanced (one CTA per SM)" if S == 0 else f"split x{S}",
            "l2": ("inputs larger than L2: %.2f GB of K/V per step vs %d MB L2" %
                   (decode_bytes / 1e9, l2_bytes >> 20)) if big_inputs else
                  "L2 flushed before every step (2x L2 written, then 2x L2 read so the "
                  "written lines are back in HBM before the step), excluded from timing",
            "parallelism": f"replicas x{world}",
        },
        "seq_steps_per_s": round(aggregate_rate(world, p.B, ms), 1),
        "pct_of_nominal_8tbs": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "copies": "pipelined: upload and readback streams, double-buffered"},
        "gpu_launches": K * launches_per_step,
        "roofline": {
            "kernel": "pkvqk_paged_decode call: paged_decode_kernel"
                      + (" + balanced_combine_kernel" if S == 0 else
                         " + lse_combine_kernel" if S > 1 else ""),
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": decode_bytes,
            "avg_launch_ms": round(dec_avg_ms, 5),
            "timing": "second pass of the K steps, CUDA events around each call",
        },
        "clocks": clk,
        "append_avg_ms": round(statistics.fmean(append_ms), 5),
        "e2e_gpu_launches": K_e2e * launches_per_step,
    }
    if prefill:
        flops = attention_flops(p)
        tpeak, tpeak_kind = load_peaks("bf16_tflops", 1900.0)
        tflops = flops / (dec_avg_ms * 1e-3) / 1e12
        line["metric"] = PREFILL_METRIC
        line["value"] = round(aggregate_rate(world, flops, ms) / 1e12, 2)
        line["unit"] = "TFLOP/s"
        line["e2e"]["value"] = round(aggregate_rate(world, flops, e2e_ms) / 1e12, 2)
        line["e2e"]["unit"] = "TFLOP/s"
        line["config"]["schedule"] = f"256-row CTA tiles (2 x 128, ping-pong) x split {S}"
        line["config"]["flops_per_step"] = flops
        line["config"]["kv_bytes_per_step"] = decode_bytes
        del line["pct_of_nominal_8tbs"]
        line["tokens_per_s"] = round(aggregate_rate(world, p.T, ms), 1)
        line["roofline"] = {
            "kernel": "pkvqk_paged_prefill call: paged_prefill_kernel"
                      + (" + lse_combine_kernel" if S > 1 else ""),
            "bound": "tensor",
            "achieved": round(tflops, 2),
            "peak": tpeak,
            "peak_kind": tpeak_kind + " (bf16 burst)",
            "unit": "TFLOP/s",
            "frac": round(tflops / tpeak, 4),
            "traffic": None,
            "algorithmic_flops_per_launch": flops,
            "avg_launch_ms": round(dec_avg_ms, 5),
            "timing": "second pass of the K steps, CUDA events around each call",
            "hbm_gbs_of_kv": round(achieved, 2),
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not prefill:
        cb = run_cpu_baseline_child(args.cpu_seconds, args.cpu_max_seqs, args.cpu_ctx)
        if "error" in cb:
            line["cpu_baseline"] = {"error": cb["error"]}
        else:
            line["cpu_baseline"] = {
                "value": round(cb["bytes"] / cb["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": f"{cb['seqs']} sequence-passes (8 seqs re-run) x ctx {cb['ctx']} of the "
                          f"16q/8kv D128 decode workload, fp64 numpy oracle, 1 BLAS thread, "
                          f"{cb['seconds']:.1f} s",
            }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
