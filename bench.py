#!/usr/bin/env python3
"""Benchmark of the paged decode-attention step on GB300.

One step = the whole hot path over one batch: fused per-head RMSNorm + neox
RoPE on q/k with the k/v append (pkvqk_norm_rope_append_cached: the rotary
sin/cos of each position come from a table that pkvqk_rope_table_build fills
once per model, for Qwen3's 40960-position context, outside every timed
region; the results are bit-identical to pkvqk_norm_rope_append's), split-KV
paged decode attention (pkvqk_paged_decode) and, when the split count is
above 1 or the schedule is the balanced one, the LSE combine kernel it
launches — all through the C ABI.

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

The same line carries `sweep`: every decode configuration of the batch x
context study measured the same way (the 12 batch x context points of the
Qwen3-0.6B decode, the 8 x 32768 long context at the heuristic split count
and at 1, 8, 32 and 128 splits, the GQA-8 serving batch of mixed lengths,
the 32 x 5-token speculative verify, and two uniform GQA shapes), each with
its own clocks; and `cpu_baseline`: the fp64 oracle timed on the host cores,
on one core and on all cores (a process pool over sequences, or over
(sequence, kv head) units for a batch smaller than the pool),
for the largest batch x context point, the long context, the GQA-8 batch and
the verify step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle as reference arm

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica (replicas only: the step has no exchange between GPUs); the sweep and
the CPU baseline run at N = 1 only.
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
ROPE_TABLE_POSITIONS = 40960          # Qwen3-0.6B's longest context
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
    "prefill_19x512_ctx16k": ("chunked_prefill",
                              {"batch": 19, "chunk": 512, "lo": 16384, "hi": 16384},
                              "chunked prefill 16q/8kv D128 bs16, batch 19 x 512-token chunk "
                              "after 16384 prior tokens (a long prompt's late chunks; 608 CTAs "
                              "= 4 waves on 152 SMs)"),
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

# The decode configurations of the batch x context study, each with the split
# count it is timed at (-1: the library's heuristic, 0: balanced schedule).
SWEEP = ([(f"decode_{b}x{c}", -1, "batch x context") for b in (1, 8, 32, 64)
          for c in (512, 2048, 8192)]
         + [("decode_long_8x32768", s, "long context") for s in (-1, 1, 8, 32, 128)]
         + [("decode_gqa8_64", -1, "GQA-8 serving batch"),
            ("verify_32x5", -1, "speculative verify"),
            ("decode_gqa8_64x4096", -1, "GQA-8 uniform"),
            ("decode_gqa4_32x8192", -1, "GQA-4 uniform")])

# The prefill configurations timed after the decode study in the default run.
PREFILL_SWEEP = ("prefill_4x2048", "prefill_8x512", "prefill_gqa8_8x512", "prefill_varlen_16",
                 "prefill_19x512_ctx16k")

# The oracle's CPU timing covers these decode configurations.
CPU_BASELINE_WORKLOADS = ("decode_64x8192", "decode_long_8x32768", "decode_gqa8_64",
                          "verify_32x5")

# dram__bytes_read.sum + dram__bytes_write.sum of one decode-kernel launch
# (1-pass ncu captures of the full-size workloads, mean of two launches after
# three warm-up steps), keyed by workload and split count (0: balanced).  A
# capture describes the kernel sources it was taken with: when the sources
# hash differently, the bench reports traffic as null.
SRC = "53582c2775d61dfe"
MEASURED_TRAFFIC = {
    ("decode_1x2048", 32): {"src": SRC, "bytes": 8468352},
    ("decode_1x512", 8): {"src": SRC, "bytes": 2176128},
    ("decode_1x8192", 64): {"src": SRC, "bytes": 33635584},
    ("decode_32x2048", 4): {"src": SRC, "bytes": 270230912},
    ("decode_32x512", 4): {"src": SRC, "bytes": 67453696},
    ("decode_32x8192", 4): {"src": SRC, "bytes": 1075746432},
    ("decode_64x2048", 2): {"src": SRC, "bytes": 538666496},
    ("decode_64x512", 2): {"src": SRC, "bytes": 135940096},
    ("decode_64x8192", 2): {"src": SRC, "bytes": 2149515264},
    ("decode_8x2048", 16): {"src": SRC, "bytes": 67362816},
    ("decode_8x512", 8): {"src": SRC, "bytes": 16885632},
    ("decode_8x8192", 16): {"src": SRC, "bytes": 270131456},
    ("decode_gqa4_32x8192", 4): {"src": SRC, "bytes": 1075707776},
    ("decode_gqa8_64", 0): {"src": SRC, "bytes": 468448000},
    ("decode_gqa8_64x4096", 2): {"src": SRC, "bytes": 539089920},
    ("decode_long_8x32768", 1): {"src": SRC, "bytes": 1075767936},
    ("decode_long_8x32768", 8): {"src": SRC, "bytes": 1075376000},
    ("decode_long_8x32768", 16): {"src": SRC, "bytes": 1075483776},
    ("decode_long_8x32768", 32): {"src": SRC, "bytes": 1075882368},
    ("decode_long_8x32768", 128): {"src": SRC, "bytes": 1076084992},
    ("verify_32x5", 6): {"src": SRC, "bytes": 710233856},
}


def kernel_src_hash():
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_cache_qk_gb300", "csrc")
    parts = []
    for f in ("decode.cu", "device_common.cuh", "kernels.h", "api.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            parts.append(hashlib.sha256(fh.read()).hexdigest())
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def measured_traffic(workload, S):
    rec = MEASURED_TRAFFIC.get((workload, S))
    return rec["bytes"] if rec and rec["src"] == kernel_src_hash() else None


def load_peaks(key="hbm_gbs", fallback=FALLBACK_HBM_GBS):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return fallback, "fallback"


def build_problem(name, device):
    """The seeded synthetic inputs of a named workload."""
    import numpy as np

    from paged_kv_cache_qk_gb300 import workloads
    builder, kw, _ = WORKLOADS[name]
    if builder == "make_problem_uniform_gqa8":
        return workloads.make_problem("gqa8_uniform", 32, 4, 128, 16, np.full(64, 4096), 1,
                                      64 * 256, workloads.BASE_SEED + 3, device=device)
    if builder == "make_problem_uniform_gqa4":
        return workloads.make_problem("gqa4_uniform", 32, 8, 128, 16, np.full(32, 8192), 1,
                                      32 * 512, workloads.BASE_SEED + 7, device=device)
    return getattr(workloads, builder)(device=device, **kw)


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
    """nvidia-smi clock / throttle sampling while the timed regions run; the
    samples carry timestamps, so any wall-clock window can be summarised."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, path):
        self.path = path
        self.proc = None
        self.samples = []
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
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        import datetime
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm, mx = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                active = {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"}
                self.samples.append((t, sm, mx, active))

    def window(self, t0, t1):
        """Median SM clock, max clock and active throttle reasons between two
        time.time() stamps (the nearest sample if none falls inside)."""
        if not self.samples:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        reasons = set()
        for s in inside:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(reasons), "samples": len(inside)}


# --------------------------------------------------------------------------
# The fp64 oracle on the host cores (cpu_baseline and the reference arm).
# A decode workload splits into independent units: a sequence (the oracle
# called as it stands on the one-sequence sub-problem), or, when the batch
# has fewer sequences than workers, a (sequence, kv head) pair (the
# sequence's q heads of that kv head over that kv head's cache).  All cores:
# a spawn pool over the units, the inputs shared through POSIX shared memory.
# --------------------------------------------------------------------------

_ORACLE_STATE = {}


def _oracle_attach(spec):
    """Pool initializer: map the shared input arrays."""
    import numpy as np
    from multiprocessing import shared_memory
    shms = []
    for key, (shm_name, shape, dtype) in spec["arrays"].items():
        shm = shared_memory.SharedMemory(name=shm_name)
        shms.append(shm)
        _ORACLE_STATE[key] = np.ndarray(shape, dtype=dtype, buffer=shm.buf)
    _ORACLE_STATE["_shms"] = shms
    _ORACLE_STATE["meta"] = spec["meta"]


def _oracle_unit(unit, state=None):
    """One unit of the fp64 oracle: sequence b over all its kv heads (g < 0),
    or over kv head g alone."""
    import oracle
    st = _ORACLE_STATE if state is None else state
    m = st["meta"]
    b, g = unit
    G, T = m["G"], m["q_len"]
    if g < 0:
        q, kc, vc = st["q"][b:b + 1], st["kc"], st["vc"]
    else:
        q = st["q"][b:b + 1, :, g * G:(g + 1) * G, :]
        kc, vc = st["kc"][:, :, g:g + 1, :], st["vc"][:, :, g:g + 1, :]
    out, _ = oracle.paged_attention(q, kc, vc, st["bt"][b:b + 1], st["sl"][b:b + 1], m["bs"],
                                    q_len=T)
    return float(out[0, 0, 0, 0])


class OracleWorkload:
    """A decode workload's inputs as host arrays, cut into independent units
    (whole sequences when the batch has at least one sequence per worker,
    else (sequence, kv head) pairs), timed through the oracle on one core or
    on a pool."""

    def __init__(self, name, workers):
        import numpy as np
        import torch
        self.name = name
        p = build_problem(name, "cpu")
        self.p = p

        def u16(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        self.arrays = {
            "q": u16(p.q).reshape(p.B, p.q_len, p.Hq, p.D),
            "kc": u16(p.k_cache), "vc": u16(p.v_cache),
            "bt": np.ascontiguousarray(p.block_tables_host),
            "sl": np.ascontiguousarray(p.seq_lens_host.astype(np.int64)),
        }
        self.meta = {"G": p.Hq // p.Hkv, "q_len": p.q_len, "bs": p.block_size}
        # longest first, so a pool finishes together
        order = np.argsort(-p.seq_lens_host, kind="stable")
        self.per_sequence = p.B >= workers
        heads = [-1] if self.per_sequence else list(range(p.Hkv))
        self.units = [(int(b), g) for b in order for g in heads]
        self.unit_kind = "sequence" if self.per_sequence else "(sequence, kv head)"
        decode_bytes = step_bytes(p)[0]
        kv_total = int(p.seq_lens_host.sum()) * len(heads)
        # a unit's share of the step's algorithmic bytes: its keys' share
        self.unit_bytes = {(b, g): decode_bytes * int(p.seq_lens_host[b]) / kv_total
                           for b, g in self.units}
        self.step_bytes = decode_bytes
        self.shms = []

    def time_one_core(self, seconds):
        """Units in order on this process (one BLAS thread expected) until
        `seconds` have passed or the workload is done; returns a record."""
        state = dict(self.arrays, meta=self.meta)
        t0 = time.perf_counter()
        done, nbytes = 0, 0.0
        for u in self.units:
            _oracle_unit(u, state)
            done += 1
            nbytes += self.unit_bytes[u]
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        return {"gbs": nbytes / dt / 1e9, "cores": 1, "seconds": dt, "units": done,
                "units_total": len(self.units), "unit": self.unit_kind}

    def _share(self):
        from multiprocessing import shared_memory
        import numpy as np
        spec = {"arrays": {}, "meta": self.meta}
        for key, a in self.arrays.items():
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            self.shms.append(shm)
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            spec["arrays"][key] = (shm.name, a.shape, a.dtype.str)
        return spec

    def open_pool(self, workers):
        import multiprocessing as mp
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        spec = self._share()
        self.pool = mp.get_context("spawn").Pool(workers, initializer=_oracle_attach,
                                                 initargs=(spec,))
        self.workers = workers
        # start every worker and map the arrays before anything is timed
        self.pool.map(_oracle_unit, self.units[-workers:], chunksize=1)

    def pass_all_cores(self):
        """One whole pass of the workload over the pool; returns seconds."""
        t0 = time.perf_counter()
        self.pool.map(_oracle_unit, self.units, chunksize=1)
        return time.perf_counter() - t0

    def time_all_cores(self, seconds, max_passes=20):
        total, passes = 0.0, 0
        while passes < max_passes and (passes == 0 or total < seconds):
            total += self.pass_all_cores()
            passes += 1
        return {"gbs": passes * self.step_bytes / total / 1e9, "cores": self.workers,
                "seconds": total, "passes": passes, "units_total": len(self.units),
                "unit": self.unit_kind}

    def close(self):
        pool = getattr(self, "pool", None)
        if pool is not None:
            pool.close()
            pool.join()
            self.pool = None
        for shm in self.shms:
            shm.close()
            shm.unlink()
        self.shms = []


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_child(seconds):
    """Time the oracle on each CPU-baseline workload, one core then all."""
    res = {"nproc": os.cpu_count(), "cores_available": host_cores(), "workloads": {}}
    for name in CPU_BASELINE_WORKLOADS:
        w = OracleWorkload(name, res["cores_available"])
        try:
            one = w.time_one_core(seconds)
            w.open_pool(res["cores_available"])
            allc = w.time_all_cores(seconds)
        finally:
            w.close()
        res["workloads"][name] = {"one_core": one, "all_cores": allc,
                                  "description": WORKLOADS[name][2]}
        del w
    return res


def run_cpu_baseline_child(seconds):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
           "--cpu-seconds", str(seconds)]
    r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr.decode(errors="replace")[-300:]}
    return json.loads(r.stdout.decode().strip().splitlines()[-1])


def cpu_baseline_record(cb, headline):
    """The JSON line's cpu_baseline object from the child's measurements."""
    if "error" in cb:
        return {"error": cb["error"]}
    ws = cb["workloads"]
    head = headline if headline in ws else CPU_BASELINE_WORKLOADS[0]
    h = ws[head]
    per = {}
    for name, r in ws.items():
        per[name] = {
            "one_core_gbs": round(r["one_core"]["gbs"], 4),
            "all_cores_gbs": round(r["all_cores"]["gbs"], 4),
            "cores": r["all_cores"]["cores"],
            "sample": (f"one core: {r['one_core']['units']} of {r['one_core']['units_total']} "
                       f"{r['one_core']['unit']} units in {r['one_core']['seconds']:.1f} s; all cores: "
                       f"{r['all_cores']['passes']} whole pass(es) in "
                       f"{r['all_cores']['seconds']:.1f} s"),
        }
    return {
        "value": round(h["all_cores"]["gbs"], 4), "unit": "GB/s",
        "cores": h["all_cores"]["cores"], "kind": "oracle",
        "sample": (f"{WORKLOADS[head][2]}: the fp64 numpy oracle over {h['all_cores']['unit']} "
                   f"units, a spawn process pool of {h['all_cores']['cores']} workers with one "
                   f"BLAS thread each, {h['all_cores']['passes']} whole pass(es) of the workload "
                   f"in {h['all_cores']['seconds']:.1f} s"),
        "one_core": {"value": round(h["one_core"]["gbs"], 4), "unit": "GB/s", "cores": 1,
                     "sample": per[head]["sample"].split(";")[0]},
        "nproc": cb["nproc"],
        "workloads": per,
    }


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

    Decode workloads: each step is one whole pass of the workload through the
    oracle, its (sequence, kv head) units spread over a spawn pool of one
    worker per host core (GB/s).  Multi-query (prefill) workloads: the oracle
    over the last tokens of one sequence's chunk, each with its whole causal
    context, per step (TFLOP/s, the same algorithmic flop count as the GPU
    arm)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    name = args.workload
    builder, kw, desc = WORKLOADS[name]
    import numpy as np
    import torch

    import oracle

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    if name in PREFILL_WORKLOADS:
        # one sequence of the workload, the last `tail` tokens of its chunk
        p = build_problem(name, "cpu")
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
        work, cores = flops, os.cpu_count()
        closer = None
    else:
        cores = host_cores()
        w = OracleWorkload(name, cores)
        w.open_pool(cores)

        def once():
            w.pass_all_cores()
        sample = (f"one whole pass of the workload per step: {len(w.units)} {w.unit_kind} "
                  f"units over a spawn process pool of {cores} workers, one BLAS thread each")
        metric, unit, scale = METRIC, "GB/s", 1e9
        work = w.step_bytes
        closer = w.close
    try:
        for _ in range(args.warmup):
            once()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            once()
        dt = (time.perf_counter() - t0) / max(1, args.steps)
    finally:
        if closer is not None:
            closer()
    rate = work / dt / scale
    line = {
        "impl": "reference", "metric": metric, "value": rate, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "sample": sample},
        "cpu_baseline": {"value": rate, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# The GPU arm
# --------------------------------------------------------------------------

class StepRunner:
    """One workload on the GPU through the C ABI: its buffers, its split
    count, one step (append + attention call), and the timed passes."""

    def __init__(self, lib, name, p, S_arg, dev, stream, flush):
        import torch
        self.lib, self.name, self.p, self.dev, self.stream = lib, name, p, dev, stream
        self.prefill = name in PREFILL_WORKLOADS
        self.varlen = p.cu_seqlens is not None
        rows_per_kv = p.q_len * p.Hq // p.Hkv
        if self.prefill:
            S = S_arg if S_arg >= 1 else lib.choose_prefill_splits(
                p.B, p.Hkv, p.q_len, p.Hq // p.Hkv, p.max_seq_len)
            ws_bytes = lib.prefill_workspace_bytes(1, p.T, p.Hq, p.D, S)
            self.launches_per_step = 2 + (1 if S > 1 else 0)
        else:
            S = S_arg if S_arg >= 0 else lib.choose_num_splits(
                p.B, p.Hkv, rows_per_kv, p.max_seq_len, p.total_tokens, p.block_size)
            ws_bytes = lib.decode_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
            self.launches_per_step = 2 + (1 if S != 1 else 0)
        self.S = S
        self.ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev) if ws_bytes else None
        self.out = (torch.empty(p.T, p.Hq, p.D, dtype=torch.bfloat16, device=dev) if self.varlen else
                    torch.empty(p.B, p.q_len, p.Hq, p.D, dtype=torch.bfloat16, device=dev))
        self.q = p.q.clone()
        self.decode_bytes, self.append_bytes = step_bytes(p)
        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
        self.l2_bytes = l2_bytes
        self.big_inputs = self.decode_bytes > 4 * l2_bytes
        self.flush = flush
        # the rotary table: model state built once (the longest context of
        # Qwen3-0.6B, or further if a workload's positions go further)
        self.table_positions = max(ROPE_TABLE_POSITIONS, int(p.positions.max().item()) + 1)
        self.rope_table = torch.empty(lib.rope_table_bytes(self.table_positions),
                                      dtype=torch.uint8, device=dev)
        lib.rope_table_build(self.rope_table, self.table_positions, p.theta, stream=stream)
        torch.cuda.synchronize()

    def cold_l2(self):
        # write 2x L2 (evicts every input line), then read another 2x L2 so
        # the written lines go back to HBM here and not inside the next step
        self.flush[0].zero_()
        self.flush[1].max()

    def decode_call(self, qq, bt, sl, cu=None, o=None):
        p, lib, S, stream = self.p, self.lib, self.S, self.stream
        o = self.out if o is None else o
        if self.varlen:
            lib.paged_prefill_varlen(qq, p.cu_seqlens if cu is None else cu, p.q_len,
                                     p.k_cache, p.v_cache, bt, sl, o, num_splits=S,
                                     max_seq_len_hint=p.max_seq_len, workspace=self.ws,
                                     stream=stream)
        elif self.prefill:
            lib.paged_prefill(qq, p.k_cache, p.v_cache, bt, sl, o, q_len=p.q_len,
                              num_splits=S, max_seq_len_hint=p.max_seq_len, workspace=self.ws,
                              stream=stream)
        else:
            lib.paged_decode(qq, p.k_cache, p.v_cache, bt, sl, o, q_len=p.q_len,
                             num_splits=S, max_seq_len_hint=p.max_seq_len, workspace=self.ws,
                             stream=stream)

    def step(self, ev=None):
        p, stream = self.p, self.stream
        if ev is not None:
            ev[0].record(stream)
        self.lib.norm_rope_append_cached(self.q, p.k, p.v, p.positions, p.slot_mapping,
                                         p.gamma_q, p.gamma_k, p.theta, p.eps, p.k_cache,
                                         p.v_cache, self.rope_table, self.table_positions,
                                         stream=stream)
        if ev is not None:
            ev[1].record(stream)
        self.decode_call(self.q, p.block_tables, p.seq_lens)
        if ev is not None:
            ev[2].record(stream)

    def warm(self, W):
        import torch
        for _ in range(W):
            if not self.big_inputs:
                self.cold_l2()
            self.step()
        torch.cuda.synchronize()

    def time_value(self, K):
        """Pass 1, the step value: K steps as a caller issues them, with no
        event between the calls of a step (an event recorded between two
        kernels ends the programmatic-dependent overlap of the second one's
        launch and prologue with the first one's tail).  Returns total ms."""
        import torch
        stream = self.stream
        if self.big_inputs:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(K):
                self.step()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K)]
        for i in range(K):
            self.cold_l2()
            step_ev[i][0].record(stream)
            self.step()
            step_ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in step_ev)

    def time_calls(self, K):
        """Pass 2, the per-call durations: the same K steps with an event
        before and after each call on the launching stream."""
        import torch
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
        for i in range(K):
            if not self.big_inputs:
                self.cold_l2()
            self.step(evs[i])
        torch.cuda.synchronize()
        return ([e[0].elapsed_time(e[1]) for e in evs], [e[1].elapsed_time(e[2]) for e in evs])

    def time_e2e(self, K):
        """End to end: host (pinned) inputs in, host output back, every step,
        pipelined as a serving loop runs it (step i's inputs go up on an
        upload stream and its output comes back on a readback stream while
        the compute stream works on the neighbouring steps; two input and two
        output buffers alternate, events order every reuse).  Returns
        (ms per step, h2d bytes per step, d2h bytes per step)."""
        import torch
        p, dev, stream, lib = self.p, self.dev, self.stream, self.lib
        # the step's inputs packed into one pinned host buffer (16-byte
        # aligned fields), one host->device copy, typed device views into it
        names = ("q", "k", "v", "positions", "slot_mapping", "block_tables", "seq_lens")
        if self.varlen:
            names = names + ("cu_seqlens",)
        fields, off = {}, 0
        for n in names:
            t = getattr(p, n)
            nbytes = t.numel() * t.element_size()
            fields[n] = (off, nbytes, t.dtype, tuple(t.shape))
            off += (nbytes + 15) // 16 * 16
        host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
        for n, (o, nb, dt, shp) in fields.items():
            src = getattr(p, n).contiguous().view(torch.uint8).reshape(-1).cpu()
            host_buf[o:o + nb].copy_(src)
        dev_bufs = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        dev_ins = [{n: dev_bufs[k][o:o + nb].view(dt).view(shp)
                    for n, (o, nb, dt, shp) in fields.items()} for k in range(2)]
        outs = [self.out, torch.empty_like(self.out)]
        host_outs = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
                     for _ in range(2)]
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
            lib.norm_rope_append_cached(d["q"], d["k"], d["v"], d["positions"],
                                        d["slot_mapping"], p.gamma_q, p.gamma_k, p.theta, p.eps,
                                        p.k_cache, p.v_cache, self.rope_table,
                                        self.table_positions, stream=stream)
            self.decode_call(d["q"], d["block_tables"], d["seq_lens"], d.get("cu_seqlens"),
                             outs[k])
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
        for i in range(K):
            e2e_step(i)
        for ev in read_back:
            stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K, off, host_outs[0].numel() * host_outs[0].element_size()

    def schedule(self):
        if self.prefill:
            return f"256-row CTA tiles (2 x 128, ping-pong) x split {self.S}"
        return "balanced (persistent, 0.84 CTAs per SM)" if self.S == 0 else f"split x{self.S}"


def sweep_point(runner, steps, warmup, peak, group):
    """One configuration of the sweep: the step and the decode call timed as
    the headline is; returns its record."""
    p = runner.p
    t0 = time.time()
    runner.warm(warmup)
    total_ms = runner.time_value(steps)
    _, dec = runner.time_calls(steps)
    t1 = time.time()
    ms = total_ms / steps
    dec_ms = statistics.fmean(dec)
    step_gbs = (runner.decode_bytes + runner.append_bytes) / (ms * 1e-3) / 1e9
    dec_gbs = runner.decode_bytes / (dec_ms * 1e-3) / 1e9
    return {
        "workload": runner.name, "group": group, "batch": p.B, "ctx_max": p.max_seq_len,
        "total_tokens": p.total_tokens, "q_len": p.q_len, "heads_q": p.Hq, "heads_kv": p.Hkv,
        "num_splits": runner.S, "schedule": runner.schedule(), "steps": steps,
        "ms_per_step": round(ms, 5), "step_gbs": round(step_gbs, 1),
        "pct_of_nominal_8tbs": round(100.0 * step_gbs / NOMINAL_HBM_GBS, 2),
        "decode_ms": round(dec_ms, 5), "decode_gbs": round(dec_gbs, 1),
        "frac": round(dec_gbs / peak, 4),
        "seq_steps_per_s": round(p.B / (ms * 1e-3), 1),
        "algorithmic_bytes_per_launch": runner.decode_bytes,
        "traffic": measured_traffic(runner.name, runner.S),
        "l2": "inputs > 4x L2" if runner.big_inputs else "cold clean L2 before every step",
        "window": (t0, t1),        # replaced by the clocks seen in it once sampling stops
    }


def prefill_point(runner, steps, warmup, tpeak):
    """One prefill configuration of the default run: the step (append +
    prefill call) and the prefill call timed as a prefill headline is."""
    p = runner.p
    t0 = time.time()
    runner.warm(warmup)
    total_ms = runner.time_value(steps)
    app, dec = runner.time_calls(steps)
    t1 = time.time()
    ms = total_ms / steps
    dec_ms = statistics.fmean(dec)
    flops = attention_flops(p)
    tflops = flops / (dec_ms * 1e-3) / 1e12
    return {
        "workload": runner.name, "batch": p.B, "new_tokens": p.T, "ctx_max": p.max_seq_len,
        "heads_q": p.Hq, "heads_kv": p.Hkv, "num_splits": runner.S, "steps": steps,
        "ms_per_step": round(ms, 5), "step_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
        "append_ms": round(statistics.fmean(app), 5),
        "prefill_ms": round(dec_ms, 5), "tflops": round(tflops, 2),
        "frac": round(tflops / tpeak, 4), "algorithmic_flops_per_launch": flops,
        "l2": "inputs > 4x L2" if runner.big_inputs else "cold clean L2 before every step",
        "window": (t0, t1),
    }


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
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=200)
    ap.add_argument("--sweep-only", default="",
                    help="comma-separated workload names: restrict the sweep to them")
    ap.add_argument("--cpu-seconds", type=float, default=3.0,
                    help="oracle seconds per workload and core setting in cpu_baseline")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()

    if args.cpu_baseline_child:
        print(json.dumps(cpu_baseline_child(args.cpu_seconds)))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch

    from paged_kv_cache_qk_gb300 import binding as lib

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    stream = torch.cuda.current_stream()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev),
             torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev))

    desc = WORKLOADS[args.workload][2]
    p = build_problem(args.workload, dev)
    run = StepRunner(lib, args.workload, p, args.num_splits, dev, stream, flush)
    S = run.S

    # the clock sampler starts (and settles) before the warm-up, so that the
    # warm-up, not an idle pause, is what directly precedes the timed steps
    clocks = ClockSampler(local, os.path.join(tempfile.gettempdir(),
                                              f"pkvqk_bench_clocks_r{rank}.csv"))
    time.sleep(0.3)
    t_head0 = time.time()
    run.warm(args.warmup)
    if world > 1:
        torch.distributed.barrier()
    K = args.steps
    total_ms = run.time_value(K)
    if world > 1:
        torch.distributed.barrier()
    append_ms, decode_ms = run.time_calls(K)
    K_e2e = max(3, min(K, 500))
    e2e_ms, h2d, d2h = run.time_e2e(K_e2e)
    t_head1 = time.time()

    ms = total_ms / K
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dev)
    decode_bytes, append_bytes = run.decode_bytes, run.append_bytes
    bytes_step = decode_bytes + append_bytes
    value = aggregate_rate(world, bytes_step, ms) / 1e9
    e2e_value = aggregate_rate(world, bytes_step, e2e_ms) / 1e9

    peak, peak_kind = load_peaks()
    dec_avg_ms = statistics.fmean(decode_ms)
    achieved = decode_bytes / (dec_avg_ms * 1e-3) / 1e9
    prefill = run.prefill

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
            "schedule": run.schedule(),
            "l2": ("inputs larger than L2: %.2f GB of K/V per step vs %d MB L2" %
                   (decode_bytes / 1e9, l2_bytes >> 20)) if run.big_inputs else
                  "L2 flushed before every step (2x L2 written, then 2x L2 read so the "
                  "written lines are back in HBM before the step), excluded from timing",
            "parallelism": f"replicas x{world}",
            "rope_table_positions": run.table_positions,
        },
        "seq_steps_per_s": round(aggregate_rate(world, p.B, ms), 1),
        "pct_of_nominal_8tbs": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "copies": "pipelined: upload and readback streams, double-buffered"},
        "gpu_launches": K * run.launches_per_step,
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
            "traffic": measured_traffic(args.workload, S),
            "algorithmic_bytes_per_launch": decode_bytes,
            "avg_launch_ms": round(dec_avg_ms, 5),
            "timing": "second pass of the K steps, CUDA events around each call",
        },
        "clocks": None,
        "append_avg_ms": round(statistics.fmean(append_ms), 5),
        "e2e_gpu_launches": K_e2e * run.launches_per_step,
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
    del run, p

    # the batch x context study, N = 1 only (a rank's sweep would hold the
    # other GPUs idle meanwhile)
    sweep = None
    if world == 1 and not args.no_sweep and not prefill:
        only = {s for s in args.sweep_only.split(",") if s}
        sweep = []
        cache = {}
        for name, S_arg, group in SWEEP:
            if only and name not in only:
                continue
            if name not in cache:
                cache.clear()
                torch.cuda.empty_cache()
                cache[name] = build_problem(name, dev)
            r = StepRunner(lib, name, cache[name], S_arg, dev, stream, flush)
            sweep.append(sweep_point(r, args.sweep_steps, 5, peak, group))
            del r
        cache.clear()
        torch.cuda.empty_cache()
    # the prefill configurations (tensor-core kernel), N = 1 only, same timing
    psweep = None
    if world == 1 and not args.no_sweep and not prefill:
        only = {s for s in args.sweep_only.split(",") if s}
        tpeak, _ = load_peaks("bf16_tflops", 1900.0)
        psweep = []
        for name in PREFILL_SWEEP:
            if only and name not in only:
                continue
            torch.cuda.empty_cache()
            r = StepRunner(lib, name, build_problem(name, dev), -1, dev, stream, flush)
            psweep.append(prefill_point(r, args.sweep_steps, 5, tpeak))
            del r
        torch.cuda.empty_cache()
    clocks.stop()
    line["clocks"] = clocks.window(t_head0, t_head1)
    if sweep is not None:
        for rec in sweep:
            clk = clocks.window(*rec.pop("window"))
            rec["sm_mhz"] = clk["sm_mhz"] if clk else None
            rec["clock_reasons"] = clk["reasons"] if clk else None
        line["sweep"] = sweep
        line["sweep_note"] = ("every decode configuration timed as the headline: step = append "
                              "+ decode call, value pass without events inside a step, decode_ms "
                              "from a second pass with events around each call; frac = decode "
                              "GB/s / measured HBM copy GB/s; traffic = 1-pass ncu DRAM bytes "
                              "of one decode launch where captured on the current sources")
    if psweep is not None:
        for rec in psweep:
            clk = clocks.window(*rec.pop("window"))
            rec["sm_mhz"] = clk["sm_mhz"] if clk else None
            rec["clock_reasons"] = clk["reasons"] if clk else None
        line["prefill_sweep"] = psweep
        line["prefill_sweep_note"] = ("chunked and varlen prefill on the tcgen05 kernel: step = "
                                      "append + prefill call; prefill_ms from a second pass "
                                      "with events around each call; frac = TFLOP/s / measured "
                                      "bf16 cuBLAS burst peak")

    if rank == 0 and world == 1 and not args.no_cpu_baseline and not prefill:
        cb = run_cpu_baseline_child(args.cpu_seconds)
        line["cpu_baseline"] = cpu_baseline_record(cb, args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
