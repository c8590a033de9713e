#!/usr/bin/env python
"""Benchmark of the GB300 grouped-query attention block forward; prints ONE JSON line.

Headline workload: long-context prefill of B=1 sequence of T=32768 tokens (dim 4096, 32 q /
8 kv heads, d_h 128, bf16 inputs, random N(0, 0.02) weights, theta=500000 RoPE table,
causal mask, fp32 output).  A step is one full block forward (Q/K/V projection + RoPE +
cache write, causal GQA attention, W_O projection) through the C ABI, inputs resident in
HBM.  L2 is flushed (256 MiB write) before every timed step, outside the step's events.

The same line carries, under "sub_records", one fully measured record (its own step time,
roofline of the dominant kernel, e2e and clocks, timed in the same process) for each other
workload of the block: prefill B=1 x T=16, B=1 x T=2048, B=4 x T=8192, the decode step of
B=64 sequences at position 4095, and a chunked prefill (the last 2048 tokens of a
32768-token prompt against a cache of the first 30720).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-sub]
                  [--impl reference]

N > 1 runs under torchrun: one rank per GPU, each rank runs its own replica of the
workload (weak scaling; the path has no cross-sequence exchange), max time over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from transformer_gqa_attention_gb300 import inputs as gin  # noqa: E402

METRIC = "GQA block tokens/s & TFLOP/s (prefill), HBM GB/s (decode), % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
NORM_EPS = 1e-5  # attention_norm epsilon of the residual workloads (norm_eps of the 8B configs)


# ------------------------------------------------------------------ accounting
def prefill_flops(B, T, start_pos=0, causal=True, n_kv=8):
    """Algorithmic FLOPs: 2 x 41,943,040 per token for the projections plus 4*128 per
    visible (query, key) pair per query head (QK^T and PV).  A shard of n_kv of the 8 kv
    groups holds n_kv/8 of the weights and of the query heads."""
    proj = 2 * (41_943_040 // 8) * n_kv * B * T
    if causal:
        pairs = T * start_pos + T * (T + 1) // 2
    else:
        pairs = T * (start_pos + T)
    return proj, 4 * 128 * 4 * n_kv * pairs * B


def decode_bytes(B, kv_len, n_kv=8):
    """Minimum HBM bytes of one decode step: the K/V cache read (kv_len keys x n_kv heads x
    128 x bf16, K and V), the weights (W_QKV + W_O, n_kv/8 of them for a shard), x in, Delta
    out (fp32), the new K/V entries written."""
    kv = B * kv_len * n_kv * 128 * 2 * 2
    w = (41_943_040 // 8) * n_kv * 2
    return kv + w + B * 4096 * 2 + B * 4096 * 4 + B * n_kv * 128 * 2 * 2


def kernel_work(kind, w: gin.Workload):
    """(bound, algorithmic work per launch, unit) of one kernel kind on the workload."""
    n_tok = w.n_tok
    g = w.n_kv  # kv groups of the context: Q/K/V rows 768 g, W_O columns 512 g
    if kind == "qkv_gemm":
        return "tensor", 2.0 * n_tok * 4096 * 768 * g, "TFLOP/s"
    if kind == "out_gemm":
        return "tensor", 2.0 * n_tok * 512 * g * 4096, "TFLOP/s"
    if kind == "flash_prefill":
        return "tensor", float(prefill_flops(w.B, w.T, w.start_pos, w.causal, g)[1]), "TFLOP/s"
    if kind == "decode_attn":
        # decode, or a prefill of T <= 16 positions (same kernel): K and V of the whole cache
        # once, q in and H out
        kv_len = w.start_pos + w.T
        return "hbm", float(w.B * kv_len * g * 128 * 2 * 2 + 2 * n_tok * 512 * g * 2), "GB/s"
    if kind == "qkv_splitk":
        return "hbm", float(768 * g * 4096 * 2 + n_tok * 4096 * 2), "GB/s"
    if kind == "out_splitk":
        return "hbm", float(4096 * 512 * g * 2 + n_tok * 512 * g * 2), "GB/s"
    if kind == "rms_norm":
        return "hbm", float(n_tok * 4096 * 2 + n_tok * 4), "GB/s"
    return None, None, None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and blank lines (string literals are kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # string literal, copied as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def source_digest():
    """Digest of the CUDA/C++ code of the library (the kernels the ncu figures describe);
    comments and blank lines do not count."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_gqa_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kind, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources for this workload; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kind)
    if not e or e.get("source_digest") != source_digest():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                    "-lms", "200", *sel]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons, power = [], [], set(), []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if n_gpus > 1 and world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} needs torchrun with {n_gpus} ranks (WORLD_SIZE={world})")
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle timing
def oracle_sample_step(inp, w: gin.Workload, n_tokens: int, seqs: int, w64):
    """Run the fp64 oracle on a bounded sample: for a prefill, the first n_tokens positions
    of `seqs` sequences (a causal prefix is the exact computation of those rows); for a
    decode, `seqs` sequences.  Returns (seconds, units processed, bytes for decode)."""
    from oracle import gqa_oracle as orc
    wq, wk, wv, wo = w64
    t0 = time.perf_counter()
    wn = gin.to_f64(gin.norm_weight(w.seed)) if w.residual else None
    if w.kind == "prefill":
        x = gin.to_f64(inp.x[:seqs, :n_tokens])
        R = gin.to_f64(inp.R[:n_tokens])
        kw = {}
        if w.start_pos:  # a chunk continuing a cache: its first n_tokens rows against it
            n_keys = w.start_pos + n_tokens
            kw = dict(start_pos=w.start_pos, cache_k=gin.to_f64(inp.cache_k[:seqs, :n_keys]),
                      cache_v=gin.to_f64(inp.cache_v[:seqs, :n_keys]))
        if w.residual:
            orc.attention_block_residual(x, wn, wq, wk, wv, wo, R, causal=w.causal, **kw)
        else:
            orc.attention_block(x, wq, wk, wv, wo, R, causal=w.causal, **kw)
        units = seqs * n_tokens
    else:
        pos = w.start_pos
        x = gin.to_f64(inp.x[:seqs])
        ck = gin.to_f64(inp.cache_k[:seqs, :pos + 1])
        cv = gin.to_f64(inp.cache_v[:seqs, :pos + 1])
        if w.residual:
            orc.attention_decode_residual(x, wn, wq, wk, wv, wo, gin.to_f64(inp.R), ck, cv, pos)
        else:
            orc.attention_decode(x, wq, wk, wv, wo, gin.to_f64(inp.R), ck, cv, pos)
        units = seqs
    return time.perf_counter() - t0, units


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _oracle_rate(inp, w: gin.Workload, n, seqs, w64, budget_s, max_runs=10):
    """Repeat the oracle on one bounded sample until budget_s has passed (at most max_runs);
    return (total seconds, runs, units per run)."""
    times, units = [], 0
    t_start = time.perf_counter()
    while True:
        dt, u = oracle_sample_step(inp, w, n, seqs, w64)
        times.append(dt)
        units = u
        if time.perf_counter() - t_start > budget_s or len(times) >= max_runs:
            break
    return sum(times), len(times), units


def cpu_baseline(inp, w: gin.Workload, budget_s=15.0):
    """Time the oracle as it stands on the host cores on a bounded sample (~budget_s).

    Prefill: a causal prefix of sequence 0 (the exact computation of those rows).  When the
    workload is longer than the prefix, the oracle's time is also extrapolated to the full
    length from two prefix lengths with t(n) = a n + b n^2 (projections grow with n, the
    attention products with n^2), and labelled as an extrapolation."""
    w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    if w.kind == "prefill":
        n = min(w.T, 2048)
        total, runs, u = _oracle_rate(inp, w, n, 1, w64, budget_s)
        out = {"value": runs * u / total, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"oracle prefill of positions 0..{n - 1} of sequence 0, {runs} run(s), {total:.1f} s"}
        if w.T > n:
            n1 = n // 2
            t1, r1, _ = _oracle_rate(inp, w, n1, 1, w64, budget_s / 3, max_runs=3)
            ta, tb = t1 / r1, total / runs
            # t(n) = a n + b n^2 through (n1, ta) and (n, tb); if the fit gives a negative
            # coefficient (timing noise, cache effects), the pure quadratic through the longer
            # prefix, which is the smaller of the two for any non-decreasing cost per pair
            b = (tb / n - ta / n1) / (n - n1)
            a = ta / n1 - b * n1
            if a > 0 and b > 0:
                t_full = w.B * (a * w.T + b * w.T * w.T)
                how = f"t(n) = a n + b n^2 fitted to the oracle's times at n = {n1} and {n}"
            else:
                t_full = w.B * tb * (w.T / n) ** 2
                how = f"t(n) = t({n}) (n / {n})^2 (a two-point fit at n = {n1}, {n} gave a negative term)"
            out["extrapolated_full_workload"] = {
                "value": w.n_tok / t_full, "unit": "tokens/s", "seconds": t_full,
                "how": how + f", evaluated at T = {w.T} for {w.B} sequence(s); an extrapolation, not a run"}
        return out
    seqs = min(w.B, 4)
    total, runs, _ = _oracle_rate(inp, w, 1, seqs, w64, budget_s)
    per_seq = decode_bytes(1, w.start_pos + 1) - 41_943_040 * 2
    value = runs * (seqs * per_seq + 41_943_040 * 2) / total / 1e9
    return {"value": value, "unit": "GB/s", "cores": cores(), "kind": "oracle",
            "sample": f"oracle decode of {seqs} of the {w.B} sequences, {runs} run(s), {total:.1f} s"}


SINGLE_CORE_WORKLOADS = ("prefill_b1_t16", "decode_b64_pos4095")


def single_core_baseline(name: str, budget_s=4.0):
    """The oracle on ONE host core (BLAS threads 1, affinity one core) on the workload, in a
    child process so that the thread settings take effect before numpy loads."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", GQA_BENCH_ONE_CORE="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-one-core", name, "--one-core-budget", str(budget_s)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": (r.stderr.strip().splitlines() or ["failed"])[-1]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def _one_core_child(name: str, budget_s: float):
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    torch.set_num_threads(1)
    w = gin.WORKLOADS[name]
    inp = gin.make_inputs(w)
    rec = cpu_baseline(inp, w, budget_s=budget_s)
    rec["cores"] = cores()
    rec["workload"] = name
    print(json.dumps(rec))


def prefix_for_budget(n1, t1, n2, t2, budget_s, T, cap=4096):
    """Causal-prefix length whose oracle time fits budget_s, from the times t1, t2 measured at
    prefix lengths n1 < n2 under t(n) = a n + b n^2 (the projections grow with n, the
    attention products with n^2); between 16 and min(T, cap)."""
    b = max((t2 / n2 - t1 / n1) / max(1, n2 - n1), 1e-12)
    a = max(t1 / n1 - b * n1, 1e-9)
    n_fit = (-a + (a * a + 4 * b * budget_s) ** 0.5) / (2 * b)
    return int(max(16, min(T, cap, n_fit)))


def run_reference(args, w, inp):
    """The oracle as the reference arm: W untimed + K timed steps, each a bounded sample."""
    w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    total_budget = 120.0
    if w.kind == "prefill":
        # calibration at two prefix lengths; the oracle's time grows as a n + b n^2
        # (projections, then the attention products), so size the prefix from that fit
        n1, n2 = min(w.T, 512), min(w.T, 1024)
        t1, _ = oracle_sample_step(inp, w, n1, 1, w64)
        t2, _ = oracle_sample_step(inp, w, n2, 1, w64)
        n = prefix_for_budget(n1, t1, n2, t2, total_budget / max(1, args.steps + args.warmup), w.T)
        seqs = 1
        desc = f"oracle prefill of positions 0..{n - 1} of sequence 0 per step"
    else:
        n, seqs = 1, 1
        desc = "oracle decode of sequence 0 per step"
    for _ in range(args.warmup):
        oracle_sample_step(inp, w, n, seqs, w64)
    times, units = [], 0
    for _ in range(args.steps):
        dt, u = oracle_sample_step(inp, w, n, seqs, w64)
        times.append(dt)
        units += u
    total = sum(times)
    ms = 1e3 * total / len(times)
    if w.kind == "prefill":
        value, unit = units / total, "tokens/s"
    else:
        value = len(times) * (decode_bytes(1, w.start_pos + 1)) / total / 1e9
        unit = "GB/s"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"kind": "oracle", "cores": cores(), "sample": desc, "value": value,
                             "unit": unit},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def workload_config(w: gin.Workload):
    c = {"workload": w.name, "kind": w.kind, "B": w.B, "T": w.T, "start_pos": w.start_pos,
         "S_max": w.s_max, "causal": w.causal, "dim": 4096, "n_heads": 32, "n_kv_heads": 8,
         "head_dim": 128, "seed": w.seed, "l2": "flushed before every timed step (256 MiB write)"}
    if w.residual:
        c.update(residual=True, norm_eps=NORM_EPS,
                 form="h = x + Delta_attn(attention_norm(x)); attention_norm weight 1 + 0.1 N(0,1)")
    if w.n_kv != 8:
        c.update(n_kv_heads=w.n_kv, n_heads=4 * w.n_kv,
                 form=f"one rank of a {8 // w.n_kv}-way head-sharded split: kv groups 0..{w.n_kv - 1}, "
                      "partial Delta (the all-reduce over ranks is not part of the step)")
    return c


# ------------------------------------------------------------------ GPU arm
def measure_gpu(args, w: gin.Workload, inp, world, rank, local, steps, warmup):
    """Time one workload on this rank's GPU: the device-timed steps, a profiled pass of the
    same steps (per-kernel times) and the end-to-end pass through pinned host buffers.
    Returns the workload's record on rank 0 (None elsewhere)."""
    from transformer_gqa_attention_gb300 import abi
    dev = torch.device("cuda", local)
    B, T = w.B, w.T
    S_max = w.s_max
    G = w.n_kv
    if G == 8:
        wts = [t.to(dev) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    else:  # one tensor-parallel rank: kv groups 0 .. G-1 and their query heads
        from transformer_gqa_attention_gb300 import tp
        wts = [t.to(dev) for t in tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, 0, G)]
    stream = torch.cuda.current_stream(dev)
    norm_w = gin.norm_weight(w.seed).to(dev) if w.residual else None

    def new_ctx():
        c = abi.attn_create(*wts) if G == 8 else abi.attn_create_shard(*wts, G)
        if w.residual:
            abi.attn_set_norm(c, norm_w, NORM_EPS, stream)
        return c

    ctx = new_ctx()
    x = inp.x.to(dev)
    R = inp.R.to(dev)
    if w.kind == "prefill":
        if inp.cache_k is not None:  # a chunk continuing a drawn cache
            ck = inp.cache_k[:, :, :G].contiguous().to(dev)
            cv = inp.cache_v[:, :, :G].contiguous().to(dev)
        else:
            ck = torch.zeros(B, S_max, G, 128, dtype=torch.bfloat16, device=dev)
            cv = torch.zeros_like(ck)
        delta = torch.empty(B, T, 4096, dtype=torch.float32, device=dev)
        fn = abi.attn_prefill_residual if w.residual else abi.attn_prefill

        def step(xd=x, Rd=R, out=delta, c=ctx):
            fn(c, xd, B, T, Rd, w.causal, ck, cv, S_max, w.start_pos, out, stream)
    else:
        ck = inp.cache_k[:, :, :G].contiguous().to(dev)
        cv = inp.cache_v[:, :, :G].contiguous().to(dev)
        delta = torch.empty(B, 1, 4096, dtype=torch.float32, device=dev)
        fn = abi.attn_decode_residual if w.residual else abi.attn_decode

        def step(xd=x, Rd=R, out=delta, c=ctx):
            fn(c, xd, B, w.start_pos, Rd, ck, cv, S_max, out, stream)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        flush.zero_()
        step()
    abi.attn_sync_status(ctx, stream)

    # ---------------- device-timed region
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    abi.attn_sync_status(ctx, stream)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, world, dev)

    # ---------------- profiled pass: the same steps with the library's per-kernel events
    # (recorded between launches, so consecutive kernels no longer overlap here)
    torch.cuda.synchronize(dev)
    abi.attn_profile_begin(ctx)
    for i in range(steps):
        flush.zero_()
        step()
    prof = abi.attn_profile_end(ctx, stream)
    abi.attn_sync_status(ctx, stream)

    # ---------------- end to end through host buffers (pinned), double-buffered: the input
    # copy of step i+1 and the result copy of step i-1 run on their own streams (copy
    # engines) while step i computes; every step copies its inputs in and its Delta out.
    # Instead of an L2 flush (a device-timing artefact) consecutive steps alternate between
    # two contexts holding separate weight copies (2 x 84 MB > L2), so no step finds the
    # previous step's weights in L2.
    ctx_alt = new_ctx()
    ctxs = (ctx, ctx_alt)
    # the second context's first call sizes its workspace (a stream synchronisation and a
    # cudaMalloc): make it here, untimed, like the warm-up steps of the first context
    for _ in range(warmup):
        flush.zero_()
        step(c=ctx_alt)
    abi.attn_sync_status(ctx_alt, stream)
    del flush
    x_h = inp.x.pin_memory()
    R_h = inp.R.pin_memory()
    out_h = torch.empty(delta.shape, dtype=torch.float32).pin_memory()
    x_d = [torch.empty_like(x) for _ in range(2)]
    R_d = [torch.empty_like(R) for _ in range(2)]
    o_d = [torch.empty_like(delta) for _ in range(2)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(steps)]
    ev_comp = [torch.cuda.Event() for _ in range(steps)]
    ev_out = [torch.cuda.Event() for _ in range(steps)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    s_in.wait_event(e_start)
    s_out.wait_event(e_start)
    for i in range(steps):
        bsel = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])  # buffers of step i-2 no longer read
            x_d[bsel].copy_(x_h, non_blocking=True)
            R_d[bsel].copy_(R_h, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # result buffer of step i-2 copied out
        step(x_d[bsel], R_d[bsel], o_d[bsel], ctxs[bsel])
        ev_comp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            out_h.copy_(o_d[bsel], non_blocking=True)
            ev_out[i].record(s_out)
    stream.wait_event(ev_out[steps - 1])
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / steps, world, dev)
    h2d = x_h.numel() * x_h.element_size() + R_h.numel() * R_h.element_size()
    d2h = out_h.numel() * out_h.element_size()
    abi.attn_sync_status(ctx, stream)
    abi.attn_sync_status(ctx_alt, stream)
    abi.attn_destroy(ctx_alt)
    abi.attn_destroy(ctx)
    del x_d, R_d, o_d, x, R, ck, cv, delta, wts
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()

    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    n = world
    if w.kind == "prefill":
        proj, attn = prefill_flops(B, T, w.start_pos, w.causal, G)
        value = n * B * T / (ms / 1e3)
        unit = "tokens/s"
        e2e_value = n * B * T / (e2e_ms / 1e3)
        extra = {"tflops": n * (proj + attn) / (ms / 1e3) / 1e12,
                 "tflops_frac_of_" + peak_src: (proj + attn) / (ms / 1e3) / 1e12 / peaks["bf16_tflops"]}
    else:
        by = decode_bytes(B, w.start_pos + 1, G)
        value = n * by / (ms / 1e3) / 1e9
        unit = "GB/s"
        e2e_value = n * by / (e2e_ms / 1e3) / 1e9
        extra = {"tokens_per_s": n * B / (ms / 1e3),
                 "hbm_frac_of_" + peak_src: by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]}

    kinds = {k: v for k, v in prof.items() if v[1] > 0}
    # dominant kernel among those with an algorithmic-work model (the reductions have none)
    modeled = {k: v for k, v in kinds.items() if kernel_work(k, w)[0] is not None}
    dom = max(modeled, key=lambda k: modeled[k][0])
    bound, work, wunit = kernel_work(dom, w)
    avg_ms = kinds[dom][0] / kinds[dom][1]
    if bound == "tensor":
        achieved = work / (avg_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
    else:
        achieved = work / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
    roofline = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": wunit,
                "frac": achieved / peak, "peak_source": f"{peak_src} (burst)" if bound == "tensor" else peak_src,
                "traffic": ncu_traffic(dom, w.name), "work_per_launch": work,
                "avg_launch_ms": avg_ms,
                "timing": "CUDA events around each launch on the launch stream, profiled pass of the "
                          "same steps right after the timed one"}
    per_kernel = {k: {"ms_per_launch": v[0] / v[1], "launches": v[1], "share": v[0] / sum(x[0] for x in kinds.values())}
                  for k, v in kinds.items()}
    return {"metric": METRIC, "value": value, "unit": unit, "n_gpus": n, "steps": steps,
            "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) x, N(0,0.02) weights)",
            "config": workload_config(w), **extra, "roofline": roofline, "kernels": per_kernel,
            "gpu_launches": int(sum(v[1] for v in kinds.values())),
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "schedule": "pinned host buffers, input copy / compute / result copy on three streams, "
                                "double-buffered across steps; consecutive steps alternate two weight "
                                "copies (168 MB > L2) instead of an L2 flush"},
            "clocks": clocks}


HEADLINE = "prefill_b1_t32768"
SUB_WORKLOADS = ("prefill_b1_t16", "prefill_b1_t2048", "prefill_b4_t8192", "decode_b64_pos4095",
                 "prefill_b1_t2048_pos30720")
# Short steps are timed over at least this many steps so that one record spans a few ms.
MIN_SUB_STEPS = 100


def run_gpu(args, w: gin.Workload, world, rank, local):
    from transformer_gqa_attention_gb300 import _build
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    inp = gin.make_inputs(w)
    line = measure_gpu(args, w, inp, world, rank, local, args.steps, args.warmup)
    subs = {}
    if not args.no_sub and w.name == HEADLINE:
        for name in SUB_WORKLOADS:
            sw = gin.WORKLOADS[name]
            sinp = gin.make_inputs(sw)
            steps = max(args.steps, MIN_SUB_STEPS) if (sw.kind == "decode" or sw.T <= 2048) else args.steps
            subs[name] = measure_gpu(args, sw, sinp, world, rank, local, steps, args.warmup)
            del sinp
    if rank != 0:
        return
    if subs:
        line["sub_records"] = subs
    if world == 1 and not args.no_cpu_baseline and w.n_kv == 8:
        line["cpu_baseline"] = cpu_baseline(inp, w)
        line["cpu_baseline"]["single_core"] = {name: single_core_baseline(name) for name in SINGLE_CORE_WORKLOADS}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(gin.WORKLOADS))
    ap.add_argument("--impl", default="gqa", choices=["gqa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="time only --workload (no sub-records)")
    ap.add_argument("--oracle-one-core", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--one-core-budget", type=float, default=4.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_one_core:
        _one_core_child(args.oracle_one_core, args.one_core_budget)
        return
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    w = gin.WORKLOADS[args.workload]
    if args.impl == "reference":
        if w.n_kv != 8:
            raise SystemExit("the reference arm times the whole block: choose a whole-block workload")
        if rank == 0:
            run_reference(args, w, gin.make_inputs(w))
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_gpu(args, w, world, rank, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
