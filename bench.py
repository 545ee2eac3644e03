"""Benchmark: paged GQA attention on GB300, one JSON line on rank 0.

Default (headline) workload: the continuous-batching mix -- 256 sequences, half with contexts
U[32, 512] and half U[2048, 8192], 32 query heads over 8 KV heads, head_dim 128, bf16 KV in
16-token pages drawn from a shared pool with 10 % free blocks interleaved (about 3 GB of KV read
per step).  A step is one paged_attn_decode call over the whole batch (decode kernel plus
split-KV merge).  value = sequences * steps / s over all ranks; the achieved HBM bandwidth of the
same step (algorithmic KV + Q + O bytes / step time) is in `roofline`.  The same line carries,
under `configs`, every other workload timed the same way: the Llama-3-8B-shaped decode, the
speculative verify at K = 4 and K = 8, the long-context E4M3 decode and the tiny parity case.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

The K timed steps are captured once in a CUDA graph and replayed as one submission between an
event pair on the launching stream (consecutive calls run back to back, as under graphs in a
serving loop).  A workload whose KV is less than 3x the 129 MB L2 (the verify batches) rotates
its calls over enough copies of its inputs that each call reads its KV from HBM; its figure
from a single copy is reported beside it.  `e2e` times the headline's calls through the public
API one by one, with the inputs copied from pinned host memory every step.  Under torchrun every
rank runs an independent replica on its own GPU (the batch partitions across sequences with no
exchange), the K timed steps are bracketed by a barrier and a device synchronise on both sides,
and the slowest rank's time is reported.
--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload (rank 0 only).
"""

from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_gqa_attn_gb300 import accounting as A  # noqa: E402
from paged_kv_gqa_attn_gb300 import workloads as W  # noqa: E402

METRIC = "paged GQA attention: achieved HBM TB/s (% of GB300 peak); seq-steps/s"
UNIT = "seq-steps/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e datasheet bandwidth: context beside the measured peak
L2_BYTES = 129 * 1024 * 1024

DESCRIPTIONS = {
    "tiny": "tiny paged decode: B=4, ctx {1,17,33,64}, Hq 4 / Hkv 2, d 64, bs 16, bf16 KV",
    "llama8b_decode": "Llama-3-8B-shaped decode, one layer: B=64, ctx 2048, Hq 32 / Hkv 8, d 128, "
                      "bs 16, bf16 KV, pool 1.25x",
    "cb_mix": "continuous-batching mix: B=256, ctx half U[32,512] half U[2048,8192], Hq 32 / Hkv 8, "
              "d 128, bs 16, bf16 KV, 10% free blocks interleaved",
    "spec_verify_k4": "speculative verify K=4: B=16, q_len 5, prior ctx U[1024,4096], Hq 32 / Hkv 8, "
                      "d 128, bs 16, bf16 KV",
    "spec_verify_k8": "speculative verify K=8: B=16, q_len 9, prior ctx U[1024,4096], Hq 32 / Hkv 8, "
                      "d 128, bs 16, bf16 KV",
    "long_fp8": "long-context fp8 KV: B=4, ctx 131072, Hq 32 / Hkv 8, d 128, bs 16, E4M3 KV with "
                "per-(block, kv head) scales, <=64 split-KV partitions",
    "llama70b_decode": "Llama-3-70B-shaped decode, one layer: B=64, ctx 2048, Hq 64 / Hkv 8 (groups of 8), "
                       "d 128, bs 16, bf16 KV, pool 1.25x (tensor-core kernel)",
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Source files each profiled kernel is built and launched from: a traffic figure stays valid
# while none of them changes.
COMMON_SOURCES = ("pa_api.cu", "pa_kernels.h", "pa_device.cuh")
KERNEL_SOURCES = {
    "decode": ("pa_decode.cu", "pa_decode_mma.cu", "pa_merge.cu", "pa_tc.cuh") + COMMON_SOURCES,
    "verify": ("pa_verify.cu", "pa_tc.cuh") + COMMON_SOURCES,
    "prefill": ("pa_prefill.cu", "pa_tc.cuh") + COMMON_SOURCES,
    "append": ("pa_append.cu",) + COMMON_SOURCES,
    "accept": ("pa_accept.cu",) + COMMON_SOURCES,
}


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_of(text):
    """C++/CUDA source with comments and blank space removed: what the compiler sees of it (no
    string literal in these sources holds comment markers)."""
    return " ".join(_COMMENT.sub(" ", text).split())


def kernel_source_hash(files=None):
    """sha256 (first 16 hex digits) over the code (comments and spacing aside) of the named csrc
    files, or of all of them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_gqa_attn_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode())
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if its kernel's sources are unchanged
    since the capture.  Keys: attention config names, else "<op>:<config>"."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(key)
        if e and e.get("kernel_source_hash") == kernel_source_hash(KERNEL_SOURCES[e["sources"]]):
            return float(e["dram_bytes_per_launch"]), e.get("kernel", "")
    except Exception:
        pass
    return None, None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.text = ""
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(getattr(self, "text", ""))) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def ranks_max(x, dist, device):
    """The largest x over all ranks (the slowest replica's time), or x alone without a process
    group.  device: where the reduction tensor lives (the rank's GPU for NCCL, "cpu" for gloo)."""
    if not dist:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank):
    """Seed of a rank's batch: rank 0 runs the named workload itself, every other rank an
    independent batch of the same shape (weak scaling: the batch partitions across replicas)."""
    return None if rank == 0 else W.BASE_SEED + 1000 * rank


def problem_bytes(p):
    lens = p.context_lens.cpu().tolist()
    fp8 = p.kv_dtype == W.KV_FP8_E4M3
    return A.attention_bytes(lens, p.q_len, p.num_q_heads, p.num_kv_heads, p.head_dim,
                             p.block_size, 1 if fp8 else 2, fp8)


def input_tensors(p):
    ts = [p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens]
    if p.k_scale is not None:
        ts += [p.k_scale, p.v_scale]
    return ts


def cpu_oracle_rate(p, budget_s, max_seqs=None):
    """Time the oracle (as it stands) on whole sequences of the workload for about budget_s."""
    import oracle

    B = p.num_seqs
    n = B if max_seqs is None else min(B, max_seqs)
    host = p.to("cpu")
    seqs_done = 0
    t0 = time.perf_counter()
    start = 0
    while True:
        sel = [(start + i) % B for i in range(n)]
        oracle.attention_problem(host, seqs=sel)
        seqs_done += n
        start = (start + n) % B
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return seqs_done / dt, seqs_done, dt, oracle.max_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return
    p = W.make_config(args.config, device="cpu")
    import oracle

    oracle.build()
    per_step = max(1, min(p.num_seqs, args.ref_seqs_per_step))
    for _ in range(args.warmup):
        oracle.attention_problem(p, seqs=list(range(per_step)))
    t0 = time.perf_counter()
    done = 0
    for k in range(args.steps):
        sel = [(k * per_step + i) % p.num_seqs for i in range(per_step)]
        oracle.attention_problem(p, seqs=sel)
        done += per_step
    dt = time.perf_counter() - t0
    rate = done / dt
    threads = oracle.max_threads()
    sample = (f"{per_step} of {p.num_seqs} sequences per step (all {p.num_q_heads} query heads, "
              f"full contexts), fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCRIPTIONS[args.config], "name": args.config},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def pool_rotation(alg_bytes):
    """How many copies of a workload's inputs the timed calls rotate over so that every call
    reads its KV from HBM: enough copies that the others' reads (> 3x the L2) evict a copy
    before its next turn; 1 when one call alone reads > 3x the L2.  Capped at 8 (the 63 KB
    parity-only case stays L2-warm and says so)."""
    if alg_bytes >= 3 * L2_BYTES:
        return 1
    return min(8, max(4, math.ceil(3 * L2_BYTES / max(alg_bytes, 1)) + 1))


def time_attention(p, args, dev, stream, local_rank, dist, rotate):
    """Capture args.steps calls of paged_attn_decode / paged_attn_verify on p in one CUDA graph
    (call k on copy k % rotate of the inputs) and time one replay between an event pair on the
    launching stream, after a soak that the clock sampler watches.  Returns (device seconds of
    the replay, max over ranks; wall seconds; clock summary)."""
    import paged_kv_gqa_attn_gb300 as pa

    max_ctx = int(p.context_lens.max())
    copies = [(p, torch.empty_like(p.q))]
    for _ in range(rotate - 1):
        cp = dataclasses.replace(p, q=p.q.clone(), k_cache=p.k_cache.clone(), v_cache=p.v_cache.clone(),
                                 k_scale=None if p.k_scale is None else p.k_scale.clone(),
                                 v_scale=None if p.v_scale is None else p.v_scale.clone())
        copies.append((cp, torch.empty_like(p.q)))

    def step(k):
        cp, o = copies[k % rotate]
        pa.run_problem(cp, out=o, stream=stream, max_context_len=max_ctx)

    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3)):
            step(k)
    stream.synchronize()
    st = pa.check_device_errors(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"device error before timing: {pa.status_string(st)}")
    # The K timed calls are captured once in a CUDA graph and replayed as one submission: the
    # kernels of consecutive calls then run back to back, as in a serving loop under graphs, with
    # no per-call launch gaps and no events between calls (an event pair around every call adds
    # a few microseconds to each).  One event pair on the launching stream brackets the replay.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for k in range(args.steps):
                step(k)
        graph.replay()  # untimed: the first replay after the capture
    stream.synchronize()
    st = pa.check_device_errors(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"device error in the captured steps: {pa.status_string(st)}")
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        # untimed soak so that the clock sampler sees the GPU under this load
        s0 = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - s0 < args.soak_s:
                graph.replay()
                stream.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            ev_start.record(stream)
            graph.replay()
            ev_end.record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        if dist:
            dist.barrier()
    st = pa.check_device_errors(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"device error during timing: {pa.status_string(st)}")
    dev_total = max(ev_start.elapsed_time(ev_end) / 1e3, 1e-12)
    del graph, copies
    return ranks_max(dev_total, dist, dev), t1 - t0, clk.summary()


def attention_launches(pa, p, dev):
    """Kernels one call launches: decode = the mma.sync kernel (+ the merge when split);
    verify = the persistent tcgen05 kernel + its merge (+ the planner beyond 1022 sequences)."""
    B = p.num_seqs
    if p.q_len > 1:
        return 2 + (1 if B > 1022 else 0)
    _, nparts = pa.plan(torch.cuda.get_device_properties(dev).multi_processor_count, B, p.num_kv_heads,
                        int(p.context_lens.max()), p.block_size, p.q_len,
                        pa.PA_KV_FP8_E4M3 if p.kv_dtype == W.KV_FP8_E4M3 else pa.PA_KV_BF16)
    return 1 + (1 if nparts > 1 else 0)


def l2_note(alg_bytes, rotate):
    if rotate == 1:
        return (f"no flush: each step reads {alg_bytes / 1e6:.0f} MB of KV, "
                f"{alg_bytes / L2_BYTES:.1f}x the 129 MB L2")
    if rotate * alg_bytes >= 3 * L2_BYTES:
        return (f"cold: calls rotate over {rotate} copies of the inputs ({rotate * alg_bytes / 1e6:.0f} MB, "
                f"{rotate * alg_bytes / L2_BYTES:.1f}x the 129 MB L2), so each call reads its KV from HBM")
    return f"L2-warm: {rotate} copies of a {alg_bytes / 1e3:.0f} KB workload stay in the 129 MB L2 (parity-only size)"


def config_entry(name, args, dev, stream, local_rank, dist, world, kv_over, peak, seed):
    """Time one attention workload; returns (entry dict for the JSON line, problem, step seconds)."""
    import paged_kv_gqa_attn_gb300 as pa

    p = W.make_config(name, seed=seed, device=dev, **kv_over)
    alg = problem_bytes(p)
    rotate = pool_rotation(alg)
    elapsed, wall, clocks = time_attention(p, args, dev, stream, local_rank, dist, rotate)
    step_s = elapsed / args.steps
    achieved = alg / step_s / 1e9
    e = {
        "workload": DESCRIPTIONS[name],
        "kv_dtype": "fp8_e4m3" if p.kv_dtype == W.KV_FP8_E4M3 else "bf16",
        "ms_per_step": step_s * 1e3,
        "value": world * p.num_seqs * args.steps / elapsed,
        "unit": UNIT,
        "algorithmic_bytes_per_launch": alg,
        "achieved_gbs": achieved,
        "frac": achieved / peak,
        "l2": l2_note(alg, rotate),
        "gpu_launches_per_step": attention_launches(pa, p, dev),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    traffic, tkernel = profiled_traffic(name if not kv_over else
                                        f"{name}:{'fp8' if p.kv_dtype == W.KV_FP8_E4M3 else 'bf16'}")
    if traffic is not None:
        # DRAM bytes of one launch of the dominant kernel, from the committed ncu capture
        e["traffic"] = traffic
        e["traffic_kernel"] = tkernel
    if name == "tiny":
        e["note"] = "parity-only size: no roofline target"
    if rotate > 1 and name != "tiny":
        # the same calls on one copy of the inputs, for comparison (L2 keeps part of the KV)
        w_elapsed, _, _ = time_attention(p, args, dev, stream, local_rank, dist, 1)
        w_step = w_elapsed / args.steps
        e["warm_single_copy"] = {"ms_per_step": w_step * 1e3, "achieved_gbs": alg / w_step / 1e9,
                                 "frac": alg / w_step / 1e9 / peak,
                                 "l2": f"not flushed: one copy of {alg / 1e6:.0f} MB, "
                                       f"{alg / L2_BYTES:.2f}x the L2, read by every call"}
    return e, p, step_s


def run_ours(args, rank, world, local_rank):
    import paged_kv_gqa_attn_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.load_library()
    dist = torch.distributed if world > 1 else None
    # each rank owns its own batch of sequences: a replica with its own seed
    seed = replica_seed(rank)
    kv_over = {} if args.kv_dtype == "auto" else {"kv_dtype": W.KV_FP8_E4M3 if args.kv_dtype == "fp8" else W.KV_BF16}
    stream = torch.cuda.Stream(device=dev)
    pa.set_max_partitions(args.max_partitions)  # 0: the library's automatic split
    peak, peak_kind = measured_peaks()

    head, p, step_s = config_entry(args.config, args, dev, stream, local_rank, dist, world, kv_over, peak, seed)
    B = p.num_seqs
    alg_bytes = head["algorithmic_bytes_per_launch"]
    kv_pool_bytes = p.k_cache.numel() * p.k_cache.element_size() * 2
    max_ctx = int(p.context_lens.max())
    ppp, nparts = pa.plan(torch.cuda.get_device_properties(dev).multi_processor_count, B,
                          p.num_kv_heads, max_ctx, p.block_size, p.q_len,
                          pa.PA_KV_FP8_E4M3 if p.kv_dtype == W.KV_FP8_E4M3 else pa.PA_KV_BF16)
    on_tc = p.q_len > 1
    out = torch.empty_like(p.q)

    def step():
        pa.run_problem(p, out=out, stream=stream, max_context_len=max_ctx)

    # end to end through the public API with host buffers: pinned inputs copied in every step
    host_in = [t.detach().to("cpu").pin_memory() for t in input_tensors(p)]
    dev_in = input_tensors(p)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    with torch.cuda.stream(stream):
        for _ in range(2):
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)
            step()
            host_out.copy_(out, non_blocking=True)
    stream.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)
            step()
            host_out.copy_(out, non_blocking=True)
    stream.synchronize()
    e_elapsed = time.perf_counter() - e0
    e_elapsed = ranks_max(e_elapsed, dist, dev)
    e2e_value = world * B * e2e_steps / e_elapsed
    del host_in

    # every other workload, timed the same way (the headline's own figures are above)
    others = {}
    if not args.headline_only:
        for name in [c for c in args.other_configs.split(",") if c and c != args.config]:
            e, q, _ = config_entry(name, args, dev, stream, local_rank, dist, world, kv_over, peak, seed)
            others[name] = e
            del q
            torch.cuda.empty_cache()

    if rank != 0:
        return
    achieved = head["achieved_gbs"]
    traffic, traffic_kernel = profiled_traffic(args.config if args.kv_dtype == "auto" else
                                               f"{args.config}:{args.kv_dtype}")
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, nseq, dt, thr = cpu_oracle_rate(p.to("cpu"), args.cpu_budget_s, max_seqs=args.cpu_seqs)
        cpu = {"value": rate, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"{nseq} whole sequences of this workload, taken in turn ({dt:.1f} s of fp64 "
                         f"oracle work)"}
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3 KV, bf16 Q/O, fp32 accumulate" if p.kv_dtype == W.KV_FP8_E4M3
        else "bf16 KV/Q/O, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) Q/K/V, random page placement)",
        "config": {
            "workload": DESCRIPTIONS[args.config] + ("" if args.kv_dtype == "auto" else
                                                     f" (KV stored as {args.kv_dtype}: --kv-dtype)"),
            "kv_dtype": head["kv_dtype"],
            "name": args.config,
            "batch": B,
            "q_len": p.q_len,
            "max_context_len": max_ctx,
            "total_context_tokens": int(p.context_lens.sum()),
            "kv_pool_bytes": kv_pool_bytes,
            "split_kv": ({"pages_per_partition": ppp, "max_partitions": nparts,
                          "forced": args.max_partitions > 0} if not on_tc else
                         {"persistent_ctas": 2 * torch.cuda.get_device_properties(dev).multi_processor_count,
                          "split": "equal page ranges of the (kv head, sequence page) space"}),
            "l2": head["l2"],
            "parallelism": f"replicas x{world}",
            "timing": f"the {args.steps} timed calls captured in one CUDA graph, one replay between an "
                      "event pair on the launching stream",
        },
        "hbm_tbs": achieved / 1e3,
        "frac_of_peak_hbm": achieved / peak,
        "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "kernel": ("paged_attn_decode call (mma.sync decode kernel + split-KV merge)" if not on_tc else
                       "paged_attn_verify call (persistent tcgen05 verify kernel + merge)"),
            "algorithmic_bytes_per_launch": alg_bytes,
            "peak_kind": f"{peak_kind} hbm_gbs (copy bandwidth)",
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall_s_timed_region"],
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if others:
        line["configs"] = others
    print(json.dumps(line), flush=True)


class L2Flush:
    """Evict the L2 between timed steps: write one buffer of twice the L2, then read another
    of the same size, so that the written lines are written back during the flush and the L2
    is left holding clean lines of neither the inputs nor the outputs."""

    def __init__(self, dev):
        self.w = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def fill_(self, k):
        self.w.fill_(k & 0xFF)
        self.r.max()


def timed_flushed_steps(args, step, stream, flush, dev, local_rank, dist, pa):
    """Warm up, soak under the clock sampler, then time args.steps calls of step(k) with CUDA
    events around each one, L2 flushed before each (outside the events).  Returns (summed
    device seconds, max over ranks; wall seconds of the timed loop; clock sampler)."""
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3)):
            step(k)
    st = pa.check_device_errors(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"device error before timing: {pa.status_string(st)}")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        # untimed soak so that the clock sampler sees the GPU under this load
        s0 = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - s0 < args.soak_s:
                for k in range(20):
                    flush.fill_(k)
                    step(k)
                stream.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush.fill_(k & 0xFF)
                evs[k][0].record(stream)
                step(k)
                evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        if dist:
            dist.barrier()
    st = pa.check_device_errors(stream)
    if st != pa.PA_OK:
        raise RuntimeError(f"device error during timing: {pa.status_string(st)}")
    elapsed = sum(a.elapsed_time(b) / 1e3 for a, b in evs)
    elapsed = ranks_max(elapsed, dist, dev)
    return elapsed, wall, clk


ACCEPT_METRIC = "speculative acceptance: rounds/s; achieved HBM GB/s (% of GB300 peak)"
ACCEPT_UNIT = "rounds/s"


def accept_bytes(num_accepted, K, V):
    """Bytes a round must read and write: per draft position the token, p(x), q(x) and u
    (4 B each) up to and including the first rejection, the word, the draw's row (p and q at a
    rejection, p alone for a bonus: V fp32 each), and the K + 2 output ints."""
    total = 0
    for n in num_accepted:
        n = int(n)
        tested = min(n + 1, K)
        total += tested * 16 + 4 + (2 if n < K else 1) * V * 4 + (K + 2) * 4
    return total


def run_accept(args, rank, world, local_rank):
    """One step = one paged_attn_spec_accept call over the batch of rounds (decision, then one
    draw per round over the vocabulary).  L2 is flushed between steps (outside the events)."""
    import paged_kv_gqa_attn_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.load_library()
    dist = torch.distributed if world > 1 else None
    seed = replica_seed(rank)
    a = W.make_accept_config(args.accept_config, seed=seed, device=dev)
    B, K, V = a.num_seqs, a.num_draft, a.vocab
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    num_acc = torch.empty(B, dtype=torch.int32, device=dev)

    def step(k):
        pa.spec_accept(a.p, a.q, a.draft, a.u_accept, a.u_sample, out_tokens=out_tokens,
                       num_accepted=num_acc, stream=stream)

    elapsed, wall, clk = timed_flushed_steps(args, step, stream, flush, dev, local_rank, dist, pa)
    n_host = num_acc.cpu().tolist()
    alg = accept_bytes(n_host, K, V)
    value = world * B * args.steps / elapsed
    step_s = elapsed / args.steps

    # end to end: the round's distributions, drafts and uniforms come from pinned host memory,
    # the emitted tokens and counts go back
    dev_in = [a.p, a.q, a.draft, a.u_accept, a.u_sample]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = [torch.empty_like(out_tokens, device="cpu").pin_memory(),
                torch.empty_like(num_acc, device="cpu").pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for h, dv in zip(host_in, dev_in):
                dv.copy_(h, non_blocking=True)
            step(0)
            host_out[0].copy_(out_tokens, non_blocking=True)
            host_out[1].copy_(num_acc, non_blocking=True)
    stream.synchronize()
    e2e_value = world * B * e2e_steps / (time.perf_counter() - e0)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle import spec_accept as SA
        import numpy as np

        hp, hq, hd, hu, hw = (t.cpu().numpy() for t in dev_in)
        done, spent = 0, 0.0
        while spent < args.cpu_budget_s:
            t0 = time.perf_counter()
            SA.accept_batch(hp, hq, hd, hu, hw.view(np.uint32))
            spent += time.perf_counter() - t0
            done += B
        cpu = {"value": done / spent, "unit": ACCEPT_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{done} rounds of this workload ({spent:.1f} s of numpy oracle work)"}
    peak, peak_kind = measured_peaks()
    achieved = alg / step_s / 1e9
    line = {
        "metric": ACCEPT_METRIC, "value": value, "unit": ACCEPT_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 probabilities, u64 fixed-point draw",
        "data": "synthetic (seeded target logits N(0, 9), draft = target + N(0, 1) noise, softmax)",
        "config": {"workload": f"speculative acceptance: B={B} rounds of K={K} drafts over a "
                               f"{V}-token vocabulary", "name": args.accept_config, "batch": B,
                   "num_draft": K, "vocab": V, "mean_accepted": sum(n_host) / B,
                   "l2": "flushed between steps outside the timed events (2x L2 written, then 2x L2 read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(f"accept:{args.accept_config}")[0],
                     "kernel": "paged_attn_spec_accept call (scan kernel + pick kernel)",
                     "algorithmic_bytes_per_launch": alg,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy bandwidth)"},
        "e2e": {"value": e2e_value, "unit": ACCEPT_UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


PREFILL_METRIC = "paged prefill attention: new tokens/s; achieved TFLOP/s (% of GB300 bf16 peak)"
PREFILL_UNIT = "tokens/s"
PREFILL_CONFIGS = {
    "prefill_chunk512": dict(chunk=512, num_seqs=4, decodes=0),
    "prefill_chunk2048": dict(chunk=2048, num_seqs=4, decodes=0),
    "prefill_chunk512_mix": dict(chunk=512, num_seqs=4, decodes=64),
}


def prefill_flops(context_lens, q_lens, num_q_heads, head_dim):
    """Useful FLOPs: every (row, query head) scores and weights the n = L - q_len + i + 1 tokens
    it sees, 2 d flops each for Q.K and for P.V."""
    total = 0
    for L, ql in zip(context_lens, q_lens):
        first = L - ql
        # sum over i of (first + i + 1) for i in [0, ql)
        total += ql * first + ql * (ql + 1) // 2
    return 4 * head_dim * num_q_heads * total


def run_prefill(args, rank, world, local_rank):
    """One step = one paged_attn_prefill call over the packed rows of the workload (prompt chunks
    after their cached prefix, plus piggybacked decode rows in the _mix workload)."""
    import paged_kv_gqa_attn_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.load_library()
    dist = torch.distributed if world > 1 else None
    seed = replica_seed(rank)
    cfg = PREFILL_CONFIGS[args.prefill_config]
    fp8 = args.kv_dtype == "fp8"
    pv = W.chunked_prefill_workload(seed=seed, device=dev, kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16, **cfg)
    lens = pv.context_lens.cpu().tolist()
    qls = pv.q_lens
    total_q = int(pv.q.shape[0])
    max_q = max(qls)
    max_ctx = max(lens)
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    out = torch.empty_like(pv.q)

    def step(k):
        pa.prefill(pv.q, pv.k_cache, pv.v_cache, pv.block_table, pv.context_lens, pv.query_start_loc,
                   pv.scale, max_q_len=max_q, max_context_len=max_ctx, out=out, stream=stream,
                   k_scale=pv.k_scale, v_scale=pv.v_scale)

    elapsed, wall, clk = timed_flushed_steps(args, step, stream, flush, dev, local_rank, dist, pa)
    value = world * total_q * args.steps / elapsed
    step_s = elapsed / args.steps
    flops = prefill_flops(lens, qls, pv.num_q_heads, pv.head_dim)

    # end to end: the step's query rows and metadata from pinned host memory, the output back
    dev_in = [pv.q, pv.block_table, pv.context_lens, pv.query_start_loc]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for h, dv in zip(host_in, dev_in):
                dv.copy_(h, non_blocking=True)
            step(0)
            host_out.copy_(out, non_blocking=True)
    stream.synchronize()
    e2e_value = world * total_q * e2e_steps / (time.perf_counter() - e0)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        host = pv.to("cpu")
        rng = torch.Generator().manual_seed(5)
        done, spent = 0, 0.0
        while spent < args.cpu_budget_s:
            rows = torch.randint(0, total_q, (16,), generator=rng).tolist()
            t0 = time.perf_counter()
            oracle.attention_varlen_problem(host, rows=rows)
            spent += time.perf_counter() - t0
            done += len(rows)
        cpu = {"value": done / spent, "unit": PREFILL_UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"{done} random packed rows of this workload, all heads ({spent:.1f} s of fp64 "
                         f"oracle work)"}
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (cuBLAS burst)"
    except Exception:
        peak, peak_kind = 1900.0, "fallback bf16 burst"
    achieved = flops / step_s / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": PREFILL_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 KV, bf16 Q/O, f16 products, fp32 accumulate" if fp8 else "bf16 Q/KV/O, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) Q/K/V, random page placement)",
        "config": {"workload": f"chunked prefill: {cfg['num_seqs']} prompt chunks of {cfg['chunk']} tokens after "
                               f"a cached prefix U[0,4096]" + (f" + {cfg['decodes']} decode rows"
                                                              if cfg["decodes"] else "")
                               + ", Hq 32 / Hkv 8, d 128, bs 16, "
                               + ("E4M3 KV with per-(block, kv head) scales" if fp8 else "bf16 KV"),
                   "name": args.prefill_config, "total_q": total_q, "max_q_len": max_q,
                   "max_context_len": max_ctx,
                   "l2": "flushed between steps outside the timed events (2x L2 written, then 2x L2 read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(f"prefill:{args.prefill_config}" + (":fp8" if fp8 else ""))[0],
                     "kernel": "prefill_tc_kernel",
                     "algorithmic_flops_per_launch": flops, "peak_kind": peak_kind},
        "e2e": {"value": e2e_value, "unit": PREFILL_UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


APPEND_METRIC = "KV append: achieved HBM GB/s (% of GB300 peak); appended tokens/s"
APPEND_UNIT = "tokens/s"


def append_bytes(lens, n_new, num_kv_heads, head_dim, block_size, fp8):
    """Bytes a KV append must move: read the new K and V rows (bf16) and write them into the
    cache; for an fp8 cache also read the older valid tokens of every touched block (their amax
    decides the block scale) and read/write the (block, head) scales.  Re-encoding the older
    tokens when a scale changes is not counted (a lower bound)."""
    total = 0
    for L in lens:
        first = L - n_new
        rows = n_new * num_kv_heads * head_dim * 2  # one side, one element per dim
        if not fp8:
            total += 2 * (rows * 2)  # K and V: read bf16 + write bf16 (2 bytes each)
            continue
        total += 2 * rows  # read the new bf16 rows, K and V
        for blk in range(first // block_size, (L - 1) // block_size + 1):
            s0 = max(first - blk * block_size, 0)
            s1 = min(L - blk * block_size, block_size)
            total += 2 * num_kv_heads * (s0 * head_dim + (s1 - s0) * head_dim + 8)
    return total


def run_append(args, rank, world, local_rank):
    """One step = one paged_attn_append_kv call storing n_new tokens per sequence (the config's
    q_len unless --n-new says otherwise) into the config's cache.  For fp8 pools the step
    alternates between two sets of new rows of different magnitude, so that the block scales
    change at every step as they do in serving.  L2 is flushed between steps (outside the
    events) because one step moves far less than the 129 MB L2."""
    import paged_kv_gqa_attn_gb300 as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pa.load_library()
    dist = torch.distributed if world > 1 else None
    seed = replica_seed(rank)
    p = W.make_config(args.config, seed=seed, device=dev)
    n_new = args.n_new or p.q_len
    lens = p.context_lens.cpu().tolist()
    if n_new > min(lens):
        raise SystemExit(f"--n-new {n_new} exceeds the shortest context {min(lens)}")
    B, Hkv, d = p.num_seqs, p.num_kv_heads, p.head_dim
    fp8 = p.kv_dtype == W.KV_FP8_E4M3
    g = torch.Generator(device="cpu").manual_seed(W.BASE_SEED + 77)
    sets = []
    for mag in (1.0, 2.0):
        sets.append(tuple((torch.randn(B, n_new, Hkv, d, generator=g) * mag).to(torch.bfloat16).to(dev)
                          for _ in range(2)))
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    alg = append_bytes(lens, n_new, Hkv, d, p.block_size, fp8)

    def step(k):
        kn, vn = sets[k & 1]
        pa.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                     k_scale=p.k_scale, v_scale=p.v_scale, stream=stream)

    elapsed, wall, clk = timed_flushed_steps(args, step, stream, flush, dev, local_rank, dist, pa)
    value = world * B * n_new * args.steps / elapsed
    step_s = elapsed / args.steps

    # end to end: the step's new rows and metadata come from pinned host memory, the touched
    # pages of the K cache go back to the host
    host_in = [t.to("cpu").pin_memory() for t in (*sets[0], p.block_table, p.context_lens)]
    dev_in = [sets[0][0], sets[0][1], p.block_table, p.context_lens]
    touched = sorted({int(p.block_table[b, j // p.block_size]) for b, L in enumerate(lens)
                      for j in range(L - n_new, L)})
    touched_idx = torch.tensor(touched, dtype=torch.int64, device=dev)
    host_out = torch.empty((len(touched),) + tuple(p.k_cache.shape[1:]), dtype=p.k_cache.dtype,
                           pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for h, dv in zip(host_in, dev_in):
                dv.copy_(h, non_blocking=True)
            step(0)
            host_out.copy_(p.k_cache.index_select(0, touched_idx), non_blocking=True)
    stream.synchronize()
    e2e_value = world * B * n_new * e2e_steps / (time.perf_counter() - e0)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_append_rate(p, sets[0], n_new, fp8, args.cpu_budget_s)
    peak, peak_kind = measured_peaks()
    achieved = alg / step_s / 1e9
    line = {
        "metric": APPEND_METRIC, "value": value, "unit": APPEND_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 rows -> fp8_e4m3 KV (fp32 scale arithmetic)" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) rows, two magnitudes alternating)",
        "config": {"workload": f"KV append of {n_new} token(s) per sequence into: " + DESCRIPTIONS[args.config],
                   "name": args.config, "batch": B, "n_new": n_new,
                   "l2": "flushed between steps outside the timed events (2x L2 written, then 2x L2 read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(f"append:{args.config}:n{n_new}")[0],
                     "kernel": "append kernel",
                     "algorithmic_bytes_per_launch": alg,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy bandwidth)"},
        "e2e": {"value": e2e_value, "unit": APPEND_UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def cpu_append_rate(p, rows, n_new, fp8, budget_s):
    """Time the append oracle (as it stands, single-threaded numpy) on growing prefixes of the
    batch until about budget_s of work is done."""
    from oracle import append as OA

    host = p.to("cpu")
    kn, vn = rows[0].cpu(), rows[1].cpu()
    done, spent, n = 0, 0.0, 1
    while spent < budget_s and n <= p.num_seqs:
        t0 = time.perf_counter()
        OA.append_kv(kn[:n], vn[:n], host.k_cache, host.v_cache, host.block_table[:n],
                     host.context_lens[:n], n_new=n_new, block_size=p.block_size, fp8=fp8,
                     k_scale=host.k_scale, v_scale=host.v_scale)
        spent += time.perf_counter() - t0
        done += n
        n *= 2
    return {"value": done * n_new / spent, "unit": APPEND_UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} sequence appends of this workload ({spent:.1f} s of numpy oracle work)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(W.CONFIG_NAMES), default="cb_mix")
    ap.add_argument("--other-configs", default="llama8b_decode,spec_verify_k4,spec_verify_k8,long_fp8,tiny",
                    help="attention: the workloads timed after the headline and reported under 'configs'")
    ap.add_argument("--headline-only", action="store_true",
                    help="attention: time the --config workload alone")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--soak-s", type=float, default=1.5)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--cpu-seqs", type=int, default=8)
    ap.add_argument("--ref-seqs-per-step", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=["attention", "append", "accept", "prefill"], default="attention",
                    help="attention (the default step), the KV append that precedes it, or the "
                         "speculative acceptance that follows verify")
    ap.add_argument("--accept-config", choices=list(W.ACCEPT_CONFIGS), default="spec_accept_k8")
    ap.add_argument("--prefill-config", choices=list(PREFILL_CONFIGS), default="prefill_chunk512")
    ap.add_argument("--n-new", type=int, default=0, help="append: tokens per sequence (default q_len)")
    ap.add_argument("--max-partitions", type=int, default=0,
                    help="attention decode: at most this many split-KV partitions per sequence (0: automatic)")
    ap.add_argument("--kv-dtype", choices=["auto", "bf16", "fp8"], default="auto",
                    help="attention and prefill: store the workload's KV as bf16 or E4M3 (default: the workload's own)")
    args = ap.parse_args()

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.op == "append":
            run_append(args, rank, world, local_rank)
        elif args.op == "accept":
            run_accept(args, rank, world, local_rank)
        elif args.op == "prefill":
            run_prefill(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
