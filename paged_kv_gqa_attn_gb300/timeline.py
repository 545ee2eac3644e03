"""Per-CTA timeline of one verify call, or per-role cycle sums of one chunked-prefill call, from
the instrumented build of the library.

    python -m paged_kv_gqa_attn_gb300.timeline [--config spec_verify_k8] [--calls 20] [--raw FILE] [--kv-dtype fp8]
    python -m paged_kv_gqa_attn_gb300.timeline --op prefill [--chunk 2048] [--num-seqs 4] [--kv-dtype fp8]

Builds the -DPA_TIMELINE variant (a separate library under _lib/timeline; the product library
has no instrumentation), runs the named workload's verify call --calls times on one stream, and
reads the %globaltimer stamps that the persistent kernel's CTAs wrote during the last call
(entry, plan built, first scores seen by the softmax, softmax done, exit) and the time the merge
kernel wrote its last row.  Prints percentiles over the CTAs, in microseconds from the earliest
CTA entry, as one JSON line (--raw also writes every CTA's stamps).  The stamps cost a few global
stores per CTA: use them for where the time goes, and bench.py (product library) for durations.

The verify run also reads the per-step SM-clock stamps of 16 CTAs (the first eight of each half
of the grid, which pair up on SMs) over their first 64 steps and prints, as "cycles_per_step",
medians over the steps k >= 3 of: the PV-to-PV period, the softmax busy (S(k) seen -> the later
warp's P(k)) and its wait for S, the skew of the two softmax warps' P, QK(k) issued -> S(k) seen,
PV(k-2) issued -> QK(k) issued, the K and V copies' lead over QK and PV, the hand-off from the
last of P(k) (and, E4M3, V(k) converted) to PV(k) issued, and for E4M3 the V copy's landing and
conversion times.

--op prefill runs the chunked-prefill workload (num_seqs prompt chunks of --chunk tokens after a
cached prefix U[0, 4096], Llama-3-8B attention shape) and reads, per CTA, the clock64 sums that
thread 0 of the softmax and the MMA issuer keep over the steps s >= 2: softmax busy (S(s) seen ->
P(s) arrived) and its phases, softmax waiting for S, the handoff from the last softmax warp's P(s)
to PV(s) issued, the skew of the four warps' P(s) arrivals, the chain PV(s-2) issued -> S(s)
seen, and PV(s-2) issued -> QK(s) issued.  Prints their means per step in SM cycles.
"""

from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np
import torch

NSLOTS = 8
NAMES = {0: "entry", 1: "plan", 2: "first_s", 3: "softmax_done", 7: "exit"}
# per-step stamps: [16 CTAs][64 steps][10 slots] (the kernel's StepSlot order)
ST_CTAS, ST_STEPS = 16, 64
(ST_VCOPY, ST_VLANDED, ST_CONVV, ST_CONVK, ST_QK, ST_S, ST_P0, ST_PV, ST_KCOPY, ST_P1, ST_SLOTS) = range(11)


def step_summary(a, fp8):
    """Medians over every sampled CTA's steps k >= 3 (SM cycles)."""
    acc = {}

    def add(name, v):
        acc.setdefault(name, []).append(float(v))

    for t in a:
        n = int((t[:, ST_PV] > 0).sum())
        for k in range(3, n):
            p = max(t[k, ST_P0], t[k, ST_P1])
            add("period_pv", t[k, ST_PV] - t[k - 1, ST_PV])
            add("softmax_busy", p - t[k, ST_S])
            add("softmax_wait_s", t[k, ST_S] - max(t[k - 1, ST_P0], t[k - 1, ST_P1]))
            add("p_skew", abs(t[k, ST_P0] - t[k, ST_P1]))
            add("qk_to_s", t[k, ST_S] - t[k, ST_QK])
            add("pv2_to_qk", t[k, ST_QK] - t[k - 2, ST_PV])
            add("kcopy_to_qk", t[k, ST_QK] - t[k, ST_KCOPY])
            add("vcopy_to_pv", t[k, ST_PV] - t[k, ST_VCOPY])
            if fp8:
                v = max(t[k, ST_CONVV], t[k, ST_CONVK])
                add("handoff_to_pv", t[k, ST_PV] - max(p, v))
                add("vcopy_to_landed", t[k, ST_VLANDED] - t[k, ST_VCOPY])
                add("landed_to_converted", t[k, ST_CONVV] - t[k, ST_VLANDED])
            else:
                add("handoff_to_pv", t[k, ST_PV] - p)
    return {k: round(float(np.median(v)), 1) for k, v in acc.items()}, sum(len(v) for v in acc.values()) // max(len(acc), 1)


PF_SLOTS = 16


def prefill_main(args):
    import paged_kv_gqa_attn_gb300 as pa
    from paged_kv_gqa_attn_gb300 import workloads as W

    lib = pa.load_library(timeline=True)
    lib.paged_attn_timeline_read_prefill.restype = ctypes.c_int
    lib.paged_attn_timeline_read_prefill.argtypes = [ctypes.c_void_p, ctypes.c_int]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kv = W.KV_FP8_E4M3 if args.kv_dtype == "fp8" else W.KV_BF16
    pv = W.chunked_prefill_workload(device=dev, chunk=args.chunk, num_seqs=args.num_seqs, decodes=args.decodes,
                                    kv_dtype=kv)
    out = torch.empty_like(pv.q)
    max_q = max(pv.q_lens)
    max_ctx = int(pv.context_lens.max())

    def call():
        pa.prefill(pv.q, pv.k_cache, pv.v_cache, pv.block_table, pv.context_lens, pv.query_start_loc, pv.scale,
                   max_q_len=max_q, max_context_len=max_ctx, out=out, k_scale=pv.k_scale, v_scale=pv.v_scale)

    nmax = 8192
    buf = np.zeros(nmax * PF_SLOTS, dtype=np.uint64)
    for _ in range(max(1, args.calls - 1)):
        call()
    torch.cuda.synchronize()
    if lib.paged_attn_timeline_read_prefill(buf.ctypes.data, nmax) != 0:  # zeroes the slots
        raise SystemExit("timeline read failed")
    call()
    torch.cuda.synchronize()
    st = pa.check_device_errors()
    if st != pa.PA_OK:
        raise SystemExit(f"device error: {pa.status_string(st)}")
    if lib.paged_attn_timeline_read_prefill(buf.ctypes.data, nmax) != 0:
        raise SystemExit("timeline read failed")
    a = buf.reshape(nmax, PF_SLOTS).astype(np.float64)
    live = a[:, 0] > 0
    a = a[live]
    n = a[:, 9].sum()
    per_step = lambda i: round(float(a[:, i].sum() / max(n, 1)), 1)
    res = {"op": "prefill", "chunk": args.chunk, "num_seqs": args.num_seqs, "decodes": args.decodes,
           "kv": args.kv_dtype if args.kv_dtype != "auto" else "bf16", "ctas": int(live.sum()),
           "steps_summed": int(n), "kernel_us": round(float(a[:, 1].max() - a[:, 0].min()) / 1e3, 2),
           "cycles_per_step": {"softmax_busy": per_step(4), "softmax_wait_s": per_step(5),
                               "handoff_last_p_to_pv": per_step(6), "chain_pv_to_s2": per_step(7),
                               "pv_to_qk2_issue": per_step(8), "p_arrival_skew": per_step(14),
                               "softmax_phases": {"tmem_load": per_step(10), "max_rescale": per_step(11),
                                                  "weights": per_step(12), "tmem_store": per_step(13)}},
           "cta_us": {q: round(float(np.percentile((a[:, 1] - a[:, 0]) / 1e3, q)), 2) for q in (0, 50, 100)}}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["verify", "prefill"], default="verify")
    ap.add_argument("--chunk", type=int, default=2048, help="prefill: new tokens per prompt chunk")
    ap.add_argument("--num-seqs", type=int, default=4, help="prefill: prompt chunks")
    ap.add_argument("--decodes", type=int, default=0, help="prefill: piggybacked decode rows")
    ap.add_argument("--config", default="spec_verify_k8")
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--kv-dtype", choices=["auto", "bf16", "fp8"], default="auto")
    ap.add_argument("--raw", default="", help="also write every CTA's stamps (JSON) to this file")
    args = ap.parse_args()
    if args.op == "prefill":
        return prefill_main(args)

    import paged_kv_gqa_attn_gb300 as pa
    from paged_kv_gqa_attn_gb300 import workloads as W

    lib = pa.load_library(timeline=True)
    lib.paged_attn_timeline_read_verify.restype = ctypes.c_int
    lib.paged_attn_timeline_read_verify.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.paged_attn_timeline_read_verify_steps.restype = ctypes.c_int
    lib.paged_attn_timeline_read_verify_steps.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kv = {} if args.kv_dtype == "auto" else {"kv_dtype": W.KV_FP8_E4M3 if args.kv_dtype == "fp8" else W.KV_BF16}
    p = W.make_config(args.config, device=dev, **kv)
    if p.q_len == 1:
        raise SystemExit("the instrumented kernel is the verify kernel: pick a verify workload")
    out = torch.empty_like(p.q)
    ncta = 2 * torch.cuda.get_device_properties(dev).multi_processor_count
    buf = np.zeros(ncta * NSLOTS + 1, dtype=np.uint64)
    for _ in range(max(1, args.calls - 1)):
        pa.run_problem(p, out=out)
    torch.cuda.synchronize()
    lib.paged_attn_timeline_read_verify(buf.ctypes.data, ncta)  # resets the merge-end stamp
    pa.run_problem(p, out=out)
    torch.cuda.synchronize()
    st = pa.check_device_errors()
    if st != pa.PA_OK:
        raise SystemExit(f"device error: {pa.status_string(st)}")
    if lib.paged_attn_timeline_read_verify(buf.ctypes.data, ncta) != 0:
        raise SystemExit("timeline read failed")
    a = buf[: ncta * NSLOTS].reshape(ncta, NSLOTS)
    t0 = float(a[:, 0].min())
    rel = lambda i: (a[:, i].astype(np.float64) - t0) / 1e3  # us
    active = a[:, 5] > 0  # CTAs whose softmax walked at least one segment
    res = {"config": args.config, "ctas": int(ncta), "active_ctas": int(active.sum())}
    pct = (0, 10, 50, 90, 100)
    for i, name in NAMES.items():
        col = rel(i)[active] if i in (2, 3) else rel(i)
        res[name] = {q: round(float(np.percentile(col, q)), 2) for q in pct}
    res["merge_end"] = round((float(buf[-1]) - t0) / 1e3, 2)
    body = rel(3)[active] - rel(2)[active]
    res["body_us"] = {q: round(float(np.percentile(body, q)), 2) for q in (0, 50, 100)}
    res["segments_per_cta"] = {q: int(np.percentile(a[active, 5], q)) for q in (0, 50, 100)}
    steps = np.zeros(ST_CTAS * ST_STEPS * ST_SLOTS, dtype=np.int64)
    if lib.paged_attn_timeline_read_verify_steps(steps.ctypes.data) != 0:
        raise SystemExit("timeline read failed")
    st = steps.reshape(ST_CTAS, ST_STEPS, ST_SLOTS).astype(np.float64)
    res["cycles_per_step"], res["steps_sampled"] = step_summary(st, p.kv_dtype == W.KV_FP8_E4M3)
    if args.raw:
        with open(args.raw, "w") as f:
            json.dump({"slots": ["entry", "plan", "first_s", "softmax_done", "smid", "segments", "steps", "exit"],
                       "t0": int(t0), "merge_end": int(buf[-1]), "ctas": a.astype(np.int64).tolist()}, f)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
