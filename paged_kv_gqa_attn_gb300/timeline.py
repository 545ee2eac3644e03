"""Per-CTA timeline of one verify call, from the instrumented build of the library.

    python -m paged_kv_gqa_attn_gb300.timeline [--config spec_verify_k8] [--calls 20] [--raw FILE]

Builds the -DPA_TIMELINE variant (a separate library under _lib/timeline; the product library
has no instrumentation), runs the named workload's verify call --calls times on one stream, and
reads the %globaltimer stamps that the persistent kernel's CTAs wrote during the last call
(entry, plan built, first scores seen by the softmax, softmax done, exit) and the time the merge
kernel wrote its last row.  Prints percentiles over the CTAs, in microseconds from the earliest
CTA entry, as one JSON line (--raw also writes every CTA's stamps).  The stamps cost a few global
stores per CTA: use them for where the time goes, and bench.py (product library) for durations.
"""

from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np
import torch

NSLOTS = 8
NAMES = {0: "entry", 1: "plan", 2: "first_s", 3: "softmax_done", 7: "exit"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="spec_verify_k8")
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--kv-dtype", choices=["auto", "bf16", "fp8"], default="auto")
    ap.add_argument("--raw", default="", help="also write every CTA's stamps (JSON) to this file")
    args = ap.parse_args()

    import paged_kv_gqa_attn_gb300 as pa
    from paged_kv_gqa_attn_gb300 import workloads as W

    lib = pa.load_library(timeline=True)
    lib.paged_attn_timeline_read_verify.restype = ctypes.c_int
    lib.paged_attn_timeline_read_verify.argtypes = [ctypes.c_void_p, ctypes.c_int]
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
    if args.raw:
        with open(args.raw, "w") as f:
            json.dump({"slots": ["entry", "plan", "first_s", "softmax_done", "smid", "segments", "steps", "exit"],
                       "t0": int(t0), "merge_end": int(buf[-1]), "ctas": a.astype(np.int64).tolist()}, f)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
