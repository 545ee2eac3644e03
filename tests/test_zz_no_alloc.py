"""paged_attn_decode_static_scratch: the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory while they run (a host framework whose
memory manager holds the GPU's memory, a real-time loop that forbids allocation after
start-up).  This file is collected last so that a run stopping at the first failure has run
every other test; it also passes alone in a fresh process.  Each case calls the entry point
through the C ABI twice in a row (the fixed scratch array keeps the first call's contents) and
compares both outputs element by element with the fp64 oracle, under the same bound as the other
GPU parity tests (oracle.parity: bf16 KV max abs 1e-2 and mean abs 1e-3, E4M3 KV max abs 5e-2,
the flat bar wherever a bf16 value can meet it); paged_attn_decode's output on the same inputs
is a second, looser check.  Cases with forced splits make the partials go through the array, and
one test checks that two calls leave the device's free memory unchanged."""

import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _static_scratch_fn():
    lib = pa.load_library()
    fn = lib.paged_attn_decode_static_scratch
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P, P, P, P]
    lib.paged_attn_static_scratch_bytes.restype = ctypes.c_size_t
    return fn, int(lib.paged_attn_static_scratch_bytes())


def _call_static(fn, p, out):
    fp8 = p.kv_dtype == W.KV_FP8_E4M3
    B, q_len, Hq, d = p.q.shape
    NB, Hkv, bs, _ = p.k_cache.shape
    return fn(p.q.data_ptr(), p.k_cache.data_ptr(), p.v_cache.data_ptr(), p.block_table.data_ptr(),
              p.context_lens.data_ptr(), B, p.block_table.shape[1], NB, p.block_table.shape[1] * bs,
              q_len, Hq, Hkv, d, bs, p.scale, 1 if fp8 else 0,
              p.k_scale.data_ptr() if fp8 else None, p.v_scale.data_ptr() if fp8 else None,
              out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _np(t):
    return t.float().cpu().double().numpy()


def _label():
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


FP8 = W.KV_FP8_E4M3
BF16 = W.KV_BF16

# (name, workload name or shape, forced partitions (0: the library's plan))
CASES = [
    ("llama8b_decode", {}, 0),
    ("tiny", {}, 0),
    ("long_fp8", {}, 0),
    ("mixed", dict(lens=[1, 40, 700, 1500, 2100], Hq=32, Hkv=8, d=128, kv=BF16), 0),
    # groups of 8: the decode entry runs the tensor-core kernel, this entry the CUDA cores
    ("group8", dict(lens=[1, 33, 700, 2049], Hq=64, Hkv=8, d=128, kv=BF16), 0),
    ("group8_fp8", dict(lens=[1, 33, 700, 2049], Hq=64, Hkv=8, d=128, kv=FP8), 0),
    # groups of 1 (multi-head attention): the kernel's reduce-scatter has nothing to scatter
    ("group1", dict(lens=[1, 17, 300, 1300], Hq=8, Hkv=8, d=128, kv=BF16), 0),
    ("group1_fp8", dict(lens=[1, 17, 300, 1300], Hq=8, Hkv=8, d=128, kv=FP8), 0),
    ("d64_fp8", dict(lens=[3, 64, 65, 900], Hq=8, Hkv=2, d=64, kv=FP8), 0),
    # forced splits: partials and log-sum-exps through the static array, then the merge
    ("split7", dict(lens=[1, 40, 700, 1500, 2100], Hq=32, Hkv=8, d=128, kv=BF16), 7),
    ("split5_fp8", dict(lens=[2, 90, 1100, 3000], Hq=32, Hkv=8, d=128, kv=FP8), 5),
]


def _problem(name, kw):
    if not kw:
        return W.make_config(name, device="cuda")
    return W.make_problem(kw["lens"], kw["Hq"], kw["Hkv"], kw["d"], seed=900 + len(name), device="cuda",
                          kv_dtype=kw["kv"], tail_fill="nan")


@pytest.mark.parametrize("name,kw,P", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_oracle(name, kw, P):
    fn, cap = _static_scratch_fn()
    assert cap == 32 << 20
    pa.set_max_partitions(P)
    try:
        p = _problem(name, kw)
        fp8 = p.kv_dtype == W.KV_FP8_E4M3
        B = p.num_seqs
        seqs = None if B <= 8 else list(range(0, B, max(1, B // 8)))
        ref = oracle.attention_problem(p, seqs=seqs)
        pick = slice(None) if seqs is None else seqs
        dec = pa.run_problem(p)
        torch.cuda.synchronize()
        pa.check_device_errors()
        for call in range(2):
            out = torch.full_like(p.q, float("nan"))
            assert _call_static(fn, p, out) == pa.PA_OK
            torch.cuda.synchronize()
            assert torch.isfinite(out.float()).all()
            parity.check(_np(out)[pick], ref[pick], fp8, label=f"{_label()} call {call}")
            # the ordinary decode entry on the same inputs (both are within the bar of the oracle)
            tol = 2 * (parity.FP8_MAX if fp8 else parity.BF16_MAX)
            assert (out.float() - dec.float()).abs().max().item() <= tol
        assert pa.check_device_errors() == pa.PA_OK
    finally:
        pa.set_max_partitions(0)


def test_static_scratch_allocates_nothing():
    # a forced split (partials in the array): two calls leave the device's free memory and torch's
    # allocator where they were
    fn, _ = _static_scratch_fn()
    pa.set_max_partitions(6)
    try:
        p = W.make_problem([100, 900, 2500, 4000], 32, 8, 128, seed=990, device="cuda")
        outs = [torch.empty_like(p.q) for _ in range(3)]
        assert _call_static(fn, p, outs[0]) == pa.PA_OK  # first call: per-device set-up
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        alloc0 = torch.cuda.memory_allocated()
        for k in (1, 2):
            assert _call_static(fn, p, outs[k]) == pa.PA_OK
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, (free0, free1)
        assert torch.cuda.memory_allocated() == alloc0
        assert torch.equal(outs[1].view(torch.int16), outs[2].view(torch.int16))
        ref = oracle.attention_problem(p)
        parity.check(_np(outs[2]), ref, False, label=_label())
        assert pa.check_device_errors() == pa.PA_OK
    finally:
        pa.set_max_partitions(0)


def test_static_scratch_rejects_shapes_beyond_its_array():
    fn, cap = _static_scratch_fn()
    pa.set_max_partitions(0)
    p = W.make_config("cb_mix", device="cuda")  # 256 x 32 heads x 16 partitions of partials
    out = torch.zeros_like(p.q)
    assert _call_static(fn, p, out) == pa.PA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched
