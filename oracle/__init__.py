"""fp64 CPU oracle for paged GQA attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers.  The product path (the CUDA library and its binding) never
imports this package, and this package never imports the product path.

The arithmetic lives in ``paged_attn_oracle.c`` (plain C, double precision, OpenMP over
(sequence, query row, query head)); this module compiles it with gcc and marshals numpy
arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double: no -ffast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.pa_oracle_attention.restype = I
            lib.pa_oracle_attention.argtypes = [
                P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, I, ctypes.c_double, P, I, P, I]
            lib.pa_oracle_attention_masked.restype = I
            lib.pa_oracle_attention_masked.argtypes = [
                P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, ctypes.c_double, P, I, P, I]
            lib.pa_oracle_bf16_to_double.restype = ctypes.c_double
            lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.pa_oracle_e4m3_to_double.restype = ctypes.c_double
            lib.pa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.pa_oracle_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().pa_oracle_max_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().pa_oracle_bf16_to_double(int(bits)))


def e4m3_to_double(byte: int) -> float:
    return float(_load().pa_oracle_e4m3_to_double(int(byte)))


def _np(t, dtype):
    """torch tensor or numpy array -> C-contiguous numpy array of `dtype` (bit-preserving)."""
    try:
        import torch

        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def attention(q, k_cache, v_cache, block_table, context_lens, *, q_len, num_q_heads,
              num_kv_heads, head_dim, block_size, scale, kv_fp8=False, k_scale=None,
              v_scale=None, seqs=None, num_threads=0, tree_mask=None):
    """fp64 paged attention.  Returns out[B, q_len, Hq, d] (float64).

    q: bf16 bits [B, q_len, Hq, d]; caches bf16 bits or E4M3 bytes [NB, Hkv, bs, d];
    scales fp32 [NB, Hkv] for fp8; seqs: optional list of sequence indices to compute (the
    other rows of the result are left at 0); tree_mask: optional uint32 [B, q_len] ancestor
    bitmasks over the q_len new tokens (None = causal).
    """
    lib = _load()
    qa = _np(q, np.uint16)
    kc = _np(k_cache, np.uint8 if kv_fp8 else np.uint16)
    vc = _np(v_cache, np.uint8 if kv_fp8 else np.uint16)
    bt = _np(block_table, np.int32)
    cl = _np(context_lens, np.int32)
    B = int(qa.shape[0])
    nb = int(kc.shape[0])
    ks = _np(k_scale, np.float32) if kv_fp8 else None
    vs = _np(v_scale, np.float32) if kv_fp8 else None
    out = np.zeros((B, q_len, num_q_heads, head_dim), dtype=np.float64)
    sel = None if seqs is None else np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
    tm = None if tree_mask is None else _np(tree_mask, np.uint32)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.pa_oracle_attention_masked(
        ptr(qa), ptr(kc), ptr(vc), ptr(ks), ptr(vs), int(bool(kv_fp8)), ptr(bt), ptr(cl), ptr(tm),
        B, int(bt.shape[1]), nb, int(q_len), int(num_q_heads), int(num_kv_heads), int(head_dim),
        int(block_size), float(scale), ptr(sel), 0 if sel is None else int(sel.size), ptr(out),
        int(num_threads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out


def attention_problem(p, seqs=None, num_threads=0, tree_mask=None):
    """Run the oracle on a workloads.PagedAttnProblem (tensors may live on any device)."""
    return attention(
        p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, q_len=p.q_len,
        num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
        block_size=p.block_size, scale=p.scale, kv_fp8=(p.kv_dtype == "fp8_e4m3"),
        k_scale=p.k_scale, v_scale=p.v_scale, seqs=seqs, num_threads=num_threads,
        tree_mask=tree_mask)


def attention_varlen(q, k_cache, v_cache, block_table, context_lens, query_start_loc, *,
                     num_q_heads, num_kv_heads, head_dim, block_size, scale, rows=None,
                     num_threads=0, kv_fp8=False, k_scale=None, v_scale=None):
    """fp64 paged attention over packed query rows: sequence b's q_len_b new rows are
    q[qsl[b]:qsl[b+1]] ([total_q, Hq, d] bf16 bits), and its row i sees the first
    context_lens[b] - q_len_b + i + 1 cached tokens.  Each row is therefore the one-row case of
    `attention` over that many tokens, which is how it is computed here (E4M3 caches: decoded
    with their per-(block, kv head) scales, as there).  rows: optional list of packed row indices
    to compute (others stay 0).  Returns [total_q, Hq, d] float64."""
    qa = _np(q, np.uint16)
    qsl = _np(query_start_loc, np.int32)
    cl = _np(context_lens, np.int32)
    bt = _np(block_table, np.int32)
    total_q = int(qa.shape[0])
    seq_of = np.zeros(total_q, dtype=np.int64)
    for b in range(len(qsl) - 1):
        seq_of[qsl[b]:qsl[b + 1]] = b
    sel = np.arange(total_q) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((total_q, num_q_heads, head_dim), dtype=np.float64)
    if sel.size == 0:
        return out
    b_of = seq_of[sel]
    i_of = sel - qsl[b_of]
    ql_of = qsl[b_of + 1] - qsl[b_of]
    n_of = (cl[b_of] - ql_of + i_of + 1).astype(np.int32)
    res = attention(qa[sel][:, None], k_cache, v_cache, bt[b_of], np.maximum(n_of, 0), q_len=1,
                    num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                    block_size=block_size, scale=scale, num_threads=num_threads, kv_fp8=kv_fp8,
                    k_scale=k_scale, v_scale=v_scale)
    out[sel] = res[:, 0]
    return out


def attention_varlen_problem(p, rows=None, num_threads=0):
    """attention_varlen on a workloads.VarlenProblem."""
    return attention_varlen(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                            p.query_start_loc, num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads,
                            head_dim=p.head_dim, block_size=p.block_size, scale=p.scale, rows=rows,
                            num_threads=num_threads, kv_fp8=(p.kv_dtype == "fp8_e4m3"),
                            k_scale=p.k_scale, v_scale=p.v_scale)
