"""GB300 (sm_103a) paged-KV GQA attention: decode and speculative verify.

A thin Python binding over the C ABI in ``include/paged_attn.h``: it checks tensor devices
and dtypes, passes raw device pointers and sizes, and raises on a non-zero status.  All the
arithmetic runs in the library's CUDA kernels; there is no fallback.  PyTorch only provides
device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "PagedAttnError",
    "decode",
    "verify",
    "tree_verify",
    "prefill",
    "append_kv",
    "spec_accept",
    "check_device_errors",
    "set_max_partitions",
    "plan",
    "status_string",
    "version",
    "library_path",
    "load_library",
]

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_NO_MEMORY = 4
PA_ERR_DEVICE_BOUNDS = 5
PA_ERR_DEVICE_TIMEOUT = 6
PA_ERR_SCRATCH_LIMIT = 7
PA_KV_BF16 = 0
PA_KV_FP8_E4M3 = 1
PA_WAIT_LIMIT = 1 << 18   # suspending mbarrier polls before a kernel wait gives up
PA_SPIN_LIMIT = 1 << 22   # non-suspending probe iterations before an issuer loop gives up

_lib = None
_lock = threading.Lock()


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = True, timeline: Optional[bool] = None):
    """Load the in-tree shared library (building it first when it is missing or stale), or return
    the one already loaded.

    timeline=True loads the instrumented variant instead (per-CTA time stamps in the verify
    kernel, for ``paged_kv_gqa_attn_gb300.timeline``); it must be the first load of the process."""
    global _lib
    with _lock:
        if _lib is not None and timeline is not None and timeline != _lib._pa_timeline:
            raise RuntimeError("the other variant of the library is already loaded in this process")
        if _lib is None:
            timeline = bool(timeline)
            path = _build.TIMELINE_LIB_PATH if timeline else _build.LIB_PATH
            if build_if_missing and not _build.up_to_date(timeline):
                _build.build(timeline=timeline)
            if not os.path.exists(path):
                raise RuntimeError(f"paged attention library not built: {path}")
            lib = ctypes.CDLL(path)
            lib._pa_timeline = timeline
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            attn_args = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P, P, P, P]
            for name in ("paged_attn_decode", "paged_attn_verify"):
                fn = getattr(lib, name)
                fn.restype = I
                fn.argtypes = attn_args
            lib.paged_attn_tree_verify.restype = I
            lib.paged_attn_tree_verify.argtypes = attn_args[:5] + [P] + attn_args[5:]
            lib.paged_attn_prefill.restype = I
            lib.paged_attn_prefill.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, P, P, P, P]
            lib.paged_attn_append_kv.restype = I
            lib.paged_attn_append_kv.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P, P]
            lib.paged_attn_spec_accept.restype = I
            lib.paged_attn_spec_accept.argtypes = [P, P, P, P, P, I, I, I, P, P, P]
            lib.paged_attn_check_device_errors.restype = I
            lib.paged_attn_check_device_errors.argtypes = [P]
            lib.paged_attn_selftest_wait.restype = I
            lib.paged_attn_selftest_wait.argtypes = [I, ctypes.c_uint, P, P]
            lib.paged_attn_status_string.restype = ctypes.c_char_p
            lib.paged_attn_status_string.argtypes = [I]
            lib.paged_attn_set_max_partitions.restype = I
            lib.paged_attn_set_max_partitions.argtypes = [I]
            lib.paged_attn_plan.restype = I
            lib.paged_attn_plan.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]
            lib.paged_attn_version.restype = I
            lib.paged_attn_version.argtypes = []
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().paged_attn_status_string(int(status)).decode()


def version() -> int:
    return int(load_library().paged_attn_version())


def set_max_partitions(p: int) -> None:
    """Force at most p split-KV partitions per sequence (0 = automatic, 1 = no split)."""
    st = load_library().paged_attn_set_max_partitions(int(p))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_set_max_partitions")


def plan(num_sms: int, num_seqs: int, num_kv_heads: int, max_context_len: int, block_size: int = 16,
         q_len: int = 1, kv_dtype: int = PA_KV_BF16):
    """(pages_per_partition, max_partitions) the library chooses for this shape."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().paged_attn_plan(num_sms, num_seqs, num_kv_heads, max_context_len, block_size,
                                        q_len, kv_dtype, ctypes.byref(a), ctypes.byref(b))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_plan")
    return a.value, b.value


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def check_device_errors(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the error status of its device."""
    with torch.cuda.device(stream.device if stream is not None else torch.cuda.current_device()):
        return int(load_library().paged_attn_check_device_errors(_stream_handle(stream)))


def selftest_wait(helper: int, polls: int, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Launch the failure-detection self-test: a bounded kernel wait on an mbarrier that never
    completes (helper 0: the decode kernels' wait, 1: the tcgen05 kernels', 2: the
    non-suspending probe loop of the tensor-core issuers), cut off after `polls` polls.  Returns
    a one-element int64 CUDA tensor with the wait's wall time in ns; the timeout shows up as
    PA_ERR_DEVICE_TIMEOUT in check_device_errors()."""
    s = stream if stream is not None else torch.cuda.current_stream()
    elapsed = torch.zeros(1, dtype=torch.int64, device=s.device)
    with torch.cuda.device(s.device):
        st = load_library().paged_attn_selftest_wait(int(helper), int(polls), elapsed.data_ptr(), _stream_handle(s))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_selftest_wait")
    return elapsed


def _one_device(stream, **tensors):
    """Check that every tensor (and the stream, if one is given) is on one CUDA device and return
    a context that makes it the current device for the call: the library launches on the
    current device."""
    devs = {t.device for t in tensors.values() if t is not None}
    if len(devs) != 1:
        where = {k: str(t.device) for k, t in tensors.items() if t is not None}
        raise ValueError(f"tensors must be on one CUDA device, got {where}")
    dev = devs.pop()
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, tensors on {dev}")
    return torch.cuda.device(dev)


def _check_cuda(name, t, dtypes):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _call(fn_name, q, k_cache, v_cache, block_table, context_lens, scale, *, k_scale=None,
          v_scale=None, max_context_len=None, out=None, stream=None, tree_mask=None):
    lib = load_library()
    _check_cuda("q", q, (torch.bfloat16,))
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    kv_dtypes = (torch.uint8, torch.float8_e4m3fn) if fp8 else (torch.bfloat16,)
    _check_cuda("k_cache", k_cache, kv_dtypes)
    _check_cuda("v_cache", v_cache, kv_dtypes)
    _check_cuda("block_table", block_table, (torch.int32,))
    _check_cuda("context_lens", context_lens, (torch.int32,))
    if fp8:
        _check_cuda("k_scale", k_scale, (torch.float32,))
        _check_cuda("v_scale", v_scale, (torch.float32,))
    if q.dim() != 4 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape or block_table.dim() != 2:
        raise ValueError("expected q [B, q_len, Hq, d], caches [NB, Hkv, bs, d], block_table [B, M]")
    B, q_len, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if d2 != d or block_table.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("shape mismatch between q, caches, block_table and context_lens")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_cuda("out", out, (torch.bfloat16,))
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    max_blocks = int(block_table.shape[1])
    if max_context_len is None:
        max_context_len = max_blocks * bs  # an upper bound known without reading the device
    lead = [q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
            context_lens.data_ptr()]
    if fn_name == "paged_attn_tree_verify":
        _check_cuda("tree_mask", tree_mask, (torch.int32,))
        if tree_mask.shape != (B, q_len):
            raise ValueError("tree_mask must be [B, q_len]")
        lead.append(tree_mask.data_ptr())
    with _one_device(stream, q=q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     context_lens=context_lens, tree_mask=tree_mask, out=out,
                     k_scale=k_scale if fp8 else None, v_scale=v_scale if fp8 else None):
        st = getattr(lib, fn_name)(
            *lead, B, max_blocks, NB, int(max_context_len), q_len, Hq, Hkv, d, bs,
            float(scale), PA_KV_FP8_E4M3 if fp8 else PA_KV_BF16,
            k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None, out.data_ptr(),
            _stream_handle(stream))
    if st != PA_OK:
        raise PagedAttnError(st, fn_name)
    return out


def decode(q, k_cache, v_cache, block_table, context_lens, scale, **kw):
    """Single-token paged GQA decode; q [B, 1, Hq, d] bf16.  See paged_attn_decode."""
    return _call("paged_attn_decode", q, k_cache, v_cache, block_table, context_lens, scale, **kw)


def verify(q, k_cache, v_cache, block_table, context_lens, scale, **kw):
    """(K+1)-row causal speculative-verify attention; q [B, K+1, Hq, d] bf16.  See paged_attn_verify."""
    return _call("paged_attn_verify", q, k_cache, v_cache, block_table, context_lens, scale, **kw)


def tree_verify(q, k_cache, v_cache, block_table, context_lens, tree_mask, scale, **kw):
    """Verify over a tree of drafts: tree_mask int32 [B, q_len] ancestor bitmasks over the new
    tokens (bit t of row i: row i sees new token t).  See paged_attn_tree_verify."""
    return _call("paged_attn_tree_verify", q, k_cache, v_cache, block_table, context_lens, scale,
                 tree_mask=tree_mask, **kw)


def prefill(q, k_cache, v_cache, block_table, context_lens, query_start_loc, scale, *,
            max_q_len=None, max_context_len=None, out=None, stream=None, k_scale=None, v_scale=None):
    """Paged attention over packed variable-length query rows (chunked prefill, with decode or
    verify rows alongside): q [total_q, Hq, d] bf16, query_start_loc [B+1] int32 (device); caches
    bf16, or E4M3 bytes (uint8 / float8_e4m3fn) with k_scale / v_scale [NB, Hkv] fp32.
    max_q_len must bound every sequence's rows; by default it is read from query_start_loc
    (one device-to-host copy).  See paged_attn_prefill."""
    lib = load_library()
    _check_cuda("q", q, (torch.bfloat16,))
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    kv_dtypes = (torch.uint8, torch.float8_e4m3fn) if fp8 else (torch.bfloat16,)
    _check_cuda("k_cache", k_cache, kv_dtypes)
    _check_cuda("v_cache", v_cache, kv_dtypes)
    if fp8:
        _check_cuda("k_scale", k_scale, (torch.float32,))
        _check_cuda("v_scale", v_scale, (torch.float32,))
    _check_cuda("block_table", block_table, (torch.int32,))
    _check_cuda("context_lens", context_lens, (torch.int32,))
    _check_cuda("query_start_loc", query_start_loc, (torch.int32,))
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape or block_table.dim() != 2:
        raise ValueError("expected q [total_q, Hq, d], caches [NB, Hkv, bs, d], block_table [B, M]")
    total_q, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_cache.shape
    B = int(block_table.shape[0])
    if d2 != d or context_lens.shape != (B,) or query_start_loc.shape != (B + 1,):
        raise ValueError("shape mismatch between q, caches, block_table, context_lens, query_start_loc")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_cuda("out", out, (torch.bfloat16,))
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if max_q_len is None:
        qsl = query_start_loc.cpu()
        max_q_len = int((qsl[1:] - qsl[:-1]).max()) if B else 1
    max_blocks = int(block_table.shape[1])
    if max_context_len is None:
        max_context_len = max_blocks * bs
    with _one_device(stream, q=q, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                     context_lens=context_lens, query_start_loc=query_start_loc, out=out,
                     k_scale=k_scale if fp8 else None, v_scale=v_scale if fp8 else None):
        st = lib.paged_attn_prefill(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
            context_lens.data_ptr(), query_start_loc.data_ptr(), B, total_q, max(1, int(max_q_len)),
            max_blocks, NB, int(max_context_len), Hq, Hkv, d, bs, float(scale),
            PA_KV_FP8_E4M3 if fp8 else PA_KV_BF16, k_scale.data_ptr() if fp8 else None,
            v_scale.data_ptr() if fp8 else None, out.data_ptr(), _stream_handle(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_prefill")
    return out


def append_kv(k_new, v_new, k_cache, v_cache, block_table, context_lens, *, k_scale=None,
              v_scale=None, stream=None):
    """Store the new tokens' K/V [B, n_new, Hkv, d] bf16 in the paged cache, in place (and, for an
    fp8 cache, update the per-(block, head) scales).  context_lens holds the lengths after the
    append.  See paged_attn_append_kv."""
    lib = load_library()
    _check_cuda("k_new", k_new, (torch.bfloat16,))
    _check_cuda("v_new", v_new, (torch.bfloat16,))
    fp8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    kv_dtypes = (torch.uint8, torch.float8_e4m3fn) if fp8 else (torch.bfloat16,)
    _check_cuda("k_cache", k_cache, kv_dtypes)
    _check_cuda("v_cache", v_cache, kv_dtypes)
    _check_cuda("block_table", block_table, (torch.int32,))
    _check_cuda("context_lens", context_lens, (torch.int32,))
    if fp8:
        _check_cuda("k_scale", k_scale, (torch.float32,))
        _check_cuda("v_scale", v_scale, (torch.float32,))
    if k_new.dim() != 4 or k_new.shape != v_new.shape or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("expected k_new/v_new [B, n_new, Hkv, d] and caches [NB, Hkv, bs, d]")
    B, n_new, Hkv, d = k_new.shape
    NB, Hkv2, bs, d2 = k_cache.shape
    if (Hkv2, d2) != (Hkv, d) or block_table.dim() != 2 or block_table.shape[0] != B \
            or context_lens.shape != (B,):
        raise ValueError("shape mismatch between new rows, caches, block_table and context_lens")
    if fp8 and (k_scale.shape != (NB, Hkv) or v_scale.shape != (NB, Hkv)):
        raise ValueError("k_scale / v_scale must be [num_blocks, num_kv_heads]")
    with _one_device(stream, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                     block_table=block_table, context_lens=context_lens,
                     k_scale=k_scale if fp8 else None, v_scale=v_scale if fp8 else None):
        st = lib.paged_attn_append_kv(
            k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            block_table.data_ptr(), context_lens.data_ptr(), B, n_new, int(block_table.shape[1]), NB,
            Hkv, d, bs, PA_KV_FP8_E4M3 if fp8 else PA_KV_BF16,
            k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None,
            _stream_handle(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_append_kv")


def spec_accept(p, q, draft_tokens, u_accept, u_sample, *, out_tokens=None, num_accepted=None,
                stream=None):
    """Speculative acceptance for a batch of rounds: p [B, K+1, V] and q [B, K, V] fp32
    probabilities, draft_tokens [B, K] int32, u_accept [B, K] fp32 uniforms, u_sample [B] int32
    (uint32 bit patterns).  Returns (num_accepted [B] int32, out_tokens [B, K+1] int32).  See
    paged_attn_spec_accept."""
    lib = load_library()
    _check_cuda("p", p, (torch.float32,))
    _check_cuda("u_sample", u_sample, (torch.int32,))
    if p.dim() != 3:
        raise ValueError("p must be [B, K+1, V]")
    B, K1, V = p.shape
    K = K1 - 1
    if K > 0:
        _check_cuda("q", q, (torch.float32,))
        _check_cuda("draft_tokens", draft_tokens, (torch.int32,))
        _check_cuda("u_accept", u_accept, (torch.float32,))
        if q.shape != (B, K, V) or draft_tokens.shape != (B, K) or u_accept.shape != (B, K):
            raise ValueError("q [B, K, V], draft_tokens [B, K] and u_accept [B, K] must match p")
    if u_sample.shape != (B,):
        raise ValueError("u_sample must be [B]")
    if out_tokens is None:
        out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=p.device)
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    _check_cuda("out_tokens", out_tokens, (torch.int32,))
    _check_cuda("num_accepted", num_accepted, (torch.int32,))
    if out_tokens.shape != (B, K + 1) or num_accepted.shape != (B,):
        raise ValueError("out_tokens must be [B, K+1] and num_accepted [B]")
    ptr = (lambda t: t.data_ptr() if K > 0 else None)
    with _one_device(stream, p=p, u_sample=u_sample, out_tokens=out_tokens, num_accepted=num_accepted,
                     q=q if K > 0 else None, draft_tokens=draft_tokens if K > 0 else None,
                     u_accept=u_accept if K > 0 else None):
        st = lib.paged_attn_spec_accept(p.data_ptr(), ptr(q), ptr(draft_tokens), ptr(u_accept),
                                        u_sample.data_ptr(), B, K, V, out_tokens.data_ptr(),
                                        num_accepted.data_ptr(), _stream_handle(stream))
    if st != PA_OK:
        raise PagedAttnError(st, "paged_attn_spec_accept")
    return num_accepted, out_tokens


def run_problem(p, out=None, stream=None, max_context_len=None):
    """Run decode (q_len 1) or verify on a workloads.PagedAttnProblem whose tensors are on the GPU."""
    fn = decode if p.q_len == 1 else verify
    return fn(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, p.scale,
              k_scale=p.k_scale, v_scale=p.v_scale, out=out, stream=stream,
              max_context_len=max_context_len)
