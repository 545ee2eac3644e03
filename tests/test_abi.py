"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its host-side
checks and planner behave as documented.  No call here reaches a CUDA compute path."""

import ctypes
import os
import re

import pytest

import paged_kv_gqa_attn_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(paged_attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = pa.load_library()
    names = _declared_functions()
    assert "paged_attn_decode" in names and "paged_attn_verify" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    assert pa.status_string(0) == "ok"
    for s in range(1, 8):
        assert pa.status_string(s) != "unknown status"
    assert pa.status_string(99) == "unknown status"
    assert pa.version() >= 100


FAKE = 1 << 20  # a 16-byte aligned non-null address that is never dereferenced


def _decode(**over):
    lib = pa.load_library()
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=2, M=4, NB=8, maxL=64, q_len=1, Hq=8,
             Hkv=2, d=128, bs=16, scale=0.1, dt=0, ks=None, vs=None, out=FAKE, stream=None)
    a.update(over)
    fn = lib.paged_attn_verify if over.pop("verify", False) else lib.paged_attn_decode
    return fn(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["M"], a["NB"], a["maxL"],
              a["q_len"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["scale"], a["dt"], a["ks"], a["vs"],
              a["out"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(q=None), pa.PA_ERR_INVALID_ARG),
    (dict(k=None), pa.PA_ERR_INVALID_ARG),
    (dict(out=None), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), pa.PA_ERR_INVALID_ARG),
    (dict(B=-1), pa.PA_ERR_INVALID_ARG),
    (dict(maxL=65), pa.PA_ERR_INVALID_ARG),
    (dict(q_len=2), pa.PA_ERR_INVALID_ARG),
    (dict(dt=1), pa.PA_ERR_INVALID_ARG),            # fp8 without scales
    (dict(dt=7), pa.PA_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), pa.PA_ERR_INVALID_ARG),      # misaligned pool
    (dict(d=96), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=32, maxL=128), pa.PA_ERR_UNSUPPORTED),
    (dict(Hq=256, Hkv=2), pa.PA_ERR_UNSUPPORTED),   # group 128: beyond 64
])
def test_decode_argument_checks(over, status):
    assert _decode(**over) == status


@pytest.mark.parametrize("over,status", [
    (dict(q_len=17), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=32, Hkv=2, q_len=9), pa.PA_ERR_UNSUPPORTED),  # 144 rows per kv head
    (dict(Hq=32, Hkv=2, q_len=9, dt=1, ks=FAKE, vs=FAKE), pa.PA_ERR_UNSUPPORTED),  # 144 rows, E4M3
    (dict(dt=1, q_len=4), pa.PA_ERR_INVALID_ARG),   # E4M3 without scales
])
def test_verify_argument_checks(over, status):
    over["verify"] = True
    assert _decode(**over) == status


def test_empty_batch_is_a_no_op():
    assert _decode(B=0) == pa.PA_OK


def test_plan_shapes():
    pa.set_max_partitions(0)
    # 64 x 2048-token sequences, 8 kv heads on 152 SMs: 3 partitions of 44 pages (>= 8 CTAs/SM)
    assert pa.plan(152, 64, 8, 2048) == (44, 3)
    # the same with E4M3 pages: one partition per (sequence, kv head) already gives 512 CTAs, 84 %
    # of the 4-per-SM target, so no split (a merge would cost more than the idle slots)
    assert pa.plan(152, 64, 8, 2048, kv_dtype=pa.PA_KV_FP8_E4M3) == (128, 1)
    # 48 sequences: 384 CTAs, 63 % of the target: >= 4 CTAs/SM, 2 partitions of 64 pages
    assert pa.plan(152, 48, 8, 2048, kv_dtype=pa.PA_KV_FP8_E4M3) == (64, 2)
    # 4 x 131072 tokens with E4M3 pages: partitions of at most 256 pages
    assert pa.plan(152, 4, 8, 131072, kv_dtype=pa.PA_KV_FP8_E4M3) == (256, 32)
    # ragged batch up to 8192 tokens: partitions of at most 64 pages
    assert pa.plan(152, 256, 8, 8192) == (64, 8)
    # 4 x 131072 tokens: capped at 64 partitions of 128 pages
    assert pa.plan(152, 4, 8, 131072) == (128, 64)
    # tiny: one partition
    ppp, P = pa.plan(152, 4, 2, 64)
    assert P == 1 and ppp >= 4
    for p in (1, 2, 7, 64):
        pa.set_max_partitions(p)
        ppp, P = pa.plan(152, 64, 8, 2048)
        assert P <= p and ppp * P >= 128 and ppp * (P - 1) < 128
    pa.set_max_partitions(0)
    with pytest.raises(pa.PagedAttnError):
        pa.set_max_partitions(-1)


def test_plan_covers_every_page():
    pa.set_max_partitions(0)
    for maxL in [1, 15, 16, 17, 1000, 4105, 8192, 131072]:
        for B in [1, 16, 256]:
            for dt in (pa.PA_KV_BF16, pa.PA_KV_FP8_E4M3):
                ppp, P = pa.plan(152, B, 8, maxL, kv_dtype=dt)
                pages = (maxL + 15) // 16
                assert ppp * P >= pages and ppp * (P - 1) < pages and 1 <= P <= 64


def _append(**over):
    lib = pa.load_library()
    a = dict(kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, B=2, n=1, M=4, NB=8, Hkv=2, d=128,
             bs=16, dt=0, ks=None, vs=None, stream=None)
    a.update(over)
    return lib.paged_attn_append_kv(a["kn"], a["vn"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["n"],
                                    a["M"], a["NB"], a["Hkv"], a["d"], a["bs"], a["dt"], a["ks"],
                                    a["vs"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(kn=None), pa.PA_ERR_INVALID_ARG),
    (dict(cl=None), pa.PA_ERR_INVALID_ARG),
    (dict(n=-1), pa.PA_ERR_INVALID_ARG),
    (dict(n=65), pa.PA_ERR_INVALID_ARG),          # more than the table holds (4 blocks of 16)
    (dict(kn=FAKE + 8), pa.PA_ERR_INVALID_ARG),   # rows not 16-byte aligned
    (dict(dt=1), pa.PA_ERR_INVALID_ARG),          # fp8 without scales
    (dict(dt=5), pa.PA_ERR_INVALID_ARG),
    (dict(bs=32), pa.PA_ERR_UNSUPPORTED),
    (dict(d=96), pa.PA_ERR_UNSUPPORTED),
    (dict(n=0), pa.PA_OK),                        # nothing to do: no launch
    (dict(B=0), pa.PA_OK),
])
def test_append_argument_checks(over, status):
    assert _append(**over) == status


def _accept(**over):
    lib = pa.load_library()
    a = dict(p=FAKE, q=FAKE, d=FAKE, u=FAKE, w=FAKE, B=2, K=4, V=1000, out=FAKE, n=FAKE, stream=None)
    a.update(over)
    return lib.paged_attn_spec_accept(a["p"], a["q"], a["d"], a["u"], a["w"], a["B"], a["K"], a["V"],
                                      a["out"], a["n"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(p=None), pa.PA_ERR_INVALID_ARG),
    (dict(q=None), pa.PA_ERR_INVALID_ARG),
    (dict(w=None), pa.PA_ERR_INVALID_ARG),
    (dict(out=None), pa.PA_ERR_INVALID_ARG),
    (dict(K=-1), pa.PA_ERR_INVALID_ARG),
    (dict(V=0), pa.PA_ERR_INVALID_ARG),
    (dict(K=32), pa.PA_ERR_UNSUPPORTED),
    (dict(V=(1 << 21) + 1), pa.PA_ERR_UNSUPPORTED),
    (dict(B=0), pa.PA_OK),
])
def test_spec_accept_argument_checks(over, status):
    assert _accept(**over) == status


def test_spec_accept_without_drafts_needs_no_q():
    # K = 0 (plain sampling from p) accepts NULL q / draft / u_accept; B = 0 launches nothing
    assert _accept(K=0, q=None, d=None, u=None, B=0) == pa.PA_OK


def _prefill(**over):
    lib = pa.load_library()
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, qsl=FAKE, B=2, tq=10, mq=8, M=4, NB=8, maxL=64,
             Hq=8, Hkv=2, d=128, bs=16, scale=0.1, dt=0, ks=None, vs=None, out=FAKE, stream=None)
    a.update(over)
    return lib.paged_attn_prefill(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["qsl"], a["B"], a["tq"], a["mq"],
                                  a["M"], a["NB"], a["maxL"], a["Hq"], a["Hkv"], a["d"], a["bs"], a["scale"],
                                  a["dt"], a["ks"], a["vs"], a["out"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(qsl=None), pa.PA_ERR_INVALID_ARG),
    (dict(q=None), pa.PA_ERR_INVALID_ARG),
    (dict(mq=0), pa.PA_ERR_INVALID_ARG),
    (dict(tq=-1), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), pa.PA_ERR_INVALID_ARG),
    (dict(maxL=65), pa.PA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), pa.PA_ERR_INVALID_ARG),
    (dict(dt=1), pa.PA_ERR_INVALID_ARG),              # E4M3 without scales
    (dict(dt=1, ks=FAKE, vs=FAKE, k=FAKE + 8), pa.PA_ERR_INVALID_ARG),  # misaligned E4M3 pool
    (dict(Hq=32, Hkv=2), pa.PA_ERR_UNSUPPORTED),      # group 16: the tile takes groups 1, 2, 4, 8
    (dict(d=96), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=32, maxL=64), pa.PA_ERR_UNSUPPORTED),
    (dict(B=0), pa.PA_OK),
    (dict(tq=0), pa.PA_OK),
])
def test_prefill_argument_checks(over, status):
    assert _prefill(**over) == status


@pytest.mark.parametrize("helper,polls,ptr", [
    (3, 16, FAKE), (-1, 16, FAKE), (0, 0, FAKE), (1, pa.PA_WAIT_LIMIT + 1, FAKE),
    (2, pa.PA_SPIN_LIMIT + 1, FAKE), (0, 16, None), (1, 16, FAKE + 4),
])
def test_selftest_wait_argument_checks(helper, polls, ptr):
    # rejected on the host before any launch
    lib = pa.load_library()
    assert lib.paged_attn_selftest_wait(helper, polls, ptr, None) == pa.PA_ERR_INVALID_ARG


def test_wait_limits_match_the_header():
    text = open(os.path.join(ROOT, "include", "paged_attn.h")).read()
    assert re.search(r"#define PA_WAIT_LIMIT \(1u << (\d+)\)", text).group(1) == str(pa.PA_WAIT_LIMIT.bit_length() - 1)
    assert re.search(r"#define PA_SPIN_LIMIT \(1u << (\d+)\)", text).group(1) == str(pa.PA_SPIN_LIMIT.bit_length() - 1)


def test_binding_rejects_tensors_on_several_devices():
    # checked before any CUDA call: the library launches on the current device only
    import torch
    with pytest.raises(ValueError, match="one CUDA device"):
        pa._one_device(None, a=torch.zeros(1), b=torch.zeros(1, device="meta"))
