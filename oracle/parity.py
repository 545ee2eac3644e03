"""The element-wise bound the CUDA output is held to against the fp64 oracle.

TEST INFRASTRUCTURE ONLY (imported by the GPU tests and ``__graft_entry__.smoke()``); it holds
no attention arithmetic, only the comparison.

Bars (the stated targets for this path): bf16 KV max abs 1e-2 and mean abs 1e-3; fp8 (E4M3) KV
max abs 5e-2.  The output tensor is bf16.  Where the oracle value ``ref`` is large enough that
half a bf16 ulp of it reaches the bar (|ref| >= 4 for 1e-2, |ref| >= 16 for 5e-2), no bf16
value can meet the flat bar, so those elements -- and only those -- are allowed half a bf16 ulp
of their own ``ref`` plus 2e-3 of arithmetic error.  Every other element must be within the
flat bar.  The ulp is taken per element, never from a tensor-wide maximum.

Each check returns (and, when ``PA_PARITY_LOG`` names a file, appends as one JSON line) the
observed worst and mean absolute error, so that the margin under the bar is on record.
"""

from __future__ import annotations

import json
import os

import numpy as np

BF16_MAX = 1e-2
BF16_MEAN = 1e-3
FP8_MAX = 5e-2
RELAXED_EXTRA = 2e-3


def half_ulp_bf16(x):
    """Half the spacing of bf16 values (8 significant bits) around |x|, per element."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 0.5 * np.exp2(np.floor(np.log2(a)) - 7)


def element_bound(ref, fp8: bool):
    """Per-element bound: the flat bar where bf16 can meet it, else half an ulp of ref + 2e-3."""
    bar = FP8_MAX if fp8 else BF16_MAX
    hu = half_ulp_bf16(ref)
    return np.where(hu < bar, bar, hu + RELAXED_EXTRA)


def _log(rec):
    path = os.environ.get("PA_PARITY_LOG")
    if not path:
        return
    try:
        d = os.path.dirname(os.path.abspath(path))
        os.makedirs(d, exist_ok=True)
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    except OSError:
        pass


def check(got, ref, fp8: bool, label: str = "", mean_bar: bool = True):
    """Assert got (any array-like of the bf16 output, as float64) is within the element bound
    of ref everywhere, and (bf16 KV) that the mean abs error is within 1e-3.  Returns
    (max abs error, mean abs error, count of elements that used the relaxed bound)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0, 0.0, 0
    d = np.abs(got - ref)
    bound = element_bound(ref, fp8)
    relaxed = int(np.count_nonzero(bound > (FP8_MAX if fp8 else BF16_MAX)))
    excess = d - bound
    worst = np.unravel_index(int(np.argmax(excess)), excess.shape)
    rec = {"label": label, "kv": "fp8" if fp8 else "bf16", "n": int(d.size),
           "max_abs": float(d.max()), "mean_abs": float(d.mean()),
           "worst_margin": float(-excess.max()), "relaxed_elements": relaxed}
    _log(rec)
    print(f"parity {label}: max {rec['max_abs']:.3e} mean {rec['mean_abs']:.3e} "
          f"margin {rec['worst_margin']:.3e} relaxed {relaxed}/{d.size}")
    assert excess.max() <= 0, ("max abs", float(d[worst]), "at", tuple(int(i) for i in worst),
                               "ref", float(ref[worst]), "bound", float(bound[worst]), label)
    if mean_bar and not fp8:
        assert d.mean() <= BF16_MEAN, ("mean abs", float(d.mean()), label)
    return float(d.max()), float(d.mean()), relaxed
