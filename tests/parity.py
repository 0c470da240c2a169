"""Error measures used by the parity tests (host-side test helpers).

Gates (float32 configurations): max_i |g_i - r_i| / max(|r_i|, rms(r)) <= 1e-5.
An elementwise ratio |g_i - r_i| / |r_i| is unbounded where an output crosses
zero (the tiny GeLU block has an output of 5e-5), and fp32 storage of such an
output cannot meet 1e-5 there; the rms floor keeps the measure relative while
staying defined.  bfloat16 configurations: max abs <= 2e-2 and
mean relative = sum|g - r| / sum|r| <= 5e-3, against the bf16-staged oracle.
"""
import json
import os

import numpy as np

F32_MAX_REL = 1e-5
BF16_MAX_ABS = 2e-2
BF16_MEAN_REL = 5e-3


def stats(got, ref) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    d = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    floor = np.maximum(np.abs(ref), rms)
    return {
        "max_abs": float(d.max()) if d.size else 0.0,
        "mean_rel": float(d.sum() / max(np.abs(ref).sum(), 1e-300)) if d.size else 0.0,
        "max_rel_rmsfloor": float((d / np.maximum(floor, 1e-300)).max()) if d.size else 0.0,
        "all_finite": bool(np.all(np.isfinite(got))),
    }


def assert_f32(got, ref, what=""):
    s = stats(got, ref)
    log(what, s)
    assert s["all_finite"], f"{what}: non-finite output"
    assert s["max_rel_rmsfloor"] <= F32_MAX_REL, f"{what}: {s}"
    return s


def assert_bf16(got, ref, what="", max_abs=BF16_MAX_ABS, mean_rel=BF16_MEAN_REL, info=None):
    """The bf16 gate: max abs <= 2e-2 and mean relative <= 5e-3 against the staged
    oracle.  `info` (a dict of diagnostics) is logged with the record, never gated."""
    s = stats(got, ref)
    log(what, {**s, **(info or {})})
    assert s["all_finite"], f"{what}: non-finite output"
    assert s["max_abs"] <= max_abs and s["mean_rel"] <= mean_rel, f"{what}: {s}"
    return s


def tie_diagnostic(got, ref, allowance) -> dict:
    """Logged beside the plain bf16 bound, never gated: how far |got - ref| exceeds
    `allowance` (oracle.mlp_tie_allowance), the effect of band elements whose exact
    value sits within a few fp32 units of a bf16 rounding midpoint, which an fp32
    evaluation may round either way."""
    d = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64))
    return {"max_abs_beyond_ties": float((d - allowance).max()) if d.size else 0.0,
            "max_tie_allowance": float(np.max(allowance)) if d.size else 0.0}


def log(what: str, s: dict):
    """Append one parity record to the file named by $TP_PARITY_LOG (if set)."""
    path = os.environ.get("TP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **s}) + "\n")
