"""Parity measurements shared by the stated-bar tests: GPU pass against the
exact (float64) oracle, free-running and layer by layer, and an optional log of
every measured value (one JSON object per line, to $DTP_PARITY_LOG)."""
from __future__ import annotations

import json
import os

import numpy as np

from helpers import rel_l2

STATED = {"layer": 2e-3, "logit_max_abs": 5e-2, "argmax_raw": 0.995}
STATED_F32_LAYER = 1e-5


def record(tag: str, metrics: dict) -> None:
    path = os.environ.get("DTP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"tag": tag, **metrics}) + "\n")


def logit_metrics(gl, xl) -> dict:
    gl = np.asarray(gl, np.float64)
    xl = np.asarray(xl, np.float64)
    return {"logit_rel_l2": rel_l2(gl, xl), "logit_max_abs": float(np.max(np.abs(gl - xl))),
            "argmax_raw": float(np.mean(np.argmax(gl, 1) == np.argmax(xl, 1)))}


def bar_holds(prec: str, bar: str, m: dict) -> bool:
    """Whether measured metrics `m` meet stated bar `bar` for precision `prec`:
    layer_free / layer_forced <= 2e-3 (float32 path: 1e-5), logit max |diff|
    <= 5e-2, raw argmax agreement >= 99.5%."""
    lim = STATED_F32_LAYER if prec == "f32" else STATED["layer"]
    if bar == "layer_free":
        return m["layer_free_max"] <= lim
    if bar == "layer_forced":
        return m["layer_forced_max"] <= lim
    if bar == "logit_max_abs":
        return m["logit_max_abs"] <= STATED["logit_max_abs"]
    if bar == "argmax_raw":
        return m["argmax_raw"] >= STATED["argmax_raw"]
    raise KeyError(bar)


BARS = ("layer_free", "layer_forced", "logit_max_abs", "argmax_raw")


GOLDEN_MODE = {"bf16": "bf16_fused", "tf32": "tf32"}     # the library's rounding points


def expected_miss(golden: dict, workload: str, prec: str, bar: str):
    """Why the GPU is expected to miss `bar` on `workload` in `prec`, or None:
    the oracle's own rounding mode (the library's rounding points) already
    misses it against the exact oracle.  The float32 path has no such entry."""
    w = golden["workloads"].get(workload)
    mode = GOLDEN_MODE.get(prec)
    if w is None or mode is None:
        return None
    g = w["modes"][mode]
    m = {"layer_free_max": g["free_max"], "layer_forced_max": g["forced_max"],
         "logit_max_abs": g["logit_max_abs"], "argmax_raw": g["argmax_agreement"]}
    if bar_holds(prec, bar, m):
        return None
    key = {"layer_free": "layer_free_max", "layer_forced": "layer_forced_max"}.get(bar, bar)
    return (f"the oracle's {mode} mode itself gives {key} = {m[key]:.3g} against the exact "
            f"oracle on {workload} (tests/golden/mode_distance.json)")


def load_golden() -> dict:
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "mode_distance.json")
    with open(path) as f:
        return json.load(f)
