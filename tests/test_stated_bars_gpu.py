"""The stated parity bars, measured against the exact (float64) oracle, for the
tiny, small and 0.6B-shape workloads in every precision (the 8B shape is in
test_qwen3_8b_gpu.py).

Bars: per-layer relative L2 <= 2e-3 (float32 path: 1e-5), final-logit max |diff|
<= 5e-2, argmax agreement >= 99.5% (raw: every position counts).  "Per layer"
is measured two ways:
  layer_free    the hidden state entering each layer, GPU pass against oracle pass;
  layer_forced  each layer alone: the exact oracle layer fed the GPU's own input
                to that layer, against the GPU's output of it.
A bar is marked as an expected miss (xfail) exactly where the oracle's own
operand-rounding mode, with the library's rounding points, misses it against
the exact oracle (tests/golden/mode_distance.json, written from the oracle
alone): an implementation that rounds those operands is not expected to meet it
there.  Every other bar is asserted."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import load_model, rel_l2
from parity_record import BARS, bar_holds, expected_miss, load_golden, logit_metrics, record

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")

WORKLOADS = ("tiny", "small", "qwen3-0.6b-shape")
PRECS = ("f32", "tf32", "bf16")
GOLDEN = load_golden()

_cache = {}


def _exact(name):
    if name not in _cache:
        cfg = synth.CONFIGS[name].replace(precision="f32")
        w = synth.model_weights(cfg)
        toks = synth.tokens(cfg)
        xl, xh = oracle.forward(cfg, w, toks, return_hidden=True)
        _cache[name] = (w, toks, xl, xh)
    return _cache[name]


def _measure(dtp, name, prec):
    key = (name, prec)
    if key in _cache:
        return _cache[key]
    w, toks, xl, xh = _exact(name)
    cfg = synth.CONFIGS[name].replace(precision=prec)
    m = load_model(dtp, cfg)
    logits, hidden = m.forward(torch.as_tensor(toks.astype(np.int32), device=dev), hidden=True)
    torch.cuda.synchronize()
    dtp.check()
    gl, gh = logits.cpu().numpy(), hidden.cpu().numpy().astype(np.float64)
    del m, logits, hidden
    pos = np.arange(len(toks))
    free = [rel_l2(gh[l], xh[l]) for l in range(1, cfg.n_layer + 1)]
    forced = [rel_l2(gh[l + 1], oracle.forward_layer(cfg, w["layers"][l], gh[l], pos))
              for l in range(cfg.n_layer)]
    met = {"layer_free": [round(v, 7) for v in free], "layer_forced": [round(v, 7) for v in forced],
           "layer_free_max": max(free), "layer_forced_max": max(forced), **logit_metrics(gl, xl)}
    record(f"stated {name} {prec} T={len(toks)}", met)
    _cache[key] = met
    return met


def _cases():
    out = []
    for name in WORKLOADS:
        for prec in PRECS:
            if prec == "bf16" and synth.CONFIGS[name].head_dim not in (64, 128):
                continue             # the bf16 kernels tile head_dim 64 and 128 only (tiny: 16)
            for bar in BARS:
                why = expected_miss(GOLDEN, name, prec, bar)
                marks = [pytest.mark.xfail(strict=False, reason=why)] if why else []
                out.append(pytest.param(name, prec, bar, marks=marks, id=f"{name}-{prec}-{bar}"))
    return out


@pytest.mark.parametrize("name,prec,bar", _cases())
def test_stated_bar(dtp, name, prec, bar):
    m = _measure(dtp, name, prec)
    assert bar_holds(prec, bar, m), {k: v for k, v in m.items() if not isinstance(v, list)}
