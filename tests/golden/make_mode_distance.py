"""Writes mode_distance.json: how far each operand-rounding mode of the oracle
lands from the oracle's exact (float64) pass, on the seeded model workloads.
It calls only the oracle and the seeded input generator; no GPU result enters.

For every workload and mode it records, against the exact pass:
  free   the hidden state entering each layer l = 1..L (and the logits) when the
         mode runs the whole pass on its own -- relative L2 per layer;
  forced each layer alone: the mode's layer l fed the exact pass's input to
         layer l, against the exact layer l -- relative L2 per layer;
  logits relative L2, max |diff| and the share of rows whose argmax agrees.
Modes: bf16 (plain: h = bf16(rms_norm(x) * w)), bf16_fused (the norm as a
row scale after bf16(x) bf16(W * w)), tf32.  The 8B shape is run on the first
256 tokens (rows 0..255 of a causal pass depend on those tokens only).

    python tests/golden/make_mode_distance.py [workload ...]   # default: all;
    each workload's entry is replaced in the existing file as soon as it is done
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

MODES = {"bf16": dict(bf16_operands=True),
         "bf16_fused": dict(bf16_operands=True, bf16_fused_norm=True),
         "tf32": dict(tf32_operands=True)}
WORKLOADS = (("tiny", None), ("small", None), ("qwen3-0.6b-shape", None), ("qwen3-8b-shape", 256))


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def run(name, R, mode):
    """One workload in one mode: the exact pass and the mode's pass side by side,
    layer by layer (each layer's weights drawn once, in float64)."""
    cfg = synth.CONFIGS[name]
    kw = MODES[mode]
    T = cfg.T if R is None else R
    toks = synth.tokens(cfg)[:T]
    emb = synth.tok_embd(cfg)
    x_exact = emb[toks].astype(np.float64)
    x_mode = oracle.round_bf16(x_exact) if mode.startswith("bf16") else x_exact.copy()
    del emb
    pos = np.arange(T)
    free, forced = [], []
    for l in range(cfg.n_layer):
        lw = {k: v.astype(np.float64) for k, v in synth.layer_weights(cfg, l).items()}
        nxt = oracle.forward_layer(cfg, lw, x_exact, pos)
        x_mode = oracle.forward_layer(cfg, lw, x_mode, pos, **kw)
        free.append(rel(x_mode, nxt))
        forced.append(rel(oracle.forward_layer(cfg, lw, x_exact, pos, **kw), nxt))
        x_exact = nxt
        print(name, mode, l + 1, f"{free[-1]:.2e} {forced[-1]:.2e}", flush=True)
    onorm, W = synth.output_norm(cfg), synth.output_weight(cfg)
    rnd = oracle.round_tf32 if mode == "tf32" else oracle.round_bf16

    def logits(x, r):
        hn = r(oracle.rms_norm(x, onorm, cfg.rms_eps))
        return np.concatenate([oracle.linear(hn, r(W[v0:v0 + 16384]))
                               for v0 in range(0, cfg.n_vocab, 16384)], axis=1)

    ex = logits(x_exact, lambda a: a)
    lg = logits(x_mode, rnd)
    top = np.sort(ex, axis=1)[:, -2:]
    return {"T": T, "n_layer": cfg.n_layer,
            "min_top1_top2_margin": float((top[:, 1] - top[:, 0]).min()),
            "free": [round(v, 7) for v in free], "forced": [round(v, 7) for v in forced],
            "free_max": max(free), "forced_max": max(forced),
            "logit_rel_l2": rel(lg, ex), "logit_max_abs": float(np.abs(lg - ex).max()),
            "argmax_agreement": float(np.mean(np.argmax(lg, 1) == np.argmax(ex, 1)))}


def _task(args):
    name, R, mode = args
    t0 = time.time()
    out = run(name, R, mode)
    out["seconds"] = round(time.time() - t0, 1)
    return name, mode, out


def main(names):
    import multiprocessing as mp

    path = os.path.join(HERE, "mode_distance.json")
    doc = json.load(open(path)) if os.path.exists(path) else {"workloads": {}}
    doc["source"] = (__doc__.strip().split("\n\n")[0].replace("\n", " ")
                     + " Written by tests/golden/make_mode_distance.py.")
    tasks = [(name, R, mode) for name, R in WORKLOADS if not names or name in names
             for mode in MODES]
    # one process per (workload, mode); BLAS threads shared out among them
    os.environ.setdefault("OMP_NUM_THREADS", str(max(1, (os.cpu_count() or 1) // len(MODES))))
    with mp.get_context("spawn").Pool(min(len(tasks), 2 * len(MODES))) as pool:
        for name, mode, out in pool.imap_unordered(_task, tasks):
            w = doc["workloads"].setdefault(name, {"modes": {}})
            w["T"], w["n_layer"] = out["T"], out["n_layer"]
            w["min_top1_top2_margin"] = out.pop("min_top1_top2_margin")
            w["modes"][mode] = out
            json.dump(doc, open(path, "w"), indent=1)


if __name__ == "__main__":
    main(sys.argv[1:])
