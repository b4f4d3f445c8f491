"""The 8B shape (36 layers, d = 4096, T = 4096, V = 151936) in the launch
configuration the benchmark times.

Causality makes rows 0..R-1 of the pass depend on the first R tokens only, so
the oracle runs the whole 36-layer model on the R-token prefix (streamed layer
by layer) and the GPU's hidden rows and logits of those rows are compared:
  * bf16 kernels against the oracle with the kernels' rounding points: the
    derived bounds of test_forward_gpu.py, free-running and layer by layer;
  * every precision against the exact oracle: the stated bars, as in
    test_stated_bars_gpu.py (expected misses are where the oracle's own
    rounding mode misses the bar, tests/golden/mode_distance.json);
  * long-range attention inside the pass: for layers 0, 17 and 35 the oracle's
    layer is fed the GPU's whole 4096-row input and compared on rows spread
    over the sequence up to T-1, where each query attends to thousands of keys.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import argmax_agreement_near_tie, rel_l2
from parity_record import BARS, bar_holds, expected_miss, load_golden, logit_metrics, record

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")

CFG = synth.CONFIGS["qwen3-8b-shape"]
R = 256
LONG_LAYERS = (0, 17, 35)
LONG_ROWS = np.unique(np.concatenate([np.linspace(0, CFG.T - 1, 24).astype(int),
                                      [3968, 4000, 4031, 4032, 4063, 4064, 4094, 4095]]))

GOLDEN = load_golden()


def _gpu_pass(dtp, prec, keep_layers=()):
    cfg = CFG.replace(precision=prec)
    m = dtp.Model(cfg)
    for l in range(cfg.n_layer):
        m.load_layer(l, synth.layer_weights(cfg, l))
    m.load_globals(synth.tok_embd(cfg), synth.output_norm(cfg), synth.output_weight(cfg))
    toks = synth.tokens(cfg)
    logits, hidden = m.forward(torch.as_tensor(toks.astype(np.int32), device=dev), hidden=True)
    torch.cuda.synchronize()
    dtp.check()
    out = {"hidden": hidden[:, :R].cpu().numpy().astype(np.float64),
           "logits": logits[:R].cpu().numpy(),
           "full": {l: hidden[l].cpu().numpy() for l in keep_layers}}
    del m, logits, hidden
    gc.collect()
    torch.cuda.empty_cache()
    return out


@pytest.fixture(scope="module")
def run8b(dtp):
    runs = {"bf16": _gpu_pass(dtp, "bf16", keep_layers=sorted({l for k in LONG_LAYERS
                                                                for l in (k, k + 1)})),
            "tf32": _gpu_pass(dtp, "tf32"), "f32": _gpu_pass(dtp, "f32")}
    toks = synth.tokens(CFG)
    emb = synth.tok_embd(CFG)
    x_ex = emb[toks[:R]].astype(np.float64)
    x_bf = oracle.round_bf16(x_ex)
    del emb
    pos = np.arange(R)
    res = {"exact_hidden": [x_ex], "fused_hidden": [x_bf], "fused_forced": [],
           "forced": {p: [] for p in runs}, "long": {}}
    for l in range(CFG.n_layer):
        # float64 once, so the exact-mode calls below convert nothing
        lw = {k: v.astype(np.float64) for k, v in synth.layer_weights(CFG, l).items()}
        x_ex = oracle.forward_layer(CFG, lw, x_ex, pos)
        res["exact_hidden"].append(x_ex)
        x_bf = oracle.forward_layer(CFG, lw, x_bf, pos, bf16_operands=True, bf16_fused_norm=True)
        res["fused_hidden"].append(x_bf)
        gb = runs["bf16"]["hidden"]
        res["fused_forced"].append(rel_l2(gb[l + 1], oracle.forward_layer(
            CFG, lw, gb[l], pos, bf16_operands=True, bf16_fused_norm=True)))
        for p in ("f32", "tf32"):
            g = runs[p]["hidden"]
            res["forced"][p].append(rel_l2(g[l + 1], oracle.forward_layer(CFG, lw, g[l], pos)))
        res["forced"]["bf16"].append(rel_l2(gb[l + 1], oracle.forward_layer(CFG, lw, gb[l], pos)))
        if l in LONG_LAYERS:
            full = runs["bf16"]["full"]
            ref = oracle.forward_layer(CFG, lw, full[l].astype(np.float64), np.arange(CFG.T),
                                       bf16_operands=True, bf16_fused_norm=True, rows=LONG_ROWS)
            got = full[l + 1][LONG_ROWS].astype(np.float64)
            res["long"][l] = [rel_l2(got[i], ref[i]) for i in range(len(LONG_ROWS))]
        del lw
    onorm, W = synth.output_norm(CFG), synth.output_weight(CFG)

    def head(x, rnd):
        hn = rnd(oracle.rms_norm(x, onorm, CFG.rms_eps))
        return np.concatenate([oracle.linear(hn, rnd(W[v0:v0 + 16384]))
                               for v0 in range(0, CFG.n_vocab, 16384)], axis=1)

    res["exact_logits"] = head(x_ex, lambda a: a)
    res["fused_logits"] = head(x_bf, oracle.round_bf16)
    del W
    res["runs"] = runs
    return res


def _stated_metrics(res, prec):
    g = res["runs"][prec]
    free = [rel_l2(g["hidden"][l], res["exact_hidden"][l]) for l in range(1, CFG.n_layer + 1)]
    forced = res["forced"][prec]
    m = {"layer_free": [round(v, 7) for v in free], "layer_forced": [round(v, 7) for v in forced],
         "layer_free_max": max(free), "layer_forced_max": max(forced),
         **logit_metrics(g["logits"], res["exact_logits"])}
    return m


def test_bf16_kernels_against_the_same_rounding_points(run8b):
    """Free-running: hidden state entering layer l within 2u sqrt(l), logits
    within 2u sqrt(L+1) + u, near-tie-adjusted argmax >= 99.5% (u = 2^-8).
    Layer by layer: each layer within 2u of the oracle's layer on the GPU's
    own input (one layer's rounding differences, no accumulation)."""
    u = 2.0 ** -8
    g = run8b["runs"]["bf16"]
    rh = run8b["fused_hidden"]
    layer_err = [rel_l2(g["hidden"][l], rh[l]) for l in range(CFG.n_layer + 1)]
    assert layer_err[0] == 0.0
    for l in range(1, CFG.n_layer + 1):
        assert layer_err[l] <= 2 * u * np.sqrt(l), (l, layer_err)
    lrel = rel_l2(g["logits"], run8b["fused_logits"])
    assert lrel <= 2 * u * np.sqrt(CFG.n_layer + 1) + u, lrel
    lmax = float(np.max(np.abs(g["logits"] - run8b["fused_logits"])))
    agree, structured = argmax_agreement_near_tie(g["logits"], run8b["fused_logits"], 2 * lmax)
    forced = run8b["fused_forced"]
    record("8b bf16 vs fused-rounding oracle", {
        "layer_rel_l2": [round(e, 7) for e in layer_err], "logit_rel_l2": lrel,
        "logit_max_abs": lmax, "argmax_near_tie": agree, "forced": [round(e, 7) for e in forced]})
    assert structured == 0 and agree >= 0.995
    assert max(forced) <= 2 * u, forced


def test_long_range_attention_rows(run8b):
    """Layers 0, 17, 35 on the GPU's own 4096-row input, rows up to T-1: one
    layer's bf16 rounding differences (2u, u = 2^-8) at every sampled row."""
    worst = {l: max(v) for l, v in run8b["long"].items()}
    record("8b long-range rows", {"rows": LONG_ROWS.tolist(),
                                  "per_layer_max": {str(k): v for k, v in worst.items()}})
    assert set(run8b["long"]) == set(LONG_LAYERS) and LONG_ROWS.max() == CFG.T - 1
    for l, errs in run8b["long"].items():
        assert max(errs) <= 2 * 2.0 ** -8, (l, errs)


def _cases():
    out = []
    for prec in ("f32", "tf32", "bf16"):
        for bar in BARS:
            why = expected_miss(GOLDEN, CFG.name, prec, bar)
            marks = [pytest.mark.xfail(strict=False, reason=why)] if why else []
            out.append(pytest.param(prec, bar, marks=marks, id=f"8b-{prec}-{bar}"))
    return out


@pytest.mark.parametrize("prec,bar", _cases())
def test_stated_bar_8b(run8b, prec, bar):
    m = _stated_metrics(run8b, prec)
    if bar == BARS[0]:
        record(f"stated qwen3-8b-shape {prec} rows 0..{R - 1}", m)
    assert bar_holds(prec, bar, m), {k: v for k, v in m.items() if not isinstance(v, list)}


def test_long_sequence_rows_at_16k(dtp):
    """The 8B shape at T = 16384, the attention sweep's longest sequence, through
    the whole bf16 pass (128 query tiles, up to 128 key tiles per query tile):
    layers 0 and 35 on the GPU's own 16384-row input, compared on rows spread to
    T - 1, within one layer's bf16 rounding bound (2u, u = 2^-8)."""
    cfg = CFG.replace(T=16384)
    T, d = cfg.T, cfg.n_embd
    rows = np.unique(np.concatenate([np.linspace(0, T - 1, 24).astype(int), [16256, 16300, T - 1]]))
    m = dtp.Model(cfg)
    for l in range(cfg.n_layer):
        m.load_layer(l, synth.layer_weights(cfg, l))
    m.load_globals(synth.tok_embd(cfg), synth.output_norm(cfg), synth.output_weight(cfg))
    toks = torch.as_tensor(synth.tokens(cfg).astype(np.int32), device=dev)
    hidden = torch.empty((cfg.n_layer + 1, T, d), dtype=torch.float32, device=dev)
    dtp.fwd_prefill_ex(m.c, m.packed, toks, m.workspace(T), hidden=hidden)   # no logits
    torch.cuda.synchronize()
    dtp.check()
    layers = (0, 35)
    x_in = {l: hidden[l].cpu().numpy().astype(np.float64) for l in layers}
    x_out = {l: hidden[l + 1][torch.as_tensor(rows, device=dev)].cpu().numpy().astype(np.float64)
             for l in layers}
    del m, hidden
    gc.collect()
    torch.cuda.empty_cache()
    worst = {}
    for l in layers:
        lw = {k: v.astype(np.float64) for k, v in synth.layer_weights(cfg, l).items()}
        ref = oracle.forward_layer(cfg, lw, x_in[l], np.arange(T), bf16_operands=True,
                                   bf16_fused_norm=True, rows=rows)
        errs = [rel_l2(x_out[l][i], ref[i]) for i in range(len(rows))]
        worst[str(l)] = max(errs)
        assert max(errs) <= 2 * 2.0 ** -8, (l, errs)
    record("8b T=16384 long-range rows", {"rows": rows.tolist(), "per_layer_max": worst})
