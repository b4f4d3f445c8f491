"""Pins for how the oracle wires the pinned ops into a layer and a pass
(docs.rs memra-engine 0.130.0, src/forward.rs, `Model::forward`: the loop body
adds the attention output, projected by Wo, to the residual stream; the FFN
RMSNorm reads that updated stream; the FFN output, projected by Wdown, is
added to it; after the last layer the stream goes through output_norm and then
the lm_head).

Each pin is a special case whose answer follows from that statement alone:
  * with Wo = 0 and Wdown = 0 a layer is the identity, so the logits are the
    closed form rms_norm(E[token]) * output_norm times W_out^T;
  * at T = 1 attention returns the group head's v, so a layer reduces to two
    residual blocks of plain matrix algebra, written out here with numpy;
  * each branch enters the stream linearly through its output projection;
  * with Wo = 0 the layer sees its input only through RMSNorm, so scaling the
    stream leaves the added branch unchanged (eps = 0).
The planted cases rewrite one line of the oracle's source in a scratch module
(never the oracle itself) and check that a pin fails.  The hand-worked bf16
fixture pins the rounding points of the fused-norm diagnostic mode.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle
import synth
from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny_weights():
    return synth.model_weights(TINY, seed=0)


def _zeroed(weights, names):
    w2 = dict(weights)
    w2["layers"] = [dict(lw, **{n: np.zeros_like(lw[n]) for n in names}) for lw in weights["layers"]]
    return w2


def _layer0(weights, **repl):
    return dict(weights["layers"][0], **repl)


def _np_rms(x, w, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, np.float64)


# ------------------------------------------------------------------------------ the pins
def pin_identity_layers(orc, weights):
    """Wo = Wdown = 0: every layer returns its input, and the logits are the
    closed form of output_norm + lm_head on the embedding rows."""
    w0 = _zeroed(weights, ("wo", "w_down"))
    toks = synth.tokens(TINY)
    x = np.asarray(weights["tok_embd"], np.float64)[toks]
    y = orc.forward_layer(TINY, w0["layers"][0], x, np.arange(len(toks)))
    assert np.array_equal(y, x), "a layer with Wo = Wdown = 0 must return its input"
    logits = orc.forward(TINY, w0, toks)
    ref = _np_rms(x, weights["output_norm"], TINY.rms_eps) @ np.asarray(weights["output"], np.float64).T
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-14)


def pin_single_token_closed_form(orc, weights):
    """T = 1: softmax over one key is 1, so head i's attention output is the v of
    kv head i // (n_head / n_head_kv); the layer is then
      x1 = x + A Wo^T,  A = [v_(i // G)]_i,  v = rms(x) w_attn Wv^T
      x2 = x1 + (silu(z Wg^T) * (z Wu^T)) Wd^T,  z = rms(x1) w_ffn."""
    cfg, hd = TINY, TINY.head_dim
    G = cfg.n_head // cfg.n_head_kv
    lw = {k: np.asarray(v, np.float64) for k, v in weights["layers"][0].items()}
    for tok in (3, 77, 200):
        x = np.asarray(weights["tok_embd"], np.float64)[[tok]]
        h = _np_rms(x, lw["attn_norm"], cfg.rms_eps)
        v = h @ lw["wv"].T
        A = np.concatenate([v[:, (i // G) * hd:(i // G + 1) * hd] for i in range(cfg.n_head)], axis=1)
        x1 = x + A @ lw["wo"].T
        z = _np_rms(x1, lw["ffn_norm"], cfg.rms_eps)
        g, u = z @ lw["w_gate"].T, z @ lw["w_up"].T
        x2 = x1 + ((g / (1 + np.exp(-g))) * u) @ lw["w_down"].T
        got = orc.forward_layer(cfg, weights["layers"][0], x, np.arange(1))
        np.testing.assert_allclose(got, x2, rtol=1e-12, atol=1e-15)


def pin_branches_enter_linearly(orc, weights):
    """Each branch is added to the stream through its output projection: with the
    other branch's projection zero, scaling Wo (or Wdown) by c scales the
    layer's increment by c, and the attention weights matter only through Wo."""
    toks = synth.tokens(TINY)
    x = np.asarray(weights["tok_embd"], np.float64)[toks]
    pos = np.arange(len(toks))
    lw = weights["layers"][0]
    f = lambda **r: orc.forward_layer(TINY, _layer0(weights, **r), x, pos) - x
    zd, zo = np.zeros_like(lw["w_down"]), np.zeros_like(lw["wo"])
    base = f(w_down=zd)
    assert np.linalg.norm(base) > 1e-3
    for c in (2.0, -0.5):
        np.testing.assert_allclose(f(w_down=zd, wo=c * lw["wo"]), c * base, rtol=1e-11, atol=1e-14)
    ffn = f(wo=zo)
    assert np.linalg.norm(ffn) > 1e-3
    for c in (2.0, -0.5):
        np.testing.assert_allclose(f(wo=zo, w_down=c * lw["w_down"]), c * ffn, rtol=1e-11, atol=1e-14)
    # with Wo = 0 nothing of the attention block reaches the stream
    np.testing.assert_allclose(f(wo=zo, wq=3 * lw["wq"], wk=-lw["wk"], wv=2 * lw["wv"],
                                 q_norm=0.5 * lw["q_norm"], attn_norm=7 * lw["attn_norm"]),
                               ffn, rtol=1e-12, atol=1e-15)


def pin_prenorm_scale_invariance(orc, weights):
    """Wo = 0, eps = 0: the FFN sees the stream only through RMSNorm, so the
    increment f(c x) - c x equals f(x) - x for any c > 0."""
    cfg = TINY.replace(rms_eps=0.0)
    toks = synth.tokens(TINY)
    x = np.asarray(weights["tok_embd"], np.float64)[toks]
    pos = np.arange(len(toks))
    lw = _layer0(weights, wo=np.zeros_like(weights["layers"][0]["wo"]))
    inc = orc.forward_layer(cfg, lw, x, pos) - x
    for c in (0.125, 9.0):
        np.testing.assert_allclose(orc.forward_layer(cfg, lw, c * x, pos) - c * x, inc,
                                   rtol=1e-9, atol=1e-12)


PINS = (pin_identity_layers, pin_single_token_closed_form, pin_branches_enter_linearly,
        pin_prenorm_scale_invariance)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_composition_pin(pin, tiny_weights):
    pin(om, tiny_weights)


# ------------------------------------------------------------------------------ planted slips
def _planted(old: str, new: str):
    """A scratch copy of the oracle module with one source line rewritten."""
    src = open(om.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_planted")
    exec(compile(src.replace(old, new), "oracle_planted", "exec"), mod.__dict__)
    return mod


def _caught(mod, weights):
    failed = []
    for pin in PINS:
        try:
            pin(mod, weights)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


PLANTS = {
    "no_attention_residual": ('    x1 = x + linear(attn, L["wo"])', '    x1 = linear(attn, L["wo"])'),
    "no_ffn_residual": ('    return x1 + linear(act, L["w_down"])', '    return linear(act, L["w_down"])'),
    "ffn_norm_on_layer_input": ('    gt, up = normed_linears(x1, lw["ffn_norm"], ("w_gate", "w_up"))',
                                '    gt, up = normed_linears(x, lw["ffn_norm"], ("w_gate", "w_up"))'),
    "attn_norm_weight_in_ffn": ('    gt, up = normed_linears(x1, lw["ffn_norm"], ("w_gate", "w_up"))',
                                '    gt, up = normed_linears(x1, lw["attn_norm"], ("w_gate", "w_up"))'),
    "ffn_residual_from_layer_input": ('    return x1 + linear(act, L["w_down"])',
                                      '    return x + linear(act, L["w_down"])'),
    "no_output_norm": (
        '    hn = op(rms_norm(x, np.asarray(weights["output_norm"], dtype=F64), cfg.rms_eps))\n'
        '    logits = linear(',
        '    hn = op(x)\n    logits = linear('),
    "post_norm_stream": ('    x1 = x + linear(attn, L["wo"])',
                         '    x1 = rms_norm(x + linear(attn, L["wo"]), lw["ffn_norm"], eps)'),
}


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_planted_wiring_slip_is_caught(name, tiny_weights):
    mod = _planted(*PLANTS[name])
    assert _caught(mod, tiny_weights), f"planted slip {name} passed every composition pin"


def test_planting_machinery_keeps_a_correct_copy_green(tiny_weights):
    mod = _planted('    x1 = x + linear(attn, L["wo"])', '    x1 = x + linear(attn, L["wo"])  # same')
    assert _caught(mod, tiny_weights) == []


# ------------------------------------------------------------------------------ bf16 rounding points
def _ev(e):
    return float(eval(e, {"sqrt": math.sqrt}))


def test_bf16_rounding_points_hand_fixture():
    """The plain bf16 placement (h = bf16(rms_norm(x) * w), then bf16(W)) and the
    fused diagnostic (bf16(x) times bf16(W * w), then 1/rms) against values
    worked out by hand."""
    d = json.load(open(os.path.join(GOLDEN, "bf16_fused_norm_hand.json")))
    for c in d["cases"]:
        x, w, W = (np.array(c[k], np.float64) for k in ("x", "w", "W"))
        plain = oracle.linear(oracle.round_bf16(oracle.rms_norm(x[None, :], w, 0.0)),
                              oracle.round_bf16(W))[0]
        fused = oracle.bf16_fused_normed_linear(x[None, :], w, W, 0.0)[0]
        np.testing.assert_allclose(plain, [_ev(e) for e in c["plain"]], rtol=0, atol=1e-15)
        np.testing.assert_allclose(fused, [_ev(e) for e in c["fused"]], rtol=1e-15, atol=1e-15)


def test_fused_and_plain_bf16_modes_agree_when_nothing_rounds():
    """Inputs on which no rounding happens (bf16-exact x and W, power-of-two norm
    weights, a power-of-two rms): the two placements give the same layer."""
    cfg = TINY.replace(n_layer=1)
    d = cfg.n_embd
    rs = np.random.default_rng(5)
    lw = synth.layer_weights(cfg, 0)
    lw = {k: (oracle.round_bf16(v) if v.ndim == 2 else v) for k, v in lw.items()}
    lw["attn_norm"] = 2.0 ** rs.integers(-1, 2, d)
    lw["ffn_norm"] = 2.0 ** rs.integers(-1, 2, d)
    x = rs.choice([-1.0, 1.0], size=(4, d))          # rms exactly 1
    pos = np.arange(4)
    a = oracle.forward_layer(cfg.replace(rms_eps=0.0), lw, x, pos, bf16_operands=True)
    b = oracle.forward_layer(cfg.replace(rms_eps=0.0), lw, x, pos, bf16_operands=True,
                             bf16_fused_norm=True)
    # the attention block rounds identically; the FFN input x1 is no longer
    # exact, so compare the attention half through Wdown = 0
    lw0 = dict(lw, w_down=np.zeros_like(lw["w_down"]))
    a0 = oracle.forward_layer(cfg.replace(rms_eps=0.0), lw0, x, pos, bf16_operands=True)
    b0 = oracle.forward_layer(cfg.replace(rms_eps=0.0), lw0, x, pos, bf16_operands=True,
                              bf16_fused_norm=True)
    assert np.array_equal(a0, b0)
    assert np.isfinite(a).all() and np.isfinite(b).all()


@pytest.mark.parametrize("gated", [False, True])
def test_layer_rows_equal_the_rows_of_the_whole_layer(gated):
    """forward_layer(rows=r) is row r of the whole layer: every step after the
    attention acts on each row alone, and a query row's attention reads the
    keys of all earlier rows."""
    cfg = synth.CONFIGS["small"].replace(n_layer=1, T=40, attn_gate=gated)
    lw = synth.layer_weights(cfg, 0)
    x = synth.normal(0, 71, (40, cfg.n_embd)).astype(np.float64)
    pos = np.arange(40)
    rows = np.array([0, 7, 8, 31, 39])
    for mode in ({}, {"bf16_operands": True}, {"bf16_operands": True, "bf16_fused_norm": True}):
        full = oracle.forward_layer(cfg, lw, x, pos, **mode)
        part = oracle.forward_layer(cfg, lw, x, pos, rows=rows, **mode)
        np.testing.assert_allclose(part, full[rows], rtol=1e-12, atol=1e-14)
