"""Pins for the CPU oracle: closed forms, invariants, hand-derived fixtures,
brute force on tiny inputs and float64 library routines.  None of these
re-types the oracle's own formula; each is chosen so that a plausible slip
(dropped eps, wrong pair split, wrong GQA map, swapped gate/up, off-by-one
causal mask, transposed weight) fails at least one of them -- the
`test_planted_*` cases plant exactly those slips in the oracle and check that.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _eval_golden(v):
    if isinstance(v, str):
        return float(eval(v, {"cos": math.cos, "sin": math.sin}))
    return float(v)


# ---------------------------------------------------------------- bf16 rounding
def test_round_bf16_hand_fixture():
    g = json.load(open(os.path.join(GOLDEN, "bf16_rounding_hand.json")))
    for c in g["cases"]:
        assert oracle.round_bf16(np.array([c["x"]]))[0] == c["y"], c


def test_round_bf16_matches_torch_on_f32_values():
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- RMSNorm
def test_rms_norm_unit_weight_closed_form():
    x = rng.standard_normal((7, 33)) * 3.0
    eps = 0.25
    y = oracle.rms_norm(x, np.ones(33), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-13)
    # direction preserved
    np.testing.assert_allclose(y / np.linalg.norm(y, axis=1, keepdims=True),
                               x / np.linalg.norm(x, axis=1, keepdims=True), rtol=1e-13)


def test_rms_norm_scale_invariant_without_eps_and_weight_is_plain_multiply():
    x = rng.standard_normal((5, 16))
    w = 1.0 + 0.1 * rng.standard_normal(16)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, w, 0.0), oracle.rms_norm(x, w, 0.0), rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 0.0), oracle.rms_norm(x, np.ones(16), 0.0) * w,
                               rtol=1e-14)


def test_rms_norm_matches_torch_f64():
    x = rng.standard_normal((9, 64))
    w = 1.0 + 0.1 * rng.standard_normal(64)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-6)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), ref.numpy(), rtol=1e-13, atol=0)


def test_qk_norm_is_per_head_row():
    T, nh, hd = 5, 3, 8
    x = rng.standard_normal((T, nh * hd)) * np.repeat([0.1, 10.0, 1000.0], hd)[None, :]
    w = 1.0 + 0.1 * rng.standard_normal(hd)
    y = oracle.qk_norm(x, w, hd, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x.reshape(T, nh, hd)), (hd,),
                                       torch.from_numpy(w), eps=1e-6).reshape(T, nh * hd)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13)
    # each (token, head) row has unit RMS before the scale
    u = oracle.qk_norm(x, np.ones(hd), hd, 0.0).reshape(T, nh, hd)
    np.testing.assert_allclose(np.mean(u * u, axis=2), 1.0, rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_hand_fixture():
    g = json.load(open(os.path.join(GOLDEN, "rope_neox_hand.json")))
    for c in g["cases"]:
        y = oracle.rope_neox(np.array([c["x"]]), np.array([c["pos"]]), 1, 4, 4, 100.0)[0]
        np.testing.assert_allclose(y, [_eval_golden(v) for v in c["y"]], rtol=1e-15, atol=1e-15)
    p = g["partial"]
    y = oracle.rope_neox(np.array([p["x"]]), np.array([p["pos"]]), 1, 4, 2, 100.0)[0]
    np.testing.assert_allclose(y, [_eval_golden(v) for v in p["y"]], rtol=1e-15, atol=1e-15)


def test_rope_invariants():
    T, nh, hd, r = 40, 3, 16, 12
    x = rng.standard_normal((T, nh * hd))
    pos = np.arange(T)
    y = oracle.rope_neox(x, pos, nh, hd, r, 1e4)
    X, Y = x.reshape(T, nh, hd), y.reshape(T, nh, hd)
    # position 0 is the identity, bit for bit
    assert np.array_equal(Y[0], X[0])
    # dims >= r pass through unchanged
    assert np.array_equal(Y[:, :, r:], X[:, :, r:])
    # every (i, i + r/2) pair keeps its norm
    h = r // 2
    np.testing.assert_allclose(Y[:, :, :h] ** 2 + Y[:, :, h:r] ** 2, X[:, :, :h] ** 2 + X[:, :, h:r] ** 2,
                               rtol=1e-12)
    # linear and orthogonal: R^T R = I on the rotated block
    M = np.stack([oracle.rope_neox(np.eye(hd)[i][None, :], np.array([17]), 1, hd, r, 1e4)[0]
                  for i in range(hd)])
    np.testing.assert_allclose(M @ M.T, np.eye(hd), atol=1e-14)


def test_rope_relative_position():
    # <R_p q, R_s k> depends only on p - s
    hd = 32
    q = rng.standard_normal((1, hd))
    k = rng.standard_normal((1, hd))

    def dot(p, s):
        return float(oracle.rope_neox(q, np.array([p]), 1, hd, hd, 1e6)[0]
                     @ oracle.rope_neox(k, np.array([s]), 1, hd, hd, 1e6)[0])
    for p, s, c in [(5, 2, 100), (9, 9, 1000), (3, 40, 7)]:
        assert abs(dot(p, s) - dot(p + c, s + c)) < 1e-9


def test_rope_full_rotary_matches_v3_table_definition():
    # v3/model.rs: freq_i = 1 / theta^(2i/dims), angle = t * freq_i (dims = head_dim)
    hd, base = 8, 1e6
    ang = oracle.rope_angles(np.array([0, 1, 7]), hd, base)
    for t, row in zip([0, 1, 7], ang):
        for i in range(hd // 2):
            assert row[i] == pytest.approx(t * (1.0 / base ** ((2 * i) / hd)), rel=1e-15)


# ---------------------------------------------------------------- attention
def _brute_attention(q, k, v, nh, nkv, hd, scale):
    """Scalar loops: for each (t, head) a softmax over keys 0..t."""
    T = q.shape[0]
    out = np.zeros_like(q)
    grp = nh // nkv
    for t in range(T):
        for i in range(nh):
            j = i // grp
            logits = [sum(q[t, i * hd + d] * k[s, j * hd + d] for d in range(hd)) * scale
                      for s in range(t + 1)]
            m = max(logits)
            e = [math.exp(a - m) for a in logits]
            z = sum(e)
            for d in range(hd):
                out[t, i * hd + d] = sum(e[s] * v[s, j * hd + d] for s in range(t + 1)) / z
    return out


@pytest.mark.parametrize("T,nh,nkv,hd", [(1, 2, 1, 4), (5, 4, 2, 3), (8, 6, 3, 2), (7, 4, 4, 5)])
def test_sdpa_brute_force(T, nh, nkv, hd):
    q = rng.standard_normal((T, nh * hd))
    k = rng.standard_normal((T, nkv * hd))
    v = rng.standard_normal((T, nkv * hd))
    scale = 1 / math.sqrt(hd)
    np.testing.assert_allclose(oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, scale),
                               _brute_attention(q, k, v, nh, nkv, hd, scale), rtol=1e-12, atol=1e-13)


def test_sdpa_matches_torch_sdpa_f64():
    T, nh, nkv, hd = 37, 8, 2, 16
    q = rng.standard_normal((T, nh * hd))
    k = rng.standard_normal((T, nkv * hd))
    v = rng.standard_normal((T, nkv * hd))
    tq = torch.from_numpy(q).reshape(T, nh, hd).transpose(0, 1)[None]
    tk = torch.from_numpy(k).reshape(T, nkv, hd).transpose(0, 1)[None]
    tv = torch.from_numpy(v).reshape(T, nkv, hd).transpose(0, 1)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    ref = ref[0].transpose(0, 1).reshape(T, nh * hd).numpy()
    np.testing.assert_allclose(oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 1 / math.sqrt(hd)), ref,
                               rtol=1e-12, atol=1e-13)


def test_sdpa_special_cases():
    T, nh, nkv, hd = 9, 4, 2, 6
    k = rng.standard_normal((T, nkv * hd))
    v = rng.standard_normal((T, nkv * hd))
    # q = 0: uniform weights over the visible keys -> running mean of v (group head)
    out = oracle.sdpa_causal_gqa(np.zeros((T, nh * hd)), k, v, nh, nkv, hd, 0.3)
    V = v.reshape(T, nkv, hd)
    running = np.cumsum(V, axis=0) / np.arange(1, T + 1)[:, None, None]
    for i in range(nh):
        np.testing.assert_allclose(out[:, i * hd:(i + 1) * hd], running[:, i // 2], rtol=1e-13)
    # first query sees only key 0: output = v[0] of its group head
    q = rng.standard_normal((T, nh * hd))
    out = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 0.3)
    for i in range(nh):
        np.testing.assert_allclose(out[0, i * hd:(i + 1) * hd], V[0, i // 2], rtol=1e-14)


def test_sdpa_gqa_equals_mha_with_repeated_kv():
    T, nh, nkv, hd = 11, 8, 2, 4
    q = rng.standard_normal((T, nh * hd))
    k = rng.standard_normal((T, nkv * hd))
    v = rng.standard_normal((T, nkv * hd))
    rep = lambda a: np.repeat(a.reshape(T, nkv, hd), nh // nkv, axis=1).reshape(T, nh * hd)
    assert np.array_equal(oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 0.5),
                          oracle.sdpa_causal_gqa(q, rep(k), rep(v), nh, nh, hd, 0.5))


def test_sdpa_causal_and_row_subset():
    T, nh, nkv, hd = 16, 2, 1, 4
    q = rng.standard_normal((T, nh * hd))
    k = rng.standard_normal((T, nkv * hd))
    v = rng.standard_normal((T, nkv * hd))
    full = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[9:] += 5.0
    v2[9:] -= 3.0
    changed = oracle.sdpa_causal_gqa(q, k2, v2, nh, nkv, hd, 0.5)
    np.testing.assert_array_equal(full[:9], changed[:9])
    assert not np.allclose(full[9:], changed[9:])
    rows = np.array([0, 3, 15])
    np.testing.assert_allclose(oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 0.5, rows=rows), full[rows],
                               rtol=1e-13)


# ---------------------------------------------------------------- SwiGLU, linear
def test_swiglu_closed_forms_and_torch():
    g = rng.standard_normal(1000) * 4
    u = rng.standard_normal(1000)
    ref = torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)
    np.testing.assert_allclose(oracle.swiglu(g, u), ref.numpy(), rtol=1e-14)
    # silu(x) - silu(-x) = x ; silu(0) = 0 ; gate and up are not interchangeable
    np.testing.assert_allclose(oracle.silu(g) - oracle.silu(-g), g, rtol=1e-12, atol=1e-15)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.swiglu(np.array([2.0]), np.array([0.0]))[0] == 0.0
    assert oracle.swiglu(np.array([0.0]), np.array([2.0]))[0] == 0.0
    assert oracle.swiglu(np.array([1.0]), np.array([3.0]))[0] == pytest.approx(3.0 / (1 + math.exp(-1)))


def test_linear_exact_on_integers_and_orientation():
    x = rng.integers(-5, 6, (4, 3)).astype(float)
    W = rng.integers(-5, 6, (7, 3)).astype(float)          # [out, in]
    y = oracle.linear(x, W)
    assert y.shape == (4, 7)
    for t in range(4):
        for o in range(7):
            assert y[t, o] == sum(x[t, c] * W[o, c] for c in range(3))


# ---------------------------------------------------------------- logit helpers
def test_argmax_top2_prime_gate():
    assert oracle.argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.top2([5.0, 1.0, 5.0]) == (0, 5.0, 2, 5.0)
    assert oracle.top2([1.0, 4.0, 2.0, 3.0]) == (1, 4.0, 3, 3.0)
    a = np.array([0.0, 2.0, 1.5])
    assert oracle.prime_gate_verdict(a, a + 0.01)[0] == "match"
    assert oracle.prime_gate_verdict(a, np.array([0.0, 1.4, 1.6]))[0] == "near_tie_flip"
    assert oracle.prime_gate_verdict(np.array([0.0, 3.0, 1.0]), np.array([0.0, 1.0, 1.2]))[0] == "structured"
    assert oracle.prime_gate_verdict(a, a + 9.0)[0] == "structured"
    assert oracle.prime_gate_verdict(a, np.array([0.0, np.nan, 1.0]))[0] == "structured"


# ---------------------------------------------------------------- whole forward
TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module")
def tiny_weights():
    return synth.model_weights(TINY, seed=0)


def test_forward_causal_prefix(tiny_weights):
    toks = synth.tokens(TINY)
    full, hid = oracle.forward(TINY, tiny_weights, toks, return_hidden=True)
    for k in (1, 5, 16):
        pre, hpre = oracle.forward(TINY, tiny_weights, toks[:k], return_hidden=True)
        np.testing.assert_allclose(pre, full[:k], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(hpre, hid[:, :k], rtol=1e-12, atol=1e-14)
    toks2 = toks.copy()
    toks2[10:] = (toks2[10:] + 1) % TINY.n_vocab
    changed = oracle.forward(TINY, tiny_weights, toks2)
    np.testing.assert_allclose(changed[:10], full[:10], rtol=1e-12, atol=1e-14)
    assert not np.allclose(changed[10:], full[10:])


def test_forward_gqa_equals_expanded_mha(tiny_weights):
    cfg = TINY
    rep = cfg.n_head // cfg.n_head_kv
    w2 = dict(tiny_weights)
    w2["layers"] = []
    for lw in tiny_weights["layers"]:
        m = dict(lw)
        for nm in ("wk", "wv"):
            m[nm] = np.repeat(lw[nm].reshape(cfg.n_head_kv, cfg.head_dim, cfg.n_embd), rep, axis=0
                              ).reshape(cfg.n_head * cfg.head_dim, cfg.n_embd)
        w2["layers"].append(m)
    toks = synth.tokens(cfg)
    np.testing.assert_allclose(oracle.forward(cfg.replace(n_head_kv=cfg.n_head), w2, toks),
                               oracle.forward(cfg, tiny_weights, toks), rtol=1e-11, atol=1e-13)


def test_forward_bf16_mode_close_to_exact(tiny_weights):
    toks = synth.tokens(TINY)
    a = oracle.forward(TINY, tiny_weights, toks)
    b = oracle.forward(TINY, tiny_weights, toks, bf16_operands=True)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-5 < rel < 5e-2


def test_forward_single_token_has_no_attention_mixing(tiny_weights):
    # T = 1: attention returns v of each group head, so the result must not
    # depend on wq, wk, q_norm or k_norm at all.
    toks = synth.tokens(TINY)[:1]
    base = oracle.forward(TINY, tiny_weights, toks)
    w2 = dict(tiny_weights)
    w2["layers"] = [dict(lw, wq=-3 * lw["wq"], wk=lw["wk"][::-1].copy(), q_norm=lw["q_norm"] * 0.1)
                    for lw in tiny_weights["layers"]]
    np.testing.assert_allclose(oracle.forward(TINY, w2, toks), base, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- planted mistakes
def _pins_fail(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_rope_interleaved_pairs_is_caught(monkeypatch):
    def wrong(x, pos, n_heads, head_dim, n_dims, freq_base):   # GPT-J style (2i, 2i+1) pairs
        x = np.asarray(x, float)
        T = x.shape[0]
        y = x.reshape(T, n_heads, head_dim).copy()
        ang = om.rope_angles(pos, n_dims, freq_base)
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        a, b = y[:, :, 0:n_dims:2].copy(), y[:, :, 1:n_dims:2].copy()
        y[:, :, 0:n_dims:2] = a * c - b * s
        y[:, :, 1:n_dims:2] = a * s + b * c
        return y.reshape(x.shape)
    monkeypatch.setattr(oracle, "rope_neox", wrong)
    assert _pins_fail(test_rope_hand_fixture)


def test_planted_rope_sign_is_caught(monkeypatch):
    real = om.rope_neox
    monkeypatch.setattr(oracle, "rope_neox",
                        lambda x, pos, *a: real(x, -np.asarray(pos), *a))
    assert _pins_fail(test_rope_hand_fixture)


def test_planted_gqa_modulo_map_is_caught(monkeypatch):
    def wrong(q, k, v, nh, nkv, hd, scale, rows=None):       # head i -> kv head i % nkv
        out = np.zeros((q.shape[0], nh * hd))
        for i in range(nh):
            j = i % nkv
            out[:, i * hd:(i + 1) * hd] = om.sdpa_causal_gqa(
                q[:, i * hd:(i + 1) * hd], k[:, j * hd:(j + 1) * hd], v[:, j * hd:(j + 1) * hd],
                1, 1, hd, scale)
        return out
    monkeypatch.setattr(oracle, "sdpa_causal_gqa", wrong)
    assert _pins_fail(test_sdpa_matches_torch_sdpa_f64)


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    def wrong(q, k, v, nh, nkv, hd, scale, rows=None):        # key t+1 also visible
        T = q.shape[0]
        out = np.zeros((T, nh * hd))
        for i in range(nh):
            j = i // (nh // nkv)
            s = q[:, i * hd:(i + 1) * hd] @ k[:, j * hd:(j + 1) * hd].T * scale
            s[np.triu(np.ones((T, T), bool), 2)] = -np.inf
            p = np.exp(s - s.max(1, keepdims=True))
            out[:, i * hd:(i + 1) * hd] = p / p.sum(1, keepdims=True) @ v[:, j * hd:(j + 1) * hd]
        return out
    monkeypatch.setattr(oracle, "sdpa_causal_gqa", wrong)
    assert _pins_fail(lambda: test_sdpa_brute_force(5, 4, 2, 3))


def test_planted_swapped_gate_up_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "swiglu", lambda g, u: om.silu(u) * np.asarray(g))
    assert _pins_fail(test_swiglu_closed_forms_and_torch)


def test_planted_rms_eps_outside_root_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "rms_norm",
                        lambda x, w, eps: np.asarray(x) / (np.sqrt(np.mean(np.square(x), -1, keepdims=True)) + eps) * w)
    assert _pins_fail(test_rms_norm_unit_weight_closed_form)


def test_planted_transposed_weight_is_caught(monkeypatch):
    # reading the [out, in] weight memory as if it were [in, out]
    monkeypatch.setattr(oracle, "linear",
                        lambda x, W: np.asarray(x) @ np.asarray(W).reshape(W.shape[1], W.shape[0]))
    assert _pins_fail(test_linear_exact_on_integers_and_orientation)


# ---------------------------------------------------------------- gated attention
def _gated_from(cfg, w, gate_rows):
    """Gated weights: per head, that head's q rows then `gate_rows(head)`."""
    hd, h = cfg.head_dim, cfg.n_head
    w2 = dict(w)
    w2["layers"] = []
    for lw in w["layers"]:
        blocks = []
        for i in range(h):
            blocks.append(lw["wq"][i * hd:(i + 1) * hd])
            blocks.append(gate_rows(lw, i))
        w2["layers"].append(dict(lw, wq=np.concatenate(blocks, axis=0)))
    return w2


def test_gated_attention_zero_gate_halves_attention():
    # sigmoid(0) = 1/2: the gated model with zero gate rows is the ungated model
    # with Wo halved -- this also pins the per-head [q | gate] row layout
    w = synth.model_weights(TINY)
    gcfg = TINY.replace(attn_gate=True)
    wg = _gated_from(TINY, w, lambda lw, i: np.zeros((TINY.head_dim, TINY.n_embd)))
    wh = dict(w)
    wh["layers"] = [dict(lw, wo=0.5 * lw["wo"]) for lw in w["layers"]]
    toks = synth.tokens(TINY)
    np.testing.assert_allclose(oracle.forward(gcfg, wg, toks), oracle.forward(TINY, wh, toks),
                               rtol=1e-12, atol=1e-14)


def test_planted_gate_layout_swap_is_caught(monkeypatch):
    # reading the q region as [all q heads | all gate heads] instead of per head
    real = om.forward_layer

    def wrong(cfg, lw, x, pos, bf16_operands=False, kv_out=None, *args, **kw):
        if getattr(cfg, "attn_gate", False):
            h, hd = cfg.n_head, cfg.head_dim
            wq = lw["wq"].reshape(2, h, hd, -1).transpose(1, 0, 2, 3).reshape(2 * h * hd, -1)
            lw = dict(lw, wq=wq)
        return real(cfg, lw, x, pos, bf16_operands, kv_out, *args, **kw)
    monkeypatch.setattr(om, "forward_layer", wrong)
    assert _pins_fail(test_gated_attention_zero_gate_halves_attention)


# ---------------------------------------------------------------- chunked prefill
def _chunked(cfg, w, toks, sizes, bf16=False):
    state, outs, p = [], [], 0
    for c in sizes:
        outs.append(oracle.forward_chunk(cfg, w, toks[p:p + c], state, bf16_operands=bf16))
        p += c
    return np.concatenate(outs), state


@pytest.mark.parametrize("sizes", [(16,), (5, 7, 4), (1, 1, 14), (15, 1)])
def test_forward_chunk_concatenates_to_the_full_pass(tiny_weights, sizes):
    """Causality: the chunks' logits are the whole pass's rows, and the state
    ends up holding every layer's (k, v) of the whole pass."""
    toks = synth.tokens(TINY)
    kv = []
    full = oracle.forward(TINY, tiny_weights, toks, kv_out=kv)
    got, state = _chunked(TINY, tiny_weights, toks, sizes)
    np.testing.assert_allclose(got, full, rtol=1e-11, atol=1e-13)
    assert len(state) == TINY.n_layer
    for (k, v), (k2, v2) in zip(state, kv):
        np.testing.assert_allclose(k, k2, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(v, v2, rtol=1e-11, atol=1e-13)


def test_forward_chunk_bf16_mode_concatenates(tiny_weights):
    toks = synth.tokens(TINY)
    full = oracle.forward(TINY, tiny_weights, toks, bf16_operands=True)
    got, _ = _chunked(TINY, tiny_weights, toks, (6, 10), bf16=True)
    # same values rounded the same way; only BLAS summation order may differ
    assert np.linalg.norm(got - full) / np.linalg.norm(full) < 1e-2


def test_sdpa_offset_equals_row_subset():
    a = synth.attention_inputs(24, 4, 2, 8, seed=3)
    q, k, v = a["q"], a["k"], a["v"]
    full = oracle.sdpa_causal_gqa(q, k, v, 4, 2, 8, 0.3)
    for p0 in (0, 1, 9, 23):
        np.testing.assert_allclose(oracle.sdpa_causal_gqa(q[p0:], k, v, 4, 2, 8, 0.3, p0=p0),
                                   full[p0:], rtol=1e-12, atol=1e-14)


def test_planted_chunk_positions_restart_is_caught(monkeypatch, tiny_weights):
    """A chunk that restarts RoPE positions at 0 (or masks from its own first
    row) fails the concatenation pin."""
    real = om.forward_layer

    def wrong(cfg, lw, x, pos, *args, **kw):
        return real(cfg, lw, x, np.arange(len(pos)), *args, **kw)
    monkeypatch.setattr(om, "forward_layer", wrong)
    assert _pins_fail(lambda: test_forward_chunk_concatenates_to_the_full_pass(tiny_weights,
                                                                              (5, 7, 4)))


# ---------------------------------------------------------------- tf32 rounding
def test_round_tf32_hand_fixture():
    """11 significant bits, nearest, ties to even (hand-worked values)."""
    u = 2.0 ** -10                                   # one tf32 ulp at 1.0
    cases = [(1.0, 1.0), (1.0 + u, 1.0 + u), (1.0 + u / 2, 1.0),        # tie -> even (1.0)
             (1.0 + 3 * u / 2, 1.0 + 2 * u),                            # tie -> even (1+2u)
             (1.0 + 0.49 * u, 1.0), (1.0 + 0.51 * u, 1.0 + u),
             (-3.0 - u, -3.0), (2.0 ** 20 * (1 + u / 2), 2.0 ** 20), (0.0, 0.0)]
    for x, want in cases:
        assert oracle.round_tf32(x) == want, (x, want)


def test_round_tf32_matches_bit_rounding_on_f32_values():
    """On float32 inputs, round_tf32 equals nearest-even rounding of the bit
    pattern (add 0xFFF plus the kept lsb, clear the 13 dropped bits), and it is
    idempotent and keeps at most 11 significant bits."""
    x = (synth.normal(9, 900, (20000,)) * np.exp(synth.normal(9, 901, (20000,)) * 4)).astype(np.float32)
    x[:4] = [1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -(1.0 + 2.0 ** -11), 1.5]   # exact ties
    u = x.view(np.uint32).astype(np.uint64)
    want = ((u + 0xFFF + ((u >> 13) & 1)) & ~np.uint64(0x1FFF)).astype(np.uint32).view(np.float32)
    got = oracle.round_tf32(x)
    np.testing.assert_array_equal(got, want.astype(np.float64))
    np.testing.assert_array_equal(oracle.round_tf32(got), got)
    m, _ = np.frexp(got)
    np.testing.assert_array_equal(m * 2048, np.rint(m * 2048))


def test_forward_tf32_mode_between_exact_and_bf16(tiny_weights):
    toks = synth.tokens(TINY)
    a = oracle.forward(TINY, tiny_weights, toks)
    t = oracle.forward(TINY, tiny_weights, toks, tf32_operands=True)
    b = oracle.forward(TINY, tiny_weights, toks, bf16_operands=True)
    rt = np.linalg.norm(a - t) / np.linalg.norm(a)
    rb = np.linalg.norm(a - b) / np.linalg.norm(a)
    # 3 more significant bits: the error shrinks about 8x
    assert 1e-6 < rt < rb / 3


# ---------------------------------------------------------------- e4m3 quantisation
def test_round_e4m3_hand_fixture():
    """OCP E4M3: 4 significant bits, subnormal step 2^-9 below 2^-6, max 448,
    nearest with ties to even (hand-worked values)."""
    cases = [(1.0, 1.0), (1.0625, 1.0),                  # tie between 1 and 1.125 -> even (1)
             (1.1875, 1.25),                            # tie between 1.125 and 1.25 -> even
             (1.09, 1.125), (-3.3, -3.25), (448.0, 448.0), (464.0, 448.0),   # tie -> even (448)
             (470.0, 448.0), (1e6, 448.0), (-1e6, -448.0),                    # saturation
             (2.0 ** -6, 2.0 ** -6), (2.0 ** -9, 2.0 ** -9), (2.0 ** -10, 0.0),  # tie -> 0
             (3 * 2.0 ** -11, 2.0 ** -9), (5 * 2.0 ** -10, 2.0 ** -8),       # tie 2.5 ulp -> 2
             (0.0137, 7 * 2.0 ** -9), (0.0, 0.0)]
    for x, want in cases:
        assert oracle.round_e4m3(x) == want, (x, oracle.round_e4m3(x), want)


def test_round_e4m3_matches_torch_float8_in_range():
    """torch's float8_e4m3fn cast (nearest-even) agrees on every value below the
    saturation point, including the subnormal range and exact ties."""
    x = synth.normal(10, 1000, (30000,)) * np.exp2(np.round(synth.normal(10, 1001, (30000,)) * 5))
    x = x[np.abs(x) < 464].astype(np.float32)
    ties = (np.arange(1, 64, dtype=np.float32) + 0.5) * np.float32(2.0 ** -9)
    x = np.concatenate([x, ties, -ties])
    want = torch.as_tensor(x).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(oracle.round_e4m3(x), want)


def test_fake_quant_rows_e4m3_properties():
    a = synth.normal(10, 1002, (64, 300)) * np.exp(synth.normal(10, 1003, (64, 1)) * 3)
    a[5] = 0.0
    q = oracle.fake_quant_rows_e4m3(a)
    amax = np.abs(a).max(axis=1)
    # each row's largest element maps to +-448, so it comes back (up to the
    # float64 rounding of s = amax / 448)
    np.testing.assert_allclose(np.abs(q).max(axis=1), amax, rtol=1e-15, atol=0)
    assert not q[5].any()
    # relative error at most half an e4m3 ulp (2^-4) in the normal range; the
    # subnormal range (|a| < 2^-6 * s) has absolute error <= 2^-10 * s
    s = (amax / 448.0)[:, None]
    err = np.abs(q - a)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(a), 2.0 ** -10 * s) * (1 + 1e-12))
    # scaling a row by a power of two scales its quantisation exactly
    np.testing.assert_array_equal(oracle.fake_quant_rows_e4m3(a * 2.0 ** 7), q * 2.0 ** 7)
    # per-row: rows are independent
    np.testing.assert_array_equal(oracle.fake_quant_rows_e4m3(a[:7])[3], q[3])


def test_forward_fp8_mode_is_coarser_than_bf16(tiny_weights):
    toks = synth.tokens(TINY)
    a = oracle.forward(TINY, tiny_weights, toks)
    b = oracle.forward(TINY, tiny_weights, toks, bf16_operands=True)
    f = oracle.forward(TINY, tiny_weights, toks, fp8_operands=True)
    rb = np.linalg.norm(a - b) / np.linalg.norm(a)
    rf = np.linalg.norm(a - f) / np.linalg.norm(a)
    # 4 significant bits instead of 8, partly offset by the per-row scales
    assert rb < rf < 0.2
