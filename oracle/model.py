"""Float64 CPU oracle of the dense prefill forward pass (test infrastructure only).

Each function names the passage it restates.  "forward.rs" is the page
docs.rs memra-engine 0.130.0 src/forward.rs (`impl Model`, `Model::forward`);
"v3/model.rs" is the page docs.rs needle-core v3/model.rs.

Readings taken where the pages leave a step open (they show the kernels' call
sites, not their bodies):
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * w (eps inside the root, plain
    multiply by w) -- the reading of the llama.cpp qwen3 graph that forward.rs
    says it matches.
  * NeoX RoPE: pairs (i, i + n_dims/2) for i < n_dims/2, theta_i =
    base^(-2i/n_dims), angle = pos * theta_i, dims >= n_dims unchanged.  With
    n_dims == head_dim this is exactly the v3/model.rs table.
  * GQA: query head i reads kv head i // (n_head / n_head_kv).
  * Causal: key s is visible to query t iff s <= t.
  * SwiGLU (`ffn_act`): act = silu(gate) * up, silu(x) = x / (1 + e^-x).
  * Gated attention (the FusedQ gate of docs.rs memra-engine 0.101.0
    src/spec.rs, `qwen35_tparallel_fa_layer`: `q_gate_split`, `sigmoid`,
    `mul`): the Q projection yields, per head, head_dim q values followed by
    head_dim gate values; the attention output is multiplied elementwise by
    sigmoid(gate) before the O projection.
  * Chunked prefill (the pages' "growing KV" reading of the causal pass): a
    chunk at positions p0 .. p0+C-1 attends to the keys/values of positions
    0 .. p0-1 kept from earlier chunks, then to its own; its logits are the
    full pass's rows p0 .. p0+C-1.
  * bf16-operand mode: matrices are rounded to bf16 once; every GEMM input
    activation (normed h = bf16(rms_norm(x) * w), attention output, SwiGLU act,
    final normed x) and the q/k/v handed to attention are rounded to bf16
    (nearest, ties to even); all sums and the residual stream stay in float64.
    This is the plain reading of "bf16 operands" and the default.
  * bf16 mode with the norm fused (`bf16_fused_norm=True`, a diagnostic): the
    RMSNorm before the QKV and gate/up projections is applied as a row scale
    after the product, as a fused kernel may compute it.  The matrix input is
    bf16(x), the matrix is bf16(W * w) (the norm weight multiplies W's columns
    before the rounding), and 1/rms(x) scales each row of the product.  Without
    rounding this is the same function as the plain mode; only the rounding
    points move.
  * tf32-operand mode: the same GEMM operands rounded to TensorFloat-32 (10-bit
    fraction, nearest, ties to even) instead, and q/k/v as well (that mode's
    tensor-core attention reads tf32); the gate stays unrounded.
  * fp8-operand mode (the quantised-weight variant; the pages' T-parallel path
    quantises weights and activations to 8 bits in blocks): every GEMM operand
    is quantised per row to OCP E4M3 with a float32 scale max|row| / 448 --
    weights per output channel, activations per token -- and used dequantised;
    the attention output and SwiGLU act are rounded to bf16 before that (they
    are stored as bf16); the embedding, q/k/v and gate are bf16 as in bf16 mode.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------------------
# bf16 rounding (bf16-operand mode)
# --------------------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits), ties to even.

    Written out on the float64 value: x = m * 2^e with m in [0.5, 1); keep
    round-half-even(m * 2^8) / 2^8.  Finite normal-range inputs only (the
    forward pass never leaves that range)."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def round_tf32(x) -> np.ndarray:
    """Round to the nearest TensorFloat-32 value (11 significant bits: the f32
    exponent with a 10-bit fraction), ties to even; same construction as
    round_bf16 with 2^11 in place of 2^8."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 2048.0), e - 11)


E4M3_MAX = 448.0


def round_e4m3(x) -> np.ndarray:
    """Round to the nearest OCP FP8 E4M3 value, ties to even, saturating at
    +-448: 4 significant bits for |x| >= 2^-6 (x = m * 2^e, m in [0.5, 1):
    keep round-half-even(m * 2^4) / 2^4), and the fixed subnormal step 2^-9
    below 2^-6."""
    x = np.asarray(x, dtype=F64)
    _, e = np.frexp(x)
    quantum = np.ldexp(1.0, np.maximum(e - 4, -9))
    return np.clip(np.rint(x / quantum) * quantum, -E4M3_MAX, E4M3_MAX)


def fake_quant_rows_e4m3(a) -> np.ndarray:
    """Per-row e4m3 quantisation, returned dequantised: each row r gets the
    scale s_r = max|a[r]| / 448 (0 for a zero row) and a[r] -> s_r * e4m3(a[r] / s_r).
    A GEMM of two such operands is s_a s_w (q_a q_w^T): the row scales of the
    activation (per token) and of the weight (per output channel) factor out of
    every dot product."""
    a = np.asarray(a, dtype=F64)
    amax = np.max(np.abs(a), axis=-1, keepdims=True)
    s = amax / E4M3_MAX
    safe = np.where(s > 0, s, 1.0)
    return np.where(s > 0, round_e4m3(a / safe) * s, 0.0)


def _rounders(bf16_operands: bool, tf32_operands: bool, fp8_operands: bool = False):
    """Roundings of a mode: (GEMM input written from float32 -- the normed h, z and
    final hn; GEMM input stored as bf16 first -- attention output and SwiGLU act;
    weight matrices; attention operands q/k/v; the attention gate).
      bf16: bf16 everywhere (the tensor-core attention reads bf16 q/k/v and gate).
      tf32: tf32 for the GEMM operands and for q/k/v (that mode's tensor-core
            attention reads tf32); the gate stays float32.
      fp8:  per-row e4m3 for the GEMM operands (the attention output and act are
            bf16 before they are quantised); bf16 attention operands and gate."""
    ident = lambda a: a
    if bf16_operands + tf32_operands + fp8_operands > 1:
        raise ValueError("the operand modes are exclusive")
    if bf16_operands:
        return round_bf16, round_bf16, round_bf16, round_bf16, round_bf16
    if tf32_operands:
        return round_tf32, round_tf32, round_tf32, round_tf32, ident
    if fp8_operands:
        fq = fake_quant_rows_e4m3
        return fq, (lambda a: fq(round_bf16(a))), fq, round_bf16, round_bf16
    return ident, ident, ident, ident, ident


# --------------------------------------------------------------------------------------
# Ops
# --------------------------------------------------------------------------------------
def rms_norm(x, w, eps: float) -> np.ndarray:
    """forward.rs, Model::forward, the RMSNorm step (nrows rows of ncols values,
    a weight vector and eps): each row (last axis) is divided by
    sqrt(mean(row^2) + eps) and multiplied elementwise by w."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)


def qk_norm(x, w, head_dim: int, eps: float) -> np.ndarray:
    """forward.rs, Model::forward, the QK-norm comment: the token-major buffer
    [T, n_heads*head_dim] is n_heads*T contiguous rows of head_dim, and
    `rms_norm(ncols=head_dim, nrows=n_heads*T)` normalises each row with the
    shared scale vector w[head_dim]."""
    x = np.asarray(x, dtype=F64)
    return rms_norm(x.reshape(-1, head_dim), w, eps).reshape(x.shape)


def rope_angles(pos, n_dims: int, freq_base: float) -> np.ndarray:
    """Angle table [len(pos), n_dims/2]: angle[t, i] = pos[t] * base^(-2i/n_dims)
    (v3/model.rs `V3Model::rope`: freq = 1/theta^(2i/dims), angle = t*freq; the
    forward.rs call passes rope_dim_count as n_dims and freq_scale 1.0)."""
    i = np.arange(n_dims // 2, dtype=F64)
    theta = np.power(F64(freq_base), -2.0 * i / n_dims)
    return np.asarray(pos, dtype=F64)[:, None] * theta[None, :]


def rope_neox(x, pos, n_heads: int, head_dim: int, n_dims: int, freq_base: float) -> np.ndarray:
    """forward.rs, Model::forward, the NeoX RoPE step applied to q and to k
    (rope_dim_count rotated dims, base freq_base, frequency scale 1, one
    position per token): rotate, for every (token,
    head) row of head_dim, the pairs (i, i + n_dims/2), i < n_dims/2, by
    angle[token, i]; dims n_dims..head_dim pass through."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    y = x.reshape(T, n_heads, head_dim).copy()
    half = n_dims // 2
    ang = rope_angles(pos, n_dims, freq_base)
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = y[:, :, :half].copy()
    b = y[:, :, half:n_dims].copy()
    y[:, :, :half] = a * c - b * s
    y[:, :, half:n_dims] = a * s + b * c
    return y.reshape(x.shape)


def sdpa_causal_gqa(q, k, v, n_head: int, n_head_kv: int, head_dim: int, scale: float,
                    rows=None, p0: int = 0) -> np.ndarray:
    """forward.rs, Model::forward, the attention step: causal, as many keys as
    queries, scale = 1/sqrt(head_dim):
    out[t, head i] = sum_{s <= t} softmax_s(q[t,i] . k[s,j] * scale) v[s,j],
    j = i // (n_head / n_head_kv).  q [T, n_head*hd], k/v [T, n_head_kv*hd].

    `rows` (optional) restricts the output to those query rows; each row
    is computed from the keys 0..row only, exactly as in the full result.

    p0 > 0: the query rows sit at positions p0, p0+1, ... and k/v hold the keys
    of positions 0 .. p0+T-1 (the earlier positions first), so query row r
    sees keys 0 .. p0+r: one chunk of a chunked prefill."""
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    T = q.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    group = n_head // n_head_kv
    out = np.zeros((len(rows), n_head * head_dim), dtype=F64)
    qpos = rows + p0                                     # position of each query row
    n_keys = int(qpos.max()) + 1 if len(rows) else 0
    key_idx = np.arange(n_keys)
    hidden = key_idx[None, :] > qpos[:, None]           # key s not visible to query t
    for i in range(n_head):
        j = i // group
        qi = q[rows, i * head_dim:(i + 1) * head_dim]
        kj = k[:n_keys, j * head_dim:(j + 1) * head_dim]
        vj = v[:n_keys, j * head_dim:(j + 1) * head_dim]
        s = (qi @ kj.T) * scale
        s[hidden] = -np.inf
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, i * head_dim:(i + 1) * head_dim] = p @ vj
    return out


def silu(x) -> np.ndarray:
    x = np.asarray(x, dtype=F64)
    return x / (1.0 + np.exp(-x))


def swiglu(gate, up) -> np.ndarray:
    """forward.rs, Model::forward, the FFN activation of the dense arm over
    t*n_ff values (the T-parallel page names the same step silu_mul):
    act = silu(gate) * up elementwise."""
    return silu(gate) * np.asarray(up, dtype=F64)


def linear(x, W) -> np.ndarray:
    """forward.rs, Model::forward, the projection matmul: W is [out_features,
    in_features] and x is token-major [T, in_features]; y = x W^T [T, out]."""
    return np.asarray(x, dtype=F64) @ np.asarray(W, dtype=F64).T


def bf16_fused_normed_linear(x, w_norm, W, eps: float) -> np.ndarray:
    """rms_norm(x) * w_norm followed by the projection W, with the rounding points
    of a norm fused into a bf16 GEMM: the GEMM multiplies bf16(x) by
    bf16(W * w_norm) (w_norm scales W's columns, i.e. the input features, before
    the rounding) and each output row is then scaled by 1/sqrt(mean(x^2) + eps),
    computed from the unrounded x.  Without the two roundings this equals
    linear(rms_norm(x, w_norm, eps), W)."""
    x = np.asarray(x, dtype=F64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    Wn = np.asarray(W, dtype=F64) * np.asarray(w_norm, dtype=F64)[None, :]
    return r * linear(round_bf16(x), round_bf16(Wn))


# --------------------------------------------------------------------------------------
# Whole forward
# --------------------------------------------------------------------------------------
def _mats(w: dict, rnd) -> dict:
    """Layer tensors in float64, every matrix passed through `rnd`."""
    out = {}
    for name, a in w.items():
        a = np.asarray(a, dtype=F64)
        out[name] = rnd(a) if a.ndim == 2 else a
    return out


def forward_layer(cfg, lw: dict, x, pos, bf16_operands: bool = False, kv_out=None,
                  kv_prefix=None, tf32_operands: bool = False,
                  fp8_operands: bool = False, bf16_fused_norm: bool = False,
                  rows=None) -> np.ndarray:
    """One decoder layer, forward.rs `Model::forward` loop body, on the residual
    stream x [T, n_embd]; returns the new x.  If `kv_out` is a list, the layer's
    attention inputs (k after QK-norm and RoPE, and v) are appended to it.

    `rows` (optional) returns only those rows of the new x [len(rows), n_embd]:
    keys and values come from every row of x, attention runs for the listed
    query rows only, and the O projection, residual and FFN, which act on each
    row alone, only for them.

    `kv_prefix` = (k, v) of the p0 positions before x (which then sits at
    positions pos = p0 .. p0+T-1): attention runs over those keys followed by
    x's own, the only way earlier positions reach later ones."""
    op, opm, opw, opa, opg = _rounders(bf16_operands, tf32_operands, fp8_operands)
    if bf16_fused_norm and not bf16_operands:
        raise ValueError("bf16_fused_norm needs bf16_operands")
    if bf16_fused_norm:     # the normed projections round W * w themselves
        lw_rest = {n: a for n, a in lw.items() if n not in ("wq", "wk", "wv", "w_gate", "w_up")}
        L = _mats(lw_rest, opw)
    else:
        L = _mats(lw, opw)
    d, h, g, hd = cfg.n_embd, cfg.n_head, cfg.n_head_kv, cfg.head_dim
    eps = cfg.rms_eps
    scale = 1.0 / np.sqrt(F64(hd))

    def normed_linears(xin, w_norm, names):
        """rms_norm(xin) * w_norm followed by each matrix.  With bf16_fused_norm
        the matrix input is bf16(xin), the norm weight multiplies the matrix's
        columns before its bf16 rounding, and the row's 1/rms scales the product
        -- the same function of xin, with those rounding points."""
        if bf16_fused_norm:
            return [bf16_fused_normed_linear(xin, w_norm, lw[n], eps) for n in names]
        hn = op(rms_norm(xin, w_norm, eps))
        return [linear(hn, L[n]) for n in names]

    # attention block
    q, k, v = normed_linears(x, lw["attn_norm"], ("wq", "wk", "wv"))
    gate = None
    if getattr(cfg, "attn_gate", False):
        qg = q.reshape(q.shape[0], h, 2, hd)
        q, gate = qg[:, :, 0, :].reshape(-1, h * hd), opg(qg[:, :, 1, :].reshape(-1, h * hd))
    q = qk_norm(q, L["q_norm"], hd, eps)
    k = qk_norm(k, L["k_norm"], hd, eps)
    q = opa(rope_neox(q, pos, h, hd, cfg.rope_dim_count, cfg.rope_freq_base))
    k = opa(rope_neox(k, pos, g, hd, cfg.rope_dim_count, cfg.rope_freq_base))
    v = opa(v)
    if kv_out is not None:
        kv_out.append((k, v))
    p0 = 0
    if kv_prefix is not None:
        p0 = kv_prefix[0].shape[0]
        k = np.concatenate([np.asarray(kv_prefix[0], dtype=F64), k])
        v = np.concatenate([np.asarray(kv_prefix[1], dtype=F64), v])
    if rows is not None:
        rows = np.asarray(rows)
        x = np.asarray(x, dtype=F64)[rows]
        gate = None if gate is None else gate[rows]
    attn = sdpa_causal_gqa(q, k, v, h, g, hd, scale, rows=rows, p0=p0)
    if gate is not None:
        attn = attn / (1.0 + np.exp(-gate))          # attn * sigmoid(gate)
    attn = opm(attn)
    x1 = x + linear(attn, L["wo"])
    # ffn block (dense SwiGLU)
    gt, up = normed_linears(x1, lw["ffn_norm"], ("w_gate", "w_up"))
    act = opm(swiglu(gt, up))
    return x1 + linear(act, L["w_down"])


def forward(cfg, weights: dict, tokens, bf16_operands: bool = False, return_hidden: bool = False,
            layer_source=None, kv_out=None, tf32_operands: bool = False,
            fp8_operands: bool = False, bf16_fused_norm: bool = False):
    """forward.rs `Model::forward`: logits [T, n_vocab] for `tokens`, positions 0..T-1.

    weights: {"tok_embd" [V,d], "layers": [dict per layer], "output_norm" [d],
    "output" [V,d]}.  `layer_source(l)` may replace weights["layers"][l] (lets a
    caller stream layers of a large model).  `kv_out` (a list) collects every
    layer's (k, v) as in forward_layer.  With return_hidden, also returns
    hidden [n_layer+1, T, d]: the residual stream entering each layer, then the
    stream entering output_norm."""
    tokens = np.asarray(tokens, dtype=np.int64)
    T = tokens.shape[0]
    op, _, opw, _, _ = _rounders(bf16_operands, tf32_operands, fp8_operands)
    emb = np.asarray(weights["tok_embd"], dtype=F64)
    x = emb[tokens]
    if bf16_operands or fp8_operands:       # the table is stored as bf16
        x = round_bf16(x)
    pos = np.arange(T)
    hidden = [x.copy()] if return_hidden else None
    for l in range(cfg.n_layer):
        lw = layer_source(l) if layer_source is not None else weights["layers"][l]
        x = forward_layer(cfg, lw, x, pos, bf16_operands, kv_out, tf32_operands=tf32_operands,
                          fp8_operands=fp8_operands, bf16_fused_norm=bf16_fused_norm)
        if return_hidden:
            hidden.append(x.copy())
    hn = op(rms_norm(x, np.asarray(weights["output_norm"], dtype=F64), cfg.rms_eps))
    logits = linear(hn, opw(np.asarray(weights["output"], dtype=F64)))
    if return_hidden:
        return logits, np.stack(hidden)
    return logits


def forward_chunk(cfg, weights: dict, tokens, kv_state: list, bf16_operands: bool = False,
                  tf32_operands: bool = False, fp8_operands: bool = False,
                  bf16_fused_norm: bool = False):
    """Chunked prefill: logits [C, n_vocab] for the next C tokens of a sequence
    whose first p0 positions went through earlier calls.  forward.rs
    `Model::forward` is causal, so those positions reach these only through
    each layer's keys and values: kv_state holds, per layer, the (k, v) of
    positions 0..p0-1 (empty list on the first chunk) and is extended in place
    with this chunk's.  The chunks' logits, concatenated, are forward(tokens)'s."""
    tokens = np.asarray(tokens, dtype=np.int64)
    C = tokens.shape[0]
    op, _, opw, _, _ = _rounders(bf16_operands, tf32_operands, fp8_operands)
    first = len(kv_state) == 0
    p0 = 0 if first else kv_state[0][0].shape[0]
    x = np.asarray(weights["tok_embd"], dtype=F64)[tokens]
    if bf16_operands or fp8_operands:
        x = round_bf16(x)
    pos = p0 + np.arange(C)
    for l in range(cfg.n_layer):
        new = []
        prefix = None if first else kv_state[l]
        x = forward_layer(cfg, weights["layers"][l], x, pos, bf16_operands, new, prefix,
                          tf32_operands, fp8_operands, bf16_fused_norm)
        k, v = new[0]
        if first:
            kv_state.append((k, v))
        else:
            kv_state[l] = (np.concatenate([kv_state[l][0], k]),
                           np.concatenate([kv_state[l][1], v]))
    hn = op(rms_norm(x, np.asarray(weights["output_norm"], dtype=F64), cfg.rms_eps))
    return linear(hn, opw(np.asarray(weights["output"], dtype=F64)))


# --------------------------------------------------------------------------------------
# Logit helpers (forward.rs `argmax`, `top2`, `prime_gate_verdict`)
# --------------------------------------------------------------------------------------
def argmax(logits) -> int:
    """First index holding the maximum (a strict `>` scan keeps the lowest index on ties)."""
    best, bv = 0, -np.inf
    for i, v in enumerate(np.asarray(logits).tolist()):
        if v > bv:
            bv, best = v, i
    return best


def top2(logits):
    """(i1, v1, i2, v2): the largest and second-largest entries, first index on ties."""
    i1, v1, i2, v2 = 0, -np.inf, 0, -np.inf
    for i, v in enumerate(np.asarray(logits).tolist()):
        if v > v1:
            i2, v2 = i1, v1
            i1, v1 = i, v
        elif v > v2:
            i2, v2 = i, v
    return i1, v1, i2, v2


def prime_gate_verdict(reference, candidate, maxdiff_bound: float = 8.0, margin_bound: float = 1.0):
    """Classify two logit vectors: "structured" if the max |diff| is non-finite or
    above maxdiff_bound; else "match" if the argmaxes agree; else "near_tie_flip"
    if the reference's top1-top2 margin is within margin_bound; else
    "structured".  Returns (class, ref_argmax, cand_argmax, ref_margin, maxdiff)."""
    t1, tv1, _, tv2 = top2(reference)
    b1, _, _, _ = top2(candidate)
    diff = np.abs(np.asarray(reference, dtype=F64) - np.asarray(candidate, dtype=F64))
    maxdiff = float(diff.max()) if diff.size else 0.0
    margin = tv1 - tv2
    if not np.isfinite(maxdiff) or maxdiff > maxdiff_bound:
        cls = "structured"
    elif t1 == b1:
        cls = "match"
    elif margin <= margin_bound:
        cls = "near_tie_flip"
    else:
        cls = "structured"
    return cls, t1, b1, margin, maxdiff
