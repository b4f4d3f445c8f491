"""Per-op parity: each C-ABI entry point against the oracle on seeded inputs.

Tolerances: float32 kernels vs the float64 oracle at 2e-6 relative (a few
float32 roundings); bf16-output kernels at 1 bf16 ulp (2^-8 relative) on top of
that; the bf16 tensor-core GEMM gets exactly bf16 operands, so only the float32
accumulation differs (K * 2^-24 relative bound, 1e-5 used)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")


def t32(a):
    return torch.as_tensor(np.ascontiguousarray(a, np.float32), device=dev)


def bf16_round32(a):
    """float32 array rounded to bf16 values (as float32), via torch on the host."""
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def max_rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


# ----------------------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("rows,cols", [(1, 64), (7, 4096), (300, 1000), (5, 13)])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_rms_norm(dtp, rows, cols, ydt):
    x = synth.normal(1, 100, (rows, cols)) * 3
    w = synth.normal(1, 101, (cols,), mean=1.0, std=0.1)
    y = torch.empty((rows, cols), dtype=ydt, device=dev)
    dtp.rms_norm(t32(x), t32(w), y, 1e-6)
    ref = oracle.rms_norm(x, w, 1e-6)
    tol = 2e-6 if ydt == torch.float32 else 2 ** -8
    np.testing.assert_allclose(y.float().cpu().numpy(), ref, rtol=tol, atol=tol * 1e-3)


# ----------------------------------------------------------------------------- QK-norm + RoPE
@pytest.mark.parametrize("T,nh,hd,r", [(1, 2, 16, 16), (37, 4, 64, 64), (300, 3, 128, 64), (129, 8, 128, 128)])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_qk_norm_rope(dtp, T, nh, hd, r, dt):
    x = synth.normal(2, 200, (T, nh * hd))
    w = synth.normal(2, 201, (hd,), mean=1.0, std=0.1)
    xin = x if dt == torch.float32 else bf16_round32(x)
    xt = t32(xin).to(dt)
    dtp.qk_norm_rope_neox(xt, t32(w), None, nh, hd, r, 1e6, 1e-6)
    ref = oracle.rope_neox(oracle.qk_norm(xin, w, hd, 1e-6), np.arange(T), nh, hd, r, 1e6)
    tol = 3e-6 if dt == torch.float32 else 2 ** -8
    np.testing.assert_allclose(xt.float().cpu().numpy(), ref, rtol=tol, atol=tol * 4)


def test_rope_only_with_positions(dtp):
    T, nh, hd = 50, 2, 32
    x = synth.normal(3, 300, (T, nh * hd))
    pos = (np.arange(T) * 37 + 5).astype(np.int32)
    xt = t32(x)
    dtp.qk_norm_rope_neox(xt, None, torch.as_tensor(pos, device=dev), nh, hd, hd, 1e4, 1e-6)
    ref = oracle.rope_neox(x, pos, nh, hd, hd, 1e4)
    np.testing.assert_allclose(xt.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)


def test_rope_position_and_pair_indexing_bit_exact(dtp):
    """Recover, from the kernel's output alone, which position rotated each row
    and which dims were paired: both must equal the definition exactly."""
    T, nh, hd, r = 4096, 2, 16, 8
    base = 1e8     # theta_i = 1e8^(-2i/8): theta_3 = 1e-6, so T*theta_3 < pi (no wrap)
    half = r // 2
    x = np.zeros((T, nh, hd), np.float32)
    x[:, 0, 3] = 1.0          # one-hot at dim 3 (< half): pairs with dim 3 + half = 7
    x[:, 1, 9] = 1.0          # dim 9 >= r: passes through
    xt = t32(x.reshape(T, nh * hd))
    dtp.qk_norm_rope_neox(xt, None, None, nh, hd, r, base, 0.0)
    y = xt.cpu().numpy().reshape(T, nh, hd).astype(np.float64)
    nz0 = sorted(set(np.nonzero(np.abs(y[1:, 0]) > 0)[1].tolist()))
    assert nz0 == [3, 7]
    assert np.array_equal(y[:, 1], x[:, 1])
    theta = base ** (-2.0 * 3 / r)
    recovered = np.rint(np.arctan2(y[:, 0, 7], y[:, 0, 3]) / theta).astype(np.int64)
    assert np.array_equal(recovered, np.arange(T))


# ----------------------------------------------------------------------------- SwiGLU
@pytest.mark.parametrize("n", [1, 1000, 123457])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_swiglu(dtp, n, dt):
    g = synth.normal(4, 400, (n,)) * 4
    u = synth.normal(4, 401, (n,))
    if dt == torch.bfloat16:
        g, u = bf16_round32(g), bf16_round32(u)
    out = torch.empty(n, dtype=dt, device=dev)
    dtp.swiglu(t32(g).to(dt), t32(u).to(dt), out)
    ref = oracle.swiglu(g, u)
    tol = 2e-6 if dt == torch.float32 else 2 ** -8
    np.testing.assert_allclose(out.float().cpu().numpy(), ref, rtol=tol, atol=tol * 1e-3)


# ----------------------------------------------------------------------------- linear
@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (130, 200, 72), (256, 512, 512), (77, 1000, 136)])
@pytest.mark.parametrize("resid", [False, True])
def test_linear_f32(dtp, M, N, K, resid):
    x = synth.normal(5, 500, (M, K))
    W = synth.normal(5, 501, (N, K), std=0.05)
    r = synth.normal(5, 502, (M, N)) if resid else None
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    dtp.linear(t32(x), t32(W), y, residual=None if r is None else t32(r))
    ref = oracle.linear(x, W) + (r if resid else 0)
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=0, atol=2e-6 * np.abs(ref).max())


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (128, 256, 64), (130, 200, 72), (256, 768, 512),
                                   (300, 1000, 136), (513, 2048, 1024), (64, 384, 4096),
                                   (77, 1001, 136)])   # odd row stride: direct-store epilogue
@pytest.mark.parametrize("mode", ["f32", "bf16", "resid"])
def test_linear_bf16_tensor_core(dtp, M, N, K, mode):
    x = bf16_round32(synth.normal(6, 600, (M, K)))
    W = bf16_round32(synth.normal(6, 601, (N, K), std=0.05))
    xt, Wt = t32(x).bfloat16(), t32(W).bfloat16()
    ref = oracle.linear(x, W)
    if mode == "bf16":
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dtp.linear(xt, Wt, y)
        np.testing.assert_allclose(y.float().cpu().numpy(), ref, rtol=2 ** -8,
                                   atol=1e-5 * np.abs(ref).max())
        return
    r = synth.normal(6, 602, (M, N)) if mode == "resid" else None
    y = t32(r) if r is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    dtp.linear(xt, Wt, y, residual=y if r is not None else None)     # in-place residual add
    if r is not None:
        ref = ref + r
    torch.cuda.synchronize()
    dtp.check()
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=0, atol=1e-5 * np.abs(ref).max())


def test_linear_bf16_long_k_and_many_tiles(dtp):
    # several persistent waves of 128x256 tiles and a 12288-long reduction
    M, N, K = 1024, 4096, 12288
    x = bf16_round32(synth.normal(7, 700, (M, K)))
    W = bf16_round32(synth.normal(7, 701, (N, K), std=0.02))
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    dtp.linear(t32(x).bfloat16(), t32(W).bfloat16(), y)
    rows = np.array([0, 1, 127, 128, 500, 1023])
    ref = oracle.linear(x[rows], W)
    # tensor-core accumulation adds each K=16 partial product into float32 with up
    # to ~1 ulp of error per step: bound (K/16) * 2^-23 * max|y|, with a 2x margin
    tol = 2 * (K / 16) * 2.0 ** -23 * np.abs(ref).max()
    np.testing.assert_allclose(y.cpu().numpy()[rows], ref, rtol=0, atol=tol)


@pytest.mark.parametrize("M,N", [(1024, 5120), (1024, 5000), (1152, 4900), (1, 4096)])
@pytest.mark.parametrize("mode", ["f32", "bf16", "resid"])
def test_linear_bf16_cluster_pairs(dtp, M, N, mode):
    """The GEMM runs as CTA pairs on M-adjacent tiles, each CTA loading half of
    the shared weight box for both.  More tiles than SMs, a ragged last N block
    (N = 5000, 4900), an odd number of M blocks (1152 = 9 x 128: the last pair's
    second tile lies wholly past M) and a single row."""
    K = 512
    x = bf16_round32(synth.normal(16, 1600, (M, K)))
    W = bf16_round32(synth.normal(16, 1601, (N, K), std=0.05))
    xt, Wt = t32(x).bfloat16(), t32(W).bfloat16()
    ref = oracle.linear(x, W)
    if mode == "bf16":
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dtp.linear(xt, Wt, y)
        torch.cuda.synchronize()
        dtp.check()
        np.testing.assert_allclose(y.float().cpu().numpy(), ref, rtol=2 ** -8,
                                   atol=1e-5 * np.abs(ref).max())
        return
    r = synth.normal(16, 1602, (M, N)) if mode == "resid" else None
    y = t32(r) if r is not None else torch.full((M, N), float("nan"), device=dev)
    dtp.linear(xt, Wt, y, residual=y if r is not None else None)
    torch.cuda.synchronize()
    dtp.check()
    if r is not None:
        ref = ref + r
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=0, atol=1e-5 * np.abs(ref).max())


# ----------------------------------------------------------------------------- attention
@pytest.mark.parametrize("T,nh,nkv,hd", [(1, 4, 2, 16), (17, 4, 2, 64), (130, 8, 4, 64), (300, 4, 1, 128)])
def test_sdpa_f32(dtp, T, nh, nkv, hd):
    q = synth.normal(8, 800, (T, nh * hd))
    k = synth.normal(8, 801, (T, nkv * hd))
    v = synth.normal(8, 802, (T, nkv * hd))
    out = torch.empty((T, nh * hd), dtype=torch.float32, device=dev)
    sc = 1 / math.sqrt(hd)
    dtp.sdpa_causal_gqa(t32(q), t32(k), t32(v), out, nh, nkv, hd, sc)
    ref = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, sc)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=2e-6 * np.abs(ref).max())


def test_sdpa_gqa_head_map_bit_exact(dtp):
    """v of kv head j is the constant j, so each output head must read back
    exactly the kv head the definition assigns: j = i // (n_head / n_head_kv)."""
    T, nh, nkv, hd = 64, 8, 2, 16
    q = synth.normal(9, 900, (T, nh * hd))
    k = synth.normal(9, 901, (T, nkv * hd))
    v = np.repeat(np.arange(nkv, dtype=np.float32), hd)[None, :].repeat(T, 0)
    out = torch.empty((T, nh * hd), dtype=torch.float32, device=dev)
    dtp.sdpa_causal_gqa(t32(q), t32(k), t32(v), out, nh, nkv, hd, 0.25)
    got = np.rint(out.cpu().numpy().reshape(T, nh, hd)).astype(int)
    want = (np.arange(nh) // (nh // nkv))[None, :, None].repeat(T, 0).repeat(hd, 2)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------------------- tcgen05 attention
def _sdpa_bf16(dtp, q, k, v, nh, nkv, hd):
    T = q.shape[0]
    out = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_BF16), dtype=torch.uint8, device=dev)
    dtp.sdpa_causal_gqa(t32(q).bfloat16(), t32(k).bfloat16(), t32(v).bfloat16(), out, nh, nkv, hd,
                        1 / math.sqrt(hd), ws)
    torch.cuda.synchronize()
    dtp.check()
    return out.float().cpu().numpy()


def _attn_close(got, ref, vmax):
    # P is rounded to bf16 for the PV product (2^-9 relative) and so is the output
    err = np.abs(got - ref)
    assert err.max() <= 8e-3 * vmax, err.max()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 3e-3


@pytest.mark.parametrize("T,nh,nkv,hd", [(1, 4, 2, 128), (100, 4, 2, 64), (128, 8, 4, 128),
                                         (129, 4, 1, 64), (300, 8, 2, 128), (1024, 16, 8, 128)])
def test_sdpa_bf16_tensor_core(dtp, T, nh, nkv, hd):
    q = bf16_round32(synth.normal(10, 1000, (T, nh * hd)))
    k = bf16_round32(synth.normal(10, 1001, (T, nkv * hd)))
    v = bf16_round32(synth.normal(10, 1002, (T, nkv * hd)))
    got = _sdpa_bf16(dtp, q, k, v, nh, nkv, hd)
    ref = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 1 / math.sqrt(hd))
    _attn_close(got, ref, np.abs(v).max())


def test_sdpa_bf16_large_scores_rescale(dtp):
    # scores spread over hundreds of log2 units across key tiles: exercises the
    # running-max rescale of O in TMEM
    T, nh, nkv, hd = 640, 2, 1, 64
    q = bf16_round32(synth.normal(11, 1100, (T, nh * hd)) * 6)
    k = bf16_round32(synth.normal(11, 1101, (T, nkv * hd)) * 6 * np.linspace(0.2, 2.0, T)[:, None])
    v = bf16_round32(synth.normal(11, 1102, (T, nkv * hd)))
    got = _sdpa_bf16(dtp, q, k, v, nh, nkv, hd)
    ref = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, 1 / math.sqrt(hd))
    _attn_close(got, ref, np.abs(v).max())


def test_sdpa_bf16_gqa_head_map_bit_exact(dtp):
    T, nh, nkv, hd = 200, 8, 2, 64
    q = bf16_round32(synth.normal(12, 1200, (T, nh * hd)))
    k = bf16_round32(synth.normal(12, 1201, (T, nkv * hd)))
    v = np.repeat(np.array([3.0, 7.0], np.float32), hd)[None, :].repeat(T, 0)
    got = np.rint(_sdpa_bf16(dtp, q, k, v, nh, nkv, hd).reshape(T, nh, hd)).astype(int)
    want = np.array([3, 3, 3, 3, 7, 7, 7, 7])[None, :, None].repeat(T, 0).repeat(hd, 2)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("T", [1024, 4096, 8192, 16384])
@pytest.mark.parametrize("r", [64, 128])
def test_attention_sweep(dtp, T, r):
    """Causal GQA SDPA with QK-norm + NeoX RoPE, h=32, g=8, hd=128, q/k/v ~ N(0,1)
    in bf16; checked on sampled query rows (each computed by the oracle from
    all keys up to it) including the first and last tiles."""
    sw = synth.ATTN_SWEEP
    nh, nkv, hd = sw["n_head"], sw["n_head_kv"], sw["head_dim"]
    inp = synth.attention_inputs(T, nh, nkv, hd)
    q, k, v = (bf16_round32(inp[n]) for n in ("q", "k", "v"))
    qt, kt, vt = t32(q).bfloat16(), t32(k).bfloat16(), t32(v).bfloat16()
    base, eps = sw["rope_freq_base"], sw["rms_eps"]
    dtp.qk_norm_rope_neox(qt, t32(inp["q_norm"]), None, nh, hd, r, base, eps)
    dtp.qk_norm_rope_neox(kt, t32(inp["k_norm"]), None, nkv, hd, r, base, eps)
    out = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_BF16), dtype=torch.uint8, device=dev)
    dtp.sdpa_causal_gqa(qt, kt, vt, out, nh, nkv, hd, 1 / math.sqrt(hd), ws)
    torch.cuda.synchronize()
    dtp.check()
    rows = np.unique(np.concatenate([[0, 1, 127, 128, T // 2, T - 129, T - 2, T - 1],
                                     np.random.default_rng(T + r).integers(0, T, 8)]))
    pos = np.arange(T)
    qr = oracle.round_bf16(oracle.rope_neox(oracle.qk_norm(q, inp["q_norm"], hd, eps), pos, nh, hd, r, base))
    kr = oracle.round_bf16(oracle.rope_neox(oracle.qk_norm(k, inp["k_norm"], hd, eps), pos, nkv, hd, r, base))
    ref = oracle.sdpa_causal_gqa(qr, kr, v, nh, nkv, hd, 1 / math.sqrt(hd), rows=rows)
    got = out.float().cpu().numpy()[rows]
    _attn_close(got, ref, np.abs(v).max())


# ----------------------------------------------------------------------------- fused epilogues
@pytest.mark.parametrize("T,d,nh,nkv,hd,r", [(1, 64, 2, 1, 64, 64), (130, 512, 8, 4, 64, 64),
                                              (300, 1024, 4, 2, 128, 64), (257, 512, 8, 2, 128, 128),
                                              # more tiles than SMs (8 x 24, 32 x 6)
                                              (1024, 512, 32, 8, 128, 128), (4096, 256, 16, 4, 64, 64)])
def test_qkv_norm_rope_fused(dtp, T, d, nh, nkv, hd, r):
    """QKV GEMM with per-head RMSNorm + NeoX RoPE in its epilogue, against the oracle
    on the same bf16 operands; outputs agree to one bf16 rounding."""
    nq, nk = nh * hd, nkv * hd
    h = bf16_round32(synth.normal(13, 1300, (T, d)))
    W = bf16_round32(synth.normal(13, 1301, (nq + 2 * nk, d), std=0.05))
    qn = synth.normal(13, 1302, (hd,), mean=1.0, std=0.1)
    kn = synth.normal(13, 1303, (hd,), mean=1.0, std=0.1)
    q = torch.empty((T, nq), dtype=torch.bfloat16, device=dev)
    k = torch.empty((T, nk), dtype=torch.bfloat16, device=dev)
    ldvt = (T + 7) // 8 * 8
    vt = torch.zeros((nk, ldvt), dtype=torch.float16, device=dev)     # f16 copies of bf16(v)
    dtp.qkv_norm_rope(t32(h).bfloat16(), t32(W).bfloat16(), t32(qn), t32(kn), q, k, vt, nh, nkv, hd,
                      r, 1e6, 1e-6)
    torch.cuda.synchronize()
    dtp.check()
    qkv = oracle.linear(h, W)
    pos = np.arange(T)
    rq = oracle.round_bf16(oracle.rope_neox(oracle.qk_norm(qkv[:, :nq], qn, hd, 1e-6), pos, nh, hd, r, 1e6))
    rk = oracle.round_bf16(oracle.rope_neox(oracle.qk_norm(qkv[:, nq:nq + nk], kn, hd, 1e-6), pos, nkv, hd, r, 1e6))
    rv = oracle.round_bf16(qkv[:, nq + nk:])
    np.testing.assert_allclose(q.float().cpu().numpy(), rq, rtol=2 ** -7, atol=1e-5)
    np.testing.assert_allclose(k.float().cpu().numpy(), rk, rtol=2 ** -7, atol=1e-5)
    vt_got = vt.float().cpu().numpy()[:, :T].T
    np.testing.assert_allclose(vt_got, rv, rtol=2 ** -7, atol=1e-5)
    assert np.array_equal(oracle.round_bf16(vt_got), vt_got)     # f16 of bf16 values: still bf16 values
    assert not vt[:, T:].any()                       # padding columns untouched


@pytest.mark.parametrize("hd,r", [(128, 64), (64, 64), (128, 128)])
def test_qkv_epilogue_rope_position_and_pair_indexing_bit_exact(dtp, hd, r):
    """The forward pass's own RoPE (the fused QKV epilogue, T = 4096): every token
    feeds the same q/k row, whose first r/2 dims are 1 and the rest of the
    rotated half 0, so after the QK-norm pair (i, i + r/2) holds c (cos, sin)(pos *
    theta_i), c = 1 / rms(row).  From the bf16 outputs alone, the integer
    position that best explains each row's r/2 angles must be the row's own
    index, every pair's angle must match it, and dims >= r must not rotate."""
    T, d, nh, nkv = 4096, 64, 2, 1
    half, base = r // 2, 1e4
    nq, nk = nh * hd, nkv * hd
    pattern = np.zeros(hd)
    pattern[:half] = 1.0
    pattern[r:] = np.linspace(0.5, 1.5, hd - r)        # pass-through dims
    W = np.zeros((nq + 2 * nk, d), np.float32)
    for head in range(nh + nkv):                        # q heads, then the k head
        W[head * hd:(head + 1) * hd, 0] = pattern
    W[nq + nk:, 0] = 1.0                                # v: untouched by the epilogue's RoPE
    h = np.zeros((T, d), np.float32)
    h[:, 0] = 1.0                                       # every token: q = k = pattern
    q = torch.empty((T, nq), dtype=torch.bfloat16, device=dev)
    k = torch.empty((T, nk), dtype=torch.bfloat16, device=dev)
    vt = torch.zeros((nk, T), dtype=torch.float16, device=dev)
    ones = t32(np.ones(hd, np.float32))
    dtp.qkv_norm_rope(t32(h).bfloat16(), t32(W).bfloat16(), ones, ones, q, k, vt, nh, nkv, hd,
                      r, base, 1e-6)
    torch.cuda.synchronize()
    dtp.check()
    theta = base ** (-2.0 * np.arange(half) / r)
    cand = np.exp(1j * np.arange(T)[:, None] * theta[None, :])       # [position, pair]
    rows = np.concatenate([q.float().cpu().numpy().reshape(T, nh, hd),
                           k.float().cpu().numpy().reshape(T, nkv, hd)], axis=1)
    for head in range(nh + nkv):
        y = rows[:, head].astype(np.float64)
        ang = np.arctan2(y[:, half:r], y[:, :half])                    # [row, pair]
        score = np.real(np.exp(1j * ang) @ cand.conj().T)               # [row, position]
        assert np.array_equal(np.argmax(score, axis=1), np.arange(T)), head
        err = np.angle(np.exp(1j * (ang - np.arange(T)[:, None] * theta[None, :])))
        assert np.abs(err).max() <= 2e-2, (head, np.abs(err).max())    # bf16: ~2^-8 rad
        np.testing.assert_allclose(np.hypot(y[:, half:r], y[:, :half]),
                                   1 / np.sqrt(np.mean(pattern ** 2) + 1e-6), rtol=2 ** -7)
        if r < hd:                                     # scaled by the norm only, never rotated
            ratio = y[:, r:] / pattern[r:]
            np.testing.assert_allclose(ratio, ratio[:, :1].repeat(hd - r, 1), rtol=2 ** -7)


@pytest.mark.parametrize("T,d,F", [(1, 64, 64), (200, 512, 1536), (513, 1024, 3072),
                                   (1024, 256, 2560)])   # 8 x 20 tiles: more than SMs
def test_gate_up_swiglu_fused(dtp, T, d, F):
    """gate/up GEMM with SwiGLU in its epilogue on the interleaved weight layout."""
    z = bf16_round32(synth.normal(14, 1400, (T, d)))
    Wg = bf16_round32(synth.normal(14, 1401, (F, d), std=0.05))
    Wu = bf16_round32(synth.normal(14, 1402, (F, d), std=0.05))
    W = np.empty((2 * F, d), np.float32)
    for b in range(F // 64):                          # the layout dtp_pack_layer writes
        W[128 * b:128 * b + 64] = Wg[64 * b:64 * b + 64]
        W[128 * b + 64:128 * b + 128] = Wu[64 * b:64 * b + 64]
    act = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
    dtp.gate_up_swiglu(t32(z).bfloat16(), t32(W).bfloat16(), act)
    torch.cuda.synchronize()
    dtp.check()
    ref = oracle.round_bf16(oracle.swiglu(oracle.linear(z, Wg), oracle.linear(z, Wu)))
    np.testing.assert_allclose(act.float().cpu().numpy(), ref, rtol=2 ** -7, atol=1e-5)


def test_bounded_wait_gives_up_and_context_survives(dtp):
    """A pipeline wait on a barrier nothing arrives at ends with an error status
    instead of a hang; the context stays usable afterwards."""
    dtp.selftest_wait_timeout()
    with pytest.raises(dtp.DtpError) as e:
        dtp.check()
    assert e.value.code == -6
    dtp.check()                                      # cleared
    x = bf16_round32(synth.normal(15, 1500, (64, 128)))
    W = bf16_round32(synth.normal(15, 1501, (256, 128)))
    y = torch.empty((64, 256), dtype=torch.float32, device=dev)
    dtp.linear(t32(x).bfloat16(), t32(W).bfloat16(), y)
    torch.cuda.synchronize()
    dtp.check()
    np.testing.assert_allclose(y.cpu().numpy(), oracle.linear(x, W), rtol=0, atol=1e-4)
