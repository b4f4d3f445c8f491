"""The seeded input generator: reproducible, slice-consistent, right distributions."""
import numpy as np

import synth


def test_streams_are_reproducible_and_slice_consistent():
    a = synth.normal(0, 77, (10001,), std=0.02)
    assert np.array_equal(a, synth.normal(0, 77, (10001,), std=0.02))
    for start, n in [(0, 1), (1, 1), (3, 10), (9990, 11), (5000, 1)]:
        assert np.array_equal(synth.normal(0, 77, (n,), std=0.02, start=start), a[start:start + n])
    assert not np.array_equal(a, synth.normal(1, 77, (10001,), std=0.02))
    assert not np.array_equal(a, synth.normal(0, 78, (10001,), std=0.02))


def test_normal_moments():
    x = synth.normal(3, 5, (2_000_000,)).astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 1) < 3e-3
    assert abs(np.mean(x ** 3)) < 1e-2 and abs(np.mean(x ** 4) - 3) < 3e-2
    w = synth.normal(3, 6, (100000,), mean=1.0, std=0.1).astype(np.float64)
    assert abs(w.mean() - 1) < 2e-3 and abs(w.std() - 0.1) < 2e-3


def test_uniform_tokens():
    t = synth.uniform_int(0, synth.TID_TOKENS, 512000, 256)
    assert t.min() == 0 and t.max() == 255
    c = np.bincount(t, minlength=256)
    assert c.min() > 1700 and c.max() < 2300
    cfg = synth.CONFIGS["qwen3-8b-shape"]
    toks = synth.tokens(cfg)
    assert toks.shape == (4096,) and toks.max() < cfg.n_vocab


def test_config_flop_counts():
    # algorithmic work per config: GEMM = 2*T*params (no embedding), attention = L*h*2*hd*T*(T+1)
    c = synth.CONFIGS["qwen3-8b-shape"]
    assert abs(c.gemm_flops() / 6.200e13 - 1) < 1e-3
    assert abs(c.attn_flops() / 4.949e12 - 1) < 1e-3
    s = synth.CONFIGS["small"]
    assert abs((s.gemm_flops() + s.attn_flops()) / 1.510e10 - 1) < 1e-3


def test_bf16_bits_round_trip():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5], np.float32)
    assert np.array_equal(synth.from_bf16_bits(synth.to_bf16_bits(x)),
                          np.array([1.0, 1.0, 1.015625, -2.5], np.float32))
