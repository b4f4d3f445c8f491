"""The C-ABI library without a GPU: it loads, exports every function that
include/dtp.h declares, and rejects bad arguments on the host before touching
the device."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dtp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dtp_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dtp_fwd_prefill", "dtp_rms_norm", "dtp_qk_norm_rope_neox", "dtp_sdpa_causal_gqa",
              "dtp_swiglu", "dtp_linear", "dtp_check", "dtp_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(dtp):
    lib = ctypes.CDLL(dtp.build())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(dtp, name="small", **kw):
    return dtp.config_from(synth.CONFIGS[name].replace(**kw))


def test_host_batch_workspace_buys_logit_buffers(dtp):
    """Each logit buffer past the two of dtp_workspace_size_host_batch adds one
    T x n_vocab float32 block (rounded up to the 256-byte alignment); counts
    outside 2..8 size to 0."""
    c = _cfg(dtp)
    T = 200
    block = (T * c.n_vocab * 4 + 255) // 256 * 256
    two = dtp.workspace_size_host_batch(c, T)
    assert two > dtp.workspace_size_host(c, T)
    for nb in range(2, 9):
        assert dtp.workspace_size_host_batch(c, T, nb) == two + (nb - 2) * block
    assert dtp.workspace_size_host_batch(c, T, 1) == 0
    assert dtp.workspace_size_host_batch(c, T, 9) == 0


def test_sizes_and_config_validation(dtp):
    c = _cfg(dtp)
    assert dtp.packed_size(c) > 0 and dtp.workspace_size(c, 256) > 0
    assert dtp.workspace_size_host(c, 256) > dtp.workspace_size(c, 256)
    assert dtp.workspace_size(c, 0) == 0
    for bad in (dict(n_head=7), dict(rope_dim_count=3), dict(rope_dim_count=200), dict(n_embd=0),
                dict(head_dim=48)):   # 48: not tiled by the bf16 path
        assert dtp.packed_size(_cfg(dtp, **bad)) == 0
        assert dtp.last_error()
    # float32 path accepts any even head_dim
    assert dtp.packed_size(_cfg(dtp, head_dim=48, rope_dim_count=48, precision="f32")) > 0


def test_packed_size_is_the_sum_of_tensors(dtp):
    cfg = synth.CONFIGS["qwen3-8b-shape"]
    n = dtp.packed_size(dtp.config_from(cfg))
    params = cfg.n_layer * (cfg.n_qkv * cfg.n_embd + cfg.n_embd * cfg.n_head * cfg.head_dim
                            + 3 * cfg.n_ff * cfg.n_embd) + 2 * cfg.n_vocab * cfg.n_embd
    assert 2 * params <= n <= 2 * params + 4 * (cfg.n_layer * (2 * cfg.n_embd + 2 * cfg.head_dim)
                                                + cfg.n_embd) + 256 * (12 * cfg.n_layer + 3)


def test_host_side_rejections(dtp):
    L = dtp.lib()
    c = _cfg(dtp)
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails validation first
    assert L.dtp_fwd_prefill(None, fake, 1 << 40, fake, 4, fake, None, fake, 1 << 40, None) == -1
    assert L.dtp_fwd_prefill(ctypes.byref(c), fake, 1 << 40, fake, 0, fake, None, fake, 1 << 40, None) == -1
    assert L.dtp_fwd_prefill(ctypes.byref(c), None, 1 << 40, fake, 4, fake, None, fake, 1 << 40, None) == -1
    assert L.dtp_fwd_prefill(ctypes.byref(c), fake, 16, fake, 4, fake, None, fake, 1 << 40, None) == -4
    assert L.dtp_fwd_prefill(ctypes.byref(c), fake, 1 << 40, fake, 4, fake, None, fake, 16, None) == -4
    assert "workspace" in dtp.last_error()
    toks = (ctypes.c_uint32 * 4)(1, 2, 40000, 3)       # 40000 >= n_vocab 32000
    logits = (ctypes.c_float * 4)()
    assert L.dtp_fwd_prefill_host(ctypes.byref(c), fake, 1 << 40, toks, 4, logits, fake, 1 << 40, None) == -3
    assert "40000" in dtp.last_error()
    assert L.dtp_rms_norm(None, fake, fake, 0, 4, 4, 1e-6, None) == -1
    assert L.dtp_rms_norm(fake, fake, fake, 0, 0, 4, 1e-6, None) == -1
    assert L.dtp_qk_norm_rope_neox(fake, 0, None, None, 4, 2, 16, 17, 1e4, 1e-6, None) == -1
    assert L.dtp_sdpa_causal_gqa(fake, fake, fake, fake, 0, 8, 6, 4, 16, 0.25, None, 0, None) == -1
    assert L.dtp_sdpa_causal_gqa(fake, fake, fake, fake, 1, 8, 8, 8, 32, 0.25, None, 0, None) == -2
    assert L.dtp_linear(fake, fake, fake, 0, 0, 0, 4, 4, None, None) == -1
    assert L.dtp_linear(fake, fake, fake, 1, 1, 4, 4, 4, fake, None) == -1   # residual needs f32 out
    assert L.dtp_linear(fake, fake, fake, 1, 0, 4, 4, 12, None, None) == -2  # K % 8
    assert L.dtp_timer_read(99, None, None) == -1
    assert dtp.workspace_size_varlen(c, 256, 4) > dtp.workspace_size(c, 256)
    assert dtp.workspace_size_varlen(c, 256, 0) == 0
    outs = dtp._binding.FwdOutputs(0x10000, 0, None, None, None)
    assert L.dtp_fwd_prefill_varlen(ctypes.byref(c), fake, 1 << 40, fake, None, 2, 256,
                                    ctypes.byref(outs), fake, 1 << 40, None) == -1
    assert L.dtp_fwd_prefill_varlen(ctypes.byref(c), fake, 1 << 40, fake, fake, 0, 256,
                                    ctypes.byref(outs), fake, 1 << 40, None) == -1


def test_chunk_state_size_and_rejections(dtp):
    """dtp_kv_state_size follows the documented layout; dtp_fwd_prefill_chunk
    rejects bad ranges and buffers before enqueueing anything."""
    L = dtp.lib()
    up = lambda x, a: (x + a - 1) // a * a
    for prec in ("bf16", "e4m3", "tf32", "f32"):
        cfg = synth.CONFIGS["small"].replace(precision=prec)
        c = dtp.config_from(cfg)
        nk = cfg.n_head_kv * cfg.head_dim
        for max_T in (1, 100, 256, 4099):
            if prec != "f32":           # K then V^T
                eb = 4 if prec == "tf32" else 2
                per = up(max_T * nk * eb, 256) + up(nk * up(max_T, 8) * eb, 256)
            else:
                per = 2 * up(max_T * nk * 4, 256)
            assert dtp.kv_state_size(c, max_T) == cfg.n_layer * per
        assert dtp.kv_state_size(c, 0) == 0
    c = _cfg(dtp)
    fake = ctypes.c_void_p(0x10000)   # never dereferenced
    big = 1 << 40
    outs = dtp._binding.FwdOutputs(0x10000, 0, None, None, None)
    call = lambda C, p0, max_T, sb=big, o=outs, st=fake: L.dtp_fwd_prefill_chunk(
        ctypes.byref(c), fake, big, fake, C, p0, st, sb, max_T, ctypes.byref(o), fake, big, None)
    assert call(0, 0, 64) == -1                      # empty chunk
    assert call(16, -1, 64) == -1                    # negative start
    assert call(16, 50, 64) == -1                    # runs past max_T
    assert "max_T" in dtp.last_error()
    assert call(16, 0, 64, st=None) == -1
    assert call(16, 0, 64, st=ctypes.c_void_p(0x10010)) == -1      # not 256-byte aligned
    assert call(16, 0, 64, sb=dtp.kv_state_size(c, 64) - 1) == -4   # short state
    kv = dtp._binding.FwdOutputs(0x10000, 0, None, 0x10000, None)
    assert call(16, 0, 64, o=kv) == -1               # the state is the cache


def test_e4m3_entry_points_reject_on_the_host(dtp):
    L = dtp.lib()
    fake = ctypes.c_void_p(0x10000)   # never dereferenced
    assert L.dtp_linear_e4m3(fake, fake, fake, fake, fake, 4, 4, 24, None, None) == -2   # K % 16
    assert L.dtp_linear_e4m3(None, fake, fake, fake, fake, 4, 4, 32, None, None) == -1
    assert L.dtp_linear_e4m3(fake, fake, fake, fake, fake, 0, 4, 32, None, None) == -1
    assert L.dtp_quantize_rows_e4m3(fake, 7, 4, 16, fake, fake, None) == -1             # dtype
    assert L.dtp_quantize_rows_e4m3(fake, 1, 4, 12, fake, fake, None) == -2             # bf16 cols % 8
    assert L.dtp_rms_norm_e4m3(fake, fake, fake, fake, 4, 6, 1e-6, None) == -2          # cols % 4
    # e4m3 configs: the tensor-core tiling rules of the bf16 path
    c = _cfg(dtp, precision="e4m3")
    assert dtp.packed_size(c) > 0 and dtp.workspace_size(c, 256) > dtp.workspace_size(_cfg(dtp), 256)
    assert dtp.packed_size(_cfg(dtp, precision="e4m3", head_dim=48)) == 0
    # packed e4m3 weights: 1 byte per matrix element, a float32 scale per row
    cfg = synth.CONFIGS["qwen3-8b-shape"]
    n8 = dtp.packed_size(dtp.config_from(cfg.replace(precision="e4m3")))
    n16 = dtp.packed_size(dtp.config_from(cfg))
    emb = cfg.n_vocab * cfg.n_embd * 2
    assert abs((n8 - emb) / (n16 - emb) - 0.5) < 0.01
