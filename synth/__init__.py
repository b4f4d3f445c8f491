"""Seeded synthetic inputs for the dense prefill forward pass.

This module is the one piece shared by the CUDA path's tests/bench and the CPU
oracle.  It draws inputs only -- weights, norm scales, token ids and attention
operands -- and holds none of the forward pass's arithmetic.

Distributions follow the workload descriptions: every matrix (embedding,
projections, FFN, lm_head) is N(0, 0.02); every norm scale vector is
1 + N(0, 0.1); token ids are uniform in [0, n_vocab); attention-sweep operands
are N(0, 1).  Each tensor is its own counter-based stream (SplitMix64 +
Box-Muller, see synth.c) keyed by (seed, tensor id).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                             ctypes.c_void_p]
            lib.synth_normal_f32.restype = None
            lib.synth_uniform_u32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                              ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p]
            lib.synth_uniform_u32.restype = None
            lib.synth_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_word.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def word(seed: int, tensor_id: int, counter: int) -> int:
    """Raw 64-bit word `counter` of stream (seed, tensor_id)."""
    return int(_load().synth_word(seed, tensor_id, counter))


def normal(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0,
           start: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """float32 array of `shape` = elements [start, start+size) of the stream."""
    n = int(np.prod(shape)) if len(tuple(shape)) else 1
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    if n:
        _load().synth_normal_f32(seed, tensor_id, start, n, float(mean), float(std),
                                 out.ctypes.data)
    return out


def uniform_int(seed: int, tensor_id: int, n: int, bound: int, start: int = 0) -> np.ndarray:
    """uint32 array of n integers uniform in [0, bound)."""
    out = np.empty((n,), dtype=np.uint32)
    if n:
        _load().synth_uniform_u32(seed, tensor_id, start, n, int(bound), out.ctypes.data)
    return out


# --------------------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Shape of a Qwen3-style dense decoder stack plus the prompt length T."""
    name: str
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    rope_dim_count: int
    n_ff: int
    n_vocab: int
    T: int
    rope_freq_base: float = 1e6
    rms_eps: float = 1e-6
    precision: str = "bf16"          # "f32" (exact), "tf32" or "bf16" (tf32 / bf16 GEMM
                                     # operands, f32 accumulate), "e4m3" (per-row e4m3
                                     # weights and GEMM inputs)
    attn_gate: bool = False          # sigmoid output gate fused into the Q projection

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)

    @property
    def n_qkv(self) -> int:
        """Rows of the fused QKV weight: q (and its gate, per head) + k + v."""
        return (self.n_head * (2 if self.attn_gate else 1) + 2 * self.n_head_kv) * self.head_dim

    def gemm_flops(self, T: int | None = None) -> float:
        """2*T*sum(out*in) over every projection, the FFN and the lm_head."""
        T = self.T if T is None else T
        d, hd = self.n_embd, self.head_dim
        per_layer = (self.n_qkv * d + d * self.n_head * hd + 3 * self.n_ff * d)
        return 2.0 * T * (self.n_layer * per_layer + self.n_vocab * d)

    def attn_flops(self, T: int | None = None) -> float:
        """Causal QK^T + PV over the visible keys (diagonal included)."""
        T = self.T if T is None else T
        return float(self.n_layer) * self.n_head * 2.0 * self.head_dim * T * (T + 1)


CONFIGS = {
    "tiny": ModelConfig("tiny", n_layer=2, n_embd=64, n_head=4, n_head_kv=2, head_dim=16,
                        rope_dim_count=16, n_ff=128, n_vocab=256, T=16, precision="f32"),
    "small": ModelConfig("small", n_layer=4, n_embd=512, n_head=8, n_head_kv=4, head_dim=64,
                         rope_dim_count=64, n_ff=1536, n_vocab=32000, T=256, precision="bf16"),
    "qwen3-0.6b-shape": ModelConfig("qwen3-0.6b-shape", n_layer=28, n_embd=1024, n_head=16,
                                    n_head_kv=8, head_dim=128, rope_dim_count=128, n_ff=3072,
                                    n_vocab=151936, T=2048, precision="bf16"),
    "qwen3-8b-shape": ModelConfig("qwen3-8b-shape", n_layer=36, n_embd=4096, n_head=32,
                                  n_head_kv=8, head_dim=128, rope_dim_count=128, n_ff=12288,
                                  n_vocab=151936, T=4096, precision="bf16"),
}

# Attention-only sweep: causal GQA SDPA with fused QK-norm + NeoX RoPE.
ATTN_SWEEP = dict(n_head=32, n_head_kv=8, head_dim=128, rope_dims=(64, 128),
                  T=(1024, 4096, 8192, 16384), rope_freq_base=1e6, rms_eps=1e-6)

# --------------------------------------------------------------------------------------
# Tensor ids (one stream each)
# --------------------------------------------------------------------------------------
TID_TOKENS = 1
TID_TOK_EMBD = 2
TID_OUTPUT_NORM = 3
TID_OUTPUT = 4
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm",
                 "w_gate", "w_up", "w_down")
NORM_TENSORS = ("attn_norm", "q_norm", "k_norm", "ffn_norm")
TID_ATTN_Q, TID_ATTN_K, TID_ATTN_V, TID_ATTN_QN, TID_ATTN_KN = 11, 12, 13, 14, 15


def layer_tid(layer: int, name: str) -> int:
    return 1000 + 64 * layer + LAYER_TENSORS.index(name)


def layer_shapes(cfg: ModelConfig) -> dict:
    d, hd, h, g, F = cfg.n_embd, cfg.head_dim, cfg.n_head, cfg.n_head_kv, cfg.n_ff
    return {
        "attn_norm": (d,), "wq": (h * hd * (2 if cfg.attn_gate else 1), d), "wk": (g * hd, d),
        "wv": (g * hd, d),
        "q_norm": (hd,), "k_norm": (hd,), "wo": (d, h * hd), "ffn_norm": (d,),
        "w_gate": (F, d), "w_up": (F, d), "w_down": (d, F),
    }


def layer_tensor(cfg: ModelConfig, layer: int, name: str, seed: int = 0) -> np.ndarray:
    shape = layer_shapes(cfg)[name]
    if name in NORM_TENSORS:
        return normal(seed, layer_tid(layer, name), shape, mean=1.0, std=0.1)
    return normal(seed, layer_tid(layer, name), shape, mean=0.0, std=0.02)


def layer_weights(cfg: ModelConfig, layer: int, seed: int = 0) -> dict:
    return {name: layer_tensor(cfg, layer, name, seed) for name in LAYER_TENSORS}


def tok_embd(cfg: ModelConfig, seed: int = 0) -> np.ndarray:
    return normal(seed, TID_TOK_EMBD, (cfg.n_vocab, cfg.n_embd), std=0.02)


def output_norm(cfg: ModelConfig, seed: int = 0) -> np.ndarray:
    return normal(seed, TID_OUTPUT_NORM, (cfg.n_embd,), mean=1.0, std=0.1)


def output_weight(cfg: ModelConfig, seed: int = 0) -> np.ndarray:
    return normal(seed, TID_OUTPUT, (cfg.n_vocab, cfg.n_embd), std=0.02)


def tokens(cfg: ModelConfig, seed: int = 0, T: int | None = None) -> np.ndarray:
    T = cfg.T if T is None else T
    return uniform_int(seed, TID_TOKENS, T, cfg.n_vocab)


def model_weights(cfg: ModelConfig, seed: int = 0) -> dict:
    """Every tensor of the model as float32 arrays (small configs only)."""
    return {
        "tok_embd": tok_embd(cfg, seed),
        "layers": [layer_weights(cfg, l, seed) for l in range(cfg.n_layer)],
        "output_norm": output_norm(cfg, seed),
        "output": output_weight(cfg, seed),
    }


def attention_inputs(T: int, n_head: int, n_head_kv: int, head_dim: int, seed: int = 0) -> dict:
    """Attention-sweep operands: q [T, h*hd], k/v [T, g*hd] ~ N(0,1); norm scales 1+N(0,0.1)."""
    return {
        "q": normal(seed, TID_ATTN_Q, (T, n_head * head_dim)),
        "k": normal(seed, TID_ATTN_K, (T, n_head_kv * head_dim)),
        "v": normal(seed, TID_ATTN_V, (T, n_head_kv * head_dim)),
        "q_norm": normal(seed, TID_ATTN_QN, (head_dim,), mean=1.0, std=0.1),
        "k_norm": normal(seed, TID_ATTN_KN, (head_dim,), mean=1.0, std=0.1),
    }


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns.

    Storage conversion for handing bf16 inputs to either side; finite inputs only."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + (((b >> 16) & 1) + 0x7FFF)) >> 16
    return r.astype(np.uint16)


def from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
