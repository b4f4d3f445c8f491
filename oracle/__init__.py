"""CPU oracle for the dense (Qwen3-style) prefill forward pass -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the
prefill pass computes, in float64 numpy, written from the pages:

  * docs.rs memra-engine 0.130.0, src/forward.rs -- `Model::forward` (the op
    order: embed -> per layer {rms_norm, wq/wk/wv matmul, q/k rms_norm over
    head_dim rows, rope_neox, sdpa_naive causal, wo matmul, add, rms_norm,
    gate/up matmul, ffn_act, down matmul, add} -> output_norm -> lm_head),
    plus `argmax`, `top2` and `prime_gate_verdict`;
  * docs.rs needle-core v3/model.rs -- `V3Model::rope` / `rope_at` (the
    cos/sin tables freq_i = theta^(-2i/dims), angle = pos * freq_i).

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg may
import it.  It shares no code with the CUDA path (`dense_transformer_prefill_gb300`)
and imports nothing from it; its inputs come from the seeded generator in
`synth`, which holds none of the method's arithmetic.

Every function is pinned by `tests/test_oracle_pins.py` (closed forms,
invariants, brute force on tiny inputs, library routines in float64).
"""
from .model import (  # noqa: F401
    argmax,
    bf16_fused_normed_linear,
    forward,
    forward_chunk,
    forward_layer,
    linear,
    prime_gate_verdict,
    qk_norm,
    rms_norm,
    rope_angles,
    rope_neox,
    round_bf16,
    round_tf32,
    round_e4m3,
    fake_quant_rows_e4m3,
    sdpa_causal_gqa,
    silu,
    swiglu,
    top2,
)
