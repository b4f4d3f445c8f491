"""bf16 attention's P V^T product runs on f16 operands: v enters as the exact f16
copy of its bf16 value, so a |v| beyond 65504 (the f16 range) cannot be held.
The library flags it on the device and dtp_check reports DTP_ERR_VALUE_RANGE;
values up to the range limit pass unflagged."""
import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")


def _run(dtp, v_scale_at, value):
    T, nh, nkv, hd = 64, 4, 2, 64
    bf = lambda a: torch.as_tensor(a, device=dev).bfloat16()
    q = bf(synth.normal(31, 1, (T, nh * hd)))
    k = bf(synth.normal(31, 2, (T, nkv * hd)))
    v = synth.normal(31, 3, (T, nkv * hd))
    v[v_scale_at] = value
    v = bf(v)
    out = torch.empty_like(q)
    ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_BF16), dtype=torch.uint8,
                     device=dev)
    dtp.sdpa_causal_gqa(q, k, v, out, nh, nkv, hd, 1 / math.sqrt(hd), ws)
    return out


def test_v_at_the_f16_limit_passes(dtp):
    out = _run(dtp, (5, 7), 65280.0)          # the largest bf16 value <= 65504: 255 * 2^8
    dtp.check()
    assert torch.isfinite(out.float()).all()


def test_v_beyond_the_f16_range_is_reported(dtp):
    _run(dtp, (5, 7), 70000.0)                 # bf16(70000) = 70144 > 65504
    with pytest.raises(dtp.DtpError) as e:
        dtp.check()
    assert e.value.code == -7
    dtp.check()                                # the error word was cleared
