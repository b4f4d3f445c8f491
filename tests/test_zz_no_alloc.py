"""The allocation-free attention entry point, dtp_sdpa_causal_gqa_noalloc.

It serves callers that cannot allocate device memory where they call
attention (an op handed only its tensors, a runtime that forbids cudaMalloc
after start-up).  Its transposed-V scratch lives in a fixed 8 MiB array inside
the library instead of a caller workspace.  These checks call it through the
C ABI and compare it with dtp_sdpa_causal_gqa on the same inputs, twice in a
row with different shapes (the shared scratch keeps the previous call's
contents), and check that an oversized call is refused before any launch.

This file is collected last on purpose: a failure here leaves every other
test already run."""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth

c_int, c_float, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
ARGS = [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_float, c_void_p]


def _fn(dtp):
    f = dtp.lib().dtp_sdpa_causal_gqa_noalloc
    f.argtypes = ARGS
    f.restype = c_int
    return f


def test_oversized_call_is_refused(dtp):
    f = _fn(dtp)
    fake = c_void_p(0x10000)          # never dereferenced: the size check comes first
    # 8 kv heads x 128 dims x 4104 tokens (rounded up) x 2 bytes > 8 MiB
    assert f(fake, fake, fake, fake, 4097, 32, 8, 128, 0.1, None) == -4
    assert "8388608" in dtp.last_error()


@pytest.mark.gpu
def test_matches_workspace_entry_point_twice_in_a_row(dtp):
    f = _fn(dtp)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call, (T, nh, nkv, hd, seed) in enumerate([(300, 8, 2, 128, 21), (129, 4, 2, 64, 22)]):
        bf = lambda a: torch.as_tensor(a, device=dev).bfloat16()
        q = bf(synth.normal(seed, 1, (T, nh * hd)))
        k = bf(synth.normal(seed, 2, (T, nkv * hd)))
        v = bf(synth.normal(seed, 3, (T, nkv * hd)))
        sc = 1 / math.sqrt(hd)
        ref = torch.empty((T, nh * hd), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(dtp.sdpa_workspace_size(T, nkv, hd, dtp.DTP_BF16), dtype=torch.uint8,
                         device=dev)
        dtp.sdpa_causal_gqa(q, k, v, ref, nh, nkv, hd, sc, ws)
        out = torch.full((T, nh * hd), float("nan"), dtype=torch.bfloat16, device=dev)
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), T, nh, nkv, hd, sc, stream)
        assert rc == 0, dtp.last_error()
        torch.cuda.synchronize()
        dtp.check()
        got, want = out.float().cpu().numpy(), ref.float().cpu().numpy()
        vmax = float(v.float().abs().max())
        # the attention tolerance of tests/test_ops_gpu.py
        assert np.all(np.isfinite(got)), call
        assert np.abs(got - want).max() <= 8e-3 * vmax, call
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 3e-3, call
