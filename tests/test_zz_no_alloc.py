"""The allocation-free attention entry point, dtp_sdpa_causal_gqa_noalloc.

It serves callers that cannot allocate device memory where they call
attention (an op handed only its tensors, a runtime that forbids cudaMalloc
after start-up).  Its transposed-V scratch lives in a fixed 8 MiB array inside
the library instead of a caller workspace.  These checks call it through the
C ABI and compare it with dtp_sdpa_causal_gqa (bit for bit) and with the
oracle on the same inputs, twice in a row with different shapes (the shared
scratch keeps the previous call's contents) and once at the size limit, and
check that an oversized call is refused before any launch.

This file is collected last on purpose: a failure here leaves every other
test already run."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
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


def test_limit_is_accepted_on_a_machine_without_a_gpu(dtp):
    """At exactly 8 MiB (8 kv heads x 128 dims x 4096 tokens x 2 bytes) the size
    check passes; without a GPU the call then stops at the device lookup
    (DTP_ERR_CUDA), one token more stops at the size check (DTP_ERR_WORKSPACE).
    Only where no GPU is present: past the size check the pointers would be used."""
    if torch.cuda.is_available():
        pytest.skip("the accepted call would launch on the fake pointers")
    f = _fn(dtp)
    fake = c_void_p(0x10000)
    assert f(fake, fake, fake, fake, 4096, 32, 8, 128, 0.1, None) == -5
    assert f(fake, fake, fake, fake, 4097, 32, 8, 128, 0.1, None) == -4


def _inputs(dev, T, nh, nkv, hd, seed):
    bf = lambda a: torch.as_tensor(a, device=dev).bfloat16()
    return (bf(synth.normal(seed, 1, (T, nh * hd))), bf(synth.normal(seed, 2, (T, nkv * hd))),
            bf(synth.normal(seed, 3, (T, nkv * hd))))


@pytest.mark.gpu
def test_matches_workspace_entry_point_twice_in_a_row(dtp):
    """Two calls in a row (different shapes; the second reads scratch the first
    wrote), then a call at the 8 MiB limit.  Each equals dtp_sdpa_causal_gqa bit
    for bit (the same kernels on the same values) and the oracle within the
    attention tolerance of test_ops_gpu.py, on all rows or, at the limit, on
    rows spread to T-1."""
    f = _fn(dtp)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(300, 8, 2, 128, 21, None), (129, 4, 2, 64, 22, None),
             (4096, 32, 8, 128, 23, np.array([0, 1, 127, 128, 2047, 3968, 4000, 4095]))]
    for call, (T, nh, nkv, hd, seed, rows) in enumerate(cases):
        q, k, v = _inputs(dev, T, nh, nkv, hd, seed)
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
        assert torch.equal(out, ref), call
        rows = np.arange(T) if rows is None else rows
        want = oracle.sdpa_causal_gqa(q.double().cpu().numpy(), k.double().cpu().numpy(),
                                      v.double().cpu().numpy(), nh, nkv, hd, sc, rows=rows)
        got = out.float().cpu().numpy()[rows]
        vmax = float(v.float().abs().max())
        assert np.all(np.isfinite(got)), call
        assert np.abs(got - want).max() <= 8e-3 * vmax, call
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 3e-3, call
