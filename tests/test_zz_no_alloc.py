"""lla_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin that its host application only hands input and output buffers, or a
latency-critical loop that must not call the allocator while it runs) get an entry point whose
scratch is a fixed array owned by the library. These tests check it through the C ABI against
lla_forward on two calls in a row (the second with different inputs, so nothing carried over in
the shared scratch can pass unnoticed), and that an oversized problem is refused up front. Both
entry points run the same stages in the same order on the same inputs, so their outputs must be
bitwise equal (the parity bound against the oracle is checked as well).
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W

TOL = {"f32": 1e-3, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def rel_err(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,shape", [("bf16", (1, 2, 300, 64, 64)), ("f32", (2, 1, 200, 32, 16))])
def test_noalloc_matches_forward_on_consecutive_calls(lla, dtype, shape):
    B, H, T, d, dv = shape
    for seed in (21, 22):  # two calls in a row, different inputs
        q, k, v = (t.cuda() for t in W.make_iid(B, H, T, d, dv, dtype, seed=seed))
        ref = lla.lla_forward(q, k, v, 8.0, 0.01)
        out = torch.full_like(ref, float("nan"))
        lla.lla_forward_noalloc(q, k, v, 8.0, 0.01, out)
        assert lla.lla_stream_status() == 0
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref)
        assert rel_err(out, ref) <= TOL[dtype]


@pytest.mark.gpu
def test_noalloc_checks_out(lla):
    q, k, v = (t.cuda() for t in W.make_iid(1, 1, 64, 16, 16, "f32", seed=23))
    for bad in (torch.empty(1, 1, 64, 8, device="cuda"),                      # wrong shape
                torch.empty(1, 1, 64, 16, device="cuda", dtype=torch.bfloat16),  # wrong dtype
                torch.empty(1, 1, 16, 64, device="cuda").transpose(2, 3)):     # not contiguous
        with pytest.raises(ValueError):
            lla.lla_forward_noalloc(q, k, v, 4.0, 0.01, bad)


def test_noalloc_refuses_problems_beyond_its_scratch(lla):
    lib = lla._load()
    need = lla.lla_workspace_size(4, 8, 4096, 64, 64, torch.bfloat16)
    assert need > lla.NOALLOC_SCRATCH_BYTES
    # rejected on the host before any pointer is used or the device is touched
    fake = ctypes.c_void_p(256)
    st = lib.lla_forward_noalloc(fake, fake, fake, fake, 4, 8, 4096, 64, 64, 8.0, 0.01, 1, None)
    assert st == 2  # LLA_ERR_UNSUPPORTED
