"""bf16 forwards with d < 64 on the tensor cores, through zero-padded copies of q, k and v.

Zero key features leave the LLA intercept unchanged: the logits gain nothing, the moments of the
padded features are exactly zero, so the ridge system (C_kk + lambda' I) y = q - kbar ("Parallax"
blog, s.2 Canonical Formulation) is block-diagonal with lambda' I and a zero right-hand side on the
padded block, and y is zero there; zero value features give zero output columns. So the padded
forward must meet the bf16 bound against the float64 oracle at the caller's d and dv, and agree
with the CUDA-core path on the same inputs.
"""
import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import lla_forward_oracle
from parity import record

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def run(lla, q, k, v, h, lam, **kw):
    out = lla.lla_forward(q.cuda(), k.cuda(), v.cuda(), h, lam, **kw)
    assert lla.lla_stream_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d,dv,T", [(32, 32, 1), (32, 32, 300), (16, 16, 129), (32, 16, 257),
                                    (16, 64, 200), (32, 64, 65)])
def test_padded_forward_matches_oracle(lla, d, dv, T):
    q, k, v = W.make_iid(2, 2, T, d, dv, "bf16", seed=700 + d + dv + T)
    h = float(np.sqrt(d))
    got = run(lla, q, k, v, h, 1e-2).reshape(-1, dv)
    ref = lla_forward_oracle(q, k, v, h, 1e-2).reshape(-1, dv)
    record(got, ref, v.float().numpy(), TOL_BF16)


def test_padded_and_cuda_core_paths_agree(lla):
    q, k, v = W.make_iid(1, 4, 512, 32, 32, "bf16", seed=711)
    h = float(np.sqrt(32))
    tc = run(lla, q, k, v, h, 1e-2)
    cc = run(lla, q, k, v, h, 1e-2, path=lla.PATH_CUDA_CORE)
    ref = lla_forward_oracle(q, k, v, h, 1e-2).reshape(tc.shape)
    record(tc.reshape(-1, 32), ref.reshape(-1, 32), v.float().numpy(), TOL_BF16,
           case="padded tensor-core path, B1 H4 T512 d32")
    record(cc.reshape(-1, 32), ref.reshape(-1, 32), v.float().numpy(), TOL_BF16,
           case="CUDA-core path, B1 H4 T512 d32")
    assert float(np.linalg.norm(tc - cc) / np.linalg.norm(cc)) <= TOL_BF16


def test_padded_page_form_matches_oracle(lla):
    q, k, v = W.make_iid(1, 2, 300, 32, 32, "bf16", seed=712)
    h = float(np.sqrt(32))
    got = run(lla, q, k, v, h, 1e-2, form=lla.FORM_PAGE).reshape(-1, 32)
    ref = lla_forward_oracle(q, k, v, h, 1e-2).reshape(-1, 32)
    record(got, ref, v.float().numpy(), TOL_BF16)


def test_padded_launches_and_stream_order(lla):
    """The padding and the copy back are two more launches on the caller's stream."""
    q, k, v = (t.cuda() for t in W.make_iid(1, 2, 256, 32, 32, "bf16", seed=713))
    s = torch.cuda.Stream()
    n0 = lla.launch_count()
    with torch.cuda.stream(s):
        out = lla.lla_forward(q, k, v, float(np.sqrt(32)), 1e-2)
    s.synchronize()
    assert lla.launch_count() - n0 == 8 + 2
    assert lla.lla_stream_status() == 0
    assert torch.isfinite(out).all() and out.shape == (1, 2, 256, 32)
