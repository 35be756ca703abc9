"""GPU parity of the matrix-free conjugate-gradient strategy (lla_forward_ex with path LLA_PATH_CG).

The strategy solves each query's ridge system (C_kk + lambda' I) y = q - kbar by CG, every
product with C_kk being one streaming pass over the prefix, instead of accumulating and
factoring the moments ("Parallax" blog, s.2 "Difficulties in Scaling LLA"). It must meet the same
bound as the dense strategy against the float64 oracle: relative Frobenius error <= 2e-2 for
bf16 inputs (the only inputs it serves: bf16 with d = dv = 64).
"""
import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import lla_forward_oracle

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


class _WithOptions:
    """The binding with fixed per-call options on lla_forward."""

    def __init__(self, lla, **opts):
        self._lla, self._opts = lla, opts

    def lla_forward(self, *args, **kw):
        return self._lla.lla_forward(*args, **{**self._opts, **kw})

    def __getattr__(self, name):
        return getattr(self._lla, name)


@pytest.fixture
def cg(lla):
    return _WithOptions(lla, path=lla.PATH_CG, cg=(1024, 1e-3))


def rel_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def run(lla, q, k, v, h, lam):
    out = lla.lla_forward(q.cuda(), k.cuda(), v.cuda(), h, lam)
    assert lla.lla_stream_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T", [1, 2, 33, 128, 129, 203, 700])
def test_cg_matches_oracle_all_rows(cg, T):
    q, k, v = W.make_iid(1, 2, T, 64, 64, "bf16", seed=300 + T)
    got = run(cg, q, k, v, 8.0, 1e-2).reshape(-1, 64)
    ref = lla_forward_oracle(q, k, v, 8.0, 1e-2).reshape(-1, 64)
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= TOL_BF16


def test_cg_headline_sampled_rows(cg):
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    rows = W.sample_rows(w.B * w.H, w.T, 128, seed=7)
    got = run(cg, q, k, v, w.h, w.lam).reshape(-1, w.dv)[rows]
    ref = lla_forward_oracle(q, k, v, w.h, w.lam, rows=rows)
    assert rel_err(got, ref) <= TOL_BF16


def test_cg_agrees_with_dense(lla):
    q, k, v = W.make_iid(2, 2, 512, 64, 64, "bf16", seed=31)
    dense = run(lla, q, k, v, 8.0, 1e-2)
    it = run(_WithOptions(lla, path=lla.PATH_CG), q, k, v, 8.0, 1e-2)
    assert rel_err(it.reshape(-1, 64), dense.reshape(-1, 64)) <= TOL_BF16


def test_cg_large_ridge_is_softmax(cg):
    # lambda -> infinity: y -> 0 after the first step; the output is causal softmax attention.
    from oracle import softmax_attention_oracle
    q, k, v = W.make_iid(1, 1, 300, 64, 64, "bf16", seed=5)
    got = run(cg, q, k, v, 8.0, 1e12).reshape(-1, 64)
    ref = softmax_attention_oracle(q, k, v, 8.0).reshape(-1, 64)
    assert rel_err(got, ref) <= TOL_BF16


def test_cg_nonfinite_input_reports_numerical(cg):
    q, k, v = W.make_iid(1, 1, 256, 64, 64, "bf16", seed=9)
    q[0, 0, 200, 3] = float("nan")
    out = cg.lla_forward(q.cuda(), k.cuda(), v.cuda(), 8.0, 1e-2)
    assert cg.lla_stream_status() == 4  # LLA_ERR_NUMERICAL
    got = out.float().cpu()
    assert torch.isnan(got[0, 0, 200]).all()
    assert torch.isfinite(got[0, 0, :128]).all()


def test_cg_parameters_are_checked(lla):
    q, k, v = (t.cuda() for t in W.make_iid(1, 1, 64, 64, 64, "bf16", seed=3))
    for bad in ((-1, 1e-3), (2000, 1e-3), (10, -0.5), (10, 1.5)):
        with pytest.raises(lla.LlaError) as ei:
            lla.lla_forward(q, k, v, 8.0, 1e-2, path=lla.PATH_CG, cg=bad)
        assert ei.value.status == 1  # LLA_ERR_INVALID_ARG
