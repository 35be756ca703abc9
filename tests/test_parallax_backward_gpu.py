"""GPU parity of the causal Parallax backward (lla_parallax_backward), through the C ABI.

Each gradient (dq, dk, dv, dr) must match the float64 oracle (oracle.parallax_backward_oracle, the
chain rule through the forward of the "Parallax" blog, s.2 and Appendix B with eta = 0) within the
bounds of the forward: relative Frobenius error <= 1e-3 for fp32 inputs and <= 2e-2 for bf16
inputs, per gradient.
"""
import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import parallax_backward_oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def make(B, H, T, d, dv, dtype, seed):
    q, k, v = W.make_iid(B, H, T, d, dv, dtype, seed)
    r = W.make_probe(B, H, T, d, dtype, seed + 1000)
    g = torch.Generator().manual_seed(seed + 2000)
    do = torch.randn(B, H, T, dv, generator=g).to(q.dtype)
    return q, k, v, r, do


def f64(t):
    return t.double().cpu().numpy()


def rel_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


SHAPES = [(1, 1, 1, 16, 16), (1, 2, 37, 16, 32), (2, 2, 130, 32, 32), (1, 2, 300, 64, 64),
          (1, 1, 200, 64, 16), (1, 1, 97, 32, 64)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_parallax_backward_matches_oracle(lla, shape, dtype):
    B, H, T, d, dv = shape
    q, k, v, r, do = make(B, H, T, d, dv, dtype, seed=T + d + dv)
    h = float(np.sqrt(d))
    got = lla.lla_parallax_backward(*(x.cuda() for x in (q, k, v, r, do)), h)
    assert lla.lla_stream_status() == 0
    ref = parallax_backward_oracle(q, k, v, r, do, h)
    scale = np.linalg.norm(ref[2])  # dv = sum_i a_ij dO_i never vanishes
    for name, g, rf in zip(("dq", "dk", "dv", "dr"), got, ref):
        assert g.dtype == q.dtype and tuple(g.shape) == rf.shape
        assert np.isfinite(f64(g)).all(), name
        err = np.linalg.norm(f64(g) - rf)
        # A single-key prefix (T = 1) has dq = dk = dr = 0 exactly: there the error is measured
        # against the scale of dv.
        assert err <= TOL[dtype] * (np.linalg.norm(rf) if np.linalg.norm(rf) > 0 else scale), name


def test_parallax_backward_headline_heads(lla):
    # B4 H8 T4096 d = dv = 64 bf16 (the headline workload with its probe and an i.i.d. N(0,1)
    # upstream gradient); two whole heads checked against the oracle.
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, w.seed + 1000)
    g = torch.Generator().manual_seed(w.seed + 2000)
    do = torch.randn(w.B, w.H, w.T, w.dv, generator=g).to(q.dtype)
    got = lla.lla_parallax_backward(*(x.cuda() for x in (q, k, v, r, do)), w.h)
    assert lla.lla_stream_status() == 0
    for b, hh in ((0, 0), (3, 7)):
        ref = parallax_backward_oracle(q[b, hh], k[b, hh], v[b, hh], r[b, hh], do[b, hh], w.h)
        for name, gg, rf in zip(("dq", "dk", "dv", "dr"), got, ref):
            assert rel_err(f64(gg[b, hh]), rf) <= TOL["bf16"], (name, b, hh)


def test_parallax_backward_zero_probe_is_softmax_backward(lla):
    B, H, T, d = 2, 2, 500, 64
    q, k, v, _, do = make(B, H, T, d, d, "f32", seed=9)
    r = torch.zeros_like(q)
    dq, dk, dv, dr = lla.lla_parallax_backward(*(x.cuda() for x in (q, k, v, r, do)), 8.0)
    tq, tk, tv = (x.double().requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=1 / 8.0)
    (o * do.double()).sum().backward()
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert rel_err(f64(got), ref.numpy()) <= 1e-4


def test_parallax_backward_is_deterministic(lla):
    xs = [x.cuda() for x in make(1, 4, 700, 64, 64, "bf16", seed=4)]
    a = lla.lla_parallax_backward(*xs, 8.0)
    b = lla.lla_parallax_backward(*xs, 8.0)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_parallax_backward_argument_errors(lla):
    lib = lla._load()
    p = 256
    ptrs = [p] * 9
    assert lib.lla_parallax_backward(*ptrs, 1, 1, 8, 48, 64, 8.0, 1, None) == 2  # d = 48
    assert lib.lla_parallax_backward(*ptrs, 1, 1, 8, 64, 64, 0.0, 1, None) == 1  # h = 0
    assert lib.lla_parallax_backward(*ptrs, 1, 1, 8, 64, 64, 8.0, 5, None) == 1  # dtype
    assert lib.lla_parallax_backward(*ptrs, 0, 1, 8, 64, 64, 8.0, 1, None) == 0  # empty
    assert lib.lla_parallax_backward(*([None] + ptrs[1:]), 1, 1, 8, 64, 64, 8.0, 1, None) == 1


@pytest.mark.parametrize("T", [1, 2, 31, 127, 128, 129, 300, 1000])
def test_parallax_backward_tensor_cores_matches_oracle(lla, T):
    # bf16 d = dv = 64 runs the tcgen05 passes (rows and columns tiles of 128, blocks of 32).
    q, k, v, r, do = make(1, 2, T, 64, 64, "bf16", seed=50 + T)
    got = lla.lla_parallax_backward(*(x.cuda() for x in (q, k, v, r, do)), 8.0)
    assert lla.lla_stream_status() == 0
    ref = parallax_backward_oracle(q, k, v, r, do, 8.0)
    scale = np.linalg.norm(ref[2])
    for name, g, rf in zip(("dq", "dk", "dv", "dr"), got, ref):
        err = np.linalg.norm(f64(g) - rf)
        assert err <= TOL["bf16"] * (np.linalg.norm(rf) if np.linalg.norm(rf) > 0 else scale), name


def test_parallax_backward_tensor_and_cuda_cores_agree(lla):
    xs = [x.cuda() for x in make(2, 2, 777, 64, 64, "bf16", seed=8)]
    tc = lla.lla_parallax_backward(*xs, 8.0)
    cc = lla.lla_parallax_backward(*xs, 8.0, path=lla.PATH_CUDA_CORE)
    assert lla.lla_stream_status() == 0
    for name, a, b in zip(("dq", "dk", "dv", "dr"), tc, cc):
        assert rel_err(f64(a), f64(b)) <= TOL["bf16"], name
