"""GPU parity: liblla's causal Parallax forward against the float64 oracle, through the C ABI.

Tolerances (relative Frobenius error over the checked rows) as for LLA: 1e-3 for fp32 inputs,
2e-2 for bf16 inputs (the bf16 output rounding is part of the budget). Inputs are rounded to
their element type first and the oracle reads the rounded values. The probe r is drawn by
``workloads.make_probe`` (N(0, 1/d), seed = the inputs' seed + 100).
"""
import math

import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import parallax_forward_oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def rel_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def run(lla, q, k, v, r, h, path=0):
    out = lla.lla_parallax_forward(q.cuda(), k.cuda(), v.cuda(), r.cuda(), h, path=path)
    assert lla.lla_stream_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


def inputs(B, H, T, d, dv, dtype, seed):
    q, k, v = W.make_iid(B, H, T, d, dv, dtype, seed=seed)
    return q, k, v, W.make_probe(B, H, T, d, dtype, seed=seed + 100)


def check(lla, q, k, v, r, h, dtype, rows=None):
    got = run(lla, q, k, v, r, h)
    e = got.shape[-1]
    flat = got.reshape(-1, e)
    if rows is None:
        ref = parallax_forward_oracle(q, k, v, r, h).reshape(-1, e)
    else:
        ref = parallax_forward_oracle(q, k, v, r, h, rows=rows)
        flat = flat[rows]
    assert np.isfinite(flat).all()
    err = rel_err(flat, ref)
    assert err <= TOL[dtype], f"relative error {err:.3e}"
    return err


def test_tensor_core_shape_all_rows(lla):
    # bf16 d = dv = 64: several 128-query tiles and 32-key blocks, ragged tail.
    q, k, v, r = inputs(2, 2, 300, 64, 64, "bf16", seed=301)
    check(lla, q, k, v, r, 8.0, "bf16")


def test_headline_shape_sampled(lla):
    w = W.WORKLOADS[3]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100)
    rows = W.sample_rows(w.B * w.H, w.T, 384, seed=12)
    check(lla, q, k, v, r, w.h, w.dtype, rows=rows)


def test_long_shape_sampled(lla):
    w = W.WORKLOADS[5]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100)
    rows = W.sample_rows(w.B * w.H, w.T, 192, seed=5)
    check(lla, q, k, v, r, w.h, w.dtype, rows=rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,dv", [(16, 16), (32, 32), (64, 64), (16, 64), (64, 16), (32, 64)])
def test_ragged_shapes(lla, dtype, d, dv):
    q, k, v, r = inputs(1, 2, 203, d, dv, dtype, seed=400 + d + dv)
    check(lla, q, k, v, r, math.sqrt(d), dtype)


@pytest.mark.parametrize("T", [1, 2, 3, 31, 32, 33, 65, 128, 129])
def test_short_sequences_tensor_core(lla, T):
    q, k, v, r = inputs(1, 2, T, 64, 64, "bf16", seed=500 + T)
    check(lla, q, k, v, r, 8.0, "bf16")


def test_paths_agree(lla):
    q, k, v, r = inputs(1, 2, 257, 64, 64, "bf16", seed=77)
    outs = {path: run(lla, q, k, v, r, 8.0, path=path)
            for path in (lla.PATH_CUDA_CORE, lla.PATH_TENSOR_CORE)}
    ref = parallax_forward_oracle(q, k, v, r, 8.0).reshape(outs[1].shape)
    for path, o in outs.items():
        assert rel_err(o, ref) <= 2e-2, (path, rel_err(o, ref))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_probe_is_softmax(lla, dtype):
    q, k, v, _ = inputs(1, 2, 150, 64, 64, dtype, seed=6)
    out = run(lla, q, k, v, torch.zeros_like(q), 8.0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), is_causal=True, scale=1 / 8.0).numpy()
    assert rel_err(out, ref) <= TOL[dtype]


def test_first_token_returns_v1(lla):
    for dtype in ("f32", "bf16"):
        q, k, v, r = inputs(2, 3, 9, 64, 64, dtype, seed=8)
        out = run(lla, q, k, v, r, 5.0)
        assert np.abs(out[:, :, 0] - v[:, :, 0].double().numpy()).max() < 1e-2


def test_empty_problem_is_noop(lla):
    q = torch.zeros(1, 1, 0, 64, device="cuda", dtype=torch.bfloat16)
    out = lla.lla_parallax_forward(q, q, q, q, 8.0)
    assert out.shape == (1, 1, 0, 64)


def test_invalid_arguments_raise(lla):
    q = torch.zeros(1, 1, 8, 48, device="cuda")
    with pytest.raises(lla.LlaError) as ei:
        lla.lla_parallax_forward(q, q, q, q, 4.0)
    assert ei.value.status == 2
    q = torch.zeros(1, 1, 8, 16, device="cuda")
    with pytest.raises(lla.LlaError):
        lla.lla_parallax_forward(q, q, q, q, 0.0)
    lib = lla._load()
    # a misaligned probe pointer is rejected on the host
    assert lib.lla_parallax_forward(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr() + 4,
                                    q.data_ptr(), 1, 1, 8, 16, 16, 4.0, 0, None) == 1
