"""Golden fixtures (tests/golden/): values written from the float64 oracle by
tests/golden/make_golden.py (the pages print no worked numerical example).

On the CPU, the oracle must reproduce every stored value (a change to its arithmetic shows up
here). On the GPU, the CUDA path must match the stored values within the parity bounds
(relative Frobenius error <= 1e-3 for fp32 inputs).
"""
import importlib.util
import json
import os

import numpy as np
import pytest
import torch

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def make_golden_module():
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def rel_err(got, ref):
    return float(np.linalg.norm(np.asarray(got) - np.asarray(ref)) / np.linalg.norm(ref))


@pytest.mark.parametrize("name", ["lla_forward_tiny.json", "parallax_forward_tiny.json",
                                  "parallax_backward_tiny.json"])
def test_oracle_reproduces_golden(name):
    fresh = make_golden_module().fixtures()[name]
    stored = load(name)
    if isinstance(stored["values"], dict):
        for key in stored["values"]:
            np.testing.assert_allclose(fresh["values"][key], stored["values"][key], rtol=1e-12,
                                       atol=1e-14)
    else:
        np.testing.assert_allclose(fresh["values"], stored["values"], rtol=1e-12, atol=1e-14)


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


@pytest.mark.gpu
def test_gpu_lla_forward_matches_golden(lla):
    mg = make_golden_module()
    fx = load("lla_forward_tiny.json")
    _, q, k, v, _ = mg.tiny_inputs()
    out = lla.lla_forward(q.cuda(), k.cuda(), v.cuda(), fx["h"], fx["lambda"])
    assert lla.lla_stream_status() == 0
    got = out.double().cpu().numpy().reshape(-1, out.shape[-1])[fx["rows"]]
    assert rel_err(got, fx["values"]) <= 1e-3


@pytest.mark.gpu
def test_gpu_parallax_forward_matches_golden(lla):
    mg = make_golden_module()
    fx = load("parallax_forward_tiny.json")
    _, q, k, v, r = mg.tiny_inputs()
    out = lla.lla_parallax_forward(q.cuda(), k.cuda(), v.cuda(), r.cuda(), fx["h"])
    assert lla.lla_stream_status() == 0
    got = out.double().cpu().numpy().reshape(-1, out.shape[-1])[fx["rows"]]
    assert rel_err(got, fx["values"]) <= 1e-3


@pytest.mark.gpu
def test_gpu_parallax_backward_matches_golden(lla):
    mg = make_golden_module()
    fx = load("parallax_backward_tiny.json")
    xs = [x.cuda() for x in mg.backward_inputs()]
    got = lla.lla_parallax_backward(*xs, fx["h"])
    assert lla.lla_stream_status() == 0
    for key, g in zip(("dq", "dk", "dv", "dr"), got):
        ref = np.asarray(fx["values"][key]).reshape(g.shape)
        assert rel_err(g.double().cpu().numpy(), ref) <= 1e-3, key
