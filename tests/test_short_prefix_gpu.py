"""GPU parity of rows whose causal prefix holds at most d keys, on every path and dtype.

With n <= d keys the centred key covariance has rank below d, so the ridge system
(C_kk + lambda e^-m I) y = q - kbar ("Parallax" blog, s.2 Canonical Formulation) is singular up
to the effective ridge lambda e^-m. When the keys share a large common offset and the query is
aligned with it, m is large, that ridge tiny, and y's part outside the keys' span, of size
|q - kbar| / (lambda e^-m), must cancel in k . y - kbar . y. The solves list such rows (every one
for fp32 inputs; for bf16 those whose |y| is past what the readout can cancel, or whose
factorisation failed) and an exact float64 pass in the dual form over the n keys recomputes their
output. Every row of every head up to d + 6 is checked here, next to a sample of later rows.

Bounds: relative Frobenius error <= 1e-3 (fp32 inputs) or 2e-2 (bf16), the worst row within 5x.
"""
import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import lla_forward_oracle
from parity import record

TOL = {"f32": 1e-3, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def offset_inputs(seed, d, offset, direction, dtype, T=300, BH=4):
    """i.i.d. N(0,1) q, k, v with `offset` added to every key, along one unit vector
    (direction="one") or in every coordinate ("all"); bf16 rounds all three."""
    q, k, v = W.make_iid(1, BH, T, d, d, "f32", seed=seed)
    if direction == "one":
        u = torch.randn(d, generator=torch.Generator().manual_seed(seed + 1))
        k = k + offset * u / u.norm()
    else:
        k = k + offset
    if dtype == "bf16":
        return W._cast(q, "bf16"), W._cast(k, "bf16"), W._cast(v, "bf16")
    return q, k, v


def check(lla, q, k, v, h, lam, dtype, path=0):
    B, H, T, d = q.shape
    out = lla.lla_forward(q.cuda(), k.cuda(), v.cuda(), h, lam, path=path)
    assert lla.lla_stream_status() == 0
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, v.shape[-1])
    rows = {bh * T + i for bh in range(B * H) for i in range(min(T, d + 6))}
    rows |= set(W.sample_rows(B * H, T, 40, seed=T + d))
    rows = sorted(rows)
    ref = lla_forward_oracle(q, k, v, h, lam, rows=rows)
    record(got[rows], ref, v.float().numpy(), TOL[dtype])


@pytest.mark.gpu
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("offset,direction", [(0.0, "all"), (16.0, "all"), (32.0, "one")])
def test_short_prefixes_f32_cuda_cores(lla, d, offset, direction):
    """fp32 inputs (the CUDA-core path): every prefix of at most d keys is recomputed exactly."""
    q, k, v = offset_inputs(int(800 + d + offset), d, offset, direction, "f32")
    check(lla, q, k, v, float(np.sqrt(d)), 1e-2, "f32")


@pytest.mark.gpu
@pytest.mark.parametrize("offset,direction", [(16.0, "all"), (32.0, "one")])
def test_short_prefixes_bf16_cuda_core_path(lla, offset, direction):
    """bf16 inputs with the CUDA-core path forced: rows listed by the size of |y|."""
    q, k, v = offset_inputs(int(900 + offset), 64, offset, direction, "bf16")
    check(lla, q, k, v, 8.0, 1e-2, "bf16", path=lla.PATH_CUDA_CORE)


@pytest.mark.gpu
@pytest.mark.parametrize("offset,direction", [(16.0, "all"), (32.0, "one")])
def test_short_prefixes_bf16_padded(lla, offset, direction):
    """bf16 inputs with d = 32 run zero-padded on the d = 64 tensor-core path, where a prefix of
    up to 64 keys is listed by the same rule (the padded features change no output)."""
    q, k, v = offset_inputs(int(950 + offset), 32, offset, direction, "bf16")
    check(lla, q, k, v, float(np.sqrt(32)), 1e-2, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_prefixes_with_repeated_keys(lla, dtype):
    """Keys that repeat earlier ones (linearly dependent prefixes: more null directions of the
    dual system than the centring's own) under a large common offset. T = 64: every row is within
    the exact pass's reach (a longer prefix with fewer than d + 1 affinely independent keys and a
    tiny effective ridge is not, and reports LLA_ERR_NUMERICAL)."""
    q, k, v = offset_inputs(990, 64, 16.0, "all", dtype, T=64)
    k = k.clone()
    for j in range(5, 64, 7):
        k[:, :, j] = k[:, :, j - 4]
    check(lla, q, k, v, 8.0, 1e-2, dtype)


@pytest.mark.gpu
def test_forward_with_listed_rows_replays_from_a_cuda_graph(lla):
    """The exact pass runs on the library's side stream, forked after the solve and joined after
    the readout; captured into a CUDA graph (rows listed: large common key offset), the fork and
    join stay inside the capture and a replay reproduces the eager call bit for bit."""
    q, k, v = (t.cuda() for t in offset_inputs(1001, 64, 16.0, "all", "bf16"))
    out = torch.empty_like(v)
    lla.lla_forward(q, k, v, 8.0, 1e-2, out=out)  # first call: creates the side stream
    torch.cuda.synchronize()
    ref = out.clone()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        lla.lla_forward(q, k, v, 8.0, 1e-2, out=out, stream=s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert lla.lla_stream_status() == 0
    assert torch.equal(out, ref)


@pytest.mark.gpu
def test_concurrent_forwards_on_two_streams_share_the_side_stream(lla):
    """Two forwards with listed rows, on two streams with no ordering between them, each fork
    to and join back from the one side stream of the device: each result equals its own call run
    alone, bit for bit."""
    a = [t.cuda() for t in offset_inputs(1101, 64, 16.0, "all", "bf16")]
    b = [t.cuda() for t in offset_inputs(1102, 64, 32.0, "one", "bf16")]
    ref_a = lla.lla_forward(*a, 8.0, 1e-2)
    ref_b = lla.lla_forward(*b, 8.0, 1e-2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out_a, out_b = torch.empty_like(ref_a), torch.empty_like(ref_b)
    for _ in range(3):
        with torch.cuda.stream(s1):
            lla.lla_forward(*a, 8.0, 1e-2, out=out_a, stream=s1)
        with torch.cuda.stream(s2):
            lla.lla_forward(*b, 8.0, 1e-2, out=out_b, stream=s2)
    torch.cuda.synchronize()
    assert lla.lla_stream_status() == 0
    assert torch.equal(out_a, ref_a) and torch.equal(out_b, ref_b)
