"""GPU parity of decode (one query per head against a key/value cache), through the C ABI.

lla_decode must return the LLA prediction of the query over all L cached positions and
lla_parallax_decode the Parallax output, the oracle's lla_row / parallax_row over the full cache
("Parallax" blog, s.2), within the bounds of the prefill forward: relative Frobenius error
<= 1e-3 for fp32 inputs and <= 2e-2 for bf16 inputs.
"""
import math

import numpy as np
import pytest
import torch

from oracle import lla_row, parallax_row

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "bf16": 2e-2}
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def make(B, H, L, d, dv, dtype, seed, probe=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, d, generator=g)
    k = torch.randn(B, H, L, d, generator=g)
    v = torch.randn(B, H, L, dv, generator=g)
    r = torch.randn(B, H, d, generator=g) / math.sqrt(d) if probe else None
    cast = lambda t: None if t is None else t.to(DT[dtype])
    return cast(q), cast(k), cast(v), cast(r)


def f64(t):
    return t.double().cpu().numpy()


def rel_err(got, ref):
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


SHAPES = [(2, 3, 1, 64, 64), (2, 3, 7, 16, 32), (1, 4, 100, 32, 64), (2, 2, 1000, 64, 64),
          (1, 2, 5000, 64, 16), (3, 1, 777, 32, 32)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_lla_decode_matches_oracle(lla, shape, dtype):
    B, H, L, d, dv = shape
    q, k, v, _ = make(B, H, L, d, dv, dtype, seed=L + d + dv)
    h, lam = math.sqrt(d), 1e-2
    out = lla.lla_decode(q.cuda(), k.cuda(), v.cuda(), h, lam)
    assert lla.lla_stream_status() == 0
    got = f64(out).reshape(-1, dv)
    Q, K, V = f64(q).reshape(-1, d), f64(k).reshape(-1, L, d), f64(v).reshape(-1, L, dv)
    ref = np.stack([lla_row(Q[i], K[i], V[i], h, lam) for i in range(B * H)])
    assert rel_err(got, ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_parallax_decode_matches_oracle(lla, shape, dtype):
    B, H, L, d, dv = shape
    q, k, v, r = make(B, H, L, d, dv, dtype, seed=7 * L + d, probe=True)
    h = math.sqrt(d)
    out = lla.lla_parallax_decode(q.cuda(), k.cuda(), v.cuda(), r.cuda(), h)
    assert lla.lla_stream_status() == 0
    got = f64(out).reshape(-1, dv)
    Q, R = f64(q).reshape(-1, d), f64(r).reshape(-1, d)
    K, V = f64(k).reshape(-1, L, d), f64(v).reshape(-1, L, dv)
    ref = np.stack([parallax_row(Q[i], K[i], V[i], R[i], h) for i in range(B * H)])
    assert rel_err(got, ref) <= TOL[dtype]


def test_lla_decode_is_the_last_row_of_the_forward(lla):
    # The query at position L-1 of a sequence attends to exactly the L cached positions.
    B, H, L, d = 2, 2, 700, 64
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(B, H, L, d, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    fwd = lla.lla_forward(q, k, v, 8.0, 1e-2)[:, :, -1].float()
    dec = lla.lla_decode(q[:, :, -1].contiguous(), k, v, 8.0, 1e-2).float()
    assert lla.lla_stream_status() == 0
    assert rel_err(dec.cpu().numpy(), fwd.cpu().numpy()) <= 2e-2


def test_parallax_decode_zero_probe_is_softmax(lla):
    B, H, L, d = 2, 2, 3000, 64
    q, k, v, _ = make(B, H, L, d, d, "f32", seed=11)
    r = torch.zeros_like(q)
    out = lla.lla_parallax_decode(q.cuda(), k.cuda(), v.cuda(), r.cuda(), 8.0)
    s = torch.einsum("bhd,bhld->bhl", q.double(), k.double()) / 8.0
    ref = torch.einsum("bhl,bhle->bhe", torch.softmax(s, dim=-1), v.double())
    assert rel_err(f64(out), ref.numpy()) <= 1e-5


def test_decode_is_deterministic(lla):
    q, k, v, r = make(2, 4, 4096, 64, 64, "bf16", seed=5, probe=True)
    q, k, v, r = q.cuda(), k.cuda(), v.cuda(), r.cuda()
    a = lla.lla_decode(q, k, v, 8.0, 1e-2)
    b = lla.lla_decode(q, k, v, 8.0, 1e-2)
    c = lla.lla_parallax_decode(q, k, v, r, 8.0)
    d_ = lla.lla_parallax_decode(q, k, v, r, 8.0)
    assert torch.equal(a, b) and torch.equal(c, d_)


def test_decode_argument_errors(lla):
    lib = lla._load()
    p = ctypes_ptr = 256
    assert lib.lla_decode(p, p, p, p, 1, 1, 0, 64, 64, 8.0, 1e-2, 1, None) == 1  # L = 0
    assert lib.lla_decode(p, p, p, p, 1, 1, 8, 48, 64, 8.0, 1e-2, 1, None) == 2  # d = 48
    assert lib.lla_decode(p, p, p, p, 1, 1, 8, 64, 64, -1.0, 1e-2, 1, None) == 1  # h < 0
    assert lib.lla_decode(p, p, p, p, 0, 1, 8, 64, 64, 8.0, 1e-2, 1, None) == 0  # empty batch
    assert lib.lla_parallax_decode(p, p, p, None, p, 1, 1, 8, 64, 64, 8.0, 1, None) == 1
    del ctypes_ptr


# Tensor-core split kernel (bf16, d = dv = 64): the chunk's sums as tcgen05 contractions with
# exact hi/lo operands, the shift of the sums moved only when a tile's maximum logit exceeds it
# by more than 8 ln 2 h (then the accumulators in tensor memory are rescaled).
TC_LENGTHS = [1, 63, 64, 65, 200, 1000, 4099, 20000]


@pytest.mark.parametrize("L", TC_LENGTHS)
def test_lla_decode_tensor_cores_match_oracle_and_cuda_cores(lla, L):
    B, H, d = 2, 3, 64
    q, k, v, _ = make(B, H, L, d, d, "bf16", seed=100 + L)
    h, lam = 8.0, 1e-2
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    tc = lla.lla_decode(qc, kc, vc, h, lam)
    assert lla.lla_stream_status() == 0
    cc = lla.lla_decode(qc, kc, vc, h, lam, path=lla.PATH_CUDA_CORE)
    assert lla.lla_stream_status() == 0
    Q, K, V = f64(q).reshape(-1, d), f64(k).reshape(-1, L, d), f64(v).reshape(-1, L, d)
    ref = np.stack([lla_row(Q[i], K[i], V[i], h, lam) for i in range(B * H)])
    got_tc, got_cc = f64(tc).reshape(-1, d), f64(cc).reshape(-1, d)
    assert rel_err(got_tc, ref) <= TOL["bf16"]
    assert rel_err(got_cc, ref) <= TOL["bf16"]
    assert rel_err(got_tc, got_cc) <= TOL["bf16"]


@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_lla_decode_tensor_cores_moving_logit_scale(lla, direction):
    # Key norms grow (or shrink) along the cache, so each tile's maximum logit keeps exceeding the
    # shift of the sums by more than the slack (rising: the accumulators are rescaled many times)
    # or never does after the first tile (falling).
    B, H, L, d = 1, 4, 6000, 64
    g = torch.Generator().manual_seed(41 if direction == "rising" else 43)
    q = torch.randn(B, H, d, generator=g)
    ramp = torch.linspace(0.2, 3.0, L) if direction == "rising" else torch.linspace(3.0, 0.2, L)
    k = torch.randn(B, H, L, d, generator=g) * ramp[None, None, :, None]
    v = torch.randn(B, H, L, d, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    h, lam = 8.0, 1e-2
    out = lla.lla_decode(q.cuda(), k.cuda(), v.cuda(), h, lam)
    assert lla.lla_stream_status() == 0
    Q, K, V = f64(q).reshape(-1, d), f64(k).reshape(-1, L, d), f64(v).reshape(-1, L, d)
    ref = np.stack([lla_row(Q[i], K[i], V[i], h, lam) for i in range(B * H)])
    assert rel_err(f64(out).reshape(-1, d), ref) <= TOL["bf16"]


@pytest.mark.parametrize("path", ["tensor", "cuda"])
def test_lla_decode_long_cache_with_empty_splits(lla, path):
    # One head and a long cache: the cache is split 512 ways in chunks of 196 keys, so the last
    # splits get no keys at all; their partials must drop out of the merge.
    B, H, L, d = 1, 1, 100000, 64
    q, k, v, _ = make(B, H, L, d, d, "bf16", seed=61)
    h, lam = 8.0, 1e-2
    out = lla.lla_decode(q.cuda(), k.cuda(), v.cuda(), h, lam,
                         path=lla.PATH_CUDA_CORE if path == "cuda" else lla.PATH_AUTO)
    assert lla.lla_stream_status() == 0
    got = f64(out).reshape(-1, d)
    assert np.isfinite(got).all()
    ref = lla_row(f64(q).reshape(d), f64(k).reshape(L, d), f64(v).reshape(L, d), h, lam)
    assert rel_err(got[0], ref) <= TOL["bf16"]
