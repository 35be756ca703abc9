"""GPU parity of the tensor-core path (bf16, d = dv = 64) in the method's boundary regime.

LLA exists for queries near or beyond the edge of the key distribution: there the softmax
estimator is biased inward and LLA's local linear fit extrapolates ("Parallax" blog, s.1 on the
boundary bias of Nadaraya-Watson; s.2 "Additive Correction to Softmax", where the correction
factor 1 + eta grows with the query's distance from the weighted key mean). The stress workload
(rank-8 keys plus small noise, half of the queries beyond every key along one direction, values
an affine map of the keys plus noise) is built for that regime; here it is rounded to bf16, which
sends it down the tensor-core moments, solve and readout. A second input gives i.i.d. keys a
large common offset, so that the raw second moments that the tensor-core path accumulates are
far larger than their centred part.

Bound: relative Frobenius error <= 2e-2 (bf16 inputs), and the worst row within 5x that.
"""
import numpy as np
import pytest
import torch

from local_linear_attention_gb300 import workloads as W
from oracle import lla_forward_oracle
from parity import record

TOL = 2e-2


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


_CACHE = {}


def stress_bf16(with_u1=False):
    if "s" not in _CACHE:
        w = W.WORKLOADS[4]
        _CACHE["s"] = W.make_stress(w.B, w.H, w.T, w.d, w.dv, "bf16", w.seed, return_u1=True)
    return _CACHE["s"] if with_u1 else _CACHE["s"][:3]


def forward(lla, q, k, v, h, lam):
    out = lla.lla_forward(q.cuda(), k.cuda(), v.cuda(), h, lam)
    assert lla.lla_stream_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


def check_rows(lla, q, k, v, h, lam, rows):
    got = forward(lla, q, k, v, h, lam)
    e = got.shape[-1]
    ref = lla_forward_oracle(q, k, v, h, lam, rows=rows)
    return record(got.reshape(-1, e)[rows], ref, v.float().numpy(), TOL)


def stress_rows(BH, T, seed):
    rows = W.sample_rows(BH, T, 160, seed=seed)
    return sorted(set(rows) | {0, 1, 2, 17, 63, 64, 65, 200, T - 1})


@pytest.mark.gpu
@pytest.mark.parametrize("lam", [1e-2, 1.0])
@pytest.mark.parametrize("h", [4.0, 8.0, 16.0])
def test_stress_bf16_tensor_cores(lla, lam, h):
    q, k, v = stress_bf16()
    B, H, T, _ = q.shape
    check_rows(lla, q, k, v, h, lam, stress_rows(B * H, T, seed=int(300 + 10 * h + lam)))


@pytest.mark.gpu
@pytest.mark.parametrize("h", [4.0, 8.0, 16.0])
def test_stress_bf16_tensor_cores_small_ridge(lla, h):
    q, k, v = stress_bf16()
    B, H, T, _ = q.shape
    check_rows(lla, q, k, v, h, 1e-4, stress_rows(B * H, T, seed=int(400 + h)))


def test_stress_queries_outside_the_hull_are_checked():
    """The rows the stress checks sample include queries beyond every key of their causal prefix
    along the shift direction u_1 (outside the key hull, the case the construction is for): at
    least a third of them, early and late ones alike."""
    q, k, _, u1 = stress_bf16(with_u1=True)
    B, H, T, d = q.shape
    Q, K, U = q.reshape(-1, T, d).double(), k.reshape(-1, T, d).double(), u1.reshape(-1, d)
    for seed in [int(300 + 10 * h + lam) for h in (4.0, 8.0, 16.0) for lam in (1e-2, 1.0)]:
        rows = stress_rows(B * H, T, seed)
        beyond = []
        for rr in rows:
            bh, i = divmod(rr, T)
            pk = K[bh, : i + 1] @ U[bh]
            beyond.append(bool(Q[bh, i] @ U[bh] < pk.min()))
        assert sum(beyond) >= len(rows) // 3
        late = [b for rr, b in zip(rows, beyond) if rr % T > T // 2]
        assert sum(late) >= len(late) // 4


def offset_keys(seed, offset, direction):
    """i.i.d. N(0,1) keys plus a common offset: `offset` along one unit vector (direction="one")
    or in every coordinate (direction="all"), rounded to bf16 with q and v."""
    B, H, T, d = 1, 4, 1100, 64
    q, k, v = W.make_iid(B, H, T, d, d, "f32", seed=seed)
    if direction == "one":
        g = torch.Generator().manual_seed(seed + 1)
        u = torch.randn(d, generator=g)
        k = k + offset * u / u.norm()
    else:
        k = k + offset
    return W._cast(q, "bf16"), W._cast(k, "bf16"), W._cast(v, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("offset,direction", [(8.0, "one"), (32.0, "one"), (1.0, "all"),
                                              (4.0, "all"), (16.0, "all")])
def test_offset_keys_bf16_tensor_cores(lla, offset, direction):
    """Keys whose common offset is large against their spread: the raw moments sum p k k^T grow
    with offset^2 while the centred ones do not (8 and 32 standard deviations along one
    direction). An offset along the query direction also shifts the logits by q . c / h, which
    makes the absolute ridge lambda e^{-m} of the max-shifted moments tiny; on rank-deficient
    early prefixes (fewer keys than d) the primal y then carries a component of size
    |q - kbar| / (lambda e^{-m}) outside the keys' span that fp32 cannot cancel in the readout.
    Those rows are listed by the solve and recomputed exactly in the dual form over their keys
    (the exact pass), so every offset here meets the bound, early rows included."""
    q, k, v = offset_keys(int(500 + offset), offset, direction)
    B, H, T, _ = q.shape
    rows = W.sample_rows(B * H, T, 200, seed=int(600 + offset))
    early = {bh * T + i for bh in range(B * H) for i in range(70)}  # every row of the exact pass
    rows = sorted(set(rows) | early | {300})
    check_rows(lla, q, k, v, 8.0, 1e-2, rows)
