"""The numerical design of the exact pass over short prefixes, checked on the CPU.

The forward recomputes rows whose causal prefix holds few keys (n <= 64) in float64, in the dual
form of the weighted ridge regression over the n keys ("Parallax" blog, s.2 Canonical
Formulation):
    o = vbar + Vc^T W^(1/2) (K' + lambda' I)^-1 W^(1/2) Xc (q - kbar),  K' = W^(1/2) Xc Xc^T W^(1/2),
with the centring's null vector W^(1/2) 1 deflated and the ridge floored at 1e-12 of K''s largest
diagonal entry. These tests restate that algorithm in numpy (not the kernel's code, which the GPU
tests check) and hold it against the oracle where the primal form fails: a tiny effective ridge
lambda e^-m, more keys than dimensions, repeated keys. They also show that the floor is needed:
without it the rounding of the right-hand side along K''s null directions is divided by lambda'.
"""
import numpy as np
import pytest
import torch

from oracle import lla_row

FLOOR = 1e-12  # the ridge floor the exact pass uses, relative to K''s largest diagonal entry


def dual_row(q, K, V, h, lam, floor=FLOOR, deflate=True):
    s = K @ q / h
    m = s.max()
    w = np.exp(s - m)
    om = w.sum()
    lp = lam * np.exp(-m)
    sw = np.sqrt(w)
    kb, vb = w @ K / om, w @ V / om
    xc, vc = K - kb, V - vb
    kk = (sw[:, None] * xc) @ (sw[:, None] * xc).T
    if deflate:
        kk = kk + np.trace(kk) / om * np.outer(sw, sw)
    ridge = max(lp, floor * np.diag(kk).max()) if floor else lp
    z = np.linalg.solve(kk + ridge * np.eye(len(w)), sw * (xc @ (q - kb)))
    return vb + (sw * z) @ vc


def offset_prefix(seed, n, d, offset, direction):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(d, generator=g, dtype=torch.float64).numpy()
    K = torch.randn(n, d, generator=g, dtype=torch.float64).numpy()
    V = torch.randn(n, d, generator=g, dtype=torch.float64).numpy()
    if direction == "one":
        u = torch.randn(d, generator=g, dtype=torch.float64).numpy()
        K = K + offset * u / np.linalg.norm(u)
        q = q + offset * u / np.linalg.norm(u) / 8.0
    else:
        K = K + offset
        q = q + offset / 8.0
    return q, K, V


def rel(a, b):
    return np.abs(a - b).max() / (np.abs(b).max() + 1.0)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("offset,direction", [(0.0, "all"), (16.0, "all"), (32.0, "one")])
def test_dual_form_matches_the_oracle_on_short_prefixes(d, offset, direction):
    """Below d keys the floored dual form is exact to ~1e-6; at n = d and d + 1 random keys are
    nearly singular (the smallest variance ~1e-5 of the largest) and the floor biases that
    direction by ~floor / 1e-5 = 1e-7 relative to it, ~1e-4 of the output at most here."""
    h, lam = float(np.sqrt(d)), 1e-2
    for n in (1, 2, d // 2, d - 1, d, d + 1, 64):
        q, K, V = offset_prefix(int(100 * d + n + offset), n, d, offset, direction)
        err = rel(dual_row(q, K, V, h, lam), lla_row(q, K, V, h, lam))
        assert err < (1e-5 if n < d else 3e-4), (n, err)


def test_repeated_keys():
    q, K, V = offset_prefix(7, 40, 64, 16.0, "all")
    K[10::7] = K[3]  # repeated keys: more null directions of K' than the centring's own
    for lam in (1e-2, 1e-30):
        assert rel(dual_row(q, K, V, 8.0, lam), lla_row(q, K, V, 8.0, lam)) < 1e-3


def test_the_floor_is_needed_under_a_tiny_effective_ridge():
    """More keys than dimensions (n = 40 > d = 32) and lambda e^-m ~ 1e-20: the floored dual form
    stays exact, the plain one divides rounding by lambda'."""
    q, K, V = offset_prefix(11, 40, 32, 16.0, "all")
    h, lam = float(np.sqrt(32)), 1e-2
    s = K @ q / h
    assert lam * np.exp(-s.max()) < 1e-15  # the regime the floor is for
    ref = lla_row(q, K, V, h, lam)
    assert rel(dual_row(q, K, V, h, lam), ref) < 1e-5
    assert rel(dual_row(q, K, V, h, lam, floor=0.0), ref) > 1e-3
