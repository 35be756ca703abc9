"""Pins for the float64 Parallax oracle (CPU only).

The pages print no worked numerical example of Parallax either, so the oracle is pinned to what
the pages and the mathematics fix:

* a zero probe gives causal softmax attention ("Parallax" blog s.2, "Strong regularization
  limit"; s.6 "With W_R = 0, Parallax is exactly Softmax Attention"), checked against ``torch``
  SDPA in float64;
* LLA is the same template with the solved probe rho* and the factor (1 + eta) (blog
  Appendix B): the pinned LLA oracle minus softmax equals (1 + eta) times (Parallax(rho*) minus
  softmax), with rho* and eta from the pages' own definitions;
* the streaming combination the pages print for the kernel, (1 + d2/d1) O1/d1 - O2/d1 (blog
  Appendix C, item 3), evaluated from whole-prefix sums;
* the wide-bandwidth limit (blog s.2 "Wide bandwidth limit"): uniform weights, so the output is
  the prefix mean of the values minus the plain (numpy) value-key covariance times the probe;
* invariants: constant values, the first token, value-affine equivariance, joint rotation of q,
  k and the probe, and affinity in the probe.

``test_pins_catch_planted_mistakes`` plants plausible mistakes into copies of the row function
and checks that at least one pin fails for each.
"""
import numpy as np
import pytest
import torch

from oracle import lla_row, parallax_forward_oracle, parallax_row


def rnd(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def forward_with(row_fn, q, k, v, r, h):
    return np.stack([row_fn(q[i], k[: i + 1], v[: i + 1], r[i], h) for i in range(q.shape[0])])


def softmax_rows(q, k, v, h):
    out = []
    for i in range(q.shape[0]):
        s = k[: i + 1] @ q[i] / h
        w = np.exp(s - s.max())
        out.append(w @ v[: i + 1] / w.sum())
    return np.stack(out)


# --------------------------------------------------------------------------- pin functions
# Each takes a row function with parallax_row's signature and returns the max violation.

def pin_zero_probe_softmax(row_fn):
    T, d, e, h = 11, 4, 4, 1.7
    q, k, v = rnd(1, T, d), rnd(2, T, d), rnd(3, T, e)
    o = forward_with(row_fn, q, k, v, np.zeros((T, d)), h)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(k)[None], torch.tensor(v)[None],
        is_causal=True, scale=1.0 / h)[0].numpy()
    return np.abs(o - ref).max() / np.abs(ref).max()


def pin_lla_relation(row_fn):
    # rho* = Sigma^-1 mu with z = k - q and raw weights w = exp(q.k/h) (blog s.2 Canonical
    # Formulation); tbar = mu^T rho* / omega and 1 + eta = 1 / (1 - tbar) (Appendix B).
    T, d, e = 12, 4, 4
    worst = 0.0
    for seed, (h, lam) in enumerate([(1.3, 0.05), (2.5, 0.4)]):
        q, k, v = rnd(10 + seed, T, d), rnd(20 + seed, T, d), rnd(30 + seed, T, e)
        o_sa = softmax_rows(q, k, v, h)
        for i in range(1, T):
            K, V = k[: i + 1], v[: i + 1]
            w = np.exp(K @ q[i] / h)
            Z = K - q[i]
            mu = w @ Z
            rho = np.linalg.solve((Z * w[:, None]).T @ Z + lam * np.eye(d), mu)
            eta = 1.0 / (1.0 - mu @ rho / w.sum()) - 1.0
            lla = lla_row(q[i], K, V, h, lam)
            par = row_fn(q[i], K, V, rho, h)
            worst = max(worst, np.abs((lla - o_sa[i]) - (1.0 + eta) * (par - o_sa[i])).max())
    return worst


def pin_streaming_combination(row_fn):
    T, d, e, h = 13, 4, 4, 1.1
    q, k, v, r = rnd(40, T, d), rnd(41, T, d), rnd(42, T, e), rnd(43, T, d)
    o = forward_with(row_fn, q, k, v, r, h)
    worst = 0.0
    for i in range(T):
        K, V = k[: i + 1], v[: i + 1]
        P1 = np.exp(K @ q[i] / h)
        P2 = P1 * (K @ r[i])
        d1, d2, O1, O2 = P1.sum(), P2.sum(), P1 @ V, P2 @ V
        worst = max(worst, np.abs((1.0 + d2 / d1) * O1 / d1 - O2 / d1 - o[i]).max())
    return worst


def pin_wide_bandwidth(row_fn):
    T, d, e = 10, 4, 4
    q, k, v, r = rnd(50, T, d), rnd(51, T, d), rnd(52, T, e), rnd(53, T, d)
    o = forward_with(row_fn, q, k, v, r, 1e14)
    worst = 0.0
    for i in range(1, T):
        C = np.cov(v[: i + 1].T, k[: i + 1].T, bias=True)[:e, e:]
        ref = v[: i + 1].mean(axis=0) - C @ r[i]
        worst = max(worst, np.abs(ref - o[i]).max())
    return worst


def pin_constant_values(row_fn):
    T, d, h = 9, 4, 1.2
    q, k, r = rnd(60, T, d), rnd(61, T, d), rnd(62, T, d, scale=3.0)
    c = np.array([1.5, -2.0, 0.25, 4.0])
    o = forward_with(row_fn, q, k, np.tile(c, (T, 1)), r, h)
    return np.abs(o - c).max()


def pin_first_token(row_fn):
    worst = 0.0
    for seed, h in enumerate([0.7, 3.0]):
        q, k, v, r = rnd(seed, 1, 4), rnd(seed + 5, 1, 4), rnd(seed + 9, 1, 4), rnd(seed + 13, 1, 4)
        worst = max(worst, np.abs(row_fn(q[0], k, v, r[0], h) - v[0]).max())
    return worst


PINS = {
    "zero_probe_softmax": (pin_zero_probe_softmax, 1e-12),
    "lla_relation": (pin_lla_relation, 1e-9),
    "streaming_combination": (pin_streaming_combination, 1e-11),
    "wide_bandwidth": (pin_wide_bandwidth, 1e-11),
    "constant_values": (pin_constant_values, 1e-12),
    "first_token": (pin_first_token, 1e-12),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_parallax_oracle_pin(name):
    fn, tol = PINS[name]
    assert fn(parallax_row) < tol


# --------------------------------------------------------------------------- invariants

def test_value_affine_equivariance():
    T, d, e, h = 10, 3, 2, 1.5
    q, k, v, r = rnd(70, T, d), rnd(71, T, d), rnd(72, T, e), rnd(73, T, d)
    M, c = rnd(74, e, e), rnd(75, e)
    o = parallax_forward_oracle(q, k, v, r, h)
    o2 = parallax_forward_oracle(q, k, v @ M + c, r, h)
    assert np.abs(o2 - (o @ M + c)).max() < 1e-11


def test_joint_rotation_invariance():
    T, d, e, h = 10, 4, 3, 1.5
    q, k, v, r = rnd(80, T, d), rnd(81, T, d), rnd(82, T, e), rnd(83, T, d)
    Rot, _ = np.linalg.qr(rnd(84, d, d))
    o = parallax_forward_oracle(q, k, v, r, h)
    o2 = parallax_forward_oracle(q @ Rot.T, k @ Rot.T, v, r @ Rot.T, h)
    assert np.abs(o2 - o).max() < 1e-11


def test_affine_in_probe():
    T, d, e, h = 9, 3, 3, 0.9
    q, k, v = rnd(90, T, d), rnd(91, T, d), rnd(92, T, e)
    r1, r2 = rnd(93, T, d), rnd(94, T, d)
    f = lambda r: parallax_forward_oracle(q, k, v, r, h)  # noqa: E731
    assert np.abs(f(r1 + r2) + f(np.zeros_like(r1)) - f(r1) - f(r2)).max() < 1e-11


def test_forward_shapes_and_rows():
    B, H, T, d, e = 2, 3, 7, 4, 2
    q, k, r = rnd(95, B, H, T, d), rnd(96, B, H, T, d), rnd(97, B, H, T, d)
    v = rnd(98, B, H, T, e)
    full = parallax_forward_oracle(q, k, v, r, 1.3)
    assert full.shape == (B, H, T, e)
    rows = [0, 6, 7, 20, B * H * T - 1]
    part = parallax_forward_oracle(q, k, v, r, 1.3, rows=rows)
    assert np.array_equal(part, full.reshape(-1, e)[rows])


# --------------------------------------------------------------------------- planted mistakes

def _mutant(kind):
    def row(q_i, K, V, r_i, h):
        s = K @ q_i / (h * h if kind == "h_squared" else h)
        w = np.exp(s - s.max())
        p = w if kind == "unnormalised" else w / w.sum()
        vbar, kbar = p @ V, p @ K
        if kind == "uncentred":
            sigma = (V * p[:, None]).T @ K
        else:
            sigma = ((V - vbar) * p[:, None]).T @ (K - kbar)
        if kind == "transposed":
            sigma = sigma.T
        probe = r_i / h if kind == "probe_scaled" else r_i
        corr = sigma @ probe
        return vbar + corr if kind == "sign" else vbar - corr
    return row


@pytest.mark.parametrize("kind", ["h_squared", "unnormalised", "uncentred", "transposed",
                                  "probe_scaled", "sign"])
def test_pins_catch_planted_mistakes(kind):
    row = _mutant(kind)
    failed = [name for name, (fn, tol) in PINS.items() if not fn(row) < tol]
    assert failed, f"no pin caught the planted mistake {kind!r}"
