"""Pins for the float64 oracle (CPU only).

The pages print no worked numerical example of LLA, so the oracle is pinned to what the pages
and the mathematics fix instead:

* library routines for special cases: weighted ridge regression with intercept
  (scikit-learn ``Ridge``), and causal softmax attention (``torch`` SDPA in float64);
* closed-form limits stated on the pages: large ridge gives softmax attention, wide bandwidth
  gives unweighted ridge-with-intercept, the first token returns its own value, an exactly
  affine key->value map is reproduced, also when the query lies outside the keys' hull;
* the pages' other forms of the same output: the weighted form sum w(1-t)v / sum w(1-t) with the
  solved probe rho* ("Parallax" blog, Appendix B), the additive correction
  o_SA - (1+eta) Sigma_KV rho* (blog s.2 "Additive Correction to Softmax") and eta as omega
  times a squared Mahalanobis distance (blog Appendix E);
* invariants (constant values, value-affine equivariance, joint rotation of q and k);
* brute-force minimisation of the objective on tiny inputs.

``test_pins_catch_planted_mistakes`` plants plausible mistakes into copies of the oracle's
row function and checks that at least one pin fails for each.
"""
import math

import numpy as np
import pytest
import torch

from oracle import lla_forward_oracle, lla_moments_oracle, lla_row, softmax_attention_oracle


def rnd(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def forward_with(row_fn, q, k, v, h, lam):
    T = q.shape[0]
    return np.stack([row_fn(q[i], k[: i + 1], v[: i + 1], h, lam) for i in range(T)])


# --------------------------------------------------------------------------- pin functions
# Each takes a row function with lla_row's signature and returns the max violation.

def pin_first_token(row_fn):
    worst = 0.0
    for seed, (h, lam) in enumerate([(0.7, 1e-3), (3.0, 1.0), (1.0, 1e4)]):
        q, k, v = rnd(seed, 1, 4), rnd(seed + 10, 1, 4), rnd(seed + 20, 1, 3)
        worst = max(worst, np.abs(row_fn(q[0], k, v, h, lam) - v[0]).max())
    return worst


def pin_large_ridge_softmax(row_fn):
    T, d, e, h = 9, 3, 2, 1.3
    q, k, v = rnd(1, T, d), rnd(2, T, d), rnd(3, T, e)
    o = forward_with(row_fn, q, k, v, h, 1e13)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(k)[None], torch.tensor(v)[None],
        is_causal=True, scale=1.0 / h)[0].numpy()
    return np.abs(o - ref).max() / np.abs(ref).max()


def pin_affine_extrapolation(row_fn):
    # v = A k + c exactly, tiny ridge: every query with more than d affinely independent keys in
    # its prefix gets A q + c, including queries far outside the keys' convex hull.
    T, d, e, h = 14, 3, 2, 2.0
    k = rnd(4, T, d)
    q = rnd(5, T, d) * 3.0 + 4.0          # mostly outside the hull of the keys
    A, c = rnd(6, e, d), rnd(7, e)
    v = k @ A.T + c
    o = forward_with(row_fn, q, k, v, h, 1e-11)
    ref = q @ A.T + c
    return (np.abs(o[d + 1:] - ref[d + 1:]).max() / np.abs(ref).max())


def pin_wide_bandwidth_ridge(row_fn):
    sk = pytest.importorskip("sklearn.linear_model")
    T, d, e, lam = 10, 3, 2, 0.37
    q, k, v = rnd(8, T, d), rnd(9, T, d), rnd(10, T, e)
    o = forward_with(row_fn, q, k, v, 1e14, lam)
    worst = 0.0
    for i in range(T):
        r = sk.Ridge(alpha=lam, fit_intercept=True, solver="svd").fit(k[: i + 1], v[: i + 1])
        worst = max(worst, np.abs(r.predict(q[i:i + 1])[0] - o[i]).max())
    return worst


def pin_weighted_ridge_library(row_fn):
    # Raw (unshifted) kernel weights exp(q.k/h) and absolute lambda, solved by scikit-learn.
    sk = pytest.importorskip("sklearn.linear_model")
    T, d, e = 11, 3, 2
    worst = 0.0
    for seed, (h, lam) in enumerate([(0.9, 0.05), (2.5, 1e-3), (1.7, 3.0)]):
        q, k, v = rnd(30 + seed, T, d), rnd(40 + seed, T, d), rnd(50 + seed, T, e)
        o = forward_with(row_fn, q, k, v, h, lam)
        for i in range(T):
            w = np.exp(k[: i + 1] @ q[i] / h)
            r = sk.Ridge(alpha=lam, fit_intercept=True, solver="svd").fit(
                k[: i + 1], v[: i + 1], sample_weight=w)
            worst = max(worst, np.abs(r.predict(q[i:i + 1])[0] - o[i]).max())
    return worst


def _page_quantities(q_i, K, V, h, lam):
    """omega, mu, Sigma, rho* with query-centred z = k - q (blog s.2 Canonical Formulation)."""
    w = np.exp(K @ q_i / h)
    Z = K - q_i
    omega = w.sum()
    mu = w @ Z
    Sigma = (Z * w[:, None]).T @ Z + lam * np.eye(K.shape[1])
    rho = np.linalg.solve(Sigma, mu)
    return w, Z, omega, mu, Sigma, rho


def pin_page_weighted_form(row_fn):
    # Blog Appendix B: the LLA forward is sum_j w_j (1 - t_j) v_j / sum_j w_j (1 - t_j),
    # t_j = rho*^T z_j, rho* = Sigma^-1 mu.
    T, d, e = 13, 4, 3
    worst = 0.0
    for seed, (h, lam) in enumerate([(1.1, 0.02), (3.0, 0.5)]):
        q, k, v = rnd(60 + seed, T, d), rnd(70 + seed, T, d), rnd(80 + seed, T, e)
        o = forward_with(row_fn, q, k, v, h, lam)
        for i in range(T):
            w, Z, _, _, _, rho = _page_quantities(q[i], k[: i + 1], v[: i + 1], h, lam)
            a = w * (1.0 - Z @ rho)
            worst = max(worst, np.abs(a @ v[: i + 1] / a.sum() - o[i]).max())
    return worst


def pin_additive_correction(row_fn):
    # Blog s.2 "Additive Correction to Softmax": o = o_SA - (1 + eta) Sigma_KV rho*,
    # eta = tbar / (1 - tbar), tbar = E_p[rho*^T z], Sigma_KV = E_p[(v - vbar)(k - kbar)^T].
    T, d, e, h, lam = 12, 3, 2, 1.4, 0.08
    q, k, v = rnd(90, T, d), rnd(91, T, d), rnd(92, T, e)
    o = forward_with(row_fn, q, k, v, h, lam)
    worst = 0.0
    for i in range(T):
        K, V = k[: i + 1], v[: i + 1]
        w, Z, omega, _, _, rho = _page_quantities(q[i], K, V, h, lam)
        p = w / omega
        vbar, kbar = p @ V, p @ K
        Skv = ((V - vbar) * p[:, None]).T @ (K - kbar)
        tbar = p @ (Z @ rho)
        eta = tbar / (1.0 - tbar)
        worst = max(worst, np.abs(vbar - (1.0 + eta) * Skv @ rho - o[i]).max())
    return worst


def pin_constant_values(row_fn):
    T, d, h, lam = 10, 3, 1.2, 1e-2
    q, k = rnd(100, T, d), rnd(101, T, d)
    c = np.array([1.5, -2.0, 0.25])
    o = forward_with(row_fn, q, k, np.tile(c, (T, 1)), h, lam)
    return np.abs(o - c).max()


def _offset_prefix(seed, n, d, e, offset):
    """n keys N(0,1) + `offset` in every coordinate and a query aligned with that offset, so that
    the max logit m is large and the effective ridge lambda e^-m tiny; values N(0,1)."""
    K = rnd(seed, n, d) + offset
    q = rnd(seed + 1, d) + offset / 8.0
    V = rnd(seed + 2, n, e)
    return q, K, V


def pin_min_norm_interpolation(row_fn):
    # Fewer keys than dimensions and lambda e^-m ~ 1e-100: the fit interpolates every key,
    # b + W (k_j - q) = v_j, and the ridge picks the smallest |W|_F among the interpolants, whose
    # closed form needs neither the weights nor the centring: W^T = pinv(K_{1:} - k_0) (V_{1:} - v_0),
    # b = v_0 + W (q - k_0).
    d, e, h, lam = 64, 8, 8.0, 1e-2
    worst = 0.0
    for seed, n in enumerate([2, 9, 24, 40]):
        q, K, V = _offset_prefix(200 + 3 * seed, n, d, e, 16.0)
        Wt = np.linalg.pinv(K[1:] - K[0]) @ (V[1:] - V[0])
        ref = V[0] + (q - K[0]) @ Wt
        worst = max(worst, np.abs(row_fn(q, K, V, h, lam) - ref).max() / np.abs(ref).max())
    return worst


def pin_exact_normal_equations(row_fn):
    # The objective's stationarity conditions over (b, W), uncentred and unshifted (raw weights
    # exp(q.k/h), absolute lambda), solved in 50-digit arithmetic: prefixes shorter than d under a
    # tiny effective ridge, one with a moderate ridge and one longer than d.
    mp = pytest.importorskip("mpmath")
    worst = 0.0
    with mp.workdps(50):
        for seed, (n, d, e, h, lam, off) in enumerate([(4, 6, 2, 1.0, 1e-2, 12.0),
                                                      (3, 5, 2, 0.5, 1e-3, 9.0),
                                                      (5, 6, 3, 2.0, 0.3, 1.0),
                                                      (9, 4, 2, 1.5, 1e-4, 6.0)]):
            q, K, V = _offset_prefix(300 + 3 * seed, n, d, e, off)
            X = mp.matrix([[1] + [mp.mpf(K[j, a]) - mp.mpf(q[a]) for a in range(d)]
                           for j in range(n)])
            w = [mp.exp(mp.fsum(mp.mpf(K[j, a]) * mp.mpf(q[a]) for a in range(d)) / h)
                 for j in range(n)]
            M = X.T * mp.diag(w) * X
            for a in range(1, d + 1):
                M[a, a] += lam
            got = row_fn(q, K, V, h, lam)
            for c in range(e):
                rhs = X.T * mp.diag(w) * mp.matrix(V[:, c].tolist())
                b = float(mp.lu_solve(M, rhs)[0])
                worst = max(worst, abs(got[c] - b) / max(1.0, abs(b)))
    return worst


PINS = {
    "first_token": (pin_first_token, 1e-10),
    "large_ridge_softmax": (pin_large_ridge_softmax, 1e-8),
    "affine_extrapolation": (pin_affine_extrapolation, 1e-7),
    "wide_bandwidth_ridge": (pin_wide_bandwidth_ridge, 1e-9),
    "weighted_ridge_library": (pin_weighted_ridge_library, 1e-9),
    "page_weighted_form": (pin_page_weighted_form, 1e-9),
    "additive_correction": (pin_additive_correction, 1e-9),
    "constant_values": (pin_constant_values, 1e-10),
    "min_norm_interpolation": (pin_min_norm_interpolation, 1e-9),
    "exact_normal_equations": (pin_exact_normal_equations, 1e-9),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(name):
    fn, tol = PINS[name]
    assert fn(lla_row) < tol


# --------------------------------------------------------------------------- more pins


def test_eta_nonnegative_mahalanobis():
    """Blog Appendix E: eta = omega * (q - kbar)^T A^-1 (q - kbar) >= 0, A = Sigma - omega zbar zbar^T."""
    T, d, e, h, lam = 15, 4, 2, 1.1, 0.03
    q, k, v = rnd(110, T, d), rnd(111, T, d), rnd(112, T, e)
    for i in range(T):
        K = k[: i + 1]
        w, Z, omega, mu, Sigma, rho = _page_quantities(q[i], K, v[: i + 1], h, lam)
        zbar = mu / omega
        tbar = zbar @ rho
        A = Sigma - omega * np.outer(zbar, zbar)
        eta_m = omega * zbar @ np.linalg.solve(A, zbar)
        assert eta_m >= -1e-12
        assert abs(tbar / (1 - tbar) - eta_m) <= 1e-9 * max(1.0, eta_m)


def test_softmax_oracle_matches_sdpa():
    T, d, e, h = 17, 5, 3, 2.2
    q, k, v = rnd(120, 2, T, d), rnd(121, 2, T, d), rnd(122, 2, T, e)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True, scale=1 / h).numpy()
    assert np.abs(softmax_attention_oracle(q, k, v, h) - ref).max() < 1e-12


def test_value_affine_equivariance():
    T, d, e, h, lam = 12, 3, 3, 1.5, 0.02
    q, k, v = rnd(130, T, d), rnd(131, T, d), rnd(132, T, e)
    M, c = rnd(133, e, 2), rnd(134, 2)
    o = lla_forward_oracle(q, k, v, h, lam)
    o2 = lla_forward_oracle(q, k, v @ M + c, h, lam)
    assert np.abs(o2 - (o @ M + c)).max() < 1e-9


def test_joint_rotation_invariance():
    T, d, e, h, lam = 12, 4, 2, 1.3, 0.05
    q, k, v = rnd(140, T, d), rnd(141, T, d), rnd(142, T, e)
    R, _ = np.linalg.qr(rnd(143, d, d))
    o = lla_forward_oracle(q, k, v, h, lam)
    o2 = lla_forward_oracle(q @ R.T, k @ R.T, v, h, lam)
    assert np.abs(o - o2).max() < 1e-9


def test_brute_force_minimisation():
    """Minimise the LLA objective over (b, W) with a generic iterative solver on tiny inputs."""
    scipy_opt = pytest.importorskip("scipy.optimize")
    T, d, e, h, lam = 6, 2, 2, 0.8, 0.15
    q, k, v = rnd(150, T, d), rnd(151, T, d), rnd(152, T, e)
    for i in [0, 2, 5]:
        K, V = k[: i + 1], v[: i + 1]
        w = np.exp(K @ q[i] / h)

        def resid(x):
            b, W = x[:e], x[e:].reshape(e, d)
            r = np.sqrt(w)[:, None] * (V - b - (K - q[i]) @ W.T)
            return np.concatenate([r.ravel(), math.sqrt(lam) * W.ravel()])

        x = scipy_opt.least_squares(resid, np.zeros(e + e * d), xtol=1e-15, ftol=1e-15,
                                    gtol=1e-15, method="trf").x
        assert np.abs(x[:e] - lla_row(q[i], K, V, h, lam)).max() < 1e-5


def test_forward_shapes_and_rows():
    B, H, T, d, e = 2, 3, 7, 3, 2
    q, k, v = rnd(160, B, H, T, d), rnd(161, B, H, T, d), rnd(162, B, H, T, e)
    full = lla_forward_oracle(q, k, v, 1.0, 0.1)
    assert full.shape == (B, H, T, e)
    rows = [0, 6, 7, 20, B * H * T - 1]
    part = lla_forward_oracle(q, k, v, 1.0, 0.1, rows=rows)
    flat = full.reshape(-1, e)
    assert np.abs(part - flat[rows]).max() == 0.0


# --------------------------------------------------------------------------- moments oracle


def test_moments_first_query_and_loops():
    T, d, e, h = 6, 3, 2, 1.7
    q, k, v = rnd(170, 1, 1, T, d), rnd(171, 1, 1, T, d), rnd(172, 1, 1, T, e)
    mo = lla_moments_oracle(q, k, v, h, range(T))
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    # first query: one key, weight 1 after the max shift
    assert abs(mo["m"][0] - Q[0] @ K[0] / h) < 1e-14 and abs(mo["omega"][0] - 1.0) < 1e-14
    assert np.abs(mo["Skk"][0] - np.outer(K[0], K[0])).max() < 1e-14
    # element-wise loop sums on a later query
    i = 4
    s = [sum(Q[i, a] * K[j, a] for a in range(d)) / h for j in range(i + 1)]
    m = max(s)
    w = [math.exp(sj - m) for sj in s]
    for a in range(d):
        assert abs(mo["sk"][i][a] - sum(w[j] * K[j, a] for j in range(i + 1))) < 1e-12
        for b in range(d):
            assert abs(mo["Skk"][i][a, b] - sum(w[j] * K[j, a] * K[j, b] for j in range(i + 1))) < 1e-12
        for c in range(e):
            assert abs(mo["Svk"][i][c, a] - sum(w[j] * V[j, c] * K[j, a] for j in range(i + 1))) < 1e-12


def test_moments_centred_form_reproduces_forward():
    """vbar + C_vk (C_kk + lam e^-m I)^-1 (q - kbar) from the moments equals the oracle."""
    T, d, e, h, lam = 20, 4, 3, 1.6, 0.04
    q, k, v = rnd(180, 1, 2, T, d), rnd(181, 1, 2, T, d), rnd(182, 1, 2, T, e)
    idx = list(range(2 * T))
    mo = lla_moments_oracle(q, k, v, h, idx)
    ref = lla_forward_oracle(q, k, v, h, lam, rows=idx)
    Q = q.reshape(-1, d)
    for n in idx:
        om, sk, sv = mo["omega"][n], mo["sk"][n], mo["sv"][n]
        kbar, vbar = sk / om, sv / om
        Ckk = mo["Skk"][n] - om * np.outer(kbar, kbar)
        Cvk = mo["Svk"][n] - om * np.outer(vbar, kbar)
        y = np.linalg.solve(Ckk + lam * np.exp(-mo["m"][n]) * np.eye(d), Q[n] - kbar)
        assert np.abs(vbar + Cvk @ y - ref[n]).max() < 1e-9


# --------------------------------------------------------------------------- planted mistakes


def _mutant(kind):
    """The oracle's row with one plausible mistake planted (or, for "joint_lstsq", the joint
    least-squares solve over (b, W), which leaves the ridge limit once sqrt(lambda e^-m) falls
    below its rank cut)."""
    def joint(q_i, K, V, h, lam):
        n, d = K.shape
        s = K @ q_i / h
        m = s.max()
        sw = np.sqrt(np.exp(s - m))
        A = np.zeros((n + d, d + 1))
        A[:n, 0] = sw
        A[:n, 1:] = sw[:, None] * (K - q_i[None, :])
        A[n:, 1:] = np.sqrt(lam * np.exp(-m)) * np.eye(d)
        Bm = np.zeros((n + d, V.shape[1]))
        Bm[:n] = sw[:, None] * V
        return np.linalg.lstsq(A, Bm, rcond=None)[0][0]

    def row(q_i, K, V, h, lam):
        n, d = K.shape
        s = K @ q_i / (h * h if kind == "h_squared" else h)
        m = s.max()
        w = np.exp(s - m)
        lam_t = {"lam_unscaled": lam, "lam_relative": lam * w.sum()}.get(kind, lam * np.exp(-m))
        p = {"unweighted_means": np.full(n, 1.0 / n), "means_unnormalised": w}.get(kind, w / w.sum())
        kbar, vbar = p @ K, p @ V
        sw = w if kind == "weights_squared" else np.sqrt(w)
        Xw = sw[:, None] * (K - (q_i if kind == "keys_centred_at_query" else kbar))
        Vw = sw[:, None] * (V - vbar)
        U, S, Vt = np.linalg.svd(Xw, full_matrices=False)
        cut = 0.0 if kind == "no_rank_cut" else \
            np.finfo(np.float64).eps * max(n, d) * np.linalg.norm(sw[:, None] * K)
        ridge = lam_t * lam_t if kind == "ridge_squared" else lam_t
        f = np.where(S > cut, S / (S * S + ridge), 0.0)
        Wt = Vt.T @ (f[:, None] * (U.T @ Vw))
        sign = -1.0 if kind == "intercept_sign" else 1.0
        return vbar + sign * (q_i - kbar) @ Wt
    return joint if kind == "joint_lstsq" else row


@pytest.mark.parametrize("kind", ["h_squared", "lam_unscaled", "lam_relative", "weights_squared",
                                  "unweighted_means", "means_unnormalised",
                                  "keys_centred_at_query", "ridge_squared",
                                  "intercept_sign", "no_rank_cut", "joint_lstsq"])
def test_pins_catch_planted_mistakes(kind):
    row = _mutant(kind)
    failed = [name for name, (fn, tol) in PINS.items() if not fn(row) < tol]
    assert failed, f"no pin caught the planted mistake {kind!r}"
