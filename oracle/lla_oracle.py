"""Float64 CPU oracle for the causal forward pass of Local Linear Attention (LLA).

TEST INFRASTRUCTURE. Only the test suite (``tests/``), ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run this module. The product
path (``local_linear_attention_gb300``) never imports it, and this module imports nothing
from the product: the two share no code. Inputs are plain arrays; the seeded generators that
feed both sides hold none of the method's arithmetic.

What is computed, and where it is defined
-----------------------------------------
Sources (cited by page title and section):

* [P1] "Parallax" (Tilde Research blog, blog.tilderesearch.com/blog/parallax),
  section 2 "Parallax & Local Linear Attention", paragraph "Canonical Formulation".
* [P2] "Parallax: Parameterized Local Linear Attention for Language Modeling"
  (arXiv 2605.29157, HTML), section 2, the test-time-regression paragraph and the
  LLA paragraph that follows it.

Both pages define LLA as follows. For query q_i, fit the local linear estimator
``f(x) = b + W (x - q_i)`` to the causal prefix of key/value pairs ``{(k_j, v_j)}_{j <= i}``
by weighted least squares with kernel weights ``w_ij = exp(q_i . k_j / h)`` and ridge penalty
``lambda * ||W||_F^2`` on the slope only. The prediction at the query is ``f(q_i) = b``, the
intercept. (The display equation with the prediction was lost when the pages were extracted;
the intercept of this weighted ridge problem is the plainest reading of "the prediction of the
local linear estimator at q_i", and it agrees with the pages' additive-correction form and
their softmax / affine limits, which the oracle's tests check.)

The oracle solves that problem one query at a time in two exact textbook steps: no normal
equations, no moments, no blocking. (1) The intercept is not penalised, so for any slope W the
best b is ``vbar - W (kbar - q_i)`` with kbar, vbar the weighted means of the keys and values;
putting it back leaves a ridge regression of the weighted-centred values on the
weighted-centred keys, whose slope is ``W^T = V S (S^2 + lambda I)^-1 U^T Vw`` through the thin
SVD ``Xw = U S V^T`` of the square-root-weighted centred keys Xw (Vw the same for the values).
(2) The prediction is ``b = vbar + W (q_i - kbar)``. Multiplying the whole objective by
``exp(-m_i)`` with ``m_i = max_j q_i . k_j / h`` leaves the minimiser unchanged and keeps
``exp`` finite; the ridge term is scaled by the same factor, so lambda stays absolute against
the raw kernel weights ``exp(q . k / h)`` as written on the pages.

Singular values of Xw at the rounding level of the centring carry no data: the centring makes
``sum_j w_j (k_j - kbar) = 0`` (one exact null vector), and linearly dependent keys add more; in
exact arithmetic the values' part along them is zero, so the ridge solution gives them zero
weight. Below ``eps * max(n, d) * |W^(1/2) K|_F`` they are cut (given zero weight) instead of
dividing rounding noise by a ridge that may be far smaller than it (with lambda e^-m ~ 1e-22, as
on early prefixes seen by a query aligned with a large common key offset). A joint least-squares
solve over (b, W) instead would return, once sqrt(lambda e^-m) fell below its own rank cut, the
minimum-norm (b, W) rather than this ridge limit.

Parity pins: every function here is pinned by the CPU tests in ``tests/test_oracle_pins.py``
(library routines, closed-form limits printed on the pages, invariants, brute force).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "lla_row",
    "lla_forward_oracle",
    "lla_moments_oracle",
    "softmax_attention_oracle",
]


def _f64(x) -> np.ndarray:
    """Convert a torch tensor or array-like to a float64 numpy array (bf16 -> f64 is exact)."""
    if hasattr(x, "detach"):  # torch tensor, without importing torch here
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def lla_row(q_i: np.ndarray, K: np.ndarray, V: np.ndarray, h: float, lam: float) -> np.ndarray:
    """Prediction of LLA for one query over its causal prefix ([P1] s.2 Canonical Formulation).

    q_i: [d]; K: [n, d] prefix keys k_1..k_n (n >= 1, j <= i inclusive); V: [n, e] prefix values.
    Minimises  sum_j w_j ||v_j - b - W (k_j - q_i)||^2 + lam ||W||_F^2  over (b, W) and returns b.
    """
    n, d = K.shape
    s = K @ q_i / h                      # logits q_i . k_j / h
    m = s.max()
    w = np.exp(s - m)                    # kernel weights times the common factor exp(-m)
    lam_t = lam * np.exp(-m)             # ridge scaled by the same factor
    omega = w.sum()
    kbar, vbar = w @ K / omega, w @ V / omega
    sw = np.sqrt(w)
    Xw = sw[:, None] * (K - kbar)        # square-root-weighted centred keys   [n, d]
    Vw = sw[:, None] * (V - vbar)        # square-root-weighted centred values [n, e]
    U, S, Vt = np.linalg.svd(Xw, full_matrices=False)
    cut = np.finfo(np.float64).eps * max(n, d) * np.linalg.norm(sw[:, None] * K)
    f = np.where(S > cut, S / (S * S + lam_t), 0.0)
    Wt = Vt.T @ (f[:, None] * (U.T @ Vw))  # the slope, transposed [d, e]
    return vbar + (q_i - kbar) @ Wt        # the intercept b


def _flatten(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim == 2:
        q, k, v = q[None], k[None], v[None]
    lead = q.shape[:-2]
    T, d = q.shape[-2:]
    e = v.shape[-1]
    return q.reshape(-1, T, d), k.reshape(-1, T, d), v.reshape(-1, T, e), lead


def lla_forward_oracle(q, k, v, h: float, lam: float, rows=None) -> np.ndarray:
    """Causal LLA forward in float64.

    q, k: [..., T, d]; v: [..., T, e] (any leading batch/head dims, or plain [T, d]).
    rows: None for every query (returns [..., T, e]); otherwise an iterable of flat query
    indices ``r = bh * T + i`` (bh = flattened leading index, i = 0-based position) and the
    result is [len(rows), e] in that order.
    """
    Q, K, V, lead = _flatten(q, k, v)
    BH, T, d = Q.shape
    e = V.shape[-1]
    if rows is None:
        out = np.zeros((BH, T, e))
        for bh in range(BH):
            for i in range(T):
                out[bh, i] = lla_row(Q[bh, i], K[bh, : i + 1], V[bh, : i + 1], h, lam)
        return out.reshape(*lead, T, e) if lead else out[0]
    rows = np.asarray(list(rows), dtype=np.int64)
    out = np.zeros((len(rows), e))
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), T)
        out[n] = lla_row(Q[bh, i], K[bh, : i + 1], V[bh, : i + 1], h, lam)
    return out


def lla_moments_oracle(q, k, v, h: float, idx):
    """Max-shifted kernel-weighted moments of the causal prefix, float64.

    For each flat query index r = bh * T + i: m = max_{j<=i} q_i.k_j/h, w_j = exp(q_i.k_j/h - m),
    omega = sum w_j, sk = sum w_j k_j, sv = sum w_j v_j, Skk = sum w_j k_j k_j^T,
    Svk = sum w_j v_j k_j^T. These are the raw (origin-centred) sums from which the pages'
    omega_i, mu_i and Sigma_i ([P1] s.2 Canonical Formulation) follow by re-centring at q_i.
    Returns a dict of arrays with a leading axis of len(idx).
    """
    Q, K, V, _ = _flatten(q, k, v)
    BH, T, d = Q.shape
    e = V.shape[-1]
    idx = np.asarray(list(idx), dtype=np.int64)
    n = len(idx)
    res = {
        "m": np.zeros(n), "omega": np.zeros(n), "sk": np.zeros((n, d)), "sv": np.zeros((n, e)),
        "Skk": np.zeros((n, d, d)), "Svk": np.zeros((n, e, d)),
    }
    for t, r in enumerate(idx):
        bh, i = divmod(int(r), T)
        Kp, Vp = K[bh, : i + 1], V[bh, : i + 1]
        s = Kp @ Q[bh, i] / h
        m = s.max()
        w = np.exp(s - m)
        res["m"][t] = m
        res["omega"][t] = w.sum()
        res["sk"][t] = w @ Kp
        res["sv"][t] = w @ Vp
        res["Skk"][t] = (Kp * w[:, None]).T @ Kp
        res["Svk"][t] = (Vp * w[:, None]).T @ Kp
    return res


def softmax_attention_oracle(q, k, v, h: float) -> np.ndarray:
    """Causal softmax attention with logit scale 1/h (the Nadaraya-Watson estimator, [P1] s.1).

    Used only as the large-ridge limit LLA must reach ([P1] s.2 "Strong regularization limit").
    """
    Q, K, V, lead = _flatten(q, k, v)
    BH, T, d = Q.shape
    out = np.zeros((BH, T, V.shape[-1]))
    for bh in range(BH):
        S = Q[bh] @ K[bh].T / h
        S = np.where(np.tril(np.ones((T, T), dtype=bool)), S, -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        out[bh] = (P / P.sum(axis=1, keepdims=True)) @ V[bh]
    return out.reshape(*lead, T, V.shape[-1]) if lead else out[0]
