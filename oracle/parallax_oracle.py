"""Float64 CPU oracle for the causal Parallax forward with a given probe.

TEST INFRASTRUCTURE. Only the test suite (``tests/``), ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run this module. The product path
(``local_linear_attention_gb300``) never imports it, and this module imports nothing from the
product.

What is computed, and where it is defined
-----------------------------------------
Sources (cited by page title and section):

* [P1] "Parallax" (Tilde Research blog), section 2, paragraphs "Parallax" and "Additive
  Correction to Softmax", and Appendix B "LLA as an additive correction -- the derivation".
* [P1-C] the same blog, Appendix C "Hopper decode kernel", item 3, which prints the output
  combination of the streaming kernel.

The pages write LLA as softmax attention plus a correction: ``o_i = o_SA_i - (1 + eta_i)
Sigma_KV^(i) rho*_i``, where ``o_SA_i`` is the causal softmax output with weights
``p_ij = exp(q_i . k_j / h) / sum_l exp(q_i . k_l / h)``, ``Sigma_KV^(i)`` is the
``p_i``-weighted covariance of values and keys over the causal prefix,
``E_p[v k^T] - vbar kbar^T`` (Appendix B's cross-moment factorisation), and ``rho*_i`` is
LLA's solved probe. Parallax drops ``eta`` and takes the probe ``rho_i`` as an input (the
pages learn it as ``W_R x_i``; here it is a given tensor R). So for each query

    o_i = o_SA_i - Sigma_KV^(i) rho_i.

The pages' display equations were lost in extraction; this is the plainest reading of their
text ("the softmax output minus a learned projection of the local KV covariance"), and it is
the combination ``(1 + d2/d1) O1/d1 - O2/d1`` that Appendix C prints for the streaming kernel
with ``O1 = P V``, ``d1 = rowsum P``, ``O2 = (P .* (R K^T)) V``, ``d2 = rowsum(P .* (R K^T))``.

The oracle evaluates the covariance form directly (explicit weighted means and the explicit
covariance matrix), not the streaming form. Pins: ``tests/test_parallax_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

from .lla_oracle import _f64

__all__ = ["parallax_row", "parallax_forward_oracle"]


def parallax_row(q_i: np.ndarray, K: np.ndarray, V: np.ndarray, r_i: np.ndarray,
                 h: float) -> np.ndarray:
    """Parallax output for one query over its causal prefix K [n, d], V [n, e] ([P1] s.2).

    o = vbar - Sigma_KV r_i with p = softmax(K q_i / h), vbar = p V, kbar = p K and
    Sigma_KV = sum_j p_j (v_j - vbar)(k_j - kbar)^T  (an e x d matrix).
    """
    s = K @ q_i / h
    w = np.exp(s - s.max())
    p = w / w.sum()
    vbar = p @ V
    kbar = p @ K
    sigma_kv = ((V - vbar) * p[:, None]).T @ (K - kbar)
    return vbar - sigma_kv @ r_i


def parallax_forward_oracle(q, k, v, r, h: float, rows=None) -> np.ndarray:
    """Causal Parallax forward in float64.

    q, k, r: [..., T, d]; v: [..., T, e]. rows: None for every query (returns [..., T, e]);
    otherwise flat query indices ``bh * T + i`` and the result is [len(rows), e].
    """
    Q, K, V, R = _f64(q), _f64(k), _f64(v), _f64(r)
    if Q.ndim == 2:
        Q, K, V, R = Q[None], K[None], V[None], R[None]
    lead = Q.shape[:-2]
    T, d = Q.shape[-2:]
    e = V.shape[-1]
    Q, K, R = Q.reshape(-1, T, d), K.reshape(-1, T, d), R.reshape(-1, T, d)
    V = V.reshape(-1, T, e)
    if rows is None:
        out = np.zeros((Q.shape[0], T, e))
        for bh in range(Q.shape[0]):
            for i in range(T):
                out[bh, i] = parallax_row(Q[bh, i], K[bh, : i + 1], V[bh, : i + 1], R[bh, i], h)
        return out.reshape(*lead, T, e) if lead else out[0]
    rows = np.asarray(list(rows), dtype=np.int64)
    out = np.zeros((len(rows), e))
    for n, rr in enumerate(rows):
        bh, i = divmod(int(rr), T)
        out[n] = parallax_row(Q[bh, i], K[bh, : i + 1], V[bh, : i + 1], R[bh, i], h)
    return out


# ----------------------------------------------------------------------------- backward
# The pages' Appendix F ("Parallax backward (closed form)") names the row scalars, the cached
# quantities (o_i, vbar_i, tbar_i, omega_i, m_i) and the row-tile / column-tile split, but its
# formulas were lost in extraction. The backward below is the gradient of the forward above
# (parallax_row), taken step by step in the forward's own order:
#
#   p_j = softmax_j(q_i . k_j / h),  t_j = r_i . k_j,  tbar = sum_j p_j t_j,
#   o_i = vbar - Sigma_KV r_i = sum_j a_j v_j,  a_j = p_j (1 + tbar - t_j)
#
# (vbar - Sigma_KV r = sum p v - sum p (v - vbar)(t - tbar) = sum p (1 + tbar - t) v, since
# sum p (t - tbar) = 0). With the upstream gradient dO_i and g_j = dO_i . v_j:
#   dv_j += a_j dO_i;
#   through t (directly, and through tbar = sum p t):  dt_j = p_j (G - g_j),  G = sum_j p_j g_j
#     = dO_i . vbar, so dr_i = sum_j dt_j k_j and dk_j += dt_j r_i;
#   through p (directly in a, and through tbar):  u_j = dL/dp_j = (1 + tbar - t_j) g_j + G t_j;
#     the softmax gives ds_j = p_j (u_j - D),  D = sum_j p_j u_j = dO_i . o_i + G tbar, and
#     s_j = q_i . k_j / h gives dq_i = sum_j ds_j k_j / h and dk_j += ds_j q_i / h.
# D and G are the row scalars the pages' kernel caches beyond the softmax statistics.


def parallax_backward_row(q_i, K, V, r_i, do_i, h):
    """Gradient of parallax_row(q_i, K, V, r_i, h) . do_i with respect to q_i, r_i and the prefix
    K [n, d], V [n, e]. Returns (dq_i [d], dr_i [d], dK [n, d], dV [n, e])."""
    s = K @ q_i / h
    w = np.exp(s - s.max())
    p = w / w.sum()
    t = K @ r_i
    tbar = p @ t
    a = p * (1.0 + tbar - t)
    o = a @ V
    g = V @ do_i
    G = p @ g
    dt = p * (G - g)
    u = (1.0 + tbar - t) * g + G * t
    D = do_i @ o + G * tbar
    ds = p * (u - D)
    dq = K.T @ ds / h
    dr = K.T @ dt
    dK = np.outer(ds, q_i) / h + np.outer(dt, r_i)
    dV = np.outer(a, do_i)
    return dq, dr, dK, dV


def parallax_backward_oracle(q, k, v, r, do, h: float):
    """Causal Parallax backward in float64: gradients of sum_i parallax(i) . do_i.

    q, k, r: [..., T, d]; v, do: [..., T, e]. Returns (dq, dk, dv, dr) shaped like q, k, v, r.
    """
    Q, K, V, R, DO = _f64(q), _f64(k), _f64(v), _f64(r), _f64(do)
    squeeze = Q.ndim == 2
    if squeeze:
        Q, K, V, R, DO = Q[None], K[None], V[None], R[None], DO[None]
    lead = Q.shape[:-2]
    T, d = Q.shape[-2:]
    e = V.shape[-1]
    Q, K, R = Q.reshape(-1, T, d), K.reshape(-1, T, d), R.reshape(-1, T, d)
    V, DO = V.reshape(-1, T, e), DO.reshape(-1, T, e)
    dq, dk, dr = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(R)
    dv = np.zeros_like(V)
    for bh in range(Q.shape[0]):
        for i in range(T):
            gq, gr, gK, gV = parallax_backward_row(Q[bh, i], K[bh, : i + 1], V[bh, : i + 1],
                                                   R[bh, i], DO[bh, i], h)
            dq[bh, i] = gq
            dr[bh, i] = gr
            dk[bh, : i + 1] += gK
            dv[bh, : i + 1] += gV
    outs = []
    for x, last in ((dq, d), (dk, d), (dv, e), (dr, d)):
        x = x.reshape(*lead, T, last)
        outs.append(x[0] if squeeze else x)
    return tuple(outs)
