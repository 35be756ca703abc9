"""Pins for the float64 Parallax backward oracle (CPU only).

The pages' Appendix F ("Parallax backward (closed form)") lost its formulas in extraction, so the
backward oracle is the gradient of the forward oracle taken by the chain rule. It is pinned to:

* central finite differences of the forward oracle (``parallax_forward_oracle``, a separate
  function): the directional derivative of sum_i o_i . dO_i along random directions in q, k, v and
  the probe r;
* a zero probe: Parallax is causal softmax attention ("Parallax" blog s.6 "With W_R = 0, Parallax
  is exactly Softmax Attention"), so dq, dk and dv equal the backward of ``torch`` SDPA in float64;
* linearity in the probe: o_i = vbar_i - Sigma_KV^(i) r_i (blog s.2), so dr_i = -Sigma_KV^(i)T dO_i
  with the covariance computed directly;
* invariants: shifting every key by one vector leaves every output unchanged (the logit shift is
  constant over a row and the covariance is shift-free), so sum_j dk_j = 0; shifting every value by
  c shifts every output by c, so sum_j dv_j = sum_i dO_i.

``test_pins_catch_planted_mistakes`` plants plausible mistakes into copies of the row gradient and
checks that at least one pin fails for each.

The same pins (finite differences, the SDPA backward at r = 0, dr = -Sigma_KV^T dO, and agreement of
an unbatched call with the matching head of a batched one) also run on ``parallax_backward_oracle``
itself, the whole-tensor function the GPU tests compare against, with several heads of unequal
content; ``test_whole_tensor_pins_catch_planted_mistakes`` plants mistakes of its bookkeeping (a
swapped return order, a causal slice that drops the diagonal, transposed heads, values taken from
another head) and checks that at least one pin fails for each.
"""
import numpy as np
import pytest
import torch

from oracle import parallax_backward_oracle, parallax_backward_row, parallax_forward_oracle


def rnd(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def backward_with(row_fn, q, k, v, r, do, h):
    T = q.shape[0]
    dq, dk, dv, dr = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(r)
    for i in range(T):
        gq, gr, gK, gV = row_fn(q[i], k[: i + 1], v[: i + 1], r[i], do[i], h)
        dq[i], dr[i] = gq, gr
        dk[: i + 1] += gK
        dv[: i + 1] += gV
    return dq, dk, dv, dr


def inputs(seed, T=7, d=4, e=3, rscale=0.5):
    q, k = rnd(seed, T, d), rnd(seed + 1, T, d)
    v, do = rnd(seed + 2, T, e), rnd(seed + 3, T, e)
    r = rnd(seed + 4, T, d, scale=rscale)
    return q, k, v, r, do


# ----------------------------------------------------------------------------- pins
def pin_finite_differences(row_fn, seed=0, h=1.7):
    q, k, v, r, do = inputs(seed)
    grads = backward_with(row_fn, q, k, v, r, do, h)
    eps = 1e-5
    for which in range(4):  # q, k, v, r
        delta = rnd(seed + 10 + which, *(q, k, v, r)[which].shape)
        plus = [x.copy() for x in (q, k, v, r)]
        minus = [x.copy() for x in (q, k, v, r)]
        plus[which] += eps * delta
        minus[which] -= eps * delta
        lp = np.sum(parallax_forward_oracle(*plus, h) * do)
        lm = np.sum(parallax_forward_oracle(*minus, h) * do)
        fd = (lp - lm) / (2 * eps)
        an = np.sum(grads[which] * delta)
        if not abs(fd - an) <= 1e-7 * max(1.0, abs(fd)):
            return False
    return True


def pin_zero_probe_is_sdpa_backward(row_fn, seed=20, h=1.3):
    q, k, v, _, do = inputs(seed, T=9, d=5, e=4)
    r = np.zeros_like(q)
    dq, dk, dv, _ = backward_with(row_fn, q, k, v, r, do, h)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=True, scale=1.0 / h)[0, 0]
    (o * torch.tensor(do)).sum().backward()
    return all(np.allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12)
               for a, b in ((dq, tq), (dk, tk), (dv, tv)))


def pin_probe_gradient_is_covariance(row_fn, seed=30, h=2.1):
    q, k, v, r, do = inputs(seed)
    _, _, _, dr = backward_with(row_fn, q, k, v, r, do, h)
    for i in range(q.shape[0]):
        K, V = k[: i + 1], v[: i + 1]
        s = K @ q[i] / h
        p = np.exp(s - s.max())
        p /= p.sum()
        cov = ((V - p @ V) * p[:, None]).T @ (K - p @ K)  # e x d
        if not np.allclose(dr[i], -cov.T @ do[i], rtol=1e-10, atol=1e-12):
            return False
    return True


def pin_shift_invariants(row_fn, seed=40, h=1.1):
    q, k, v, r, do = inputs(seed, T=8)
    _, dk, dv, _ = backward_with(row_fn, q, k, v, r, do, h)
    return (np.allclose(dk.sum(axis=0), 0.0, atol=1e-11)
            and np.allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-11, atol=1e-11))


PINS = (pin_finite_differences, pin_zero_probe_is_sdpa_backward,
        pin_probe_gradient_is_covariance, pin_shift_invariants)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_oracle_pin(pin):
    assert pin(parallax_backward_row)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_backward_oracle_finite_differences_more_seeds(seed):
    assert pin_finite_differences(parallax_backward_row, seed=100 * seed, h=0.7 + seed)


# ----------------------------------------------------------------------------- planted mistakes
def _mutant(mistake):
    def row(q_i, K, V, r_i, do_i, h):
        s = K @ q_i / h
        w = np.exp(s - s.max())
        p = w / w.sum()
        t = K @ r_i
        tbar = p @ t
        a = p * (1.0 + tbar - t) if mistake != "a_without_tbar" else p * (1.0 - t)
        o = a @ V
        g = V @ do_i
        G = p @ g
        dt = p * (G - g) if mistake != "dt_sign" else p * (g - G)
        u = (1.0 + tbar - t) * g + (G * t if mistake != "u_without_Gt" else 0.0)
        D = do_i @ o + (G * tbar if mistake != "D_without_Gtbar" else 0.0)
        ds = p * (u - D)
        dq = K.T @ ds / (h if mistake != "dq_without_h" else 1.0)
        dr = K.T @ dt
        dK = np.outer(ds, q_i) / h + (np.outer(dt, r_i) if mistake != "dk_without_probe" else 0.0)
        dV = np.outer(a, do_i)
        return dq, dr, dK, dV
    return row


@pytest.mark.parametrize("mistake", ["a_without_tbar", "dt_sign", "u_without_Gt",
                                     "D_without_Gtbar", "dq_without_h", "dk_without_probe"])
def test_pins_catch_planted_mistakes(mistake):
    row = _mutant(mistake)
    assert not all(pin(row) for pin in PINS)


# ----------------------------------------------------------------------------- the whole-tensor function
# The GPU tests compare against parallax_backward_oracle itself ([B, H, T, .] tensors, the causal
# accumulation of dk and dv over every row, the return order (dq, dk, dv, dr)). These pins apply
# to that function directly, on inputs with several heads of unequal content (B = 2, H = 3), so
# that a head mix-up, a wrong causal slice or a swapped return value fails at least one of them.

def whole_inputs(seed, B=2, H=3, T=6, d=4, e=3, rscale=0.5):
    q, k = rnd(seed, B, H, T, d), rnd(seed + 1, B, H, T, d)
    v, do = rnd(seed + 2, B, H, T, e), rnd(seed + 3, B, H, T, e)
    r = rnd(seed + 4, B, H, T, d, scale=rscale)
    # heads of different scale, so that gradients of one head cannot stand in for another's
    scale = (1.0 + np.arange(B * H)).reshape(B, H, 1, 1) / 3.0
    return q * scale, k, v * scale, r, do


def whole_pin_finite_differences(fn, seed=60, h=1.4):
    q, k, v, r, do = whole_inputs(seed)
    grads = fn(q, k, v, r, do, h)
    if len(grads) != 4:
        return False
    dq, dk, dv, dr = grads
    eps = 1e-5
    for which, g in enumerate((dq, dk, dv, dr)):  # d/dq, d/dk, d/dv, d/dr
        x = (q, k, v, r)[which]
        if g.shape != x.shape:
            return False
        delta = rnd(seed + 20 + which, *x.shape)
        plus = [y.copy() for y in (q, k, v, r)]
        minus = [y.copy() for y in (q, k, v, r)]
        plus[which] += eps * delta
        minus[which] -= eps * delta
        fd = (np.sum(parallax_forward_oracle(*plus, h) * do)
              - np.sum(parallax_forward_oracle(*minus, h) * do)) / (2 * eps)
        if not abs(fd - np.sum(g * delta)) <= 1e-7 * max(1.0, abs(fd)):
            return False
    return True


def whole_pin_zero_probe_is_sdpa_backward(fn, seed=70, h=0.9):
    q, k, v, _, do = whole_inputs(seed)
    dq, dk, dv, _ = fn(q, k, v, np.zeros_like(q), do, h)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=1.0 / h)
    (o * torch.tensor(do)).sum().backward()
    return all(np.allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12)
               for a, b in ((dq, tq), (dk, tk), (dv, tv)))


def whole_pin_probe_gradient_is_covariance(fn, seed=80, h=1.9):
    q, k, v, r, do = whole_inputs(seed)
    dr = fn(q, k, v, r, do, h)[3]
    B, H, T, _ = q.shape
    for b in range(B):
        for hh in range(H):
            for i in range(T):
                K, V = k[b, hh, : i + 1], v[b, hh, : i + 1]
                s = K @ q[b, hh, i] / h
                p = np.exp(s - s.max())
                p /= p.sum()
                cov = ((V - p @ V) * p[:, None]).T @ (K - p @ K)
                if not np.allclose(dr[b, hh, i], -cov.T @ do[b, hh, i], rtol=1e-10, atol=1e-12):
                    return False
    return True


def whole_pin_unbatched_matches_batched(fn, seed=90, h=1.2):
    """A [T, .] call (no leading dimensions) equals the matching head of a batched call."""
    q, k, v, r, do = whole_inputs(seed)
    full = fn(q, k, v, r, do, h)
    one = fn(q[1, 2], k[1, 2], v[1, 2], r[1, 2], do[1, 2], h)
    return all(a.shape == b[1, 2].shape and np.allclose(a, b[1, 2], rtol=1e-12, atol=1e-14)
               for a, b in zip(one, full))


WHOLE_PINS = (whole_pin_finite_differences, whole_pin_zero_probe_is_sdpa_backward,
              whole_pin_probe_gradient_is_covariance, whole_pin_unbatched_matches_batched)


@pytest.mark.parametrize("pin", WHOLE_PINS, ids=lambda f: f.__name__)
def test_backward_oracle_whole_tensor_pin(pin):
    assert pin(parallax_backward_oracle)


def _whole_mutant(mistake):
    """parallax_backward_oracle with one planted mistake of the whole-tensor bookkeeping."""
    def fn(q, k, v, r, do, h):
        q, k, v, r, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, r, do))
        squeeze = q.ndim == 2
        if squeeze:
            q, k, v, r, do = q[None], k[None], v[None], r[None], do[None]
        lead, (T, d), e = q.shape[:-2], q.shape[-2:], v.shape[-1]
        Q, K, R = q.reshape(-1, T, d), k.reshape(-1, T, d), r.reshape(-1, T, d)
        V, DO = v.reshape(-1, T, e), do.reshape(-1, T, e)
        dq, dk, dr, dv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(R), np.zeros_like(V)
        nbh = Q.shape[0]
        for bh in range(nbh):
            src = (bh + 1) % nbh if mistake == "value_of_next_head" else bh
            for i in range(T):
                gq, gr, gK, gV = parallax_backward_row(Q[bh, i], K[bh, : i + 1], V[src, : i + 1],
                                                       R[bh, i], DO[bh, i], h)
                dq[bh, i], dr[bh, i] = gq, gr
                if mistake == "slice_drops_diagonal":
                    dk[bh, :i] += gK[:i]
                    dv[bh, :i] += gV[:i]
                else:
                    dk[bh, : i + 1] += gK
                    dv[bh, : i + 1] += gV
        outs = []
        for x, last in ((dq, d), (dk, d), (dv, e), (dr, d)):
            if mistake == "heads_transposed" and len(lead) == 2:
                x = x.reshape(lead[1], lead[0], T, last).swapaxes(0, 1)
            else:
                x = x.reshape(*lead, T, last)
            outs.append(x[0] if squeeze else x)
        if mistake == "swap_dk_dr":
            outs[1], outs[3] = outs[3], outs[1]
        return tuple(outs)
    return fn


@pytest.mark.parametrize("mistake", ["swap_dk_dr", "slice_drops_diagonal", "heads_transposed",
                                     "value_of_next_head"])
def test_whole_tensor_pins_catch_planted_mistakes(mistake):
    fn = _whole_mutant(mistake)
    assert not all(pin(fn) for pin in WHOLE_PINS)


def test_whole_tensor_mutant_without_mistake_passes():
    """The mutant scaffold itself is faithful: with no planted mistake every pin holds."""
    fn = _whole_mutant("none")
    assert all(pin(fn) for pin in WHOLE_PINS)
