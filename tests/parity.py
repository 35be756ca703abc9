"""Error metrics of the GPU parity tests and the record of achieved errors.

Two metrics compare a GPU result with the float64 oracle over the checked rows:

* ``rel_err``: the relative Frobenius error ||O - O_ref||_F / ||O_ref||_F (the gated bound:
  1e-3 for fp32 inputs, 2e-2 for bf16 inputs);
* ``row_max_err``: the worst single row, max_i ||o_i - o_ref,i||_2 / (||o_ref,i||_2 + rms(V)), so
  that a few badly wrong rows cannot hide inside a large Frobenius norm. rms(V) keeps rows whose
  reference output is near zero from dividing by almost nothing.

Every check appends its numbers to ``RECORDS``; ``conftest.py`` prints them at the end of the run.
"""
from __future__ import annotations

import os

import numpy as np

RECORDS: list[dict] = []

# The worst row may exceed the Frobenius bound (a single row has few elements, and bf16 output
# rounding alone is ~2e-3 per element); it is gated at this multiple of that bound.
ROW_FACTOR = 5.0


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def row_max_err(got, ref, v_rms: float) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    e = got.shape[-1]
    g, r = got.reshape(-1, e), ref.reshape(-1, e)
    if g.shape[0] == 0:
        return 0.0
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1) + v_rms
    return float((num / den).max())


def current_case() -> str:
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::", 1)[-1]


def record(got, ref, v, tol: float, case: str | None = None, row_tol: float | None = None):
    """Computes both metrics, records them and asserts both bounds. Returns (rel, row_max)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    v_rms = float(np.sqrt(np.mean(np.asarray(v, dtype=np.float64) ** 2))) if np.size(v) else 1.0
    rel = rel_err(got, ref)
    rmax = row_max_err(got, ref, v_rms)
    row_tol = ROW_FACTOR * tol if row_tol is None else row_tol
    e = got.shape[-1] if got.ndim else 1
    RECORDS.append({"case": case or current_case(), "rows": int(got.size // max(e, 1)),
                    "rel": rel, "tol": tol, "row_max": rmax, "row_tol": row_tol})
    assert np.isfinite(got).all(), "non-finite output"
    assert rel <= tol, f"relative Frobenius error {rel:.3e} > {tol:.1e}"
    assert rmax <= row_tol, f"worst-row error {rmax:.3e} > {row_tol:.1e}"
    return rel, rmax
