import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C-ABI)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle time)")


def to_oracle(t):
    """torch tensor -> numpy array in a form the oracle decodes exactly
    (bfloat16 travels as its raw 16 bits)."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.float64):
        return t.numpy()
    raise TypeError(t.dtype)


def max_rel_err(got, ref):
    """Infinity-norm relative error of a whole tensor: max|got-ref| / max|ref|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / den)


def _blocks(a, rows_per_block=1 << 16):
    """Views of a 2-D array [rows, n] in blocks of rows (bounds the temporaries)."""
    for i in range(0, a.shape[0], rows_per_block):
        yield i, a[i:i + rows_per_block]


def row_rel_err(got, ref):
    """Largest relative error of a row: for every row along the last axis (a token
    of y, a feature row of S, the z vector of a head), max|got-ref| over the row
    divided by max|ref| over that row; the maximum over all rows.  A row whose
    reference is exactly zero contributes its largest |got|.

    Unlike max_rel_err this does not let the largest rows of a tensor set the bar
    for the small ones: y_t is a normalised average over t tokens and shrinks
    along the sequence, so a tensor-wide bar set by the first tokens would not
    see errors in the last ones."""
    ref = np.asarray(ref)
    got = np.asarray(got)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    n = ref.shape[-1] if ref.ndim else 1
    g2, r2 = got.reshape(-1, n), ref.reshape(-1, n)
    worst = 0.0
    for i, rb in _blocks(r2):
        gb = g2[i:i + rb.shape[0]].astype(np.float64)
        rb = rb.astype(np.float64)
        den = np.max(np.abs(rb), axis=1)
        num = np.max(np.abs(gb - rb), axis=1)
        err = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
        worst = max(worst, float(np.max(err)) if err.size else 0.0)
    return worst


def elem_diag(got, ref):
    """Elementwise diagnostic (reported, not asserted): max over elements of
    |got-ref| / max(|ref|, 1e-3 * rms(ref))."""
    ref = np.asarray(ref)
    got = np.asarray(got)
    r1, g1 = ref.reshape(-1), got.reshape(-1)
    if r1.size == 0:
        return 0.0
    rms = 0.0
    for i in range(0, r1.size, 1 << 24):
        rb = r1[i:i + (1 << 24)].astype(np.float64)
        rms += float(np.dot(rb, rb))
    rms = (rms / r1.size) ** 0.5
    floor = max(1e-3 * rms, np.finfo(np.float64).tiny)
    worst = 0.0
    for i in range(0, r1.size, 1 << 24):
        rb = r1[i:i + (1 << 24)].astype(np.float64)
        gb = g1[i:i + (1 << 24)].astype(np.float64)
        worst = max(worst, float(np.max(np.abs(gb - rb) / np.maximum(np.abs(rb), floor))))
    return worst


def assert_close(got, ref, tol, what=""):
    """The parity bar: finite, and both the tensor-wide and the per-row relative
    error within tol; prints the errors and the elementwise diagnostic."""
    got = np.asarray(got)
    assert np.isfinite(got).all(), f"{what}: not finite"
    t_err = max_rel_err(got, ref)
    r_err = row_rel_err(got, ref)
    print(f"[parity] {what}: tensor {t_err:.3e}  row {r_err:.3e}  elem-diag {elem_diag(got, ref):.3e}  (bar {tol})")
    assert t_err <= tol, f"{what}: max rel err {t_err:.3e} > {tol}"
    assert r_err <= tol, f"{what}: per-row rel err {r_err:.3e} > {tol}"
    return t_err, r_err


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
