"""Lays logical matrices out in BLAS-style storage for tests.

Input plumbing only: given the logical operand (already op()-applied) it
produces the flat buffer a caller would pass, with op N/T, row/column order,
a padded leading dimension and a batch stride.  No GEMM arithmetic here.
"""
import numpy as np


def stored_shape(op, rows, cols):
    """Shape of the stored matrix for a logical rows x cols operand."""
    return (rows, cols) if op == "N" else (cols, rows)


def tight_ld(order, srows, scols):
    return max(1, scols if order == "row" else srows)


def to_storage(logical, op="N", order="row", ld=None, batch_stride=None):
    """logical: array (L, rows, cols) -> (flat buffer, ld, batch stride).

    The stored matrix is logical[l] (op N) or its transpose (op T); row-major
    puts stored row r at r*ld, column-major puts stored column s at s*ld.
    """
    logical = np.asarray(logical)
    if logical.ndim == 2:
        logical = logical[None]
    L, rows, cols = logical.shape
    sr, sc = stored_shape(op, rows, cols)
    if ld is None:
        ld = tight_ld(order, sr, sc)
    outer = sr if order == "row" else sc
    inner_extent = sc if order == "row" else sr
    assert ld >= inner_extent
    per = outer * ld
    if batch_stride is None:
        batch_stride = per
    assert batch_stride >= per or L == 1
    total = (L - 1) * batch_stride + per
    buf = np.zeros(total, dtype=logical.dtype)
    for l in range(L):
        stored = logical[l] if op == "N" else logical[l].T
        block = np.zeros((outer, ld), dtype=logical.dtype)
        if order == "row":
            block[:, :sc] = stored
        else:
            block[:, :sr] = stored.T
        buf[l * batch_stride: l * batch_stride + per] = block.reshape(-1)
    return buf, ld, batch_stride


def from_storage(buf, L, rows, cols, order="row", ld=None, batch_stride=None):
    """Inverse of to_storage for an op-N operand (used for C and D)."""
    if ld is None:
        ld = tight_ld(order, rows, cols)
    outer = rows if order == "row" else cols
    per = outer * ld
    if batch_stride is None:
        batch_stride = per
    out = np.zeros((L, rows, cols), dtype=buf.dtype)
    for l in range(L):
        block = buf[l * batch_stride: l * batch_stride + per].reshape(outer, ld)
        out[l] = block[:, :cols] if order == "row" else block[:, :rows].T
    return out
