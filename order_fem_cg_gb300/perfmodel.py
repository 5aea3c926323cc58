"""Streaming performance model and the byte counts of each BS operation.

"Portable high-order finite element kernels I: Streaming Operations",
performance model: streaming B bytes takes T(B) = T0 + B / Wmax (eq. (8)),
so the effective bandwidth is W_eff(B) = B / (T0 + B / Wmax) (eq. (9)), and
80% of Wmax is reached at the Fischer-Brown point B_0.8 = 4 T0 Wmax
(eq. (10)).  The fit method is not given on the pages; ordinary least
squares of T on B over a size sweep is used here.

Byte counts: the minimal unique HBM traffic of each operation (8-byte
values, 4-byte indices), the figure of merit the pages measure in GB/s.
"""

from __future__ import annotations

import numpy as np


def t_model(B, T0, Wmax):
    """Eq. (8): time to stream B bytes."""
    return T0 + np.asarray(B, dtype=np.float64) / Wmax


def w_eff(B, T0, Wmax):
    """Eq. (9): effective bandwidth when streaming B bytes."""
    B = np.asarray(B, dtype=np.float64)
    return B / (T0 + B / Wmax)


def b_08(T0, Wmax):
    """Eq. (10): bytes needed to reach 80% of Wmax."""
    return 4.0 * T0 * Wmax


def fit(B, T):
    """Least-squares fit of T = T0 + B / Wmax; returns (T0, Wmax)."""
    B = np.asarray(B, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    A = np.stack([np.ones_like(B), B], axis=1)
    (T0, inv_w), *_ = np.linalg.lstsq(A, T, rcond=None)
    return float(T0), float(1.0 / inv_w)


# ----------------------------------------------------------- byte counts

def bytes_copy(n):
    return 16 * n            # read x, write y


def bytes_axpy(n):
    return 24 * n            # read x, y; write y


def bytes_norm(n):
    return 8 * n             # read x


def bytes_dot(n):
    return 16 * n            # read x, y


def bytes_cg_update(n):
    return 48 * n            # read p, Ap, x, r; write x, r


def bytes_gather(NL, NG, nnz, nblocks):
    # read q_L (each unmasked local once) and localIds; read rowStarts,
    # write q_G; read blockStarts
    return 8 * nnz + 4 * nnz + 4 * (NG + 1) + 8 * NG + 4 * (nblocks + 1)


def bytes_scatter(NL, NG_referenced):
    # read scatterIds, write q_L, read each referenced q_G value once
    # (all N_G of them unless the mesh masks some global nodes)
    return 4 * NL + 8 * NL + 8 * NG_referenced


def bytes_cg_iteration(NL, NG, nnz, nblocks):
    """scatter + gather + dot + fused update + norm on global-length vectors."""
    return (bytes_scatter(NL, NG) + bytes_gather(NL, NG, nnz, nblocks) + bytes_dot(NG)
            + bytes_cg_update(NG) + bytes_norm(NG))


# ------------------------------------------------ DRAM traffic of the design

def moved_bytes(op, NL, NG, nnz):
    """Bytes the library's kernels move for one call (not the figure of
    merit: the algorithmic bytes above are).  Streaming operations move
    their algorithmic bytes.  The two-pass gather and scatter route every
    local value through a work array in HBM: scatter reads q_G and its
    pass-1 offsets, writes the work array, reads it back with its pass-2
    offsets and writes q_L (8 N_G + 20 nnz + 8 N_L); gather reads q_L and
    its offsets, writes and reads the work array with its offsets, reads
    each row's staged position and writes q_G (8 NL + 20 nnz + 10 N_G).
    Run tables (under 5%) are left out.  Used to scale DRAM traffic measured
    on one mesh to another."""
    n = NL
    if op == "copy":
        return bytes_copy(n)
    if op == "axpy":
        return bytes_axpy(n)
    if op == "norm":
        return bytes_norm(n)
    if op == "dot":
        return bytes_dot(n)
    if op == "cg_update":
        return bytes_cg_update(n)
    if op == "scatter":
        return 8 * NG + 20 * nnz + 8 * NL
    if op == "gather":
        return 8 * NL + 20 * nnz + 10 * NG
    raise ValueError(op)
