"""Float64 oracle of the Mamba-2 block's gated RMSNorm, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906), sections
"_layer_norm_bwd speed-up" and the B200 results: after the SSD scan the
Mamba-2 block normalises the layer output, and the backward of that
normalisation (`_layer_norm_bwd`) is a memory-bound row reduction whose
concurrency (rows handled per program) decides its speed.  The page names
the kernel but does not write out the operation.  Reading (the plainest one
the rest supports): the Mamba-2 block's gated RMSNorm, with the gate applied
before the norm and the mean of squares taken over groups of columns,

    g[r, j]   = y[r, j] * silu(z[r, j])          silu(u) = u * sigmoid(u)
                (g = y when there is no gate)
    rstd[r,k] = 1 / sqrt(mean_{j in group k} g[r, j]^2 + eps)
    out[r, j] = g[r, j] * rstd[r, k(j)] * w[j]

for rows r (tokens) and groups k of ``group_size`` contiguous columns.  The
reverse mode for an upstream gradient dout, derived by hand (n = g * rstd is
the normalised value, dn = dout * w):

    dw[j]    = sum_r dout[r, j] * n[r, j]
    dg[r, j] = rstd[r, k] * (dn[r, j] - n[r, j] * mean_{i in group k} dn[r, i] n[r, i])
    dy[r, j] = dg[r, j] * silu(z[r, j])                       (dg without a gate)
    dz[r, j] = dg[r, j] * y[r, j] * sigmoid(z) * (1 + z * (1 - sigmoid(z)))

The sum over rows in dw is the cross-row reduction that page "Cake RMSNorm"
(blog.secrett2633.cloud, flashinfer PR 6997), section "Fixed-order tree
fold reduction", folds across thread blocks in a fixed order; here it is a
plain float64 sum.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def _sigmoid(u):
    # both branches of the logistic function, each evaluated where it does not overflow
    e = np.exp(-np.abs(u))
    return np.where(u >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _grouped(a, group_size):
    rows, dim = a.shape
    if dim % group_size:
        raise ValueError("dim must be a multiple of group_size")
    return a.reshape(rows, dim // group_size, group_size)


def gated_rmsnorm_fwd(y, z: Optional[np.ndarray], w, group_size: int, eps: float):
    """Forward of the gated RMSNorm on (rows, dim) arrays; returns (out, rstd)
    with rstd of shape (rows, dim // group_size)."""
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if z is None:
        g = y
    else:
        z = np.asarray(z, dtype=np.float64)
        g = y * (z * _sigmoid(z))
    gg = _grouped(g, group_size)
    rstd = 1.0 / np.sqrt((gg * gg).mean(axis=2) + eps)
    out = (gg * rstd[:, :, None]).reshape(g.shape) * w[None, :]
    return out, rstd


def gated_rmsnorm_bwd(y, z: Optional[np.ndarray], w, dout, group_size: int, eps: float):
    """Reverse mode of ``gated_rmsnorm_fwd`` for the upstream gradient dout;
    returns (dy, dz, dw) (dz is None without a gate)."""
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    if z is None:
        g = y
    else:
        z = np.asarray(z, dtype=np.float64)
        sz = _sigmoid(z)
        silu = z * sz
        g = y * silu
    gg = _grouped(g, group_size)
    rstd = 1.0 / np.sqrt((gg * gg).mean(axis=2) + eps)
    n = gg * rstd[:, :, None]
    dn = _grouped(dout * w[None, :], group_size)
    dw = (dout * n.reshape(g.shape)).sum(axis=0)
    c = (dn * n).mean(axis=2)
    dg = (rstd[:, :, None] * (dn - n * c[:, :, None])).reshape(g.shape)
    if z is None:
        return dg, None, dw
    dy = dg * silu
    dz = dg * y * sz * (1.0 + z * (1.0 - sz))
    return dy, dz, dw
