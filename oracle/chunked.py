"""Chunked float64 evaluation of the Mamba-2 SSD layer (numpy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

This is the same layer as ``ssd_ref`` (the token-by-token recurrence), taken
by chunks of Q tokens the way the chunked scan splits it (page "llm-mamba-200"
(gigipick.blogspot.com), section 3, "shared memory caching": split the
sequence into chunks and hand each chunk's final (carry-out) state to the next
chunk as its carry-in state; page "B200 Helion Mamba-2"
(aitrends.kr/articles/109906), section "Helion based B200 kernel redesign":
the cross-chunk state passing, forward and backward, is an associative scan).
It is written independently of the C oracle so that their agreement pins the
chunk decomposition; it also returns the intermediates (chunk-local decay
cumsum, chunk states, carry-in states, their gradients).

Per row b, head h (group g), chunk c holding tokens t0..t1-1 (local i, j):

  de_t   = softplus(dt_t + dt_bias_h),  l_i = sum_{k<=i} de_k A_h  (chunk-local)
  seg_t  = seq_idx[b, t] (0 when absent); s_in = seg of token t0-1 (seg_0 at t0=0)
  S_c    = sum_{j: seg_j = seg_last} exp(l_last - l_j) de_j  x_j (outer) B_j
  a_c    = exp(l_last) if every token of c has segment s_in, else 0
  H[0]   = initial_states (or 0);  H[c+1] = a_c H[c] + S_c;  final = H[nc]
  y_i    = sum_{j<=i, seg_j = seg_i} (C_i . B_j) exp(l_i - l_j) de_j x_j
           + [seg_i = s_in] exp(l_i) H[c] C_i + D_h x_i
"""
from __future__ import annotations

import math

import numpy as np


def softplus(z):
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def _decay(l, s):
    """E_ij = exp(l_i - l_j) for j <= i in the same segment, else 0; the
    exponent is only formed where the entry is kept."""
    n = len(l)
    keep = np.tril(np.ones((n, n), dtype=bool)) & (s[:, None] == s[None, :])
    diff = np.where(keep, l[:, None] - l[None, :], -np.inf)
    return np.exp(diff), keep


def _chunk_fwd_quantities(de, A_h, s, s_in):
    l = np.cumsum(de * A_h)
    E, keep = _decay(l, s)
    sv = (s == s[-1])
    w = np.where(sv, np.exp(np.where(sv, l[-1] - l, 0.0)), 0.0)   # exp(l_last - l_j) on kept j
    cv = (s == s_in)
    a_c = math.exp(l[-1]) if np.all(s == s_in) else 0.0
    return l, E, w, cv, a_c


def ssd_chunked_fwd(x, dt, dt_bias, A, B, C, D, chunk, initial_states=None,
                    seq_idx=None):
    """Returns (y, final_states, inter) with inter holding dt_eff (b,H,L),
    l (b,H,L) (chunk-local cumsums), a_chunk (b,H,nc), S (b,H,nc,P,N) and
    H_in (b,H,nc+1,P,N)."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = int(chunk)
    nc = -(-L // Q)
    seg = np.zeros((b, L), dtype=np.int64) if seq_idx is None else np.asarray(seq_idx, np.int64)
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    inter = dict(dt_eff=np.zeros((b, H, L)), l=np.zeros((b, H, L)),
                 a_chunk=np.zeros((b, H, nc)), S=np.zeros((b, H, nc, P, N)),
                 H_in=np.zeros((b, H, nc + 1, P, N)))
    for bi in range(b):
        for h in range(H):
            g = h * G // H
            de_all = softplus(dt[bi, :, h] + dt_bias[h])
            inter["dt_eff"][bi, h] = de_all
            Hc = np.zeros((P, N)) if initial_states is None else np.array(initial_states[bi, h], np.float64)
            inter["H_in"][bi, h, 0] = Hc
            for c in range(nc):
                t0, t1 = c * Q, min(L, (c + 1) * Q)
                s = seg[bi, t0:t1]
                s_in = seg[bi, t0 - 1] if t0 > 0 else seg[bi, 0]
                de = de_all[t0:t1]
                l, E, w, cv, a_c = _chunk_fwd_quantities(de, A[h], s, s_in)
                inter["l"][bi, h, t0:t1] = l
                X = x[bi, t0:t1, h, :]
                Bm = B[bi, t0:t1, g, :]
                Cm = C[bi, t0:t1, g, :]
                M = (Cm @ Bm.T) * E * de[None, :]
                y_carry = (cv * np.exp(l))[:, None] * (Cm @ Hc.T)
                y[bi, t0:t1, h, :] = M @ X + y_carry + D[h] * X
                S_c = (X * (w * de)[:, None]).T @ Bm
                inter["S"][bi, h, c] = S_c
                inter["a_chunk"][bi, h, c] = a_c
                Hc = a_c * Hc + S_c
                inter["H_in"][bi, h, c + 1] = Hc
            fin[bi, h] = Hc
    return y, fin, inter


def ssd_chunked_bwd(x, dt, dt_bias, A, B, C, D, dy, chunk, initial_states=None,
                    seq_idx=None, dfinal_states=None):
    """Reverse mode of ``ssd_chunked_fwd``.  Returns a dict with dx, ddt,
    ddt_bias, dA, dB, dC, dD, dinitial_states and the intermediates dS
    (b,H,nc,P,N) = dL/dS_c and da_chunk (b,H,nc) = dL/da_c."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = int(chunk)
    nc = -(-L // Q)
    seg = np.zeros((b, L), dtype=np.int64) if seq_idx is None else np.asarray(seq_idx, np.int64)
    _, _, inter = ssd_chunked_fwd(x, dt, dt_bias, A, B, C, D, Q, initial_states, seq_idx)
    out = dict(dx=np.zeros((b, L, H, P)), ddt=np.zeros((b, L, H)), ddt_bias=np.zeros(H),
               dA=np.zeros(H), dB=np.zeros((b, L, G, N)), dC=np.zeros((b, L, G, N)),
               dD=np.zeros(H), dinitial_states=np.zeros((b, H, P, N)),
               dS=np.zeros((b, H, nc, P, N)), da_chunk=np.zeros((b, H, nc)))
    for bi in range(b):
        for h in range(H):
            g = h * G // H
            de_all = inter["dt_eff"][bi, h]
            z_all = dt[bi, :, h] + dt_bias[h]
            # state passing backward: Gtot[c] = dL/dH[c]
            Gt = np.zeros((P, N)) if dfinal_states is None else np.array(dfinal_states[bi, h], np.float64)
            for c in range(nc - 1, -1, -1):
                t0, t1 = c * Q, min(L, (c + 1) * Q)
                s = seg[bi, t0:t1]
                s_in = seg[bi, t0 - 1] if t0 > 0 else seg[bi, 0]
                de = de_all[t0:t1]
                l, E, w, cv, a_c = _chunk_fwd_quantities(de, A[h], s, s_in)
                X = x[bi, t0:t1, h, :]
                dY = dy[bi, t0:t1, h, :]
                Bm = B[bi, t0:t1, g, :]
                Cm = C[bi, t0:t1, g, :]
                Hc = inter["H_in"][bi, h, c]
                dS = Gt                                   # dL/dS_c = dL/dH[c+1]
                out["dS"][bi, h, c] = dS
                da = float(np.sum(dS * Hc))               # dL/da_c
                out["da_chunk"][bi, h, c] = da
                el = np.exp(l)
                dHloc = (dY * (cv * el)[:, None]).T @ Cm  # from the carry term of y
                Gt = dHloc + a_c * Gt                     # dL/dH[c]
                n = t1 - t0
                dX = np.zeros((n, P))
                dBm = np.zeros((n, N))
                dCm = np.zeros((n, N))
                dde = np.zeros(n)                         # direct d/d dt_eff
                dl = np.zeros(n)                          # d/d l_i
                # chunk state S_c = sum_j u_j x_j (outer) B_j, u_j = w_j de_j
                u = w * de
                XdS = X @ dS                              # (n, N): x_j^T dS
                dX += u[:, None] * (Bm @ dS.T)
                dBm += u[:, None] * XdS
                du = np.sum(XdS * Bm, axis=1)
                dde += w * du
                dl[-1] += np.sum(u * du)
                dl -= u * du
                # intra-chunk output  y_i += sum_j M_ij x_j, M = CB * E * de_j
                CB = Cm @ Bm.T
                M = CB * E * de[None, :]
                dX += M.T @ dY
                dM = dY @ X.T
                dCB = dM * E * de[None, :]
                dCm += dCB @ Bm
                dBm += dCB.T @ Cm
                dde += np.sum(dM * CB * E, axis=0)
                R = dM * M
                dl += R.sum(axis=1)
                dl -= R.sum(axis=0)
                # carry term  y_i += cv_i exp(l_i) H C_i
                y_carry = (cv * el)[:, None] * (Cm @ Hc.T)
                dCm += (cv * el)[:, None] * (dY @ Hc)
                dl += np.sum(dY * y_carry, axis=1)
                # skip term
                dX += D[h] * dY
                out["dD"][h] += float(np.sum(dY * X))
                # chunk decay a_c = exp(l_last) (only when no reset inside c)
                if a_c != 0.0:
                    dl[-1] += a_c * da
                # l_i = cumsum(de A): d(dA_k) = sum_{i>=k} dl_i
                d_dA = np.cumsum(dl[::-1])[::-1]
                dde_tot = dde + A[h] * d_dA
                out["dA"][h] += float(np.sum(de * d_dA))
                ddt_c = dde_tot * sigmoid(z_all[t0:t1])
                out["ddt"][bi, t0:t1, h] = ddt_c
                out["ddt_bias"][h] += float(np.sum(ddt_c))
                out["dx"][bi, t0:t1, h, :] = dX
                out["dB"][bi, t0:t1, g, :] += dBm
                out["dC"][bi, t0:t1, g, :] += dCm
            out["dinitial_states"][bi, h] = Gt
    return out
