"""What storing the carry-in states and dS in bf16 costs, in isolation.

The tensor-core path keeps the chunk carries and their gradient in fp32 in
registers but hands them to the tensor core as bf16 tiles (H_in for the
chunk output's carry term and the dB/dC products, dS for dx and dB).  In
float64, on bf16-valued inputs of a workload-shaped problem, this computes
the change of y, dx, dB and dC that rounding H_in and dS to bf16 alone makes
(every other quantity exact) and checks that it stays well inside the
layer's bf16 tolerance of 2e-2 max|ref|: under a fifth of it."""
import numpy as np
import pytest
import torch

from mamba_selective_state_gb300.inputs import make_inputs
from oracle import chunked

BOUND = 2e-2 / 5


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("init", [False, True])
def test_bf16_carry_rounding_costs_under_a_fifth_of_the_tolerance(init):
    inp = make_inputs(batch=1, seqlen=1024, nheads=2, headdim=64, dstate=128, ngroups=1, chunk=128,
                      dtype="bf16", init=init, seed=13)
    f = inp.f64
    x, dt, bias, A, B, C, D, dy = (f(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D", "dy"])
    y, _, inter = chunked.ssd_chunked_fwd(x, dt, bias, A, B, C, D, 128, f("initial_states"))
    g = chunked.ssd_chunked_bwd(x, dt, bias, A, B, C, D, dy, 128, f("initial_states"))
    b, L, H, P = x.shape
    Q, nc = 128, L // 128
    dy_max = dx_max = dB_max = dC_max = 0.0
    for h in range(H):
        for c in range(nc):
            t = slice(c * Q, (c + 1) * Q)
            l = inter["l"][0, h, t]
            el = np.exp(l)                       # one sequence: every token sees the carry
            w = np.exp(l[-1] - l)
            u = w * inter["dt_eff"][0, h, t]
            Hc = inter["H_in"][0, h, c]
            dHc = _bf16(Hc) - Hc
            dSc = g["dS"][0, h, c]
            ddS = _bf16(dSc) - dSc
            Cm, Bm, X, dY = C[0, t, 0], B[0, t, 0], x[0, t, h], dy[0, t, h]
            dy_max = max(dy_max, np.abs(el[:, None] * (Cm @ dHc.T)).max())      # y carry term
            dx_max = max(dx_max, np.abs(u[:, None] * (Bm @ ddS.T)).max())      # dx state term
            dB_max = max(dB_max, np.abs(u[:, None] * (X @ ddS)).max())         # dB state term
            dC_max = max(dC_max, np.abs(el[:, None] * (dY @ dHc)).max())       # dC carry term
    rel = dict(y=dy_max / np.abs(y).max(), dx=dx_max / np.abs(g["dx"]).max(),
               dB=dB_max / np.abs(g["dB"]).max(), dC=dC_max / np.abs(g["dC"]).max())
    print("bf16 carry/dS rounding, max|change| / max|ref|:", rel)
    assert all(v <= BOUND for v in rel.values()), rel
