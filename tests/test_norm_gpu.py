"""Gated RMSNorm of the Mamba-2 block: CUDA path vs the float64 oracle,
element by element, through the C ABI.

Small cases cover every team shape of the kernels (a team of 1, 3, 12 and 16
warps per group, idle lanes in a team, the largest groups of each dtype),
ragged row counts, one row, more rows than the backward's row slices, and the
ungated norm; they compare every element.  The norms that follow the five
layer workloads run at full size: out, rstd, dy and dz are compared on 64
sampled rows, dweight (a sum over every row) in full.  Tolerance:
max|diff| <= 2e-2 max|ref| (bf16) or 1e-4 max|ref| (fp32), per tensor; rstd
is fp32 in both and held to 1e-4."""
import numpy as np
import pytest
import torch

from mamba_selective_state_gb300.inputs import WORKLOADS, make_norm_inputs, make_norm_workload
from oracle import gated_norm
from tests.ref_helpers import TOL, rel_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def run_device(inp):
    from mamba_selective_state_gb300.runner import NormDevice
    dev = NormDevice(inp, device="cuda")
    dev.fwd()
    dev.bwd()
    torch.cuda.synchronize()
    return dev, dev.results()


def _f64(t, rows):
    if t is None:
        return None
    t = t if rows is None else t[torch.as_tensor(rows)]
    return t.to(torch.float64).numpy()


def oracle(inp, rows=None):
    """The oracle on every row, or on the rows listed in ``rows``."""
    y, z, dout = _f64(inp.y, rows), _f64(inp.z, rows), _f64(inp.dout, rows)
    w = inp.f64("weight")
    out, rstd = gated_norm.gated_rmsnorm_fwd(y, z, w, inp.group_size, inp.eps)
    dy, dz, dw = gated_norm.gated_rmsnorm_bwd(y, z, w, dout, inp.group_size, inp.eps)
    ref = dict(out=out, rstd=rstd, dy=dy, dweight=dw)
    if dz is not None:
        ref["dz"] = dz
    return ref


def check(got, ref, dtype):
    errs = rel_errors(got, ref)
    tol = dict.fromkeys(errs, TOL[dtype])
    tol["rstd"] = 1e-4
    bad = {k: e for k, e in errs.items() if not e <= tol[k]}
    assert not bad, f"{bad} (all: {errs})"


SMALL = {
    # rows, dim, group_size, dtype, gate
    "tiny_fp32": (256, 64, 64, "f32", True),                 # 16 pieces: half a warp idle
    "bf16_ragged_rows_G8": (333, 1024, 128, "bf16", True),
    "bf16_one_row": (1, 512, 512, "bf16", True),
    "bf16_ungated": (200, 768, 256, "bf16", False),
    "bf16_team_of_3": (130, 1536, 768, "bf16", True),        # 96 pieces: 3 warps, 2 teams per CTA
    "bf16_team_of_12": (50, 6144, 3072, "bf16", True),       # 384 pieces: 512-thread CTAs
    "bf16_largest_group": (20, 8192, 4096, "bf16", True),    # 512 pieces: 16 warps
    "fp32_largest_group": (40, 4096, 2048, "f32", True),
    "fp32_ungated_small_group": (70, 384, 96, "f32", False),
    "bf16_more_rows_than_slices": (5000, 256, 256, "bf16", True),  # 1024 slices of ~5 rows
    "fp32_one_piece_groups": (90, 64, 4, "f32", True),       # 16 groups of one piece
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    rows, dim, gs, dtype, gate = SMALL[name]
    inp = make_norm_inputs(rows, dim, gs, dtype=dtype, gate=gate, seed=7)
    _, got = run_device(inp)
    check(got, oracle(inp), dtype)


def test_backward_is_bitwise_deterministic():
    inp = make_norm_inputs(3000, 2048, 256, dtype="bf16", seed=3)
    dev, first = run_device(inp)
    dev.bwd()
    torch.cuda.synchronize()
    second = dev.results()
    for k in ("dy", "dz", "dweight"):
        assert torch.equal(first[k], second[k]), k


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload_sampled_rows(name):
    from mamba_selective_state_gb300.runner import NormDevice
    inp = make_norm_workload(name, seed=0)
    dev = NormDevice(inp, device="cuda")
    dev.fwd()
    dev.bwd()
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(inp.rows, size=64, replace=False))
    ref = oracle(inp, rows)
    del ref["dweight"]  # the sampled rows' share only; the full sum is checked below
    idx = torch.as_tensor(rows, device="cuda")
    sampled = {k: getattr(dev, k)[idx].to("cpu", torch.float64) for k in ref}
    check(sampled, ref, inp.dtype)
    # dweight sums over every row: the oracle's column sums, taken by row blocks
    w = inp.f64("weight")
    dw = np.zeros(inp.dim)
    step = max(1, (1 << 22) // inp.dim)
    for r0 in range(0, inp.rows, step):
        sl = slice(r0, min(inp.rows, r0 + step))
        z = None if inp.z is None else inp.z[sl].to(torch.float64).numpy()
        dw += gated_norm.gated_rmsnorm_bwd(inp.y[sl].to(torch.float64).numpy(), z, w,
                                           inp.dout[sl].to(torch.float64).numpy(),
                                           inp.group_size, inp.eps)[2]
    check({"dweight": dev.dweight.to("cpu", torch.float64)}, {"dweight": dw}, inp.dtype)
