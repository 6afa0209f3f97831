"""Pins of the float64 gated-RMSNorm oracle (``oracle/gated_norm.py``), CPU.

Each pin checks the oracle against something other than itself:
  * torch's own ``rms_norm`` and ``silu`` (library routines, float64) on the
    grouped view, and torch autograd through them for the backward;
  * central finite differences of the forward for every gradient;
  * closed forms (a constant group; a gate of zero);
  * invariants that hold with eps = 0 (scale invariance of each group, and the
    gradient orthogonal to the input that follows from it);
  * groups are independent: a grouped call equals one call per group.
A last test plants plausible mistakes in a copy of the oracle and checks that
at least one pin fails for each.
"""
import os
import types

import numpy as np
import pytest
import torch

from oracle import gated_norm

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "gated_norm.py")


def _case(rows=5, dim=12, gs=4, seed=0, gate=True):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((rows, dim))
    z = rng.standard_normal((rows, dim)) * 2.0 if gate else None
    w = rng.standard_normal(dim)
    dout = rng.standard_normal((rows, dim))
    return y, z, w, dout, gs


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def _library(y, z, w, dout, gs, eps):
    """The same operation composed from torch's rms_norm and silu, float64,
    with its gradients from torch autograd."""
    yt = torch.tensor(y, requires_grad=True)
    zt = None if z is None else torch.tensor(z, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    g = yt if zt is None else yt * torch.nn.functional.silu(zt)
    rows, dim = g.shape
    n = torch.nn.functional.rms_norm(g.reshape(rows, dim // gs, gs), (gs,), eps=eps)
    out = n.reshape(rows, dim) * wt
    out.backward(torch.tensor(dout))
    return (out.detach().numpy(), yt.grad.numpy(), None if zt is None else zt.grad.numpy(),
            wt.grad.numpy())


def pin_library(mod, gate=True, eps=1e-5, seed=0, gs=4):
    y, z, w, dout, gs = _case(gs=gs, seed=seed, gate=gate)
    out, _ = mod.gated_rmsnorm_fwd(y, z, w, gs, eps)
    dy, dz, dw = mod.gated_rmsnorm_bwd(y, z, w, dout, gs, eps)
    ref = _library(y, z, w, dout, gs, eps)
    ok = _rel(out, ref[0]) < 1e-12 and _rel(dy, ref[1]) < 1e-12 and _rel(dw, ref[3]) < 1e-12
    if gate:
        ok = ok and _rel(dz, ref[2]) < 1e-12
    return ok


def pin_finite_differences(mod, gate=True, eps=1e-3, seed=1):
    y, z, w, dout, gs = _case(rows=3, dim=6, gs=3, seed=seed, gate=gate)
    dy, dz, dw = mod.gated_rmsnorm_bwd(y, z, w, dout, gs, eps)

    def loss(yy, zz, ww):
        return float((mod.gated_rmsnorm_fwd(yy, zz, ww, gs, eps)[0] * dout).sum())

    h = 1e-6
    ok = True
    for name, arr, grad in (("y", y, dy), ("z", z, dz), ("w", w, dw)):
        if arr is None:
            continue
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {"y": y, "z": z, "w": w}
            p = arr.copy(); p[idx] += h
            m = arr.copy(); m[idx] -= h
            args_p = dict(args, **{name: p}); args_m = dict(args, **{name: m})
            fd[idx] = (loss(args_p["y"], args_p["z"], args_p["w"])
                       - loss(args_m["y"], args_m["z"], args_m["w"])) / (2 * h)
        ok = ok and _rel(grad, fd) < 1e-7
    return ok


def pin_constant_group(mod):
    # one row, no gate, every entry of a group equal to c: mean of squares is c^2
    c, eps, gs = -0.75, 1e-2, 8
    y = np.full((1, 2 * gs), c)
    y[0, gs:] = 2.0
    w = np.linspace(-1.0, 1.0, 2 * gs)
    out, rstd = mod.gated_rmsnorm_fwd(y, None, w, gs, eps)
    want = np.concatenate([np.full(gs, c / np.sqrt(c * c + eps)),
                           np.full(gs, 2.0 / np.sqrt(4.0 + eps))]) * w
    return (_rel(out[0], want) < 1e-14
            and abs(rstd[0, 0] - 1 / np.sqrt(c * c + eps)) < 1e-13)


def pin_zero_gate(mod):
    # z = 0: silu(0) = 0, so g = 0, out = 0, dy = 0, and since sigmoid(0) = 1/2,
    # dz = dout * w * y / (2 sqrt(eps))
    y, _, w, dout, gs = _case(rows=3, dim=8, gs=4, seed=2)
    z = np.zeros_like(y)
    eps = 1e-4
    out, _ = mod.gated_rmsnorm_fwd(y, z, w, gs, eps)
    dy, dz, dw = mod.gated_rmsnorm_bwd(y, z, w, dout, gs, eps)
    want_dz = dout * w[None, :] * y / (2.0 * np.sqrt(eps))
    return (np.abs(out).max() == 0 and np.abs(dy).max() == 0 and np.abs(dw).max() == 0
            and _rel(dz, want_dz) < 1e-13)


def pin_scale_invariance(mod):
    # eps = 0, no gate: out is unchanged when a group of a row is scaled by s > 0,
    # so the gradient of any loss is orthogonal to y within every group
    y, _, w, dout, gs = _case(rows=4, dim=12, gs=6, seed=3, gate=False)
    out, _ = mod.gated_rmsnorm_fwd(y, None, w, gs, 0.0)
    s = np.ones_like(y)
    s[1, :gs] = 3.5
    s[2, gs:] = 0.125
    out2, _ = mod.gated_rmsnorm_fwd(y * s, None, w, gs, 0.0)
    dy, _, _ = mod.gated_rmsnorm_bwd(y, None, w, dout, gs, 0.0)
    dots = (dy * y).reshape(4, 2, gs).sum(axis=2)
    return _rel(out2, out) < 1e-14 and np.abs(dots).max() < 1e-12


def pin_groups_independent(mod):
    y, z, w, dout, gs = _case(rows=3, dim=12, gs=4, seed=4)
    eps = 1e-5
    out, rstd = mod.gated_rmsnorm_fwd(y, z, w, gs, eps)
    dy, dz, dw = mod.gated_rmsnorm_bwd(y, z, w, dout, gs, eps)
    ok = True
    for k in range(3):
        sl = slice(k * gs, (k + 1) * gs)
        o1, r1 = mod.gated_rmsnorm_fwd(y[:, sl], z[:, sl], w[sl], gs, eps)
        d1 = mod.gated_rmsnorm_bwd(y[:, sl], z[:, sl], w[sl], dout[:, sl], gs, eps)
        ok = ok and np.array_equal(o1, out[:, sl]) and np.array_equal(r1[:, 0], rstd[:, k])
        ok = ok and np.array_equal(d1[0], dy[:, sl]) and np.array_equal(d1[1], dz[:, sl])
        ok = ok and _rel(d1[2], dw[sl]) < 1e-15
    return ok


PINS = {
    "library_gated": lambda m: pin_library(m, gate=True),
    "library_plain": lambda m: pin_library(m, gate=False),
    "library_one_group": lambda m: pin_library(m, gate=True, gs=12, seed=5),
    "finite_differences_gated": lambda m: pin_finite_differences(m, gate=True),
    "finite_differences_plain": lambda m: pin_finite_differences(m, gate=False),
    "constant_group": pin_constant_group,
    "zero_gate": pin_zero_gate,
    "scale_invariance": pin_scale_invariance,
    "groups_independent": pin_groups_independent,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    assert PINS[name](gated_norm), name


def test_sigmoid_is_stable_for_large_arguments():
    z = np.array([-800.0, -40.0, 0.0, 40.0, 800.0])
    s = gated_norm._sigmoid(z)
    assert np.all(np.isfinite(s))
    assert s[0] == 0.0 and s[-1] == 1.0 and s[2] == 0.5


def test_rejects_ragged_groups():
    with pytest.raises(ValueError):
        gated_norm.gated_rmsnorm_fwd(np.ones((2, 10)), None, np.ones(10), 4, 1e-5)


MUTANTS = {
    "gate_after_norm_missing": ("g = y * (z * _sigmoid(z))", "g = y * z"),
    "mean_over_row_not_group": ("rstd = 1.0 / np.sqrt((gg * gg).mean(axis=2) + eps)\n    out",
                                "rstd = 1.0 / np.sqrt((gg * gg).mean(axis=(1, 2))[:, None] + eps) + 0 * gg[:, :, 0]\n    out"),
    "eps_outside_sqrt": ("rstd = 1.0 / np.sqrt((gg * gg).mean(axis=2) + eps)\n    out",
                         "rstd = 1.0 / (np.sqrt((gg * gg).mean(axis=2)) + eps)\n    out"),
    "bwd_drop_projection": ("(dn - n * c[:, :, None])", "dn"),
    "bwd_projection_sign": ("(dn - n * c[:, :, None])", "(dn + n * c[:, :, None])"),
    "bwd_dw_unnormalised": ("dw = (dout * n.reshape(g.shape)).sum(axis=0)",
                            "dw = (dout * g).sum(axis=0)"),
    "bwd_dz_missing_product_rule": ("sz * (1.0 + z * (1.0 - sz))", "sz"),
    "bwd_dy_missing_gate": ("dy = dg * silu", "dy = dg"),
    "bwd_dn_missing_weight": ("dn = _grouped(dout * w[None, :], group_size)",
                              "dn = _grouped(dout, group_size)"),
    "bwd_sum_for_mean": ("c = (dn * n).mean(axis=2)", "c = (dn * n).sum(axis=2)"),
}


def _mutant(edit):
    src = open(SRC).read()
    old, new = edit
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    mod = types.ModuleType("gated_norm_mutant")
    exec(compile(src.replace(old, new), "gated_norm_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mod = _mutant(MUTANTS[name])
    failed = []
    for pin, fn in PINS.items():
        try:
            ok = fn(mod)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin)
    assert failed, f"no pin catches mutant {name}"
