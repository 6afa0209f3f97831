"""Test helpers: run the float64 oracle on an ``SSDInputs`` (whole problem or
one sampled group) and compare device results against it."""
import numpy as np

from oracle import ssd_ref

FWD = ["x", "dt", "dt_bias", "A", "B", "C", "D"]
TOL = {"bf16": 2e-2, "f32": 1e-4}   # max|diff| <= TOL * max|ref|, per tensor


def oracle_full(inp, want_dinit=None):
    f = inp.f64
    args = [f(n) for n in FWD]
    kw = dict(initial_states=f("initial_states"), seq_idx=f("seq_idx"))
    y, fin = ssd_ref.ssd_fwd(*args, **kw)
    out = dict(y=y, final_states=fin)
    if want_dinit is None:
        want_dinit = inp.initial_states is not None
    g = ssd_ref.ssd_bwd(*args, f("dy"), dfinal_states=f("dfinal_states"), want_dinit=want_dinit,
                        **kw)
    out.update(g)
    return out


def oracle_group(inp, g):
    """Oracle outputs restricted to group g (every batch row, the group's
    heads, every token); dB and dC of the group sum the per-head results in
    head order."""
    f = inp.f64
    x, dt, bias, A, B, C, D = [f(n) for n in FWD]
    init = f("initial_states")
    return ssd_ref.ssd_group(x, dt, bias, A, B, C, D, f("dy"), g, inp.ngroups,
                             initial_states=init, seq_idx=f("seq_idx"),
                             dfinal_states=f("dfinal_states"), want_dinit=init is not None)


def slice_group(got, inp, g):
    H, G = inp.nheads, inp.ngroups
    hpg = H // G
    hs = slice(g * hpg, (g + 1) * hpg)
    out = {}
    for k, v in got.items():
        v = v.numpy() if hasattr(v, "numpy") else v
        if k in ("y", "dx", "ddt"):
            out[k] = v[:, :, hs]
        elif k in ("final_states", "dinitial_states"):
            out[k] = v[:, hs]
        elif k in ("dA", "dD", "ddt_bias"):
            out[k] = v[hs]
        elif k in ("dB", "dC"):
            out[k] = v[:, :, g:g + 1]
    return out


def rel_errors(got, ref):
    errs = {}
    for k, r in ref.items():
        gk = got[k]
        gk = gk.numpy() if hasattr(gk, "numpy") else np.asarray(gk)
        assert gk.shape == r.shape, (k, gk.shape, r.shape)
        assert np.all(np.isfinite(gk)), k
        errs[k] = float(np.abs(gk - r).max() / max(np.abs(r).max(), 1e-30))
    return errs


def assert_close(got, ref, dtype):
    errs = rel_errors(got, ref)
    bad = {k: e for k, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"tolerance {TOL[dtype]}: {bad} (all: {errs})"
    return errs
