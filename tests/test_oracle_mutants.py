"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/ssd_oracle.c`` to a temporary directory, plants one
mistake by a textual edit (a dropped term, a wrong sign, a wrong index or
operand), compiles the copy and runs a short battery of pins against it: the
closed forms, the independent chunked evaluation, packing, and finite
differences of the forward.  At least one pin must fail for every mutant,
and all of them must pass for the unmodified source.  CPU only.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

from mamba_selective_state_gb300.inputs import make_inputs
from oracle import chunked, ssd_ref

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "ssd_oracle.c")

MUTANTS = {
    "drop_skip_term": ("yt[p] = acc + D[h] * xt[p];", "yt[p] = acc;"),
    "decay_sign": ("double a = exp(de * A[h]);", "double a = exp(-de * A[h]);"),
    "softplus_no_log1p": ("log1p(exp(-fabs(z)))", "exp(-fabs(z))"),
    "output_reads_B": ("const double* Ct = C + ((bi * d.L + t) * d.G + g) * N;",
                       "const double* Ct = B + ((bi * d.L + t) * d.G + g) * N;"),
    "reset_ignored": ("return seq_idx[bi * d->L + t] != seq_idx[bi * d->L + t - 1];",
                      "return 0;"),
    "group_map_interleaved": ("return h * d->G / d->H;", "return h % d->G;"),
    "init_ignored_fwd": ("if (initial_states) memcpy(hs, initial_states", "if (0) memcpy(hs, initial_states"),
    "bwd_drop_decay_term": ("s_xb + A[h] * a * s_hp", "s_xb"),
    "bwd_dB_missing_dt": ("dBt[n] += de * accb;", "dBt[n] += accb;"),
    "bwd_dC_uses_prev_state": ("accc += ht[p * N + n] * dyt[p];", "accc += hprev[p * N + n] * dyt[p];"),
    "bwd_carry_through_reset": ("const double carry = reset ? 0.0 : a;", "const double carry = a;"),
    "bwd_no_sigmoid": ("ddt_eff * sigmoid(z)", "ddt_eff"),
    "bwd_dA_missing_decay": ("pdA[bi * H + h] += de * a * s_hp;", "pdA[bi * H + h] += de * s_hp;"),
    "bwd_dx_missing_skip": ("dxt[p] = D[h] * dyt[p] + de * acc;", "dxt[p] = de * acc;"),
    "bwd_dx_transposed_state": ("acc += gcur[p * N + n] * Bt[n];", "acc += gcur[n * N + p % N] * Bt[n];"),
}


def _build(tmp_path, name, edit):
    src = open(SRC).read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutation anchor not found: {old}"
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c = d / "ssd_oracle.c"
    c.write_text(src)
    so = d / "lib.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(c),
                    "-o", str(so), "-lm"], check=True)
    return ssd_ref.load_library(str(so))


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def battery(lib):
    """Returns {pin name: passed} for a small set of pins run on ``lib``."""
    res = {}
    LN2 = math.log(2.0)
    # geometric closed form with init (distinguishes B from C)
    L, P, N = 12, 2, 3
    x = np.array([1.5, -0.5]); Bv = np.array([0.2, -1.0, 0.4]); Cv = np.array([-0.3, 0.8, 0.5])
    init = (np.arange(P * N, dtype=float).reshape(1, 1, P, N) * 0.1 - 0.2)
    y, fin = lib.ssd_fwd(np.broadcast_to(x, (1, L, 1, P)).copy(), np.zeros((1, L, 1)),
                         np.zeros(1), np.array([-0.7]),
                         np.broadcast_to(Bv, (1, L, 1, N)).copy(),
                         np.broadcast_to(Cv, (1, L, 1, N)).copy(), np.array([0.3]),
                         initial_states=init)
    a = 2.0 ** -0.7
    u = LN2 * np.outer(x, Bv)
    ok = True
    for t in range(L):
        h = a ** (t + 1) * init[0, 0] + u * (1 - a ** (t + 1)) / (1 - a)
        ok &= _rel(y[0, t, 0], h @ Cv + 0.3 * x) < 1e-12
    res["geometric"] = bool(ok)
    # chunked (independent numpy) vs this build, fwd and bwd, with resets and groups
    inp = make_inputs(batch=2, seqlen=21, nheads=4, headdim=3, dstate=4, ngroups=2, init=True,
                      dfinal=True, seq_lengths=[6, 9, 6], seed=21)
    f = inp.f64
    args = [f(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D"]]
    kw = dict(initial_states=f("initial_states"), seq_idx=f("seq_idx"))
    y, fin = lib.ssd_fwd(*args, **kw)
    y2, fin2, _ = chunked.ssd_chunked_fwd(*args, 5, **kw)
    res["chunked_fwd"] = _rel(y, y2) < 1e-12 and _rel(fin, fin2) < 1e-12
    g = lib.ssd_bwd(*args, f("dy"), dfinal_states=f("dfinal_states"), **kw)
    g2 = chunked.ssd_chunked_bwd(*args, f("dy"), 5, dfinal_states=f("dfinal_states"), **kw)
    res["chunked_bwd"] = all(_rel(g[k], g2[k]) < 1e-11 for k in g)
    # finite differences of this build's own forward on a few coordinates
    names = ["x", "dt", "dt_bias", "A", "B", "C", "D", "initial_states"]
    gn = ["dx", "ddt", "ddt_bias", "dA", "dB", "dC", "dD", "dinitial_states"]
    arrs = [f(n) for n in names]

    def loss():
        yy, ff = lib.ssd_fwd(*arrs[:7], initial_states=arrs[7], seq_idx=f("seq_idx"))
        return float(np.sum(f("dy") * yy) + np.sum(f("dfinal_states") * ff))
    ok = True
    rng = np.random.default_rng(0)
    for k in range(len(names)):
        flat = arrs[k].reshape(-1)
        for i in rng.choice(flat.size, size=min(6, flat.size), replace=False):
            old = flat[i]
            flat[i] = old + 1e-6; lp = loss()
            flat[i] = old - 1e-6; lm = loss()
            flat[i] = old
            fd = (lp - lm) / 2e-6
            ok &= abs(fd - g[gn[k]].reshape(-1)[i]) <= 1e-5 * max(1.0, abs(fd))
    res["finite_differences"] = bool(ok)
    return res


def test_unmodified_oracle_passes_battery(tmp_path):
    res = battery(_build(tmp_path, "clean", None))
    assert all(res.values()), res


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    res = battery(_build(tmp_path, name, MUTANTS[name]))
    assert not all(res.values()), f"mutant {name} passed every pin: {res}"
