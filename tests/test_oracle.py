"""Pins of the float64 oracle against facts that do not come from the oracle:
closed forms, invariants, independent evaluation orders and finite
differences.  CPU only."""
import math

import numpy as np
import pytest

from mamba_selective_state_gb300.inputs import make_inputs
from oracle import chunked, scan, ssd_ref

LN2 = math.log(2.0)
FWD_NAMES = ["x", "dt", "dt_bias", "A", "B", "C", "D"]


def fwd_args(inp):
    return [inp.f64(n) for n in FWD_NAMES]


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def const_problem(L, P, N, A_h, D_h, x, Bv, Cv, init):
    """One row, one head: dt + dt_bias = 0 on every token (dt_eff = ln 2)."""
    xs = np.broadcast_to(np.asarray(x, float), (1, L, 1, P)).copy()
    dt = np.zeros((1, L, 1))
    Bs = np.broadcast_to(np.asarray(Bv, float), (1, L, 1, N)).copy()
    Cs = np.broadcast_to(np.asarray(Cv, float), (1, L, 1, N)).copy()
    return xs, dt, np.zeros(1), np.array([A_h]), Bs, Cs, np.array([D_h]), init


# --- P1: constant inputs give a geometric series -----------------------------
def test_geometric_closed_form():
    L, P, N = 20, 2, 3
    A_h, D_h = -0.7, 0.3
    x = np.array([1.5, -0.5])
    Bv = np.array([0.2, -1.0, 0.4])
    Cv = np.array([-0.3, 0.8, 0.5])       # B != C so that swapping them shows
    init = np.arange(P * N, dtype=float).reshape(1, 1, P, N) * 0.1 - 0.2
    xs, dt, bias, A, Bs, Cs, D, init = const_problem(L, P, N, A_h, D_h, x, Bv, Cv, init)
    y, fin = ssd_ref.ssd_fwd(xs, dt, bias, A, Bs, Cs, D, initial_states=init)
    a = math.exp(LN2 * A_h)
    u = LN2 * np.outer(x, Bv)
    for t in range(L):
        k = t + 1
        h = a ** k * init[0, 0] + u * (1 - a ** k) / (1 - a)
        assert rel(y[0, t, 0], h @ Cv + D_h * x) < 1e-13
    h_last = a ** L * init[0, 0] + u * (1 - a ** L) / (1 - a)
    assert rel(fin[0, 0], h_last) < 1e-13


# --- P2: dt -> 0 leaves only the skip term and the undecayed carry -----------
def test_dt_to_zero():
    inp = make_inputs(batch=2, seqlen=17, nheads=4, headdim=3, dstate=5, ngroups=2,
                      init=True, seed=3)
    args = fwd_args(inp)
    args[2] = np.full_like(args[2], -100.0)        # dt_eff ~ 3.7e-44
    init = inp.f64("initial_states")
    y, fin = ssd_ref.ssd_fwd(*args, initial_states=init)
    x, C, D = args[0], args[5], args[6]
    g = np.arange(4) * 2 // 4
    expect = np.einsum("bhpn,blhn->blhp", init, C[:, :, g, :]) + D[None, None, :, None] * x
    assert np.abs(y - expect).max() < 1e-12
    assert np.abs(fin - init).max() < 1e-12
    y0, _ = ssd_ref.ssd_fwd(*args)
    assert np.abs(y0 - D[None, None, :, None] * x).max() < 1e-30


# --- P3: a single token -------------------------------------------------------
def test_single_token():
    rng = np.random.default_rng(5)
    P, N = 4, 6
    x = rng.standard_normal((1, 1, 1, P))
    Bv = rng.standard_normal((1, 1, 1, N))
    Cv = rng.standard_normal((1, 1, 1, N))
    y, fin = ssd_ref.ssd_fwd(x, np.zeros((1, 1, 1)), np.zeros(1), np.array([-3.0]), Bv, Cv,
                             np.array([0.25]))
    expect = LN2 * float(Cv[0, 0, 0] @ Bv[0, 0, 0]) * x[0, 0, 0] + 0.25 * x[0, 0, 0]
    assert rel(y[0, 0, 0], expect) < 1e-14
    assert rel(fin[0, 0], LN2 * np.outer(x[0, 0, 0], Bv[0, 0, 0])) < 1e-14


def test_two_tokens_by_hand():
    """L = 2, P = N = 1: y_1 = C_1 (a_1 dt_0 x_0 B_0 + dt_1 x_1 B_1) + D x_1,
    with dt_eff = ln 2 on both tokens and a = 2**A."""
    x = np.array([2.0, -1.0]).reshape(1, 2, 1, 1)
    Bs = np.array([0.5, 3.0]).reshape(1, 2, 1, 1)
    Cs = np.array([-1.0, 0.25]).reshape(1, 2, 1, 1)
    A_h, D_h = -1.0, 0.5                          # a = 2**-1 = 0.5 on every token
    y, fin = ssd_ref.ssd_fwd(x, np.zeros((1, 2, 1)), np.zeros(1), np.array([A_h]), Bs, Cs,
                             np.array([D_h]))
    h0 = LN2 * 2.0 * 0.5                          # ln2
    h1 = 0.5 * h0 + LN2 * (-1.0) * 3.0            # -2.5 ln2
    assert abs(y[0, 0, 0, 0] - (-1.0 * h0 + 0.5 * 2.0)) < 1e-15
    assert abs(y[0, 1, 0, 0] - (0.25 * h1 + 0.5 * -1.0)) < 1e-15
    assert abs(fin[0, 0, 0, 0] - h1) < 1e-15


# --- P4 / P10: the pair combine is associative; Hillis-Steele == sequential --
def test_combine_associative_identity_reset():
    rng = np.random.default_rng(0)
    for _ in range(50):
        p, q, r = [(rng.uniform(0, 1), rng.standard_normal((3, 4))) for _ in range(3)]
        lhs = scan.combine(scan.combine(p, q), r)
        rhs = scan.combine(p, scan.combine(q, r))
        assert abs(lhs[0] - rhs[0]) < 1e-15 and np.abs(lhs[1] - rhs[1]).max() < 1e-13
        e = scan.combine(scan.IDENTITY, p)
        assert e[0] == p[0] and np.array_equal(e[1], p[1])
        e = scan.combine(p, scan.IDENTITY)
        assert e[0] == p[0] and np.array_equal(e[1], p[1])
        z = scan.combine(p, (0.0, q[1]))          # a reset discards the left span
        assert z[0] == 0.0 and np.array_equal(z[1], q[1])
    # the combine is not commutative: the order of spans matters
    p, q = (0.5, np.ones(2)), (0.25, 2 * np.ones(2))
    assert not np.allclose(scan.combine(p, q)[1], scan.combine(q, p)[1])


@pytest.mark.parametrize("n", [1, 2, 5, 8, 31, 32, 33, 100])
def test_hillis_steele_equals_sequential(n):
    rng = np.random.default_rng(n)
    pairs = [(rng.uniform(0, 1), rng.standard_normal(3)) for _ in range(n)]
    hs = scan.hillis_steele_scan(pairs)
    sq = scan.sequential_scan(pairs)
    for (a1, b1), (a2, b2) in zip(hs, sq):
        assert abs(a1 - a2) < 1e-15 and np.abs(b1 - b2).max() < 1e-12


def test_scan_of_pairs_reproduces_recurrence():
    """States from scanning (a_t, dt_eff_t x_t B_t) match the oracle's output."""
    inp = make_inputs(batch=1, seqlen=23, nheads=1, headdim=1, dstate=1, init=True, seed=7)
    args = fwd_args(inp)
    x, dt, bias, A, B, C, D = args
    init = inp.f64("initial_states")
    y, fin = ssd_ref.ssd_fwd(*args, initial_states=init)
    de = np.log1p(np.exp(dt[0, :, 0] + bias[0]))
    a = np.exp(de * A[0])
    b = de * x[0, :, 0, 0] * B[0, :, 0, 0]
    hs = scan.states_from_scan(list(a), list(b), init[0, 0, 0, 0])
    for t in range(23):
        assert abs(y[0, t, 0, 0] - (hs[t] * C[0, t, 0, 0] + D[0] * x[0, t, 0, 0])) < 1e-12
    assert abs(fin[0, 0, 0, 0] - hs[-1]) < 1e-12


# --- P5: chunked evaluation equals the sequential recurrence ------------------
CHUNK_CASES = [
    dict(L=37, Q=1, seqs=None, init=False),
    dict(L=37, Q=3, seqs=None, init=True),
    dict(L=37, Q=8, seqs=[5, 11, 2, 19], init=True),
    dict(L=64, Q=64, seqs=None, init=True),
    dict(L=37, Q=37, seqs=[16, 1, 20], init=False),
    dict(L=40, Q=8, seqs=[8, 8, 24], init=True),       # resets on chunk starts
]


@pytest.mark.parametrize("case", CHUNK_CASES)
def test_chunked_equals_sequential(case):
    inp = make_inputs(batch=2, seqlen=case["L"], nheads=4, headdim=3, dstate=5, ngroups=2,
                      init=case["init"], dfinal=True, seq_lengths=case["seqs"], seed=11)
    args = fwd_args(inp)
    kw = dict(initial_states=inp.f64("initial_states"), seq_idx=inp.f64("seq_idx"))
    y, fin = ssd_ref.ssd_fwd(*args, **kw)
    y2, fin2, inter = chunked.ssd_chunked_fwd(*args, case["Q"], **kw)
    assert rel(y2, y) < 1e-13 and rel(fin2, fin) < 1e-13
    g = ssd_ref.ssd_bwd(*args, inp.f64("dy"), dfinal_states=inp.f64("dfinal_states"), **kw)
    g2 = chunked.ssd_chunked_bwd(*args, inp.f64("dy"), case["Q"],
                                 dfinal_states=inp.f64("dfinal_states"), **kw)
    for k in g:
        assert rel(g2[k], g[k]) < 1e-12, k


def test_state_passing_is_the_pair_scan():
    """Carry-in states of the chunked evaluation equal the Hillis-Steele scan of
    the chunk pairs (a_c, S_c) applied to the initial state."""
    inp = make_inputs(batch=1, seqlen=50, nheads=2, headdim=2, dstate=3, init=True,
                      seq_lengths=[20, 30], seed=2)
    _, _, inter = chunked.ssd_chunked_fwd(*fwd_args(inp), 8,
                                          initial_states=inp.f64("initial_states"),
                                          seq_idx=inp.f64("seq_idx"))
    for h in range(2):
        a = inter["a_chunk"][0, h]
        S = inter["S"][0, h]
        pre = scan.hillis_steele_scan(scan.as_array_pairs(a, S))
        for c in range(len(a)):
            hc = scan.apply(pre[c], inp.f64("initial_states")[0, h])
            assert np.abs(hc - inter["H_in"][0, h, c + 1]).max() < 1e-12


# --- P6: a packed row equals the separate sequences ---------------------------
def test_packed_equals_separate():
    lens = [7, 13, 4, 9]
    L = sum(lens)
    inp = make_inputs(batch=1, seqlen=L, nheads=4, headdim=3, dstate=4, ngroups=2, init=True,
                      dfinal=True, seq_lengths=lens, seed=4)
    args = fwd_args(inp)
    init, dfin, dy = inp.f64("initial_states"), inp.f64("dfinal_states"), inp.f64("dy")
    y, fin = ssd_ref.ssd_fwd(*args, initial_states=init, seq_idx=inp.f64("seq_idx"))
    gp = ssd_ref.ssd_bwd(*args, dy, initial_states=init, seq_idx=inp.f64("seq_idx"),
                         dfinal_states=dfin)
    t0 = 0
    sums = dict(dA=0.0, dD=0.0, ddt_bias=0.0)
    for k, n in enumerate(lens):
        sl = slice(t0, t0 + n)
        part = [args[0][:, sl], args[1][:, sl], args[2], args[3], args[4][:, sl],
                args[5][:, sl], args[6]]
        kin = init if k == 0 else None
        kdf = dfin if k == len(lens) - 1 else None
        ys, fs = ssd_ref.ssd_fwd(*part, initial_states=kin)
        assert rel(y[:, sl], ys) < 1e-14
        gs = ssd_ref.ssd_bwd(*part, dy[:, sl], initial_states=kin, dfinal_states=kdf)
        for name in ("dx", "ddt", "dB", "dC"):
            assert rel(gp[name][:, sl], gs[name]) < 1e-13, name
        for name in sums:
            sums[name] = sums[name] + gs[name]
        if k == 0:
            assert rel(gp["dinitial_states"], gs["dinitial_states"]) < 1e-13
        t0 += n
    assert rel(fin, fs) < 1e-14
    for name in sums:
        assert rel(gp[name], sums[name]) < 1e-12, name


# --- P7: resuming from the final state ----------------------------------------
def test_resume_from_final_state():
    L, k = 30, 11
    inp = make_inputs(batch=2, seqlen=L, nheads=2, headdim=3, dstate=4, init=True, dfinal=True,
                      seed=6)
    args = fwd_args(inp)
    init, dfin, dy = inp.f64("initial_states"), inp.f64("dfinal_states"), inp.f64("dy")
    y, fin = ssd_ref.ssd_fwd(*args, initial_states=init)
    first = [a[:, :k] if a.ndim >= 3 else a for a in args]
    second = [a[:, k:] if a.ndim >= 3 else a for a in args]
    y1, f1 = ssd_ref.ssd_fwd(*first, initial_states=init)
    y2, f2 = ssd_ref.ssd_fwd(*second, initial_states=f1)
    assert rel(np.concatenate([y1, y2], axis=1), y) < 1e-14 and rel(f2, fin) < 1e-14
    g = ssd_ref.ssd_bwd(*args, dy, initial_states=init, dfinal_states=dfin)
    g2 = ssd_ref.ssd_bwd(*second, dy[:, k:], initial_states=f1, dfinal_states=dfin)
    g1 = ssd_ref.ssd_bwd(*first, dy[:, :k], initial_states=init,
                         dfinal_states=g2["dinitial_states"])
    assert rel(g1["dinitial_states"], g["dinitial_states"]) < 1e-13
    assert rel(np.concatenate([g1["dx"], g2["dx"]], 1), g["dx"]) < 1e-13
    assert rel(g1["dA"] + g2["dA"], g["dA"]) < 1e-12


# --- P8: scale invariance and linearity in x ----------------------------------
def test_scale_invariance_and_linearity():
    inp = make_inputs(batch=1, seqlen=19, nheads=2, headdim=3, dstate=4, seed=8)
    x, dt, bias, A, B, C, D = fwd_args(inp)
    y, _ = ssd_ref.ssd_fwd(x, dt, bias, A, B, C, D)
    ys, _ = ssd_ref.ssd_fwd(x, dt, bias, A, 4.0 * B, C / 4.0, D)
    assert rel(ys, y) < 1e-14
    x2 = np.random.default_rng(1).standard_normal(x.shape)
    y2, _ = ssd_ref.ssd_fwd(x2, dt, bias, A, B, C, D)
    y3, _ = ssd_ref.ssd_fwd(2.0 * x - 3.0 * x2, dt, bias, A, B, C, D)
    assert rel(y3, 2.0 * y - 3.0 * y2) < 1e-13


def test_head_to_group_map():
    """Heads are split into G contiguous blocks; block k reads group k's B, C.
    Running each block alone with its group's B, C reproduces the outputs."""
    H, G = 6, 3
    inp = make_inputs(batch=1, seqlen=15, nheads=H, headdim=2, dstate=3, ngroups=G, seed=9)
    x, dt, bias, A, B, C, D = fwd_args(inp)
    y, _ = ssd_ref.ssd_fwd(x, dt, bias, A, B, C, D)
    hg = H // G
    for g in range(G):
        hs = slice(g * hg, (g + 1) * hg)
        yg, _ = ssd_ref.ssd_fwd(x[:, :, hs], dt[:, :, hs], bias[hs], A[hs], B[:, :, g:g + 1],
                                C[:, :, g:g + 1], D[hs])
        assert rel(y[:, :, hs], yg) < 1e-15


# --- P9: finite differences of the forward pin every gradient -----------------
def _loss(inp_arrays, dy, dfin, seq):
    x, dt, bias, A, B, C, D, init = inp_arrays
    y, fin = ssd_ref.ssd_fwd(x, dt, bias, A, B, C, D, initial_states=init, seq_idx=seq)
    return float(np.sum(dy * y) + np.sum(dfin * fin))


@pytest.mark.parametrize("shape", [
    dict(L=9, H=2, P=2, N=3, G=1, seqs=None),
    dict(L=12, H=4, P=2, N=2, G=2, seqs=[5, 3, 4]),
    dict(L=7, H=2, P=3, N=2, G=2, seqs=[1, 6]),
])
def test_finite_differences(shape):
    inp = make_inputs(batch=2, seqlen=shape["L"], nheads=shape["H"], headdim=shape["P"],
                      dstate=shape["N"], ngroups=shape["G"], init=True, dfinal=True,
                      seq_lengths=shape["seqs"], seed=13, init_std=0.5)
    names = ["x", "dt", "dt_bias", "A", "B", "C", "D", "initial_states"]
    arrs = [inp.f64(n) for n in names]
    dy, dfin, seq = inp.f64("dy"), inp.f64("dfinal_states"), inp.f64("seq_idx")
    g = ssd_ref.ssd_bwd(*arrs[:7], dy, initial_states=arrs[7], seq_idx=seq,
                        dfinal_states=dfin)
    grad_names = ["dx", "ddt", "ddt_bias", "dA", "dB", "dC", "dD", "dinitial_states"]
    eps = 1e-6
    for k, (name, gname) in enumerate(zip(names, grad_names)):
        fd = np.zeros_like(arrs[k])
        flat = arrs[k].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(arrs, dy, dfin, seq)
            flat[i] = old - eps
            lm = _loss(arrs, dy, dfin, seq)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * eps)
        err = np.abs(fd - g[gname]).max() / max(np.abs(fd).max(), 1e-12)
        assert err < 1e-6, (gname, err)


def test_dfinal_only_gradient_is_decay_product():
    """With dy = 0 and dfinal = 1 on one element, dinit is the product of all
    decays a_t (no input terms reach the initial state)."""
    inp = make_inputs(batch=1, seqlen=10, nheads=1, headdim=1, dstate=1, init=True, seed=12)
    args = fwd_args(inp)
    dfin = np.ones((1, 1, 1, 1))
    g = ssd_ref.ssd_bwd(*args, np.zeros((1, 10, 1, 1)), initial_states=inp.f64("initial_states"),
                        dfinal_states=dfin)
    x, dt, bias, A = args[:4]
    de = np.log1p(np.exp(dt[0, :, 0] + bias[0]))
    assert rel(g["dinitial_states"][0, 0, 0, 0], np.exp(np.sum(de) * A[0])) < 1e-13


def test_group_restriction_equals_full_run():
    """The group-restricted run (one group's heads, each with a copy of the
    group's B and C; dB, dC summed over the heads) equals the slice of the
    full run: heads of other groups do not touch this group's outputs."""
    inp = make_inputs(batch=2, seqlen=37, nheads=6, headdim=3, dstate=4, ngroups=3, chunk=16,
                      dtype="f32", init=True, dfinal=True, seq_lengths=[20, 17], seed=4)
    f = inp.f64
    args = [f(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D"]]
    kw = dict(initial_states=f("initial_states"), seq_idx=f("seq_idx"))
    y, fin = ssd_ref.ssd_fwd(*args, **kw)
    full = ssd_ref.ssd_bwd(*args, f("dy"), dfinal_states=f("dfinal_states"), **kw)
    for g in range(3):
        hs = slice(2 * g, 2 * g + 2)
        got = ssd_ref.ssd_group(*args, f("dy"), g, 3, dfinal_states=f("dfinal_states"), **kw)
        np.testing.assert_allclose(got["y"], y[:, :, hs], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got["final_states"], fin[:, hs], rtol=1e-12, atol=1e-14)
        for k in ("dx", "ddt"):
            np.testing.assert_allclose(got[k], full[k][:, :, hs], rtol=1e-12, atol=1e-14)
        for k in ("dA", "dD", "ddt_bias"):
            np.testing.assert_allclose(got[k], full[k][hs], rtol=1e-12, atol=1e-14)
        for k in ("dB", "dC"):
            np.testing.assert_allclose(got[k], full[k][:, :, g:g + 1], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got["dinitial_states"], full["dinitial_states"][:, hs],
                                   rtol=1e-12, atol=1e-14)
