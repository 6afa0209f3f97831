"""Context parallelism of the SSD layer, pinned on the CPU.

The sequence is split into contiguous shards, every shard is evaluated on its
own by the float64 oracle, and the shards are joined by the exclusive folds
of ``oracle/context_parallel.py`` (forward: the state entering each shard;
backward: the gradient reaching each shard's final state).  The result must
equal the unsharded oracle -- y, final_states and every gradient -- for
splits inside segments, on segment boundaries (in some rows only), with a
reset inside a shard, one-token shards, initial states and an upstream
dfinal_states.  Two gloo ranks (spawned processes, 127.0.0.1) run the same
with the exchange as collectives.  Planted mistakes in a copy of the module
must each break the equality."""
import json
import os
import socket
import subprocess
import sys
import types

import numpy as np
import pytest

from mamba_selective_state_gb300.inputs import make_inputs
from oracle import context_parallel as cp
from oracle import ssd_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "context_parallel.py")
NAMES = ["x", "dt", "dt_bias", "A", "B", "C", "D", "dy", "initial_states", "dfinal_states"]


def seq_rows(L, lengths_per_row):
    ids = [np.repeat(np.arange(len(lens), dtype=np.int32), lens) for lens in lengths_per_row]
    assert all(len(r) == L for r in ids)
    return np.stack(ids)


def problem(L=48, seq=None, init=True, dfinal=True, seed=5):
    inp = make_inputs(batch=2, seqlen=L, nheads=4, headdim=3, dstate=5, ngroups=2, chunk=16,
                      dtype="f32", init=init, dfinal=dfinal, seed=seed)
    d = {n: inp.f64(n) for n in NAMES}
    d["seq_idx"] = seq
    return d


def full(d):
    kw = dict(initial_states=d["initial_states"], seq_idx=d["seq_idx"])
    args = [d[n] for n in ("x", "dt", "dt_bias", "A", "B", "C", "D")]
    y, fin = ssd_ref.ssd_fwd(*args, **kw)
    g = ssd_ref.ssd_bwd(*args, d["dy"], dfinal_states=d["dfinal_states"], **kw)
    g.update(y=y, final_states=fin)
    if d["initial_states"] is None:
        g.pop("dinitial_states", None)
    return g


def sharded(d, sizes, mod=cp):
    out = mod.context_parallel(ssd_ref.ssd_fwd, ssd_ref.ssd_bwd, d, sizes,
                               dfinal_states=d["dfinal_states"])
    if d["initial_states"] is None:
        out.pop("dinitial_states")
    return out


def max_rel(got, ref):
    return max(float(np.abs(got[k] - ref[k]).max() / max(np.abs(ref[k]).max(), 1e-300))
               for k in ref)


CASES = {
    # name: (L, per-row segment lengths or None, shard sizes, init, dfinal)
    "no_segments_three_shards": (48, None, [17, 16, 15], True, True),
    "reset_inside_a_shard": (48, [[10, 38], [30, 18]], [16, 16, 16], True, True),
    "segment_starts_on_a_shard_boundary_in_one_row": (48, [[16, 32], [20, 28]], [16, 16, 16],
                                                      True, True),
    "one_token_shards": (20, [[7, 13], [7, 13]], [1, 6, 1, 1, 11], True, True),
    "no_init_no_dfinal": (40, [[5, 5, 30], [40]], [13, 27], False, False),
    "many_segments_two_shards": (60, [[1, 1, 20, 38], [59, 1]], [30, 30], True, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_sharded_equals_unsharded(name):
    L, segs, sizes, init, dfinal = CASES[name]
    d = problem(L, None if segs is None else seq_rows(L, segs), init, dfinal)
    assert max_rel(sharded(d, sizes), full(d)) < 1e-11


def test_one_shard_is_the_unsharded_call():
    d = problem(32, seq_rows(32, [[12, 20], [32]]))
    assert max_rel(sharded(d, [32]), full(d)) < 1e-13


def test_shard_decay_closed_form():
    # dt_eff = softplus(dt + bias); decay = exp(A * sum dt_eff); a reset zeroes the row
    dt = np.zeros((2, 3, 1))
    bias = np.array([np.log(np.expm1(0.5))])     # softplus(bias) = 0.5
    dec = cp.shard_decay(dt, bias, np.array([-2.0]), seq_idx=np.array([[0, 0, 0], [4, 4, 5]]))
    assert abs(dec[0, 0] - np.exp(-3.0)) < 1e-15 and dec[1, 0] == 0.0


def test_breaks_compare_neighbouring_shards():
    brk = cp.shard_breaks(first_ids=[[0, 0], [0, 2], [1, 2]], last_ids=[[0, 1], [0, 2], [1, 3]])
    assert brk.tolist() == [[False, False], [False, True], [True, False]]


MUTANTS = {
    "forward_ignores_breaks": ("h[np.asarray(breaks[r], dtype=bool)] = 0.0\n        entering",
                               "pass\n        entering"),
    "reset_does_not_cut_decay": ("dec[reset, :] = 0.0", "pass"),
    "reverse_drops_decay": ("g = decays[r][:, :, None, None] * g + dinits0[r]",
                            "g = g + dinits0[r]"),
    "reverse_ignores_breaks": ("g[np.asarray(breaks[r], dtype=bool)] = 0.0",
                               "pass"),
    "reverse_drops_local_dinit": ("g = decays[r][:, :, None, None] * g + dinits0[r]",
                                  "g = decays[r][:, :, None, None] * g"),
    "forward_inclusive_fold": ("entering[r] = h\n        h = decays[r][:, :, None, None] * h + finals0[r]",
                               "h = decays[r][:, :, None, None] * h + finals0[r]\n        entering[r] = h"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_equality_catches_mutant(name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, old
    mod = types.ModuleType("cp_mutant")
    exec(compile(src.replace(old, new), "cp_mutant.py", "exec"), mod.__dict__)
    worst = 0.0
    for case in CASES.values():
        L, segs, sizes, init, dfinal = case
        d = problem(L, None if segs is None else seq_rows(L, segs), init, dfinal)
        worst = max(worst, max_rel(sharded(d, sizes, mod), full(d)))
    assert worst > 1e-6, name


# ---------------------------------------------------------------------------
# two gloo ranks: the exchange as collectives
# ---------------------------------------------------------------------------
WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import numpy as np, torch, torch.distributed as dist
from oracle import context_parallel as cp, ssd_ref
from tests.test_context_parallel import problem, seq_rows, full, max_rel
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
L = 48
d = problem(L, seq_rows(L, [[16, 32], [10, 38]]))      # row 0 starts a segment at the split
s, e = rank * L // world, (rank + 1) * L // world
cut = lambda a: None if a is None else a[:, s:e]
args = [cut(d["x"]), cut(d["dt"]), d["dt_bias"], d["A"], cut(d["B"]), cut(d["C"]), d["D"]]
seq = cut(d["seq_idx"])

def gather(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    out = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return np.stack([o.numpy() for o in out])

fin0 = ssd_ref.ssd_fwd(*args, seq_idx=seq)[1]
dec = cp.shard_decay(cut(d["dt"]), d["dt_bias"], d["A"], seq_idx=seq)
ids = gather(np.stack([seq[:, 0], seq[:, -1]]).astype(np.int64))
brk = cp.shard_breaks(ids[:, 0], ids[:, 1])
h_in, final = cp.carries_in(gather(dec), gather(fin0), brk, d["initial_states"])
y = ssd_ref.ssd_fwd(*args, initial_states=h_in[rank], seq_idx=seq)[0]
d0 = ssd_ref.ssd_bwd(*args, cut(d["dy"]), initial_states=h_in[rank], seq_idx=seq)["dinitial_states"]
g_out = cp.dfinals_out(gather(dec), gather(d0), brk, d["dfinal_states"])
g = ssd_ref.ssd_bwd(*args, cut(d["dy"]), initial_states=h_in[rank], seq_idx=seq,
                    dfinal_states=g_out[rank])
got = dict(y=np.concatenate(list(gather(y)), axis=1), final_states=final,
           dinitial_states=gather(g["dinitial_states"])[0])
for k in ("dx", "ddt", "dB", "dC"):
    got[k] = np.concatenate(list(gather(g[k])), axis=1)
for k in ("dA", "dD", "ddt_bias"):
    got[k] = gather(g[k]).sum(axis=0)
print(json.dumps({{"rank": rank, "err": max_rel(got, full(d))}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_match_the_unsharded_oracle():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for pr in procs:
        out, err = pr.communicate(timeout=240)
        assert pr.returncode == 0, err[-3000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["err"] < 1e-11 for o in outs), outs
