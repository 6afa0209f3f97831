"""Context parallelism on the GPU: the sequence split into shards run one
after another on one GPU through ssd_fwd / ssd_bwd, joined by
ssd_shard_decay and the two ssd_shard_fold folds, compared with the float64
oracle of the unsharded layer (not with the GPU's own unsharded run).
Tolerances as for the layer: max|diff| <= 2e-2 max|ref| (bf16), 1e-4 (fp32)."""
import numpy as np
import pytest
import torch

from mamba_selective_state_gb300.inputs import make_inputs
from tests.ref_helpers import assert_close, oracle_full

pytestmark = pytest.mark.gpu

CASES = {
    # resets inside shards, a sequence start exactly on a shard boundary
    # (token 250), a one-token shard, initial states and dfinal
    "bf16_N64_resets": (dict(batch=2, seqlen=700, nheads=4, headdim=64, dstate=64, ngroups=2,
                             chunk=128, dtype="bf16", init=True, dfinal=True,
                             seq_lengths=[250, 3, 300, 147]), [250, 1, 300, 149]),
    "bf16_N128_plain": (dict(batch=1, seqlen=600, nheads=4, headdim=64, dstate=128, ngroups=1,
                             chunk=128, dtype="bf16", init=True, dfinal=True), [128, 200, 272]),
    "fp32_small": (dict(batch=2, seqlen=200, nheads=2, headdim=16, dstate=16, ngroups=1, chunk=32,
                        dtype="f32", init=True, dfinal=True, seq_lengths=[60, 1, 139]),
                   [60, 70, 1, 69]),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("name", sorted(CASES))
def test_sharded_layer_matches_unsharded_oracle(name):
    from mamba_selective_state_gb300.context_parallel import (StackExchange, run_sharded,
                                                              shard_bounds, shard_inputs)
    cfg, sizes = CASES[name]
    inp = make_inputs(seed=5, **cfg)
    bounds = shard_bounds(inp.seqlen, sizes)
    shards = [shard_inputs(inp, s, e) for s, e in bounds]
    out = run_sharded(shards, list(range(len(shards))), StackExchange(len(shards)),
                      initial_states=inp.initial_states, dfinal_states=inp.dfinal_states)
    torch.cuda.synchronize()
    got = {"y": torch.cat([out["y"][r] for r in range(len(shards))], dim=1),
           "final_states": out["final_states"]}
    for k in ("dx", "ddt", "dB", "dC"):
        got[k] = torch.cat([out[k][r] for r in range(len(shards))], dim=1)
    for k in ("dA", "dD", "ddt_bias", "dinitial_states"):
        got[k] = out[k]
    got = {k: v.detach().to("cpu", torch.float64) for k, v in got.items()}
    assert_close(got, oracle_full(inp), inp.dtype)


def test_shard_fold_matches_its_definition():
    """The fold kernels against the recurrence that defines them, written out
    on the host in float64 for random pairs, with sequence starts on some
    shard boundaries."""
    from mamba_selective_state_gb300 import _lib
    g = torch.Generator().manual_seed(0)
    R, b, H, P, N = 5, 3, 2, 4, 8
    dec = torch.rand((R, b, H), generator=g)
    loc = torch.randn((R, b, H, P, N), generator=g)
    bnd = torch.randn((b, H, P, N), generator=g)
    first = torch.tensor([[0, 0, 0], [0, 1, 0], [1, 1, 2], [1, 2, 2], [3, 2, 2]], dtype=torch.int32)
    last = torch.tensor([[0, 0, 0], [0, 1, 1], [1, 2, 2], [2, 2, 2], [3, 3, 2]], dtype=torch.int32)
    for rev in (False, True):
        out = torch.empty((R, b, H, P, N), device="cuda")
        tot = torch.empty((b, H, P, N), device="cuda")
        _lib.ssd_shard_fold(dec.cuda(), loc.cuda(), first.cuda(), last.cuda(), bnd.cuda(), out, tot,
                            reverse=rev)
        torch.cuda.synchronize()
        v = bnd.double().clone()
        want = torch.empty((R, b, H, P, N), dtype=torch.float64)
        order = range(R - 1, -1, -1) if rev else range(R)
        for r in order:
            brk = torch.zeros(b, dtype=torch.bool) if r == 0 else (first[r] != last[r - 1])
            if not rev:
                v[brk] = 0.0
            want[r] = v
            v = dec[r].double()[:, :, None, None] * v + loc[r].double()
            if rev:
                v[brk] = 0.0
        np.testing.assert_allclose(out.cpu().double().numpy(), want.numpy(), rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(tot.cpu().double().numpy(), v.numpy(), rtol=1e-6, atol=1e-6)
