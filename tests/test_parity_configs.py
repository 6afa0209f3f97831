"""Every GPU parity case draws valid inputs and the oracle runs on it (CPU
only), so that a mistake in a case's definition shows up without a GPU."""
import pytest

from mamba_selective_state_gb300.inputs import make_inputs
from tests.ref_helpers import oracle_full
from tests.test_parity_gpu import SMALL


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_case_is_well_formed(name):
    cfg = SMALL[name]
    inp = make_inputs(seed=3, **cfg)
    assert inp.seqlen == cfg["seqlen"] and inp.dtype == cfg["dtype"]
    if inp.batch * inp.seqlen * inp.nheads <= 4 * 4096:  # keep the CPU suite quick
        ref = oracle_full(inp)
        assert ref["y"].shape == (inp.batch, inp.seqlen, inp.nheads, inp.headdim)


def test_norm_parity_cases_pass_validation():
    """Every gated-norm GPU case is inside the library's limits (its
    workspace query succeeds) and the oracle runs on it."""
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.inputs import WORKLOADS, make_norm_inputs, norm_shape
    from oracle import gated_norm
    from tests.test_norm_gpu import SMALL as NORM_SMALL
    shapes = [(c[0], c[1], c[2], c[3], c[4]) for c in NORM_SMALL.values()]
    shapes += [(s["rows"], s["dim"], s["group_size"], s["dtype"], True)
               for s in map(norm_shape, WORKLOADS)]
    for rows, dim, gs, dtype, gate in shapes:
        prob = _lib.make_norm_problem(rows, dim, gs, 1e-5, _lib.SSD_BF16 if dtype == "bf16"
                                      else _lib.SSD_F32, gate=gate)
        assert _lib.ssd_gated_rmsnorm_bwd_workspace_bytes(prob) > 0, (rows, dim, gs, dtype)
    for rows, dim, gs, dtype, gate in shapes[:len(NORM_SMALL)]:
        inp = make_norm_inputs(rows, dim, gs, dtype=dtype, gate=gate, seed=7)
        out, rstd = gated_norm.gated_rmsnorm_fwd(inp.f64("y"), inp.f64("z"), inp.f64("weight"),
                                                 gs, inp.eps)
        assert out.shape == (rows, dim) and rstd.shape == (rows, dim // gs)


def test_norm_shapes_follow_the_layer_workloads():
    """The norm after each layer workload has one row per token, H*P columns
    and H*P/G columns per group (the packed workload's rows are its drawn
    total)."""
    from mamba_selective_state_gb300.inputs import WORKLOADS, make_workload, norm_shape
    for name, cfg in WORKLOADS.items():
        s = norm_shape(name)
        dim = cfg["nheads"] * cfg["headdim"]
        assert s["dim"] == dim and s["group_size"] * cfg["ngroups"] == dim
        if "nseq" in cfg:
            inp = make_workload(name, seed=0)
            assert s["rows"] == inp.batch * inp.seqlen
        else:
            assert s["rows"] == cfg["batch"] * cfg["seqlen"]
