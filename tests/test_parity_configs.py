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
