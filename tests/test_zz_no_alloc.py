"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device
memory where they call the layer (a plain C host without access to the
framework's allocator, or a loop where allocating is not allowed).  It uses
the library's own statically sized device array instead of a caller
workspace.

Checked through the C ABI against ssd_fwd (which uses a caller workspace), on
two calls in a row (the array keeps the previous call's contents), within the
parity tolerance of the bf16 tests.  This file is collected last on purpose."""
import pytest
import torch

from mamba_selective_state_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from mamba_selective_state_gb300 import _lib
    return _lib


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def test_noalloc_forward_matches_workspace_forward_twice(lib):
    from mamba_selective_state_gb300.runner import SSDDevice
    cases = [
        dict(batch=1, seqlen=700, nheads=8, headdim=64, dstate=64, ngroups=4, chunk=128, dtype="bf16",
             seq_lengths=[256, 3, 300, 141], seed=21),
        dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2, chunk=128, dtype="bf16",
             init=True, seed=22),
    ]
    for cfg in cases:
        inp = make_inputs(**cfg)
        dev = SSDDevice(inp, device="cuda", backward=False)
        assert lib.ssd_fwd_workspace_bytes(dev.fwd_prob) <= lib.SSD_NOALLOC_SCRATCH_BYTES
        dev.fwd()
        torch.cuda.synchronize()
        y_ref, fin_ref = dev.y.clone(), dev.final.clone()
        for _ in range(2):
            dev.y.zero_()
            dev.final.zero_()
            rc = lib.ssd_fwd_noalloc(dev.fwd_prob, dev.x, dev.dt, dev.dt_bias, dev.A, dev.B, dev.C,
                                     dev.D, dev.init, dev.seq_idx, dev.y, dev.final)
            assert rc == lib.SSD_OK, lib.status_string(rc)
            torch.cuda.synchronize()
            assert _rel(dev.y, y_ref) <= TOL
            assert _rel(dev.final, fin_ref) <= TOL


def test_noalloc_rejects_problems_beyond_the_array(lib):
    p = lib.make_problem(2, 8192, 64, 64, 128, 8, 128, lib.SSD_BF16, 0)
    assert lib.ssd_fwd_workspace_bytes(p) > lib.SSD_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = lib.ssd_fwd_noalloc(p, fake, fake, fake, fake, fake, fake, fake, None, None, fake, fake,
                             stream=0)
    assert rc == lib.SSD_ERR_WORKSPACE_TOO_SMALL
