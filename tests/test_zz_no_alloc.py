"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device
memory where they call the layer (a plain C host without access to the
framework's allocator, or a loop where allocating is not allowed).  It uses
the library's own statically sized device array instead of a caller
workspace.

Checked through the C ABI against ssd_fwd (which uses a caller workspace) on
two calls in a row: the array keeps the previous call's contents, and the
larger case runs first so that the smaller one starts on a dirty array.  Both
entry points run the same deterministic kernels, so the outputs must agree
bit for bit, and the array's status word (read with
ssd_fwd_noalloc_read_device_status) must be clean after every call.  This
file is collected last on purpose."""
import pytest
import torch

from mamba_selective_state_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from mamba_selective_state_gb300 import _lib
    return _lib


def _noalloc(lib, dev):
    return lib.ssd_fwd_noalloc(dev.fwd_prob, dev.x, dev.dt, dev.dt_bias, dev.A, dev.B, dev.C,
                               dev.D, dev.init, dev.seq_idx, dev.y, dev.final)


CASES = [
    # larger first: the smaller case then starts on the leftovers of this one
    dict(batch=2, seqlen=1500, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=128,
         dtype="bf16", init=True, seq_lengths=[700, 1, 799], seed=23),
    dict(batch=1, seqlen=700, nheads=8, headdim=64, dstate=64, ngroups=4, chunk=128, dtype="bf16",
         seq_lengths=[256, 3, 300, 141], seed=21),
    dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2, chunk=128, dtype="bf16",
         init=True, seed=22),
]


def test_noalloc_forward_matches_workspace_forward_twice(lib):
    from mamba_selective_state_gb300.runner import SSDDevice
    for cfg in CASES:
        inp = make_inputs(**cfg)
        dev = SSDDevice(inp, device="cuda", backward=False)
        assert lib.ssd_fwd_workspace_bytes(dev.fwd_prob) <= lib.SSD_NOALLOC_SCRATCH_BYTES
        dev.fwd()
        torch.cuda.synchronize()
        assert dev.device_status() == lib.SSD_OK
        y_ref, fin_ref = dev.y.clone(), dev.final.clone()
        for _ in range(2):
            dev.y.fill_(float("nan"))
            dev.final.fill_(float("nan"))
            rc = _noalloc(lib, dev)
            assert rc == lib.SSD_OK, lib.status_string(rc)
            assert lib.ssd_fwd_noalloc_read_device_status() == lib.SSD_OK
            assert torch.equal(dev.y, y_ref)
            assert torch.equal(dev.final, fin_ref)


def test_noalloc_reports_a_device_side_timeout(lib):
    """A scan tile that never publishes (the testing flag) makes its
    successors exhaust their bounded wait; the timeout is recorded in the
    library array's status word and read back through the C ABI, and the next
    normal call clears it and is exact again."""
    from mamba_selective_state_gb300.runner import SSDDevice
    cfg = dict(batch=1, seqlen=64 * 40 + 5, nheads=2, headdim=64, dstate=16, ngroups=1, chunk=64,
               dtype="bf16", init=True, seed=1)
    inp = make_inputs(**cfg)
    dev = SSDDevice(inp, device="cuda", backward=False)
    dev.fwd()
    torch.cuda.synchronize()
    y_ref, fin_ref = dev.y.clone(), dev.final.clone()
    drop = SSDDevice(inp, device="cuda", backward=False,
                     extra_flags=lib.SSD_TEST_DROP_SCAN_PUBLISH)
    rc = lib.ssd_fwd_noalloc(drop.fwd_prob, drop.x, drop.dt, drop.dt_bias, drop.A, drop.B, drop.C,
                             drop.D, drop.init, drop.seq_idx, drop.y, drop.final)
    assert rc == lib.SSD_OK
    assert lib.ssd_fwd_noalloc_read_device_status() == lib.SSD_ERR_TIMEOUT
    assert _noalloc(lib, dev) == lib.SSD_OK
    assert lib.ssd_fwd_noalloc_read_device_status() == lib.SSD_OK
    assert torch.equal(dev.y, y_ref) and torch.equal(dev.final, fin_ref)


def test_noalloc_rejects_problems_beyond_the_array(lib):
    p = lib.make_problem(2, 8192, 64, 64, 128, 8, 128, lib.SSD_BF16, 0)
    assert lib.ssd_fwd_workspace_bytes(p) > lib.SSD_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = lib.ssd_fwd_noalloc(p, fake, fake, fake, fake, fake, fake, fake, None, None, fake, fake,
                             stream=0)
    assert rc == lib.SSD_ERR_WORKSPACE_TOO_SMALL
