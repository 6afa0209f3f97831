"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Small cases span several chunks and token blocks with ragged tails and run the
oracle on the whole problem; the five layer workloads run at full size in the
launch configuration the benchmark times and are compared on one sampled
group (every batch row, all heads of the group, every token).  Tolerance:
max|diff| <= 2e-2 max|ref| (bf16) or 1e-4 max|ref| (fp32), per tensor."""
import numpy as np
import pytest
import torch

from mamba_selective_state_gb300.inputs import WORKLOADS, make_inputs, make_workload
from tests.ref_helpers import assert_close, oracle_full, oracle_group, slice_group

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def run_device(inp, **kw):
    from mamba_selective_state_gb300.runner import SSDDevice
    dev = SSDDevice(inp, device="cuda", **kw)
    dev.fwd()
    # the backward's first kernel resets the status word: read the forward's first
    assert dev.device_status() == 0
    dev.bwd()
    torch.cuda.synchronize()
    assert dev.device_status() == 0
    return dev, dev.results()


SMALL = {
    "tiny_fp32": dict(batch=1, seqlen=256, nheads=4, headdim=16, dstate=16, ngroups=1,
                      chunk=64, dtype="f32"),
    "fp32_ragged_init_resets": dict(batch=2, seqlen=250, nheads=4, headdim=16, dstate=32,
                                    ngroups=2, chunk=64, dtype="f32", init=True, dfinal=True,
                                    seq_lengths=[64, 1, 100, 85]),
    "fp32_P64_N128": dict(batch=1, seqlen=200, nheads=2, headdim=64, dstate=128, ngroups=1,
                          chunk=128, dtype="f32", init=True),
    "bf16_N128_G2": dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2,
                         chunk=128, dtype="bf16", init=True, dfinal=True,
                         seq_lengths=[100, 128, 72]),
    "bf16_N16_Q64": dict(batch=3, seqlen=333, nheads=6, headdim=64, dstate=16, ngroups=1,
                         chunk=64, dtype="bf16"),
    "bf16_N64_G4_varlen": dict(batch=1, seqlen=700, nheads=8, headdim=64, dstate=64, ngroups=4,
                               chunk=128, dtype="bf16", seq_lengths=[256, 3, 300, 141]),
    "bf16_Q256_init": dict(batch=1, seqlen=600, nheads=4, headdim=64, dstate=128, ngroups=1,
                           chunk=256, dtype="bf16", init=True),
    "bf16_P128_N64": dict(batch=1, seqlen=160, nheads=2, headdim=128, dstate=64, ngroups=1,
                          chunk=32, dtype="bf16", init=True, dfinal=True),
    "bf16_P32_N32_Q16": dict(batch=2, seqlen=100, nheads=4, headdim=32, dstate=32, ngroups=2,
                             chunk=16, dtype="bf16", seq_lengths=[16, 16, 68]),
    "bf16_single_token": dict(batch=2, seqlen=1, nheads=2, headdim=64, dstate=64, ngroups=1,
                              chunk=64, dtype="bf16", init=True, dfinal=True),
    "bf16_shorter_than_chunk": dict(batch=1, seqlen=37, nheads=2, headdim=64, dstate=128,
                                    ngroups=2, chunk=128, dtype="bf16"),
    "bf16_many_chunks": dict(batch=1, seqlen=64 * 40 + 5, nheads=2, headdim=64, dstate=16,
                             ngroups=1, chunk=64, dtype="bf16", init=True, dfinal=True),
    # 201 chunks: 26 scan segments of 8 chunks, joined across 4 checkpoint spans
    "bf16_many_segments": dict(batch=2, seqlen=64 * 200 + 7, nheads=2, headdim=64, dstate=32,
                               ngroups=1, chunk=64, dtype="bf16", init=True, dfinal=True,
                               seq_lengths=[5000, 1, 7806]),
    "fp32_many_segments": dict(batch=1, seqlen=32 * 150, nheads=2, headdim=16, dstate=16,
                               ngroups=1, chunk=32, dtype="f32", init=True, dfinal=True),
    # sequence starts on chunk boundaries, a one-token sequence, a ragged end
    "bf16_chunk_aligned_resets": dict(batch=2, seqlen=128 * 5 + 17, nheads=4, headdim=64,
                                      dstate=128, ngroups=1, chunk=128, dtype="bf16", init=True,
                                      dfinal=True, seq_lengths=[128, 256, 1, 127, 128, 17]),
    # chunk 32: tensor-core chunk states next to the CUDA-core scan and backward
    # two chunks, and exactly four (every x tile of the single-pass forward
    # used once, no refill)
    "bf16_two_chunks": dict(batch=1, seqlen=200, nheads=2, headdim=64, dstate=128, ngroups=1,
                            chunk=128, dtype="bf16", init=True),
    "bf16_four_chunks_exact": dict(batch=2, seqlen=512, nheads=2, headdim=64, dstate=64, ngroups=2,
                                   chunk=128, dtype="bf16", dfinal=True),
    "bf16_Q32_mixed": dict(batch=1, seqlen=32 * 9 + 11, nheads=4, headdim=64, dstate=64,
                           ngroups=2, chunk=32, dtype="bf16", init=True, dfinal=True,
                           seq_lengths=[100, 199]),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    inp = make_inputs(seed=3, **SMALL[name])
    _, got = run_device(inp)
    ref = oracle_full(inp)
    assert_close(got, ref, inp.dtype)


# tensor-core backward: one to eight heads per group, sequence starts on
# chunk boundaries and inside chunks, d_state 16 to 128
FEW_CTAS = ["bf16_N16_Q64", "bf16_Q256_init", "bf16_chunk_aligned_resets", "bf16_N64_G4_varlen"]


@pytest.mark.parametrize("name", FEW_CTAS)
def test_persistent_kernels_walk_several_units(name):
    """The persistent token-gradient kernel on two CTAs (SSD_TEST_FEW_CTAS),
    so that each CTA of a small problem walks several work units in turn (the
    copies and products of one unit's first head overlapping the previous
    unit's last heads): the same bits as with one CTA per unit, and the
    oracle's values."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=5, **SMALL[name])
    _, one = run_device(inp)
    _, few = run_device(inp, extra_flags=_lib.SSD_TEST_FEW_CTAS)
    for k in one:
        assert torch.equal(one[k], few[k]), k
    assert_close(few, oracle_full(inp), inp.dtype)


# the multi-kernel path's forward scan with its segments' local scans across
# lanes (warp-shuffle Hillis-Steele steps) instead of inside each thread
SHUFFLE_SCAN = ["bf16_many_segments", "fp32_many_segments", "bf16_chunk_aligned_resets",
                "fp32_ragged_init_resets"]


@pytest.mark.parametrize("name", SHUFFLE_SCAN)
def test_warp_shuffle_scan_variant(name):
    """SSD_SCAN_WARP_SHUFFLE: the same layer to rounding, against the oracle
    and against the sequential in-thread scan on the same path."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=7, **SMALL[name])
    multi = _lib.SSD_PATH_MULTI_KERNEL
    _, seq = run_device(inp, extra_flags=multi)
    _, shf = run_device(inp, extra_flags=multi | _lib.SSD_SCAN_WARP_SHUFFLE)
    assert_close(shf, oracle_full(inp), inp.dtype)
    assert_close(shf, {k: v.numpy() for k, v in seq.items()}, inp.dtype)


# bf16, headdim 64, d_state 64 or 128: the single-pass forward's shape set
SINGLE_PASS = ["bf16_N128_G2", "bf16_N64_G4_varlen", "bf16_Q256_init", "bf16_single_token",
               "bf16_shorter_than_chunk", "bf16_Q32_mixed", "bf16_chunk_aligned_resets", "bf16_two_chunks",
               "bf16_four_chunks_exact"]


@pytest.mark.parametrize("name", SINGLE_PASS)
def test_small_parity_single_pass(name):
    """The single-pass forward (forced on these small problems, which by
    default take the separate kernels) against the oracle."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=3, **SMALL[name])
    _, got = run_device(inp, extra_flags=_lib.SSD_PATH_SINGLE_PASS)
    assert_close(got, oracle_full(inp), inp.dtype)


def test_single_pass_is_deterministic_and_matches_multi_kernel():
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.runner import SSDDevice
    inp = make_inputs(seed=9, **SMALL["bf16_N64_G4_varlen"])
    dev = SSDDevice(inp, device="cuda", backward=False, extra_flags=_lib.SSD_PATH_SINGLE_PASS)
    dev.fwd()
    torch.cuda.synchronize()
    y0, f0 = dev.y.clone(), dev.final.clone()
    dev.fwd()
    torch.cuda.synchronize()
    assert torch.equal(dev.y, y0) and torch.equal(dev.final, f0)
    multi = SSDDevice(inp, device="cuda", backward=False, extra_flags=_lib.SSD_PATH_MULTI_KERNEL)
    multi.fwd()
    torch.cuda.synchronize()
    d = (multi.y.float() - y0.float()).abs().max() / y0.float().abs().max()
    assert float(d) <= 2e-2


def test_single_pass_positive_decay_rate():
    """A head with A > 0 (a growing state) takes the exact exponential for
    every entry of the mask (the split decay needs l nonincreasing)."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=4, **SMALL["bf16_N128_G2"])
    inp.A = inp.A.clone()
    inp.A[1] = 0.01
    _, got = run_device(inp, extra_flags=_lib.SSD_PATH_SINGLE_PASS)
    assert_close(got, oracle_full(inp), inp.dtype)


# shapes of the single-pass forward and the state chains, where the backward
# takes the intermediates the forward kept
KEPT = ["bf16_N128_G2", "bf16_N64_G4_varlen", "bf16_chunk_aligned_resets", "bf16_four_chunks_exact",
        "bf16_shorter_than_chunk"]


@pytest.mark.parametrize("name", KEPT)
def test_kept_forward_intermediates(name):
    """Forward with SSD_KEEP_FWD_STATES, then the backward that takes its
    dt_eff, chunk cumsums, decays and carry-in states instead of recomputing
    them: against the oracle, and against the recomputing backward."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=12, **SMALL[name])
    sp = _lib.SSD_PATH_SINGLE_PASS
    _, kept = run_device(inp, extra_flags=sp | _lib.SSD_KEEP_FWD_STATES)
    assert_close(kept, oracle_full(inp), inp.dtype)
    _, rec = run_device(inp, extra_flags=sp)
    # the forward does not depend on the flag; the gradients agree to rounding
    assert torch.equal(kept["y"], rec["y"]) and torch.equal(kept["final_states"], rec["final_states"])
    for k in kept:
        scale = float(rec[k].abs().max()) or 1.0
        assert float((kept[k] - rec[k]).abs().max()) <= 1e-2 * scale, k


# shapes of the separate kernels: CUDA-core fp32, tensor-core bf16 at d_state
# 16 and 128, chunk 64 and 256, and a scan over many segments and checkpoints
KEPT_MK = ["tiny_fp32", "fp32_ragged_init_resets", "bf16_N16_Q64", "bf16_N128_G2",
           "bf16_many_segments", "bf16_Q256_init"]


@pytest.mark.parametrize("name", KEPT_MK)
def test_kept_forward_intermediates_on_the_multi_kernel_path(name):
    """On the separate kernels the forward keeps dt_eff, the chunk cumsums
    and decays and the carry-in states (bf16 and fp32; its scan writes the
    fp32 ones over the chunk states), and the backward takes them instead of
    recomputing: against the oracle, and bit for bit against the recomputing
    backward, which runs the same deterministic kernels on the same inputs."""
    from mamba_selective_state_gb300 import _lib
    mk = _lib.SSD_PATH_MULTI_KERNEL
    inp = make_inputs(seed=13, **SMALL[name])
    _, kept = run_device(inp, extra_flags=mk | _lib.SSD_KEEP_FWD_STATES)
    assert_close(kept, oracle_full(inp), inp.dtype)
    _, rec = run_device(inp, extra_flags=mk)
    for k in kept:
        assert torch.equal(kept[k], rec[k]), k


def test_kept_multi_kernel_backward_runs_twice():
    """Two backwards after one kept forward: the second finds the reverse
    scan's flags and ticket reset (no forward recompute resets them there)
    and gives the same bits."""
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=15, **SMALL["bf16_many_segments"])
    dev, a = run_device(inp, extra_flags=_lib.SSD_PATH_MULTI_KERNEL | _lib.SSD_KEEP_FWD_STATES)
    for _ in range(2):
        dev.bwd()
        torch.cuda.synchronize()
        assert dev.device_status() == 0
        b = dev.results()
        for k in a:
            assert torch.equal(a[k], b[k]), k


def test_kept_stamp_tells_which_forward_kept():
    """The separate-kernel backward needs the fp32 carry-in states that only
    the separate-kernel forward keeps: after a single-pass forward, or a
    forward that keeps nothing, it reports SSD_ERR_NO_KEPT_STATES.  The
    state-chain backward takes the intermediates of either forward."""
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.runner import SSDDevice
    keep, mk, sp = _lib.SSD_KEEP_FWD_STATES, _lib.SSD_PATH_MULTI_KERNEL, _lib.SSD_PATH_SINGLE_PASS
    inp = make_inputs(seed=16, **SMALL["bf16_N128_G2"])
    dev = SSDDevice(inp, device="cuda", extra_flags=mk | keep)
    base_f, base_b = dev.fwd_prob.flags & ~(mk | keep), dev.bwd_prob.flags & ~(mk | keep)
    for fwd_flags in (sp | keep, mk):
        dev.fwd_prob.flags = base_f | fwd_flags
        dev.fwd()
        dev.bwd()
        torch.cuda.synchronize()
        assert dev.device_status() == _lib.SSD_ERR_NO_KEPT_STATES, fwd_flags
    # separate-kernel forward, state-chain backward
    dev.fwd_prob.flags = base_f | mk | keep
    dev.bwd_prob.flags = base_b | sp | keep
    dev.fwd()
    dev.bwd()
    torch.cuda.synchronize()
    assert dev.device_status() == 0
    assert_close(dev.results(), oracle_full(inp), inp.dtype)


def test_missing_kept_intermediates_are_reported():
    """A backward told to take the forward's intermediates from a workspace
    whose last forward did not keep them reports SSD_ERR_NO_KEPT_STATES in
    the status word; the next kept forward and backward are clean again."""
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.runner import SSDDevice
    inp = make_inputs(seed=14, **SMALL["bf16_N64_G4_varlen"])
    flags = _lib.SSD_PATH_SINGLE_PASS | _lib.SSD_KEEP_FWD_STATES
    dev = SSDDevice(inp, device="cuda", extra_flags=flags)
    dev.fwd_prob.flags &= ~_lib.SSD_KEEP_FWD_STATES   # a forward that keeps nothing
    dev.fwd()
    dev.fwd_prob.flags |= _lib.SSD_KEEP_FWD_STATES
    dev.bwd()
    torch.cuda.synchronize()
    assert dev.device_status() == _lib.SSD_ERR_NO_KEPT_STATES
    assert "kept" in _lib.status_string(_lib.SSD_ERR_NO_KEPT_STATES)
    dev.fwd()
    dev.bwd()
    torch.cuda.synchronize()
    assert dev.device_status() == 0


def test_null_init_equals_zero_init():
    cfg = dict(SMALL["bf16_N128_G2"])
    cfg["init"] = False
    inp = make_inputs(seed=5, **cfg)
    _, got0 = run_device(inp)
    inp.initial_states = torch.zeros((inp.batch, inp.nheads, inp.headdim, inp.dstate))
    _, got1 = run_device(inp, want_dinit=False)
    for k in got0:
        assert torch.equal(got0[k], got1[k]), k


@pytest.mark.parametrize("single_pass", [False, True])
def test_backward_is_bitwise_deterministic(single_pass):
    from mamba_selective_state_gb300 import _lib
    inp = make_inputs(seed=7, **SMALL["bf16_N64_G4_varlen"])
    dev, a = run_device(inp, extra_flags=_lib.SSD_PATH_SINGLE_PASS if single_pass else 0)
    dev.fwd()
    dev.bwd()
    torch.cuda.synchronize()
    b = dev.results()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_scan_across_checkpoints_is_bitwise_deterministic():
    """The scan's look-back folds the published segment aggregates in a fixed
    order, so repeated calls give the same bits whichever tiles finish first."""
    inp = make_inputs(seed=11, **SMALL["bf16_many_segments"])
    dev, a = run_device(inp)
    for _ in range(3):
        dev.fwd()
        dev.bwd()
        torch.cuda.synchronize()
        assert dev.device_status() == 0
        b = dev.results()
        for k in a:
            assert torch.equal(a[k], b[k]), k


def test_scan_wait_timeout_is_reported_not_hung():
    """A scan tile that never publishes makes its successors exhaust their
    bounded wait: the call completes and the status word says TIMEOUT; the
    next normal call on the same context is fine."""
    from mamba_selective_state_gb300 import _lib
    cfg = dict(SMALL["bf16_many_chunks"])
    inp = make_inputs(seed=1, **cfg)
    from mamba_selective_state_gb300.runner import SSDDevice
    dev = SSDDevice(inp, device="cuda", backward=False,
                    extra_flags=_lib.SSD_TEST_DROP_SCAN_PUBLISH)
    dev.fwd()
    assert dev.device_status() == _lib.SSD_ERR_TIMEOUT
    _, got = run_device(inp)
    assert_close(got, oracle_full(inp), inp.dtype)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload_sampled_group(name):
    inp = make_workload(name, seed=0, dfinal=False)
    _, got = run_device(inp)
    if inp.ngroups == 1 and inp.nheads * inp.seqlen * inp.batch <= 4 * 256 * 64:
        ref = oracle_full(inp)
        assert_close(got, ref, inp.dtype)
        return
    g = int(np.random.default_rng(0).integers(inp.ngroups))
    ref = oracle_group(inp, g)
    assert_close(slice_group(got, inp, g), ref, inp.dtype)
