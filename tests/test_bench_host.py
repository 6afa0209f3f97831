"""Host-side logic of bench.py (CPU only): the algorithmic byte model, the
guard on the recorded DRAM traffic, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_kernel_model_counts_compulsory_bytes():
    cfg = dict(batch=2, seqlen=300, nheads=4, headdim=16, dstate=8, ngroups=2, chunk=64)
    m, layer_io = bench.kernel_model(cfg, 2)
    T, nc = 2 * 300, 5
    tokx, tokbc = T * 4 * 16 * 2, T * 2 * 8 * 2
    st32 = 2 * 4 * nc * 16 * 8 * 4
    per_tok = 2 * 4 * nc * 64 * 4
    # chunk_scan reads x, B, C, the carry-in states, l and dt, writes y
    assert m["chunk_scan"]["bytes"] == 2 * tokx + 2 * tokbc + st32 // 2 + 2 * per_tok
    # forward scan: fp32 chunk states in, carry-in states out in the dtype
    assert m["state_passing_fwd"]["bytes"] == st32 + st32 // 2
    # reverse scan: dHloc and the fp32 carry-in states in, dS out
    assert m["state_passing_bwd"]["bytes"] == 2 * st32 + st32 // 2
    # a kept backward on the separate kernels zeroes one scan flag per (row,
    # head, 512-element state block, scan segment: 16 chunks forward, 8 in
    # reverse) -- here 2 x 4 x 1 x 1 -- and writes the status word
    assert m["kept_scan_reset"]["bytes"] == 4 * 8 + 4
    # the layer's own inputs and outputs, forward plus backward
    assert layer_io == (2 * tokx + T * 4 * 2 + 2 * tokbc) + (3 * tokx + 2 * T * 4 * 2 + 4 * tokbc)


def test_recorded_traffic_only_for_unchanged_sources(monkeypatch):
    name = "chunk_bwd_tc"
    files, nbytes, sha = bench.NCU_TRAFFIC[name]
    # the figure belongs to one workload
    assert bench.ncu_traffic(name, "tiny_fp32") is None
    assert bench.ncu_traffic("no_such_kernel", bench.NCU_TRAFFIC_WORKLOAD) is None
    # a different source hash (the kernel changed since the capture) -> null
    monkeypatch.setitem(bench.NCU_TRAFFIC, name, (files, nbytes, "0" * 40))
    assert bench.ncu_traffic(name, bench.NCU_TRAFFIC_WORKLOAD) is None


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--workload", "tiny_fp32"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_fp32"


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_other_ranks_exit_without_work(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=rank)
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--workload", "tiny_fp32"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]


def test_norm_model_counts_compulsory_bytes():
    rows, dim, G = 100, 64, 4
    m = bench.norm_model(rows, dim, G, True, 2)
    e = rows * dim * 2
    # forward: y, z in; out, rstd out; weight once
    assert m["gated_norm_fwd"]["bytes"] == 3 * e + rows * G * 4 + dim * 4
    # backward: y, z, dout in; dy, dz out; weight in, dweight out
    assert m["gated_norm_bwd"]["bytes"] == 5 * e + 2 * dim * 4
    m1 = bench.norm_model(rows, dim, G, False, 4)
    assert m1["gated_norm_bwd"]["bytes"] == 3 * rows * dim * 4 + 2 * dim * 4


def test_norm_reference_arm_prints_one_contract_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--op",
                          "gated_rmsnorm", "--steps", "1", "--warmup", "3", "--workload",
                          "tiny_fp32"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["op"] == "gated_rmsnorm" and d["value"] > 0
    assert d["config"]["rows"] == 256 and d["config"]["group_size"] == 64


def test_cpu_baseline_reports_all_cores_and_one_core():
    d = bench.cpu_baseline("tiny_fp32", target_s=0.3, min_s=0.2, single_core_s=0.1)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] >= 1
    one = d["single_core"]
    assert one["cores"] == 1 and one["value"] > 0 and "tokens" in one["sample"]


def test_layer_summary_against_both_roofs():
    model = {"chunk_state": dict(bytes=10, flops=1000), "dt_cumsum": dict(bytes=5, flops=0)}
    kernels = {"chunk_state_tc": {"launches": 4}, "dt_cumsum": {"launches": 4},
               "unknown": {"launches": 2}}
    d = bench.layer_summary(kernels, model, steps=2, ms_per_step=1.0, layer_io=2e9,
                            hbm_peak=4000.0, tc_peak=0.5)
    assert d["flops_per_step"] == 2000            # two chunk_state launches per step
    assert abs(d["achieved_GBps"] - 2000.0) < 1e-9 and abs(d["frac_of_hbm"] - 0.5) < 1e-12
    assert abs(d["achieved_TFLOPps"] - 2e-6) < 1e-18
    assert abs(d["frac_of_tensor"] - 4e-6) < 1e-18


def test_kernel_model_flops_match_a_hand_count():
    """One chunk of 128 tokens, two heads of one group, headdim 64, d_state
    32: the matrix products the two backward kernels issue, counted by hand
    (2 flops per multiply-add)."""
    cfg = dict(batch=1, seqlen=128, nheads=2, headdim=64, dstate=32, ngroups=1, chunk=128)
    m, _ = bench.kernel_model(cfg, 2)
    # token kernel: C B^T once (128x128x32), per head dy x^T (128x128x64),
    # B dS^T and C H^T (128x64x32 each), M^T dY (128x64x128)
    cb = 2 * 128 * 128 * 32
    per_head = 2 * 128 * 128 * 64 + 2 * (2 * 128 * 64 * 32) + 2 * 128 * 64 * 128
    assert m["chunk_bwd"]["flops"] == cb + 2 * per_head == 11534336
    # dB/dC kernel, per head: dy x^T, dy H and x dS (128x32x64 each); once
    # per group, on the heads' summed dCB: S B and S^T C (128x32x128 each)
    per_head = 2 * 128 * 128 * 64 + 2 * (2 * 128 * 32 * 64)
    per_group = 2 * (2 * 128 * 32 * 128)
    assert m["chunk_bwd_dbc"]["flops"] == 2 * per_head + per_group == 8388608
    # chunk_scan at chunk 128: C B^T and C_rev B^T once, per head A_hat X
    # (128x64x128) and C H^T (128x64x32)
    assert m["chunk_scan"]["flops"] == 2 * cb + 2 * (2 * 128 * 64 * 128 + 2 * 128 * 64 * 32)


def test_kernel_model_single_pass_forward_is_the_compulsory_io():
    """The single-pass forward's algorithmic bytes are exactly the forward's
    compulsory IO (x, dt, B, C in; y out) plus the two state tensors; the
    tensor-core path's evaluation chunk is 128 whatever chunk_size asks."""
    cfg = dict(batch=2, seqlen=1000, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=256)
    assert bench.eval_chunk(cfg, 2) == 128 and bench.eval_chunk(cfg, 4) == 256
    m, _ = bench.kernel_model(cfg, 2)
    T = 2 * 1000
    io = 2 * T * 8 * 64 * 2 + T * 8 * 2 + 2 * T * 2 * 128 * 2 + 2 * 2 * 8 * 64 * 128 * 4
    assert m["ssd_fwd_fused"]["bytes"] == io
    # per (row, head, 128-token chunk): C B^T, C H^T, S^T (128 rows issued), A_hat X
    per = 2 * 128 * 128 * 128 + 2 * 128 * 64 * 128 + 2 * 128 * 64 * 128 + 2 * 128 * 128 * 64
    assert m["ssd_fwd_fused"]["flops"] == 2 * 8 * 8 * per
