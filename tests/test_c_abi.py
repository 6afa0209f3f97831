"""The boundary seen from C (CPU only): a C99 program compiled against
include/ssd.h and linked with libssd.so agrees with the ctypes binding on
the layout of the ABI's structs, the workspace sizes and the status codes of
rejected calls."""
import ctypes
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE = os.path.join(ROOT, "tests", "c_abi_probe.c")


@pytest.fixture(scope="module")
def lib():
    from mamba_selective_state_gb300 import build_ext
    build_ext.build()
    from mamba_selective_state_gb300 import _lib
    return _lib


def _cuda_lib_dirs():
    dirs = []
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
              "/usr/local/cuda/targets/x86_64-linux/lib"):
        if os.path.isdir(d):
            dirs.append(d)
    return dirs


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++11")])
def test_c_consumer_agrees_with_binding(lib, tmp_path, compiler, std):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    exe = tmp_path / "probe"
    src = PROBE
    if compiler == "g++":  # the header must also be usable from C++
        src = str(tmp_path / "probe.cc")
        shutil.copy(PROBE, src)
    pkg = os.path.dirname(lib.LIB_PATH)
    cmd = [compiler, std, "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o",
           str(exe), "-L", pkg, "-lssd", f"-Wl,-rpath,{pkg}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="",
               LD_LIBRARY_PATH=":".join(_cuda_lib_dirs() + [os.environ.get("LD_LIBRARY_PATH", "")]))
    out = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0, out.stderr
    d = json.loads(out.stdout)
    P, NP = lib.ssd_problem, lib.ssd_norm_problem
    assert d["sizeof_problem"] == ctypes.sizeof(P)
    assert d["off_chunk"] == P.chunk_size.offset and d["off_dtype"] == P.dtype.offset
    assert d["off_flags"] == P.flags.offset
    assert d["sizeof_norm"] == ctypes.sizeof(NP)
    assert d["off_eps"] == NP.eps.offset and d["off_ndtype"] == NP.dtype.offset
    assert d["off_nflags"] == NP.flags.offset
    p = lib.make_problem(2, 300, 8, 64, 128, 2, 128, lib.SSD_BF16)
    assert d["fwd_ws"] == lib.ssd_fwd_workspace_bytes(p) > 0
    assert d["bwd_ws"] == lib.ssd_bwd_workspace_bytes(p) > d["fwd_ws"]
    assert d["bad_ws"] == 0
    np_ = lib.make_norm_problem(300, 4096, 512, 1e-5, lib.SSD_BF16, gate=True)
    assert d["norm_ws"] == lib.ssd_gated_rmsnorm_bwd_workspace_bytes(np_) > 0
    assert d["fwd_null_x"] == lib.SSD_ERR_INVALID_ARGUMENT
    assert d["fwd_small_ws"] == lib.SSD_ERR_WORKSPACE_TOO_SMALL
    assert d["norm_no_z"] == lib.SSD_ERR_INVALID_ARGUMENT
    assert d["status_ok"] == "ok" and d["version"] == lib.version()
