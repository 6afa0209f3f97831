"""Thin ctypes binding over libssd (include/ssd.h): the same entry points,
argument marshalling only.  Every step of the layer runs in the library's
CUDA kernels; there is no fallback of any kind -- if libssd.so is missing or
does not load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd.so")

SSD_OK = 0
SSD_ERR_INVALID_ARGUMENT = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_WORKSPACE_TOO_SMALL = 3
SSD_ERR_CUDA = 4
SSD_ERR_TIMEOUT = 5
SSD_ERR_NO_KEPT_STATES = 6
SSD_F32 = 0
SSD_BF16 = 1
SSD_HAS_INIT = 1
SSD_HAS_SEQ_IDX = 2
SSD_HAS_DFINAL = 4
SSD_WANT_DINIT = 8
SSD_KEEP_FWD_STATES = 16
SSD_TEST_DROP_SCAN_PUBLISH = 1 << 16
SSD_PATH_MULTI_KERNEL = 1 << 17
SSD_PATH_SINGLE_PASS = 1 << 18
SSD_TEST_FEW_CTAS = 1 << 19
SSD_SCAN_WARP_SHUFFLE = 1 << 20
SSD_NORM_HAS_Z = 1

# every symbol include/ssd.h declares
EXPORTS = ["ssd_fwd_workspace_bytes", "ssd_bwd_workspace_bytes", "ssd_fwd", "ssd_bwd",
           "ssd_status_string", "ssd_read_device_status", "ssd_version", "ssd_profile_start",
           "ssd_profile_stop", "ssd_profile_count", "ssd_profile_get", "ssd_fwd_noalloc",
           "ssd_fwd_noalloc_read_device_status", "ssd_shard_decay", "ssd_shard_fold",
           "ssd_gated_rmsnorm_fwd", "ssd_gated_rmsnorm_bwd_workspace_bytes",
           "ssd_gated_rmsnorm_bwd"]
SSD_NOALLOC_SCRATCH_BYTES = 32 << 20


class ssd_problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class ssd_norm_problem(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("group_size", ctypes.c_int64), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class SSDError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssd.so not built at {LIB_PATH}; run "
                          "`python -m mamba_selective_state_gb300.build_ext`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pp = ctypes.POINTER(ssd_problem)
    lib.ssd_fwd_workspace_bytes.argtypes = [pp]
    lib.ssd_fwd_workspace_bytes.restype = sz
    lib.ssd_bwd_workspace_bytes.argtypes = [pp]
    lib.ssd_bwd_workspace_bytes.restype = sz
    lib.ssd_fwd.argtypes = [pp] + [vp] * 11 + [vp, sz, vp]
    lib.ssd_fwd.restype = i32
    lib.ssd_bwd.argtypes = [pp] + [vp] * 19 + [vp, sz, vp]
    lib.ssd_bwd.restype = i32
    lib.ssd_status_string.argtypes = [i32]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_read_device_status.argtypes = [vp, vp]
    lib.ssd_read_device_status.restype = i32
    lib.ssd_version.restype = ctypes.c_char_p
    lib.ssd_profile_start.restype = i32
    lib.ssd_profile_stop.restype = i32
    lib.ssd_profile_count.restype = i32
    lib.ssd_profile_get.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p),
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
    lib.ssd_profile_get.restype = i32
    lib.ssd_fwd_noalloc.argtypes = [pp] + [vp] * 11 + [vp]
    lib.ssd_fwd_noalloc.restype = i32
    lib.ssd_fwd_noalloc_read_device_status.argtypes = [vp]
    lib.ssd_fwd_noalloc_read_device_status.restype = i32
    lib.ssd_shard_decay.argtypes = [pp] + [vp] * 7 + [vp]
    lib.ssd_shard_decay.restype = i32
    i64 = ctypes.c_int64
    lib.ssd_shard_fold.argtypes = [i64] * 5 + [vp] * 7 + [i32, vp]
    lib.ssd_shard_fold.restype = i32
    npp = ctypes.POINTER(ssd_norm_problem)
    lib.ssd_gated_rmsnorm_fwd.argtypes = [npp] + [vp] * 5 + [vp]
    lib.ssd_gated_rmsnorm_fwd.restype = i32
    lib.ssd_gated_rmsnorm_bwd_workspace_bytes.argtypes = [npp]
    lib.ssd_gated_rmsnorm_bwd_workspace_bytes.restype = sz
    lib.ssd_gated_rmsnorm_bwd.argtypes = [npp] + [vp] * 8 + [sz, vp]
    lib.ssd_gated_rmsnorm_bwd.restype = i32
    return lib


LIB = _load()


def status_string(code: int) -> str:
    return LIB.ssd_status_string(int(code)).decode()


def version() -> str:
    return LIB.ssd_version().decode()


def make_problem(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype,
                 flags=0) -> ssd_problem:
    if isinstance(dtype, torch.dtype):
        dtype = SSD_BF16 if dtype == torch.bfloat16 else SSD_F32
    return ssd_problem(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype, flags)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ssd_fwd_workspace_bytes(prob: ssd_problem) -> int:
    return int(LIB.ssd_fwd_workspace_bytes(ctypes.byref(prob)))


def ssd_bwd_workspace_bytes(prob: ssd_problem) -> int:
    return int(LIB.ssd_bwd_workspace_bytes(ctypes.byref(prob)))


def ssd_fwd(prob, x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, y, final_states,
            workspace, workspace_bytes=None, stream=None, check=True) -> int:
    """Enqueue the forward on ``stream`` (default: torch's current stream).
    Tensor arguments may also be raw device addresses (ints)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = LIB.ssd_fwd(ctypes.byref(prob), _p(x), _p(dt), _p(dt_bias), _p(A), _p(B), _p(C), _p(D),
                     _p(initial_states), _p(seq_idx), _p(y), _p(final_states), _p(workspace),
                     workspace_bytes, _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_fwd")
    return rc


def ssd_bwd(prob, x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, dy, dfinal_states,
            dx, ddt, ddt_bias, dA, dB, dC, dD, dinitial_states, workspace,
            workspace_bytes=None, stream=None, check=True) -> int:
    """Enqueue the backward on ``stream`` (default: torch's current stream)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = LIB.ssd_bwd(ctypes.byref(prob), _p(x), _p(dt), _p(dt_bias), _p(A), _p(B), _p(C), _p(D),
                     _p(initial_states), _p(seq_idx), _p(dy), _p(dfinal_states), _p(dx), _p(ddt),
                     _p(ddt_bias), _p(dA), _p(dB), _p(dC), _p(dD), _p(dinitial_states),
                     _p(workspace), workspace_bytes, _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_bwd")
    return rc


def ssd_read_device_status(workspace, stream=None) -> int:
    return int(LIB.ssd_read_device_status(_p(workspace), _stream(stream)))


def profile_start() -> None:
    rc = LIB.ssd_profile_start()
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_profile_start")


def profile_stop() -> dict:
    """Stop per-kernel timing; returns {kernel name: (launches, total ms)}."""
    rc = LIB.ssd_profile_stop()
    if rc not in (SSD_OK, SSD_ERR_WORKSPACE_TOO_SMALL):
        raise SSDError(rc, "ssd_profile_stop")
    out = {}
    for i in range(LIB.ssd_profile_count()):
        name, n, ms = ctypes.c_char_p(), ctypes.c_int(), ctypes.c_double()
        if LIB.ssd_profile_get(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms)) == SSD_OK:
            out[name.value.decode()] = (int(n.value), float(ms.value))
    if rc == SSD_ERR_WORKSPACE_TOO_SMALL:
        out["_dropped"] = (1, 0.0)
    return out


def ssd_fwd_noalloc(prob, x, dt, dt_bias, A, B, C, D, initial_states, seq_idx, y, final_states,
                    stream=None) -> int:
    """Forward with the library-owned workspace (no workspace argument, no
    allocation); returns the status code."""
    return int(LIB.ssd_fwd_noalloc(ctypes.byref(prob), _p(x), _p(dt), _p(dt_bias), _p(A), _p(B),
                                   _p(C), _p(D), _p(initial_states), _p(seq_idx), _p(y),
                                   _p(final_states), _stream(stream)))


def ssd_fwd_noalloc_read_device_status(stream=None) -> int:
    """Device status word of the last ssd_fwd_noalloc call (synchronises)."""
    return int(LIB.ssd_fwd_noalloc_read_device_status(_stream(stream)))


def ssd_shard_decay(prob, dt, dt_bias, A, seq_idx, decay, first_ids=None, last_ids=None,
                    stream=None, check=True) -> int:
    """One shard's decay (b, H) and the segment ids of its first and last tokens."""
    rc = LIB.ssd_shard_decay(ctypes.byref(prob), _p(dt), _p(dt_bias), _p(A), _p(seq_idx), _p(decay),
                             _p(first_ids), _p(last_ids), _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_shard_decay")
    return rc


def ssd_shard_fold(decay, local, first_ids, last_ids, boundary, out, total=None, reverse=False,
                   stream=None, check=True) -> int:
    """The exclusive fold over the shards (forward or from the right);
    shapes are read from ``local`` (R, b, H, P, N)."""
    R, b, H, P, N = local.shape
    rc = LIB.ssd_shard_fold(R, b, H, P, N, _p(decay), _p(local), _p(first_ids), _p(last_ids),
                            _p(boundary), _p(out), _p(total), int(bool(reverse)), _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_shard_fold")
    return rc


def make_norm_problem(rows, dim, group_size, eps, dtype, gate=True) -> ssd_norm_problem:
    if isinstance(dtype, torch.dtype):
        dtype = SSD_BF16 if dtype == torch.bfloat16 else SSD_F32
    return ssd_norm_problem(rows, dim, group_size, eps, dtype, SSD_NORM_HAS_Z if gate else 0)


def ssd_gated_rmsnorm_bwd_workspace_bytes(prob: ssd_norm_problem) -> int:
    return int(LIB.ssd_gated_rmsnorm_bwd_workspace_bytes(ctypes.byref(prob)))


def ssd_gated_rmsnorm_fwd(prob, y, z, weight, out, rstd=None, stream=None, check=True) -> int:
    """Enqueue the gated RMSNorm forward on ``stream`` (default: torch's
    current stream)."""
    rc = LIB.ssd_gated_rmsnorm_fwd(ctypes.byref(prob), _p(y), _p(z), _p(weight), _p(out),
                                   _p(rstd), _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_gated_rmsnorm_fwd")
    return rc


def ssd_gated_rmsnorm_bwd(prob, y, z, weight, dout, dy, dz, dweight, workspace,
                          workspace_bytes=None, stream=None, check=True) -> int:
    """Enqueue the gated RMSNorm backward on ``stream``."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = LIB.ssd_gated_rmsnorm_bwd(ctypes.byref(prob), _p(y), _p(z), _p(weight), _p(dout),
                                   _p(dy), _p(dz), _p(dweight), _p(workspace), workspace_bytes,
                                   _stream(stream))
    if check and rc != SSD_OK:
        raise SSDError(rc, "ssd_gated_rmsnorm_bwd")
    return rc
