"""ctypes wrapper over the float64 C oracle (``ssd_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).  The shared library is
built with gcc on first use (or by ``build_oracle()``) next to the source.

Inputs are numpy arrays; they are converted to contiguous float64 (seq_idx to
int32).  Layouts: x, dy (b,L,H,P); dt (b,L,H); B, C (b,L,G,N); states
(b,H,P,N); seq_idx (b,L); A, D, dt_bias (H).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile ssd_oracle.c into libssd_oracle.so (portable flags, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    L = ctypes.c_long
    lib.oracle_ssd_fwd.argtypes = [L] * 6 + [dp] * 7 + [dp, ip, dp, dp]
    lib.oracle_ssd_fwd.restype = ctypes.c_int
    lib.oracle_ssd_bwd.argtypes = [L] * 6 + [dp] * 7 + [dp, ip, dp, dp] + [dp] * 8
    lib.oracle_ssd_bwd.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_last_threads.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


def load_library(path):
    """Load another build of the oracle source (used by the tests that plant
    mistakes in a copy of it); returns an object with ``ssd_fwd``/``ssd_bwd``."""
    lib = _configure(ctypes.CDLL(path))

    class _Variant:
        def ssd_fwd(self, *a, **k):
            return ssd_fwd(*a, _lib_override=lib, **k)

        def ssd_bwd(self, *a, **k):
            return ssd_bwd(*a, _lib_override=lib, **k)
    return _Variant()


def set_threads(n: int) -> None:
    """Cap the OpenMP threads the oracle uses (0 = all available)."""
    _load().oracle_set_threads(int(n))


def last_threads() -> int:
    """Threads the most recent oracle call actually ran on."""
    return int(_load().oracle_last_threads())


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    if a.dtype == np.int32:
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(x, B):
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return b, L, H, P, N, G


def ssd_fwd(x, dt, dt_bias, A, B, C, D, initial_states=None, seq_idx=None,
            _lib_override=None):
    """Sequential float64 forward.  Returns (y, final_states)."""
    lib = _lib_override or _load()
    x, dt, dt_bias, A, B, C, D = map(_f64, (x, dt, dt_bias, A, B, C, D))
    init = _f64(initial_states)
    seq = None if seq_idx is None else np.ascontiguousarray(seq_idx, dtype=np.int32)
    b, L, H, P, N, G = _dims(x, B)
    y = np.empty((b, L, H, P))
    fin = np.empty((b, H, P, N))
    rc = lib.oracle_ssd_fwd(b, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A),
                            _ptr(B), _ptr(C), _ptr(D), _ptr(init), _ptr(seq),
                            _ptr(y), _ptr(fin))
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_fwd failed with code {rc}")
    return y, fin


def ssd_bwd(x, dt, dt_bias, A, B, C, D, dy, initial_states=None, seq_idx=None,
            dfinal_states=None, want_dinit=True, _lib_override=None):
    """Hand-derived reverse mode in float64.  Returns a dict of gradients:
    dx, ddt, ddt_bias, dA, dB, dC, dD and (if want_dinit) dinitial_states."""
    lib = _lib_override or _load()
    x, dt, dt_bias, A, B, C, D, dy = map(_f64, (x, dt, dt_bias, A, B, C, D, dy))
    init, dfin = _f64(initial_states), _f64(dfinal_states)
    seq = None if seq_idx is None else np.ascontiguousarray(seq_idx, dtype=np.int32)
    b, L, H, P, N, G = _dims(x, B)
    out = dict(dx=np.empty((b, L, H, P)), ddt=np.empty((b, L, H)),
               ddt_bias=np.empty(H), dA=np.empty(H), dB=np.empty((b, L, G, N)),
               dC=np.empty((b, L, G, N)), dD=np.empty(H))
    dinit = np.empty((b, H, P, N)) if want_dinit else None
    rc = lib.oracle_ssd_bwd(b, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(dt_bias), _ptr(A),
                            _ptr(B), _ptr(C), _ptr(D), _ptr(init), _ptr(seq), _ptr(dy),
                            _ptr(dfin), _ptr(out["dx"]), _ptr(out["ddt"]),
                            _ptr(out["ddt_bias"]), _ptr(out["dA"]), _ptr(out["dB"]),
                            _ptr(out["dC"]), _ptr(out["dD"]), _ptr(dinit))
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_bwd failed with code {rc}")
    if want_dinit:
        out["dinitial_states"] = dinit
    return out


def ssd_group(x, dt, dt_bias, A, B, C, D, dy, g, ngroups, initial_states=None, seq_idx=None,
              dfinal_states=None, want_dinit=True):
    """Forward and backward restricted to group ``g`` of ``ngroups`` (every
    batch row, the group's contiguous block of heads, every token).  Each
    head runs as its own group with a copy of the group's B and C (so the
    oracle's threads spread over the heads); dB and dC of the group are then
    the sums of the per-head results in head order.  Returns a dict with y,
    final_states and the gradients, restricted the same way (dB, dC with a
    group axis of length 1)."""
    H = x.shape[2]
    hpg = H // ngroups
    hs = slice(g * hpg, (g + 1) * hpg)
    Bg = np.repeat(np.asarray(B)[:, :, g:g + 1, :], hpg, axis=2)
    Cg = np.repeat(np.asarray(C)[:, :, g:g + 1, :], hpg, axis=2)
    init_s = None if initial_states is None else np.asarray(initial_states)[:, hs]
    dfin_s = None if dfinal_states is None else np.asarray(dfinal_states)[:, hs]
    args = [np.asarray(x)[:, :, hs], np.asarray(dt)[:, :, hs], np.asarray(dt_bias)[hs],
            np.asarray(A)[hs], Bg, Cg, np.asarray(D)[hs]]
    y, fin = ssd_fwd(*args, initial_states=init_s, seq_idx=seq_idx)
    gr = ssd_bwd(*args, np.asarray(dy)[:, :, hs], initial_states=init_s, seq_idx=seq_idx,
                 dfinal_states=dfin_s, want_dinit=want_dinit)
    dB = np.zeros_like(gr["dB"][:, :, :1])
    dC = np.zeros_like(dB)
    for k in range(hpg):
        dB[:, :, 0] += gr["dB"][:, :, k]
        dC[:, :, 0] += gr["dC"][:, :, k]
    out = dict(y=y, final_states=fin, dx=gr["dx"], ddt=gr["ddt"], ddt_bias=gr["ddt_bias"],
               dA=gr["dA"], dD=gr["dD"], dB=dB, dC=dC)
    if want_dinit:
        out["dinitial_states"] = gr["dinitial_states"]
    return out


def inputs_f64(inp):
    """Pull the float64 views the oracle needs out of an ``SSDInputs``-like
    object (duck-typed: anything with ``f64(name)``)."""
    names = ["x", "dt", "dt_bias", "A", "B", "C", "D", "initial_states",
             "seq_idx", "dy", "dfinal_states"]
    return {n: inp.f64(n) for n in names}
