"""Seeded synthetic inputs for the Mamba-2 SSD layer (forward + backward).

This module only draws random numbers and rounds them to the storage dtype;
it holds none of the layer's arithmetic.  Both the CUDA path and the float64
oracle receive the *same* rounded values: the device gets the bf16/fp32
tensors, the oracle gets their exact float64 upcast.

Recipe (per workload; numpy PCG64 ``default_rng(seed)``, draw order fixed):

  [lengths (packed workloads only)], dt_target, A, x, dt, B, C, D,
  [initial_states], dy, [dfinal_states]

  x, dt, dy ~ N(0, 1)
  dt_bias_h = log(expm1(dt_target_h)),  dt_target_h = exp(U(ln 1e-3, ln 1e-1))
      (the bias centres softplus(dt + dt_bias) on dt_target_h)
  A_h = -exp(U(0, ln 16))
  B, C ~ N(0, 1) / sqrt(d_state)
  D ~ N(0, 1)
  initial_states ~ N(0, 0.1**2)   (only when requested)
  dfinal_states ~ N(0, 1)         (only when requested)

Packed variable-length rows draw ``nseq`` integer lengths uniform in
[min_len, max_len] and redraw the whole set until the sum is <= max_total;
seq_idx then holds the segment id of every token of the single row.

x, dt, B, C, dy are stored in the workload's dtype (bf16 by round-to-nearest-
even from fp32, or fp32); A, D, dt_bias, initial_states, dfinal_states are
always fp32; seq_idx is int32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# The five workloads of the layer benchmark, named by what they are.
WORKLOADS = {
    "tiny_fp32": dict(batch=1, seqlen=256, nheads=4, headdim=16, dstate=16,
                      ngroups=1, chunk=64, dtype="f32"),
    "b2_L8192_bf16": dict(batch=2, seqlen=8192, nheads=64, headdim=64,
                          dstate=128, ngroups=8, chunk=128, dtype="bf16"),
    "long_L65536_bf16": dict(batch=1, seqlen=65536, nheads=32, headdim=64,
                             dstate=128, ngroups=1, chunk=256, dtype="bf16",
                             init=True),
    "smallstate_N16_bf16": dict(batch=8, seqlen=4096, nheads=48, headdim=64,
                                dstate=16, ngroups=1, chunk=64, dtype="bf16"),
    "varlen_16seq_bf16": dict(nseq=16, min_len=256, max_len=4096,
                              max_total=32768, nheads=64, headdim=64,
                              dstate=64, ngroups=4, chunk=128, dtype="bf16"),
}


@dataclasses.dataclass
class SSDInputs:
    """One problem's inputs as CPU torch tensors in their storage dtypes."""
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str                      # "bf16" or "f32"
    x: torch.Tensor                 # (b, L, H, P)
    dt: torch.Tensor                # (b, L, H)
    dt_bias: torch.Tensor           # (H,) fp32
    A: torch.Tensor                 # (H,) fp32
    B: torch.Tensor                 # (b, L, G, N)
    C: torch.Tensor                 # (b, L, G, N)
    D: torch.Tensor                 # (H,) fp32
    dy: torch.Tensor                # (b, L, H, P)
    initial_states: Optional[torch.Tensor] = None   # (b, H, P, N) fp32
    seq_idx: Optional[torch.Tensor] = None          # (b, L) int32
    dfinal_states: Optional[torch.Tensor] = None    # (b, H, P, N) fp32
    seq_lengths: Optional[list] = None

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def f64(self, name: str) -> Optional[np.ndarray]:
        """Exact float64 (or int32) numpy copy of one input, for the oracle."""
        t = getattr(self, name)
        if t is None:
            return None
        if t.dtype == torch.int32:
            return t.numpy().copy()
        return t.to(torch.float64).numpy().copy()

    def dims(self) -> dict:
        return dict(batch=self.batch, seqlen=self.seqlen, nheads=self.nheads,
                    headdim=self.headdim, dstate=self.dstate,
                    ngroups=self.ngroups, chunk=self.chunk)


def _round(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f32":
        return t.clone()
    raise ValueError(f"unknown dtype {dtype!r}")


def draw_lengths(rng, nseq, min_len, max_len, max_total):
    """Integer lengths uniform in [min_len, max_len], redrawn until sum <= max_total."""
    while True:
        lens = rng.integers(min_len, max_len + 1, size=nseq)
        if int(lens.sum()) <= max_total:
            return [int(v) for v in lens]


def make_inputs(batch=1, seqlen=64, nheads=2, headdim=8, dstate=8, ngroups=1,
                chunk=16, dtype="f32", init=False, dfinal=False,
                seq_lengths=None, seed=0, rng=None,
                init_std=0.1) -> SSDInputs:
    """Draw one problem.  ``seq_lengths`` (a list summing to seqlen, batch 1
    or per-row identical) turns on seq_idx with those segment lengths."""
    if rng is None:
        rng = np.random.default_rng(seed)
    b, L, H, P, N, G = batch, seqlen, nheads, headdim, dstate, ngroups
    if H % G != 0:
        raise ValueError("ngroups must divide nheads")
    f32 = np.float32
    dt_target = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=H))
    A = -np.exp(rng.uniform(0.0, math.log(16.0), size=H))
    x = rng.standard_normal((b, L, H, P), dtype=f32)
    dt = rng.standard_normal((b, L, H), dtype=f32)
    sc = f32(1.0 / math.sqrt(N))
    Bm = rng.standard_normal((b, L, G, N), dtype=f32) * sc
    Cm = rng.standard_normal((b, L, G, N), dtype=f32) * sc
    D = rng.standard_normal(H)
    init_t = None
    if init:
        init_t = torch.from_numpy(
            (rng.standard_normal((b, H, P, N), dtype=f32) * f32(init_std)))
    dy = rng.standard_normal((b, L, H, P), dtype=f32)
    dfin_t = None
    if dfinal:
        dfin_t = torch.from_numpy(rng.standard_normal((b, H, P, N), dtype=f32))
    seq_t = None
    if seq_lengths is not None:
        if sum(seq_lengths) != L:
            raise ValueError("seq_lengths must sum to seqlen")
        ids = np.repeat(np.arange(len(seq_lengths), dtype=np.int32), seq_lengths)
        seq_t = torch.from_numpy(np.ascontiguousarray(
            np.broadcast_to(ids, (b, L)).astype(np.int32)))
    dt_bias = np.log(np.expm1(dt_target))
    return SSDInputs(
        batch=b, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G,
        chunk=chunk, dtype=dtype,
        x=_round(x, dtype), dt=_round(dt, dtype),
        dt_bias=torch.from_numpy(dt_bias.astype(f32)),
        A=torch.from_numpy(A.astype(f32)),
        B=_round(Bm, dtype), C=_round(Cm, dtype),
        D=torch.from_numpy(D.astype(f32)),
        dy=_round(dy, dtype),
        initial_states=init_t, seq_idx=seq_t, dfinal_states=dfin_t,
        seq_lengths=list(seq_lengths) if seq_lengths is not None else None)


def make_workload(name: str, seed: int = 0, **overrides) -> SSDInputs:
    """Draw one of the named workloads (``WORKLOADS``) with seed ``seed``."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    rng = np.random.default_rng(seed)
    if "nseq" in cfg:
        lens = draw_lengths(rng, cfg.pop("nseq"), cfg.pop("min_len"),
                            cfg.pop("max_len"), cfg.pop("max_total"))
        cfg["batch"] = 1
        cfg["seqlen"] = sum(lens)
        cfg["seq_lengths"] = lens
    return make_inputs(rng=rng, **cfg)


# ---------------------------------------------------------------------------
# Gated RMSNorm of the Mamba-2 block (the normalisation after the scan).
#
# Recipe (numpy PCG64 ``default_rng(seed)``, draw order y, z, weight, dout):
#   y, z, dout ~ N(0, 1)   (y has the scan output's unit scale, z the gate's)
#   weight = 1 + 0.1 * N(0, 1)   (the usual all-ones start, perturbed so that
#                                 a dropped or misplaced weight shows)
#   eps = 1e-5
# Shapes follow the layer workloads: rows = tokens (batch * seqlen, or the
# packed total), dim = nheads * headdim, group_size = dim / ngroups.

@dataclasses.dataclass
class NormInputs:
    """One gated-RMSNorm problem's inputs as CPU torch tensors."""
    rows: int
    dim: int
    group_size: int
    eps: float
    dtype: str                      # "bf16" or "f32"
    y: torch.Tensor                 # (rows, dim)
    z: Optional[torch.Tensor]       # (rows, dim), None without a gate
    weight: torch.Tensor            # (dim,) fp32
    dout: torch.Tensor              # (rows, dim)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def f64(self, name: str) -> Optional[np.ndarray]:
        t = getattr(self, name)
        return None if t is None else t.to(torch.float64).numpy().copy()


def make_norm_inputs(rows, dim, group_size, dtype="bf16", gate=True, eps=1e-5, seed=0,
                     rng=None) -> NormInputs:
    if dim % group_size != 0:
        raise ValueError("group_size must divide dim")
    if rng is None:
        rng = np.random.default_rng(seed)
    f32 = np.float32
    y = rng.standard_normal((rows, dim), dtype=f32)
    z = rng.standard_normal((rows, dim), dtype=f32)
    w = 1.0 + 0.1 * rng.standard_normal(dim)
    dout = rng.standard_normal((rows, dim), dtype=f32)
    return NormInputs(rows=rows, dim=dim, group_size=group_size, eps=eps, dtype=dtype,
                      y=_round(y, dtype), z=_round(z, dtype) if gate else None,
                      weight=torch.from_numpy(w.astype(f32)), dout=_round(dout, dtype))


def norm_shape(name: str, seed: int = 0) -> dict:
    """(rows, dim, group_size, dtype) of the gated norm that follows the scan
    of layer workload ``name``."""
    cfg = WORKLOADS[name]
    if "nseq" in cfg:
        rng = np.random.default_rng(seed)
        rows = sum(draw_lengths(rng, cfg["nseq"], cfg["min_len"], cfg["max_len"],
                                cfg["max_total"]))
    else:
        rows = cfg["batch"] * cfg["seqlen"]
    dim = cfg["nheads"] * cfg["headdim"]
    return dict(rows=rows, dim=dim, group_size=dim // cfg["ngroups"], dtype=cfg["dtype"])


def make_norm_workload(name: str, seed: int = 0, gate=True, **overrides) -> NormInputs:
    shape = norm_shape(name, seed)
    shape.update(overrides)
    return make_norm_inputs(gate=gate, seed=seed, **shape)
