"""Device buffers for one SSD problem and the calls that run it through the
C ABI.  Allocation and argument marshalling only; the layer runs in libssd.
"""
from __future__ import annotations

import torch

from . import _lib
from .inputs import NormInputs, SSDInputs


class SSDDevice:
    """Inputs copied to ``device``, outputs, gradients and workspace allocated.

    ``dfinal``/``want_dinit`` select the optional backward arguments; by
    default they follow the inputs (dfinal_states present -> used; initial
    states present -> dinitial_states wanted)."""

    def __init__(self, inp: SSDInputs, device="cuda", backward=True, dfinal=None,
                 want_dinit=None, extra_flags=0):
        self.inp = inp
        self.device = torch.device(device)
        dev = self.device
        to = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
        self.x, self.dt, self.B, self.C = to(inp.x), to(inp.dt), to(inp.B), to(inp.C)
        self.dt_bias, self.A, self.D = to(inp.dt_bias), to(inp.A), to(inp.D)
        self.init = to(inp.initial_states)
        self.seq_idx = to(inp.seq_idx)
        use_dfinal = (inp.dfinal_states is not None) if dfinal is None else dfinal
        self.dfinal = to(inp.dfinal_states) if use_dfinal else None
        self.want_dinit = (inp.initial_states is not None) if want_dinit is None else want_dinit
        self.dy = to(inp.dy) if backward else None
        dt_t = inp.torch_dtype
        b, L, H, P, N, G = inp.batch, inp.seqlen, inp.nheads, inp.headdim, inp.dstate, inp.ngroups
        flags = extra_flags
        if self.init is not None:
            flags |= _lib.SSD_HAS_INIT
        if self.seq_idx is not None:
            flags |= _lib.SSD_HAS_SEQ_IDX
        self.fwd_prob = _lib.make_problem(b, L, H, P, N, G, inp.chunk, dt_t, flags)
        bflags = flags
        if self.dfinal is not None:
            bflags |= _lib.SSD_HAS_DFINAL
        if self.want_dinit:
            bflags |= _lib.SSD_WANT_DINIT
        self.bwd_prob = _lib.make_problem(b, L, H, P, N, G, inp.chunk, dt_t, bflags)
        self.y = torch.empty((b, L, H, P), dtype=dt_t, device=dev)
        self.final = torch.empty((b, H, P, N), dtype=torch.float32, device=dev)
        ws = _lib.ssd_bwd_workspace_bytes(self.bwd_prob) if backward else \
            _lib.ssd_fwd_workspace_bytes(self.fwd_prob)
        if ws == 0:
            raise _lib.SSDError(_lib.SSD_ERR_INVALID_ARGUMENT, "workspace size")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        if backward:
            self.dx = torch.empty_like(self.x)
            self.ddt = torch.empty_like(self.dt)
            self.dB = torch.empty_like(self.B)
            self.dC = torch.empty_like(self.C)
            self.ddt_bias = torch.empty(H, dtype=torch.float32, device=dev)
            self.dA = torch.empty(H, dtype=torch.float32, device=dev)
            self.dD = torch.empty(H, dtype=torch.float32, device=dev)
            self.dinit = (torch.empty((b, H, P, N), dtype=torch.float32, device=dev)
                          if self.want_dinit else None)

    def fwd(self, stream=None, check=True):
        return _lib.ssd_fwd(self.fwd_prob, self.x, self.dt, self.dt_bias, self.A, self.B, self.C,
                            self.D, self.init, self.seq_idx, self.y, self.final, self.workspace,
                            stream=stream, check=check)

    def bwd(self, stream=None, check=True):
        return _lib.ssd_bwd(self.bwd_prob, self.x, self.dt, self.dt_bias, self.A, self.B, self.C,
                            self.D, self.init, self.seq_idx, self.dy, self.dfinal, self.dx,
                            self.ddt, self.ddt_bias, self.dA, self.dB, self.dC, self.dD,
                            self.dinit, self.workspace, stream=stream, check=check)

    def device_status(self, stream=None):
        return _lib.ssd_read_device_status(self.workspace, stream)

    def results(self) -> dict:
        """Outputs and gradients as CPU float64 tensors."""
        out = dict(y=self.y, final_states=self.final)
        if self.dy is not None:
            out.update(dx=self.dx, ddt=self.ddt, dB=self.dB, dC=self.dC, ddt_bias=self.ddt_bias,
                       dA=self.dA, dD=self.dD)
            if self.dinit is not None:
                out["dinitial_states"] = self.dinit
        return {k: v.detach().to("cpu", torch.float64) for k, v in out.items()}


class NormDevice:
    """Device buffers of one gated-RMSNorm problem (inputs, out, rstd, the
    gradients and the backward workspace) and its calls through the C ABI."""

    def __init__(self, inp: NormInputs, device="cuda"):
        self.inp = inp
        dev = torch.device(device)
        to = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
        self.y, self.z, self.weight, self.dout = to(inp.y), to(inp.z), to(inp.weight), to(inp.dout)
        self.prob = _lib.make_norm_problem(inp.rows, inp.dim, inp.group_size, inp.eps,
                                           inp.torch_dtype, gate=inp.z is not None)
        self.out = torch.empty_like(self.y)
        self.rstd = torch.empty((inp.rows, inp.dim // inp.group_size), dtype=torch.float32,
                                device=dev)
        self.dy = torch.empty_like(self.y)
        self.dz = None if self.z is None else torch.empty_like(self.z)
        self.dweight = torch.empty(inp.dim, dtype=torch.float32, device=dev)
        ws = _lib.ssd_gated_rmsnorm_bwd_workspace_bytes(self.prob)
        if ws == 0:
            raise _lib.SSDError(_lib.SSD_ERR_INVALID_ARGUMENT, "norm workspace size")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def fwd(self, stream=None, check=True):
        return _lib.ssd_gated_rmsnorm_fwd(self.prob, self.y, self.z, self.weight, self.out,
                                          self.rstd, stream=stream, check=check)

    def bwd(self, stream=None, check=True):
        return _lib.ssd_gated_rmsnorm_bwd(self.prob, self.y, self.z, self.weight, self.dout,
                                          self.dy, self.dz, self.dweight, self.workspace,
                                          stream=stream, check=check)

    def results(self) -> dict:
        out = dict(out=self.out, rstd=self.rstd, dy=self.dy, dweight=self.dweight)
        if self.dz is not None:
            out["dz"] = self.dz
        return {k: v.detach().to("cpu", torch.float64) for k, v in out.items()}
