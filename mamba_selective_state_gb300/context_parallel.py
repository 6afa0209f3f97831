"""Context parallelism of the SSD layer: the sequence split into contiguous
shards, each shard run through ssd_fwd / ssd_bwd as a problem of its own,
the shards joined by the two folds of ssd_shard_fold (see include/ssd.h).

Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906) names context
parallelism as the integration goal of its module; the decomposition follows
from the recurrence: a shard maps the state entering it, h, to
dec * h + final(0), and its dinitial_states is affine in the gradient at its
final state.

``run_sharded`` drives the shards this process owns.  The exchange between
shards is an argument: ``StackExchange`` when one process runs every shard
one after another (one GPU), ``DistExchange`` when every rank owns one shard
(torch.distributed all-gather / all-reduce, NCCL on GPUs).  Marshalling and
the exchange only: every step of the layer and both folds run in libssd.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch

from . import _lib
from .inputs import SSDInputs


def shard_bounds(seqlen: int, sizes: Sequence[int]):
    """[start, end) token ranges of contiguous shards of the given sizes."""
    if sum(sizes) != seqlen or min(sizes) < 1:
        raise ValueError("shard sizes must be positive and sum to seqlen")
    out, s = [], 0
    for n in sizes:
        out.append((s, s + n))
        s += n
    return out


def shard_inputs(inp: SSDInputs, start: int, end: int) -> SSDInputs:
    """The inputs of tokens [start, end) of every row, as a problem of its own
    (no initial or final-state gradient: the folds supply them)."""
    cut = lambda t: None if t is None else t[:, start:end].contiguous()  # noqa: E731
    return dataclasses.replace(inp, seqlen=end - start, x=cut(inp.x), dt=cut(inp.dt),
                               B=cut(inp.B), C=cut(inp.C), dy=cut(inp.dy),
                               seq_idx=cut(inp.seq_idx), initial_states=None,
                               dfinal_states=None)


class StackExchange:
    """All shards in this process: a gather is a stack in shard order, a sum
    over shards a plain sum."""

    def __init__(self, nshards: int):
        self.nshards = nshards

    def gather(self, parts: List[torch.Tensor]) -> torch.Tensor:
        return torch.stack(parts)

    def sum(self, t: torch.Tensor) -> torch.Tensor:
        return t


class DistExchange:
    """One shard per rank, rank order = shard order (torch.distributed)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.nshards = dist.get_world_size(group)

    def gather(self, parts: List[torch.Tensor]) -> torch.Tensor:
        (t,) = parts
        t = t.contiguous()
        # gathered along the leading dimension (the form every backend takes),
        # then viewed as one slice per shard
        out = torch.empty((self.nshards * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype,
                          device=t.device)
        self.dist.all_gather_into_tensor(out, t, group=self.group)
        return out.view((self.nshards,) + tuple(t.shape))

    def sum(self, t: torch.Tensor) -> torch.Tensor:
        self.dist.all_reduce(t, group=self.group)
        return t


@dataclasses.dataclass
class _Shard:
    index: int
    inp: SSDInputs
    dev: dict


def _buffers(inp: SSDInputs, device) -> dict:
    to = lambda t: None if t is None else t.to(device).contiguous()  # noqa: E731
    b, L, H, P, N, G = inp.batch, inp.seqlen, inp.nheads, inp.headdim, inp.dstate, inp.ngroups
    d = dict(x=to(inp.x), dt=to(inp.dt), B=to(inp.B), C=to(inp.C), dy=to(inp.dy),
             dt_bias=to(inp.dt_bias), A=to(inp.A), D=to(inp.D), seq=to(inp.seq_idx))
    f32 = dict(dtype=torch.float32, device=device)
    d["y"] = torch.empty((b, L, H, P), dtype=inp.torch_dtype, device=device)
    d["final"] = torch.empty((b, H, P, N), **f32)
    d["dinit"] = torch.empty((b, H, P, N), **f32)
    d["dx"], d["ddt"] = torch.empty_like(d["x"]), torch.empty_like(d["dt"])
    d["dB"], d["dC"] = torch.empty_like(d["B"]), torch.empty_like(d["C"])
    for k in ("ddt_bias", "dA", "dD"):
        d[k] = torch.empty(H, **f32)
    d["decay"] = torch.empty((b, H), **f32)
    d["first"] = torch.empty(b, dtype=torch.int32, device=device)
    d["last"] = torch.empty(b, dtype=torch.int32, device=device)
    base = _lib.SSD_HAS_SEQ_IDX if inp.seq_idx is not None else 0
    mk = lambda fl: _lib.make_problem(b, L, H, P, N, G, inp.chunk, inp.torch_dtype, base | fl)  # noqa: E731
    d["prob0"] = mk(0)
    d["prob_init"] = mk(_lib.SSD_HAS_INIT)
    d["bprob0"] = mk(_lib.SSD_HAS_INIT | _lib.SSD_WANT_DINIT)
    d["bprob"] = mk(_lib.SSD_HAS_INIT | _lib.SSD_WANT_DINIT | _lib.SSD_HAS_DFINAL)
    ws = max(_lib.ssd_bwd_workspace_bytes(d["bprob"]), _lib.ssd_fwd_workspace_bytes(d["prob0"]))
    d["ws"] = torch.empty(ws, dtype=torch.uint8, device=device)
    return d


class ShardedLayer:
    """The shards this process owns (``indices``: their places in sequence
    order), with their device buffers allocated once; ``run`` is one forward
    and backward of the layer over the whole sequence, joined with the other
    shards through ``exchange``."""

    def __init__(self, shards: List[SSDInputs], indices: List[int], exchange, device="cuda"):
        self.own = [_Shard(i, s, _buffers(s, device)) for i, s in zip(indices, shards)]
        self.exchange = exchange
        self.device = device
        s0 = shards[0]
        self.dims = (s0.batch, s0.nheads, s0.headdim, s0.dstate)

    def run(self, initial_states: Optional[torch.Tensor] = None,
            dfinal_states: Optional[torch.Tensor] = None, stream=None) -> dict:
        """Returns, per owned shard, y and the per-token gradients (views of
        the shard buffers, valid until the next run), and the layer-wide
        final_states, dA, dD, ddt_bias and dinitial_states (the latter from
        shard 0, on its owner)."""
        b, H, P, N = self.dims
        device, st, exchange = self.device, stream, self.exchange
        f32 = dict(dtype=torch.float32, device=device)
        init = None if initial_states is None else initial_states.to(device).contiguous()
        dfin = None if dfinal_states is None else dfinal_states.to(device).contiguous()

        def fwd(d, prob, init_t):
            _lib.ssd_fwd(prob, d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], init_t,
                         d["seq"], d["y"], d["final"], d["ws"], stream=st)

        def bwd(d, prob, init_t, dfin_t):
            _lib.ssd_bwd(prob, d["x"], d["dt"], d["dt_bias"], d["A"], d["B"], d["C"], d["D"], init_t,
                         d["seq"], d["dy"], dfin_t, d["dx"], d["ddt"], d["ddt_bias"], d["dA"], d["dB"],
                         d["dC"], d["dD"], d["dinit"], d["ws"], stream=st)

        # 1. every owned shard from a zero state, its decay and boundary segment ids
        for s in self.own:
            d = s.dev
            fwd(d, d["prob0"], None)
            _lib.ssd_shard_decay(d["prob0"], d["dt"], d["dt_bias"], d["A"], d["seq"], d["decay"],
                                 d["first"], d["last"], stream=st)
        # 2. exchange, the forward fold, every owned shard again from its entering state
        FIN0 = exchange.gather([s.dev["final"] for s in self.own])
        DEC = exchange.gather([s.dev["decay"] for s in self.own])
        FIRST = exchange.gather([s.dev["first"] for s in self.own])
        LAST = exchange.gather([s.dev["last"] for s in self.own])
        R = FIN0.shape[0]
        enter = torch.empty((R, b, H, P, N), **f32)
        final = torch.empty((b, H, P, N), **f32)
        _lib.ssd_shard_fold(DEC, FIN0, FIRST, LAST, init, enter, final, reverse=False, stream=st)
        for s in self.own:
            fwd(s.dev, s.dev["prob_init"], enter[s.index])
        # 3. backward: dinit with no upstream final gradient, the reverse fold,
        #    then every owned shard's backward with its upstream gradient
        for s in self.own:
            bwd(s.dev, s.dev["bprob0"], enter[s.index], None)
        D0 = exchange.gather([s.dev["dinit"] for s in self.own])
        gout = torch.empty((R, b, H, P, N), **f32)
        _lib.ssd_shard_fold(DEC, D0, FIRST, LAST, dfin, gout, None, reverse=True, stream=st)
        out = dict(final_states=final)
        for k in ("y", "dx", "ddt", "dB", "dC"):
            out[k] = {}
        psum = {k: torch.zeros(H, **f32) for k in ("dA", "dD", "ddt_bias")}
        for s in self.own:
            d = s.dev
            bwd(d, d["bprob"], enter[s.index], gout[s.index])
            for k in ("y", "dx", "ddt", "dB", "dC"):
                out[k][s.index] = d[k]
            for k in psum:
                psum[k] += d[k]
            if s.index == 0:
                out["dinitial_states"] = d["dinit"]
        for k, v in psum.items():
            out[k] = exchange.sum(v)
        return out


def run_sharded(shards: List[SSDInputs], indices: List[int], exchange, device="cuda",
                initial_states: Optional[torch.Tensor] = None,
                dfinal_states: Optional[torch.Tensor] = None, stream=None) -> dict:
    """One forward and backward of the layer over a sequence split into
    shards (see ShardedLayer)."""
    return ShardedLayer(shards, indices, exchange, device).run(initial_states, dfinal_states, stream)
