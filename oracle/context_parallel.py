"""Context parallelism of the SSD layer in float64: the sequence split into
contiguous shards (one per rank), each shard run on its own, and the shards
joined by one exclusive scan of per-shard (decay, state) pairs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906) names context
parallelism, the sequence sharded across ranks, as the extension its drop-in
module is meant to support; it gives no method.  The plainest one follows
from the recurrence itself (page "llm-mamba-200", sections 2-3): a shard
maps the state entering it, h, to the state leaving it as

    final(h) = dec * h + final(0)

with dec the product of the shard's per-token decays exp(dt_eff * A) for
each (row, head) -- or 0 when a new segment starts inside the shard, since
the reset cuts the entering state off -- and final(0) the shard's final
state from a zero start.  These (dec, final(0)) pairs compose with the same
operator as the chunks of one sequence, (a, b) o (a', b') = (a a', a' b + b'),
so one exclusive fold over the shards, in rank order, gives every shard the
state entering it; a shard whose first token starts a new segment enters
from zero.  Each shard is then run again from that state.

The backward mirrors it from the right.  The gradient reaching a shard's
final state is the gradient with respect to the state entering the next
shard (zero when that shard starts a new segment), and a shard's
dinitial_states is affine in the gradient at its final state:

    dinit(g) = dec * g + dinit(0)

with dinit(0) from the shard's backward with no upstream gradient at its
final state.  A right-to-left fold over the shards gives every shard its
upstream dfinal_states; each shard then runs its backward with it.  Per-token
gradients stay on their shard; dA, dD and ddt_bias are sums over shards.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def _softplus(z):
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def shard_decay(dt, dt_bias, A, seq_idx=None):
    """Product of a shard's per-token decays for every (row, head), (b, H),
    or 0 for the rows in which a new segment starts after the shard's first
    token.  dt: (b, Ls, H) of the shard; seq_idx: (b, Ls) or None."""
    dt = np.asarray(dt, dtype=np.float64)
    dt_eff = _softplus(dt + np.asarray(dt_bias, dtype=np.float64)[None, None, :])
    dec = np.exp((dt_eff * np.asarray(A, dtype=np.float64)[None, None, :]).sum(axis=1))
    if seq_idx is not None:
        seq = np.asarray(seq_idx)
        reset = (seq[:, 1:] != seq[:, :-1]).any(axis=1)
        dec[reset, :] = 0.0
    return dec


def shard_breaks(first_ids, last_ids):
    """Whether each shard's first token starts a new segment, (R, b): shard
    r > 0 breaks in row bi when its first token's segment id differs from the
    previous shard's last token's.  first_ids, last_ids: (R, b); shard 0
    never breaks (the initial state feeds its first segment)."""
    first_ids = np.asarray(first_ids)
    last_ids = np.asarray(last_ids)
    brk = np.zeros(first_ids.shape, dtype=bool)
    brk[1:] = first_ids[1:] != last_ids[:-1]
    return brk


def carries_in(decays, finals0, breaks, initial_states=None):
    """Left-to-right exclusive fold over the shards.

    decays (R, b, H), finals0 (R, b, H, P, N), breaks (R, b) bool,
    initial_states (b, H, P, N) or None.  Returns the state entering every
    shard, (R, b, H, P, N), and the state after the last one."""
    decays = np.asarray(decays, dtype=np.float64)
    finals0 = np.asarray(finals0, dtype=np.float64)
    R = finals0.shape[0]
    h = (np.zeros(finals0.shape[1:]) if initial_states is None
         else np.asarray(initial_states, dtype=np.float64).copy())
    entering = np.empty_like(finals0)
    for r in range(R):
        if r > 0:
            h[np.asarray(breaks[r], dtype=bool)] = 0.0
        entering[r] = h
        h = decays[r][:, :, None, None] * h + finals0[r]
    return entering, h


def dfinals_out(decays, dinits0, breaks, dfinal_states=None):
    """Right-to-left exclusive fold over the shards.

    decays (R, b, H), dinits0 (R, b, H, P, N) (each shard's dinitial_states
    with no upstream gradient at its final state), breaks (R, b) bool,
    dfinal_states (b, H, P, N) or None (the layer's upstream gradient at the
    last shard's final state).  Returns the upstream gradient at every
    shard's final state, (R, b, H, P, N)."""
    decays = np.asarray(decays, dtype=np.float64)
    dinits0 = np.asarray(dinits0, dtype=np.float64)
    R = dinits0.shape[0]
    g = (np.zeros(dinits0.shape[1:]) if dfinal_states is None
         else np.asarray(dfinal_states, dtype=np.float64).copy())
    out = np.empty_like(dinits0)
    for r in range(R - 1, -1, -1):
        out[r] = g
        g = decays[r][:, :, None, None] * g + dinits0[r]  # d loss / d state entering shard r
        if r > 0:
            g[np.asarray(breaks[r], dtype=bool)] = 0.0      # shard r did not read the previous final
    return out


def shard_bounds(seqlen: int, sizes: Sequence[int]):
    """[start, end) token ranges of contiguous shards of the given sizes."""
    if sum(sizes) != seqlen or min(sizes) < 1:
        raise ValueError("shard sizes must be positive and sum to seqlen")
    ends = np.cumsum(sizes)
    return [(int(e - s), int(e)) for s, e in zip(sizes, ends)]


def context_parallel(fwd, bwd, inputs: dict, sizes: Sequence[int],
                     dfinal_states: Optional[np.ndarray] = None):
    """The layer evaluated shard by shard with the two folds above, the
    exchange done in one process.  ``fwd``/``bwd`` evaluate one shard (the
    float64 oracle's ``ssd_fwd``/``ssd_bwd`` signatures); ``inputs`` holds
    x, dt, dt_bias, A, B, C, D, dy and optional initial_states, seq_idx.
    Returns y, final_states and the gradients as the unsharded call would."""
    x, dt, dy = inputs["x"], inputs["dt"], inputs["dy"]
    seq = inputs.get("seq_idx")
    init = inputs.get("initial_states")
    params = [inputs[n] for n in ("dt_bias", "A")]
    bounds = shard_bounds(x.shape[1], sizes)

    def cut(a, s, e):
        return None if a is None else a[:, s:e]

    def args(s, e):
        return [cut(x, s, e), cut(dt, s, e), inputs["dt_bias"], inputs["A"], cut(inputs["B"], s, e),
                cut(inputs["C"], s, e), inputs["D"]]

    # 1. every shard from a zero state: its final state and its decay
    fin0 = np.stack([fwd(*args(s, e), seq_idx=cut(seq, s, e))[1] for s, e in bounds])
    dec = np.stack([shard_decay(cut(dt, s, e), *params, seq_idx=cut(seq, s, e)) for s, e in bounds])
    if seq is None:
        brk = np.zeros((len(bounds), x.shape[0]), dtype=bool)
    else:
        brk = shard_breaks([seq[:, s] for s, _ in bounds], [seq[:, e - 1] for _, e in bounds])
    # 2. exclusive fold, then every shard again from the state entering it
    h_in, final = carries_in(dec, fin0, brk, init)
    ys = [fwd(*args(s, e), initial_states=h_in[r], seq_idx=cut(seq, s, e))[0]
          for r, (s, e) in enumerate(bounds)]
    # 3. backward: each shard's dinit with no upstream final gradient, the
    #    reverse fold, then every shard's backward with its upstream gradient
    d0 = np.stack([bwd(*args(s, e), cut(dy, s, e), initial_states=h_in[r],
                       seq_idx=cut(seq, s, e))["dinitial_states"]
                   for r, (s, e) in enumerate(bounds)])
    g_out = dfinals_out(dec, d0, brk, dfinal_states)
    grads = [bwd(*args(s, e), cut(dy, s, e), initial_states=h_in[r], seq_idx=cut(seq, s, e),
                 dfinal_states=g_out[r]) for r, (s, e) in enumerate(bounds)]
    out = dict(y=np.concatenate(ys, axis=1), final_states=final)
    for k in ("dx", "ddt", "dB", "dC"):
        out[k] = np.concatenate([g[k] for g in grads], axis=1)
    for k in ("dA", "dD", "ddt_bias"):
        out[k] = np.sum([g[k] for g in grads], axis=0)
    out["dinitial_states"] = grads[0]["dinitial_states"]
    return out
