"""The associative pair-combine of the SSM recurrence, and a log-step scan.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Page "llm-mamba-200" (gigipick.blogspot.com), section 2 ("principle of the
parallel associative scan"): each step t is turned into a pair (A_t, B_t x_t)
and the pairs are folded left to right with an associative operator, so the
state after t steps is a prefix "sum" of the pairs.  The operator itself is
lost from the extracted text; for a scalar decay per head it is read as

    (a, b) o (a', b') = (a * a', a' * b + b')

where the left operand is the earlier span: applying the earlier span and
then the later one to a state h gives a' * (a * h + b) + b'.  The identity is
(1, 0); a pair (0, b') (a sequence reset) discards everything to its left.

The same page, section "Hillis-Steele based implementation", scans with one
thread per element and steps d = 1, 2, 4, ... < n, each element combining
with the one d places to its left, all elements of a step reading the values
of the previous step (the barrier between steps).
"""
from __future__ import annotations

import numpy as np


def combine(left, right):
    """(a, b) o (a', b') = (a a', a' b + b'); ``left`` is the earlier span."""
    a, b = left
    a2, b2 = right
    return (a * a2, a2 * b + b2)


IDENTITY = (1.0, 0.0)


def sequential_scan(pairs):
    """Inclusive prefix of ``pairs`` folded left to right, one at a time."""
    out = []
    acc = None
    for p in pairs:
        acc = p if acc is None else combine(acc, p)
        out.append(acc)
    return out


def hillis_steele_scan(pairs):
    """Inclusive prefix by the log-step scheme: at step d every element i >= d
    becomes V[i-d] o V[i], reading only the previous step's values."""
    v = list(pairs)
    n = len(v)
    d = 1
    while d < n:
        nxt = list(v)
        for i in range(d, n):
            nxt[i] = combine(v[i - d], v[i])
        v = nxt
        d *= 2
    return v


def apply(pair, h):
    """Apply a span (a, b) to an incoming state h: a * h + b."""
    a, b = pair
    return a * h + b


def states_from_scan(a_seq, b_seq, h0):
    """States after each step of h_t = a_t h_{t-1} + b_t, computed by scanning
    the pairs (a_t, b_t) and applying each prefix to h0."""
    pre = hillis_steele_scan(list(zip(a_seq, b_seq)))
    return [apply(p, h0) for p in pre]


def as_array_pairs(a, b):
    """Helper: pair lists from numpy arrays (a: (T,), b: (T, ...))."""
    return [(np.float64(a[i]), np.asarray(b[i], dtype=np.float64)) for i in range(len(a))]
