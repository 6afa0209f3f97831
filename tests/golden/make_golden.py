"""Writes oracle_small.json: outputs of the float64 oracle on one small seeded
problem (resets, initial state, upstream final-state gradient, two groups).

The fixture guards the oracle against unnoticed drift: any change to the
oracle's arithmetic that moves these numbers must be regenerated here and
justified.  It calls only the input generator and ``oracle/``.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from mamba_selective_state_gb300.inputs import make_inputs  # noqa: E402
from oracle import ssd_ref  # noqa: E402

CASE = dict(batch=1, seqlen=12, nheads=2, headdim=2, dstate=3, ngroups=2, chunk=4,
            dtype="f32", init=True, dfinal=True, seq_lengths=[5, 7], seed=17)


def compute():
    inp = make_inputs(**CASE)
    f = inp.f64
    args = [f(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D"]]
    kw = dict(initial_states=f("initial_states"), seq_idx=f("seq_idx"))
    y, fin = ssd_ref.ssd_fwd(*args, **kw)
    g = ssd_ref.ssd_bwd(*args, f("dy"), dfinal_states=f("dfinal_states"), **kw)
    out = dict(y=y, final_states=fin, **g)
    return {k: v.reshape(-1).tolist() for k, v in out.items()}


if __name__ == "__main__":
    data = dict(case=CASE, values=compute())
    with open(os.path.join(HERE, "oracle_small.json"), "w") as fh:
        json.dump(data, fh, indent=1)
