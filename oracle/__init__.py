"""Float64 CPU oracle of the Mamba-2 SSD layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and imports nothing from it.

  ssd_ref      -- ctypes wrapper over ``ssd_oracle.c``: the sequential
                  recurrence (forward) and its hand-derived reverse mode.
  chunked      -- numpy float64 evaluation of the same layer by chunks
                  (chunk states, state passing, intra-chunk output), forward
                  and backward, returning the intermediates as well.
  scan         -- the pair-combine operator of the associative scan and a
                  Hillis-Steele log-step scan built on it.
  gated_norm   -- numpy float64 gated RMSNorm of the Mamba-2 block (the
                  normalisation after the scan), forward and hand-derived
                  reverse mode.
  context_parallel -- the layer over a sequence split into shards, joined by
                  exclusive folds of per-shard (decay, state) pairs and of
                  dinitial states (context parallelism).
"""
