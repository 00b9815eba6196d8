"""CPU oracle for the compressed-KV sparse-attention (CSA) decode path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

The oracle is a plain, slow, obviously-correct restatement of what the path
computes, written in numpy float64 from the method's own definitions:

* ``codecs``    -- E2M1 / E4M3(FN) / UE8M0 / FP16 element codecs, the per-block
                   power-of-two scale rule and the packed 68-byte indexer row
                   and 583-byte KV row (DS4X README, "Packed cache ABI").
* ``indexer``   -- CSA indexer score and the exact top-k with the float total
                   order and lower-index tie break (DS4X README,
                   "Optimization details" and "CSA score/top-512 fusion").
* ``attention`` -- exact softmax attention of a decode query over the selected
                   packed KV rows (DS4X README, "Packed cache ABI" row layout;
                   shared K = V over the 512-element row); dense attention over
                   every row (the HCA layers, DS4X README, "Optimization
                   details"), the split-KV log-sum-exp combine, and attention
                   over the selected rows plus the raw sliding window.
* ``prefill``   -- the multi-query (chunked prefill) scorer with E4M3-quantised
                   queries and a causal visibility rule, then per-query top-k
                   and attention (DS4X README, "Packed prefill implementation").
* ``layout``    -- row sizes and the persistent allocation formula
                   (DS4X README, "Packed cache ABI").
* ``checkpoint`` -- the packed-row checkpoint layout, written and read in plain
                   Python (payload version 3: DS4X README, "Optimization
                   details"; the window in logical order: ds4 README, "Disk KV
                   Cache").

It shares no code with the CUDA path (``compressed_kv_sparse_csa_gb300``) and
neither imports the other.  Every function is pinned by a ``-m "not gpu"``
test in ``tests/test_oracle_*.py`` (the checkpoint layout in
``tests/test_checkpoint.py``, at fixed offsets) against something other than
itself (page values, library conversions, brute force, closed forms).
"""

from . import attention, checkpoint, codecs, indexer, layout, prefill  # noqa: F401
