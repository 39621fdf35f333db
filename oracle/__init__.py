"""Float64 CPU oracle for chunked causal attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
product path (the CUDA library and its Python binding) never imports, links or
executes anything here, and this package never imports the product.

Modules
-------
plan       integer chunk-boundary rules (SPPO "FLOPs-based partition"; uniform
           "length-based" partition; edge re-split; InfiniPipe split chunks).
attention  the plain definition of causal softmax attention in float64 with an
           explicit score matrix, its analytic backward, sampled-row forms for
           long sequences, and the chunk-by-chunk method with the log-sum-exp
           merge that the chunked schedule is built on.

Every function states the passage it follows. Parity is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py`` against brute force,
closed forms, invariants, finite differences and torch float64 routines.
"""
