"""Oracle for the GLA prefill forward pass and the gated delta rule — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or run anything in this package. The product
path (``chunkwise_recurrent_prefill_gb300``) never does, and this package never
imports the product path: the two share no code, headers, tables or helpers.

Contents:
  gla_oracle.c   fp64 token-by-token recurrence (plain C, OpenMP over heads).
  gla_ref.py     ctypes binding to it, an independent pure-numpy token loop, and an
                 fp64 numpy restatement of the chunkwise algorithm.
  gdn_ref.py     the gated delta rule: fp64 numpy token loop and chunk algebra, pinned by
                 ``tests/test_gdn_oracle_pins.py`` (its formula is a reading from outside the
                 pages, which name the method but print no recurrence).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute-force decay-matrix attention, the ungated textbook case, closed forms,
state carry, linearity, exact rational arithmetic). No function is parity-unpinned.
"""
from .gla_ref import (  # noqa: F401
    build,
    recurrent,
    recurrent_head,
    recurrent_np,
    chunkwise_np,
    num_threads,
)
