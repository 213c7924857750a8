"""Oracle for the GLA prefill forward pass and the gated delta rule — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or run anything in this package. The product
path (``chunkwise_recurrent_prefill_gb300``) never does, and this package never
imports the product path: the two share no code, headers, tables or helpers.

Contents:
  gla_oracle.c   fp64 token-by-token recurrence (plain C, OpenMP over heads).
  gla_ref.py     ctypes binding to it, an independent pure-numpy token loop, and an
                 fp64 numpy restatement of the chunkwise algorithm.
  gdn_oracle.c   the gated delta rule's fp64 token loop in plain C (OpenMP over heads).
  gdn_ref.py     the gated delta rule: fp64 numpy token loop, ctypes binding to the C loop,
                 and the chunk algebra, pinned by
                 ``tests/test_gdn_oracle_pins.py`` (its formula is a reading from outside the
                 pages, which name the method but print no recurrence).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute-force decay-matrix attention, the ungated textbook case, closed forms,
state carry, linearity, exact rational arithmetic). No function is parity-unpinned.
"""
from . import gdn_ref as _gdn_ref
from . import gla_ref as _gla_ref
from .gla_ref import (  # noqa: F401
    recurrent,
    recurrent_head,
    recurrent_np,
    chunkwise_np,
    num_threads,
)


def build(force: bool = False) -> None:
    """Compile every C oracle (gcc, OpenMP) into ``oracle/_build``."""
    _gla_ref.build(force)
    _gdn_ref.build(force)
