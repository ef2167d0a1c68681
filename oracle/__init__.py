"""CPU oracle for the decode megakernel: forward pass, lowering, DAG validator.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import, call or execute anything here;
the library and its kernels never do, and this package imports nothing from
the library.  Inputs come from ``synth`` (seeded generators only).

Pinned by ``tests/test_oracle_pins.py`` (brute-force loops, closed forms,
invariants, library routines on special cases and the pages' worked values
in ``tests/golden/``).  Nothing here is "parity unpinned".
"""
from . import forward, lowering, validate, graph  # noqa: F401
