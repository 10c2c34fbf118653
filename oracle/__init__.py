"""fp64 CPU oracle of the tensor-parallel MLP block and the sequence-parallel
LayerNorm.

TEST INFRASTRUCTURE: imported only by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg.  The library never imports it, and it
imports nothing from the library.  Parity status of every function is pinned
by ``tests/test_oracle_pins.py`` (see the design notes for the list of pins).
"""
from . import bf16, mlp, layernorm  # noqa: F401
