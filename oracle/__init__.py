"""Float64 CPU oracle of the DSA step (lightning indexer, top-k, sparse absorbed MLA).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg, never by the product path.
It shares no code with the CUDA path; only the seeded input generators in
``workloads.py`` serve both.

Parity pins: every function of ``dsa_oracle`` is pinned by tests that do not
re-use its own formulas (pure-Python brute force in ``brute.py``, the OCP
E4M3 table, library routines, closed forms and invariants); no function is
left "parity unpinned".
"""
from . import dsa_oracle, brute  # noqa: F401
