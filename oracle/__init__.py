"""CPU oracle (test infrastructure only).

Imported by the tests, by ``__graft_entry__.smoke`` and by the benchmark's
CPU-baseline leg — never by the product path.  See ``oracle.model``.
"""
from . import model, philox  # noqa: F401
