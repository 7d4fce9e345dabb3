"""CPU oracle (test infrastructure only).

Imported by the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``; never by the product path.
"""
