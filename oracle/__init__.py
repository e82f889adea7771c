"""CPU oracle for the OScaR decode path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  Nothing in the product path does.
"""
