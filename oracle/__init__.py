"""CPU oracle for the DFlash speculative round (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.
"""
