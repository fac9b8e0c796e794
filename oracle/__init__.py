"""CPU oracle for the NVFP4 routed-expert MoE layer.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.
The arithmetic lives in ``nvfp4_oracle.c`` (plain C, fp64 sums).
"""
