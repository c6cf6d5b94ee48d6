"""CPU oracle for the per-FSDP-unit cycle.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import anything here.  The
library never imports it, and it imports nothing from the library.
"""
