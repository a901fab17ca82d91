"""CPU oracle (test infrastructure only).

Importable only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  It shares no code with ``paged_sliding_window_swa_gb300``.
"""
