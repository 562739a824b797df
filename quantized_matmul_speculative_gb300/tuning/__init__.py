"""Benchmark sweep behind the dispatch table (see sweep.py and make_table.py)."""
