"""Paged KV cache on GB300: paged decode attention, cache write, block copy and
a host block allocator, behind the C ABI of include/pa.h.

Importing the package loads nothing; the CUDA library is loaded on first use
and its absence is an error (there is no CPU path).
"""
__all__ = ["api", "workloads", "build"]
