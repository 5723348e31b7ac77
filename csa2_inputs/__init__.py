"""Seeded synthetic input generators (host: numpy; device: ``libcsa2_inputs``).

Shared by the CUDA path's tests and benchmark and by the CPU oracle's tests.  It
contains no arithmetic of the method: only counter-based random draws and the
layout bookkeeping (page tables, slots) of the synthetic workloads.
"""
from .gen import *  # noqa: F401,F403
