"""Seeded synthetic inputs for the TriAttention eviction pass.

This package is shared by the tests, ``bench.py`` and the smoke check. It
produces caches and calibration statistics; it contains none of the eviction
method's arithmetic (no scoring, normalisation, selection or compaction).

* :mod:`synth.counter_rng` - a counter-based normal generator whose host
  (numpy) and device (CUDA, ``synth/csrc/synth_gen.cu``) forms give identical
  bits, so the oracle can regenerate any segment on the host instead of
  reading device memory.
* :mod:`synth.workloads` - the five workload shapes and their seeds.
"""
from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401
