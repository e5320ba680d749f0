"""Selective KV-cache refresh on GB300 (sm_103a).

    selective_kv_cache_gb300.kvr        ctypes binding of libkvr (include/kvr.h)
    selective_kv_cache_gb300.harness    device set-up of a workload (tests, bench)
    selective_kv_cache_gb300.workloads  seeded synthetic inputs
    selective_kv_cache_gb300.build      nvcc build of libkvr.so (in-tree)

Importing the package loads nothing; importing `kvr` loads libkvr.so and fails
if it has not been built.
"""
__version__ = "0.1.0"
