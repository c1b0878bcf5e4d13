"""libpagedattn: paged decode attention for sm_103a (GB300).

The compute path is the C-ABI shared library ``libpagedattn`` built from ``csrc/``;
``paged_kv_cache_63_gb300.lib`` is its thin ctypes binding (argument marshalling
only). ``workloads`` draws the seeded synthetic inputs used by tests and benchmarks.
"""

__all__ = ["lib", "workloads"]


def __getattr__(name):
    if name in ("lib", "workloads"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
