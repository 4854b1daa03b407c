"""Routed-expert FFN of one MoE layer for GB300 (sm_103a).

The compute lives in libmoe_gb300.so (C ABI: include/moe.h); this package
holds its ctypes binding (`_lib`), a small device-buffer owner (`layer`), the
adaptive expert cache's planner binding (`cache`), the routing-trace codec
binding (`trace`), the build script (`build`) and the seeded synthetic input
generator (`synth`).
"""
from . import synth  # noqa: F401

__all__ = ["synth", "lib", "layer", "cache", "trace"]


def __getattr__(name):
    if name == "lib":
        from . import _lib
        return _lib
    if name in ("layer", "cache", "trace"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
