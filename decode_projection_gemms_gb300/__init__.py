"""GB300 (sm_103a) decode-time KDA projection GEMMs.

The compute path is ``libkdaproj.so`` (hand-written CUDA, C ABI in
``include/kdaproj.h``); :mod:`.binding` marshals torch tensors into it. Build
the library with :func:`decode_projection_gemms_gb300.build.build`.
"""
from __future__ import annotations

__all__ = ["KdaPlan", "KpCfg", "KdaProjError", "skinny_gemm", "select_config", "make_events",
           "table_load", "table_clear", "device_error", "check_device"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
