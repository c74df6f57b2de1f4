"""GB300 (sm_103a) decode step for quantised Llama-architecture models.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/dls.h``); ``dls`` is its ctypes binding.
"""
from . import dls  # noqa: F401
from .dls import DlsError, Model, load  # noqa: F401

__all__ = ["dls", "DlsError", "Model", "load"]
