"""Speculative Pipeline Decoding on one GB300: the per-cycle hot path as sm_103a CUDA kernels.

The C ABI lives in include/spd.h and the kernels in csrc/; ``binding`` marshals Python and torch
arguments to it.  Build the library with ``build_ext.build()``.
"""
from .binding import (Config, Engine, SpdError, attention, attention_workspace_bytes,  # noqa: F401
                      grouped_gemv, lib, library_path, exported_symbols)
from . import binding  # noqa: F401
