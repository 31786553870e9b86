"""Mixed-format (FP8 / TQ3) paged decode attention for GB300 (sm_103a).

The compute path is the CUDA library ``libmkv.so`` (C ABI in
``include/mkv.h``); this package only marshals arguments to it.  The first
call into the library loads it and raises ImportError if it has not been
built (``python -m mixed_format_paged_gb300.build``): there is no fallback.
"""
from . import binding
from .binding import *  # noqa: F401,F403  (the C-ABI names)
from .pool import MkvPool

__all__ = ["binding", "MkvPool"] + binding.EXPORTED
