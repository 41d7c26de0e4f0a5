"""libfibatt: Fibottention per-head sparse self-attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libfibatt.so`` (``include/fibatt.h``);
this package only builds it (``build.build_library``) and binds it
(``api``).  Importing the package does not load the library; the first call
does, and fails loudly if it has not been built.
"""
from .api import (FibattError, FibottentionFunction, Support, bwd, fibottention, fwd,
                  window_schedule, wythoff_row, wythoff_row_modified)

__all__ = ["FibattError", "FibottentionFunction", "Support", "bwd", "fibottention", "fwd",
           "window_schedule", "wythoff_row", "wythoff_row_modified"]
