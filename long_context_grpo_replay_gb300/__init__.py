"""Exact response-replay attention for long-context GRPO on GB300 (sm_103a).

The compute path is the C-ABI CUDA library ``libls`` (``include/ls.h``); this
package holds its build script (``build.py``), the ctypes binding
(``binding.py``) with one function per C entry point, and the seeded synthetic
input generators (``inputs.py``).  Importing the package does not load the
library; the first binding call does, and fails loudly if it was not built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "binding", "build"]


def __getattr__(name):
    if name in ("binding", "build"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
