"""GB300-native DSpark sequential Markov sampling of draft tokens.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/markov.h``); ``api`` is its thin Python binding.  Importing the
package does not load the library: ``api`` loads it on first use and raises
if it is missing, so a missing build fails loudly instead of falling back.
"""
import importlib

from . import workloads  # noqa: F401  (pure input generation, no arithmetic)

__all__ = ["workloads", "api"]


def __getattr__(name):
    if name in ("api", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
