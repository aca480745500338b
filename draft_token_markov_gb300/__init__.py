"""GB300-native DSpark sequential Markov sampling of draft tokens.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/markov.h``); ``api`` is its thin Python binding.  Importing the
package does not load the library: ``api`` loads it on first use and raises
if it is missing, so a missing build fails loudly instead of falling back.
"""
from . import workloads  # noqa: F401  (pure input generation, no arithmetic)

__all__ = ["workloads", "api"]


def __getattr__(name):
    if name == "api":
        from . import api
        return api
    raise AttributeError(name)
