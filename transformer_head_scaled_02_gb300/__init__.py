"""GB300-native multi-head attention forward (sm_103a).

The compute path is the C-ABI library ``libmha.so`` built from ``csrc/`` (its
interface is ``include/mha.h``).  ``_lib`` binds it with ctypes under the same
names; ``Mha`` (in ``mha``) is a small torch-tensor front end that only
marshals arguments.  Nothing here computes attention on the CPU: if the
library is missing, loading it raises ImportError.

``workloads`` (seeded synthetic inputs) imports neither torch nor the library.
"""

__all__ = ["Mha", "workloads"]


def __getattr__(name):
    if name == "Mha":
        from .mha import Mha
        return Mha
    raise AttributeError(name)
