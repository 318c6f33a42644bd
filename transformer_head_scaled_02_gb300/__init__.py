"""GB300-native multi-head attention forward (sm_103a).

The compute path is the C-ABI library ``libmha.so`` built from ``csrc/``; this
package only marshals arguments into it (see ``_lib``) and offers a small
torch-tensor wrapper (``Mha``).  Nothing here computes attention on the CPU:
if the library is missing, loading it raises.
"""
__all__ = ["workloads"]
