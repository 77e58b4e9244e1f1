"""GB300-native memory-efficient biased Evoformer attention.

``evo_attn`` holds the ctypes binding to the sm_103a C-ABI library
(``libevo_attn.so``); ``workload`` the seeded synthetic inputs.  Importing the
package does not load the library; the first binding call does, and fails
loudly if it has not been built.
"""
from . import workload  # noqa: F401

__all__ = ["workload"]
