"""GB300-native tensor-parallel MLP block (Megatron column/row split, all shards on one GPU).

The compute path is the CUDA library ``libtpmlp.so`` (hand-written sm_103a
kernels behind the C ABI declared in ``include/tpmlp.h``).  ``binding``
marshals torch tensors to that ABI; ``inputs`` holds the seeded synthetic
input recipes.  Importing the package loads nothing: the library is opened
on first use and its absence raises instead of falling back to anything.
"""
__all__ = ["binding", "inputs"]
