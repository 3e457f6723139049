"""B300-native MoE layer forward: route -> permute -> grouped FFN -> combine.

The compute lives in ``libmoe_b300.so`` (hand-written sm_103a CUDA behind a
C ABI, declared in ``include/moe.h``). ``binding`` marshals torch tensors to
that ABI and raises if the library or a GPU is missing; there is no CPU path.
Importing this package loads nothing; the library is opened on first use.
"""
__all__ = ["binding", "accounting"]
