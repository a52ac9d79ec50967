"""GB300-native sequence-partitioned causal attention (StreamBP / SeCO chunk calls).

The compute path is ``libseqattn.so`` (hand-written sm_103a kernels behind a C
ABI declared in ``include/seqattn.h``).  ``binding`` marshals torch tensors to
that ABI; importing this package does not load the library, the first call
does, and it raises if the library has not been built.
"""

from . import inputs, workloads  # noqa: F401

__all__ = ["inputs", "workloads"]
