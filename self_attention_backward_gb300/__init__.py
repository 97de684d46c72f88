"""GB300-native PSA self-attention backward (lo/hi shared-QK FlashAttention-2
backward) on hand-written sm_103a CUDA kernels behind a C ABI.

The compute path is the shared library built from ``csrc/`` (see ``build.py``);
``binding.py`` marshals torch tensors into its C calls.  Importing this package
does not load the library; the first call does, and fails loudly if it is not
built.
"""
from .inputs import WORKLOADS, WORKLOAD_ORDER, Workload, make_inputs, make_custom  # noqa: F401
