"""GB300-native PTPC-FP8 Mixture-of-Experts layer forward.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (`csrc/`, declared in `include/moe_ptpc.h`); `binding` marshals
torch tensors into those calls. Importing the package loads nothing; the
library is loaded on first use and a missing build raises.
"""

__all__ = ["binding", "synthetic", "build"]
