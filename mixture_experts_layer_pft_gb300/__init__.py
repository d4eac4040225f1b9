"""Padding-free (PFT) expert-specialised MoE layer for GB300 (sm_103a).

``binding`` holds the Python names of the C ABI (include/moe_pft.h); ``layer`` sequences one
forward + backward step; ``workloads`` draws the seeded synthetic inputs.  The CUDA library
(libmoe_pft.so, built in-tree by ``build.build()``) is loaded on the first call.
"""

from . import workloads  # noqa: F401
