"""GB300-native Permute + GroupedMatMul (+ shared-expert MatMul) hot path.

The compute runs in liba2av_gmm.so (hand-written sm_103a CUDA kernels behind
a C ABI, include/a2av_gmm.h); ``binding`` marshals torch tensors into it.
"""

from .binding import Plan, a2av_gmm  # noqa: F401
