"""B300-native (sm_103a) forward pass of the GLM MoE feed-forward sublayer.

The compute lives in libmoe_b300.so (hand-written CUDA behind the C ABI of
include/moe.h); this package holds its Python binding, the build script and
the seeded synthetic workloads.
"""
from .binding import MoeSublayer, MoeError, load_library, status_string  # noqa: F401
from .workloads import WORKLOADS, Workload, make_inputs, host_arrays  # noqa: F401
