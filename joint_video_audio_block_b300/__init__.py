"""B300-native (sm_103a) hot path of the H3 joint audio+video DiT trunk.

The compute lives in libh3.so (CUDA kernels behind the C ABI of include/h3.h); `h3` is its
ctypes binding and `runtime` holds the torch-side conveniences (device buffers, streams).
"""

from . import h3  # noqa: F401
