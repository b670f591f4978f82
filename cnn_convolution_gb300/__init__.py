"""GB300-native forward 2-D convolution (sm_103a CUDA kernels behind a C ABI)."""
from . import conv2d, workloads  # noqa: F401
from .conv2d import Conv2dDesc, Conv2dError, forward  # noqa: F401
