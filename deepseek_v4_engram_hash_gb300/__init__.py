"""GB300-native DeepSeek-V4.1 engram forward: n-gram hash -> table rows ->
wkv projection -> gate, as sm_103a CUDA kernels behind the libengram C ABI
(include/engram.h).  PyTorch supplies device memory and streams only."""
from . import configs  # noqa: F401
