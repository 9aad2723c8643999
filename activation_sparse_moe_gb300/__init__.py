"""GB300-native activation-sparse decode/prefill of a ReLU^2 MoE layer.

The compute path is libhs.so (CUDA for sm_103a, C ABI in include/hs.h); this
package holds its build script, its ctypes binding (`hs`), a helper that
uploads checkpoint-layout experts and repacks them on the device (`layer`),
and the byte model used to report achieved bandwidth (`bytemodel`).
"""
from . import hs  # noqa: F401

__all__ = ["hs"]
