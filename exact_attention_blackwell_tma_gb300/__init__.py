"""GB300-native exact attention (forward and backward) behind a C ABI.

The compute path is the CUDA library ``libattn.so`` built from ``csrc/``;
``binding`` marshals PyTorch tensors into its C entry points. Importing this
package loads nothing: the library is loaded on the first call.
"""
from . import inputs  # noqa: F401  (seeded synthetic inputs; no attention arithmetic)

__all__ = ["inputs"]
