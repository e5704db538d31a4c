"""GB300-native paged KV cache: slot-mapped append, copy-on-write block copy and
single-token decode attention over block tables, as a C-ABI CUDA library
(``libkvpaged.so``, sm_103a) with a thin ctypes binding.

``abi``    the C entry points, one Python function each (marshalling only)
``cache``  ``PagedKVCache`` (torch-owned device pools) and ``BlockAllocator``
``build``  compiles the library in-tree with nvcc
"""

from . import abi  # noqa: F401

__all__ = ["abi", "build", "cache"]
