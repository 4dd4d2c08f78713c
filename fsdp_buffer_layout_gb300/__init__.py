"""GB300-native shard step of structure-aware FSDP (RaggedShard layout,
planned distributed buffer, block-wise 8-bit AdamW) behind the C ABI of
libvsf (include/vsf.h).

``vsf`` is the ctypes binding (same names as the C functions); ``step``
holds ``ShardStep``, which owns torch-allocated device buffers for one plan
and calls the four per-step entry points.
"""
from . import vsf  # noqa: F401
from ._build import build  # noqa: F401

__all__ = ["vsf", "build"]
