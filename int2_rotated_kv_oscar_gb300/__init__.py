"""GB300 (sm_103a) OSCAR INT2 rotated KV cache: write path and fused decode attention.

The compute lives in ``liboscar_gb300.so`` (hand-written CUDA behind the C ABI
in ``include/oscar.h``); ``abi`` is its ctypes binding with the same names.
``cache`` allocates device memory with PyTorch; ``inputs`` draws seeded
synthetic data; ``calibrate`` is the offline host tool that derives the
rotations and clip thresholds.
"""

from . import abi  # noqa: F401
from .abi import (OscarError, oscar_check_device_error, oscar_create, oscar_decode_attention,  # noqa: F401
                  oscar_decode_attention_bf16, oscar_decode_workspace_bytes, oscar_destroy,
                  oscar_device_sm_count, oscar_kv_append, oscar_load_rotation, oscar_status_string)
