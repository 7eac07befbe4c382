"""kvring for GB300: a write-time FP8 ring KV cache and the attention that reads it.

The compute path is ``libkvring.so`` (CUDA kernels for sm_103a behind the C ABI
of ``include/kvring.h``); ``fp8_ring_kv_gb300.kvring`` is its ctypes binding.
"""
from .kvring import (KVRing, KVRingError, KVRingStack, kvring_reset_positions_batch, kvring_attend, kvring_attend_noalloc, kvring_create, kvring_destroy,  # noqa: F401,E501
                     kvring_calibrate, kvring_reset_positions, kvring_set_qk_norm, kvring_workspace_bytes,
                     kvring_write, kvring_write_global, load, make_config)
