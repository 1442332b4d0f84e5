"""rwkv_wkv_gb300: the WKV-7 state-slot engine for one GB300 GPU.

The compute lives in libwkv7.so (hand-written CUDA for sm_103a behind a C-ABI,
see include/wkv7.h); this package is its thin Python binding.
"""
from .wkv7 import (BF16, DEV_BAD_SEQLENS, DEV_BAD_SLOT, DEV_DECAY_RANGE, DEV_DUP_SLOT,  # noqa: F401
                   DEV_OK, DEV_WAIT_TIMEOUT, F32, HEAD_SIZE, LIB_PATH, Pool, Wkv7Error,
                   exported_symbols, launch_count, load_library)
