"""GB300 (sm_103a) Kimi Delta Attention prefill / MTP verify.

The compute lives in libkda.so (C ABI, include/kda.h); ``kda`` is its ctypes
binding.  Importing this package loads nothing; the library is loaded on the
first call and its absence is an error, never a fallback.
"""
from .kda import (CHUNK, HEAD_DIM, KdaError, host_staging_size, kda_prefill,  # noqa: F401
                  overrides, prefill_schedule,
                  kda_prefill_host, kda_verify, lib, status_string, workspace_layout,
                  workspace_size)
