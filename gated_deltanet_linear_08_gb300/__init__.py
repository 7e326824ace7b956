"""GB300-native Gated DeltaNet (GDN) linear-attention layer core.

The computation lives in libgdn.so (C ABI, include/gdn.h): a chunked tcgen05
prefill and a streaming decode (single or multi-token, optionally over a pool of
state slots), hand-written CUDA for sm_103a.  This package is
the thin Python binding over that ABI (torch tensors -> device pointers) plus
the build script and the seeded synthetic input generator.
"""
from ._binding import (GdnError, alloc_workspace, check_device_status, conv_prefill, decode, decode_slots, load,
                       prefill, prefill_noalloc, status_string, workspace_bytes)

__all__ = ["GdnError", "alloc_workspace", "check_device_status", "conv_prefill", "decode", "decode_slots", "load",
           "prefill", "prefill_noalloc", "status_string", "workspace_bytes"]
