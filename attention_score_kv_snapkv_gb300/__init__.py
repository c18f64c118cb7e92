"""GB300 (sm_103a) attention-score KV-cache compression: SnapKV, H2O, StreamingLLM.

The compute lives in libkvcompress.so (hand-written CUDA kernels behind the C ABI of
include/kvcompress.h); this package is its thin Python binding.  See _binding for the
entry points, which keep the C names.
"""

from ._binding import (  # noqa: F401
    DEV_BAD_STATE, DEV_CACHE_FULL, DEV_TIMEOUT, H2OState, KVCError, compressed_decode_attn,
    compressed_decode_attn_noalloc,
    h2o_decode_step, h2o_prefill, h2o_prefill_from_votes, h2o_step_ctas_per_unit,
    kvc_device_status, kvc_selftest_wait_timeout, kvc_set_wait_timeout_ns, kvc_version, lib,
    library_path, prefill_attention_lse, sink_window_append, snapkv_compress,
    snapkv_prefill_attention, snapkv_select, snapkv_vote_plan, snapkv_votes_from_lse,
    snapkv_workspace_bytes)
