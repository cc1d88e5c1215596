"""GB300-native Gated DeltaNet slot-pool step: libgdn (sm_103a CUDA kernels
behind a C ABI, declared in include/gdn.h) and its thin Python binding."""
from .binding import (  # noqa: F401
    BF16, F32, DEV_ERR_SLOT_OOB, DEV_ERR_TIMEOUT, K_COMMIT_INDEX, K_DECODE, K_GATED_RMSNORM, K_KDA_DECODE,
    K_KDA_PREFILL, K_KDA_VERIFY, K_MIXED, K_PREFILL,
    K_SLOT_COPY, K_SLOT_ZERO, K_SPEC_COMMIT, K_SPEC_VERIFY, K_STATE_PACK, Dims, GdnError,
    LayerParams, StatePool, chunk_prefill, chunk_prefill_gated, chunk_prefill_noalloc, chunk_prefill_workspace_size,
    decode_step, gated_rmsnorm, kda_decode_step, kda_prefill, kda_spec_verify, selftest_wait_timeout, launch_count, launch_count_reset, launch_counts, load, mixed_step, slot_copy,
    slot_zero, BoundsError, debug_bounds, debug_bounds_take, selftest_bounds,
    spec_commit, spec_commit_index, spec_verify, state_pack, state_record_bytes, state_unpack,
)
