// KDA prefill in the chunked form on the tensor cores (tcgen05, tf32 state
// products; dk = dv = 128, conv width 4, bf16); see kda_tc32.cu.
#pragma once
#include "gdn_common.cuh"

namespace gdn {
bool kda_tc32_supported(const gdn_dims& d, const void* qkv, const void* a, const void* out, const gdn_params& p);
// the recurrence (outputs, checkpoint and final SSM states); the conv
// histories come from the prefill's history kernel, launched by the caller
cudaError_t kda_tc32_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                            const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                            int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                            int32_t ckpt_block, const void* qkv, const void* a, const void* b, void* out,
                            uint32_t* dev_err, cudaStream_t s);
}  // namespace gdn
