// Tensor-core (tcgen05) chunked prefills for dk = dv = 128: bf16 operands
// (prefill_tc.cu) and tf32 operands (prefill_tc32.cu).
#pragma once
#include "gdn_common.cuh"

namespace gdn {
bool prefill_tc_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p);
size_t prefill_tc_workspace(const gdn_dims& d, int32_t n_seq, int64_t total);
cudaError_t prefill_tc_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt,
                              const gdn_params& p, const int32_t* slot_ids, const int32_t* cu_seqlens,
                              const int64_t* start_pos, int32_t n_seq, int64_t total,
                              const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                              const void* qkv, const void* a, const void* b, void* out,
                              void* workspace, uint32_t* dev_err, cudaStream_t s);
// The same chunk form with every product in tf32 and the features computed in
// the chain (prefill_tc32.cu): dk = dv = 128, width 4, bf16 activations and
// conv history.  Needs no workspace.
bool prefill_tc32_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p);
// the readout epilogue fused into the output (gdn_chunk_prefill_gated): out
// receives y = o / sqrt(mean(o^2) + eps) * weight * silu(z)
struct Tc32Epilogue {
  const void* z;         // [total][hv][dv] bf16, 16-byte aligned
  const float* weight;   // [dv] fp32, 16-byte aligned
  float eps;
};
cudaError_t prefill_tc32_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                                const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                                int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                                int32_t ckpt_block, const void* qkv, const void* a, const void* b, void* out,
                                uint32_t* dev_err, cudaStream_t s, const Tc32Epilogue* epi = nullptr);
// The single-launch mixed step (prefill_tc32.cu): decode requests as the
// TMA-fed decode items and continuations as tf32 chains plus their conv
// histories, in one persistent launch.  queue: mixed_fused_queue_bytes(n_pre)
// bytes of device memory, 8-byte aligned.
bool mixed_fused_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p);
size_t mixed_fused_queue_bytes(int32_t n_pre);
cudaError_t mixed_fused_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                               const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                               int32_t n_seq, int32_t n_decode, int64_t total, const int32_t* ckpt_ids,
                               int32_t max_ckpt, int32_t ckpt_block, const void* qkv, const void* av,
                               const void* bv, void* out, void* queue, uint32_t* dev_err, cudaStream_t s);
// conv histories of a prefill's checkpoints and final state (prefill.cu)
cudaError_t conv_history_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt,
                                const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                                int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                                int32_t ckpt_block, const void* qkv, uint32_t* dev_err, cudaStream_t s);
}  // namespace gdn
