// Persistent TMA-fed decode path (dk = 128, conv width 4); see decode_tma.cu.
#pragma once
#include "gdn_common.cuh"

namespace gdn {
// True when the shape, dtypes and pointer alignment fit the TMA-fed kernel.
bool decode_tma_supported(const gdn_dims& d, const void* qkv, const gdn_params& p);
// kda: the per-key-channel decay variant (a [B][hv][dk], dt_bias [hv][dk])
cudaError_t decode_tma_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_params& p,
                              const int32_t* slot_ids, int32_t B, const void* qkv, const void* a,
                              const void* b, void* out, uint32_t* dev_err, bool kda, cudaStream_t s);
// whether gdn_decode_step takes the TMA-fed kernel for batch B
bool decode_takes_tma(const gdn_dims& d, int32_t B, const void* qkv, const gdn_params& p);
int sm_count();
// CTAs per SM for the persistent kernels: 0 = the default choice of each
// kernel, 1 or 2 forced by GDN_TMA_CTAS (for measurement).
int tma_ctas_per_sm();

// Persistent TMA-fed speculative verify (dk = 128, conv width 4, T <= 16);
// kda: the per-key-channel decay variant (a [B][T][hv][dk], dt_bias [hv][dk],
// both 16-byte aligned).
bool verify_tma_supported(const gdn_dims& d, int32_t T, const void* qkv, const gdn_params& p);
cudaError_t verify_tma_launch(const gdn_dims& d, const gdn_pool& work, const gdn_pool& spec,
                              const gdn_params& p, const int32_t* slot_ids, const int32_t* spec_ids,
                              int32_t B, int32_t T, const void* qkv, const void* a, const void* b,
                              void* out, uint32_t* dev_err, bool kda, cudaStream_t s);
}  // namespace gdn
