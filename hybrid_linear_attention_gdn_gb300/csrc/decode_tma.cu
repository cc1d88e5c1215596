// Persistent, TMA-fed GDN decode step (dk = 128, conv width 4).
//
// One CTA per SM (or two) walks a static list of work items, each one
// request and one QK head with the G V heads that read it; the item's work
// (a producer lane streaming its bundle and state rows through a ring of
// shared-memory stages, eight consumer warps running the gated delta rule on
// them) is in decode_tma_item.cuh, shared with the single-launch mixed step.
#include "gdn_common.cuh"
#include "decode_tma.cuh"
#include "decode_tma_item.cuh"

#include <cstddef>
#include <cstdlib>

namespace gdn {
namespace {

using namespace dtma;

template <typename Tact, typename Tconv, int STAGES, int MINB, bool KDA>
__global__ void __launch_bounds__(kThr, MINB) decode_tma_kernel(const TmaArgs a) {
  using SM = TmaSmem<Tact, Tconv, STAGES, KDA>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SM& S = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  volatile int* abort_flag = &S.abort;
  [[maybe_unused]] const int nreq = a.n_items / a.hk;
  if (tid == 0) init_barriers<SM, STAGES>(S);
  __syncthreads();
  // programmatic dependent launch: everything above touches only this CTA's
  // shared memory
  pdl_wait();
  pdl_trigger();

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    uint32_t n = 0, vk = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
      const int r = item / a.hk, hq = item % a.hk;
      const int32_t slot = a.slot_ids[GDN_G(r, nreq)];
      if (slot_class(slot, a.num_slots)) continue;
      if (*abort_flag) break;
      ok = produce_item<Tact, Tconv, STAGES, KDA>(a, S, r, hq, slot, vk, n);
    }
    if (!ok || *abort_flag) producer_drain<SM, STAGES>(a, S, vk, n);
    return;
  }

  // -------------------------------------------------------------- consumers
  uint32_t n = 0, vk = 0;
  int item = blockIdx.x;
  int32_t slot_next = item < a.n_items ? a.slot_ids[GDN_G(item / a.hk, nreq)] : -1;
  for (; item < a.n_items; item += gridDim.x) {
    const int r = item / a.hk, hq = item % a.hk;
    const int32_t slot = slot_next;
    const int nitem = item + gridDim.x;
    if (nitem < a.n_items) slot_next = a.slot_ids[GDN_G(nitem / a.hk, nreq)];
    const int cls = slot_class(slot, a.num_slots);
    if (cls) {
      consume_skipped<Tact>(a, r, hq, cls);
      continue;
    }
    const int bb = vk & 1;
    if (!*abort_flag && !mbar_wait(&S.bfull[bb], (vk >> 1) & 1)) *abort_flag = 1;
    named_sync(kBarCons, kCons);
    if (*abort_flag) break;
    ++vk;
    if (!consume_bundle<Tact, Tconv, STAGES, KDA>(a, S, r, hq, slot, bb, n)) break;
  }
  if (*abort_flag && tid == 0) report(a.err, GDN_DEV_ERR_TIMEOUT);
}

template <typename Tact, typename Tconv, int STAGES, int MINB, bool KDA>
cudaError_t launch_tma(const TmaArgs& a, cudaStream_t s) {
  using SM = TmaSmem<Tact, Tconv, STAGES, KDA>;
  static_assert(bundle_aligned<Tact, Tconv, STAGES, KDA>(), "bulk-copy destinations must be 16-byte aligned");
  static_assert(vectors_aligned<Tact, Tconv, STAGES, KDA>(), "float4 reads must be 16-byte aligned");
  auto k = decode_tma_kernel<Tact, Tconv, STAGES, MINB, KDA>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SM));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int slots = sm_count() * MINB;
  const int grid = a.n_items < slots ? a.n_items : slots;
  return launch_pdl(k, dim3((unsigned)grid), dim3(kThr), sizeof(SM), s, dim3(1), a);
}

// One CTA per SM with a 10-stage ring, or two per SM with 4 stages each (one
// CTA's item prologue then overlaps the other's state stream).  Measured on
// the Qwen3.5-shaped layer: two per SM is better below ~6 items per SM (batch
// 32: 0.76 vs 0.71 of HBM peak; batch 48: 0.82 vs 0.80), one per SM above
// (batch 64: 0.88 vs 0.83; batch 128: 0.93 vs 0.89).
template <typename Tact, typename Tconv>
cudaError_t launch_tma_dt(const TmaArgs& a, bool kda, cudaStream_t s) {
  const int forced = tma_ctas_per_sm();
  const bool two = forced ? forced == 2 : a.n_items < 6 * sm_count();
  if (kda) return two ? launch_tma<Tact, Tconv, 4, 2, true>(a, s) : launch_tma<Tact, Tconv, 10, 1, true>(a, s);
  return two ? launch_tma<Tact, Tconv, 4, 2, false>(a, s) : launch_tma<Tact, Tconv, 10, 1, false>(a, s);
}

}  // namespace

int tma_ctas_per_sm() {  // read on every call, so a process can time both
  const char* e = std::getenv("GDN_TMA_CTAS");
  return (e && e[0] == '2') ? 2 : (e && e[0] == '1') ? 1 : 0;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

bool decode_tma_supported(const gdn_dims& d, const void* qkv, const gdn_params& p) {
  const size_t ea = dtype_size(d.act_dtype), ec = dtype_size(d.conv_dtype);
  const int64_t C = channels(d);
  const int G = d.hv / d.hk;
  if (d.dk != kDK || d.conv_width != kW) return false;
  if (d.dv % kRows || G * d.dv > kMaxGR) return false;
  if ((C * ea) % 16 || (C * ec) % 16) return false;
  if ((kDK * ea) % 16 || (kDK * ec) % 16 || ((size_t)G * d.dv * ea) % 16 || ((size_t)G * d.dv * ec) % 16)
    return false;
  if (!aligned(qkv, 16) || !aligned(p.conv_w, 16)) return false;
  return true;
}

cudaError_t decode_tma_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_params& p,
                              const int32_t* slot_ids, int32_t B, const void* qkv, const void* av,
                              const void* bv, void* out, uint32_t* dev_err, bool kda, cudaStream_t s) {
  TmaArgs a;
  a.ssm = pool.ssm;
  a.conv = pool.conv;
  a.num_slots = pool.num_slots;
  a.conv_w = p.conv_w;
  a.A_log = p.A_log;
  a.dt_bias = p.dt_bias;
  a.slot_ids = slot_ids;
  a.qkv = qkv;
  a.a = av;
  a.b = bv;
  a.out = out;
  a.err = dev_err;
  a.hk = d.hk;
  a.hv = d.hv;
  a.dv = d.dv;
  a.C = (int32_t)channels(d);
  a.G = d.hv / d.hk;
  a.n_items = B * d.hk;
  if (d.act_dtype == GDN_BF16 && d.conv_dtype == GDN_BF16)
    return launch_tma_dt<__nv_bfloat16, __nv_bfloat16>(a, kda, s);
  if (d.act_dtype == GDN_BF16) return launch_tma_dt<__nv_bfloat16, float>(a, kda, s);
  return launch_tma_dt<float, float>(a, kda, s);
}

}  // namespace gdn
