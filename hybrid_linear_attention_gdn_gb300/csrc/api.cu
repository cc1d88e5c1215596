// Host-side pieces shared by all entry points: argument checks, status
// strings and launch counters.
#include "gdn_common.cuh"

#include <cstdio>

namespace gdn {

std::atomic<uint64_t> g_launches[GDN_K_COUNT];

namespace {
struct BoundsUnit {
  const char* unit;
  BoundsReader read;
};
// filled by static initialisers of the checked build's units (no locking:
// they run before the library is usable)
BoundsUnit g_bounds_units[32];
int g_n_bounds_units = 0;
}  // namespace

void register_bounds_reader(const char* unit, BoundsReader r) {
  if (g_n_bounds_units < 32) g_bounds_units[g_n_bounds_units++] = BoundsUnit{unit, r};
}

gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_INVALID_ARG;
  if (d->hk <= 0 || d->hv <= 0 || d->dk <= 0 || d->dv <= 0 || d->conv_width <= 0)
    return GDN_ERR_INVALID_ARG;
  if (d->hv % d->hk) return GDN_ERR_INVALID_ARG;
  if (d->act_dtype != GDN_F32 && d->act_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (d->conv_dtype != GDN_F32 && d->conv_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (d->dk != 16 && d->dk != 64 && d->dk != 128) return GDN_ERR_UNSUPPORTED;
  if (d->dv > 256) return GDN_ERR_UNSUPPORTED;
  if (d->conv_width < 2 || d->conv_width > 8) return GDN_ERR_UNSUPPORTED;
  if (d->act_dtype == GDN_F32 && d->conv_dtype == GDN_BF16) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

gdn_status check_pool(const gdn_dims& d, const gdn_pool& p) {
  if (p.num_slots < 0) return GDN_ERR_INVALID_ARG;
  if (p.num_slots == 0) return GDN_OK;
  if (!p.ssm || !p.conv) return GDN_ERR_INVALID_ARG;
  if (!aligned(p.ssm, 16) || !aligned(p.conv, 16)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // namespace gdn

extern "C" const char* gdn_status_string(int32_t s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_SCRATCH_LIMIT: return "GDN_ERR_SCRATCH_LIMIT";
    default: return "GDN_UNKNOWN_STATUS";
  }
}

extern "C" uint64_t gdn_launch_count(int32_t k) {
  if (k < 0 || k >= GDN_K_COUNT) return 0;
  return gdn::g_launches[k].load(std::memory_order_relaxed);
}

extern "C" void gdn_launch_count_reset(void) {
  for (int k = 0; k < GDN_K_COUNT; ++k) gdn::g_launches[k].store(0);
}

extern "C" gdn_status gdn_debug_bounds_take(uint32_t* count, char* where, size_t where_len, int64_t* index,
                                           int64_t* limit) {
#ifndef GDN_DEBUG_BOUNDS
  (void)count, (void)where, (void)where_len, (void)index, (void)limit;
  return GDN_ERR_UNSUPPORTED;
#else
  if (!count) return GDN_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return GDN_ERR_CUDA;
  *count = 0;
  if (where && where_len) where[0] = 0;
  bool first = true;
  for (int u = 0; u < gdn::g_n_bounds_units; ++u) {
    gdn::BoundsWord w;
    if (!gdn::g_bounds_units[u].read(&w)) return GDN_ERR_CUDA;
    if (!w.count) continue;
    *count += w.count;
    if (first) {
      first = false;
      static const char* kinds[3] = {"global", "shared", "TMEM"};
      if (where && where_len)
        snprintf(where, where_len, "%s:%d %s", gdn::g_bounds_units[u].unit, w.line,
                 (w.kind >= 0 && w.kind < 3) ? kinds[w.kind] : "?");
      if (index) *index = w.index;
      if (limit) *limit = w.limit;
    }
  }
  return GDN_OK;
#endif
}
