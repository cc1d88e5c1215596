// Slot copy-on-write, slot zeroing, speculative commit (by copy or by index),
// and state pack / unpack.
//
// TokenSpeed Qwen3.5 page, "Riesgo de correctitud: estado obsoleto": the
// allocator hands out slot ids without clearing GPU memory, so a new working
// slot is safe only after a copy from a clean checkpoint or an explicit zero.
// "Scheduler dual": the spec_cache snapshot of the accepted draft step becomes
// the working state (rollback = keep the working slot).
//
// "Disaggregacion Prefill-Decode": slot states travel as contiguous records
// (pack: slots -> records; unpack: records -> slots).
//
// The data moves are pure HBM streams: each CTA moves one 32 KiB piece of one
// slot (SSM bytes followed by the conv history, viewed as one byte range) with
// 128-bit accesses, 8 in flight per thread before the first store.  A staging
// record is the same byte range, stored contiguously.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;                              // uint4 per thread
constexpr size_t kPiece = (size_t)kThreads * kVec * 16;  // bytes per CTA

enum { MODE_COPY = 0, MODE_ZERO = 1, MODE_COMMIT = 2, MODE_PACK = 3, MODE_UNPACK = 4 };

struct SlotOpArgs {
  const char* src_ssm;
  const char* src_conv;
  int32_t src_n;
  char* dst_ssm;
  char* dst_conv;
  int32_t dst_n;
  size_t ssm_bytes;   // per slot
  size_t conv_bytes;  // per slot
  size_t src_sstride, src_cstride;  // bytes between consecutive slots / records
  size_t dst_sstride, dst_cstride;
  const int32_t* src_ids;     // copy, pack: [n]; commit: spec ids [n][T]
  const int32_t* dst_ids;     // copy, zero, commit, unpack: [n]
  const int32_t* accept_len;  // commit: [n]
  int32_t T;
  int32_t n;
  uint32_t* err;
};

// bytes from the first to the end of the last of `n` slots (or records) of
// `part` bytes each, `stride` bytes apart
__device__ __forceinline__ long long slots_extent(int32_t n, size_t stride, size_t part) {
  return n > 0 ? (long long)((size_t)(n - 1) * stride + part) : 0;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) slot_op_kernel(SlotOpArgs a) {
  pdl_wait();
  pdl_trigger();
  const bool leader = blockIdx.x == 0 && threadIdx.x == 0;
  const size_t total = a.ssm_bytes + a.conv_bytes;
  // the two sides in 16-byte units, and the id arrays
  const auto src_ssm = GDN_GV(reinterpret_cast<const uint4*>(a.src_ssm),
                              slots_extent(a.src_n, a.src_sstride, a.ssm_bytes) / 16);
  const auto src_conv = GDN_GV(reinterpret_cast<const uint4*>(a.src_conv),
                               slots_extent(a.src_n, a.src_cstride, a.conv_bytes) / 16);
  const auto dst_ssm = GDN_GV(reinterpret_cast<uint4*>(a.dst_ssm), slots_extent(a.dst_n, a.dst_sstride, a.ssm_bytes) / 16);
  const auto dst_conv =
      GDN_GV(reinterpret_cast<uint4*>(a.dst_conv), slots_extent(a.dst_n, a.dst_cstride, a.conv_bytes) / 16);
  const auto src_ids = GDN_GV(a.src_ids, (long long)a.n * (MODE == MODE_COMMIT ? a.T : 1));
  const auto dst_ids = GDN_GV(a.dst_ids, a.n);
  const auto accept_len = GDN_GV(a.accept_len, a.n);
  for (int32_t r = blockIdx.y; r < a.n; r += gridDim.y) {
    int32_t src = 0, dst;
    if (MODE == MODE_COMMIT) {
      const int32_t L = accept_len[r];
      if (L < 0 || L > a.T) {
        if (leader) report(a.err, GDN_DEV_ERR_SLOT_OOB);
        continue;
      }
      if (L == 0) continue;
      src = src_ids[(size_t)r * a.T + (L - 1)];
    } else if (MODE == MODE_COPY || MODE == MODE_PACK) {
      src = src_ids[r];
    } else if (MODE == MODE_UNPACK) {
      src = r;
    }
    dst = MODE == MODE_PACK ? r : dst_ids[r];
    const int cd = slot_class(dst, a.dst_n);
    const int cs = MODE == MODE_ZERO ? 0 : slot_class(src, a.src_n);
    // pack writes a zero record for a padding or out-of-range id
    const bool zero_fill = MODE == MODE_ZERO || (MODE == MODE_PACK && cs != 0);
    if ((cd | cs) && !(MODE == MODE_PACK && cd == 0)) {
      if ((cd == 2 || cs == 2) && leader) report(a.err, GDN_DEV_ERR_SLOT_OOB);
      continue;
    }
    if (MODE == MODE_PACK && cs == 2 && leader) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    const size_t begin = (size_t)blockIdx.x * kPiece;
    if (begin >= total) continue;
    // byte offsets of this slot's (record's) two parts
    const size_t dss = (size_t)dst * a.dst_sstride, dcs = (size_t)dst * a.dst_cstride;
    const size_t sss = (size_t)src * a.src_sstride, scs = (size_t)src * a.src_cstride;
    uint4 v[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const size_t off = begin + ((size_t)i * kThreads + threadIdx.x) * 16;
      v[i] = make_uint4(0, 0, 0, 0);
      if (!zero_fill && off < total)
        v[i] = off < a.ssm_bytes ? src_ssm[(sss + off) / 16] : src_conv[(scs + off - a.ssm_bytes) / 16];
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const size_t off = begin + ((size_t)i * kThreads + threadIdx.x) * 16;
      if (off < total)
        __stcs(off < a.ssm_bytes ? dst_ssm.at((dss + off) / 16) : dst_conv.at((dcs + off - a.ssm_bytes) / 16), v[i]);
    }
  }
}

gdn_status launch_slot_op(int mode, const gdn_dims* dims, const gdn_pool* src,
                          const gdn_pool& dst, const int32_t* src_ids,
                          const int32_t* dst_ids, const int32_t* accept_len,
                          int32_t T, int32_t n, uint32_t* dev_err, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n < 0) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  if ((st = check_pool(*dims, dst)) != GDN_OK) return st;
  if (src && (st = check_pool(*dims, *src)) != GDN_OK) return st;
  if (!dst_ids || (mode != MODE_ZERO && !src_ids)) return GDN_ERR_INVALID_ARG;
  if (mode == MODE_COMMIT && (!accept_len || T <= 0)) return GDN_ERR_INVALID_ARG;
  SlotOpArgs a;
  a.ssm_bytes = ssm_slot_bytes(*dims);
  a.conv_bytes = conv_slot_bytes(*dims);
  if (a.ssm_bytes % 16 || a.conv_bytes % 16) return GDN_ERR_UNSUPPORTED;
  a.src_sstride = a.dst_sstride = a.ssm_bytes;
  a.src_cstride = a.dst_cstride = a.conv_bytes;
  a.src_ssm = src ? reinterpret_cast<const char*>(src->ssm) : nullptr;
  a.src_conv = src ? reinterpret_cast<const char*>(src->conv) : nullptr;
  a.src_n = src ? src->num_slots : 0;
  a.dst_ssm = reinterpret_cast<char*>(dst.ssm);
  a.dst_conv = reinterpret_cast<char*>(dst.conv);
  a.dst_n = dst.num_slots;
  a.src_ids = src_ids;
  a.dst_ids = dst_ids;
  a.accept_len = accept_len;
  a.T = T;
  a.n = n;
  a.err = dev_err;
  const size_t pieces = (a.ssm_bytes + a.conv_bytes + kPiece - 1) / kPiece;
  dim3 grid((unsigned)pieces, (unsigned)(n < 65535 ? n : 65535));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (mode == MODE_COPY) {
    e = launch_pdl(slot_op_kernel<MODE_COPY>, dim3(grid), dim3(kThreads), 0, s, dim3(1), a);
    count_launch(GDN_K_SLOT_COPY);
  } else if (mode == MODE_ZERO) {
    e = launch_pdl(slot_op_kernel<MODE_ZERO>, dim3(grid), dim3(kThreads), 0, s, dim3(1), a);
    count_launch(GDN_K_SLOT_ZERO);
  } else {
    e = launch_pdl(slot_op_kernel<MODE_COMMIT>, dim3(grid), dim3(kThreads), 0, s, dim3(1), a);
    count_launch(GDN_K_SPEC_COMMIT);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Pack (pool -> staging records) or unpack (staging records -> pool).  The
// staging side is addressed by record index r, with both halves of a record
// at a stride of one whole record.
gdn_status launch_state_xfer(bool pack, const gdn_dims* dims, const gdn_pool& pool,
                             const int32_t* ids, int32_t n, const void* staging,
                             size_t staging_bytes, uint32_t* dev_err, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n < 0) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  if ((st = check_pool(*dims, pool)) != GDN_OK) return st;
  if (!ids || !staging) return GDN_ERR_INVALID_ARG;
  SlotOpArgs a;
  a.ssm_bytes = ssm_slot_bytes(*dims);
  a.conv_bytes = conv_slot_bytes(*dims);
  if (a.ssm_bytes % 16 || a.conv_bytes % 16) return GDN_ERR_UNSUPPORTED;
  const size_t rec = a.ssm_bytes + a.conv_bytes;
  if (reinterpret_cast<uintptr_t>(staging) % 16) return GDN_ERR_INVALID_ARG;
  if (staging_bytes / rec < (size_t)n) return GDN_ERR_INVALID_ARG;
  char* st_ssm = const_cast<char*>(reinterpret_cast<const char*>(staging));
  char* st_conv = st_ssm + a.ssm_bytes;
  if (pack) {
    a.src_ssm = reinterpret_cast<const char*>(pool.ssm);
    a.src_conv = reinterpret_cast<const char*>(pool.conv);
    a.src_n = pool.num_slots;
    a.src_sstride = a.ssm_bytes;
    a.src_cstride = a.conv_bytes;
    a.dst_ssm = st_ssm;
    a.dst_conv = st_conv;
    a.dst_n = n;
    a.dst_sstride = a.dst_cstride = rec;
    a.src_ids = ids;
    a.dst_ids = nullptr;
  } else {
    a.src_ssm = st_ssm;
    a.src_conv = st_conv;
    a.src_n = n;
    a.src_sstride = a.src_cstride = rec;
    a.dst_ssm = reinterpret_cast<char*>(pool.ssm);
    a.dst_conv = reinterpret_cast<char*>(pool.conv);
    a.dst_n = pool.num_slots;
    a.dst_sstride = a.ssm_bytes;
    a.dst_cstride = a.conv_bytes;
    a.src_ids = nullptr;
    a.dst_ids = ids;
  }
  a.accept_len = nullptr;
  a.T = 0;
  a.n = n;
  a.err = dev_err;
  const size_t pieces = (rec + kPiece - 1) / kPiece;
  dim3 grid((unsigned)pieces, (unsigned)(n < 65535 ? n : 65535));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e =
      pack ? launch_pdl(slot_op_kernel<MODE_PACK>, grid, dim3(kThreads), 0, s, dim3(1), a)
           : launch_pdl(slot_op_kernel<MODE_UNPACK>, grid, dim3(kThreads), 0, s, dim3(1), a);
  count_launch(GDN_K_STATE_PACK);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Index-update commit: one thread per request; only int32 indices move.
constexpr int kIdxThreads = 128;

__global__ void __launch_bounds__(kIdxThreads)
    commit_index_kernel(const int32_t* __restrict__ spec_ids,
                        const int32_t* __restrict__ accept_len, int32_t* __restrict__ slot_ids,
                        int32_t* __restrict__ freed, int32_t B, int32_t T, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int32_t r = blockIdx.x * kIdxThreads + threadIdx.x;
  if (r >= B) return;
  const long long BT = (long long)B * T;
  const auto sp = GDN_GV(spec_ids, BT) + (size_t)r * T;
  const auto fr = GDN_GV(freed, BT) + (size_t)r * T;
  const auto slots = GDN_GV(slot_ids, B);
  const int32_t L = GDN_GV(accept_len, B)[r];
  if (L == 0) {
    for (int32_t t = 0; t < T; ++t) fr[t] = sp[t];
    return;
  }
  const int32_t acc = (L >= 1 && L <= T) ? sp[L - 1] : -1;
  if (acc < 0) {
    report(err, GDN_DEV_ERR_SLOT_OOB);
    for (int32_t t = 0; t < T; ++t) fr[t] = -1;
    return;
  }
  fr[0] = slots[r];
  int32_t k = 1;
  for (int32_t t = 0; t < T; ++t)
    if (t != L - 1) fr[k++] = sp[t];
  slots[r] = acc;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_slot_copy(const gdn_dims* dims, gdn_pool src, gdn_pool dst,
                                    const int32_t* src_ids, const int32_t* dst_ids,
                                    int32_t n, uint32_t* dev_err, void* stream) {
  return gdn::launch_slot_op(gdn::MODE_COPY, dims, &src, dst, src_ids, dst_ids,
                             nullptr, 0, n, dev_err, stream);
}

extern "C" gdn_status gdn_slot_zero(const gdn_dims* dims, gdn_pool pool, const int32_t* ids,
                                    int32_t n, uint32_t* dev_err, void* stream) {
  return gdn::launch_slot_op(gdn::MODE_ZERO, dims, nullptr, pool, nullptr, ids, nullptr,
                             0, n, dev_err, stream);
}

extern "C" gdn_status gdn_spec_commit(const gdn_dims* dims, gdn_pool spec, gdn_pool work,
                                      const int32_t* spec_ids, const int32_t* accept_len,
                                      const int32_t* slot_ids, int32_t B, int32_t T,
                                      uint32_t* dev_err, void* stream) {
  return gdn::launch_slot_op(gdn::MODE_COMMIT, dims, &spec, work, spec_ids, slot_ids,
                             accept_len, T, B, dev_err, stream);
}

extern "C" gdn_status gdn_spec_commit_index(const int32_t* spec_ids, const int32_t* accept_len,
                                            int32_t* slot_ids, int32_t* freed_ids, int32_t B,
                                            int32_t T, uint32_t* dev_err, void* stream) {
  if (B < 0 || T < 1) return GDN_ERR_INVALID_ARG;
  if (B == 0) return GDN_OK;
  if (!spec_ids || !accept_len || !slot_ids || !freed_ids) return GDN_ERR_INVALID_ARG;
  const unsigned blocks = (unsigned)((B + gdn::kIdxThreads - 1) / gdn::kIdxThreads);
  cudaError_t e = gdn::launch_pdl(gdn::commit_index_kernel, dim3(blocks), dim3(gdn::kIdxThreads),
                                  0, reinterpret_cast<cudaStream_t>(stream), dim3(1), spec_ids,
                                  accept_len, slot_ids, freed_ids, B, T, dev_err);
  gdn::count_launch(GDN_K_COMMIT_INDEX);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" size_t gdn_state_record_bytes(const gdn_dims* dims) {
  if (gdn::check_dims(dims) != GDN_OK) return 0;
  return gdn::ssm_slot_bytes(*dims) + gdn::conv_slot_bytes(*dims);
}

extern "C" gdn_status gdn_state_pack(const gdn_dims* dims, gdn_pool pool, const int32_t* ids,
                                     int32_t n, void* staging, size_t staging_bytes,
                                     uint32_t* dev_err, void* stream) {
  return gdn::launch_state_xfer(true, dims, pool, ids, n, staging, staging_bytes, dev_err,
                                stream);
}

extern "C" gdn_status gdn_state_unpack(const gdn_dims* dims, const void* staging,
                                       size_t staging_bytes, gdn_pool pool, const int32_t* ids,
                                       int32_t n, uint32_t* dev_err, void* stream) {
  return gdn::launch_state_xfer(false, dims, pool, ids, n, staging, staging_bytes, dev_err,
                                stream);
}

// ---------------------------------------------------------------------------
// Self-test of the bounded waits that every mbarrier-fed kernel here relies on:
// one CTA waits on a barrier phase that nothing completes; the wait gives up
// after the library's limit (kWaitLimitNs), the kernel records
// GDN_DEV_ERR_TIMEOUT and returns, and the context stays usable.
// ---------------------------------------------------------------------------
namespace gdn {
namespace {
__global__ void wait_selftest_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) report(err, GDN_DEV_ERR_TIMEOUT);
}

#ifdef GDN_DEBUG_BOUNDS
// Positive control of the checked build: one thread indexes a global and a
// shared view one element past their declared extents and asks for a span
// that ends past its view.  Each view covers only the first half of its
// buffer, so even an index that escaped its check would stay inside real
// memory; with the checks working, the two indices go to the scratch buffer
// and the span is refused.
__device__ int g_bounds_probe[8];
__global__ void bounds_selftest_kernel() {
  __shared__ int probe[8];
  if (threadIdx.x != 0) return;
  const auto gv = GDN_GV(g_bounds_probe, 4);
  gv[4] = 1;
  const auto sv = GDN_SV(probe, 4);
  sv[4] = 1;
  if (gv.has(2, 4)) g_bounds_probe[0] = probe[4];
}
#endif
}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_wait_timeout(uint32_t* dev_err, void* stream) {
  using namespace gdn;
  if (!dev_err) return GDN_ERR_INVALID_ARG;
  const cudaError_t e = launch_plain(wait_selftest_kernel, dim3(1), dim3(32), 0,
                                     reinterpret_cast<cudaStream_t>(stream), dim3(1), dev_err);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_bounds(void* stream) {
#ifdef GDN_DEBUG_BOUNDS
  const cudaError_t e = gdn::launch_plain(gdn::bounds_selftest_kernel, dim3(1), dim3(32), 0,
                                          reinterpret_cast<cudaStream_t>(stream), dim3(1));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
#else
  (void)stream;
  return GDN_ERR_UNSUPPORTED;
#endif
}
