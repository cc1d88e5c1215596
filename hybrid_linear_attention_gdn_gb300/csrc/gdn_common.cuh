// Shared helpers for the libgdn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstdlib>
#include <utility>

#include "gdn.h"

namespace gdn {

// ---- element conversion ---------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---- streaming 128-bit global access (data touched once per launch) --------
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// ---- device error word ----------------------------------------------------
__device__ __forceinline__ void report(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// ---- bounds-checked build ----------------------------------------------------
// Compiled with -DGDN_DEBUG_BOUNDS (the separate libgdn_debug.so), every
// computed index of the kernels goes through one of the checks below: global
// (GDN_G), shared (GDN_S) and TMEM (GDN_T) element indices, and spans of bulk
// copies (GDN_SPAN_G / GDN_SPAN_S).  An index outside its buffer is recorded
// in this translation unit's bounds word (how many, and the first one's line,
// kind, index and limit); the access is then redirected to element 0 (an
// index) or skipped (a span), so a failing check neither faults nor traps.
// The host reads and clears the words with gdn_debug_bounds_take().  In the
// normal build every check is the identity and compiles away.
struct BoundsWord {
  unsigned int count;
  int line, kind;  // kind: 0 global, 1 shared, 2 TMEM
  long long index, limit;
};
#ifdef GDN_DEBUG_BOUNDS
#ifndef GDN_TU
#define GDN_TU "?"
#endif
namespace {
__device__ BoundsWord g_bounds_word;
__device__ __noinline__ void bounds_fail(int line, int kind, long long i, long long n) {
  if (atomicAdd(&g_bounds_word.count, 1u) == 0) {
    g_bounds_word.line = line;
    g_bounds_word.kind = kind;
    g_bounds_word.index = i;
    g_bounds_word.limit = n;
  }
}
template <typename I>
__device__ __forceinline__ I bounds_ix(I i, long long n, int line, int kind) {
  if ((unsigned long long)(long long)i < (unsigned long long)n) return i;
  bounds_fail(line, kind, (long long)i, n);
  return I(0);
}
// [off, off + len) inside [0, n)
__device__ __forceinline__ bool bounds_span(long long off, long long len, long long n, int line, int kind) {
  if (off >= 0 && len >= 0 && off + len <= n) return true;
  bounds_fail(line, kind, off + len, n);
  return false;
}
}  // namespace
#define GDN_G(i, n) ::gdn::bounds_ix((i), (long long)(n), __LINE__, 0)
#define GDN_S(i, n) ::gdn::bounds_ix((i), (long long)(n), __LINE__, 1)
#define GDN_T(i, n) ::gdn::bounds_ix((i), (long long)(n), __LINE__, 2)
#define GDN_SPAN_G(off, len, n) ::gdn::bounds_span((long long)(off), (long long)(len), (long long)(n), __LINE__, 0)
#define GDN_SPAN_S(off, len, n) ::gdn::bounds_span((long long)(off), (long long)(len), (long long)(n), __LINE__, 1)
#else
#define GDN_G(i, n) (i)
#define GDN_S(i, n) (i)
#define GDN_T(i, n) (i)
#define GDN_SPAN_G(off, len, n) true
#define GDN_SPAN_S(off, len, n) true
#endif
// A buffer seen by a kernel: a pointer and, in the checked build, the
// buffer's extent (elements) and the line that made the view.  Indexing,
// at() and sub-views are checked there; a failed check is recorded and the
// access goes to a small per-unit scratch buffer instead.  In the normal
// build a View is its pointer.
#ifdef GDN_DEBUG_BOUNDS
namespace {
__device__ __align__(16) unsigned char g_bounds_sink[256];
}  // namespace
#endif
template <typename T, int KIND>
struct View {
  T* p;
#ifdef GDN_DEBUG_BOUNDS
  long long n;
  int line;
#endif
  // element i (checked: i inside the view)
  __device__ __forceinline__ T& operator[](long long i) const { return *at(i, 1); }
  // pointer to element i, where w elements from i on are inside the view
  __device__ __forceinline__ T* at(long long i, long long w = 1) const {
#ifdef GDN_DEBUG_BOUNDS
    if (i < 0 || i + w > n || w * (long long)sizeof(T) > (long long)sizeof(g_bounds_sink)) {
      bounds_fail(line, KIND, i + w - 1, n);
      return reinterpret_cast<T*>(g_bounds_sink);
    }
#endif
    return p + i;
  }
  // whether elements [i, i + w) are inside the view (a failure is recorded);
  // for asynchronous copies, which are skipped rather than redirected
  __device__ __forceinline__ bool has([[maybe_unused]] long long i, [[maybe_unused]] long long w) const {
#ifdef GDN_DEBUG_BOUNDS
    if (i < 0 || i + w > n) {
      bounds_fail(line, KIND, i + w - 1, n);
      return false;
    }
#endif
    return true;
  }
  // the view from element off on
  __device__ __forceinline__ View operator+(long long off) const {
    View v = *this;
#ifdef GDN_DEBUG_BOUNDS
    if (off < 0 || off > n) {
      bounds_fail(line, KIND, off, n);
      v.n = 0;
      return v;
    }
    v.n = n - off;
#endif
    v.p = p + off;
    return v;
  }
};
// a view of the buffer p[0 .. n) (n ignored in the normal build)
template <int KIND, typename T>
__device__ __forceinline__ View<T, KIND> make_view(T* p, [[maybe_unused]] long long n,
                                                   [[maybe_unused]] int line) {
  View<T, KIND> v;
  v.p = p;
#ifdef GDN_DEBUG_BOUNDS
  v.n = n;
  v.line = line;
#endif
  return v;
}
template <typename V, typename T, int KIND>
__device__ __forceinline__ V& vec_at(const View<T, KIND>& v, long long i) {
  static_assert(sizeof(V) % sizeof(T) == 0, "a vector of whole elements");
  return *reinterpret_cast<V*>(v.at(i, (long long)(sizeof(V) / sizeof(T))));
}
// the same on a plain pointer (unchecked)
template <typename V, typename T>
__device__ __forceinline__ V& vec_at(T* p, long long i) {
  return *reinterpret_cast<V*>(p + i);
}
// The V at byte offset `off` of a shared-memory tile of `bytes` bytes
// (checked: the V lies inside the tile; a failure is recorded against the
// caller's line and the access goes to the tile's start).
template <typename V>
__device__ __forceinline__ V& tile_at(unsigned char* tile, [[maybe_unused]] unsigned bytes, unsigned off,
                                      [[maybe_unused]] int line = __builtin_LINE()) {
#ifdef GDN_DEBUG_BOUNDS
  if ((unsigned long long)off + sizeof(V) > bytes) {
    bounds_fail(line, 1, (long long)off + (long long)sizeof(V) - 1, bytes);
    off = 0;
  }
#endif
  return *reinterpret_cast<V*>(tile + off);
}
#define GDN_GV(p, n) ::gdn::make_view<0>((p), (long long)(n), __LINE__)
#define GDN_SV(p, n) ::gdn::make_view<1>((p), (long long)(n), __LINE__)

// byte distance from `base` to `p`
__host__ __device__ __forceinline__ long long byte_off(const void* base, const void* p) {
  return (long long)(reinterpret_cast<const unsigned char*>(p) - reinterpret_cast<const unsigned char*>(base));
}
// `bytes` at global `p` inside the buffer [base, base + extent bytes)
#define GDN_GBYTES(p, bytes, base, extent) GDN_SPAN_G(::gdn::byte_off((base), (p)), (bytes), (extent))
// `bytes` at shared `p` inside the CTA's shared-memory struct `S`
#define GDN_SBYTES(p, bytes, S) GDN_SPAN_S(::gdn::byte_off(&(S), (p)), (bytes), sizeof(S))

// 0 = usable, 1 = padding (-1), 2 = out of range
__device__ __forceinline__ int slot_class(int32_t id, int32_t n) {
  if (id == -1) return 1;
  return (id < 0 || id >= n) ? 2 : 0;
}

// ---- thread-block cluster barrier (split arrive / wait) --------------------
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}

// ---- mbarrier + bulk async copy (TMA engine, 1-D) --------------------------
// Every wait is bounded: a phase that does not complete within kWaitLimitNs
// (1 s of %globaltimer) makes the wait return false; callers then report
// GDN_DEV_ERR_TIMEOUT and wind down instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// a barrier no thread waits on any more, before its memory is reused or the
// barrier initialised again
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for the phase of parity `parity` to complete; false after the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
// global -> shared bulk copy; bytes and both addresses multiples of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// 16-byte global -> shared copy without a barrier (completion by group):
// both addresses 16-byte aligned
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled while the previous kernel in the stream finishes; every kernel of
// this library calls pdl_wait() before its first access to global memory (the
// wait returns once every earlier grid in the stream has completed and its
// writes are visible; at once for a plain launch), then pdl_trigger() so that
// the next kernel can in turn be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
// barrier over a subset of warps that also ORs `v` over its threads: every
// participant gets the same result
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
// barrier over a subset of warps (id 1..15; nthreads a multiple of 32)
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// Packed fp32 pairs (Blackwell f32x2 instructions, round to nearest: each
// half is bit-identical to the scalar operation).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 join4(float2 lo, float2 hi) { return make_float4(lo.x, lo.y, hi.x, hi.y); }

// ---- math (CUDA library functions; fp32) -----------------------------------
// e^x as 2^(x log2 e) on the PTX ex2.approx.ftz instruction (relative error
// ~2^-22 plus |x| 2^-24 from rounding the product; subnormal results flush to
// zero).  For values that become bf16 tensor-core operands, where it is far
// below the operand rounding; it is several times faster than expf here.
__device__ __forceinline__ float exp_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}
__device__ __forceinline__ float silu_f(float y) { return y / (1.0f + expf(-y)); }
// the same with the approximate exponential and division (ex2.approx,
// rcp.approx: a few ulp of fp32), for prologues that run it on every draft
__device__ __forceinline__ float silu_fast_f(float y) { return __fdividef(y, 1.f + exp_ftz(-y)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f(float x) {
  return x > 20.0f ? x : log1pf(expf(x));
}
// The chunked forms take the decay between tokens j and t as
// exp(b_t - b_j), with b the cumulative log decay.  A token whose decay is 0
// (log decay -inf: a = +inf, or exp(A_log) * softplus overflowing) would make
// that -inf - (-inf).  They floor each token's log decay here instead.  At
// -128 the exponential is exactly 0 in fp32 (expf underflows below about
// -104, and 2^x on ex2.approx.ftz flushes below about -87), so the decay
// stays 0 and every difference stays finite; any log decay below -104
// already has an exponential of 0, so the floor changes no finite decay.  A
// floor this close to the underflow keeps the cumulative sums after a floored
// token small, where fp32 still resolves their differences finely.  The
// comparison lets NaN through (fmaxf would turn it into the floor), so a NaN
// gate poisons the state exactly as the token recurrence does.
constexpr float kLogDecayFloor = -128.0f;
__device__ __forceinline__ float floor_log_decay(float g) { return g < kLogDecayFloor ? kLogDecayFloor : g; }
// alpha = exp(-exp(A_log) * softplus(a + dt_bias))
__device__ __forceinline__ float gate_alpha(float A_log, float dt_bias, float a) {
  return expf(-expf(A_log) * softplus_f(a + dt_bias));
}

constexpr float kNormEps = 1e-6f;

// ---- host side ------------------------------------------------------------
extern std::atomic<uint64_t> g_launches[GDN_K_COUNT];
inline void count_launch(int k) { g_launches[k].fetch_add(1, std::memory_order_relaxed); }

inline int64_t channels(const gdn_dims& d) {
  return 2 * (int64_t)d.hk * d.dk + (int64_t)d.hv * d.dv;
}
inline size_t dtype_size(int32_t t) { return t == GDN_BF16 ? 2 : 4; }

// launch k<<<grid, block, smem, s>>>(args...), optionally as clusters of
// `cluster` CTAs and as a programmatic dependent of the previous work in the
// stream (pdl; GDN_NO_PDL=1 turns that off, for measurement)
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(bool pdl, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      dim3 cluster, Args&&... args) {
  static const bool no_pdl = [] {
    const char* e = std::getenv("GDN_NO_PDL");
    return e && e[0] == '1';
  }();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl && !no_pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster.x;
    attr[n].val.clusterDim.y = cluster.y;
    attr[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}
// Programmatic dependent launch pays off for the decode and per-head verify
// kernels and the slot operations (the next launch overlaps the previous
// kernel's tail: decode batch 64, 0.85 -> 0.89 of HBM); it measured slower
// for the persistent verify kernel and the prefill kernels, which launch in
// plain stream order (their pdl_wait() then returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, dim3 cluster,
                       Args&&... args) {
  return launch_ex(true, k, grid, block, smem, s, cluster, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, dim3 cluster,
                         Args&&... args) {
  return launch_ex(false, k, grid, block, smem, s, cluster, std::forward<Args>(args)...);
}
inline size_t ssm_slot_bytes(const gdn_dims& d) {
  return (size_t)d.hv * d.dv * d.dk * sizeof(float);
}
inline size_t conv_slot_bytes(const gdn_dims& d) {
  return (size_t)(d.conv_width - 1) * channels(d) * dtype_size(d.conv_dtype);
}

// Bounds words of the checked build: each translation unit registers a
// reader that copies its word out and clears it.
using BoundsReader = bool (*)(BoundsWord*);
void register_bounds_reader(const char* unit, BoundsReader r);
#ifdef GDN_DEBUG_BOUNDS
namespace {
bool read_bounds_word(BoundsWord* w) {
  if (cudaMemcpyFromSymbol(w, g_bounds_word, sizeof *w) != cudaSuccess) return false;
  const BoundsWord zero = {};
  return cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof zero) == cudaSuccess;
}
const int g_bounds_registered = (register_bounds_reader(GDN_TU, read_bounds_word), 0);
}  // namespace
#endif

// Host-side validation shared by every entry point.
gdn_status check_dims(const gdn_dims* d);
gdn_status check_pool(const gdn_dims& d, const gdn_pool& p);
inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace gdn
