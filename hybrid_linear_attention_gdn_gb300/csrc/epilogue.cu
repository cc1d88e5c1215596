// Readout epilogue: gated RMS norm of every (token, V head) row.
//
// Not written on the pages.  The published Gated DeltaNet block ("Gated Delta
// Networks", ICLR 2025) normalises each head's readout and gates it with the
// SiLU of a separate projection z:
//   y = o / sqrt(mean(o^2) + eps) * w * silu(z),   w [dv] shared by the heads.
//
// HBM bound (o and z read once, y written once: 3 x 256 bytes per bf16 row of
// 128).  Two forms:
//  * streamed (rows of 64 to 512 bytes, 16-byte aligned tensors): each warp
//    copies 2 KB of consecutive rows of o and of z into shared memory by
//    16-byte cp.async copies, all in flight at once without holding
//    registers, then normalises them.  A row is LPR = row bytes / 16 lanes;
//    lane l copies, and later reads back, the 16-byte pieces l % LPR of its
//    rows, so no lane reads another's copies and no barrier is needed; the
//    sum of squares reduces over the row's lanes by shuffles, and y leaves by
//    16-byte stores.  (The same layout with the loads straight into
//    registers measured 0.63 of the copy bandwidth: too few bytes in flight.)
//  * general: each warp takes four rows and issues all their loads before the
//    first reduction; lane l holds the EPL consecutive elements from l * EPL
//    of a row (one vector access when the row is full-width and aligned).
// In both, y may be o: every element is read before its row's reduction and
// written after it, by the same lane.
#include "gdn_common.cuh"
#include "decode_tma.cuh"  // sm_count

#include <cstdlib>
#include <cstring>

namespace gdn {
namespace {

constexpr int kWarps = 8;        // warps per CTA
constexpr int kRowsPerWarp = 4;  // rows a warp loads before its first reduction
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

// silu(z) = z / (1 + e^-z) with the approximate exponential and division
// (ex2.approx and rcp.approx, a few ulp of fp32: far below the bf16 rounding
// of the outputs).  An IEEE division here cost several times the two
// special-function operations per element that the norm needs.
__device__ __forceinline__ float silu_approx(float z) { return __fdividef(z, 1.f + exp_ftz(-z)); }

// EPL consecutive elements of one row, by one vector access when VEC (the row
// is full-width and 16-byte aligned; the vector is EPL * sizeof(T) <= 16 bytes)
template <typename T, int EPL> struct VecOf;
template <> struct VecOf<__nv_bfloat16, 1> { using t = unsigned short; };
template <> struct VecOf<__nv_bfloat16, 2> { using t = unsigned int; };
template <> struct VecOf<__nv_bfloat16, 4> { using t = uint2; };
template <> struct VecOf<__nv_bfloat16, 8> { using t = uint4; };
template <> struct VecOf<float, 1> { using t = float; };
template <> struct VecOf<float, 2> { using t = float2; };
template <> struct VecOf<float, 4> { using t = float4; };
template <> struct VecOf<float, 8> { using t = float4; };  // unused: 32 bytes are never one access

// row: a view of one row's dv elements
template <typename T, int EPL, bool VEC, typename R>
__device__ __forceinline__ void load_part(const R& row, int j0, int dv, float (&v)[EPL]) {
  if constexpr (VEC) {
    T tmp[EPL];
    const typename VecOf<T, EPL>::t u = vec_at<const typename VecOf<T, EPL>::t>(row, j0);
    memcpy(tmp, &u, sizeof(tmp));
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = to_f32(tmp[e]);
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = j0 + e < dv ? to_f32(row[j0 + e]) : 0.f;
  }
}

template <typename T, int EPL, bool VEC, typename R>
__device__ __forceinline__ void store_part(const R& row, int j0, int dv, const float (&v)[EPL]) {
  if constexpr (VEC) {
    T tmp[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) tmp[e] = from_f32<T>(v[e]);
    typename VecOf<T, EPL>::t u;
    memcpy(&u, tmp, sizeof(tmp));
    vec_at<typename VecOf<T, EPL>::t>(row, j0) = u;
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if (j0 + e < dv) row[j0 + e] = from_f32<T>(v[e]);
  }
}

template <typename T, int EPL, bool VEC>
__global__ void __launch_bounds__(32 * kWarps)
    gated_rmsnorm_kernel(const T* o, const T* __restrict__ z, const float* __restrict__ w, float eps,
                         int64_t rows, int dv, T* y) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
  if (r0 >= rows) return;
  const int j0 = lane * EPL;
  const auto ov_ = GDN_GV(o, rows * dv), zv_ = GDN_GV(z, rows * dv);
  const auto yv_ = GDN_GV(y, rows * dv);
  const auto wv_ = GDN_GV(w, dv);
  float ov[kRowsPerWarp][EPL], zv[kRowsPerWarp][EPL], wv[EPL];
  // every load of the warp's rows in flight before the first reduction
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    if (r0 + i < rows) {
      load_part<T, EPL, VEC>(ov_ + (r0 + i) * dv, j0, dv, ov[i]);
      load_part<T, EPL, VEC>(zv_ + (r0 + i) * dv, j0, dv, zv[i]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) ov[i][e] = zv[i][e] = 0.f;
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) wv[e] = j0 + e < dv ? wv_[j0 + e] : 0.f;
  float ss[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    ss[i] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) ss[i] = fmaf(ov[i][e], ov[i][e], ss[i]);
  }
#pragma unroll
  for (int m = 16; m; m >>= 1)
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], m);
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    if (r0 + i >= rows) break;
    const float inv = rsqrtf(ss[i] / (float)dv + eps);
    float yv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float gate = silu_approx(zv[i][e]);
      yv[e] = ov[i][e] * inv * wv[e] * gate;
    }
    store_part<T, EPL, VEC>(yv_ + (r0 + i) * dv, j0, dv, yv);
  }
}

// ---- streamed form -----------------------------------------------------------
constexpr int kSWarps = 8;          // warps per CTA
constexpr int kSGroupBytes = 2048;  // bytes of o (and of z) per warp: 8 rows of 256 bytes

// LPR lanes per row (row bytes / 16); a warp's group is kSGroupBytes of
// consecutive rows (RPG rows).  One group per warp, many CTAs: every load of
// the group is in flight before the first is waited for, and the CTAs that
// follow keep each SM's copies going while earlier ones compute and store.
// (Measured on the Qwen3.5-shaped readout, 32768 tokens x 32 heads: 1.04 of
// the measured copy bandwidth; the same copies walked by a persistent grid,
// several groups per warp through a ring of stages, reached 0.80 - 0.85.)
template <typename T, int LPR>
__global__ void __launch_bounds__(32 * kSWarps)
    gated_rmsnorm_stream_kernel(const T* o, const T* z, const float* __restrict__ w, float eps, int64_t rows,
                                int dv, T* y) {
  constexpr int E = 16 / sizeof(T);              // elements per 16-byte piece
  constexpr int RPG = kSGroupBytes / (16 * LPR);  // rows per group
  constexpr int RPI = 32 / LPR;                   // rows per warp-wide access
  constexpr int NI = RPG / RPI;                   // accesses per group (per lane)
  static_assert(RPG % RPI == 0 && NI >= 1, "whole accesses per group");
  __shared__ __align__(16) uint4 stage[kSWarps][2][kSGroupBytes / 16];  // [warp][o | z]
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int piece = lane % LPR, sub = lane / LPR;  // 16-byte piece of the row, row within an access
  const int64_t g = (int64_t)blockIdx.x * kSWarps + warp;
  if (g * RPG >= rows) return;
  const auto ov = GDN_GV(reinterpret_cast<const uint4*>(o), rows * LPR);
  const auto zv = GDN_GV(reinterpret_cast<const uint4*>(z), rows * LPR);
  const auto yv = GDN_GV(reinterpret_cast<uint4*>(y), rows * LPR);
  const auto sv = GDN_SV(&stage[0][0][0], kSWarps * 2 * (kSGroupBytes / 16));
  const int so = warp * 2 * (kSGroupBytes / 16), sz = so + kSGroupBytes / 16;  // this warp's o and z parts
  // every piece of the group this lane reads: into shared memory, all in flight
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int64_t row = g * RPG + i * RPI + sub;
    if (row < rows) {
      const int64_t src = row * LPR + piece;
      const int dst = i * 32 + lane;
      if (sv.has(so + dst, 1) && ov.has(src, 1)) cp_async16(sv.p + so + dst, ov.p + src);
      if (sv.has(sz + dst, 1) && zv.has(src, 1)) cp_async16(sv.p + sz + dst, zv.p + src);
    }
  }
  cp_async_commit();
  // the lane's weights meanwhile: elements piece * E .. piece * E + E - 1
  float wv[E];
  {
    const auto wg = GDN_GV(w, dv);
#pragma unroll
    for (int e = 0; e < E; ++e) wv[e] = wg[piece * E + e];
  }
  cp_async_wait_all();  // this lane's copies have landed (it reads only those)
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int64_t row = g * RPG + i * RPI + sub;
    const uint4 ou = sv[so + i * 32 + lane], zu = sv[sz + i * 32 + lane];
    T ot[E], zt[E];
    memcpy(ot, &ou, 16);
    memcpy(zt, &zu, 16);
    float of[E], ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      of[e] = to_f32(ot[e]);
      ss = fmaf(of[e], of[e], ss);
    }
#pragma unroll
    for (int m = LPR / 2; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float inv = rsqrtf(ss / (float)dv + eps);
    T yt[E];
#pragma unroll
    for (int e = 0; e < E; ++e) yt[e] = from_f32<T>(of[e] * inv * wv[e] * silu_approx(to_f32(zt[e])));
    uint4 yu;
    memcpy(&yu, yt, 16);
    if (row < rows) yv[row * LPR + piece] = yu;
  }
}

template <typename T, int LPR>
cudaError_t launch_stream(const T* o, const T* z, const float* w, float eps, int64_t rows, int dv, T* y,
                          cudaStream_t s) {
  constexpr int RPG = kSGroupBytes / (16 * LPR);
  const int64_t groups = (rows + RPG - 1) / RPG;
  const int64_t ctas = (groups + kSWarps - 1) / kSWarps;
  if (ctas > 2147483647LL) return cudaErrorInvalidValue;
  return launch_pdl(gated_rmsnorm_stream_kernel<T, LPR>, dim3((unsigned)ctas), dim3(32 * kSWarps), 0, s, dim3(1),
                    o, z, w, eps, rows, dv, y);
}

template <typename T, int EPL>
cudaError_t launch_epl(const T* o, const T* z, const float* w, float eps, int64_t rows, int dv, T* y,
                       bool vec, cudaStream_t s) {
  const dim3 grid((unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta));
  const dim3 block(32 * kWarps);
  constexpr bool kCanVec = EPL * sizeof(T) <= 16;
  if (kCanVec && vec)
    return launch_pdl(gated_rmsnorm_kernel<T, EPL, kCanVec>, grid, block, 0, s, dim3(1), o, z, w, eps, rows,
                      dv, y);
  return launch_pdl(gated_rmsnorm_kernel<T, EPL, false>, grid, block, 0, s, dim3(1), o, z, w, eps, rows, dv,
                    y);
}

// GDN_EPILOGUE=rows selects the general form at every shape (read on every
// call, so one process can time both)
bool stream_epilogue() {
  const char* e = std::getenv("GDN_EPILOGUE");
  return !(e && e[0] == 'r');
}

template <typename T>
cudaError_t launch_rmsnorm_t(const void* o, const void* z, const float* w, float eps, int64_t rows, int dv,
                             void* y, cudaStream_t s) {
  const T* ot = static_cast<const T*>(o);
  const T* zt = static_cast<const T*>(z);
  T* yt = static_cast<T*>(y);
  // streamed: rows of 64, 128, 256 or 512 bytes, every tensor 16-byte aligned
  const size_t row_bytes = (size_t)dv * sizeof(T);
  const bool al16 = aligned(o, 16) && aligned(z, 16) && aligned(y, 16);
  if (al16 && stream_epilogue()) {
    if (row_bytes == 64) return launch_stream<T, 4>(ot, zt, w, eps, rows, dv, yt, s);
    if (row_bytes == 128) return launch_stream<T, 8>(ot, zt, w, eps, rows, dv, yt, s);
    if (row_bytes == 256) return launch_stream<T, 16>(ot, zt, w, eps, rows, dv, yt, s);
    if (row_bytes == 512) return launch_stream<T, 32>(ot, zt, w, eps, rows, dv, yt, s);
  }
  // vector accesses when every lane holds EPL elements of a full-width row and
  // every row starts 16-byte aligned
  const int epl = dv <= 32 ? 1 : dv <= 64 ? 2 : dv <= 128 ? 4 : 8;
  const bool vec = dv == 32 * epl && aligned(o, 16) && aligned(z, 16) && aligned(y, 16) &&
                   ((size_t)dv * sizeof(T)) % 16 == 0;
  if (epl == 1) return launch_epl<T, 1>(ot, zt, w, eps, rows, dv, yt, vec, s);
  if (epl == 2) return launch_epl<T, 2>(ot, zt, w, eps, rows, dv, yt, vec, s);
  if (epl == 4) return launch_epl<T, 4>(ot, zt, w, eps, rows, dv, yt, vec, s);
  return launch_epl<T, 8>(ot, zt, w, eps, rows, dv, yt, vec, s);
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, const void* o, const void* z,
                                        const float* weight, float eps, int64_t n_tokens, void* y,
                                        void* stream) {
  using namespace gdn;
  const gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n_tokens < 0 || !(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (n_tokens == 0) return GDN_OK;
  if (!o || !z || !weight || !y) return GDN_ERR_INVALID_ARG;
  if (dims->dv > 256) return GDN_ERR_UNSUPPORTED;
  const int64_t rows = n_tokens * dims->hv;
  if ((rows + kRowsPerCta - 1) / kRowsPerCta > 2147483647LL) return GDN_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dims->act_dtype == GDN_BF16
          ? launch_rmsnorm_t<__nv_bfloat16>(o, z, weight, eps, rows, dims->dv, y, s)
          : launch_rmsnorm_t<float>(o, z, weight, eps, rows, dims->dv, y, s);
  count_launch(GDN_K_GATED_RMSNORM);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
