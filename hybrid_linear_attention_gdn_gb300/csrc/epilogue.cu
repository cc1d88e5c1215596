// Readout epilogue: gated RMS norm of every (token, V head) row.
//
// Not written on the pages.  The published Gated DeltaNet block ("Gated Delta
// Networks", ICLR 2025) normalises each head's readout and gates it with the
// SiLU of a separate projection z:
//   y = o / sqrt(mean(o^2) + eps) * w * silu(z),   w [dv] shared by the heads.
//
// HBM bound (o and z read once, y written once: 3 x 256 bytes per bf16 row of
// 128): each warp takes four rows and issues all their loads before the first
// reduction; lane l holds the EPL consecutive elements from l * EPL of a row
// (one vector access when the row is full-width and aligned), the sum of
// squares by a warp shuffle.  y may be o (each element is read before the
// row's reduction and written after it, by the same lane).  A variant with
// 16-byte accesses (two rows per warp-wide access, eight rows per warp)
// measured slower: 0.63 against 0.76 of the copy bandwidth.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 8;        // warps per CTA
constexpr int kRowsPerWarp = 4;  // rows a warp loads before its first reduction
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

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
      const float gate = zv[i][e] / (1.f + exp_ftz(-zv[i][e]));  // silu(z)
      yv[e] = ov[i][e] * inv * wv[e] * gate;
    }
    store_part<T, EPL, VEC>(yv_ + (r0 + i) * dv, j0, dv, yv);
  }
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

template <typename T>
cudaError_t launch_rmsnorm_t(const void* o, const void* z, const float* w, float eps, int64_t rows, int dv,
                             void* y, cudaStream_t s) {
  const T* ot = static_cast<const T*>(o);
  const T* zt = static_cast<const T*>(z);
  T* yt = static_cast<T*>(y);
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
