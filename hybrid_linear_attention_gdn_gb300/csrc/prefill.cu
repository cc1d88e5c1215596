// Chunked GDN prefill with block-aligned checkpoints.
//
// TokenSpeed Qwen3.5 page, "Ciclo de vida de slots": prefill fills the
// working slot, and checkpoint slots receive clean snapshots that become
// reusable at block-aligned prefix boundaries.  The state recurrence is
// evaluated in the chunkwise WY/UT form of the delta rule (Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence
// Length", NeurIPS 2024, with the Gated DeltaNet decay): for a chunk of n
// tokens with local cumulative log-decay b_i = sum_{j<=i} g_j,
//   A = strict_lower(diag(beta) (K K^T (.) Gamma)),  Gamma_ij = e^{b_i - b_j}
//   T = (I + A)^{-1} diag(beta)
//   W = T diag(e^b) K,  U = T V,  Delta = U - W S
//   O = diag(e^b) Q S + (Q K^T (.) Gamma (.) lower-incl-diag) Delta
//   S' = e^{b_n} S + (diag(e^{b_n - b}) K)^T Delta
// Chunks are 64 tokens aligned to absolute positions, so every checkpoint
// boundary (a multiple of the checkpoint block, itself a multiple of 64) is
// a chunk boundary.
//
// Three kernels, in stream order:
//   features: conv1d + SiLU + L2 norm + gates per (token, QK head) -> workspace
//   chunks:   one CTA per (sequence, V head, dv tile) walks the chunks in
//             order, keeping its slice of S in shared memory
//   history:  one thread per (sequence, channel) writes the conv history of
//             every checkpoint and the final one (it reads the old history
//             before overwriting it, and runs after `features` read it)
#include "gdn_common.cuh"
#include "decode_tma.cuh"
#include "prefill_history.cuh"
#include "prefill_tc.cuh"

#include <cstdlib>
#include <cstring>

namespace gdn {
namespace {

using namespace pfx;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;
template <typename V>
__device__ __forceinline__ int seq_of_token(const V& cu, int n_seq, int64_t t) {
  int lo = 0, hi = n_seq - 1;  // last n with cu[n] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// features: grid (total tokens, hk)
// ---------------------------------------------------------------------------
template <int DK, typename Tact, typename Tconv>
__global__ void __launch_bounds__(kThreads) features_kernel(const PrefillArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sq_[DK], sk_[DK];
  __shared__ float sred[2][kWarps];
  __shared__ float sr[2];
  const auto sq = GDN_SV(sq_, DK), sk = GDN_SV(sk_, DK);
  const PrefillViews<Tact, Tconv> g(a);
  const int64_t t = blockIdx.x;
  const int hq = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = seq_of_token(g.cu_seqlens, a.n_seq, t);
  const int32_t slot = g.slot_ids[n];
  if (slot_class(slot, a.num_slots)) return;  // the chunk kernel zeroes its outputs
  const int64_t t0 = g.cu_seqlens[n];
  const int64_t i = t - t0;  // index within the sequence
  if (i < 0) return;         // inconsistent cu_seqlens: reported by the chunk kernel
  const auto qkv = g.qkv;
  const auto hist = g.conv + (size_t)slot * (a.W - 1) * a.C;
  const int nch = 2 * DK + a.G * a.dv;
  for (int idx = tid; idx < nch; idx += kThreads) {
    int c;
    if (idx < DK) c = hq * DK + idx;
    else if (idx < 2 * DK) c = a.hk * DK + hq * DK + (idx - DK);
    else c = 2 * a.hk * DK + hq * a.G * a.dv + (idx - 2 * DK);
    const auto w = g.conv_w + (size_t)c * a.W;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) {
      if (j < a.W) {
        const int64_t m = i - (a.W - 1) + j;  // window element j, sequence-relative
        const float xv = m >= 0 ? to_f32(qkv[(t0 + m) * a.C + c])
                                : to_f32(hist[(size_t)(a.W - 1 + m) * a.C + c]);
        acc = fmaf(w[j], xv, acc);
      }
    }
    const float y = silu_f(acc);
    if (idx < DK) sq[idx] = y;
    else if (idx < 2 * DK) sk[idx - DK] = y;
    else g.ws_v[(size_t)t * a.hv * a.dv + (size_t)hq * a.G * a.dv + (idx - 2 * DK)] = y;
  }
  __syncthreads();
  float pq = 0.f, pk = 0.f;
  for (int m = tid; m < DK; m += kThreads) {
    pq = fmaf(sq[m], sq[m], pq);
    pk = fmaf(sk[m], sk[m], pk);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    pq += __shfl_xor_sync(0xffffffffu, pq, o);
    pk += __shfl_xor_sync(0xffffffffu, pk, o);
  }
  if (lane == 0) {
    const int w = GDN_S(warp, kWarps);
    sred[0][w] = pq;
    sred[1][w] = pk;
  }
  __syncthreads();
  if (tid == 0) {
    float x = 0.f, y = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      x += sred[0][w];
      y += sred[1][w];
    }
    sr[0] = rsqrtf(x + kNormEps) * rsqrtf((float)DK);
    sr[1] = rsqrtf(y + kNormEps);
  }
  __syncthreads();
  const auto oq = g.ws_q + ((size_t)t * a.hk + hq) * DK;
  const auto ok = g.ws_k + ((size_t)t * a.hk + hq) * DK;
  for (int m = tid; m < DK; m += kThreads) {
    oq[m] = sq[m] * sr[0];
    ok[m] = sk[m] * sr[1];
  }
  if (tid < a.G) {
    const int h = hq * a.G + tid;
    const float av = to_f32(g.a[(size_t)t * a.hv + h]);
    const float bv = to_f32(g.b[(size_t)t * a.hv + h]);
    g.ws_g[(size_t)t * a.hv + h] = floor_log_decay(-expf(g.A_log[h]) * softplus_f(av + g.dt_bias[h]));
    g.ws_beta[(size_t)t * a.hv + h] = sigmoid_f(bv);
  }
}

// ---------------------------------------------------------------------------
// chunks: grid (hv * n_tiles, n_seq); S slice St[DVT][DK] lives in smem
// ---------------------------------------------------------------------------
template <int DK, int DVT>
struct ChunkSmem {
  static constexpr int LK = DK + 1;   // padded row strides (column walks
  static constexpr int LV = DVT + 1;  // across rows stay conflict-free)
  static constexpr int LC = kChunk + 1;
  static constexpr size_t floats =
      (size_t)DVT * LK            // St
      + 3 * (size_t)kChunk * LK   // K, Q, W
      + 2 * (size_t)kChunk * LV   // V, U (then Delta)
      + 2 * (size_t)kChunk * LC   // A (then QK), T
      + 3 * kChunk;               // b, beta, e^b
  static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, int DVT, typename Tact>
__global__ void __launch_bounds__(kThreads, 1) chunk_kernel(const PrefillArgs a) {
  pdl_wait();
  pdl_trigger();
  using L = ChunkSmem<DK, DVT>;
  extern __shared__ float sm_[];
  const auto sm = GDN_SV(sm_, L::floats);
  const auto St = sm;
  const auto K = St + DVT * L::LK;
  const auto Q = K + kChunk * L::LK;
  const auto Wm = Q + kChunk * L::LK;
  const auto V = Wm + kChunk * L::LK;
  const auto U = V + kChunk * L::LV;
  const auto A = U + kChunk * L::LV;
  const auto Tm = A + kChunk * L::LC;
  const auto sb = Tm + kChunk * L::LC;
  const auto sbeta = sb + kChunk;
  const auto seb = sbeta + kChunk;
  const PrefillViews<Tact, float> g(a);  // (the conv history is not touched here)

  const int tid = threadIdx.x;
  const int n_tiles = (a.dv + DVT - 1) / DVT;
  const int n = blockIdx.y;
  const int h = blockIdx.x / n_tiles;
  const int j0 = (blockIdx.x % n_tiles) * DVT;
  const int ncols = min(DVT, a.dv - j0);
  const int hq = h / a.G;
  const int64_t t0 = g.cu_seqlens[n], len = (int64_t)g.cu_seqlens[n + 1] - t0;
  const int64_t p0 = g.start_pos[n];
  const int32_t slot = g.slot_ids[n];
  const auto out = g.out;
  if (t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0) {
    if (blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * ncols; e += kThreads) {
      const int64_t r = e / ncols;
      out[((t0 + r) * a.hv + h) * a.dv + j0 + (e % ncols)] = from_f32<Tact>(0.f);
    }
    return;
  }
  const auto gS = g.ssm + (((size_t)slot * a.hv + h) * a.dv + j0) * DK;
  for (int e = tid; e < DVT * DK; e += kThreads) {
    const int j = e / DK, m = e % DK;
    St[j * L::LK + m] = j < ncols ? gS[(size_t)j * DK + m] : 0.f;
  }

  int64_t pos = p0;
  const int64_t p1 = p0 + len;
  while (pos < p1) {
    const int64_t cend = min(p1, (pos / kChunk + 1) * kChunk);
    const int nr = (int)(cend - pos);
    const int64_t tb = t0 + (pos - p0);  // packed index of row 0
    __syncthreads();  // previous chunk done with K, Q, V, St
    for (int e = tid; e < kChunk * DK; e += kThreads) {
      const int r = e / DK, m = e % DK;
      const bool ok = r < nr;
      K[r * L::LK + m] = ok ? g.ws_k[((tb + r) * a.hk + hq) * DK + m] : 0.f;
      Q[r * L::LK + m] = ok ? g.ws_q[((tb + r) * a.hk + hq) * DK + m] : 0.f;
    }
    for (int e = tid; e < kChunk * DVT; e += kThreads) {
      const int r = e / DVT, j = e % DVT;
      V[r * L::LV + j] = (r < nr && j < ncols) ? g.ws_v[((tb + r) * a.hv + h) * a.dv + j0 + j] : 0.f;
    }
    if (tid < 32) {  // inclusive prefix sum of g (warp 0, two 32-wide halves)
      float carry = 0.f;
      for (int half = 0; half < 2; ++half) {
        const int r = half * 32 + tid;
        float v = r < nr ? g.ws_g[(tb + r) * a.hv + h] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, v, o);
          if (tid >= o) v += u;
        }
        v += carry;
        sb[r] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
      }
    }
    if (tid >= 64 && tid < 128) {
      const int r = tid - 64;
      sbeta[r] = r < nr ? g.ws_beta[(tb + r) * a.hv + h] : 0.f;
    }
    __syncthreads();
    if (tid < kChunk) seb[tid] = expf(sb[tid]);
    // A = strict_lower(diag(beta) (K K^T (.) Gamma))
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
      const int r = e / kChunk, c = e % kChunk;
      float v = 0.f;
      if (c < r && r < nr) {
        float d = 0.f;
        for (int m = 0; m < DK; ++m) d = fmaf(K[r * L::LK + m], K[c * L::LK + m], d);
        v = sbeta[r] * d * expf(sb[r] - sb[c]);
      }
      A[r * L::LC + c] = v;
    }
    __syncthreads();
    // T = (I + A)^{-1} diag(beta): forward substitution, one row at a time
    for (int r = 0; r < nr; ++r) {
      if (tid < kChunk) {
        const int c = tid;
        float v = 0.f;
        if (c <= r) {
          v = (c == r) ? sbeta[r] : 0.f;
          for (int m = c; m < r; ++m) v = fmaf(-A[r * L::LC + m], Tm[m * L::LC + c], v);
        }
        Tm[r * L::LC + c] = v;
      }
      __syncthreads();
    }
    // A <- Q K^T (.) Gamma (.) lower-incl-diag ;  W = T diag(e^b) K ;  U = T V
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
      const int r = e / kChunk, c = e % kChunk;
      float v = 0.f;
      if (c <= r && r < nr) {
        float d = 0.f;
        for (int m = 0; m < DK; ++m) d = fmaf(Q[r * L::LK + m], K[c * L::LK + m], d);
        v = d * expf(sb[r] - sb[c]);
      }
      A[r * L::LC + c] = v;
    }
    for (int e = tid; e < kChunk * DK; e += kThreads) {
      const int r = e / DK, m = e % DK;
      float v = 0.f;
      if (r < nr)
        for (int c = 0; c <= r; ++c) v = fmaf(Tm[r * L::LC + c] * seb[c], K[c * L::LK + m], v);
      Wm[r * L::LK + m] = v;
    }
    for (int e = tid; e < kChunk * DVT; e += kThreads) {
      const int r = e / DVT, j = e % DVT;
      float v = 0.f;
      if (r < nr)
        for (int c = 0; c <= r; ++c) v = fmaf(Tm[r * L::LC + c], V[c * L::LV + j], v);
      U[r * L::LV + j] = v;
    }
    __syncthreads();
    // Delta = U - W S   (in place)
    for (int e = tid; e < kChunk * DVT; e += kThreads) {
      const int r = e / DVT, j = e % DVT;
      if (r < nr) {
        float v = U[r * L::LV + j];
        for (int m = 0; m < DK; ++m) v = fmaf(-Wm[r * L::LK + m], St[j * L::LK + m], v);
        U[r * L::LV + j] = v;
      }
    }
    __syncthreads();
    // O = diag(e^b) Q S + (QK^T (.) Gamma) Delta
    for (int e = tid; e < kChunk * DVT; e += kThreads) {
      const int r = e / DVT, j = e % DVT;
      if (r < nr && j < ncols) {
        float qs = 0.f;
        for (int m = 0; m < DK; ++m) qs = fmaf(Q[r * L::LK + m], St[j * L::LK + m], qs);
        float v = seb[r] * qs;
        for (int c = 0; c <= r; ++c) v = fmaf(A[r * L::LC + c], U[c * L::LV + j], v);
        out[((tb + r) * a.hv + h) * a.dv + j0 + j] = from_f32<Tact>(v);
      }
    }
    __syncthreads();
    // S' = e^{b_n} S + (diag(e^{b_n - b}) K)^T Delta
    const float blast = sb[nr - 1];
    for (int e = tid; e < DVT * DK; e += kThreads) {
      const int j = e / DK, m = e % DK;
      float v = expf(blast) * St[j * L::LK + m];
      for (int c = 0; c < nr; ++c)
        v = fmaf(expf(blast - sb[c]) * K[c * L::LK + m], U[c * L::LV + j], v);
      St[j * L::LK + m] = v;
    }
    pos = cend;
    if (pos % a.ckpt_block == 0) {
      const int64_t idx = pos / a.ckpt_block - p0 / a.ckpt_block - 1;
      if (idx >= 0 && idx < a.max_ckpt) {
        const int32_t cid = g.ckpt_ids[(size_t)n * a.max_ckpt + idx];
        if (slot_class(cid, a.ck_num_slots) == 0) {
          __syncthreads();
          const auto cS = g.ck_ssm + (((size_t)cid * a.hv + h) * a.dv + j0) * DK;
          for (int e = tid; e < ncols * DK; e += kThreads)
            cS[(size_t)(e / DK) * DK + (e % DK)] = St[(e / DK) * L::LK + (e % DK)];
        }
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < ncols * DK; e += kThreads)
    gS[(size_t)(e / DK) * DK + (e % DK)] = St[(e / DK) * L::LK + (e % DK)];
}

// ---------------------------------------------------------------------------
// history: grid (ceil(C / 256), n_seq, groups); one thread per channel
// (history_channel, prefill_history.cuh)
// ---------------------------------------------------------------------------
template <typename Tact, typename Tconv>
__global__ void __launch_bounds__(kThreads) history_kernel(const PrefillArgs a) {
  pdl_wait();
  pdl_trigger();
  history_channel<Tact, Tconv>(a, blockIdx.y, blockIdx.z, (int)(blockIdx.x * kThreads + threadIdx.x));
}

// channels x sequences x groups of kCkGroup checkpoints
dim3 history_grid(const PrefillArgs& a) {
  const int groups = a.max_ckpt > kCkGroup ? (a.max_ckpt + kCkGroup - 1) / kCkGroup : 1;
  return dim3((unsigned)((a.C + kThreads - 1) / kThreads), (unsigned)a.n_seq, (unsigned)groups);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t q, k, v, g, beta, total;
};

WsLayout ws_layout(const gdn_dims& d, int64_t total) {
  WsLayout w;
  size_t off = 0;
  w.q = off; off += align256(sizeof(float) * (size_t)total * d.hk * d.dk);
  w.k = off; off += align256(sizeof(float) * (size_t)total * d.hk * d.dk);
  w.v = off; off += align256(sizeof(float) * (size_t)total * d.hv * d.dv);
  w.g = off; off += align256(sizeof(float) * (size_t)total * d.hv);
  w.beta = off; off += align256(sizeof(float) * (size_t)total * d.hv);
  w.total = off;
  return w;
}

template <int DK, int DVT, typename Tact, typename Tconv>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t s) {
  if (a.total > 0) {
    cudaError_t e = launch_plain(features_kernel<DK, Tact, Tconv>, dim3((unsigned)a.total, (unsigned)a.hk),
                               dim3(kThreads), 0, s, dim3(1), a);
    if (e != cudaSuccess) return e;
  }
  using L = ChunkSmem<DK, DVT>;
  auto ck = chunk_kernel<DK, DVT, Tact>;
  cudaError_t e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.dv + DVT - 1) / DVT;
  e = launch_plain(ck, dim3((unsigned)(a.hv * n_tiles), (unsigned)a.n_seq), dim3(kThreads), L::bytes, s, dim3(1), a);
  if (e != cudaSuccess) return e;
  return launch_plain(history_kernel<Tact, Tconv>, history_grid(a), dim3(kThreads), 0, s, dim3(1), a);
}

template <int DK, int DVT>
cudaError_t dispatch_prefill(const PrefillArgs& a, int act, int cv, cudaStream_t s) {
  if (act == GDN_F32 && cv == GDN_F32) return launch_prefill_t<DK, DVT, float, float>(a, s);
  if (act == GDN_BF16 && cv == GDN_BF16)
    return launch_prefill_t<DK, DVT, __nv_bfloat16, __nv_bfloat16>(a, s);
  return launch_prefill_t<DK, DVT, __nv_bfloat16, float>(a, s);
}

cudaError_t launch_history(const PrefillArgs& a, int act, int cv, cudaStream_t s) {
  const dim3 grid = history_grid(a);
  if (act == GDN_F32 && cv == GDN_F32)
    return launch_plain(history_kernel<float, float>, grid, dim3(kThreads), 0, s, dim3(1), a);
  if (act == GDN_BF16 && cv == GDN_BF16)
    return launch_plain(history_kernel<__nv_bfloat16, __nv_bfloat16>, grid, dim3(kThreads), 0, s, dim3(1), a);
  return launch_plain(history_kernel<__nv_bfloat16, float>, grid, dim3(kThreads), 0, s, dim3(1), a);
}

// Prefill paths.  The tf32 tensor-core path takes dk = dv = 128, width 4,
// bf16 activations and conv history; every other shape runs the fp32
// CUDA-core path.  GDN_PREFILL_PATH (read on every call, so a process can
// time or test each) forces one: "cuda" the CUDA-core path, "bf16" the
// tensor-core path with bf16 operands (dk = dv = 128, width 4), whose operand
// roundings put its outputs above the 2e-3 the tf32 path meets.
enum class PrefillPath { kCuda, kTf32, kBf16 };
PrefillPath prefill_path(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p) {
  const char* e = std::getenv("GDN_PREFILL_PATH");
  if (e && !std::strcmp(e, "cuda")) return PrefillPath::kCuda;
  if (e && !std::strcmp(e, "bf16"))
    return prefill_tc_supported(d, qkv, out, p) ? PrefillPath::kBf16 : PrefillPath::kCuda;
  return prefill_tc32_supported(d, qkv, out, p) ? PrefillPath::kTf32 : PrefillPath::kCuda;
}

}  // namespace

// The conv histories of a prefill's checkpoints and of its final state, for
// prefill paths that write only the SSM states (the KDA recurrence).
cudaError_t conv_history_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt,
                                const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                                int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                                int32_t ckpt_block, const void* qkv, uint32_t* dev_err, cudaStream_t s) {
  PrefillArgs p = {};
  p.ssm = pool.ssm;
  p.conv = pool.conv;
  p.num_slots = pool.num_slots;
  p.ck_ssm = ckpt.ssm;
  p.ck_conv = ckpt.conv;
  p.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  p.slot_ids = slot_ids;
  p.cu_seqlens = cu_seqlens;
  p.start_pos = start_pos;
  p.n_seq = n_seq;
  p.total = total;
  p.ckpt_ids = ckpt_ids;
  p.max_ckpt = max_ckpt;
  p.ckpt_block = ckpt_block;
  p.qkv = qkv;
  p.err = dev_err;
  p.hk = d.hk;
  p.hv = d.hv;
  p.dk = d.dk;
  p.dv = d.dv;
  p.W = d.conv_width;
  p.C = (int32_t)channels(d);
  p.G = d.hv / d.hk;
  return launch_history(p, d.act_dtype, d.conv_dtype, s);
}

}  // namespace gdn

// Sized for either path (the tensor-core path needs about half of it).
extern "C" size_t gdn_chunk_prefill_workspace_size(const gdn_dims* dims, int32_t n_seq,
                                                   int64_t total_tokens) {
  if (gdn::check_dims(dims) != GDN_OK || total_tokens < 0 || n_seq < 0) return 0;
  const size_t v1 = gdn::ws_layout(*dims, total_tokens).total;
  const size_t tc = gdn::prefill_tc_workspace(*dims, n_seq, total_tokens);
  return total_tokens == 0 ? 0 : (v1 > tc ? v1 : tc);
}

// The chunked prefill: host-side checks, then (launch = true) the kernels.
static gdn_status chunk_prefill_impl(bool launch, const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                     const gdn_params* params, const int32_t* slot_ids,
                                     const int32_t* cu_seqlens, const int64_t* start_pos, int32_t n_seq,
                                     int64_t total_tokens, const int32_t* ckpt_ids, int32_t max_ckpt,
                                     int32_t ckpt_block, const void* qkv, const void* a, const void* b,
                                     void* out, void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                     void* stream, const gdn::Tc32Epilogue* epi = nullptr) {
  using namespace gdn;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n_seq < 0 || total_tokens < 0 || max_ckpt < 0) return GDN_ERR_INVALID_ARG;
  if (ckpt_block <= 0 || ckpt_block % kChunk) return GDN_ERR_INVALID_ARG;
  if (n_seq == 0) return GDN_OK;
  if (n_seq > 65535 || total_tokens > 2147483647LL || max_ckpt > kCkGroup * 65535)
    return GDN_ERR_UNSUPPORTED;
  if ((st = check_pool(*dims, pool)) != GDN_OK) return st;
  if (max_ckpt > 0 && (st = check_pool(*dims, ckpt)) != GDN_OK) return st;
  if (!params || !params->conv_w || !params->A_log || !params->dt_bias) return GDN_ERR_INVALID_ARG;
  if (!slot_ids || !cu_seqlens || !start_pos || (max_ckpt > 0 && !ckpt_ids))
    return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!qkv || !a || !b || !out)) return GDN_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(*dims, total_tokens);
  const PrefillPath path = prefill_path(*dims, qkv, out, *params);
  const size_t need = path == PrefillPath::kTf32   ? 0
                      : path == PrefillPath::kBf16 ? prefill_tc_workspace(*dims, n_seq, total_tokens)
                                                   : wl.total;
  if (total_tokens > 0 && need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return GDN_ERR_INVALID_ARG;
  if (dims->hv / dims->hk * dims->dv + 2 * dims->dk > 4096) return GDN_ERR_UNSUPPORTED;
  if (!launch) return GDN_OK;
  PrefillArgs p = {};
  p.ssm = pool.ssm;
  p.conv = pool.conv;
  p.num_slots = pool.num_slots;
  p.ck_ssm = ckpt.ssm;
  p.ck_conv = ckpt.conv;
  p.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  p.conv_w = params->conv_w;
  p.A_log = params->A_log;
  p.dt_bias = params->dt_bias;
  p.slot_ids = slot_ids;
  p.cu_seqlens = cu_seqlens;
  p.start_pos = start_pos;
  p.n_seq = n_seq;
  p.total = total_tokens;
  p.ckpt_ids = ckpt_ids;
  p.max_ckpt = max_ckpt;
  p.ckpt_block = ckpt_block;
  p.qkv = qkv;
  p.a = a;
  p.b = b;
  p.out = out;
  p.err = dev_err;
  if (char* ws = reinterpret_cast<char*>(workspace)) {  // the tf32 path needs none (may be null)
    p.ws_q = reinterpret_cast<float*>(ws + wl.q);
    p.ws_k = reinterpret_cast<float*>(ws + wl.k);
    p.ws_v = reinterpret_cast<float*>(ws + wl.v);
    p.ws_g = reinterpret_cast<float*>(ws + wl.g);
    p.ws_beta = reinterpret_cast<float*>(ws + wl.beta);
  }
  p.hk = dims->hk;
  p.hv = dims->hv;
  p.dk = dims->dk;
  p.dv = dims->dv;
  p.W = dims->conv_width;
  p.C = (int32_t)channels(*dims);
  p.G = dims->hv / dims->hk;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
  const int act = dims->act_dtype, cv = dims->conv_dtype;
  if (path == PrefillPath::kTf32) {
    // the readout epilogue fuses into the output when its operands allow the
    // tile copies; otherwise it runs after the prefill, in place
    const bool fuse = epi && aligned(epi->z, 16) && aligned(epi->weight, 16);
    e = prefill_tc32_launch(*dims, pool, ckpt, *params, slot_ids, cu_seqlens, start_pos, n_seq, total_tokens,
                            ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, out, dev_err, s, fuse ? epi : nullptr);
    if (fuse) epi = nullptr;
    if (e == cudaSuccess) e = launch_history(p, act, cv, s);
  } else if (path == PrefillPath::kBf16) {
    e = prefill_tc_launch(*dims, pool, ckpt, *params, slot_ids, cu_seqlens, start_pos, n_seq,
                          total_tokens, ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, out, workspace,
                          dev_err, s);
    if (e == cudaSuccess) e = launch_history(p, act, cv, s);
  } else {
    switch (dims->dk) {
      case 16: e = dispatch_prefill<16, 16>(p, act, cv, s); break;
      case 64: e = dispatch_prefill<64, 64>(p, act, cv, s); break;
      case 128: e = dispatch_prefill<128, 64>(p, act, cv, s); break;
    }
  }
  if (e == cudaSuccess) count_launch(GDN_K_PREFILL);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  if (epi) return gdn_gated_rmsnorm(dims, out, epi->z, epi->weight, epi->eps, total_tokens, out, stream);
  return GDN_OK;
}

extern "C" gdn_status gdn_chunk_prefill(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                        const gdn_params* params, const int32_t* slot_ids,
                                        const int32_t* cu_seqlens, const int64_t* start_pos,
                                        int32_t n_seq, int64_t total_tokens,
                                        const int32_t* ckpt_ids, int32_t max_ckpt,
                                        int32_t ckpt_block, const void* qkv, const void* a,
                                        const void* b, void* out, void* workspace,
                                        size_t workspace_bytes, uint32_t* dev_err, void* stream) {
  return chunk_prefill_impl(true, dims, pool, ckpt, params, slot_ids, cu_seqlens, start_pos, n_seq,
                            total_tokens, ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, out, workspace,
                            workspace_bytes, dev_err, stream);
}

// The prefill with the readout epilogue (gated RMS norm): `y` receives
// o / sqrt(mean(o^2) + eps) * weight * silu(z) instead of the readout o.
extern "C" gdn_status gdn_chunk_prefill_gated(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                              const gdn_params* params, const int32_t* slot_ids,
                                              const int32_t* cu_seqlens, const int64_t* start_pos,
                                              int32_t n_seq, int64_t total_tokens, const int32_t* ckpt_ids,
                                              int32_t max_ckpt, int32_t ckpt_block, const void* qkv,
                                              const void* a, const void* b, const void* z,
                                              const float* weight, float eps, void* y, void* workspace,
                                              size_t workspace_bytes, uint32_t* dev_err, void* stream) {
  using namespace gdn;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (!(eps >= 0.f) || (total_tokens > 0 && (!z || !weight))) return GDN_ERR_INVALID_ARG;
  if (dims->dv > 256) return GDN_ERR_UNSUPPORTED;
  if ((st = chunk_prefill_impl(false, dims, pool, ckpt, params, slot_ids, cu_seqlens, start_pos, n_seq,
                               total_tokens, ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, y, workspace,
                               workspace_bytes, dev_err, stream)) != GDN_OK)
    return st;
  const Tc32Epilogue epi{z, weight, eps};
  return chunk_prefill_impl(true, dims, pool, ckpt, params, slot_ids, cu_seqlens, start_pos, n_seq, total_tokens,
                            ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, y, workspace, workspace_bytes, dev_err,
                            stream, total_tokens > 0 ? &epi : nullptr);
}

// Mixed batch, decode-first: the decode rows through the decode kernel, the
// continuations through the chunked prefill (rows at their absolute offsets,
// so only the per-sequence arrays are offset).  The prefill half is checked
// before anything is launched, so a host-side error launches nothing.
extern "C" gdn_status gdn_mixed_step(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                     const gdn_params* params, const int32_t* slot_ids,
                                     const int32_t* cu_seqlens, const int64_t* start_pos,
                                     int32_t n_seq, int32_t n_decode, int64_t total_tokens,
                                     const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                                     const void* qkv, const void* a, const void* b, void* out,
                                     void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                     void* stream) {
  using namespace gdn;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n_seq < 0 || n_decode < 0 || n_decode > n_seq || (int64_t)n_decode > total_tokens || max_ckpt < 0)
    return GDN_ERR_INVALID_ARG;
  const int32_t n_pre = n_seq - n_decode;
  if (n_pre > 0 && (!slot_ids || !cu_seqlens || !start_pos || (max_ckpt > 0 && !ckpt_ids)))
    return GDN_ERR_INVALID_ARG;
  const int32_t* pre_ids = n_pre > 0 ? slot_ids + n_decode : nullptr;
  const int32_t* pre_cu = n_pre > 0 ? cu_seqlens + n_decode : nullptr;
  const int64_t* pre_sp = n_pre > 0 ? start_pos + n_decode : nullptr;
  const int32_t* pre_ck = (n_pre > 0 && max_ckpt > 0) ? ckpt_ids + (size_t)n_decode * max_ckpt : nullptr;
  // one launch when both halves take their fast paths and the workspace
  // holds the work queue (after the same host checks as the separate calls)
  if (n_pre > 0 && n_decode > 0 && mixed_fused_supported(*dims, qkv, out, *params) &&
      prefill_path(*dims, qkv, out, *params) == PrefillPath::kTf32 &&
      decode_takes_tma(*dims, n_decode, qkv, *params) && workspace &&
      workspace_bytes >= mixed_fused_queue_bytes(n_pre) && aligned(workspace, 8)) {
    if (!qkv || !a || !b || !out) return GDN_ERR_INVALID_ARG;
    if ((st = check_pool(*dims, pool)) != GDN_OK) return st;
    if ((st = chunk_prefill_impl(false, dims, pool, ckpt, params, pre_ids, pre_cu, pre_sp, n_pre, total_tokens,
                                 pre_ck, max_ckpt, ckpt_block, qkv, a, b, out, nullptr, 0, dev_err, stream)) !=
        GDN_OK)
      return st;
    const cudaError_t e = mixed_fused_launch(*dims, pool, ckpt, *params, slot_ids, cu_seqlens, start_pos, n_seq,
                                             n_decode, total_tokens, ckpt_ids, max_ckpt, ckpt_block, qkv, a, b,
                                             out, workspace, dev_err, reinterpret_cast<cudaStream_t>(stream));
    count_launch(GDN_K_MIXED);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  if (n_pre > 0 &&
      (st = chunk_prefill_impl(false, dims, pool, ckpt, params, pre_ids, pre_cu, pre_sp, n_pre, total_tokens,
                               pre_ck, max_ckpt, ckpt_block, qkv, a, b, out, workspace, workspace_bytes,
                               dev_err, stream)) != GDN_OK)
    return st;
  if (n_decode > 0 &&
      (st = gdn_decode_step(dims, pool, params, slot_ids, n_decode, qkv, a, b, out, dev_err, stream)) != GDN_OK)
    return st;
  if (n_pre == 0) return GDN_OK;
  return chunk_prefill_impl(true, dims, pool, ckpt, params, pre_ids, pre_cu, pre_sp, n_pre, total_tokens,
                            pre_ck, max_ckpt, ckpt_block, qkv, a, b, out, workspace, workspace_bytes, dev_err,
                            stream);
}

// ---------------------------------------------------------------------------
// No-allocation variant: the same prefill, working in a scratch array that
// is part of the library image instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace gdn {
namespace {

// Device address of the scratch array in the current device's context.  In
// host code the array's name only stands for the symbol; its address is
// looked up on every call (a cheap query next to a prefill), so it stays
// right after a device reset or in another context.
gdn_status noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
  *out = p;
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                                const gdn_params* params, const int32_t* slot_ids,
                                                const int32_t* cu_seqlens, const int64_t* start_pos,
                                                int32_t n_seq, int64_t total_tokens,
                                                const int32_t* ckpt_ids, int32_t max_ckpt,
                                                int32_t ckpt_block, const void* qkv, const void* a,
                                                const void* b, void* out, uint32_t* dev_err,
                                                void* stream) {
  const size_t need = gdn_chunk_prefill_workspace_size(dims, n_seq, total_tokens);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    const gdn_status st = gdn::noalloc_scratch(&ws);
    if (st != GDN_OK) return st;
    ws_bytes = GDN_NOALLOC_SCRATCH_BYTES;
  }
  return gdn_chunk_prefill(dims, pool, ckpt, params, slot_ids, cu_seqlens, start_pos, n_seq,
                           total_tokens, ckpt_ids, max_ckpt, ckpt_block, qkv, a, b, out, ws,
                           ws_bytes, dev_err, stream);
}
