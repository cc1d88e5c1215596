// KDA prefill, chunked form (dk = 128, dv <= 128), fp32 accuracy.
//
// The per-key-channel gated delta rule (Kimi Delta Attention, Kimi Linear
// 2025: St <- St diag(alpha_t) + beta_t (v_t - St diag(alpha_t) k_t) k_t^T,
// o_t = St q_t) over windows of 16 tokens aligned to absolute positions (so
// every block-aligned checkpoint falls on a window end).  Inside a window,
// with a_t = prod_{m<=t} alpha_m (per channel, from the window start),
//   K~_t = k_t (.) a_t,   Q~_t = q_t (.) a_t,   K-_t = k_t (.) prod_{t<m} alpha_m,
//   A'[t][j] = sum_c k_t k_j prod_{j<m<=t} alpha_m   (t > j),
//   M[t][j]  = sum_c q_t k_j prod_{j<m<=t} alpha_m   (t >= j),
//   T = (I + diag(beta) A')^-1 diag(beta),
// the window is, for every state row (a row of St):
//   X = v - St K~^T,  Delta = X T^T,  o = St Q~^T + M Delta,
//   St <- St diag(a_last) + Delta K-.
// This is the window-level unrolling of the token step (the chunkwise WY
// algebra of the Gated DeltaNet paper with the decay kept per channel).  Every
// decay factor is a product of alphas over a token range, at most 1, formed
// from cumulative logs, so none can overflow.
//
// One CTA per (sequence, V head), 256 threads.  The state rows' products run
// on the tensor cores (mma m16n8k8 tf32, operands split hi + lo so that three
// products carry an fp32 product): warp w owns rows 16w .. 16w+15, held in
// registers in the accumulator layout for the whole sequence.  The raw
// inputs of window w+1 are staged by cp.async while window w is computed.
#include "gdn_common.cuh"
#include "kda_chunk.cuh"

#include <cstddef>

namespace gdn {
namespace {

constexpr int kCk = 16;          // window
constexpr int kCkThreads = 256;
constexpr int kD = 128;          // dk
constexpr int kMaxV = 128;       // dv
constexpr int kCh = 2 * kD + kMaxV;
constexpr int kCkMaxW = 8;       // conv taps held (right-aligned)
// padded row strides (floats) so that the tensor-core fragment loads hit 32
// distinct banks: K~ and Q~ rows are read at (row g, column tq), K- at (row
// tq, column g), T and M at (row g, column tq)
constexpr int kKQS = kD + 4;     // 132
constexpr int kKBS = kD + 8;     // 136
constexpr int kTS = kCk + 4;     // 20

struct KdaChunkArgs {
  float* ssm;
  const void* conv;
  int32_t num_slots;
  float* ck_ssm;
  int32_t ck_num_slots;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;  // [hv][dk]
  const int32_t* slot_ids;
  const int32_t* cu_seqlens;
  const int64_t* start_pos;
  int64_t total;
  const int32_t* ckpt_ids;
  int32_t max_ckpt;
  int32_t ckpt_block;
  const void* qkv;
  const void* a;  // [total][hv][dk]
  const void* b;
  void* out;
  uint32_t* err;
  int32_t hk, hv, dv, W, C, G;
};

template <typename Tact>
struct __align__(16) CkSmem {
  Tact xr[2][kCk][kCh];     // raw inputs (q | k | v rows), double-buffered
  Tact ga[2][kCk][kD];      // gate logits, double-buffered
  float bl[2][kCk];         // beta logits, double-buffered
  float xh[kCkMaxW - 1][kCh];  // conv history, one column per channel
  float cw[kCkMaxW][kCh];   // conv weights, right-aligned
  float sy[kCk][kCh];       // conv + SiLU; q and k normalised in place
  float al[kCk][kD];        // log alpha (0 past the window's end)
  float lb[kCk][kKQS];      // cumulative log alpha from the window start (padded rows)
  float kp[kCk][kKQS];      // k^ (padded rows)
  float qp[kCk][kKQS];      // q^ (padded rows)
  uint32_t kth[kCk][kKQS], ktl[kCk][kKQS];  // K~ as tf32 hi + lo
  uint32_t qth[kCk][kKQS], qtl[kCk][kKQS];  // Q~ as tf32 hi + lo
  uint32_t kbh[kCk][kKBS], kbl[kCk][kKBS];  // K- as tf32 hi + lo
  float dec[kD];            // a_last: the window's decay of the state
  float A[kCk][kCk];        // A' (t > j)
  float M[kCk][kTS];        // M (t >= j)
  uint32_t Mh[kCk][kTS], Ml[kCk][kTS];  // M as tf32 hi + lo
  uint32_t Th[kCk][kTS], Tl[kCk][kTS];  // T (lower triangle with the diagonal) as tf32 hi + lo
  float Pm[kCk][kCk + 1];   // powers of L = diag(beta) A' in the solve
  float Xm[kCk][kCk + 1];   // (I + L)^-1 in the making
  float beta[kCk];
  float so[kCk][kMaxV];     // the window's outputs
};

// Warp-level tf32 tensor-core product (m16n8k8, fp32 accumulate).  Lane =
// 4 g + tq; A holds (g, tq), (g + 8, tq), (g, tq + 4), (g + 8, tq + 4); B holds
// (tq, g), (tq + 4, g); C/D hold (g, 2tq), (g, 2tq + 1), (g + 8, 2tq), (g + 8, 2tq + 1).
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo, both tf32: the split that lets three tf32 products carry an
// fp32 product (hi*hi + hi*lo + lo*hi; lo*lo is below fp32's rounding)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = tf32_rna(x);
  lo = tf32_rna(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d += a b with b already split (hi, lo)
__device__ __forceinline__ void mma3s(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], uint32_t bh0,
                                      uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma_tf32(d, al, bh0, bh1);
  mma_tf32(d, ah, bl0, bl1);
  mma_tf32(d, ah, bh0, bh1);
}

// The A fragment of an 8-column group from the same group in the C layout
// (c[0..3] = (g, 2tq), (g, 2tq + 1), (g + 8, 2tq), (g + 8, 2tq + 1)): quad
// shuffles, then the split
__device__ __forceinline__ void c_to_a(const float (&c)[4], uint32_t (&ah)[4], uint32_t (&al)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int lo = (g << 2) | (tq >> 1), hi = lo + 2;
  const bool odd = tq & 1;
  const float x0 = __shfl_sync(0xffffffffu, c[0], lo), x1 = __shfl_sync(0xffffffffu, c[1], lo);
  const float y0 = __shfl_sync(0xffffffffu, c[2], lo), y1 = __shfl_sync(0xffffffffu, c[3], lo);
  const float u0 = __shfl_sync(0xffffffffu, c[0], hi), u1 = __shfl_sync(0xffffffffu, c[1], hi);
  const float z0 = __shfl_sync(0xffffffffu, c[2], hi), z1 = __shfl_sync(0xffffffffu, c[3], hi);
  split_tf32(odd ? x1 : x0, ah[0], al[0]);  // (g, tq)
  split_tf32(odd ? y1 : y0, ah[1], al[1]);  // (g + 8, tq)
  split_tf32(odd ? u1 : u0, ah[2], al[2]);  // (g, tq + 4)
  split_tf32(odd ? z1 : z0, ah[3], al[3]);  // (g + 8, tq + 4)
}

// first global channel of staged channel i (q, k of the QK head, then v rows)
__device__ __forceinline__ int ck_channel(int i, int hq, int h, int hk, int dv) {
  if (i < kD) return hq * kD + i;
  if (i < 2 * kD) return hk * kD + hq * kD + (i - kD);
  return 2 * hk * kD + h * dv + (i - 2 * kD);
}

// raw inputs of tokens [tok, tok + nt) into the staging buffers (ASYNC:
// 16-byte cp.async pieces, every segment a multiple of 16 bytes)
template <typename Tact, bool ASYNC>
__device__ __forceinline__ void ck_stage(const KdaChunkArgs& a, Tact (*xr)[kCh], Tact (*gs)[kD], int64_t tok, int nt,
                                         int hq, int h) {
  const auto qkv = GDN_GV(reinterpret_cast<const Tact*>(a.qkv), a.total * a.C);
  const auto ga = GDN_GV(reinterpret_cast<const Tact*>(a.a), a.total * a.hv * kD);
  const auto xv = GDN_SV(&xr[0][0], kCk * kCh), gv = GDN_SV(&gs[0][0], kCk * kD);  // one staging buffer each
  const int nch = 2 * kD + a.dv;
  if constexpr (ASYNC) {
    constexpr int E = 16 / sizeof(Tact);
    const int per_row = nch / E;
    for (int p = threadIdx.x; p < nt * per_row; p += kCkThreads) {
      const int t = p / per_row, e = (p % per_row) * E;
      const size_t src = (size_t)(tok + t) * a.C + ck_channel(e, hq, h, a.hk, a.dv);
      if (xv.has(t * kCh + e, E) && qkv.has(src, E)) cp_async16(&xr[t][e], qkv.p + src);
    }
    for (int p = threadIdx.x; p < nt * (kD / E); p += kCkThreads) {
      const int t = p / (kD / E), e = (p % (kD / E)) * E;
      const size_t src = ((size_t)(tok + t) * a.hv + h) * kD + e;
      if (gv.has(t * kD + e, E) && ga.has(src, E)) cp_async16(&gs[t][e], ga.p + src);
    }
  } else {
    for (int p = threadIdx.x; p < nt * nch; p += kCkThreads) {
      const int t = p / nch, e = p % nch;
      xv[t * kCh + e] = qkv[(size_t)(tok + t) * a.C + ck_channel(e, hq, h, a.hk, a.dv)];
    }
    for (int p = threadIdx.x; p < nt * kD; p += kCkThreads) {
      const int t = p / kD, e = p % kD;
      gv[t * kD + e] = ga[((size_t)(tok + t) * a.hv + h) * kD + e];
    }
  }
}

template <typename Tact, typename Tconv, bool ASYNC>
__global__ void __launch_bounds__(kCkThreads, 1) kda_chunk_kernel(const KdaChunkArgs a) {
  pdl_wait();
  pdl_trigger();
  using SMT = CkSmem<Tact>;
  static_assert(offsetof(SMT, ga) % 16 == 0 && offsetof(SMT, lb) % 16 == 0 && offsetof(SMT, kp) % 16 == 0 &&
                    offsetof(SMT, qp) % 16 == 0 && offsetof(SMT, dec) % 16 == 0,
                "vector-accessed shared arrays must start 16-byte aligned");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SMT& S = *reinterpret_cast<SMT*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, n = blockIdx.y, hq = h / a.G;
  const int dv = a.dv, nch = 2 * kD + dv;
  // the caller's tensors (extents in elements)
  const int n_seq = gridDim.y;
  const auto cu_seqlens = GDN_GV(a.cu_seqlens, n_seq + 1);
  const auto start_pos = GDN_GV(a.start_pos, n_seq);
  const auto slot_ids = GDN_GV(a.slot_ids, n_seq);
  const auto ckpt_ids = GDN_GV(a.ckpt_ids, (long long)n_seq * a.max_ckpt);
  const auto ssm = GDN_GV(a.ssm, (long long)a.num_slots * a.hv * dv * kD);
  const auto ck_ssm = GDN_GV(a.ck_ssm, (long long)a.ck_num_slots * a.hv * dv * kD);
  const int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1], len = t1 - t0, p0 = start_pos[n];
  if (t0 < 0 || len < 0 || t1 > a.total || p0 < 0) {
    if (h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const auto out = GDN_GV(reinterpret_cast<Tact*>(a.out), a.total * a.hv * dv);
  const int32_t slot = slot_ids[n];
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * dv; e += kCkThreads)
      out[((t0 + e / dv) * a.hv + h) * dv + e % dv] = from_f32<Tact>(0.f);
    return;
  }
  if (len == 0) return;

  // windows aligned to absolute multiples of 16: the first ends at the next one
  const int first = len < kCk - (int)(p0 % kCk) ? (int)len : kCk - (int)(p0 % kCk);
  const auto gb = GDN_GV(reinterpret_cast<const Tact*>(a.b), a.total * a.hv);
  ck_stage<Tact, ASYNC>(a, S.xr[0], S.ga[0], t0, first, hq, h);
  if constexpr (ASYNC) cp_async_commit();
  if (tid < first) S.bl[0][GDN_S(tid, kCk)] = to_f32(gb[(size_t)(t0 + tid) * a.hv + h]);

  // this thread's state: rows rA = 16 warp + g and rB = rA + 8, in the
  // tensor core's C layout: sc[j] = (rA, 8j + 2tq), (rA, 8j + 2tq + 1),
  // (rB, 8j + 2tq), (rB, 8j + 2tq + 1)
  const int g = lane >> 2, tq = lane & 3;
  const int rA = GDN_S(16 * warp + g, kMaxV - 8), rB = rA + 8;
  const bool vA = rA < dv, vB = rB < dv;
  const auto StA = ssm + (((size_t)slot * a.hv + h) * dv + (vA ? rA : 0)) * kD;
  const auto StB = ssm + (((size_t)slot * a.hv + h) * dv + (vB ? rB : 0)) * kD;
  float sc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 x = vA ? vec_at<float2>(StA, 8 * j + 2 * tq) : make_float2(0.f, 0.f);
    const float2 y = vB ? vec_at<float2>(StB, 8 * j + 2 * tq) : make_float2(0.f, 0.f);
    sc[j][0] = x.x;
    sc[j][1] = x.y;
    sc[j][2] = y.x;
    sc[j][3] = y.y;
  }
  // conv weights and history, right-aligned in kCkMaxW taps
  const auto hist = GDN_GV(reinterpret_cast<const Tconv*>(a.conv), (long long)a.num_slots * (a.W - 1) * a.C) +
                    (size_t)slot * (a.W - 1) * a.C;
  const auto conv_w = GDN_GV(a.conv_w, (long long)a.C * a.W);
  const int lead = kCkMaxW - a.W;
  for (int i0 = tid; i0 < nch; i0 += kCkThreads) {
    const int i = GDN_S(i0, kCh);
    const int ch = ck_channel(i, hq, h, a.hk, dv);
#pragma unroll
    for (int j = 0; j < kCkMaxW; ++j) S.cw[j][i] = j >= lead ? conv_w[(size_t)ch * a.W + (j - lead)] : 0.f;
#pragma unroll
    for (int j = 0; j < kCkMaxW - 1; ++j)
      S.xh[j][i] = j >= lead ? to_f32(hist[(size_t)(j - lead) * a.C + ch]) : 0.f;
  }
  const float eA = expf(GDN_GV(a.A_log, a.hv)[h]);
  // alpha channel of this thread
  const float dtb = GDN_GV(a.dt_bias, (long long)a.hv * kD)[(size_t)h * kD + (tid & (kD - 1))];
  const int64_t blk0 = p0 / a.ckpt_block;
  int64_t next_bd = (blk0 + 1) * a.ckpt_block;
  int64_t ck_idx = 0;
  if constexpr (ASYNC) cp_async_wait_all();
  __syncthreads();

  int cur = 0;
  for (int64_t w0 = 0; w0 < len; cur ^= 1) {
    const int nt = w0 == 0 ? first : (len - w0 < kCk ? (int)(len - w0) : kCk);
    const int64_t wn = w0 + nt;
    const int ntn = wn >= len ? 0 : (len - wn < kCk ? (int)(len - wn) : kCk);
    const int nxt = cur ^ 1;
    // 0. the next window's inputs
    float bnext = 0.f;
    if (ntn > 0) {
      ck_stage<Tact, ASYNC>(a, S.xr[nxt], S.ga[nxt], t0 + wn, ntn, hq, h);
      if constexpr (ASYNC) cp_async_commit();
      if (tid < ntn) bnext = to_f32(gb[(size_t)(t0 + wn + tid) * a.hv + h]);  // (tid < kCk)
    }
    // 1. conv1d + SiLU (tokens past the window's end: zero)
#pragma unroll
    for (int ci = 0; ci < 2; ++ci) {
      const int i = tid + ci * kCkThreads;
      if (i < nch && GDN_S(i, kCh) == i) {
        float w[kCkMaxW], win[kCkMaxW - 1];
#pragma unroll
        for (int j = 0; j < kCkMaxW; ++j) w[j] = S.cw[j][i];
#pragma unroll
        for (int j = 0; j < kCkMaxW - 1; ++j) win[j] = S.xh[j][i];
#pragma unroll
        for (int t = 0; t < kCk; ++t) {
          if (t < nt) {
            const float xv = to_f32(S.xr[cur][t][i]);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kCkMaxW - 1; ++j) acc = fmaf(w[j], win[j], acc);
            acc = fmaf(w[kCkMaxW - 1], xv, acc);
            S.sy[t][i] = __fdividef(acc, 1.f + exp_ftz(-acc));
#pragma unroll
            for (int j = 0; j < kCkMaxW - 2; ++j) win[j] = win[j + 1];
            win[kCkMaxW - 2] = xv;
          } else {
            S.sy[t][i] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < kCkMaxW - 1; ++j) S.xh[j][i] = win[j];
      }
    }
    // log alpha = -exp(A_log) softplus(a + dt_bias) (0 past the window's end)
    for (int e = tid; e < kCk * kD; e += kCkThreads) {
      const int t = e / kD, c = e % kD;
      const float x = to_f32(S.ga[cur][t][c]) + dtb;
      S.al[t][c] = t < nt ? floor_log_decay(-eA * (x > 20.f ? x : __logf(1.f + __expf(x)))) : 0.f;  // softplus
    }
    __syncthreads();
    // 2. per token (a warp per token): q, k normalised in place, beta
    for (int t = warp; t < kCk; t += kCkThreads / 32) {
      float* yq = S.sy[t];
      float* yk = yq + kD;
      float pq = 0.f, pk = 0.f;
      for (int i = lane; i < kD; i += 32) {
        pq = fmaf(yq[i], yq[i], pq);
        pk = fmaf(yk[i], yk[i], pk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        pq += __shfl_xor_sync(0xffffffffu, pq, o);
        pk += __shfl_xor_sync(0xffffffffu, pk, o);
      }
      const float rq = rsqrtf(pq + kNormEps) * rsqrtf((float)kD), rk = rsqrtf(pk + kNormEps);
      for (int i = lane; i < kD; i += 32) {
        yq[i] *= rq;
        yk[i] *= rk;
      }
      if (lane == 0) S.beta[t] = t < nt ? sigmoid_f(S.bl[cur][t]) : 0.f;
    }
    __syncthreads();
    // 3a. per channel (threads 0-127): the cumulative log decay from the
    //     window start, K~, Q~ (decay to token t), K- (decay from token t to
    //     the window's end), the window's decay, and padded copies of k^, q^
    if (tid < kD) {
      const int c = tid;
      float lbv[kCk];
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < kCk; ++t) {
        acc += S.al[t][c];
        lbv[t] = acc;
      }
#pragma unroll
      for (int t = 0; t < kCk; ++t) {
        const float kv = S.sy[t][kD + c], qv = S.sy[t][c];
        const float ef = __expf(lbv[t]), eb = __expf(acc - lbv[t]);
        split_tf32(kv * ef, S.kth[t][c], S.ktl[t][c]);
        split_tf32(qv * ef, S.qth[t][c], S.qtl[t][c]);
        split_tf32(kv * eb, S.kbh[t][c], S.kbl[t][c]);
        S.lb[t][c] = lbv[t];
        S.kp[t][c] = kv;
        S.qp[t][c] = qv;
      }
      S.dec[c] = __expf(acc);
    }
    __syncthreads();
    // 3b. A' and M, a thread per (t, j): the decay between tokens j and t of
    //     every channel is exp(lb[t] - lb[j]) (at most 1)
    {
      const int t = tid >> 4, j = tid & 15;
      if (t >= j) {
        float vk = 0.f, vq = 0.f;
#pragma unroll 4
        for (int c = 0; c < kD; c += 4) {
          const float4 kj = *reinterpret_cast<const float4*>(&S.kp[j][c]);
          const float4 lj = *reinterpret_cast<const float4*>(&S.lb[j][c]);
          const float4 lt = *reinterpret_cast<const float4*>(&S.lb[t][c]);
          const float4 kt4 = *reinterpret_cast<const float4*>(&S.kp[t][c]);
          const float4 qt4 = *reinterpret_cast<const float4*>(&S.qp[t][c]);
          const float f0 = kj.x * __expf(lt.x - lj.x), f1 = kj.y * __expf(lt.y - lj.y);
          const float f2 = kj.z * __expf(lt.z - lj.z), f3 = kj.w * __expf(lt.w - lj.w);
          vk = fmaf(kt4.x, f0, fmaf(kt4.y, f1, fmaf(kt4.z, f2, fmaf(kt4.w, f3, vk))));
          vq = fmaf(qt4.x, f0, fmaf(qt4.y, f1, fmaf(qt4.z, f2, fmaf(qt4.w, f3, vq))));
        }
        S.A[t][j] = vk;  // used below the diagonal only
        S.M[t][j] = vq;
      } else {
        S.A[t][j] = 0.f;  // M enters a full 16 x 16 product: zero above the diagonal
        S.M[t][j] = 0.f;
      }
    }
    __syncthreads();
    // 4. T = (I + L)^-1 diag(beta), L = diag(beta) A' strictly lower: by
    //    doubling, (I + L)^-1 = (I - L)(I + L^2)(I + L^4)(I + L^8) (L^16 = 0),
    //    a thread per entry
    {
      const int t = tid >> 4, j = tid & 15;
      const float l = t > j ? S.beta[t] * S.A[t][j] : 0.f;
      S.Pm[t][j] = l;
      S.Xm[t][j] = (t == j ? 1.f : 0.f) - l;
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        float p2 = 0.f, xp = 0.f;
#pragma unroll
        for (int m = 0; m < kCk; ++m) p2 = fmaf(S.Pm[t][m], S.Pm[m][j], p2);
        __syncthreads();
        S.Pm[t][j] = p2;
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kCk; ++m) xp = fmaf(S.Xm[t][m], S.Pm[m][j], xp);
        __syncthreads();
        S.Xm[t][j] += xp;
        __syncthreads();
      }
      split_tf32(S.Xm[t][j] * S.beta[j], S.Th[t][j], S.Tl[t][j]);
      split_tf32(S.M[t][j], S.Mh[t][j], S.Ml[t][j]);
    }
    __syncthreads();
    // 5. the state rows on the tensor cores (split tf32, fp32 accuracy), a
    //    warp per 16 rows: Xk = St K~^T and Xq = St Q~^T (16 rows x 16 tokens),
    //    Delta = (v - Xk) T^T, o = Xq + Delta M^T, St <- St diag(a_last) + Delta K-
    {
      float xk[2][4], xq[2][4];
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
        for (int i = 0; i < 4; ++i) xk[nt2][i] = xq[nt2][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        uint32_t ah[4], al[4];
        c_to_a(sc[kk], ah, al);
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2) {
          const int r8 = 8 * nt2 + g, c8 = 8 * kk + tq;
          mma3s(xk[nt2], ah, al, S.kth[r8][c8], S.kth[r8][c8 + 4], S.ktl[r8][c8], S.ktl[r8][c8 + 4]);
          mma3s(xq[nt2], ah, al, S.qth[r8][c8], S.qth[r8][c8 + 4], S.qtl[r8][c8], S.qtl[r8][c8 + 4]);
        }
      }
      // X = v - Xk (rows past dv: 0), in place
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2) {
        const int tok = 8 * nt2 + 2 * tq;
        // rA, rB < kMaxV (checked where they are set): inside sy's kCh = 2 kD + kMaxV
        xk[nt2][0] = (vA ? S.sy[tok][2 * kD + rA] : 0.f) - xk[nt2][0];
        xk[nt2][1] = (vA ? S.sy[tok + 1][2 * kD + rA] : 0.f) - xk[nt2][1];
        xk[nt2][2] = (vB ? S.sy[tok][2 * kD + rB] : 0.f) - xk[nt2][2];
        xk[nt2][3] = (vB ? S.sy[tok + 1][2 * kD + rB] : 0.f) - xk[nt2][3];
      }
      // Delta = X T^T (K = the 16 tokens j, B[j][t'] = T[t'][j])
      float dl[2][4];
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
        for (int i = 0; i < 4; ++i) dl[nt2][i] = 0.f;
#pragma unroll
      for (int kj = 0; kj < 2; ++kj) {
        uint32_t ah[4], al[4];
        c_to_a(xk[kj], ah, al);
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2) {
          const int r8 = 8 * nt2 + g, c8 = 8 * kj + tq;
          mma3s(dl[nt2], ah, al, S.Th[r8][c8], S.Th[r8][c8 + 4], S.Tl[r8][c8], S.Tl[r8][c8 + 4]);
        }
      }
      // o = Xq + Delta M^T; St <- St diag(a_last) + Delta K- (Delta as A)
      uint32_t dh[2][4], dlo[2][4];
#pragma unroll
      for (int kj = 0; kj < 2; ++kj) c_to_a(dl[kj], dh[kj], dlo[kj]);
#pragma unroll
      for (int kj = 0; kj < 2; ++kj)
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2) {
          const int r8 = 8 * nt2 + g, c8 = 8 * kj + tq;
          mma3s(xq[nt2], dh[kj], dlo[kj], S.Mh[r8][c8], S.Mh[r8][c8 + 4], S.Ml[r8][c8], S.Ml[r8][c8 + 4]);
        }
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2) {
        const int tok = 8 * nt2 + 2 * tq;
        if (vA && tok < nt) S.so[tok][rA] = xq[nt2][0];
        if (vA && tok + 1 < nt) S.so[tok + 1][rA] = xq[nt2][1];
        if (vB && tok < nt) S.so[tok][rB] = xq[nt2][2];
        if (vB && tok + 1 < nt) S.so[tok + 1][rB] = xq[nt2][3];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float d0 = S.dec[8 * j + 2 * tq], d1 = S.dec[8 * j + 2 * tq + 1];
        sc[j][0] *= d0;
        sc[j][1] *= d1;
        sc[j][2] *= d0;
        sc[j][3] *= d1;
#pragma unroll
        for (int kj = 0; kj < 2; ++kj) {
          const int r8 = 8 * kj + tq, c8 = 8 * j + g;
          mma3s(sc[j], dh[kj], dlo[kj], S.kbh[r8][c8], S.kbh[r8 + 4][c8], S.kbl[r8][c8], S.kbl[r8 + 4][c8]);
        }
      }
    }
    // a block boundary at the window's end: the rows to its checkpoint slot
    if (p0 + wn == next_bd) {
      const int64_t idx = ck_idx++;
      next_bd += a.ckpt_block;
      if (idx < a.max_ckpt) {
        const int32_t cid = ckpt_ids[(size_t)n * a.max_ckpt + idx];
        const int cc = slot_class(cid, a.ck_num_slots);
        if (cc == 0) {
          const auto dA = ck_ssm + (((size_t)cid * a.hv + h) * dv + (vA ? rA : 0)) * kD;
          const auto dB = ck_ssm + (((size_t)cid * a.hv + h) * dv + (vB ? rB : 0)) * kD;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (vA) vec_at<float2>(dA, 8 * j + 2 * tq) = make_float2(sc[j][0], sc[j][1]);
            if (vB) vec_at<float2>(dB, 8 * j + 2 * tq) = make_float2(sc[j][2], sc[j][3]);
          }
        } else if (cc == 2 && tid == 0) {
          report(a.err, GDN_DEV_ERR_SLOT_OOB);
        }
      }
    }
    __syncthreads();
    // 6. the window's outputs; the next window's beta logits and inputs land
    for (int e = tid; e < nt * dv; e += kCkThreads) {
      const int t = e / dv, i = e % dv;
      out[((size_t)(t0 + w0 + t) * a.hv + h) * dv + i] = from_f32<Tact>(S.so[GDN_S(t, kCk)][GDN_S(i, kMaxV)]);
    }
    if (tid < ntn) S.bl[nxt][GDN_S(tid, kCk)] = bnext;
    if constexpr (ASYNC) cp_async_wait_all();
    __syncthreads();
    w0 = wn;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (vA) vec_at<float2>(StA, 8 * j + 2 * tq) = make_float2(sc[j][0], sc[j][1]);
    if (vB) vec_at<float2>(StB, 8 * j + 2 * tq) = make_float2(sc[j][2], sc[j][3]);
  }
}

template <typename Tact, typename Tconv>
cudaError_t launch_ck_t(const KdaChunkArgs& a, int32_t n_seq, bool async, cudaStream_t s) {
  const size_t smem = sizeof(CkSmem<Tact>);
  auto k = async ? kda_chunk_kernel<Tact, Tconv, true> : kda_chunk_kernel<Tact, Tconv, false>;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)a.hv, (unsigned)n_seq), dim3(kCkThreads), smem, s, dim3(1), a);
}

}  // namespace

bool kda_chunk_supported(const gdn_dims& d) { return d.dk == kD && d.dv <= kMaxV && d.dv % 4 == 0; }

cudaError_t kda_chunk_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                             const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                             int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                             int32_t ckpt_block, const void* qkv, const void* av, const void* bv, void* out,
                             uint32_t* dev_err, cudaStream_t s) {
  KdaChunkArgs k = {};
  k.ssm = pool.ssm;
  k.conv = pool.conv;
  k.num_slots = pool.num_slots;
  k.ck_ssm = ckpt.ssm;
  k.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  k.conv_w = p.conv_w;
  k.A_log = p.A_log;
  k.dt_bias = p.dt_bias;
  k.slot_ids = slot_ids;
  k.cu_seqlens = cu_seqlens;
  k.start_pos = start_pos;
  k.total = total;
  k.ckpt_ids = ckpt_ids;
  k.max_ckpt = max_ckpt;
  k.ckpt_block = ckpt_block;
  k.qkv = qkv;
  k.a = av;
  k.b = bv;
  k.out = out;
  k.err = dev_err;
  k.hk = d.hk;
  k.hv = d.hv;
  k.dv = d.dv;
  k.W = d.conv_width;
  k.C = (int32_t)channels(d);
  k.G = d.hv / d.hk;
  const size_t es = dtype_size(d.act_dtype);
  const bool async = aligned(qkv, 16) && aligned(av, 16) && ((size_t)d.dv * es) % 16 == 0 &&
                     ((size_t)k.C * es) % 16 == 0;
  if (d.act_dtype == GDN_F32 && d.conv_dtype == GDN_F32) return launch_ck_t<float, float>(k, n_seq, async, s);
  if (d.act_dtype == GDN_BF16 && d.conv_dtype == GDN_BF16)
    return launch_ck_t<__nv_bfloat16, __nv_bfloat16>(k, n_seq, async, s);
  return launch_ck_t<__nv_bfloat16, float>(k, n_seq, async, s);
}

}  // namespace gdn
