// Fused GDN decode step and speculative verify over the slot pool.
//
// One CTA owns R rows (dv indices) of one V head of one request.  The fp32
// state of that head is stored transposed, St[dv][dk], so row j of St is an
// independent dk-vector: its update needs only (k^, v_j, q^), and the two dot
// products per row reduce over dk with warp shuffles - no cross-warp traffic.
//
//   lanes per row  LPR = dk/16      (each lane holds 16 consecutive-in-phase
//                                    floats of the row as 4 float4)
//   rows per warp  RW  = 32/LPR
//   rows per CTA   R   = NIT * 8 warps * RW
//
// The state rows are loaded with 128-bit streaming loads at kernel entry,
// before the slot's conv history, the activations and the gates are even
// read, so the HBM latency of the 64 KiB-per-head state overlaps the whole
// prologue (conv1d + SiLU + L2 norm + gates).  Each state element is read
// once and written once.
//
// Conv history ownership: the v channels of rows [row0, row0+R) of head h are
// read and rewritten by this CTA alone.  The q/k channels of QK head hq are
// shared by the G V heads that read hq and by all P row-parts of each, so
// those G*P CTAs form one thread-block cluster: each arrives on the cluster
// barrier once its history reads are done, and cluster rank 0 rewrites the
// q/k history after waiting - after its own state work, when the others
// have long arrived.  No distributed shared memory and no multicast is used.
#include "gdn_common.cuh"
#include "decode_tma.cuh"
#include "prefill_tc.cuh"
#include "kda_chunk.cuh"
#include "kda_tc32.cuh"

#include <cstdlib>
#include <cstring>

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxW = 8;
constexpr int kMaxT = 16;

struct StepArgs {
  float* ssm;
  void* conv;
  int32_t num_slots;
  float* spec_ssm;
  void* spec_conv;
  int32_t spec_num_slots;
  const int32_t* spec_ids;  // [B][T]
  int32_t T;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const int32_t* slot_ids;
  int32_t B;
  const void* qkv;
  const void* a;
  const void* b;
  void* out;
  uint32_t* err;
  int32_t hk, hv, dv, W, C, G, P;
};

template <int DK>
struct RowMap {
  static constexpr int LPR = DK / 16;
  static constexpr int RW = 32 / LPR;
  static constexpr int RI = kWarps * RW;
  // column of float4 number c (0..3) held by lane segment `seg`
  static __device__ __forceinline__ int col(int c, int seg) { return c * 4 * LPR + seg * 4; }
};

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

template <int DK>
__device__ __forceinline__ int channel_of(int i, int hq, int h, int hk, int dv, int row0) {
  if (i < DK) return hq * DK + i;
  if (i < 2 * DK) return hk * DK + hq * DK + (i - DK);
  return 2 * hk * DK + h * dv + row0 + (i - 2 * DK);
}

template <int DK, int NIT, typename V>
__device__ __forceinline__ void load_rows(float4 (&s)[NIT][4], const V& base, int nrows, int rloc, int seg) {
  using M = RowMap<DK>;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int row = it * M::RI + rloc;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      s[it][c] = row < nrows ? ld_stream(&vec_at<const float4>(base, (size_t)row * DK + M::col(c, seg)))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// The caller's tensors of a decode or verify step as checked views (extents
// in elements; T tokens per request).
template <int DK, typename Tact, typename Tconv, bool KDA>
struct StepViews {
  View<float, 0> ssm, spec_ssm;
  View<Tconv, 0> conv, spec_conv;
  View<const float, 0> conv_w, A_log, dt_bias;
  View<const int32_t, 0> slot_ids, spec_ids;
  View<const Tact, 0> qkv, a, b;
  View<Tact, 0> out;
  __device__ __forceinline__ explicit StepViews(const StepArgs& g, int T) {
    const long long BT = (long long)g.B * T, gate = BT * g.hv;
    ssm = GDN_GV(g.ssm, (long long)g.num_slots * g.hv * g.dv * DK);
    spec_ssm = GDN_GV(g.spec_ssm, (long long)g.spec_num_slots * g.hv * g.dv * DK);
    conv = GDN_GV(reinterpret_cast<Tconv*>(g.conv), (long long)g.num_slots * (g.W - 1) * g.C);
    spec_conv = GDN_GV(reinterpret_cast<Tconv*>(g.spec_conv), (long long)g.spec_num_slots * (g.W - 1) * g.C);
    conv_w = GDN_GV(g.conv_w, (long long)g.C * g.W);
    A_log = GDN_GV(g.A_log, g.hv);
    dt_bias = GDN_GV(g.dt_bias, (long long)g.hv * (KDA ? DK : 1));
    slot_ids = GDN_GV(g.slot_ids, g.B);
    spec_ids = GDN_GV(g.spec_ids, BT);
    qkv = GDN_GV(reinterpret_cast<const Tact*>(g.qkv), BT * g.C);
    a = GDN_GV(reinterpret_cast<const Tact*>(g.a), gate * (KDA ? DK : 1));
    b = GDN_GV(reinterpret_cast<const Tact*>(g.b), gate);
    out = GDN_GV(reinterpret_cast<Tact*>(g.out), gate * g.dv);
  }
};

// Reduce (q.q, k.k, q.k) over the dk channels of one QK head held in smem,
// with all warps; result in red_out[0..2] (shared).
template <int DK>
__device__ __forceinline__ void block_norms(const float* sq, const float* sk, float (*sred)[kWarps],
                                            float* red_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float pq = 0.f, pk = 0.f, pqk = 0.f;
  for (int i = tid; i < DK; i += kThreads) {
    pq = fmaf(sq[i], sq[i], pq);
    pk = fmaf(sk[i], sk[i], pk);
    pqk = fmaf(sq[i], sk[i], pqk);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    pq += __shfl_xor_sync(0xffffffffu, pq, o);
    pk += __shfl_xor_sync(0xffffffffu, pk, o);
    pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
  }
  if (lane == 0) {
    const int w = GDN_S(warp, kWarps);
    sred[0][w] = pq;
    sred[1][w] = pk;
    sred[2][w] = pqk;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f, c = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      a += sred[0][w];
      b += sred[1][w];
      c += sred[2][w];
    }
    red_out[0] = a;
    red_out[1] = b;
    red_out[2] = c;
  }
}

// ---------------------------------------------------------------------------
// Decode: one token per request.
// ---------------------------------------------------------------------------
// KDA (Kimi Delta Attention, the per-key-channel decay variant: a [B][hv][dk]
// gate logits, dt_bias [hv][dk]): column i of St decays by its own alpha_i,
//   u = v - St (alpha . k^) ; St' = St diag(alpha) + beta u k^T ;
//   o = St (alpha . q^) + beta u (k^ . q^).
template <int DK, int NIT, typename Tact, typename Tconv, bool KDA>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const StepArgs a) {
  pdl_wait();
  pdl_trigger();
  using M = RowMap<DK>;
  constexpr int R = NIT * M::RI;
  __shared__ float sq_[DK], sk_[DK], sv_[R], so_[R];
  __shared__ float sal_[KDA ? DK : 1];
  __shared__ float sraw_[kMaxW][2 * DK];
  __shared__ float sred[3][kWarps];
  __shared__ float sscal[8];
  const auto sq = GDN_SV(sq_, DK), sk = GDN_SV(sk_, DK), sv = GDN_SV(sv_, R), so = GDN_SV(so_, R);
  const auto sal = GDN_SV(sal_, KDA ? DK : 1);
  const auto sraw = GDN_SV(&sraw_[0][0], kMaxW * 2 * DK);  // [kMaxW][2 DK]
  const StepViews<DK, Tact, Tconv, KDA> g(a, 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.y;
  const int h = blockIdx.x / a.P, p = blockIdx.x % a.P;
  const int hq = h / a.G;
  const int row0 = p * R;
  const int nrows = min(R, a.dv - row0);
  const int csize = a.G * a.P;
  const int32_t slot = g.slot_ids[r];
  const int cls = slot_class(slot, a.num_slots);
  const auto out = g.out + (((size_t)r * a.hv + h) * a.dv + row0);
  if (cls) {  // the whole cluster shares r, so it skips together
    if (cls == 2 && blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int i = tid; i < nrows; i += kThreads) out[i] = from_f32<Tact>(0.f);
    return;
  }

  // 1. state rows in flight first
  const int seg = lane % M::LPR;
  const int rloc = warp * M::RW + lane / M::LPR;
  const auto St = g.ssm + (((size_t)slot * a.hv + h) * a.dv + row0) * DK;
  float4 s[NIT][4];
  load_rows<DK, NIT>(s, St, nrows, rloc, seg);

  // 2. conv1d + SiLU on the q/k channels of hq and the v channels of our rows
  const bool qk_writer = csize == 1 || cluster_ctarank() == 0;
  const auto conv = g.conv + (size_t)slot * (a.W - 1) * a.C;
  const auto x = g.qkv + (size_t)r * a.C;
  for (int i = tid; i < 2 * DK + nrows; i += kThreads) {
    const int c = channel_of<DK>(i, hq, h, a.hk, a.dv, row0);
    const auto w = g.conv_w + (size_t)c * a.W;
    float hist[kMaxW];
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxW - 1; ++j)
      if (j < a.W - 1) {
        hist[j] = to_f32(conv[(size_t)j * a.C + c]);
        acc = fmaf(w[j], hist[j], acc);
      }
    const float xv = to_f32(x[c]);
    acc = fmaf(w[a.W - 1], xv, acc);
    const float y = silu_f(acc);
    if (i < DK) {
      sq[i] = y;
    } else if (i < 2 * DK) {
      sk[i - DK] = y;
    } else {
      sv[i - 2 * DK] = y;
      // this CTA alone owns these channels: shift the history now
#pragma unroll
      for (int j = 0; j < kMaxW - 2; ++j)
        if (j < a.W - 2) conv[(size_t)j * a.C + c] = from_f32<Tconv>(hist[j + 1]);
      conv[(size_t)(a.W - 2) * a.C + c] = from_f32<Tconv>(xv);
    }
    if (i < 2 * DK && qk_writer) {
#pragma unroll
      for (int j = 0; j < kMaxW - 1; ++j)
        if (j < a.W - 1) sraw[j * 2 * DK + i] = hist[j];
      sraw[(a.W - 1) * 2 * DK + i] = xv;
    }
  }
  if (csize > 1) cluster_arrive_release();  // our reads of the shared history are done
  __syncthreads();

  // 3. L2 norms and gates
  block_norms<DK>(sq_, sk_, sred, sscal);
  if (tid == 0) {
    const float rq = rsqrtf(sscal[0] + kNormEps) * rsqrtf((float)DK);
    const float rk = rsqrtf(sscal[1] + kNormEps);
    sscal[3] = rq;
    sscal[4] = rk;
    sscal[5] = sscal[2] * rq * rk;  // k^ . q^
    if (!KDA) sscal[6] = gate_alpha(g.A_log[h], g.dt_bias[h], to_f32(g.a[(size_t)r * a.hv + h]));
    sscal[7] = sigmoid_f(to_f32(g.b[(size_t)r * a.hv + h]));
  }
  if (KDA) {
    const auto av = g.a + ((size_t)r * a.hv + h) * DK;
    for (int i = tid; i < DK; i += kThreads)
      sal[i] = gate_alpha(g.A_log[h], g.dt_bias[(size_t)h * DK + i], to_f32(av[i]));
  }
  __syncthreads();
  const float rq = sscal[3], rk = sscal[4], kq = sscal[5], alpha = KDA ? 1.f : sscal[6], beta = sscal[7];
  // kk = k^ (the rank-1 term); qq = alpha . q^ and, inside the dot product,
  // alpha . k^ (KDA; the scalar alpha of GDN is applied to the dot products)
  float4 kk[4], qq[4], al[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = M::col(c, seg);
    kk[c] = make_float4(sk[col] * rk, sk[col + 1] * rk, sk[col + 2] * rk, sk[col + 3] * rk);
    qq[c] = make_float4(sq[col] * rq, sq[col + 1] * rq, sq[col + 2] * rq, sq[col + 3] * rq);
    if (KDA) {
      al[c] = make_float4(sal[col], sal[col + 1], sal[col + 2], sal[col + 3]);
      qq[c] = make_float4(qq[c].x * al[c].x, qq[c].y * al[c].y, qq[c].z * al[c].z, qq[c].w * al[c].w);
    } else {
      al[c] = make_float4(alpha, alpha, alpha, alpha);
    }
  }

  // 4. gated delta rule + readout, row by row
  //    u = v - alpha St k^ ; St' = alpha St + beta u k^T ; o = St' q^
  //      = alpha (St q^) + beta u (k^ . q^)
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int row = it * M::RI + rloc;
    float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      dk_ += KDA ? dot4(make_float4(s[it][c].x * al[c].x, s[it][c].y * al[c].y, s[it][c].z * al[c].z,
                                    s[it][c].w * al[c].w),
                        kk[c])
                 : dot4(s[it][c], kk[c]);
      dq_ += dot4(s[it][c], qq[c]);
    }
#pragma unroll
    for (int o = M::LPR / 2; o; o >>= 1) {
      dk_ += __shfl_xor_sync(0xffffffffu, dk_, o);
      dq_ += __shfl_xor_sync(0xffffffffu, dq_, o);
    }
    if (row < nrows) {
      const float bu = beta * (sv[row] - alpha * dk_);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float4 v = s[it][c];
        v.x = fmaf(bu, kk[c].x, al[c].x * v.x);
        v.y = fmaf(bu, kk[c].y, al[c].y * v.y);
        v.z = fmaf(bu, kk[c].z, al[c].z * v.z);
        v.w = fmaf(bu, kk[c].w, al[c].w * v.w);
        st_stream(&vec_at<float4>(St, (size_t)row * DK + M::col(c, seg)), v);
      }
      if (seg == 0) so[row] = fmaf(bu, kq, alpha * dq_);
    }
  }
  __syncthreads();
  for (int i = tid; i < nrows; i += kThreads) out[i] = from_f32<Tact>(so[i]);

  // 5. q/k history: one writer per cluster, after every reader arrived
  if (csize > 1) cluster_wait_acquire();
  if (qk_writer) {
    for (int i = tid; i < 2 * DK; i += kThreads) {
      const int c = channel_of<DK>(i, hq, h, a.hk, a.dv, row0);
#pragma unroll
      for (int j = 0; j < kMaxW - 1; ++j)
        if (j < a.W - 1) conv[(size_t)j * a.C + c] = from_f32<Tconv>(sraw[(j + 1) * 2 * DK + i]);
    }
  }
}

// ---------------------------------------------------------------------------
// Speculative verify: T draft tokens per request from the working slot, which
// is only read; the state after draft t goes to spec slot spec_ids[r][t].
// The state rows stay in registers across the T steps.  KDA: the per-key-
// channel decay of every draft step (a [B][T][hv][dk]) from a [T][dk] table.
// ---------------------------------------------------------------------------
// offset (floats) of the KDA alpha table in the verify kernel's shared memory
__host__ __device__ constexpr size_t verify_alpha_off(int T, int nch, int R) {
  return ((size_t)T * nch + (size_t)T * R + (size_t)T * 5 + 3) & ~(size_t)3;
}

template <int DK, int NIT, typename Tact, typename Tconv, bool KDA>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const StepArgs a) {
  pdl_wait();
  pdl_trigger();
  using M = RowMap<DK>;
  constexpr int R = NIT * M::RI;
  constexpr int NCH = 2 * DK + R;  // channels handled: q, k, our v rows
  extern __shared__ __align__(16) float smem[];
  const size_t smem_floats = KDA ? verify_alpha_off(a.T, NCH, R) + (size_t)a.T * DK
                                 : (size_t)a.T * NCH + (size_t)a.T * R + (size_t)a.T * 5;
  const auto sm = GDN_SV(smem, smem_floats);
  const auto sy = sm;                                // [T][NCH]  conv+SiLU outputs
  const auto so = sm + (size_t)a.T * NCH;            // [T][R]    outputs
  const auto sscal = sm + (size_t)a.T * (NCH + R);   // [T][5]    rq, rk, kq, alpha, beta
  const auto salk = sm + (KDA ? verify_alpha_off(a.T, NCH, R) : 0);  // KDA: [T][DK] alpha
  const StepViews<DK, Tact, Tconv, KDA> g(a, a.T);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.y;
  const int h = blockIdx.x / a.P, p = blockIdx.x % a.P;
  const int hq = h / a.G;
  const int row0 = p * R;
  const int nrows = min(R, a.dv - row0);
  const int T = a.T;
  const int32_t slot = g.slot_ids[r];
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int t = 0; t < T; ++t) {
      const auto out = g.out + (((((size_t)r * T + t) * a.hv) + h) * a.dv + row0);
      for (int i = tid; i < nrows; i += kThreads) out[i] = from_f32<Tact>(0.f);
    }
    return;
  }

  const int seg = lane % M::LPR;
  const int rloc = warp * M::RW + lane / M::LPR;
  const auto St = g.ssm + (((size_t)slot * a.hv + h) * a.dv + row0) * DK;
  float4 s[NIT][4];
  load_rows<DK, NIT>(s, St, nrows, rloc, seg);

  // conv over the draft sequence; snapshot histories go straight to the spec
  // slots (v rows: this CTA; q/k channels: the first V head of the group)
  const bool qk_writer = (h % a.G) == 0 && p == 0;
  const auto conv = g.conv + (size_t)slot * (a.W - 1) * a.C;
  const auto sids = g.spec_ids + (size_t)r * T;
  for (int i = tid; i < NCH; i += kThreads) {
    if (i >= 2 * DK + nrows) continue;
    const int c = channel_of<DK>(i, hq, h, a.hk, a.dv, row0);
    const auto w = g.conv_w + (size_t)c * a.W;
    float win[kMaxW];  // win[0..W-2] = history, oldest first
#pragma unroll
    for (int j = 0; j < kMaxW - 1; ++j)
      if (j < a.W - 1) win[j] = to_f32(conv[(size_t)j * a.C + c]);
    const bool writes = i >= 2 * DK || qk_writer;
    for (int t = 0; t < T; ++t) {
      const float xv = to_f32(g.qkv[((size_t)r * T + t) * a.C + c]);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxW - 1; ++j)
        if (j < a.W - 1) acc = fmaf(w[j], win[j], acc);
      acc = fmaf(w[a.W - 1], xv, acc);
      sy[(size_t)t * NCH + i] = silu_f(acc);
      // advance the window
#pragma unroll
      for (int j = 0; j < kMaxW - 2; ++j)
        if (j < a.W - 2) win[j] = win[j + 1];
      win[a.W - 2] = xv;
      if (writes) {
        const int32_t sid = sids[t];
        if (slot_class(sid, a.spec_num_slots) == 0) {
          const auto sc = g.spec_conv + (size_t)sid * (a.W - 1) * a.C;
#pragma unroll
          for (int j = 0; j < kMaxW - 1; ++j)
            if (j < a.W - 1) sc[(size_t)j * a.C + c] = from_f32<Tconv>(win[j]);
        }
      }
    }
  }
  if (tid < T && blockIdx.x == 0 && slot_class(sids[tid], a.spec_num_slots) == 2)
    report(a.err, GDN_DEV_ERR_SLOT_OOB);
  __syncthreads();

  // per-token norms and gates: warp w handles tokens w, w+8, ...
  for (int t = warp; t < T; t += kWarps) {
    const auto yq = sy + (size_t)t * NCH;
    const auto yk = yq + DK;
    float pq = 0.f, pk = 0.f, pqk = 0.f;
    for (int i = lane; i < DK; i += 32) {
      pq = fmaf(yq[i], yq[i], pq);
      pk = fmaf(yk[i], yk[i], pk);
      pqk = fmaf(yq[i], yk[i], pqk);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      pq += __shfl_xor_sync(0xffffffffu, pq, o);
      pk += __shfl_xor_sync(0xffffffffu, pk, o);
      pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
    }
    if (lane == 0) {
      const size_t rt = (size_t)r * T + t;
      const float rq = rsqrtf(pq + kNormEps) * rsqrtf((float)DK);
      const float rk = rsqrtf(pk + kNormEps);
      sscal[t * 5 + 0] = rq;
      sscal[t * 5 + 1] = rk;
      sscal[t * 5 + 2] = pqk * rq * rk;
      if (!KDA) sscal[t * 5 + 3] = gate_alpha(g.A_log[h], g.dt_bias[h], to_f32(g.a[rt * a.hv + h]));
      sscal[t * 5 + 4] = sigmoid_f(to_f32(g.b[rt * a.hv + h]));
    }
  }
  if (KDA) {
    for (int e = tid; e < T * DK; e += kThreads) {
      const int t = e / DK, i = e % DK;
      const size_t rt = (size_t)r * T + t;
      salk[e] = gate_alpha(g.A_log[h], g.dt_bias[(size_t)h * DK + i], to_f32(g.a[(rt * a.hv + h) * DK + i]));
    }
  }
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    const auto yq = sy + (size_t)t * NCH;
    const auto yk = yq + DK;
    const auto yv = yk + DK;
    const float rq = sscal[t * 5 + 0], rk = sscal[t * 5 + 1], kq = sscal[t * 5 + 2];
    const float alpha = KDA ? 1.f : sscal[t * 5 + 3], beta = sscal[t * 5 + 4];
    float4 kk[4], qq[4], al[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 k4 = vec_at<float4>(yk, M::col(c, seg));
      const float4 q4 = vec_at<float4>(yq, M::col(c, seg));
      kk[c] = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
      qq[c] = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
      al[c] = KDA ? vec_at<float4>(salk, (size_t)t * DK + M::col(c, seg)) : make_float4(alpha, alpha, alpha, alpha);
    }
    const int32_t sid = sids[t];
    const bool keep = slot_class(sid, a.spec_num_slots) == 0;
    const auto Sp = g.spec_ssm + (keep ? (((size_t)sid * a.hv + h) * a.dv + row0) * DK : 0);
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int row = it * M::RI + rloc;
      float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // KDA: the decayed row St diag(alpha) meets k^ and q^
        const float4 sa = KDA ? make_float4(s[it][c].x * al[c].x, s[it][c].y * al[c].y, s[it][c].z * al[c].z,
                                            s[it][c].w * al[c].w)
                              : s[it][c];
        dk_ += dot4(sa, kk[c]);
        dq_ += dot4(sa, qq[c]);
      }
#pragma unroll
      for (int o = M::LPR / 2; o; o >>= 1) {
        dk_ += __shfl_xor_sync(0xffffffffu, dk_, o);
        dq_ += __shfl_xor_sync(0xffffffffu, dq_, o);
      }
      const float bu = row < nrows ? beta * (yv[row] - alpha * dk_) : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float4& v = s[it][c];
        v.x = fmaf(bu, kk[c].x, al[c].x * v.x);
        v.y = fmaf(bu, kk[c].y, al[c].y * v.y);
        v.z = fmaf(bu, kk[c].z, al[c].z * v.z);
        v.w = fmaf(bu, kk[c].w, al[c].w * v.w);
      }
      if (row < nrows) {
        if (keep) {
#pragma unroll
          for (int c = 0; c < 4; ++c) st_stream(&vec_at<float4>(Sp, (size_t)row * DK + M::col(c, seg)), s[it][c]);
        }
        if (seg == 0) so[(size_t)t * R + row] = fmaf(bu, kq, alpha * dq_);
      }
    }
  }
  __syncthreads();
  for (int t = 0; t < T; ++t) {
    const auto out = g.out + (((((size_t)r * T + t) * a.hv) + h) * a.dv + row0);
    for (int i = tid; i < nrows; i += kThreads) out[i] = from_f32<Tact>(so[(size_t)t * R + i]);
  }
}

// ---------------------------------------------------------------------------
// KDA prefill, the recurrent form (fp32, CUDA cores): one CTA per (sequence,
// V head, row part) walks the sequence token by token in windows of kTW
// tokens.  The raw inputs of window w+1 (the CTA's qkv channels and the gate
// logits) are copied into shared memory (cp.async, double-buffered) while
// window w is computed: conv1d + SiLU from the staged inputs and the conv
// history (shared memory, one column per channel, owned by the thread that
// convolves it), per-token norms, beta and the per-key-channel alphas, then
// the KDA update of the CTA's state rows, which stay in registers for the
// whole sequence.  At every block boundary the rows go to their checkpoint
// slot; at the end to the working slot.  The conv histories of the
// checkpoints and of the final state come from the prefill's history kernel.
// ---------------------------------------------------------------------------
constexpr int kTW = 16;


struct KdaPrefillArgs {
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
  int32_t hk, hv, dv, W, C, G, P;
};

// shared memory of kda_prefill_kernel (byte offsets, each 16-byte aligned)
template <int DK, int NIT, typename Tact>
struct KdaPrefillSmem {
  static constexpr int R = NIT * RowMap<DK>::RI;
  static constexpr int NCH = 2 * DK + R;  // q, k and the CTA's v rows
  static constexpr size_t xr = 0;                                             // [2][kTW][NCH] raw inputs
  static constexpr size_t ga = xr + 2 * kTW * NCH * sizeof(Tact);             // [2][kTW][DK] gate logits
  static constexpr size_t xh = ga + 2 * kTW * DK * sizeof(Tact);              // [kMaxW-1][NCH] conv history
  static constexpr size_t cw = xh + (kMaxW - 1) * NCH * sizeof(float);        // [kMaxW][NCH] conv weights
  static constexpr size_t sy = cw + kMaxW * NCH * sizeof(float);              // [kTW][NCH] conv + SiLU
  static constexpr size_t so = sy + kTW * NCH * sizeof(float);                // [kTW][R] outputs
  static constexpr size_t sc = so + kTW * R * sizeof(float);                  // [kTW][4] rq, rk, k^.q^, beta
  static constexpr size_t al = sc + kTW * 4 * sizeof(float);                  // [kTW][DK] alphas
  static constexpr size_t sb = al + kTW * DK * sizeof(float);                 // [2][kTW] beta logits
  static constexpr size_t bytes = sb + 2 * kTW * sizeof(float);
  static_assert(ga % 16 == 0 && xh % 16 == 0 && cw % 16 == 0 && sy % 16 == 0 && so % 16 == 0 && al % 16 == 0,
                "shared arrays must start 16-byte aligned");
};

// Raw inputs of tokens [tok, tok + nt) into the staging buffers: the CTA's
// channels of qkv (q, k, then its v rows) and the head's gate logits.  ASYNC:
// 16-byte cp.async pieces (every segment start and length a multiple of 16
// bytes, checked on the host); otherwise element copies.
// xr, gs: views of one staging buffer each ([kTW][NCH] and [kTW][DK])
template <int DK, int NIT, typename Tact, bool ASYNC, typename VS>
__device__ __forceinline__ void kda_stage(const KdaPrefillArgs& a, const VS& xr, const VS& gs, int64_t tok, int nt,
                                          int nrows, int hq, int h, int row0) {
  using L = KdaPrefillSmem<DK, NIT, Tact>;
  const auto qkv = GDN_GV(reinterpret_cast<const Tact*>(a.qkv), a.total * a.C);
  const auto ga = GDN_GV(reinterpret_cast<const Tact*>(a.a), a.total * a.hv * DK);
  const int nch = 2 * DK + nrows;
  if constexpr (ASYNC) {
    constexpr int E = 16 / sizeof(Tact);  // elements per piece
    const int per_row = nch / E;
    for (int p = threadIdx.x; p < nt * per_row; p += kThreads) {
      const int t = p / per_row, e = (p % per_row) * E;
      const size_t src = (size_t)(tok + t) * a.C + channel_of<DK>(e, hq, h, a.hk, a.dv, row0);
      if (xr.has(t * L::NCH + e, E) && qkv.has(src, E)) cp_async16(xr.p + t * L::NCH + e, qkv.p + src);
    }
    for (int p = threadIdx.x; p < nt * (DK / E); p += kThreads) {
      const int t = p / (DK / E), e = (p % (DK / E)) * E;
      const size_t src = ((size_t)(tok + t) * a.hv + h) * DK + e;
      if (gs.has(t * DK + e, E) && ga.has(src, E)) cp_async16(gs.p + t * DK + e, ga.p + src);
    }
  } else {
    for (int p = threadIdx.x; p < nt * nch; p += kThreads) {
      const int t = p / nch, e = p % nch;
      xr[t * L::NCH + e] = qkv[(size_t)(tok + t) * a.C + channel_of<DK>(e, hq, h, a.hk, a.dv, row0)];
    }
    for (int p = threadIdx.x; p < nt * DK; p += kThreads) {
      const int t = p / DK, e = p % DK;
      gs[t * DK + e] = ga[((size_t)(tok + t) * a.hv + h) * DK + e];
    }
  }
}

template <int DK, int NIT, typename Tact, typename Tconv, bool ASYNC>
__global__ void __launch_bounds__(kThreads, 2) kda_prefill_kernel(const KdaPrefillArgs a) {
  pdl_wait();
  pdl_trigger();
  using M = RowMap<DK>;
  using L = KdaPrefillSmem<DK, NIT, Tact>;
  constexpr int R = L::R, NCH = L::NCH;
  constexpr int kCPT = (NCH + kThreads - 1) / kThreads;  // channels per thread
  static_assert(kThreads % DK == 0, "a thread's gate channel must be fixed");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const auto xr = GDN_SV(reinterpret_cast<Tact*>(smem_raw + L::xr), 2 * kTW * NCH);
  const auto gs = GDN_SV(reinterpret_cast<Tact*>(smem_raw + L::ga), 2 * kTW * DK);
  const auto xh = GDN_SV(reinterpret_cast<float*>(smem_raw + L::xh), (kMaxW - 1) * NCH);
  const auto cwt = GDN_SV(reinterpret_cast<float*>(smem_raw + L::cw), kMaxW * NCH);
  const auto sy = GDN_SV(reinterpret_cast<float*>(smem_raw + L::sy), kTW * NCH);
  const auto so = GDN_SV(reinterpret_cast<float*>(smem_raw + L::so), kTW * R);
  const auto sscal = GDN_SV(reinterpret_cast<float*>(smem_raw + L::sc), kTW * 4);
  const auto salk = GDN_SV(reinterpret_cast<float*>(smem_raw + L::al), kTW * DK);
  const auto sb = GDN_SV(reinterpret_cast<float*>(smem_raw + L::sb), 2 * kTW);
  const int n_seq = gridDim.y;
  const auto ssm = GDN_GV(a.ssm, (long long)a.num_slots * a.hv * a.dv * DK);
  const auto ck_ssm = GDN_GV(a.ck_ssm, (long long)a.ck_num_slots * a.hv * a.dv * DK);
  const auto conv_w = GDN_GV(a.conv_w, (long long)a.C * a.W);
  const auto cu_seqlens = GDN_GV(a.cu_seqlens, n_seq + 1);
  const auto start_pos = GDN_GV(a.start_pos, n_seq);
  const auto slot_ids = GDN_GV(a.slot_ids, n_seq);
  const auto ckpt_ids = GDN_GV(a.ckpt_ids, (long long)n_seq * a.max_ckpt);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.y;
  const int h = blockIdx.x / a.P, p = blockIdx.x % a.P;
  const int hq = h / a.G;
  const int row0 = p * R;
  const int nrows = min(R, a.dv - row0);
  const int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1], len = t1 - t0, p0 = start_pos[n];
  if (t0 < 0 || len < 0 || t1 > a.total || p0 < 0) {
    if (blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const auto out = GDN_GV(reinterpret_cast<Tact*>(a.out), a.total * a.hv * a.dv);
  const int32_t slot = slot_ids[n];
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && blockIdx.x == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * nrows; e += kThreads)
      out[((t0 + e / nrows) * a.hv + h) * a.dv + row0 + e % nrows] = from_f32<Tact>(0.f);
    return;
  }
  if (len == 0) return;

  const auto gb = GDN_GV(reinterpret_cast<const Tact*>(a.b), a.total * a.hv);
  // the first window's inputs in flight before anything else
  kda_stage<DK, NIT, Tact, ASYNC>(a, xr, gs, t0, len < kTW ? (int)len : kTW, nrows, hq, h, row0);
  if constexpr (ASYNC) cp_async_commit();
  if (tid < kTW && tid < len) sb[tid] = to_f32(gb[(size_t)(t0 + tid) * a.hv + h]);

  const int seg = lane % M::LPR;
  const int rloc = warp * M::RW + lane / M::LPR;
  const auto St = ssm + (((size_t)slot * a.hv + h) * a.dv + row0) * DK;
  float4 s[NIT][4];
  load_rows<DK, NIT>(s, St, nrows, rloc, seg);

  // conv weights and history, right-aligned in kMaxW taps (the newest input
  // last; the taps before the width are zero), one column per channel
  const auto hist = GDN_GV(reinterpret_cast<const Tconv*>(a.conv), (long long)a.num_slots * (a.W - 1) * a.C) +
                    (size_t)slot * (a.W - 1) * a.C;
  const int lead = kMaxW - a.W;
  for (int i = tid; i < 2 * DK + nrows; i += kThreads) {
    const int ch = channel_of<DK>(i, hq, h, a.hk, a.dv, row0);
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) cwt[j * NCH + i] = j >= lead ? conv_w[(size_t)ch * a.W + (j - lead)] : 0.f;
#pragma unroll
    for (int j = 0; j < kMaxW - 1; ++j) xh[j * NCH + i] = j >= lead ? to_f32(hist[(size_t)(j - lead) * a.C + ch]) : 0.f;
  }
  const float eA = expf(GDN_GV(a.A_log, a.hv)[h]);
  // the alphas this thread computes are of channel tid % DK
  const float dtb = GDN_GV(a.dt_bias, (long long)a.hv * DK)[(size_t)h * DK + tid % DK];
  const int64_t blk0 = p0 / a.ckpt_block;
  // the next block boundary (absolute position) and its checkpoint index
  int64_t next_bd = (blk0 + 1) * a.ckpt_block;
  int64_t ck_idx = 0;
  if constexpr (ASYNC) cp_async_wait_all();
  __syncthreads();

  for (int64_t w0 = 0; w0 < len; w0 += kTW) {
    const int cur = (int)((w0 / kTW) & 1), nxt = cur ^ 1;
    const int nt = len - w0 < kTW ? (int)(len - w0) : kTW;
    const int64_t wn = w0 + kTW;
    const int ntn = wn >= len ? 0 : (len - wn < kTW ? (int)(len - wn) : kTW);
    // 0. the next window's inputs
    float bnext = 0.f;
    if (ntn > 0) {
      kda_stage<DK, NIT, Tact, ASYNC>(a, xr + nxt * kTW * NCH, gs + nxt * kTW * DK, t0 + wn, ntn, nrows, hq, h,
                                      row0);
      if constexpr (ASYNC) cp_async_commit();
      if (tid < ntn) bnext = to_f32(gb[(size_t)(t0 + wn + tid) * a.hv + h]);
    }
    const auto x = xr + cur * kTW * NCH;
    const auto gw = gs + cur * kTW * DK;
    // 1. conv1d + SiLU of the window's tokens (oldest tap first)
#pragma unroll
    for (int ci = 0; ci < kCPT; ++ci) {
      const int i = tid + ci * kThreads;
      if (i < 2 * DK + nrows) {
        float w[kMaxW], win[kMaxW - 1];
#pragma unroll
        for (int j = 0; j < kMaxW; ++j) w[j] = cwt[j * NCH + i];
#pragma unroll
        for (int j = 0; j < kMaxW - 1; ++j) win[j] = xh[j * NCH + i];
        // unrolled: the tokens' products and SiLUs are independent
#pragma unroll
        for (int t = 0; t < kTW; ++t) {
          if (t < nt) {
            const float xv = to_f32(x[t * NCH + i]);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxW - 1; ++j) acc = fmaf(w[j], win[j], acc);
            acc = fmaf(w[kMaxW - 1], xv, acc);
            sy[t * NCH + i] = __fdividef(acc, 1.f + exp_ftz(-acc));  // SiLU
#pragma unroll
            for (int j = 0; j < kMaxW - 2; ++j) win[j] = win[j + 1];
            win[kMaxW - 2] = xv;
          }
        }
#pragma unroll
        for (int j = 0; j < kMaxW - 1; ++j) xh[j * NCH + i] = win[j];
      }
    }
    __syncthreads();
    // 2. per token: q/k norms, k^.q^, beta (a warp per token) and the alphas
    for (int t = warp; t < nt; t += kWarps) {
      const auto yq = sy + t * NCH;
      const auto yk = yq + DK;
      float pq = 0.f, pk = 0.f, pqk = 0.f;
      for (int i = lane; i < DK; i += 32) {
        pq = fmaf(yq[i], yq[i], pq);
        pk = fmaf(yk[i], yk[i], pk);
        pqk = fmaf(yq[i], yk[i], pqk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        pq += __shfl_xor_sync(0xffffffffu, pq, o);
        pk += __shfl_xor_sync(0xffffffffu, pk, o);
        pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
      }
      if (lane == 0) {
        const float rq = rsqrtf(pq + kNormEps) * rsqrtf((float)DK);
        const float rk = rsqrtf(pk + kNormEps);
        sscal[t * 4 + 0] = rq;
        sscal[t * 4 + 1] = rk;
        sscal[t * 4 + 2] = pqk * rq * rk;
        sscal[t * 4 + 3] = sigmoid_f(sb[cur * kTW + t]);
      }
    }
    // alpha = exp(-exp(A_log) * softplus(a + dt_bias))
    for (int e = tid; e < nt * DK; e += kThreads) salk[e] = expf(-eA * softplus_f(to_f32(gw[e]) + dtb));
    __syncthreads();
    // 3. the recurrence over the window's tokens
    for (int t = 0; t < nt; ++t) {
      const auto yq = sy + t * NCH;
      const auto yk = yq + DK;
      const auto yv = yk + DK;
      const float rq = sscal[t * 4 + 0], rk = sscal[t * 4 + 1], kq = sscal[t * 4 + 2], beta = sscal[t * 4 + 3];
      // unnormalised q and k: the norms scale the dot products and the update
      float4 kr[4], qr[4], al[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        kr[c] = vec_at<float4>(yk, M::col(c, seg));
        qr[c] = vec_at<float4>(yq, M::col(c, seg));
        al[c] = vec_at<float4>(salk, t * DK + M::col(c, seg));
      }
      // a block boundary after this token: its checkpoint slot
      bool to_ck = false;
      auto ck = ck_ssm;
      if (p0 + w0 + t + 1 == next_bd) {
        const int64_t idx = ck_idx++;
        next_bd += a.ckpt_block;
        if (idx < a.max_ckpt) {
          const int32_t cid = ckpt_ids[(size_t)n * a.max_ckpt + idx];
          const int cc = slot_class(cid, a.ck_num_slots);
          if (cc == 0) {
            to_ck = true;
            ck = ck_ssm + (((size_t)cid * a.hv + h) * a.dv + row0) * DK;
          } else if (cc == 2 && tid == 0) {
            report(a.err, GDN_DEV_ERR_SLOT_OOB);
          }
        }
      }
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int row = it * M::RI + rloc;
        // the rows become St diag(alpha) in place; the update adds beta u k^T
        float2 dk2 = make_float2(0.f, 0.f), dq2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float4& v = s[it][c];
          const float2 lo = mul2(lo2(v), lo2(al[c])), hi = mul2(hi2(v), hi2(al[c]));
          v = make_float4(lo.x, lo.y, hi.x, hi.y);
          dk2 = fma2(hi, hi2(kr[c]), fma2(lo, lo2(kr[c]), dk2));
          dq2 = fma2(hi, hi2(qr[c]), fma2(lo, lo2(qr[c]), dq2));
        }
        float dk_ = dk2.x + dk2.y, dq_ = dq2.x + dq2.y;
#pragma unroll
        for (int o = M::LPR / 2; o; o >>= 1) {
          dk_ += __shfl_xor_sync(0xffffffffu, dk_, o);
          dq_ += __shfl_xor_sync(0xffffffffu, dq_, o);
        }
        dq_ *= rq;
        const float bu = row < nrows ? beta * (yv[row] - dk_ * rk) : 0.f;
        const float2 buk = make_float2(bu * rk, bu * rk);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float4& v = s[it][c];
          const float2 lo = fma2(buk, lo2(kr[c]), lo2(v)), hi = fma2(buk, hi2(kr[c]), hi2(v));
          v = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
        if (row < nrows) {
          if (to_ck) {
#pragma unroll
            for (int c = 0; c < 4; ++c) st_stream(&vec_at<float4>(ck, (size_t)row * DK + M::col(c, seg)), s[it][c]);
          }
          if (seg == 0) so[t * R + row] = fmaf(bu, kq, dq_);
        }
      }
    }
    __syncthreads();
    // 4. the window's outputs; the next window's beta logits and inputs land
    for (int e = tid; e < nt * nrows; e += kThreads) {
      const int t = e / nrows, i = e % nrows;
      out[((size_t)(t0 + w0 + t) * a.hv + h) * a.dv + row0 + i] = from_f32<Tact>(so[t * R + i]);
    }
    if (tid < ntn) sb[nxt * kTW + tid] = bnext;
    if constexpr (ASYNC) cp_async_wait_all();
    __syncthreads();
  }
  // the final state
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int row = it * M::RI + rloc;
    if (row < nrows) {
#pragma unroll
      for (int c = 0; c < 4; ++c) st_stream(&vec_at<float4>(St, (size_t)row * DK + M::col(c, seg)), s[it][c]);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int DK, int NIT, typename Tact, typename Tconv>
cudaError_t launch_decode_t(const StepArgs& a, bool kda, cudaStream_t s) {
  // the G*P CTAs of a QK head form one cluster (shared q/k history writer)
  const dim3 cluster(a.G * a.P > 1 ? (unsigned)(a.G * a.P) : 1u);
  const dim3 grid((unsigned)(a.hv * a.P), (unsigned)a.B);
  if (kda) return launch_pdl(decode_kernel<DK, NIT, Tact, Tconv, true>, grid, dim3(kThreads), 0, s, cluster, a);
  return launch_pdl(decode_kernel<DK, NIT, Tact, Tconv, false>, grid, dim3(kThreads), 0, s, cluster, a);
}

template <int DK, int NIT, typename Tact, typename Tconv>
cudaError_t launch_verify_t(const StepArgs& a, bool kda, cudaStream_t s) {
  constexpr int R = NIT * RowMap<DK>::RI;
  const size_t smem = kda ? sizeof(float) * (verify_alpha_off(a.T, 2 * DK + R, R) + (size_t)a.T * DK)
                          : sizeof(float) * ((size_t)a.T * (2 * DK + R) + (size_t)a.T * R + (size_t)a.T * 5);
  auto k = kda ? verify_kernel<DK, NIT, Tact, Tconv, true> : verify_kernel<DK, NIT, Tact, Tconv, false>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k, dim3((unsigned)(a.hv * a.P), (unsigned)a.B), dim3(kThreads), smem, s, dim3(1), a);
}

template <int DK, int NIT>
cudaError_t dispatch_dtype(bool verify, bool kda, const StepArgs& a, int act, int cv, cudaStream_t s) {
  if (act == GDN_F32 && cv == GDN_F32)
    return verify ? launch_verify_t<DK, NIT, float, float>(a, kda, s)
                  : launch_decode_t<DK, NIT, float, float>(a, kda, s);
  if (act == GDN_BF16 && cv == GDN_BF16)
    return verify ? launch_verify_t<DK, NIT, __nv_bfloat16, __nv_bfloat16>(a, kda, s)
                  : launch_decode_t<DK, NIT, __nv_bfloat16, __nv_bfloat16>(a, kda, s);
  return verify ? launch_verify_t<DK, NIT, __nv_bfloat16, float>(a, kda, s)
                : launch_decode_t<DK, NIT, __nv_bfloat16, float>(a, kda, s);
}

template <int DK, int NIT, typename Tact, typename Tconv>
cudaError_t launch_kda_prefill_t(const KdaPrefillArgs& a, int32_t n_seq, bool async, cudaStream_t s) {
  const size_t smem = KdaPrefillSmem<DK, NIT, Tact>::bytes;
  auto k = async ? kda_prefill_kernel<DK, NIT, Tact, Tconv, true> : kda_prefill_kernel<DK, NIT, Tact, Tconv, false>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k, dim3((unsigned)(a.hv * a.P), (unsigned)n_seq), dim3(kThreads), smem, s, dim3(1), a);
}

template <int DK, int NIT>
cudaError_t dispatch_kda_prefill(const KdaPrefillArgs& a, int32_t n_seq, int act, int cv, bool async,
                                 cudaStream_t s) {
  if (act == GDN_F32 && cv == GDN_F32) return launch_kda_prefill_t<DK, NIT, float, float>(a, n_seq, async, s);
  if (act == GDN_BF16 && cv == GDN_BF16)
    return launch_kda_prefill_t<DK, NIT, __nv_bfloat16, __nv_bfloat16>(a, n_seq, async, s);
  return launch_kda_prefill_t<DK, NIT, __nv_bfloat16, float>(a, n_seq, async, s);
}

// rows-per-CTA choice: fewer rows (more CTAs, smaller clusters of work) when
// the batch is small, so that enough bytes are in flight to cover HBM latency.
int choose_nit(int dk, int dv, int units, int G, bool verify) {
  if (dk == 16) return 1;
  if (verify) {  // GDN_VERIFY_NIT=1|2|4 fixes the verify tile, for measurement
    const char* e = std::getenv("GDN_VERIFY_NIT");
    const int f = e ? std::atoi(e) : 0;
    if (f == 1 || f == 2 || (f == 4 && dk == 128)) return f;
  }
  const int ri = kWarps * (32 / (dk / 16));
  int nit = dk == 64 ? 2 : 4;
  const int target = verify ? 512 : 1024;  // CTAs wanted before the largest tile is used
  while (nit > 1 && (long)units * ((dv + nit * ri - 1) / (nit * ri)) < target) nit >>= 1;
  // a cluster spans G V heads x P row-parts; keep it within the portable 8
  while (!verify && nit < (dk == 64 ? 2 : 4) && G * ((dv + nit * ri - 1) / (nit * ri)) > 8) nit <<= 1;
  return nit;
}

// Kernel choice between the persistent TMA-fed kernels (dk 128, width 4;
// decode also G*dv <= 256) and the per-head kernels, by batch (below).
// GDN_DECODE_PATH=rows / tma forces either for decode and verify, for
// measurement.
int forced_path() {  // read on every call, so a process can time both paths
  const char* e = std::getenv("GDN_DECODE_PATH");
  if (!e) return 0;
  if (!std::strcmp(e, "tma")) return 1;
  if (!std::strcmp(e, "rows")) return 2;
  return 0;
}

// Decode: the persistent TMA-fed kernel from a quarter of an item (request x
// QK head) per SM up; below that its few CTAs each stream a whole 128 KiB
// group and the per-head kernel, which spreads a request's rows over more
// CTAs, is faster (GPU time per step, Qwen3.5-shaped layer: batch 1: 4.4 us vs
// 6.9; batch 2: 4.8 vs 7.0; batch 4: 8.9 vs 7.3).
bool use_tma_decode(const gdn_dims& d, int32_t B, const void* qkv, const gdn_params& p) {
  if (!decode_tma_supported(d, qkv, p)) return false;
  const int f = forced_path();
  if (f) return f != 2;
  return 4L * B * d.hk > sm_count();
}

// Verify: the persistent TMA-fed kernel from 3 (request, V head) heads per
// SM up (Qwen3.5-shaped layer, T = 8, its work split evenly by 32-row stages:
// 0.71 / 0.78 / 0.85 / 0.88 of HBM at batch 16 / 32 / 64 / 128 against 0.68
// for the per-head kernel at batch 16); below that its per-segment prologue
// (the q/k conv) is not hidden and the per-head kernel is faster.
// GDN_DECODE_PATH=tma / rows forces either, for measurement.
bool use_tma_verify(const gdn_dims& d, int32_t B, int32_t T, const void* qkv, const gdn_params& p) {
  if (!verify_tma_supported(d, T, qkv, p)) return false;
  const int f = forced_path();
  if (f) return f == 1;
  return (long)B * d.hv >= 3L * sm_count();
}

gdn_status run_step(bool verify, bool kda, const gdn_dims* dims, const gdn_pool& work, const gdn_pool* spec,
                    const gdn_params* params, const int32_t* slot_ids, const int32_t* spec_ids,
                    int32_t B, int32_t T, const void* qkv, const void* a, const void* b, void* out,
                    uint32_t* dev_err, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (B < 0 || (verify && (T < 1))) return GDN_ERR_INVALID_ARG;
  if (verify && T > kMaxT) return GDN_ERR_UNSUPPORTED;
  if (B == 0) return GDN_OK;
  if (B > 65535) return GDN_ERR_UNSUPPORTED;
  if ((st = check_pool(*dims, work)) != GDN_OK) return st;
  if (verify && (st = check_pool(*dims, *spec)) != GDN_OK) return st;
  if (!params || !params->conv_w || !params->A_log || !params->dt_bias) return GDN_ERR_INVALID_ARG;
  if (!slot_ids || !qkv || !a || !b || !out || (verify && !spec_ids)) return GDN_ERR_INVALID_ARG;
  const int G = dims->hv / dims->hk;
  if (G > 8) return GDN_ERR_UNSUPPORTED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // KDA's gate logits and dt_bias reach the TMA-fed kernel by bulk copies
  const bool kda_aligned = !kda || (aligned(a, 16) && aligned(params->dt_bias, 16));
  if (!verify && kda_aligned && use_tma_decode(*dims, B, qkv, *params)) {
    cudaError_t e = decode_tma_launch(*dims, work, *params, slot_ids, B, qkv, a, b, out, dev_err, kda, cs);
    if (e == cudaSuccess) count_launch(kda ? GDN_K_KDA_DECODE : GDN_K_DECODE);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  if (verify && kda_aligned && use_tma_verify(*dims, B, T, qkv, *params)) {
    cudaError_t e = verify_tma_launch(*dims, work, *spec, *params, slot_ids, spec_ids, B, T, qkv, a,
                                      b, out, dev_err, kda, cs);
    if (e == cudaSuccess) count_launch(kda ? GDN_K_KDA_VERIFY : GDN_K_SPEC_VERIFY);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  StepArgs s = {};
  s.ssm = work.ssm;
  s.conv = work.conv;
  s.num_slots = work.num_slots;
  if (verify) {
    s.spec_ssm = spec->ssm;
    s.spec_conv = spec->conv;
    s.spec_num_slots = spec->num_slots;
    s.spec_ids = spec_ids;
    s.T = T;
  }
  s.conv_w = params->conv_w;
  s.A_log = params->A_log;
  s.dt_bias = params->dt_bias;
  s.slot_ids = slot_ids;
  s.B = B;
  s.qkv = qkv;
  s.a = a;
  s.b = b;
  s.out = out;
  s.err = dev_err;
  s.hk = dims->hk;
  s.hv = dims->hv;
  s.dv = dims->dv;
  s.W = dims->conv_width;
  s.C = (int32_t)channels(*dims);
  s.G = G;
  const int nit = choose_nit(dims->dk, dims->dv, B * dims->hv, G, verify);
  const int ri = kWarps * (32 / (dims->dk / 16));
  s.P = (dims->dv + nit * ri - 1) / (nit * ri);
  if (!verify && G * s.P > 8) return GDN_ERR_UNSUPPORTED;
  if ((long)dims->hv * s.P > 2147483647L) return GDN_ERR_UNSUPPORTED;
  const int act = dims->act_dtype, cv = dims->conv_dtype;
  cudaError_t e = cudaErrorInvalidValue;
  switch (dims->dk) {
    case 16: e = dispatch_dtype<16, 1>(verify, kda, s, act, cv, cs); break;
    case 64:
      e = nit == 1 ? dispatch_dtype<64, 1>(verify, kda, s, act, cv, cs)
                   : dispatch_dtype<64, 2>(verify, kda, s, act, cv, cs);
      break;
    case 128:
      e = nit == 1   ? dispatch_dtype<128, 1>(verify, kda, s, act, cv, cs)
          : nit == 2 ? dispatch_dtype<128, 2>(verify, kda, s, act, cv, cs)
                     : dispatch_dtype<128, 4>(verify, kda, s, act, cv, cs);
      break;
  }
  if (e == cudaSuccess)
    count_launch(kda ? (verify ? GDN_K_KDA_VERIFY : GDN_K_KDA_DECODE) : verify ? GDN_K_SPEC_VERIFY : GDN_K_DECODE);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

// the decode step's kernel choice for batch B, for the mixed step
bool decode_takes_tma(const gdn_dims& d, int32_t B, const void* qkv, const gdn_params& p) {
  return use_tma_decode(d, B, qkv, p);
}
}  // namespace gdn

extern "C" gdn_status gdn_decode_step(const gdn_dims* dims, gdn_pool pool, const gdn_params* params,
                                      const int32_t* slot_ids, int32_t B, const void* qkv,
                                      const void* a, const void* b, void* out, uint32_t* dev_err,
                                      void* stream) {
  return gdn::run_step(false, false, dims, pool, nullptr, params, slot_ids, nullptr, B, 1, qkv, a, b, out,
                       dev_err, stream);
}

extern "C" gdn_status gdn_kda_decode_step(const gdn_dims* dims, gdn_pool pool, const gdn_params* params,
                                          const int32_t* slot_ids, int32_t B, const void* qkv,
                                          const void* a, const void* b, void* out, uint32_t* dev_err,
                                          void* stream) {
  return gdn::run_step(false, true, dims, pool, nullptr, params, slot_ids, nullptr, B, 1, qkv, a, b, out,
                       dev_err, stream);
}

extern "C" gdn_status gdn_kda_spec_verify(const gdn_dims* dims, gdn_pool work, gdn_pool spec,
                                          const gdn_params* params, const int32_t* slot_ids,
                                          const int32_t* spec_ids, int32_t B, int32_t T, const void* qkv,
                                          const void* a, const void* b, void* out, uint32_t* dev_err,
                                          void* stream) {
  return gdn::run_step(true, true, dims, work, &spec, params, slot_ids, spec_ids, B, T, qkv, a, b, out,
                       dev_err, stream);
}

extern "C" gdn_status gdn_spec_verify(const gdn_dims* dims, gdn_pool work, gdn_pool spec,
                                      const gdn_params* params, const int32_t* slot_ids,
                                      const int32_t* spec_ids, int32_t B, int32_t T,
                                      const void* qkv, const void* a, const void* b, void* out,
                                      uint32_t* dev_err, void* stream) {
  return gdn::run_step(true, false, dims, work, &spec, params, slot_ids, spec_ids, B, T, qkv, a, b, out,
                       dev_err, stream);
}

extern "C" gdn_status gdn_kda_prefill(const gdn_dims* dims, gdn_pool pool, gdn_pool ckpt,
                                      const gdn_params* params, const int32_t* slot_ids,
                                      const int32_t* cu_seqlens, const int64_t* start_pos, int32_t n_seq,
                                      int64_t total_tokens, const int32_t* ckpt_ids, int32_t max_ckpt,
                                      int32_t ckpt_block, const void* qkv, const void* a, const void* b,
                                      void* out, uint32_t* dev_err, void* stream) {
  using namespace gdn;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (n_seq < 0 || total_tokens < 0 || max_ckpt < 0) return GDN_ERR_INVALID_ARG;
  if (ckpt_block <= 0 || ckpt_block % 64) return GDN_ERR_INVALID_ARG;
  if (n_seq == 0) return GDN_OK;
  if (n_seq > 65535 || total_tokens > 2147483647LL || max_ckpt > 4 * 65535) return GDN_ERR_UNSUPPORTED;
  if ((st = check_pool(*dims, pool)) != GDN_OK) return st;
  if (max_ckpt > 0 && (st = check_pool(*dims, ckpt)) != GDN_OK) return st;
  if (!params || !params->conv_w || !params->A_log || !params->dt_bias) return GDN_ERR_INVALID_ARG;
  if (!slot_ids || !cu_seqlens || !start_pos || (max_ckpt > 0 && !ckpt_ids)) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!qkv || !a || !b || !out)) return GDN_ERR_INVALID_ARG;
  const int G = dims->hv / dims->hk;
  KdaPrefillArgs k = {};
  k.ssm = pool.ssm;
  k.conv = pool.conv;
  k.num_slots = pool.num_slots;
  k.ck_ssm = ckpt.ssm;
  k.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  k.conv_w = params->conv_w;
  k.A_log = params->A_log;
  k.dt_bias = params->dt_bias;
  k.slot_ids = slot_ids;
  k.cu_seqlens = cu_seqlens;
  k.start_pos = start_pos;
  k.total = total_tokens;
  k.ckpt_ids = ckpt_ids;
  k.max_ckpt = max_ckpt;
  k.ckpt_block = ckpt_block;
  k.qkv = qkv;
  k.a = a;
  k.b = b;
  k.out = out;
  k.err = dev_err;
  k.hk = dims->hk;
  k.hv = dims->hv;
  k.dv = dims->dv;
  k.W = dims->conv_width;
  k.C = (int32_t)channels(*dims);
  k.G = G;
  // rows per CTA: the kernel's NIT row groups of kWarps * 32 / (dk / 16) rows
  const int rows = (dims->dk == 128 ? 2 : 1) * kWarps * (32 / (dims->dk / 16));
  k.P = (dims->dv + rows - 1) / rows;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int act = dims->act_dtype, cv = dims->conv_dtype;
  // 16-byte staging copies: qkv and a 16-byte aligned, and every channel
  // segment (q and k heads, the v rows of a CTA, a gate row) and row stride a
  // multiple of 16 bytes (the CTA row counts are multiples of 8)
  const size_t es = dtype_size(act);
  const bool async = aligned(qkv, 16) && aligned(a, 16) && ((size_t)dims->dk * es) % 16 == 0 &&
                     ((size_t)dims->dv * es) % 16 == 0 && ((size_t)k.C * es) % 16 == 0;
  cudaError_t e = cudaErrorInvalidValue;
  // the 64-token chunk form on the tensor cores where it applies (dk = dv =
  // 128, bf16, width 4), else the 16-token window form (dk 128, dv <= 128),
  // else the token recurrence; GDN_KDA_PREFILL_PATH=window or recurrent
  // forces one of the latter (read on every call)
  const char* kp = std::getenv("GDN_KDA_PREFILL_PATH");
  const bool force_rec = kp && !std::strcmp(kp, "recurrent"), force_win = kp && !std::strcmp(kp, "window");
  const bool tc = !force_rec && !force_win && kda_tc32_supported(*dims, qkv, a, out, *params);
  const bool window = !tc && !force_rec && kda_chunk_supported(*dims);
  if (tc)
    e = kda_tc32_launch(*dims, pool, ckpt, *params, slot_ids, cu_seqlens, start_pos, n_seq, total_tokens, ckpt_ids,
                        max_ckpt, ckpt_block, qkv, a, b, out, dev_err, cs);
  else if (window)
    e = kda_chunk_launch(*dims, pool, ckpt, *params, slot_ids, cu_seqlens, start_pos, n_seq, total_tokens, ckpt_ids,
                         max_ckpt, ckpt_block, qkv, a, b, out, dev_err, cs);
  else switch (dims->dk) {
    case 16: e = dispatch_kda_prefill<16, 1>(k, n_seq, act, cv, async, cs); break;
    case 64: e = dispatch_kda_prefill<64, 1>(k, n_seq, act, cv, async, cs); break;
    case 128: e = dispatch_kda_prefill<128, 2>(k, n_seq, act, cv, async, cs); break;
  }
  if (e == cudaSuccess)
    e = conv_history_launch(*dims, pool, ckpt, slot_ids, cu_seqlens, start_pos, n_seq, total_tokens, ckpt_ids,
                            max_ckpt, ckpt_block, qkv, dev_err, cs);
  if (e == cudaSuccess) count_launch(GDN_K_KDA_PREFILL);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
