// One work item of the persistent TMA-fed GDN decode step (dk = 128, conv
// width 4), as device functions shared by the decode kernel (decode_tma.cu)
// and the single-launch mixed step (prefill_tc32.cu).
//
// An item is one request and one QK head hq together with the G V heads that
// read it: G*dv state rows of 512 bytes, contiguous in the pool
// ([slot][hv][dv][dk]), plus the q/k channels of hq and the v channels of its
// V heads.  Owning the whole group means the CTA alone reads and rewrites
// that slice of the conv history, so no other CTA ever touches it.
//
// Warp roles:
//   warp 8 (producer, one lane): produce_item streams the item's "bundle"
//     (conv history, activations, conv weights; 15 bulk copies) into one of
//     two bundle buffers and then its state rows in 16 KiB chunks (32 rows)
//     through a ring of STAGES shared-memory buffers with cp.async.bulk,
//     completion tracked by mbarriers (full/empty).
//   warps 0-7 (consumers): consume_bundle runs conv1d + SiLU, L2 norms and
//     gates from the bundle, then, chunk by chunk, the gated delta rule on 32
//     rows (4 rows per warp, 8 lanes per row, 3-level shuffle reductions),
//     streaming the updated rows straight to HBM with 128-bit stores.
// The producer runs up to STAGES chunks (and the next bundle) ahead, so HBM
// reads continue while the consumers are in an item's prologue.
//
// KDA (the per-key-channel decay variant: gate logits a [B][hv][dk], dt_bias
// [hv][dk]) uses the same walk with one alpha per (V head, key channel), kept
// in shared memory per item: u = v - St (alpha . k^), St' = St diag(alpha) +
// beta u k^T, o = St (alpha . q^) + beta u (k^ . q^).
//
// Every mbarrier wait is bounded (1 s); a wait that expires sets the CTA's
// abort flag, and the callers report GDN_DEV_ERR_TIMEOUT and wind down.
#pragma once
#include <cstddef>

#include "gdn_common.cuh"

namespace gdn {
namespace dtma {

constexpr int kCW = 8;             // consumer warps
constexpr int kCons = kCW * 32;    // consumer threads
constexpr int kThr = kCons + 32;   // + producer warp
constexpr int kDK = 128;
constexpr int kLPR = kDK / 16;     // lanes per state row
constexpr int kRows = 32;          // state rows per ring stage
constexpr int kStageFloats = kRows * kDK;
constexpr uint32_t kStageBytes = kStageFloats * sizeof(float);
constexpr int kW = 4;              // conv width
constexpr int kMaxGR = 256;        // G * dv rows per item, at most
constexpr int kMaxCh = 2 * kDK + kMaxGR;
constexpr int kBarCons = 1;        // named barrier of the consumer warps

template <typename Tact, typename Tconv, int STAGES, bool KDA>
struct __align__(128) TmaSmem {
  float ring[STAGES][kStageFloats];
  // every member is a bulk-copy destination: 16-byte aligned, and so is the
  // size, so that bundle[1] is too
  struct __align__(16) Bundle {
    Tconv hist[kW - 1][kMaxCh];  // [q | k | v of the group] per history row
    Tact x[kMaxCh];
    float w[kMaxCh * kW];
    __align__(16) Tact ga[KDA ? kMaxGR / kRows * kDK : 8];      // KDA: gate logits of the G V heads
    __align__(16) float gdt[KDA ? kMaxGR / kRows * kDK : 4];   // KDA: their dt_bias
  } bundle[2];
  float sy[kMaxCh];    // conv + SiLU output: q, k, v of the group
  float so[kMaxGR];    // readout of the group's rows
  float sred[3][kCW];
  float sgate[2][8];   // alpha, beta per V head of the group
  float sal[KDA ? 8 : 1][kDK];  // KDA: alpha per (V head of the group, key channel)
  float snorm[4];      // rq, rk, k^.q^
  uint64_t full[STAGES], empty[STAGES], bfull[2], bempty[2];
  int abort;
  int bitem[2];        // the item of each bundle buffer (the mixed step's dynamic walk)
};

template <typename Tact, typename Tconv, int STAGES, bool KDA>
constexpr bool bundle_aligned() {
  using SMt = TmaSmem<Tact, Tconv, STAGES, KDA>;
  using B = typename SMt::Bundle;
  return sizeof(B) % 16 == 0 && offsetof(B, x) % 16 == 0 && offsetof(B, w) % 16 == 0 &&
         offsetof(B, ga) % 16 == 0 && offsetof(B, gdt) % 16 == 0 && offsetof(SMt, bundle) % 16 == 0 &&
         offsetof(SMt, ring) % 16 == 0;
}
// the members read as float4 start 16-byte aligned
template <typename Tact, typename Tconv, int STAGES, bool KDA>
constexpr bool vectors_aligned() {
  using SMt = TmaSmem<Tact, Tconv, STAGES, KDA>;
  return offsetof(SMt, sy) % 16 == 0 && offsetof(SMt, sal) % 16 == 0 && offsetof(SMt, ring) % 16 == 0;
}

struct TmaArgs {
  float* ssm;
  void* conv;
  int32_t num_slots;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const int32_t* slot_ids;
  const void* qkv;
  const void* a;
  const void* b;
  void* out;
  uint32_t* err;
  int32_t hk, hv, dv, C, G, n_items;
};

// thread 0: the ring's and the bundles' barriers
template <typename SM, int STAGES>
__device__ __forceinline__ void init_barriers(SM& S) {
  for (int s = 0; s < STAGES; ++s) {
    mbar_init(&S.full[s], 1);
    mbar_init(&S.empty[s], kCW);
  }
  for (int s = 0; s < 2; ++s) {
    mbar_init(&S.bfull[s], 1);
    mbar_init(&S.bempty[s], kCons);
  }
  S.abort = 0;
  fence_mbar_init();
}

// Producer lane: the bundle of item (r, hq), whose slot is usable, into
// bundle buffer vk & 1 (once the consumers released it; `tag` is recorded as
// the buffer's item), then the item's state rows through the ring, stages n,
// n + 1, ...  vk and n advance by what was issued; false when a wait expired
// or the CTA is aborting.
template <typename Tact, typename Tconv, int STAGES, bool KDA>
__device__ __forceinline__ bool produce_item(const TmaArgs& a, TmaSmem<Tact, Tconv, STAGES, KDA>& S, int r, int hq,
                                             int32_t slot, uint32_t& vk, uint32_t& n, int tag = 0) {
  volatile int* abort_flag = &S.abort;
  const int GR = a.G * a.dv, nchunks = GR / kRows, nch = 2 * kDK + GR;
  const uint32_t esz_c = sizeof(Tconv), esz_a = sizeof(Tact);
  const uint32_t bundle_bytes =
      (kW - 1) * nch * esz_c + nch * esz_a + nch * kW * 4 + (KDA ? a.G * kDK * (esz_a + 4) : 0);
  // extents of the caller's tensors (elements), for the checked build
  const int nreq = a.n_items / a.hk;
  [[maybe_unused]] const long long ssm_n = (long long)a.num_slots * a.hv * a.dv * kDK,
                                   conv_n = (long long)a.num_slots * (kW - 1) * a.C,
                                   gate_n = (long long)nreq * a.hv;
  const int bb = vk & 1;
  if (!mbar_wait(&S.bempty[bb], ((vk >> 1) & 1) ^ 1)) return false;
  S.bitem[bb] = tag;  // published by the arrival below
  mbar_arrive_expect_tx(&S.bfull[bb], bundle_bytes);
  typename TmaSmem<Tact, Tconv, STAGES, KDA>::Bundle& B = S.bundle[bb];
  const size_t cq = (size_t)hq * kDK, ck = (size_t)a.hk * kDK + cq, cv = 2 * (size_t)a.hk * kDK + (size_t)hq * GR;
  // one bundle copy: `bytes` from global src (inside [base, base + extent))
  // into the shared bundle
  auto g2s = [&](void* dst, const void* src, uint32_t bytes, [[maybe_unused]] const void* base,
                 [[maybe_unused]] long long extent) {
    if (GDN_GBYTES(src, bytes, base, extent) && GDN_SBYTES(dst, bytes, S)) bulk_g2s(dst, src, bytes, &S.bfull[bb]);
  };
  const Tconv* hist = reinterpret_cast<const Tconv*>(a.conv) + (size_t)slot * (kW - 1) * a.C;
  for (int j = 0; j < kW - 1; ++j) {
    g2s(&B.hist[j][0], hist + (size_t)j * a.C + cq, kDK * esz_c, a.conv, conv_n * esz_c);
    g2s(&B.hist[j][kDK], hist + (size_t)j * a.C + ck, kDK * esz_c, a.conv, conv_n * esz_c);
    g2s(&B.hist[j][2 * kDK], hist + (size_t)j * a.C + cv, GR * esz_c, a.conv, conv_n * esz_c);
  }
  const Tact* x = reinterpret_cast<const Tact*>(a.qkv) + (size_t)r * a.C;
  const long long x_bytes = (long long)nreq * a.C * esz_a, w_bytes = (long long)a.C * kW * 4;
  g2s(&B.x[0], x + cq, kDK * esz_a, a.qkv, x_bytes);
  g2s(&B.x[kDK], x + ck, kDK * esz_a, a.qkv, x_bytes);
  g2s(&B.x[2 * kDK], x + cv, GR * esz_a, a.qkv, x_bytes);
  g2s(&B.w[0], a.conv_w + cq * kW, kDK * kW * 4, a.conv_w, w_bytes);
  g2s(&B.w[kDK * kW], a.conv_w + ck * kW, kDK * kW * 4, a.conv_w, w_bytes);
  g2s(&B.w[2 * kDK * kW], a.conv_w + cv * kW, GR * kW * 4, a.conv_w, w_bytes);
  if (KDA) {
    const size_t h0 = (size_t)hq * a.G;
    g2s(&B.ga[0], reinterpret_cast<const Tact*>(a.a) + ((size_t)r * a.hv + h0) * kDK, a.G * kDK * esz_a, a.a,
        gate_n * kDK * esz_a);
    g2s(&B.gdt[0], a.dt_bias + h0 * kDK, a.G * kDK * 4, a.dt_bias, (long long)a.hv * kDK * 4);
  }
  ++vk;
  const float* src = a.ssm + ((size_t)slot * a.hv + (size_t)hq * a.G) * a.dv * kDK;
  for (int c = 0; c < nchunks; ++c, ++n) {
    const int st = n % STAGES;
    if (*abort_flag || !mbar_wait(&S.empty[st], ((n / STAGES) & 1) ^ 1)) return false;
    mbar_arrive_expect_tx(&S.full[st], kStageBytes);
    if (GDN_GBYTES(src + (size_t)c * kStageFloats, kStageBytes, a.ssm, ssm_n * 4) &&
        GDN_SBYTES(S.ring[GDN_S(st, STAGES)], kStageBytes, S))
      bulk_g2s(S.ring[st], src + (size_t)c * kStageFloats, kStageBytes, &S.full[st]);
  }
  return true;
}

// Producer lane after a failed wait: mark the CTA aborting, report, and let
// the copies already issued land before the CTA's memory goes away.
template <typename SM, int STAGES>
__device__ __forceinline__ void producer_drain(const TmaArgs& a, SM& S, uint32_t vk, uint32_t n) {
  S.abort = 1;
  report(a.err, GDN_DEV_ERR_TIMEOUT);
  const uint32_t first = n > (uint32_t)STAGES ? n - STAGES : 0;
  for (uint32_t m = first; m < n; ++m) mbar_wait(&S.full[m % STAGES], (m / STAGES) & 1);
  for (uint32_t m = vk > 2 ? vk - 2 : 0; m < vk; ++m) mbar_wait(&S.bfull[m & 1], (m >> 1) & 1);
}

// Consumers (all kCons threads): the outputs of item (r, hq) of an unusable
// slot are zeros (and an out-of-range id is reported once per request).
template <typename Tact>
__device__ __forceinline__ void consume_skipped(const TmaArgs& a, int r, int hq, int cls) {
  const int tid = threadIdx.x, GR = a.G * a.dv;
  const int nreq = a.n_items / a.hk;
  [[maybe_unused]] const long long out_n = (long long)nreq * a.hv * a.dv;
  Tact* const out_all = reinterpret_cast<Tact*>(a.out);
  const size_t out0 = ((size_t)r * a.hv + (size_t)hq * a.G) * a.dv;
  if (cls == 2 && hq == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
  for (int i = tid; i < GR; i += kCons) out_all[GDN_G(out0 + i, out_n)] = from_f32<Tact>(0.f);
}

// Consumers (all kCons threads), item (r, hq) of usable slot `slot` whose
// bundle has landed in buffer bb (every consumer passed its wait and the
// consumers' barrier): conv1d + SiLU (the new conv history written at once:
// the old one is in the bundle), the gates, the bundle released, the norms,
// then the state rows from ring stages n, n + 1, ... and the group's
// outputs.  n advances by the stages consumed; false when a wait expired (or
// the CTA is aborting).
template <typename Tact, typename Tconv, int STAGES, bool KDA>
__device__ __forceinline__ bool consume_bundle(const TmaArgs& a, TmaSmem<Tact, Tconv, STAGES, KDA>& S, int r, int hq,
                                               int32_t slot, int bb, uint32_t& n) {
  using SM = TmaSmem<Tact, Tconv, STAGES, KDA>;
  volatile int* abort_flag = &S.abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int GR = a.G * a.dv, nchunks = GR / kRows, nch = 2 * kDK + GR;
  const int seg = lane % kLPR;
  const int rloc = warp * (32 / kLPR) + lane / kLPR;  // row within a chunk
  const int nreq = a.n_items / a.hk;
  [[maybe_unused]] const long long ssm_n = (long long)a.num_slots * a.hv * a.dv * kDK,
                                   conv_n = (long long)a.num_slots * (kW - 1) * a.C,
                                   out_n = (long long)nreq * a.hv * a.dv, gate_n = (long long)nreq * a.hv;
  Tact* const out_all = reinterpret_cast<Tact*>(a.out);
  const size_t out0 = ((size_t)r * a.hv + (size_t)hq * a.G) * a.dv;
  const typename SM::Bundle& B = S.bundle[bb];
  // conv1d + SiLU; the old history is in the bundle, so the new one can be
  // written at once (this CTA is the only one touching these channels)
  Tconv* const hist_all = reinterpret_cast<Tconv*>(a.conv);
  const size_t hist0 = (size_t)slot * (kW - 1) * a.C;
  for (int i0 = tid; i0 < nch; i0 += kCons) {
    const int i = GDN_S(i0, kMaxCh);
    const float h0 = to_f32(B.hist[0][i]), h1 = to_f32(B.hist[1][i]), h2 = to_f32(B.hist[2][i]);
    const float xv = to_f32(B.x[i]);
    const float4 w = reinterpret_cast<const float4*>(B.w)[i];  // kW = 4 weights of channel i
    float acc = w.x * h0;
    acc = fmaf(w.y, h1, acc);
    acc = fmaf(w.z, h2, acc);
    acc = fmaf(w.w, xv, acc);
    S.sy[i] = silu_f(acc);
    const size_t c = i < kDK ? (size_t)hq * kDK + i
                   : i < 2 * kDK ? (size_t)a.hk * kDK + (size_t)hq * kDK + (i - kDK)
                                 : 2 * (size_t)a.hk * kDK + (size_t)hq * GR + (i - 2 * kDK);
    hist_all[GDN_G(hist0 + c, conv_n)] = B.hist[1][i];
    hist_all[GDN_G(hist0 + a.C + c, conv_n)] = B.hist[2][i];
    hist_all[GDN_G(hist0 + 2 * (size_t)a.C + c, conv_n)] = from_f32<Tconv>(xv);
  }
  if (KDA) {
    for (int e0 = tid; e0 < a.G * kDK; e0 += kCons) {
      const int e = GDN_S(e0, (KDA ? kMaxGR / kRows : 1) * kDK);
      const int gi = e / kDK, h = hq * a.G + gi;
      S.sal[KDA ? gi : 0][e % kDK] = gate_alpha(a.A_log[GDN_G(h, a.hv)], B.gdt[e], to_f32(B.ga[e]));
    }
  }
  if (tid < a.G) {
    const int h = GDN_G(hq * a.G + tid, a.hv), tg = GDN_S(tid, 8);
    const float bv = to_f32(reinterpret_cast<const Tact*>(a.b)[GDN_G((size_t)r * a.hv + h, gate_n)]);
    if (!KDA) {
      const float av = to_f32(reinterpret_cast<const Tact*>(a.a)[GDN_G((size_t)r * a.hv + h, gate_n)]);
      S.sgate[0][tg] = gate_alpha(a.A_log[h], a.dt_bias[h], av);
    }
    S.sgate[1][tg] = sigmoid_f(bv);
  }
  named_sync(kBarCons, kCons);
  mbar_arrive(&S.bempty[bb]);
  // L2 norms of q and k, and k^.q^
  {
    float pq = 0.f, pk = 0.f, pqk = 0.f;
    if (tid < kDK) {
      const float q = S.sy[tid], k = S.sy[kDK + tid];
      pq = q * q;
      pk = k * k;
      pqk = q * k;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      pq += __shfl_xor_sync(0xffffffffu, pq, o);
      pk += __shfl_xor_sync(0xffffffffu, pk, o);
      pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
    }
    if (lane == 0) {
      const int w = GDN_S(warp, kCW);
      S.sred[0][w] = pq;
      S.sred[1][w] = pk;
      S.sred[2][w] = pqk;
    }
    named_sync(kBarCons, kCons);
    if (tid == 0) {
      float x = 0.f, y = 0.f, z = 0.f;
      for (int w = 0; w < kCW; ++w) {
        x += S.sred[0][w];
        y += S.sred[1][w];
        z += S.sred[2][w];
      }
      const float rq = rsqrtf(x + kNormEps) * rsqrtf((float)kDK);
      const float rk = rsqrtf(y + kNormEps);
      S.snorm[0] = rq;
      S.snorm[1] = rk;
      S.snorm[2] = z * rq * rk;
    }
    named_sync(kBarCons, kCons);
  }
  const float rq = S.snorm[0], rk = S.snorm[1], kq = S.snorm[2];
  float4 kk[4], qq[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = GDN_S(c * 4 * kLPR + seg * 4, kDK - 3);
    const float4 k4 = *reinterpret_cast<const float4*>(&S.sy[kDK + col]);
    const float4 q4 = *reinterpret_cast<const float4*>(&S.sy[col]);
    kk[c] = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
    qq[c] = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
  }
  const size_t dst0 = ((size_t)slot * a.hv + (size_t)hq * a.G) * a.dv * kDK;
  // KDA: this lane's alphas of the current V head (a chunk's 32 rows belong
  // to one head; reloaded only when the head changes)
  float4 al[4];
  int g_al = -1;
  for (int c = 0; c < nchunks; ++c, ++n) {
    const int st = n % STAGES;
    if (!*abort_flag && !mbar_wait(&S.full[st], (n / STAGES) & 1)) *abort_flag = 1;
    if (*abort_flag) continue;
    const int grow = GDN_S(c * kRows + rloc, kMaxGR);  // row within the group
    const int g = GDN_S(grow / a.dv, 8);
    const float alpha = KDA ? 1.f : S.sgate[0][g], beta = S.sgate[1][g];
    const float* srow = S.ring[GDN_S(st, STAGES)] + GDN_S(rloc, kRows) * kDK;
    float4 s4[4];
    if (g != g_al) {
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        al[cc] = KDA ? *reinterpret_cast<const float4*>(&S.sal[KDA ? g : 0][GDN_S(cc * 4 * kLPR + seg * 4, kDK - 3)])
                     : make_float4(alpha, alpha, alpha, alpha);
      g_al = g;
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      s4[cc] = *reinterpret_cast<const float4*>(srow + GDN_S(cc * 4 * kLPR + seg * 4, kDK - 3));
    float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      // KDA: the decayed row St diag(alpha) meets k^ and q^
      const float4 sa = KDA ? make_float4(s4[cc].x * al[cc].x, s4[cc].y * al[cc].y, s4[cc].z * al[cc].z,
                                          s4[cc].w * al[cc].w)
                            : s4[cc];
      dk_ += sa.x * kk[cc].x + sa.y * kk[cc].y + sa.z * kk[cc].z + sa.w * kk[cc].w;
      dq_ += sa.x * qq[cc].x + sa.y * qq[cc].y + sa.z * qq[cc].z + sa.w * qq[cc].w;
    }
    __syncwarp();  // every lane has consumed its part of the stage
    if (lane == 0) mbar_arrive(&S.empty[st]);  // the producer may refill it
#pragma unroll
    for (int o = kLPR / 2; o; o >>= 1) {
      dk_ += __shfl_xor_sync(0xffffffffu, dk_, o);
      dq_ += __shfl_xor_sync(0xffffffffu, dq_, o);
    }
    const float bu = beta * (S.sy[GDN_S(2 * kDK + grow, kMaxCh)] - alpha * dk_);
    float4* const ssm4 = reinterpret_cast<float4*>(a.ssm);
    const size_t drow4 = (dst0 + (size_t)grow * kDK) / 4;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float4 v = s4[cc];
      v.x = fmaf(bu, kk[cc].x, al[cc].x * v.x);
      v.y = fmaf(bu, kk[cc].y, al[cc].y * v.y);
      v.z = fmaf(bu, kk[cc].z, al[cc].z * v.z);
      v.w = fmaf(bu, kk[cc].w, al[cc].w * v.w);
      st_stream(ssm4 + GDN_G(drow4 + (cc * 4 * kLPR + seg * 4) / 4, ssm_n / 4), v);
    }
    if (seg == 0) S.so[grow] = fmaf(bu, kq, alpha * dq_);
  }
  named_sync(kBarCons, kCons);
  if (*abort_flag) return false;
  for (int i = tid; i < GR; i += kCons) out_all[GDN_G(out0 + i, out_n)] = from_f32<Tact>(S.so[GDN_S(i, kMaxGR)]);
  return true;
}

}  // namespace dtma
}  // namespace gdn
