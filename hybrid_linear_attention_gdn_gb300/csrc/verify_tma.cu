// Persistent, TMA-fed speculative verify (dk = 128, conv width 4).
//
// TokenSpeed Qwen3.5 page, "Scheduler dual": the spec_cache keeps per-draft-
// step conv/SSM snapshots so that the state can roll back when verification
// rejects drafts.  Verify runs the T draft tokens of each request from its
// working slot and writes the state after every draft into a spec slot; the
// working slot is only read.
//
// Because nothing here is written in place, work splits freely.  The unit of
// work is one stage: 32 state rows of one request and V head.  Each CTA takes
// an equal, contiguous share of the B * hv * dv/32 stages (so the last wave
// ends evenly however B compares with the SM count) and walks it as segments
// (the stages of one request and V head it holds):
//   warp 8 (producer, one lane): per segment, a bundle of bulk copies (the
//     conv history rows and the T draft activations of the q/k channels of h's
//     QK head and of the segment's v channels, plus their conv weights), then
//     its state rows in 16 KiB chunks through a ring of mbarrier-tracked
//     shared-memory stages;
//   warps 0-7: conv + SiLU over the draft sequence (and the snapshot conv
//     histories, written straight to the spec slots), per-draft L2 norms and
//     gates; then per chunk, 4 rows per warp are held in registers through all
//     T drafts, each draft's rows streamed to its spec slot with 128-bit stores.
// Snapshot writes are T times the state reads, so HBM time is mostly stores.
// All waits are bounded (GDN_DEV_ERR_TIMEOUT).
//
// KDA (one decay per key channel): the bundle also carries the T drafts' gate
// logits of the V head and its dt_bias row; the consumers turn them into an
// alpha table [T][dk] and scale each row by it in place before its products.
#include "gdn_common.cuh"

#include <cstddef>
#include <cstdlib>
#include <type_traits>
#include "decode_tma.cuh"

namespace gdn {
namespace {

constexpr int kCW = 8;
constexpr int kCons = kCW * 32;
constexpr int kThr = kCons + 32;
constexpr int kDK = 128;
constexpr int kLPR = kDK / 16;
constexpr int kRows = 32;
constexpr int kStageFloats = kRows * kDK;
constexpr uint32_t kStageBytes = kStageFloats * sizeof(float);
constexpr int kW = 4;
constexpr int kMaxT = 16;
constexpr int kMaxR = 128;
constexpr int kMaxCh = 2 * kDK + kMaxR;
constexpr int kBarCons = 1;

// MT: drafts the shared-memory layout holds (T <= MT).  The T <= 8 layout is
// small enough for two CTAs per SM, so one CTA's prologue overlaps the other's
// stream of snapshot stores.
template <typename Tact, typename Tconv, int STAGES, int MT, bool KDA>
struct __align__(128) VSmem {
  float ring[STAGES][kStageFloats];
  // every member a multiple of 16 bytes long, so that every bulk-copy
  // destination in both bundles is 16-byte aligned
  struct __align__(16) Bundle {
    Tconv hist[kW - 1][kMaxCh];
    Tact x[MT][kMaxCh];
    float w[kMaxCh * kW];
    Tact ga[KDA ? MT : 1][KDA ? kDK : 8];  // KDA: the drafts' gate logits of the V head
    float gdt[KDA ? kDK : 4];              // KDA: its dt_bias row
  } bundle[2];
  float sy[MT][kMaxCh];   // conv + SiLU per draft: q | k | v rows
  float so[MT][kMaxR];    // readout per draft
  float snorm[MT][3];     // rq, rk, k^.q^ per draft
  float sgate[MT][2];     // alpha, beta per draft
  float sal[KDA ? MT : 1][kDK];  // KDA: alpha per draft and key channel
  int32_t ssid[MT];       // the segment's spec slot per draft
  uint64_t full[STAGES], empty[STAGES], bfull[2], bempty[2];
  int abort;
};

template <typename Tact, typename Tconv, int STAGES, int MT, bool KDA>
__host__ __device__ constexpr bool vbundle_aligned() {
  using V = VSmem<Tact, Tconv, STAGES, MT, KDA>;
  using B = typename V::Bundle;
  return sizeof(B) % 16 == 0 && offsetof(B, x) % 16 == 0 && offsetof(B, w) % 16 == 0 &&
         offsetof(B, ga) % 16 == 0 && offsetof(B, gdt) % 16 == 0 && offsetof(V, bundle) % 16 == 0;
}

struct VArgs {
  const float* ssm;
  const void* conv;
  int32_t num_slots;
  float* spec_ssm;
  void* spec_conv;
  int32_t spec_num_slots;
  const int32_t* spec_ids;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const int32_t* slot_ids;
  const void* qkv;
  const void* a;
  const void* b;
  void* out;
  uint32_t* err;
  int32_t hk, hv, dv, C, G, T;
  int32_t sph;      // stages (32 rows) per V head: dv / 32
  int64_t n_units;  // B * hv * sph
};

// The segment that starts at stage unit u of a CTA's share [.., u1): request
// r, V head h, stages s0 .. s0 + ns - 1 of the head (rows 32 s0 ..), at most
// kMaxR / 32 stages (the rows one bundle holds).
struct Seg {
  int r, h, s0, ns;
};
__device__ __forceinline__ Seg segment_at(const VArgs& a, int64_t u, int64_t u1) {
  const int64_t hu = u / a.sph;
  Seg g;
  g.r = (int)(hu / a.hv);
  g.h = (int)(hu % a.hv);
  g.s0 = (int)(u % a.sph);
  int64_t ns = a.sph - g.s0;
  if (ns > u1 - u) ns = u1 - u;
  if (ns > kMaxR / kRows) ns = kMaxR / kRows;
  g.ns = (int)ns;
  return g;
}

// two consecutive elements (8-byte aligned for fp32, 4-byte for bf16) as fp32
__device__ __forceinline__ float2 load_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void store_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// a line of global memory into L1 (no value returned, nothing to wait for)
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.L1 [%0];\n" ::"l"(p)); }

template <typename Tact, typename Tconv, int STAGES, int MT, int MINB, bool KDA>
__global__ void __launch_bounds__(kThr, MINB) verify_tma_kernel(const VArgs a) {
  pdl_wait();
  pdl_trigger();
  using SM = VSmem<Tact, Tconv, STAGES, MT, KDA>;
  static_assert(vbundle_aligned<Tact, Tconv, STAGES, MT, KDA>(), "bundle members must stay 16-byte aligned");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SM& S = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T;
  // this CTA's share of the stage units
  const int64_t u0 = (int64_t)blockIdx.x * a.n_units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * a.n_units / gridDim.x;
  volatile int* abort_flag = &S.abort;
  // extents of the caller's tensors (elements), for the checked build
  const int nreq = (int)(a.n_units / ((int64_t)a.hv * a.sph));
  [[maybe_unused]] const long long ssm_n = (long long)a.num_slots * a.hv * a.dv * kDK,
                                   conv_n = (long long)a.num_slots * (kW - 1) * a.C,
                                   spec_ssm_n = (long long)a.spec_num_slots * a.hv * a.dv * kDK,
                                   spec_conv_n = (long long)a.spec_num_slots * (kW - 1) * a.C,
                                   gate_n = (long long)nreq * T * a.hv, out_n = (long long)nreq * T * a.hv * a.dv;

  if (tid == 0) {
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
  __syncthreads();

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint32_t ec = sizeof(Tconv), ea = sizeof(Tact);
    uint32_t n = 0, vk = 0;
    bool ok = true;
    // the next segment at or after u whose working slot is in range (the
    // consumers skip the others without a bundle), or false
    auto next_valid = [&](int64_t& u, Seg& g) -> bool {
      while (u < u1) {
        g = segment_at(a, u, u1);
        u += g.ns;
        if (!slot_class(a.slot_ids[GDN_G(g.r, nreq)], a.num_slots)) return true;
      }
      return false;
    };
    // segment g's bundle into buffer vk % 2 (free once the consumers have
    // finished the prologue of the segment two before); false on a timeout
    auto issue_bundle = [&](const Seg& g) -> bool {
      const int r = g.r, h = g.h, R = g.ns * kRows, nch = 2 * kDK + R;
      const uint32_t bundle_bytes =
          (kW - 1) * nch * ec + T * nch * ea + nch * kW * 4 + (KDA ? T * kDK * ea + kDK * 4 : 0u);
      const int32_t slot = a.slot_ids[GDN_G(r, nreq)];
      const int hq = h / a.G;
      const int bb = vk & 1;
      if (!mbar_wait(&S.bempty[bb], ((vk >> 1) & 1) ^ 1)) return false;
      mbar_arrive_expect_tx(&S.bfull[bb], bundle_bytes);
      typename SM::Bundle& Bd = S.bundle[bb];
      const size_t cq = (size_t)hq * kDK, ck = (size_t)a.hk * kDK + cq,
                   cv = 2 * (size_t)a.hk * kDK + (size_t)h * a.dv + (size_t)g.s0 * kRows;
      // one bundle copy: `bytes` from global src (inside [base, base + extent))
      // into the shared bundle
      auto g2s = [&](void* dst, const void* src, uint32_t bytes, [[maybe_unused]] const void* base,
                     [[maybe_unused]] long long extent) {
        if (GDN_GBYTES(src, bytes, base, extent) && GDN_SBYTES(dst, bytes, S))
          bulk_g2s(dst, src, bytes, &S.bfull[bb]);
      };
      const Tconv* hist = reinterpret_cast<const Tconv*>(a.conv) + (size_t)slot * (kW - 1) * a.C;
      for (int j = 0; j < kW - 1; ++j) {
        g2s(&Bd.hist[j][0], hist + (size_t)j * a.C + cq, kDK * ec, a.conv, conv_n * ec);
        g2s(&Bd.hist[j][kDK], hist + (size_t)j * a.C + ck, kDK * ec, a.conv, conv_n * ec);
        g2s(&Bd.hist[j][2 * kDK], hist + (size_t)j * a.C + cv, R * ec, a.conv, conv_n * ec);
      }
      const long long x_bytes = (long long)nreq * T * a.C * ea, w_bytes = (long long)a.C * kW * 4;
      for (int t = 0; t < T; ++t) {
        const Tact* x = reinterpret_cast<const Tact*>(a.qkv) + ((size_t)r * T + t) * a.C;
        const int tt = GDN_S(t, MT);
        g2s(&Bd.x[tt][0], x + cq, kDK * ea, a.qkv, x_bytes);
        g2s(&Bd.x[tt][kDK], x + ck, kDK * ea, a.qkv, x_bytes);
        g2s(&Bd.x[tt][2 * kDK], x + cv, R * ea, a.qkv, x_bytes);
      }
      g2s(&Bd.w[0], a.conv_w + cq * kW, kDK * kW * 4, a.conv_w, w_bytes);
      g2s(&Bd.w[kDK * kW], a.conv_w + ck * kW, kDK * kW * 4, a.conv_w, w_bytes);
      g2s(&Bd.w[2 * kDK * kW], a.conv_w + cv * kW, R * kW * 4, a.conv_w, w_bytes);
      if constexpr (KDA) {
        for (int t = 0; t < T; ++t)
          g2s(&Bd.ga[GDN_S(t, MT)][0], reinterpret_cast<const Tact*>(a.a) + (((size_t)r * T + t) * a.hv + h) * kDK,
              kDK * ea, a.a, gate_n * kDK * ea);
        g2s(&Bd.gdt[0], a.dt_bias + (size_t)h * kDK, kDK * 4, a.dt_bias, (long long)a.hv * kDK * 4);
      }
      ++vk;
      return true;
    };
    // each segment's bundle goes out one segment ahead of its state chunks,
    // so it has landed when the consumers reach the segment
    int64_t u = u0;
    Seg g, gn;
    bool have = next_valid(u, g);
    if (have && !issue_bundle(g)) ok = false;
    while (have && ok && !*abort_flag) {
      const bool have_next = next_valid(u, gn);
      if (have_next && !issue_bundle(gn)) {
        ok = false;
        break;
      }
      const int h = g.h, nchunks = g.ns;
      const int32_t slot = a.slot_ids[GDN_G(g.r, nreq)];
      const float* src = a.ssm + (((size_t)slot * a.hv + h) * a.dv + (size_t)g.s0 * kRows) * kDK;
      for (int c = 0; c < nchunks; ++c, ++n) {
        const int st = n % STAGES;
        if (*abort_flag || !mbar_wait(&S.empty[st], ((n / STAGES) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.full[st], kStageBytes);
        if (GDN_GBYTES(src + (size_t)c * kStageFloats, kStageBytes, a.ssm, ssm_n * 4) &&
            GDN_SBYTES(S.ring[GDN_S(st, STAGES)], kStageBytes, S))
          bulk_g2s(S.ring[st], src + (size_t)c * kStageFloats, kStageBytes, &S.full[st]);
      }
      g = gn;
      have = have_next;
    }
    if (!ok || *abort_flag) {
      *abort_flag = 1;
      report(a.err, GDN_DEV_ERR_TIMEOUT);
      const uint32_t first = n > (uint32_t)STAGES ? n - STAGES : 0;
      for (uint32_t m = first; m < n; ++m) mbar_wait(&S.full[m % STAGES], (m / STAGES) & 1);
      for (uint32_t m = vk > 2 ? vk - 2 : 0; m < vk; ++m) mbar_wait(&S.bfull[m & 1], (m >> 1) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int seg = lane % kLPR;
  const int rloc = warp * (32 / kLPR) + lane / kLPR;
  uint32_t n = 0, vk = 0;
  for (int64_t u = u0; u < u1;) {
    const Seg g = segment_at(a, u, u1);
    u += g.ns;
    const int r = g.r, h = g.h, R = g.ns * kRows, nchunks = g.ns, nch = 2 * kDK + R;
    const int row0 = g.s0 * kRows;  // first row of the segment within the head
    const int hq = h / a.G;
    const int32_t slot = a.slot_ids[GDN_G(r, nreq)];
    // spec slot of draft t of this request
    auto sid_of = [&](int t) { return a.spec_ids[GDN_G((size_t)r * T + t, (long long)nreq * T)]; };
    const int cls = slot_class(slot, a.num_slots);
    if (cls) {
      if (cls == 2 && h == 0 && g.s0 == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
      for (int e = tid; e < T * R; e += kCons) {
        const int t = e / R, i = e % R;
        reinterpret_cast<Tact*>(a.out)[GDN_G((((size_t)r * T + t) * a.hv + h) * a.dv + row0 + i, out_n)] =
            from_f32<Tact>(0.f);
      }
      continue;
    }
    if (h == 0 && g.s0 == 0 && tid < T && slot_class(sid_of(tid), a.spec_num_slots) == 2)
      report(a.err, GDN_DEV_ERR_SLOT_OOB);
    // the drafts' spec slots, read once per segment (the loops below take
    // them from shared memory rather than reloading them per draft)
    if (tid < T) S.ssid[GDN_S(tid, MT)] = sid_of(tid);
    const int bb = vk & 1;
    if (!*abort_flag && !mbar_wait(&S.bfull[bb], (vk >> 1) & 1)) *abort_flag = 1;
    named_sync(kBarCons, kCons);
    if (*abort_flag) break;
    const typename SM::Bundle& Bd = S.bundle[bb];
    // conv over the drafts; the snapshot history after draft t is
    // [win1, win2, x_t].  q/k channels are written by the segment holding row
    // 0 of the first V head of the QK group, v channels by their own segment.
    const bool qk_writer = (h % a.G) == 0 && g.s0 == 0;
    // a channel pair (2 i, 2 i + 1) per thread: pair loads and stores (every
    // part's channel count is even, so a pair never straddles two parts).
    for (int i0 = 2 * tid; i0 < nch; i0 += 2 * kCons) {
      const int i = GDN_S(i0, kMaxCh - 1);
      const float4 wa = reinterpret_cast<const float4*>(Bd.w)[i];  // kW = 4 weights of channel i
      const float4 wb = reinterpret_cast<const float4*>(Bd.w)[i + 1];
      float2 w0 = load_pair(&Bd.hist[0][i]), w1 = load_pair(&Bd.hist[1][i]), w2 = load_pair(&Bd.hist[2][i]);
      const size_t c = i < kDK ? (size_t)hq * kDK + i
                     : i < 2 * kDK ? (size_t)a.hk * kDK + (size_t)hq * kDK + (i - kDK)
                                   : 2 * (size_t)a.hk * kDK + (size_t)h * a.dv + (size_t)row0 + (i - 2 * kDK);
      const bool writes = i >= 2 * kDK || qk_writer;
      for (int t0 = 0; t0 < T; ++t0) {
        const int t = GDN_S(t0, MT);
        const float2 xv = load_pair(&Bd.x[t][i]);
        float ax = wa.x * w0.x, ay = wb.x * w0.y;
        ax = fmaf(wa.y, w1.x, ax);
        ay = fmaf(wb.y, w1.y, ay);
        ax = fmaf(wa.z, w2.x, ax);
        ay = fmaf(wb.z, w2.y, ay);
        ax = fmaf(wa.w, xv.x, ax);
        ay = fmaf(wb.w, xv.y, ay);
        *reinterpret_cast<float2*>(&S.sy[t][i]) = make_float2(silu_fast_f(ax), silu_fast_f(ay));
        w0 = w1;
        w1 = w2;
        w2 = xv;
        const int32_t sid = S.ssid[t];
        if (writes && slot_class(sid, a.spec_num_slots) == 0) {
          Tconv* const sc = reinterpret_cast<Tconv*>(a.spec_conv);
          const size_t c0 = (size_t)sid * (kW - 1) * a.C + c;
          store_pair(&sc[GDN_G(c0, spec_conv_n - 1)], w0);
          store_pair(&sc[GDN_G(c0 + a.C, spec_conv_n - 1)], w1);
          store_pair(&sc[GDN_G(c0 + 2 * (size_t)a.C, spec_conv_n - 1)], w2);
        }
      }
    }
    if (tid < T) {
      const size_t rt = (size_t)r * T + tid;
      const int tt = GDN_S(tid, MT);
      S.sgate[tt][0] = KDA ? 1.f
                           : gate_alpha(a.A_log[GDN_G(h, a.hv)], a.dt_bias[GDN_G(h, a.hv)],
                                        to_f32(reinterpret_cast<const Tact*>(a.a)[GDN_G(rt * a.hv + h, gate_n)]));
      S.sgate[tt][1] = sigmoid_f(to_f32(reinterpret_cast<const Tact*>(a.b)[GDN_G(rt * a.hv + h, gate_n)]));
    }
    if constexpr (KDA) {
      // alpha[t][c] = exp(-exp(A_log) softplus(a[t][c] + dt_bias[c])), from the bundle
      const float A_log = a.A_log[GDN_G(h, a.hv)];
      for (int e = tid; e < T * kDK; e += kCons) {
        const int t = GDN_S(e / kDK, MT), c = e % kDK;
        S.sal[t][c] = gate_alpha(A_log, Bd.gdt[c], to_f32(Bd.ga[t][c]));
      }
    }
    named_sync(kBarCons, kCons);
    mbar_arrive(&S.bempty[bb]);
    ++vk;
    for (int t0 = warp; t0 < T; t0 += kCW) {
      const int t = GDN_S(t0, MT);
      float pq = 0.f, pk = 0.f, pqk = 0.f;
      for (int i = lane; i < kDK; i += 32) {
        const float q = S.sy[t][i], k = S.sy[t][kDK + i];
        pq = fmaf(q, q, pq);
        pk = fmaf(k, k, pk);
        pqk = fmaf(q, k, pqk);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        pq += __shfl_xor_sync(0xffffffffu, pq, o);
        pk += __shfl_xor_sync(0xffffffffu, pk, o);
        pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
      }
      if (lane == 0) {
        const float rq = rsqrtf(pq + kNormEps) * rsqrtf((float)kDK);
        const float rk = rsqrtf(pk + kNormEps);
        S.snorm[t][0] = rq;
        S.snorm[t][1] = rk;
        S.snorm[t][2] = pqk * rq * rk;
      }
    }
    named_sync(kBarCons, kCons);
    // q^ and k^ normalised in place, once per segment rather than per row
    for (int e = tid; e < T * 2 * kDK; e += kCons) {
      const int t = GDN_S(e / (2 * kDK), MT), i = e % (2 * kDK);
      S.sy[t][i] *= S.snorm[t][i < kDK ? 0 : 1];
    }
    named_sync(kBarCons, kCons);

    // NR = 1 or 2 stages at once: with two, each lane carries a row of each
    // through the drafts, so every draft's k^, q^ (and KDA alpha) slices are
    // loaded once for both rows and the two rows' reductions overlap
    auto rows_step = [&](auto nr_c, int c, const int (&st)[2]) {
      constexpr int NR = decltype(nr_c)::value;
      int row[NR];
      float4 s4[NR][4];
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        row[j] = GDN_S((c + j) * kRows + rloc, kMaxR);  // row within the segment
        const float* srow = S.ring[GDN_S(st[j], STAGES)] + GDN_S(rloc, kRows) * kDK;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          s4[j][cc] = *reinterpret_cast<const float4*>(srow + GDN_S(cc * 4 * kLPR + seg * 4, kDK - 3));
      }
      for (int t0 = 0; t0 < T; ++t0) {
        const int t = GDN_S(t0, MT);
        const float kq = S.snorm[t][2];
        const float alpha = S.sgate[t][0], beta = S.sgate[t][1];
        float4 kk[4], qq[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int col = GDN_S(cc * 4 * kLPR + seg * 4, kDK - 3);
          kk[cc] = *reinterpret_cast<const float4*>(&S.sy[t][kDK + col]);
          qq[cc] = *reinterpret_cast<const float4*>(&S.sy[t][col]);
          if constexpr (KDA) {
            // the rows become St diag(alpha) before their products
            const float4 al = *reinterpret_cast<const float4*>(&S.sal[t][col]);
#pragma unroll
            for (int j = 0; j < NR; ++j)
              s4[j][cc] = join4(mul2(lo2(s4[j][cc]), lo2(al)), mul2(hi2(s4[j][cc]), hi2(al)));
          }
        }
        // each row's dot products with k^ and q^, on packed fp32 pairs
        float dk_[NR], dq_[NR];
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          float2 dk2 = make_float2(0.f, 0.f), dq2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            dk2 = fma2(hi2(s4[j][cc]), hi2(kk[cc]), fma2(lo2(s4[j][cc]), lo2(kk[cc]), dk2));
            dq2 = fma2(hi2(s4[j][cc]), hi2(qq[cc]), fma2(lo2(s4[j][cc]), lo2(qq[cc]), dq2));
          }
          dk_[j] = dk2.x + dk2.y;
          dq_[j] = dq2.x + dq2.y;
        }
#pragma unroll
        for (int o = kLPR / 2; o; o >>= 1)
#pragma unroll
          for (int j = 0; j < NR; ++j) {
            dk_[j] += __shfl_xor_sync(0xffffffffu, dk_[j], o);
            dq_[j] += __shfl_xor_sync(0xffffffffu, dq_[j], o);
          }
        const int32_t sid = S.ssid[t];
        const bool keep = slot_class(sid, a.spec_num_slots) == 0;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          // KDA: alpha is 1 here (the rows carry the per-channel decay already)
          const float bu = beta * (S.sy[t][GDN_S(2 * kDK + row[j], kMaxCh)] - alpha * dk_[j]);
          const float2 bu2 = make_float2(bu, bu), al2 = make_float2(alpha, alpha);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const float2 lo = KDA ? lo2(s4[j][cc]) : mul2(al2, lo2(s4[j][cc]));
            const float2 hi = KDA ? hi2(s4[j][cc]) : mul2(al2, hi2(s4[j][cc]));
            s4[j][cc] = join4(fma2(bu2, lo2(kk[cc]), lo), fma2(bu2, hi2(kk[cc]), hi));
          }
          if (keep) {
            float4* const spec4 = reinterpret_cast<float4*>(a.spec_ssm);
            const size_t drow4 = (((size_t)sid * a.hv + h) * a.dv + (size_t)row0 + row[j]) * kDK / 4;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              st_stream(spec4 + GDN_G(drow4 + (cc * 4 * kLPR + seg * 4) / 4, spec_ssm_n / 4), s4[j][cc]);
          }
          if (seg == 0) S.so[t][row[j]] = fmaf(bu, kq, alpha * dq_[j]);
        }
      }
    };
    // the next segment's per-draft scalars (its working slot, the drafts'
    // spec slots and gate logits) into L1 while this segment's rows run, so
    // that its prologue does not start on cold global loads
    if (u < u1 && tid <= T) {
      const Seg gn = segment_at(a, u, u1);
      if (tid < T) {
        const size_t rt = (size_t)gn.r * T + tid;
        prefetch_l1(&a.spec_ids[GDN_G(rt, (long long)nreq * T)]);
        prefetch_l1(&reinterpret_cast<const Tact*>(a.b)[GDN_G(rt * a.hv + gn.h, gate_n)]);
        if (!KDA) prefetch_l1(&reinterpret_cast<const Tact*>(a.a)[GDN_G(rt * a.hv + gn.h, gate_n)]);
      } else {
        prefetch_l1(&a.slot_ids[GDN_G(gn.r, nreq)]);
      }
    }
    for (int c = 0; c < nchunks;) {
      const int nr = c + 1 < nchunks ? 2 : 1;
      const int st[2] = {(int)(n % STAGES), (int)((n + 1) % STAGES)};
      for (int j = 0; j < nr; ++j)
        if (!*abort_flag && !mbar_wait(&S.full[st[j]], ((n + j) / STAGES) & 1)) *abort_flag = 1;
      if (!*abort_flag) {
        if (nr == 2)
          rows_step(std::integral_constant<int, 2>{}, c, st);
        else
          rows_step(std::integral_constant<int, 1>{}, c, st);
        __syncwarp();  // the whole warp is done with its rows of the stages
        if (lane == 0)
          for (int j = 0; j < nr; ++j) mbar_arrive(&S.empty[st[j]]);
      }
      c += nr;
      n += nr;
    }
    named_sync(kBarCons, kCons);
    if (*abort_flag) break;
    for (int e = tid; e < T * R; e += kCons) {
      const int t = e / R, i = e % R;
      reinterpret_cast<Tact*>(a.out)[GDN_G((((size_t)r * T + t) * a.hv + h) * a.dv + row0 + i, out_n)] =
          from_f32<Tact>(S.so[GDN_S(t, MT)][GDN_S(i, kMaxR)]);
    }
  }
  if (*abort_flag && tid == 0) report(a.err, GDN_DEV_ERR_TIMEOUT);
}

template <typename Tact, typename Tconv, int STAGES, int MT, int MINB, bool KDA>
cudaError_t launch_v(const VArgs& a, cudaStream_t s) {
  using SM = VSmem<Tact, Tconv, STAGES, MT, KDA>;
  auto k = verify_tma_kernel<Tact, Tconv, STAGES, MT, MINB, KDA>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SM));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int slots = sm_count() * MINB;
  const int grid = a.n_units < slots ? (int)a.n_units : slots;
  return launch_plain(k, dim3((unsigned)grid), dim3(kThr), sizeof(SM), s, dim3(1), a);
}

template <typename Tact, typename Tconv, bool KDA>
cudaError_t launch_v_dt(const VArgs& a, cudaStream_t s) {
  // the two-CTA layout only where two fit on an SM, with a 4-stage ring (two
  // stages consumed at once, two filling) where that fits, else 3 stages
  constexpr bool kFit4 = 2 * (sizeof(VSmem<Tact, Tconv, 4, 8, KDA>) + 1024) <= 228 * 1024;
  constexpr bool kFit3 = 2 * (sizeof(VSmem<Tact, Tconv, 3, 8, KDA>) + 1024) <= 228 * 1024;
  if (a.T <= 8 && tma_ctas_per_sm() != 1) {
    if (kFit4) return launch_v<Tact, Tconv, 4, 8, 2, KDA>(a, s);
    if (kFit3) return launch_v<Tact, Tconv, 3, 8, 2, KDA>(a, s);
  }
  return launch_v<Tact, Tconv, 4, kMaxT, 1, KDA>(a, s);
}

template <bool KDA>
cudaError_t launch_v_kda(const gdn_dims& d, const VArgs& a, cudaStream_t s) {
  if (d.act_dtype == GDN_BF16 && d.conv_dtype == GDN_BF16) return launch_v_dt<__nv_bfloat16, __nv_bfloat16, KDA>(a, s);
  if (d.act_dtype == GDN_BF16) return launch_v_dt<__nv_bfloat16, float, KDA>(a, s);
  return launch_v_dt<float, float, KDA>(a, s);
}

}  // namespace

bool verify_tma_supported(const gdn_dims& d, int32_t T, const void* qkv, const gdn_params& p) {
  const size_t ea = dtype_size(d.act_dtype), ec = dtype_size(d.conv_dtype);
  const int64_t C = channels(d);
  if (d.dk != kDK || d.conv_width != kW || T < 1 || T > kMaxT) return false;
  if (d.dv % kRows) return false;
  if ((C * ea) % 16 || (C * ec) % 16 || (kDK * ea) % 16 || (kDK * ec) % 16) return false;
  if ((kRows * ea) % 16 || (kRows * ec) % 16) return false;
  if (!aligned(qkv, 16) || !aligned(p.conv_w, 16)) return false;
  return true;
}

cudaError_t verify_tma_launch(const gdn_dims& d, const gdn_pool& work, const gdn_pool& spec,
                              const gdn_params& p, const int32_t* slot_ids, const int32_t* spec_ids,
                              int32_t B, int32_t T, const void* qkv, const void* av, const void* bv,
                              void* out, uint32_t* dev_err, bool kda, cudaStream_t s) {
  VArgs a;
  a.ssm = work.ssm;
  a.conv = work.conv;
  a.num_slots = work.num_slots;
  a.spec_ssm = spec.ssm;
  a.spec_conv = spec.conv;
  a.spec_num_slots = spec.num_slots;
  a.spec_ids = spec_ids;
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
  a.T = T;
  if (d.dv % kRows) return cudaErrorInvalidValue;
  a.sph = d.dv / kRows;
  a.n_units = (int64_t)B * d.hv * a.sph;
  return kda ? launch_v_kda<true>(d, a, s) : launch_v_kda<false>(d, a, s);
}

}  // namespace gdn
