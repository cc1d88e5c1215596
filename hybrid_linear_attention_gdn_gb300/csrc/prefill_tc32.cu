// Chunked GDN prefill on the 5th-generation tensor cores, every product in
// tf32 (fp32 operands with 10 explicit mantissa bits, fp32 accumulation).
//
// Same contract as prefill.cu (TokenSpeed Qwen3.5 page, "Ciclo de vida de
// slots": block-aligned checkpoints of state and conv history, the final
// state in the working slot) and the same chunk form: the chunkwise WY/UT form
// of the gated delta rule (Yang et al., NeurIPS 2024; Gated Delta Networks,
// ICLR 2025), chunks of 64 tokens aligned to absolute positions, for dk = dv =
// 128, conv width 4, bf16 activations and conv history.
//
// One CTA per (V head, sequence) walks the sequence's chunks in order; nothing
// goes through a workspace.  Per chunk (transposed so that M = 128 rows of the
// tensor core are dv rows, or the chunk's 64 k^ rows and 64 q^ rows):
//   features   the 67 raw input rows (3 of history) of the head's q, k and v
//              channels arrive by three TMA tensor copies; one thread per
//              channel runs conv1d + SiLU down the chunk.  The q and k rows
//              are kept unnormalised (Y_K, Y_Q): their L2 norms come out of
//              the next product and are folded into the small operands below.
//              Written as tf32 operands: [Y_K ; Y_Q] (shared memory, K-major),
//              K~^T = (diag(e^{b_last - b}) Y_K)^T (shared memory, K-major
//              over tokens) and V^T (tensor memory).
//   P          [Y_K;Y_Q] [Y_K;Y_Q]^T (tcgen05, TMEM): its diagonal gives the
//              norms, rk_i = 1/|y_k,i|, rq_i = dk^-1/2 / |y_q,i| (with the eps)
//   A, M'      A = strict_lower(beta_i rk_i rk_j (Y_K Y_K^T)_ij Gamma_ij)
//              (fp32, for the solve), M'_ij = rq_i (Y_Q Y_K^T)_ij Gamma_ij on
//              and below the diagonal (tf32 operand)
//   T          X = (I + A)^-1 by 8 x 8 substitutions and three merge levels,
//              fp32 on the CUDA cores; written as T1 = diag(rk) X diag(beta)
//              and T2 = -diag(rk) X diag(beta e^b rk) (tf32 operands)
//   Delta'^T   = V^T T1^T + (S^T Y_K^T) T2^T = (diag(rk) Delta)^T: the WY
//              form's U - W S with W = T diag(e^b) K^, regrouped so that the
//              state meets only the T-free Y_K (S^T Y_K^T comes with
//              S^T Y_Q^T in one product whose A operand is the state itself,
//              in TMEM)
//   state      S^T <- e^{b_last} S^T (in TMEM, by the threads) + Delta'^T K~
//              (one product accumulating into the state; A = Delta'^T in TMEM)
//   output     O = (S^T Y_Q^T) diag(rq e^b) + Delta'^T M'^T, staged as a bf16
//              tile and written by one TMA tensor store; or, with the readout
//              epilogue fused (EPI), staged in fp32 and written as
//              y = O / sqrt(mean(O^2) + eps) * w * silu(z) per token, z
//              arriving by its own TMA tile
// With k^ = diag(rk) Y_K and q^ = diag(rq) Y_Q these are the chunk form's
// products exactly: the rk factors of Delta and of the state update meet in
// Delta', and M' = M diag(1/rk).
// The fp32 state S^T (dv x dk) lives in TMEM for the whole sequence: it is
// the accumulator of its own update and the A operand of the products that
// read it.  Checkpoints are staged from TMEM into the dead [K;Q] tile and
// leave by TMA tensor stores.  The conv histories of checkpoints and of the
// final state come from the history kernel of prefill.cu.
#include "gdn_common.cuh"
#include "decode_tma.cuh"
#include "decode_tma_item.cuh"
#include "prefill_history.cuh"
#include "prefill_tc.cuh"
#include "tma.cuh"
#include "umma.cuh"

#include <atomic>
#include <cstdlib>

namespace gdn {
namespace {

#include "tc32_common.cuh"

// TMEM columns (fp32, one per column).  Lanes are dv rows, except P, whose
// lanes are the [Y_K;Y_Q] rows.
constexpr uint32_t TM_S = 0;     // S^T [dv][dk], 128 columns
constexpr uint32_t TM_P = 128;   // P [128 rows][128]
constexpr uint32_t TM_E = 256;   // S^T Y_K^T [dv][64]
constexpr uint32_t TM_O1 = 320;  // S^T Y_Q^T [dv][64]
constexpr uint32_t TM_DL = 384;  // Delta'^T [dv][64]
constexpr uint32_t TM_V = 448;   // V^T [dv][64] (operand); then O2:
constexpr uint32_t TM_O2 = 448;  //   Delta'^T M'^T [dv][64] (V read by then)
constexpr uint32_t TM_COLS = 512;

struct Tc32Args {
  float* ssm;
  int32_t num_slots;
  float* ck_ssm;
  int32_t ck_num_slots;
  const __nv_bfloat16* conv;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const int32_t* slot_ids;
  const int32_t* cu_seqlens;
  const int64_t* start_pos;
  int32_t n_seq;
  int64_t total;
  const int32_t* ckpt_ids;
  int32_t max_ckpt;
  int32_t ckpt_block;
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  __nv_bfloat16* out;
  uint32_t* err;
  int32_t hk, hv, C, G;
  const float* norm_w;  // the fused epilogue's weight [dv] (EPI)
  float eps;
};

// Shared memory.  Operand tiles are fp32 in the tensor core's 128-byte
// swizzled K-major layout: a 128-byte row holds 32 elements, 8-row groups
// are 1024 bytes apart, and wider rows continue in further 32-column blocks.
struct __align__(1024) Smem32 {
  uint8_t kq[4 * 128 * 128];  // [Y_K ; Y_Q]: rows 0..63 k, 64..127 q (x dk): 4 blocks of 16 KB
  uint8_t kt[2 * 128 * 128];  // K~^T [dk][64 tokens]: 2 blocks of 16 KB
  uint8_t tm[2 * 64 * 128];   // T1 [i][j]: 2 blocks of 8 KB
  uint8_t t2[2 * 64 * 128];   // T2; after its product, the output staging tile
  uint8_t mq[2 * 64 * 128];   // M' [i][j]
  union {
    __nv_bfloat16 raw[3][kRawRows][kD];  // staged inputs: q, k, v parts
    struct {
      float A[kC * kAX];
      float X[kC * kAX];
      float Y[2048];
      float L0[8][3][64];  // per 8 x 8 diagonal block: L^2, L^4, (I - L)(I + L^2)
    } sv;  // the solve's scratch (after the features have read the inputs)
  };
  float g[2][kC], beta[2][kC], b[2][kC], eb[2][kC], ebl[2][kC];  // by chunk parity
  float rk[kC];  // 1 / sqrt(|y_k|^2 + eps) per token
  float rq[kC];  // dk^-1/2 / sqrt(|y_q|^2 + eps) per token
  __nv_bfloat16 zt[kC][kD];  // the fused epilogue's z rows of the chunk (EPI)
  uint64_t ld_bar, mma_bar, z_bar, eo_bar;
  uint32_t tmem_base;
};

__device__ __forceinline__ bool seq_ok(const Tc32Args& a, int n, int64_t& t0, int64_t& len, int64_t& p0) {
  const auto cu = GDN_GV(a.cu_seqlens, a.n_seq + 1);
  t0 = cu[n];
  len = (int64_t)cu[n + 1] - t0;
  p0 = GDN_GV(a.start_pos, a.n_seq)[n];
  return !(t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0);
}


// ---- one chain ---------------------------------------------------------------
// V head h of sequence n, by all kThreads threads of the CTA, which holds the
// 512 TMEM columns from `tmem` on.  Thread 0 issues the TMA copies and the
// tensor-core products; every wait is bounded (1 s).  The chain's barriers
// are set up here and invalidated at its end, after its last tensor store
// has completed, so the shared memory can serve the next work item.
template <typename Tconv, bool EPI>
__device__ __forceinline__ void tc32_chain(const Tc32Args& a, const CUtensorMap& qmap, const CUtensorMap& omap,
                                           const CUtensorMap& cmap, const CUtensorMap& zmap, Smem32& S,
                                           const uint32_t tmem, const int h, const int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = h / a.G;
  int64_t t0, len, p0;
  if (!seq_ok(a, n, t0, len, p0)) {
    if (h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  // the caller's tensors (extents in elements)
  const auto out = GDN_GV(a.out, a.total * a.hv * kD);
  const auto gate_a = GDN_GV(a.a, a.total * a.hv), gate_b = GDN_GV(a.b, a.total * a.hv);
  const auto ckpt_ids = GDN_GV(a.ckpt_ids, (long long)a.n_seq * a.max_ckpt);
  const int32_t slot = GDN_GV(a.slot_ids, a.n_seq)[n];
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * kD; e += kThreads)
      out[((t0 + e / kD) * a.hv + h) * kD + (e % kD)] = __float2bfloat16_rn(0.f);
    return;
  }
  if (len == 0) return;
  const int64_t p1 = p0 + len;
  const int nch = (int)((p1 + kC - 1) / kC - p0 / kC);

  if (tid == 0) {
    mbar_init(&S.ld_bar, 1);
    mbar_init(&S.mma_bar, 1);
    mbar_init(&S.z_bar, 1);
    mbar_init(&S.eo_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int lrow = 32 * (warp & 3) + lane;  // TMEM lane of this thread (dv row, or [Y_K;Y_Q] row)
  const int qq = warp >> 2;                 // which column quarter this warp handles
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

  constexpr uint32_t ID_N64 = umma::idesc_tf32(128, 64, false, false);
  constexpr uint32_t ID_N128 = umma::idesc_tf32(128, 128, false, false);
  // operand extents of the products below (their k-steps walk 32-column
  // blocks: 128 rows x 128 bytes per block of kq and kt, 64 rows of tm, t2, mq)
  static_assert(4 * 16384 <= sizeof(Smem32::kq) && 2 * 16384 <= sizeof(Smem32::kt), "operand tiles");
  static_assert(2 * 8192 <= sizeof(Smem32::tm) && 2 * 8192 <= sizeof(Smem32::t2) && 2 * 8192 <= sizeof(Smem32::mq),
                "operand tiles");
  static_assert(TM_P == TM_S + 128 && TM_E == TM_P + 128 && TM_O1 == TM_E + 64 && TM_DL == TM_O1 + 64 &&
                    TM_V == TM_DL + 64 && TM_V + 64 <= TM_COLS && TM_O2 == TM_V,
                "TMEM regions");

  // feature channels of this thread: the q/k channel pair (2 cp, 2 cp + 1)
  // (k for tid % 128 < 64, else q) for tokens 16 qq .., and v channel lrow
  // for the same tokens
  const bool isq = (tid & 127) >= 64;
  const int cp = tid & 63;
  const int gch_qk = (isq ? hq : a.hk + hq) * kD + 2 * cp;
  const int gch_v = 2 * a.hk * kD + h * kD + lrow;
  float2 wqk[4];
  float wv[4];
  {
    const auto cw = GDN_GV(a.conv_w, (long long)a.C * 4);
    const float4 w4 = vec_at<const float4>(cw, (size_t)gch_qk * 4);
    const float4 u4 = vec_at<const float4>(cw, (size_t)(gch_qk + 1) * 4);
    wqk[0] = make_float2(w4.x, u4.x); wqk[1] = make_float2(w4.y, u4.y);
    wqk[2] = make_float2(w4.z, u4.z); wqk[3] = make_float2(w4.w, u4.w);
    const float4 v4 = vec_at<const float4>(cw, (size_t)gch_v * 4);
    wv[0] = v4.x; wv[1] = v4.y; wv[2] = v4.z; wv[3] = v4.w;
  }
  const float eA = expf(GDN_GV(a.A_log, a.hv)[h]), dtb = GDN_GV(a.dt_bias, a.hv)[h];
  const int part_x[3] = {hq * kD, (a.hk + hq) * kD, 2 * a.hk * kD + h * kD};

  // checkpoint slot at the end of chunk c (-1: none): chunk c ends at the
  // absolute chunk boundary p0 / 64 + c + 1, a block boundary when
  // q = (p0 / 64) mod kpc + c + 1 is a multiple of kpc (kpc = block / 64),
  // with checkpoint index q / kpc - 1; a last chunk cut short ends on none
  const int kpc = a.ckpt_block / kC;
  const int q0 = (int)((p0 / kC) % kpc);
  const bool last_full = (p1 % kC) == 0;
  auto ckpt_slot = [&](int c) -> int32_t {
    if (c == nch - 1 && !last_full) return -1;
    const int q = q0 + c + 1;
    if (q % kpc != 0) return -1;
    const int idx = q / kpc - 1;
    if (idx >= a.max_ckpt) return -1;
    const int32_t id = ckpt_ids[(size_t)n * a.max_ckpt + idx];
    return slot_class(id, a.ck_num_slots) == 0 ? id : -1;
  };
  auto issue_raw = [&](int c) {  // thread 0: chunk c's raw rows into S.raw
    const int64_t P = (p0 / kC + c) * kC;
    const int32_t row0 = (int32_t)(t0 + (P - 3 - p0));  // packed row of raw row 0 (may be < 0)
    mbar_arrive_expect_tx(&S.ld_bar, 3u * kRawRows * kD * 2u);
#pragma unroll
    for (int q = 0; q < 3; ++q)  // a box of 128 channels from part_x[q], 67 rows (rows outside: zeros)
      if (GDN_SPAN_G(part_x[q], kD, a.C) && GDN_SBYTES(&S.raw[q][0][0], kRawRows * kD * 2, S))
        tma_load_2d(&S.raw[q][0][0], &qmap, part_x[q], row0, &S.ld_bar);
  };
  // gate inputs of chunk c's token tid - 256 (threads 256..319), loaded one
  // chunk ahead
  auto load_gates = [&](int c, float& av, float& bv) {
    const int64_t pos = (p0 / kC + c) * kC + (tid - 8 * 32);
    av = bv = 0.f;
    if (c < nch && pos >= p0 && pos < p1) {
      const size_t tok = (size_t)(t0 + pos - p0);
      av = __bfloat162float(gate_a[tok * a.hv + h]);
      bv = __bfloat162float(gate_b[tok * a.hv + h]);
    }
  };

  // gates of chunk cc into buffer buf (warps 8 and 9: thread 256 + t for
  // token t, with the inputs loaded one chunk ahead in ga, gb; outside the
  // sequence g = beta = 0), then the cumulative log decay b, e^b and
  // e^{b_last - b} (warp 8)
  const int gt = tid - 8 * 32;  // token of a gate thread
  const bool gate_thread = gt >= 0 && gt < kC;
  float ga = 0.f, gb = 0.f;
  auto gates_into = [&](int cc, int buf) {
    if (gate_thread) {
      const int64_t pos = (p0 / kC + cc) * kC + gt;
      const bool in = pos >= p0 && pos < p1;
      S.g[buf][GDN_S(gt, kC)] = in ? floor_log_decay(-eA * softplus_f(ga + dtb)) : 0.f;
      S.beta[buf][gt] = in ? sigmoid_f(gb) : 0.f;
      load_gates(cc + 1, ga, gb);
      named_sync(1, kC);
    }
    if (warp == 8) {
      float bv[2], carry = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v = S.g[buf][32 * hh + lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += u;
        }
        bv[hh] = v + carry;
        carry = __shfl_sync(0xffffffffu, bv[hh], 31);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        S.b[buf][32 * hh + lane] = bv[hh];
        S.eb[buf][32 * hh + lane] = expf(bv[hh]);
        S.ebl[buf][32 * hh + lane] = expf(carry - bv[hh]);
      }
    }
  };

  // initial state S^T rows into TMEM; the upper triangle of T1 stays zero
  const auto gS = GDN_GV(a.ssm, (long long)a.num_slots * a.hv * kD * kD) +
                  ((((size_t)slot * a.hv + h) * kD + lrow) * kD + 32 * qq);
  {
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = vec_at<const float4>(gS, 4 * i);
      v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
    }
    umma::tmem_st32(tlane + TM_S + 32 * qq, v);
  }
  for (int e = tid; e < (int)(sizeof(S.tm) / 16); e += kThreads)
    reinterpret_cast<uint4*>(S.tm)[e] = make_uint4(0u, 0u, 0u, 0u);
  int ld_issued = 0, ld_done = 0;  // raw-row loads issued (thread 0) and completed
  if (tid == 0) {
    issue_raw(0);
    ld_issued = 1;
  }
  if (gate_thread) load_gates(0, ga, gb);
  gates_into(0, 0);

  bool bad = false;
  uint32_t mph = 0;
  // all threads wait (bounded) for a phase, then synchronise; false (in
  // every thread) if any thread's wait expired
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (!mbar_wait(bar, parity)) bad = true;
    return !__syncthreads_or(bad);
  };
  auto mma_wait = [&]() -> bool {
    const bool ok = wait_all(&S.mma_bar, mph);
    mph ^= 1;
    umma::fence_after();
    return ok;
  };

  bool eo_pending = false;  // [E | O1] of chunk c issued and not yet waited for
  int c = 0;
  for (; c < nch; ++c) {
    const int64_t P = (p0 / kC + c) * kC;
    const bool full = P >= p0 && P + kC <= p1;
    const int gbuf = c & 1;
    // tokens tlo .. thi - 1 of the chunk lie inside the sequence
    const int tlo = (int)(p0 > P ? (p0 - P < kC ? p0 - P : kC) : 0);
    const int thi = (int)(p1 > P ? (p1 - P < kC ? p1 - P : kC) : 0);
    const float* gb_ = S.b[gbuf];
    const float* geb = S.eb[gbuf];
    const float* gebl = S.ebl[gbuf];
    const float* gbeta = S.beta[gbuf];
    // the previous chunk's tensor stores have read the kq tile (checkpoint
    // staging) and the t2 tile (output staging); the gates of this chunk are
    // in buffer gbuf
    if (tid == 0) bulk_wait_read();
    // the fused epilogue's z rows of this chunk (the previous chunk's output
    // step has read the tile: it ended with a CTA barrier)
    if (EPI && tid == 0) {
      mbar_arrive_expect_tx(&S.z_bar, (uint32_t)sizeof(S.zt));
      if (GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD))
        tma_load_2d(&S.zt[0][0], &zmap, h * kD, (int32_t)(t0 + (P - p0)), &S.z_bar);
    }
    // the chunk's raw rows landed
    if (!wait_all(&S.ld_bar, c & 1)) break;
    ld_done = c + 1;
    // the up to 3 rows just before the sequence start come from the conv history
    if (P - 3 < p0) {
      const int64_t lo = (P - 3 > p0 - 3) ? P - 3 : p0 - 3;
      const int64_t hi = (P + kC < p0) ? P + kC : p0;
      const auto hist = GDN_GV(reinterpret_cast<const Tconv*>(a.conv), (long long)a.num_slots * 3 * a.C) +
                        (size_t)slot * 3 * a.C;
      for (int64_t pos = lo; pos < hi; ++pos) {
        const int r = GDN_S((int)(pos - (P - 3)), kRawRows);
        for (int e = tid; e < 3 * kD; e += kThreads) {
          const int q = e / kD, ch = e % kD;
          S.raw[q][r][ch] = __float2bfloat16_rn(to_f32(hist[(size_t)(3 - (p0 - pos)) * a.C + part_x[q] + ch]));
        }
      }
      __syncthreads();
    }

    // ---- features: conv1d + SiLU, down the chunk ---------------------------
    // (each thread's raw rows are loaded into registers first, so that no
    // shared-memory store of the results has to wait for, or hold up, them)
    {
      const int tk = 16 * qq;
      // q or k: a channel pair, as packed fp32 pairs; its [Y_K ; Y_Q]
      // columns and, for k, its two K~^T rows
      float2 y[16];
      {
        // channel pair 2 cp of rows tk .. tk + 18 of the q or k part
        const auto xs = GDN_SV(reinterpret_cast<const __nv_bfloat162*>(&S.raw[isq ? 0 : 1][0][0]), kRawRows * kD / 2) +
                        (tk * (kD / 2) + cp);
        float2 x[19];
#pragma unroll
        for (int r = 0; r < 19; ++r) x[r] = __bfloat1622float2(xs[r * (kD / 2)]);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float2 acc = mul2(wqk[0], x[t]);
          acc = fma2(wqk[1], x[t + 1], acc);
          acc = fma2(wqk[2], x[t + 2], acc);
          acc = fma2(wqk[3], x[t + 3], acc);
          const bool valid = (unsigned)(tk + t - tlo) < (unsigned)(thi - tlo);
          y[t] = valid ? make_float2(umma::tf32_round(silu_tanh(acc.x)), umma::tf32_round(silu_tanh(acc.y)))
                       : make_float2(0.f, 0.f);
        }
      }
      const int R0 = (isq ? kC : 0) + tk;
#pragma unroll
      for (int t = 0; t < 16; ++t) tile_at<float2>(S.kq, sizeof(S.kq), f32_off(R0 + t, 2 * cp, 128 * 128)) = y[t];
      if (!isq) {
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          const float4 e4 = *reinterpret_cast<const float4*>(&gebl[GDN_S(tk + 4 * t4, kC - 3)]);
          tile_at<float4>(S.kt, sizeof(S.kt), f32_off(2 * cp, tk + 4 * t4, 128 * 128)) =
              make_float4(umma::tf32_round(y[4 * t4].x * e4.x), umma::tf32_round(y[4 * t4 + 1].x * e4.y),
                          umma::tf32_round(y[4 * t4 + 2].x * e4.z), umma::tf32_round(y[4 * t4 + 3].x * e4.w));
          tile_at<float4>(S.kt, sizeof(S.kt), f32_off(2 * cp + 1, tk + 4 * t4, 128 * 128)) =
              make_float4(umma::tf32_round(y[4 * t4].y * e4.x), umma::tf32_round(y[4 * t4 + 1].y * e4.y),
                          umma::tf32_round(y[4 * t4 + 2].y * e4.z), umma::tf32_round(y[4 * t4 + 3].y * e4.w));
        }
      }
      // v: channel lrow, into TMEM
      float vv[16];
      {
        const auto xv = GDN_SV(&S.raw[2][0][0], kRawRows * kD) + (tk * kD + lrow);
        float x[19];
#pragma unroll
        for (int r = 0; r < 19; ++r) x[r] = __bfloat162float(xv[r * kD]);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float acc = wv[0] * x[t];
          acc = fmaf(wv[1], x[t + 1], acc);
          acc = fmaf(wv[2], x[t + 2], acc);
          acc = fmaf(wv[3], x[t + 3], acc);
          const bool valid = (unsigned)(tk + t - tlo) < (unsigned)(thi - tlo);
          vv[t] = valid ? umma::tf32_round(silu_tanh(acc)) : 0.f;
        }
      }
      umma::tmem_st16(tlane + TM_V + tk, vv);
    }
    // operands visible to the tensor core, then P = [Y_K;Y_Q] [Y_K;Y_Q]^T
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    if (tid == 0) {
      umma::fence_after();
      const uint64_t dkq = umma::desc(smem_addr(S.kq), 16, 1024);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
        umma::mma_tf32(tmem + TM_P, umma::adv(dkq, ko), umma::adv(dkq, ko), ID_N128, s > 0);
      }
      umma::commit(&S.mma_bar);
    }
    // meanwhile X is cleared for the solve (the raw rows are read) and T2 for
    // its lower triangle (its tile held the previous chunk's output staging)
    for (int e = tid; e < kC * kAX / 4; e += kThreads)
      reinterpret_cast<float4*>(S.sv.X)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = tid; e < (int)(sizeof(S.t2) / 16); e += kThreads)
      reinterpret_cast<uint4*>(S.t2)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (!mma_wait()) break;
    // ---- norms from P's diagonal: rk_i (K block), rq_i (Q block) ------------
    // warps 0..3: lane quarter w holds the diagonal entries (lrow, lrow) in
    // the 32 x 32 block at columns 32 w ..
    if (qq == 0) {
      float v[32];
      umma::tmem_ld32(tlane + TM_P + 32 * warp, v);
      float d = v[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) d = (lane == i) ? v[i] : d;
      if (lrow < kC)
        S.rk[GDN_S(lrow, kC)] = rsqrtf(d + kNormEps);
      else
        S.rq[GDN_S(lrow - kC, kC)] = rsqrtf(d + kNormEps) * rsqrtf((float)kD);
    }
    __syncthreads();
    // ---- A (fp32, for the solve) and M' (tf32 operand) from P ---------------
    // thread: row lrow, columns 16 qq .. 16 qq + 15
    {
      float v[16];
      umma::tmem_ld16(tlane + TM_P + 16 * qq, v);
      const int c0 = 16 * qq;
      float bc[16], rkc[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 b4 = *reinterpret_cast<const float4*>(&gb_[GDN_S(c0 + 4 * i, kC - 3)]);
        bc[4 * i] = b4.x; bc[4 * i + 1] = b4.y; bc[4 * i + 2] = b4.z; bc[4 * i + 3] = b4.w;
        const float4 r4 = *reinterpret_cast<const float4*>(&S.rk[c0 + 4 * i]);
        rkc[4 * i] = r4.x; rkc[4 * i + 1] = r4.y; rkc[4 * i + 2] = r4.z; rkc[4 * i + 3] = r4.w;
      }
      if (lrow < kC) {
        const int r = lrow;
        const float br = gb_[r], fr = gbeta[r] * S.rk[r];
        float av[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) av[i] = (c0 + i < r) ? fr * rkc[i] * v[i] * exp_ftz(br - bc[i]) : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          vec_at<float4>(GDN_SV(S.sv.A, kC * kAX), ix(r, c0 + 4 * q)) =
              make_float4(av[4 * q], av[4 * q + 1], av[4 * q + 2], av[4 * q + 3]);
      } else {
        const int r = lrow - kC;
        const float br = gb_[r], fr = S.rq[r];
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) m[i] = (c0 + i <= r) ? umma::tf32_round(fr * v[i] * exp_ftz(br - bc[i])) : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tile_at<float4>(S.mq, sizeof(S.mq), f32_off(r, c0 + 4 * q, 64 * 128)) =
              make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
      }
    }
    umma::fence_before();
    __syncthreads();
    // the next chunk's gates (warps 8, 9) beside the solve's diagonal blocks
    if (c + 1 < nch && (warp == 8 || warp == 9)) gates_into(c + 1, gbuf ^ 1);
    // [E | O1] = S^T [Y_K;Y_Q]^T: the state entering the chunk (final since
    // the previous chunk's update completed) meets the chunk's keys and
    // queries on the tensor core during the solve.  Issued by a lane of warp
    // 10, idle in the solve's first phase: a thread issuing products waits
    // for the tensor core to take them, about as long as they run.
    eo_pending = true;
    if (warp == 10 && lane == 0) {
      umma::fence_after();
      const uint64_t dkq = umma::desc(smem_addr(S.kq), 16, 1024);
#pragma unroll
      for (int s = 0; s < 16; ++s)
        umma::mma_tf32_ta(tmem + TM_E, tmem + TM_S + 8 * s, umma::adv(dkq, (s >> 2) * 16384 + (s & 3) * 32),
                          ID_N128, s > 0);
      umma::commit(&S.eo_bar);
    }
    solve_T(S.sv.A, S.sv.X, S.sv.Y, S.sv.L0, TOut{S.tm, S.t2, gbeta, geb, S.rk});
    umma::fence_proxy_async();
    __syncthreads();
    // the next chunk's raw rows (the solve's scratch is dead)
    if (tid == 0 && c + 1 < nch) {
      issue_raw(c + 1);
      ld_issued = c + 2;
    }
    // E and O1 have long completed (every thread sees it before the state,
    // which they read, is scaled below)
    if (!wait_all(&S.eo_bar, c & 1)) break;
    eo_pending = false;
    umma::fence_after();
    // ---- Delta'^T = V^T T1^T + E T2^T (tensor core), S^T <- e^{b_last} S^T --
    if (tid == 0) {
      const uint64_t dtm = umma::desc(smem_addr(S.tm), 16, 1024);
      const uint64_t dt2 = umma::desc(smem_addr(S.t2), 16, 1024);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_DL, tmem + TM_V + 8 * s, umma::adv(dtm, (s >> 2) * 8192 + (s & 3) * 32), ID_N64,
                          s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_DL, tmem + TM_E + 8 * s, umma::adv(dt2, (s >> 2) * 8192 + (s & 3) * 32), ID_N64,
                          true);
      umma::commit(&S.mma_bar);
    }
    {
      const float dec = geb[kC - 1];
      float v[32];
      umma::tmem_ld32(tlane + TM_S + 32 * qq, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= dec;
      umma::tmem_st32(tlane + TM_S + 32 * qq, v);
    }
    umma::fence_before();
    if (!mma_wait()) break;
    // ---- S^T += Delta'^T K~ ; O2 = Delta'^T M'^T ------------------------------
    if (tid == 0) {
      const uint64_t dkt = umma::desc(smem_addr(S.kt), 16, 1024);
      const uint64_t dmq = umma::desc(smem_addr(S.mq), 16, 1024);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_S, tmem + TM_DL + 8 * s, umma::adv(dkt, (s >> 2) * 16384 + (s & 3) * 32), ID_N128,
                          true);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_O2, tmem + TM_DL + 8 * s, umma::adv(dmq, (s >> 2) * 8192 + (s & 3) * 32), ID_N64,
                          s > 0);
      umma::commit(&S.mma_bar);
    }
    if (!mma_wait()) break;
    // ---- output O = O1 diag(rq e^b) + O2, staged [token][dv] bf16 in t2 ------
    if constexpr (!EPI) {
      float o1[16], o2[16];
      umma::tmem_ld16(tlane + TM_O1 + 16 * qq, o1);
      umma::tmem_ld16(tlane + TM_O2 + 16 * qq, o2);
      const auto ot = GDN_SV(reinterpret_cast<__nv_bfloat16*>(S.t2), kC * kD);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        ot[(16 * qq + i) * kD + lrow] = __float2bfloat16_rn(fmaf(o1[i], S.rq[16 * qq + i] * geb[16 * qq + i], o2[i]));
    } else {
      // fp32 O staged [token][dv] in the kt tile (dead since the state update),
      // then per token y = O / sqrt(mean(O^2) + eps) * w * silu(z) into t2
      {
        float o1[16], o2[16];
        umma::tmem_ld16(tlane + TM_O1 + 16 * qq, o1);
        umma::tmem_ld16(tlane + TM_O2 + 16 * qq, o2);
        const auto of = GDN_SV(reinterpret_cast<float*>(S.kt), kC * kD);
#pragma unroll
        for (int i = 0; i < 16; ++i) of[(16 * qq + i) * kD + lrow] = fmaf(o1[i], S.rq[16 * qq + i] * geb[16 * qq + i], o2[i]);
      }
      if (!wait_all(&S.z_bar, c & 1)) break;
      const float4 w4 = vec_at<const float4>(GDN_GV(a.norm_w, kD), 4 * lane);
      const auto of = GDN_SV(reinterpret_cast<const float*>(S.kt), kC * kD);
      const auto ot = GDN_SV(reinterpret_cast<__nv_bfloat16*>(S.t2), kC * kD);
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // tokens 4 warp + k: lane holds dv 4 lane .. 4 lane + 3
        const int t = GDN_S(4 * warp + k, kC);
        const float4 o4 = vec_at<const float4>(of, t * kD + 4 * lane);
        float ss = o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w;
#pragma unroll
        for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float inv = rsqrtf(ss / (float)kD + a.eps);
        const uint2 zu = *reinterpret_cast<const uint2*>(&S.zt[t][4 * lane]);
        const float2 z01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zu.x));
        const float2 z23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zu.y));
        const __nv_bfloat162 y01 = __floats2bfloat162_rn(o4.x * inv * w4.x * silu_fast(z01.x),
                                                         o4.y * inv * w4.y * silu_fast(z01.y));
        const __nv_bfloat162 y23 = __floats2bfloat162_rn(o4.z * inv * w4.z * silu_fast(z23.x),
                                                         o4.w * inv * w4.w * silu_fast(z23.y));
        uint2 yu;
        yu.x = *reinterpret_cast<const uint32_t*>(&y01);
        yu.y = *reinterpret_cast<const uint32_t*>(&y23);
        vec_at<uint2>(ot, t * kD + 4 * lane) = yu;
      }
    }
    // checkpoint: the state rows, 128B-swizzled, into four 16 KB boxes (32
    // columns x 128 rows) in the dead kq tile, for four tensor stores
    const int32_t cid = ckpt_slot(c);
    if (cid >= 0) {
      float v[32];
      umma::tmem_ld32(tlane + TM_S + 32 * qq, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        tile_at<float4>(S.kq, sizeof(S.kq), qq * 16384 + lrow * 128 + ((j ^ (lrow & 7)) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    if (tid == 0) {
      // boxes: 128 channels x 64 tokens of the output; 32 x 128 rows of a checkpoint
      if (full && GDN_SPAN_G(t0 + (P - p0), kC, a.total) && GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD))
        tma_store_2d(&omap, S.t2, h * kD, (int32_t)(t0 + (P - p0)));
      if (cid >= 0) {
        const int32_t y = (int32_t)(((int64_t)cid * a.hv + h) * kD);
        if (GDN_SPAN_G(y, kD, (long long)a.ck_num_slots * a.hv * kD)) {
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_store_2d(&cmap, S.kq + k * 16384, 32 * k, y);
        }
      }
      bulk_commit();
    }
    if (!full) {  // rows of the chunk's tokens inside the sequence: 16-byte stores
      const auto ot = GDN_SV(reinterpret_cast<const __nv_bfloat16*>(S.t2), kC * kD);
      for (int e = tid; e < kC * (kD / 8); e += kThreads) {
        const int r = e / (kD / 8), ch = e % (kD / 8);
        const int64_t pos = P + r;
        if (pos >= p0 && pos < p1)
          vec_at<uint4>(out, ((t0 + pos - p0) * a.hv + h) * kD + ch * 8) = vec_at<const uint4>(ot, r * kD + ch * 8);
      }
    }
  }
  if (c < nch) {
    // a wait expired: let the copies and products in flight land first
    if (tid == 0) {
      report(a.err, GDN_DEV_ERR_TIMEOUT);
      umma::commit(&S.mma_bar);
      mbar_wait(&S.mma_bar, mph);
      if (eo_pending) mbar_wait(&S.eo_bar, c & 1);
      for (int k = ld_done; k < ld_issued; ++k) mbar_wait(&S.ld_bar, k & 1);
      if (EPI) mbar_wait(&S.z_bar, c & 1);
    }
  } else {
    // the final state
    float v[32];
    umma::tmem_ld32(tlane + TM_S + 32 * qq, v);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      vec_at<float4>(gS, 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
  if (tid == 0) bulk_wait_all();
  umma::fence_before();
  __syncthreads();
  if (tid == 0) {
    mbar_inval(&S.ld_bar);
    mbar_inval(&S.mma_bar);
    mbar_inval(&S.z_bar);
    mbar_inval(&S.eo_bar);
  }
}

// grid (hv, n_seq), 512 threads, one CTA per SM: one chain each.
template <typename Tconv, bool EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc32_prefill_kernel(const Tc32Args a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap cmap,
                        const __grid_constant__ CUtensorMap zmap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem32& S = *reinterpret_cast<Smem32*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int warp = threadIdx.x >> 5;
  if (warp == 0) umma::tmem_alloc(&S.tmem_base, TM_COLS);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = S.tmem_base;
  tc32_chain<Tconv, EPI>(a, qmap, omap, cmap, zmap, S, tmem, blockIdx.x, blockIdx.y);
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, TM_COLS);
}

// ---- the single-launch mixed step ---------------------------------------------
// TokenSpeed talk, "Kernel: 让 MLA 真正跑满 GPU": a decode-first batch of
// decode requests and prefill continuations, variable length, no padding.
// One persistent launch (one CTA per SM) takes work items from a queue in
// global memory, in this order:
//   chains     (V head, continuation): tc32_chain above;
//   decode     (request, QK head): the TMA-fed decode items of
//              decode_tma_item.cuh.  A CTA that takes one enters a decode
//              walk: its producer lane takes the following items itself and
//              hands each to the consumers with its bundle, until it takes a
//              non-decode item, which ends the walk for the whole CTA;
//   histories  (continuation, checkpoint group, 512 channels): the conv
//              histories of pfx::history_channel, each once every chain of
//              its continuation has finished (and so read the old history).
// Every item computes exactly what the separate launches compute, so the
// results are bit-identical to the decode step and chunked prefill called
// one after the other.  The chains come first so that the decode items fill
// the SMs the chains leave free and then the ones they release.
//
// The queue words live in the caller's workspace, each tagged with a
// per-call epoch in its upper half, so no word needs clearing before a call;
// the last CTA to finish returns them to zero (so a replayed CUDA graph, with
// its epoch baked in, starts afresh too).
constexpr int kDecStages = 10;  // the decode walk's ring: as the one-CTA-per-SM decode kernel
using DecSmem = dtma::TmaSmem<__nv_bfloat16, __nv_bfloat16, kDecStages, false>;
static_assert(dtma::bundle_aligned<__nv_bfloat16, __nv_bfloat16, kDecStages, false>(), "bulk-copy destinations");
static_assert(dtma::vectors_aligned<__nv_bfloat16, __nv_bfloat16, kDecStages, false>(), "float4 reads");
static_assert(dtma::kThr <= kThreads, "the decode walk's warps are a subset of the CTA");

struct MixedArgs {
  dtma::TmaArgs dec;      // the decode requests (rows 0 .. n_decode - 1)
  Tc32Args pf;            // the continuations
  pfx::PrefillArgs hist;  // the same continuations, for their conv histories
  unsigned long long* queue;     // [0]: next item, [1]: CTAs done, [2 ..]: chains done per continuation
  uint32_t epoch;
  int32_t n_chain, n_dec, n_hist, hist_blocks, hist_groups;
};

struct __align__(1024) MixedSmem {
  union {
    Smem32 pf;
    DecSmem dec;
  };
  int item;   // the CTA's next work item (broadcast)
  int ready;  // a history item's continuation is ready
};

// (epoch, count) words: count under this call's epoch, 0 under another
__device__ __forceinline__ uint32_t epoch_count(unsigned long long w, uint32_t epoch) {
  return (uint32_t)(w >> 32) == epoch ? (uint32_t)w : 0u;
}
// Word q carries this call's epoch from now on: a word of another call (or
// zero) becomes (epoch, 0) by one compare-and-swap, which at most one caller
// wins; false if the word stayed contended for the retry limit.  Counting is
// then a plain atomic add (no compare-and-swap on the hot word: contended
// swaps made the walk several times slower).
__device__ __forceinline__ bool epoch_install(unsigned long long* q, uint32_t epoch) {
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(q);
    if ((uint32_t)(old >> 32) == epoch) return true;
    if (atomicCAS(q, old, (unsigned long long)epoch << 32) == old) return true;
  }
  return false;
}
// add 1 to word q's count (its epoch installed first); the count before, or
// -1 if the epoch could not be installed
__device__ __forceinline__ long long epoch_add(unsigned long long* q, uint32_t epoch) {
  if (!epoch_install(q, epoch)) return -1;
  const unsigned long long old = atomicAdd(q, 1ull);
  return (uint32_t)(old >> 32) == epoch ? (long long)(uint32_t)old : -1;
}

// thread 0: the next work item (>= total, or -1 on a failure, ends the CTA's
// walk).  One atomic add; only when it lands on a word of another call (the
// first takes of this one) is the epoch installed and the add repeated: the
// install wipes such stray adds, and an add after it counts for this call.
__device__ __forceinline__ int take_item(const MixedArgs& m) {
  for (int tries = 0; tries < 4; ++tries) {
    const unsigned long long old = atomicAdd(m.queue, 1ull);
    if ((uint32_t)(old >> 32) == m.epoch) return (uint32_t)old > 0x7fffffffu ? 0x7fffffff : (int)(uint32_t)old;
    if (!epoch_install(m.queue, m.epoch)) break;
  }
  report(m.pf.err, GDN_DEV_ERR_TIMEOUT);
  return -1;
}

// The decode walk from item `first`: warps 0-8 as in the decode kernel (the
// producer lane taking the items), the other warps idle.  Returns, to every
// thread, the first item taken that is not a decode item.
__device__ __forceinline__ int mixed_decode(const MixedArgs& m, MixedSmem& M, const int first) {
  using namespace dtma;
  DecSmem& S = M.dec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const TmaArgs& a = m.dec;
  [[maybe_unused]] const int nreq = a.n_items / a.hk;
  auto is_dec = [&](int item) { return item >= m.n_chain && item < m.n_chain + m.n_dec; };
  if (tid == 0) init_barriers<DecSmem, kDecStages>(S);
  __syncthreads();
  volatile int* abort_flag = &S.abort;
  if (warp == kCW) {
    if (lane == 0) {
      // producer: every item goes through a bundle buffer, so that the
      // consumers follow the same sequence; an unusable slot's item and the
      // final non-decode item travel without copies
      uint32_t n = 0, vk = 0;
      bool ok = true;
      int item = first;
      for (;;) {
        const bool dec = is_dec(item);
        int r = 0, hq = 0;
        int32_t slot = -1;
        if (dec) {
          const int d = item - m.n_chain;
          r = d / a.hk;
          hq = d % a.hk;
          slot = a.slot_ids[GDN_G(r, nreq)];
        }
        if (*abort_flag) break;
        if (!dec || slot_class(slot, a.num_slots)) {
          const int bb = vk & 1;
          if (!mbar_wait(&S.bempty[bb], ((vk >> 1) & 1) ^ 1)) {
            ok = false;
            break;
          }
          S.bitem[bb] = item;
          mbar_arrive(&S.bfull[bb]);
          ++vk;
          if (!dec) break;
        } else {
          if (!(ok = produce_item<__nv_bfloat16, __nv_bfloat16, kDecStages, false>(a, S, r, hq, slot, vk, n, item)))
            break;
        }
        item = take_item(m);
      }
      if (!ok || *abort_flag) producer_drain<DecSmem, kDecStages>(a, S, vk, n);
    }
  } else if (warp < kCW) {
    uint32_t n = 0, vk = 0;
    for (;;) {
      const int bb = vk & 1;
      if (!*abort_flag && !mbar_wait(&S.bfull[bb], (vk >> 1) & 1)) *abort_flag = 1;
      named_sync(kBarCons, kCons);
      if (*abort_flag) break;
      const int item = S.bitem[bb];
      ++vk;
      if (!is_dec(item)) {
        if (tid == 0) M.item = item;
        break;
      }
      const int d = item - m.n_chain, r = d / a.hk, hq = d % a.hk;
      const int32_t slot = a.slot_ids[GDN_G(r, nreq)];
      const int cls = slot_class(slot, a.num_slots);
      if (cls) {
        consume_skipped<__nv_bfloat16>(a, r, hq, cls);
        named_sync(kBarCons, kCons);  // every consumer has read the item
        mbar_arrive(&S.bempty[bb]);
        continue;
      }
      if (!consume_bundle<__nv_bfloat16, __nv_bfloat16, kDecStages, false>(a, S, r, hq, slot, bb, n)) break;
    }
    if (*abort_flag && tid == 0) {
      report(a.err, GDN_DEV_ERR_TIMEOUT);
      M.item = -1;
    }
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_inval(&S.full[s]);
      mbar_inval(&S.empty[s]);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_inval(&S.bfull[s]);
      mbar_inval(&S.bempty[s]);
    }
  }
  const int next = M.item;
  __syncthreads();
  return next;
}

__global__ void __launch_bounds__(kThreads, 1)
    mixed_kernel(const MixedArgs m, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                 const __grid_constant__ CUtensorMap cmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  MixedSmem& M = *reinterpret_cast<MixedSmem*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int total = m.n_chain + m.n_dec + m.n_hist;
  const int hv = m.pf.hv;
  unsigned long long* const chains_done = m.queue + 2;
  if (warp == 0) umma::tmem_alloc(&M.pf.tmem_base, TM_COLS);
  if (tid == 0) M.item = take_item(m);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = M.pf.tmem_base;
  int item = M.item;
  __syncthreads();
  while (item >= 0 && item < total) {
    if (item < m.n_chain) {
      const int n = item / hv, h = item % hv;
      tc32_chain<__nv_bfloat16, false>(m.pf, qmap, omap, cmap, omap, M.pf, tmem, h, n);
      if (tid == 0) {
        __threadfence();  // this chain's reads of the old conv history are done
        epoch_add(chains_done + n, m.epoch);
        M.item = take_item(m);
      }
      __syncthreads();
      item = M.item;
    } else if (item < m.n_chain + m.n_dec) {
      item = mixed_decode(m, M, item);
    } else {
      const int k = item - m.n_chain - m.n_dec;
      const int n = k / (m.hist_groups * m.hist_blocks);
      const int grp = (k / m.hist_blocks) % m.hist_groups, blk = k % m.hist_blocks;
      if (tid == 0) {
        // every chain of continuation n has finished (bounded wait)
        bool ok = true;
        const uint64_t t0 = globaltimer_ns();
        while (epoch_count(*reinterpret_cast<volatile unsigned long long*>(chains_done + n), m.epoch) <
               (uint32_t)hv) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            report(m.pf.err, GDN_DEV_ERR_TIMEOUT);
            break;
          }
        }
        __threadfence();
        M.ready = ok;
      }
      __syncthreads();
      const int c = blk * kThreads + tid;
      if (M.ready && c < m.hist.C) pfx::history_channel<__nv_bfloat16, __nv_bfloat16>(m.hist, n, grp, c);
      __syncthreads();
      if (tid == 0) M.item = take_item(m);
      __syncthreads();
      item = M.item;
    }
  }
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, TM_COLS);
  // the last CTA out returns the queue words to zero
  if (tid == 0) {
    __threadfence();
    const long long done = epoch_add(m.queue + 1, m.epoch);
    if (done == (long long)gridDim.x - 1) {
      __threadfence();
      for (int i = 0; i < 2 + m.pf.n_seq; ++i) m.queue[i] = 0ull;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side (declared in prefill_tc.cuh)
// ---------------------------------------------------------------------------
bool prefill_tc32_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p) {
  if (d.dk != kD || d.dv != kD || d.conv_width != 4) return false;
  if (d.act_dtype != GDN_BF16 || d.conv_dtype != GDN_BF16) return false;
  if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(p.conv_w, 16)) return false;
  return true;
}

cudaError_t prefill_tc32_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                                const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                                int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                                int32_t ckpt_block, const void* qkv, const void* av, const void* bv, void* out,
                                uint32_t* dev_err, cudaStream_t s, const Tc32Epilogue* epi) {
  Tc32Args a;
  a.ssm = pool.ssm;
  a.num_slots = pool.num_slots;
  a.ck_ssm = ckpt.ssm;
  a.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  a.conv = reinterpret_cast<const __nv_bfloat16*>(pool.conv);
  a.conv_w = p.conv_w;
  a.A_log = p.A_log;
  a.dt_bias = p.dt_bias;
  a.slot_ids = slot_ids;
  a.cu_seqlens = cu_seqlens;
  a.start_pos = start_pos;
  a.n_seq = n_seq;
  a.total = total;
  a.ckpt_ids = ckpt_ids;
  a.max_ckpt = max_ckpt;
  a.ckpt_block = ckpt_block;
  a.a = reinterpret_cast<const __nv_bfloat16*>(av);
  a.b = reinterpret_cast<const __nv_bfloat16*>(bv);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.err = dev_err;
  a.hk = d.hk;
  a.hv = d.hv;
  a.C = (int32_t)channels(d);
  a.G = d.hv / d.hk;
  a.norm_w = epi ? epi->weight : nullptr;
  a.eps = epi ? epi->eps : 0.f;
  auto k = epi ? tc32_prefill_kernel<__nv_bfloat16, true> : tc32_prefill_kernel<__nv_bfloat16, false>;
  const size_t smem = sizeof(Smem32) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // qkv [total][C] in boxes of 128 channels x 67 rows; out (and z) [total][hv
  // * 128] in boxes of one V head x 64 tokens; checkpoint states [slots * hv *
  // 128 rows][128] fp32 in 128B-swizzled boxes of 32 x 128 (over the working
  // pool when there is no checkpoint pool: never written then)
  CUtensorMap qmap, omap, cmap, zmap;
  if ((e = tensor_map_2d(&qmap, qkv, total, a.C, 2, kD, kRawRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&omap, out, total, (int64_t)a.hv * kD, 2, kD, kC, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&zmap, epi ? epi->z : out, total, (int64_t)a.hv * kD, 2, kD, kC,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  const bool has_ck = a.ck_ssm != nullptr && a.ck_num_slots > 0;
  if ((e = tensor_map_2d(&cmap, has_ck ? a.ck_ssm : a.ssm, (int64_t)(has_ck ? a.ck_num_slots : a.num_slots) * a.hv * kD,
                         kD, 4, 32, kD, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  return launch_plain(k, dim3((unsigned)a.hv, (unsigned)n_seq), dim3(kThreads), smem, s, dim3(1), a, qmap, omap,
                      cmap, zmap);
}

// ---------------------------------------------------------------------------
bool mixed_fused_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p) {
  if (!prefill_tc32_supported(d, qkv, out, p) || !decode_tma_supported(d, qkv, p)) return false;
  const char* e = std::getenv("GDN_MIXED");  // read on every call: "split" for the separate launches
  return !(e && e[0] == 's');
}

size_t mixed_fused_queue_bytes(int32_t n_pre) { return sizeof(unsigned long long) * (2 + (size_t)n_pre); }

cudaError_t mixed_fused_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                               const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                               int32_t n_seq, int32_t n_decode, int64_t total, const int32_t* ckpt_ids,
                               int32_t max_ckpt, int32_t ckpt_block, const void* qkv, const void* av,
                               const void* bv, void* out, void* queue, uint32_t* dev_err, cudaStream_t s) {
  static std::atomic<uint32_t> epochs{0};
  uint32_t epoch = epochs.fetch_add(1) + 1;
  if (epoch == 0) epoch = epochs.fetch_add(1) + 1;
  const int32_t n_pre = n_seq - n_decode;
  MixedArgs m = {};
  // decode rows: the first n_decode rows of every per-token tensor
  m.dec.ssm = pool.ssm;
  m.dec.conv = pool.conv;
  m.dec.num_slots = pool.num_slots;
  m.dec.conv_w = p.conv_w;
  m.dec.A_log = p.A_log;
  m.dec.dt_bias = p.dt_bias;
  m.dec.slot_ids = slot_ids;
  m.dec.qkv = qkv;
  m.dec.a = av;
  m.dec.b = bv;
  m.dec.out = out;
  m.dec.err = dev_err;
  m.dec.hk = d.hk;
  m.dec.hv = d.hv;
  m.dec.dv = d.dv;
  m.dec.C = (int32_t)channels(d);
  m.dec.G = d.hv / d.hk;
  m.dec.n_items = n_decode * d.hk;
  // continuations: sequences n_decode .., rows at their absolute offsets
  const int32_t* pre_ids = slot_ids + n_decode;
  const int32_t* pre_cu = cu_seqlens + n_decode;
  const int64_t* pre_sp = start_pos + n_decode;
  const int32_t* pre_ck = max_ckpt > 0 ? ckpt_ids + (size_t)n_decode * max_ckpt : nullptr;
  Tc32Args& a = m.pf;
  a.ssm = pool.ssm;
  a.num_slots = pool.num_slots;
  a.ck_ssm = ckpt.ssm;
  a.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  a.conv = reinterpret_cast<const __nv_bfloat16*>(pool.conv);
  a.conv_w = p.conv_w;
  a.A_log = p.A_log;
  a.dt_bias = p.dt_bias;
  a.slot_ids = pre_ids;
  a.cu_seqlens = pre_cu;
  a.start_pos = pre_sp;
  a.n_seq = n_pre;
  a.total = total;
  a.ckpt_ids = pre_ck;
  a.max_ckpt = max_ckpt;
  a.ckpt_block = ckpt_block;
  a.a = reinterpret_cast<const __nv_bfloat16*>(av);
  a.b = reinterpret_cast<const __nv_bfloat16*>(bv);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.err = dev_err;
  a.hk = d.hk;
  a.hv = d.hv;
  a.C = (int32_t)channels(d);
  a.G = d.hv / d.hk;
  a.norm_w = nullptr;
  a.eps = 0.f;
  pfx::PrefillArgs& hq = m.hist;
  hq.ssm = pool.ssm;
  hq.conv = pool.conv;
  hq.num_slots = pool.num_slots;
  hq.ck_ssm = ckpt.ssm;
  hq.ck_conv = ckpt.conv;
  hq.ck_num_slots = a.ck_num_slots;
  hq.conv_w = p.conv_w;
  hq.A_log = p.A_log;
  hq.dt_bias = p.dt_bias;
  hq.slot_ids = pre_ids;
  hq.cu_seqlens = pre_cu;
  hq.start_pos = pre_sp;
  hq.n_seq = n_pre;
  hq.total = total;
  hq.ckpt_ids = pre_ck;
  hq.max_ckpt = max_ckpt;
  hq.ckpt_block = ckpt_block;
  hq.qkv = qkv;
  hq.a = av;
  hq.b = bv;
  hq.out = out;
  hq.err = dev_err;
  hq.hk = d.hk;
  hq.hv = d.hv;
  hq.dk = d.dk;
  hq.dv = d.dv;
  hq.W = d.conv_width;
  hq.C = (int32_t)channels(d);
  hq.G = d.hv / d.hk;
  m.queue = reinterpret_cast<unsigned long long*>(queue);
  m.epoch = epoch;
  m.n_chain = n_pre * d.hv;
  m.n_dec = n_decode * d.hk;
  m.hist_blocks = (hq.C + kThreads - 1) / kThreads;
  m.hist_groups = max_ckpt > pfx::kCkGroup ? (max_ckpt + pfx::kCkGroup - 1) / pfx::kCkGroup : 1;
  m.n_hist = n_pre * m.hist_groups * m.hist_blocks;
  const size_t smem = sizeof(MixedSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(mixed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap qmap, omap, cmap;
  if ((e = tensor_map_2d(&qmap, qkv, total, a.C, 2, kD, kRawRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&omap, out, total, (int64_t)a.hv * kD, 2, kD, kC, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  const bool has_ck = a.ck_ssm != nullptr && a.ck_num_slots > 0;
  if ((e = tensor_map_2d(&cmap, has_ck ? a.ck_ssm : a.ssm, (int64_t)(has_ck ? a.ck_num_slots : a.num_slots) * a.hv * kD,
                         kD, 4, 32, kD, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  const int64_t items = (int64_t)m.n_chain + m.n_dec + m.n_hist;
  const int grid = (int)(items < sm_count() ? items : sm_count());
  return launch_plain(mixed_kernel, dim3((unsigned)grid), dim3(kThreads), smem, s, dim3(1), m, qmap, omap, cmap);
}

}  // namespace gdn
