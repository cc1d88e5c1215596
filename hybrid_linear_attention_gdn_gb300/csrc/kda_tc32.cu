// KDA prefill in the chunked form on the 5th-generation tensor cores, the
// state products in tf32 (dk = dv = 128, conv width 4, bf16 activations and
// conv history).
//
// The per-key-channel gated delta rule (Kimi Delta Attention, Kimi Linear
// 2025): St <- St diag(alpha_t) + beta_t (v_t - St diag(alpha_t) k_t) k_t^T,
// o_t = St q_t, with log alpha_t = -exp(A_log) softplus(a_t + dt_bias) per
// key channel.  Same contract as the other KDA prefills (block-aligned
// checkpoints of state, the final state in the working slot; the conv
// histories come from the prefill's history kernel) and the chunk form of the
// Gated DeltaNet paper (chunkwise WY/UT) with the decay kept per channel, in
// chunks of 64 tokens aligned to absolute positions.  With lb_t the
// cumulative log decay from the chunk start (per channel):
//   K~_t = k^_t (.) e^{lb_t},  Q~_t = q^_t (.) e^{lb_t},  K-_t = k^_t (.) e^{lb_63 - lb_t},
//   A'[t][j] = sum_c k^_tc k^_jc e^{lb_tc - lb_jc}   (t > j),
//   M[t][j]  = sum_c q^_tc k^_jc e^{lb_tc - lb_jc}   (t >= j),
//   T = (I + diag(beta) A')^-1 diag(beta),
//   Delta = (V - S K~^T) T^T,  O = S Q~^T + Delta M^T,  S <- S diag(e^{lb_63}) + Delta K-
// (S is the dv x dk state, V and Delta dv x 64).
//
// A' and M cannot be one product of decayed operands: e^{lb_t - lb_j} split
// as e^{lb_t} e^{-lb_j} overflows.  They are taken in 8-token blocks with a
// reference token R between the two blocks of a pair, so that every factor
// is a product of alphas over a token range (at most 1):
//   off the diagonal (t in block I, j in block J < I, a reference block R
//     with J < R <= I): e^{lb_t - lb_j} is the row factor e^{lb_t - lb_b(R)}
//     = fl8_t e^{lb_b(I) - lb_b(R)} (fl8 from the block's first token) times
//     the column factor e^{lb_b(R) - lb_j} = e^{lb_b(R) - lb_e(J)} fr8_j (fr8
//     to the block's last token; b(), e() a block's first and last token).
//     The 28 block pairs fall into three levels of a binary split, each one
//     product for all its pairs:
//     R = block 4 (rows of blocks 4..7 against columns of 0..3), R = 2 and 6
//     (rows 2, 3 x columns 0, 1 and rows 6, 7 x columns 4, 5), R = the row
//     block itself (1 x 0, 3 x 2, 5 x 4, 7 x 6).  Levels 3 and 2 make one
//     tcgen05 product (M = 128: their k and q rows; N = 64), level 1 another
//     (N = 32), in fp16 (the 10-bit mantissa the tf32 products keep; every
//     operand lies in [-1, 1]);
//   on the eight 8 x 8 diagonal blocks: fp32 running products of alpha down
//     each row, on the CUDA cores.
// Every within-block factor is a running product of alphas (no differences
// of large cumulative sums), and the block factors exponentials of sums of
// block totals.
//
// One CTA per (V head, sequence), 512 threads, walks the sequence's chunks in
// order; the fp32 state S lives in TMEM for the whole sequence.  Per chunk:
//   gates      thread (channel pair, 8-token block): log alpha, alpha, the
//              8-block totals, from the chunk's gate logits (one TMA box,
//              loaded under the previous chunk's assembly and solve, with
//              its own barrier: the gates do not wait for the raw rows)
//   features   the 67 raw rows of the head's q, k and v channels arrive by
//              three TMA boxes (issued after the previous chunk's solve,
//              landing under the gates); conv1d + SiLU down the chunk; q and
//              k rows (fp32) into shared memory, V^T (tf32) into TMEM, and
//              each token's sums of squares over the warp's channels
//   norms      rk_t = 1/|y_k,t|, rq_t = dk^-1/2 / |y_q,t| (with the eps) from
//              those sums
//   diagonal   the 8 x 8 diagonal blocks of A' and M
//   transform  thread (channel pair, 8-token block): fl8, fr8 by running
//              products; the fp16 operands of the off-diagonal products
//   off-diag   A' and M below the diagonal blocks (two tcgen05 products),
//              issued as soon as their operands are written; the tf32
//              operand tiles [K~;Q~] and K-^T are written while they run
//   S [K~;Q~]^T  (tcgen05, A operand the state in TMEM) issued before the
//              solve, runs under it
//   solve      X = (I + diag(beta) A')^-1 as in the GDN chain; T1 = X
//              diag(beta) and T2 = -T1
//   state      Delta = V^T T1^T + E T2^T (tcgen05), S <- S diag(e^{lb_63})
//              by the threads, then S += Delta K- and O2 = Delta M^T
//   output     O = S Q~^T + O2, one TMA tensor store (row stores for chunks
//              cut by a sequence boundary); checkpoints as in the GDN chain.
#include "gdn_common.cuh"
#include "kda_tc32.cuh"
#include "tma.cuh"
#include "umma.cuh"

#include <cuda_fp16.h>

namespace gdn {
namespace {

#include "tc32_common.cuh"

constexpr int kYS = kD + 4;   // row stride (floats) of the fp32 feature and alpha rows

// TMEM columns (fp32; lanes are dv rows)
constexpr uint32_t TM_S = 0;     // S [dv][dk]
constexpr uint32_t TM_DX = 128;  // off-diagonal levels 3 and 2 [their 128 rows][64]
constexpr uint32_t TM_DY = 192;  // off-diagonal level 1 [its 64 rows (+ 64 unused)][32]
constexpr uint32_t TM_E = 256;   // S K~^T [dv][64]
constexpr uint32_t TM_O1 = 320;  // S Q~^T [dv][64]
constexpr uint32_t TM_DL = 384;  // Delta [dv][64]
constexpr uint32_t TM_V = 448;   // V^T [dv][64] (operand); then O2:
constexpr uint32_t TM_O2 = 448;  //   Delta M^T [dv][64] (V read by then)
constexpr uint32_t TM_COLS = 512;

struct KdaTcArgs {
  float* ssm;
  int32_t num_slots;
  float* ck_ssm;
  int32_t ck_num_slots;
  const __nv_bfloat16* conv;
  const float* conv_w;
  const float* A_log;    // [hv]
  const float* dt_bias;  // [hv][dk]
  const int32_t* slot_ids;
  const int32_t* cu_seqlens;
  const int64_t* start_pos;
  int32_t n_seq;
  int64_t total;
  const int32_t* ckpt_ids;
  int32_t max_ckpt;
  int32_t ckpt_block;
  const __nv_bfloat16* b;  // beta logits [total][hv]
  __nv_bfloat16* out;
  uint32_t* err;
  int32_t hk, hv, C, G;
};

// Shared memory.  The tf32 operand tiles are in the tensor core's 128-byte
// swizzled K-major layout (f32_off); the regions T and U are reused by the
// phases of a chunk in turn.
struct __align__(1024) KSmem {
  uint8_t kq[4 * 128 * 128];  // [K~ ; Q~]: rows 0..63 K~, 64..127 Q~ (x dk)
  uint8_t kt[2 * 128 * 128];  // K-^T [dk][64 tokens]
  union {                     // region T
    struct {
      uint8_t tm[2 * 64 * 128];  // T1 [i][j]
      uint8_t t2[2 * 64 * 128];  // T2 = -T1; after its product, the output staging tile
      uint8_t mq[2 * 64 * 128];  // M [i][j]
    } t;
    struct {
      float al[kC][kYS];         // alpha per token and channel
    } g;
    uint8_t by[2 * 32 * 128];    // level-1 columns (fp16 operand, over al)
  } rt;
  union {                     // region U
    struct {
      __nv_bfloat16 raw[3][kRawRows][kD];  // staged inputs: q, k, v parts
      __nv_bfloat16 ga[kC][kD];            // the chunk's gate logits
    } in;
    struct {
      float yk[kC][kYS];  // conv + SiLU of the k channels, unnormalised
      float yq[kC][kYS];
    } y;
    struct {
      uint8_t ax[2 * 128 * 128];  // levels 3 and 2: rows (fp16 operand)
      uint8_t bx[2 * 64 * 128];   //   and their columns
      uint8_t ay[2 * 64 * 128];   // level 1: rows (64 of the product's 128; it reads 8 KB past)
    } ops;
    struct {
      float A[kC * kAX];
      float X[kC * kAX];
      float Y[2048];
      float L0[8][3][64];
    } sv;  // the solve's scratch
  } ru;
  float beta[kC];
  float G8[8][kD];    // per 8-token block and channel: the sum of its log decays
  float g8f[8][kD];   // the log decay of the block's first token
  float alast[kD];    // e^{lb_63} per channel
  float rk[kC];       // 1 / sqrt(|y_k|^2 + eps)
  float rq[kC];       // dk^-1/2 / sqrt(|y_q|^2 + eps)
  float nrm[2][2][kC];  // sums of squares over half the channels: [k, q][half][token]
  float dgA[kC][8];   // diagonal blocks: beta_t A'[t][j] (j < t, local j), and
  float dgM[kC][8];   //   M[t][j] (j <= t)
  float ones[kC];
  uint64_t ld_bar, ga_bar;  // the raw rows; the gate logits (they land first: the gates start on them)
  uint64_t mma_bar, eo_bar, od_bar;  // od_bar: the two off-diagonal products (two issuers)
  uint32_t tmem_base;
};

static_assert(sizeof(KSmem) + 1024 <= 232448, "one CTA's shared memory (with the alignment slack)");
// the level-1 product reads rows 64..127 of its second column block, 8 KB
// past the end of ay: still inside the CTA's shared memory
static_assert(offsetof(KSmem, ru) + 32768 + 16384 + 8192 + 16384 <= sizeof(KSmem),
              "level-1 rows read past ay (its second column block starts 8 KB in and spans 16 KB)");

__device__ __forceinline__ bool seq_ok(const KdaTcArgs& a, int n, int64_t& t0, int64_t& len, int64_t& p0) {
  const auto cu = GDN_GV(a.cu_seqlens, a.n_seq + 1);
  t0 = cu[n];
  len = (int64_t)cu[n + 1] - t0;
  p0 = GDN_GV(a.start_pos, a.n_seq)[n];
  return !(t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0);
}

// ---- diagonal 8 x 8 blocks --------------------------------------------------------
// Warp (block B, row group RG), lane = channel group cg (channels 4 cg ..):
// rows {0, 7, 1, 6} or {2, 5, 3, 4} of the block (9 (t, j) pairs each per
// pair of rows).  Per row t, walking j down from t: p = prod_{j<m<=t} alpha_m
// (running product), M(t, j) += q_t k_j p, A'(t, j) += k_t k_j p over the
// lane's 4 channels; then a reduce-scatter over the 32 lanes leaves lane l
// with value l, which goes (norms and beta applied) to dgA / dgM.  Value
// layout per row t at offset o: M(t, 0..t), then A'(t, 0..t-1).
__host__ __device__ constexpr int diag_row(int rg, int r) {
  return rg ? (r == 0 ? 2 : r == 1 ? 5 : r == 2 ? 3 : 4) : (r == 0 ? 0 : r == 1 ? 7 : r == 2 ? 1 : 6);
}
__host__ __device__ constexpr int diag_off(int rg, int r) {
  int o = 0;
  for (int i = 0; i < r; ++i) o += 2 * diag_row(rg, i) + 1;
  return o;
}
static_assert(diag_off(0, 4) == 32 && diag_off(1, 4) == 32, "32 values per lane");

// a (.) b on packed fp32 pairs
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return join4(mul2(lo2(a), lo2(b)), mul2(hi2(a), hi2(b)));
}
// acc + a . b
__device__ __forceinline__ float dot4acc(float4 a, float4 b, float acc) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}

template <int RG>
__device__ __forceinline__ void diag_block(KSmem& S, const int B) {
  const int lane = threadIdx.x & 31;
  const auto yk = GDN_SV(&S.ru.y.yk[0][0], kC * kYS), yq = GDN_SV(&S.ru.y.yq[0][0], kC * kYS);
  const auto al = GDN_SV(&S.rt.g.al[0][0], kC * kYS);
  const int c4 = 4 * lane;
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  float4 p[4], kr[4], qr[4];
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    const float4 kj = vec_at<const float4>(yk, (8 * B + j) * kYS + c4);
    const float4 aj = j < 7 ? vec_at<const float4>(al, (8 * B + j + 1) * kYS + c4) : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = diag_row(RG, r), o = diag_off(RG, r);
      if (t == j) {
        p[r] = make_float4(1.f, 1.f, 1.f, 1.f);
        kr[r] = kj;
        qr[r] = vec_at<const float4>(yq, (8 * B + t) * kYS + c4);
      } else if (t > j) {
        p[r] = mul4(p[r], aj);
      }
      if (t >= j) {
        const float4 kp = t == j ? kj : mul4(kj, p[r]);
        acc[o + j] = dot4acc(qr[r], kp, acc[o + j]);
        if (t > j) acc[o + t + 1 + j] = dot4acc(kr[r], kp, acc[o + t + 1 + j]);
      }
    }
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = lane & s;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? acc[i] : acc[i + s];
      const float keep = up ? acc[i + s] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  // lane -> (row, column, kind)
  int r = 0;
#pragma unroll
  for (int i = 1; i < 4; ++i)
    if (lane >= diag_off(RG, i)) r = i;
  int t = diag_row(RG, 0), o = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (r == i) {
      t = diag_row(RG, i);
      o = diag_off(RG, i);
    }
  const int m = lane - o, T = 8 * B + t;
  if (m <= t)
    S.dgM[GDN_S(T, kC)][GDN_S(m, 8)] = acc[0] * S.rq[T] * S.rk[8 * B + m];
  else
    S.dgA[GDN_S(T, kC)][GDN_S(m - t - 1, 8)] = acc[0] * S.rk[T] * S.rk[8 * B + (m - t - 1)] * S.beta[T];
}

// ---- one chain ---------------------------------------------------------------
// V head h of sequence n, by all 512 threads, which hold the 512 TMEM columns
// from `tmem` on.  Thread 0 issues the TMA copies and the state-side products
// (a lane of warp 10 the one that runs under the solve); every wait is
// bounded (1 s).
__device__ __forceinline__ void kda_chain(const KdaTcArgs& a, const CUtensorMap& qmap, const CUtensorMap& amap,
                                          const CUtensorMap& omap, const CUtensorMap& cmap, KSmem& S,
                                          const uint32_t tmem, const int h, const int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = h / a.G;
  int64_t t0, len, p0;
  if (!seq_ok(a, n, t0, len, p0)) {
    if (h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const auto out = GDN_GV(a.out, a.total * a.hv * kD);
  const auto gate_b = GDN_GV(a.b, a.total * a.hv);
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
    mbar_init(&S.ga_bar, 1);
    mbar_init(&S.mma_bar, 1);
    mbar_init(&S.od_bar, 2);
    mbar_init(&S.eo_bar, 1);
    fence_mbar_init();
  }
  if (tid < kC) S.ones[tid] = 1.f;
  __syncthreads();
  const int lrow = 32 * (warp & 3) + lane;  // TMEM lane of this thread (dv row)
  const int qq = warp >> 2;                 // which column quarter this warp handles
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

  constexpr uint32_t ID_N64 = umma::idesc_tf32(128, 64, false, false);
  constexpr uint32_t ID_N128 = umma::idesc_tf32(128, 128, false, false);
  static_assert(4 * 16384 <= sizeof(KSmem::kq) && 2 * 16384 <= sizeof(KSmem::kt), "operand tiles");
  static_assert(sizeof(KSmem::rt) == 3 * 16384 && kC * kYS * 4 <= 3 * 16384,
                "region T holds T1, T2, M or alpha (then the level-1 columns)");
  static_assert(2 * kC * kYS * 4 <= sizeof(KSmem::ru) && 2 * kC * kAX * 4 + (2048 + 8 * 3 * 64) * 4 <= sizeof(KSmem::ru) &&
                    4 * 16384 <= sizeof(KSmem::ru),
                "region U holds the feature rows, the off-diagonal operands or the solve's scratch");
  static_assert(TM_DX == TM_S + 128 && TM_DY == TM_DX + 64 && TM_E >= TM_DY + 32 && TM_O1 == TM_E + 64 &&
                    TM_DL == TM_O1 + 64 && TM_V == TM_DL + 64 && TM_V + 64 <= TM_COLS && TM_O2 == TM_V,
                "TMEM regions");

  // feature channels of this thread: the q/k channel pair (2 cp, 2 cp + 1)
  // (k for tid % 128 < 64, else q) for tokens 16 qq .., and v channel lrow
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
  // gate channels of this thread (gates and transform: channels 2 gp, 2 gp + 1
  // of the 8-token block gb)
  const int gp = tid & 63, gb = tid >> 6;
  const float eA = expf(GDN_GV(a.A_log, a.hv)[h]);
  const float2 dtb = vec_at<const float2>(GDN_GV(a.dt_bias, (long long)a.hv * kD), (size_t)h * kD + 2 * gp);
  const int part_x[3] = {hq * kD, (a.hk + hq) * kD, 2 * a.hk * kD + h * kD};

  // checkpoint slot at the end of chunk c (-1: none), as in the GDN chain
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
  constexpr uint32_t kRawBytes = 3u * kRawRows * kD * 2u, kGaBytes = (uint32_t)kC * kD * 2u;
  // warp 0: chunk c's gate logits (lane 3, on ga_bar) and raw rows (lanes
  // 0..2: the q, k and v boxes at once, on ld_bar) into region U, each call
  // with its barrier's byte count.  The gate-logit box lies past the solve's
  // scratch, so it goes first, as soon as the previous chunk's off-diagonal
  // products have read their operands.
  auto issue_ga = [&](int c) {
    const int64_t P = (p0 / kC + c) * kC;
    const int32_t row = (int32_t)(t0 + (P - p0));  // packed row of the chunk's first token (may be < 0)
    if (lane == 3) {
      mbar_arrive_expect_tx(&S.ga_bar, kGaBytes);
      // 128 channels of V head h, 64 rows (rows outside: zeros)
      if (GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD) && GDN_SBYTES(&S.ru.in.ga[0][0], kC * kD * 2, S))
        tma_load_2d(&S.ru.in.ga[0][0], &amap, h * kD, row, &S.ga_bar);
    }
  };
  auto issue_raw = [&](int c) {
    const int64_t P = (p0 / kC + c) * kC;
    const int32_t row0 = (int32_t)(t0 + (P - 3 - p0));  // packed row of raw row 0 (may be < 0)
    if (lane == 0) mbar_arrive_expect_tx(&S.ld_bar, kRawBytes);
    __syncwarp();  // the phase's byte count before any of its copies
    if (lane < 3) {  // a box of 128 channels of the q, k or v part, 67 rows (rows outside: zeros)
      const int x = lane == 0 ? hq * kD : lane == 1 ? (a.hk + hq) * kD : 2 * a.hk * kD + h * kD;
      if (GDN_SPAN_G(x, kD, a.C) && GDN_SBYTES(&S.ru.in.raw[lane][0][0], kRawRows * kD * 2, S))
        tma_load_2d(&S.ru.in.raw[lane][0][0], &qmap, x, row0, &S.ld_bar);
    }
  };
  static_assert(offsetof(decltype(KSmem::ru), in.ga) >= offsetof(decltype(KSmem::ru), sv.L0) + sizeof(KSmem::ru.sv.L0),
                "the gate-logit box lies past the solve's scratch");
  // raw bits of the beta logit of chunk c's token tid (threads 0..63, 0 for
  // the other threads and outside the sequence).  An asm load, so that it is
  // issued where it stands (at the chunk start) and its latency runs under
  // the gates, not where its value is first used.
  auto load_beta = [&](int c) -> uint16_t {
    const int64_t pos = (p0 / kC + c) * kC + tid;
    uint16_t v = 0;
    if (tid < kC && pos >= p0 && pos < p1) {
      const __nv_bfloat16* src = gate_b.at((long long)(t0 + pos - p0) * a.hv + h);
      asm volatile("ld.global.nc.b16 %0, [%1];\n" : "=h"(v) : "l"(src));
    }
    return v;
  };

  // initial state rows into TMEM
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
  int ld_issued = 0, ld_done = 0, ga_issued = 0, ga_done = 0;
  if (warp == 0) {
    issue_ga(0);
    issue_raw(0);
  }
  ld_issued = ga_issued = 1;

  bool bad = false;
  uint32_t mph = 0;
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

  bool eo_pending = false, od_pending = false;
  int c = 0;
  for (; c < nch; ++c) {
    const int64_t P = (p0 / kC + c) * kC;
    const bool full = P >= p0 && P + kC <= p1;
    const int tlo = (int)(p0 > P ? (p0 - P < kC ? p0 - P : kC) : 0);
    const int thi = (int)(p1 > P ? (p1 - P < kC ? p1 - P : kC) : 0);
    const uint16_t bl = load_beta(c);
    // the previous chunk's tensor stores have read kq (checkpoint staging)
    // and t2 (output staging)
    if (tid == 0) bulk_wait_read();
    // the gate logits (issued under the previous chunk's assembly) have
    // landed; the raw rows (issued after its solve) are awaited after the gates
    if (!wait_all(&S.ga_bar, c & 1)) break;
    ga_done = c + 1;
    // ---- gates: log alpha, alpha, 8-block totals (thread: channels 2 gp, 2 gp + 1
    //      of the 8-token block gb) ---------------------------------------------
    {
      const auto ga = GDN_SV(reinterpret_cast<const __nv_bfloat162*>(&S.ru.in.ga[0][0]), kC * kD / 2);
      const auto al = GDN_SV(&S.rt.g.al[0][0], kC * kYS);
      float2 G = make_float2(0.f, 0.f), f = G;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int tt = 8 * gb + t;
        const bool valid = (unsigned)(tt - tlo) < (unsigned)(thi - tlo);
        const float2 x = __bfloat1622float2(ga[tt * (kD / 2) + gp]);
        const float x0 = x.x + dtb.x, x1 = x.y + dtb.y;
        const float s0 = x0 > 20.f ? x0 : __logf(1.f + __expf(x0)), s1 = x1 > 20.f ? x1 : __logf(1.f + __expf(x1));
        const float g0 = valid ? floor_log_decay(-eA * s0) : 0.f, g1 = valid ? floor_log_decay(-eA * s1) : 0.f;
        vec_at<float2>(al, tt * kYS + 2 * gp) = make_float2(__expf(g0), __expf(g1));
        G.x += g0;
        G.y += g1;
        if (t == 0) f = make_float2(g0, g1);
      }
      vec_at<float2>(&S.G8[GDN_S(gb, 8)][0], 2 * gp) = G;
      vec_at<float2>(&S.g8f[GDN_S(gb, 8)][0], 2 * gp) = f;
    }
    if (tid < kC)
      S.beta[tid] =
          (unsigned)(tid - tlo) < (unsigned)(thi - tlo) ? sigmoid_f(__bfloat162float(__ushort_as_bfloat16(bl))) : 0.f;

    // each thread's own wait (the copies' writes are visible to it after
    // it); an expired wait is acted on at the barrier after the features
    if (mbar_wait(&S.ld_bar, c & 1))
      ld_done = c + 1;
    else
      bad = true;
    // the up to 3 rows just before the sequence start come from the conv history
    if (P - 3 < p0) {
      const int64_t lo = (P - 3 > p0 - 3) ? P - 3 : p0 - 3;
      const int64_t hi = (P + kC < p0) ? P + kC : p0;
      const auto hist = GDN_GV(a.conv, (long long)a.num_slots * 3 * a.C) + (size_t)slot * 3 * a.C;
      for (int64_t pos = lo; pos < hi; ++pos) {
        const int r = GDN_S((int)(pos - (P - 3)), kRawRows);
        for (int e = tid; e < 3 * kD; e += kThreads) {
          const int q = e / kD, ch = e % kD;
          S.ru.in.raw[q][r][ch] = hist[(size_t)(3 - (p0 - pos)) * a.C + part_x[q] + ch];
        }
      }
      __syncthreads();
    }

    // ---- features: conv1d + SiLU, down the chunk ---------------------------
    float2 y[16];
    float vv[16];
    {
      const int tk = 16 * qq;
      {
        const auto xs = GDN_SV(reinterpret_cast<const __nv_bfloat162*>(&S.ru.in.raw[isq ? 0 : 1][0][0]),
                               kRawRows * kD / 2) +
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
          y[t] = valid ? make_float2(silu_tanh(acc.x), silu_tanh(acc.y)) : make_float2(0.f, 0.f);
        }
      }
      // the tokens' sums of squares over the warp's 64 channels: a
      // reduce-scatter leaves lanes 2 t and 2 t + 1 with token t's
      {
        float ss[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) ss[t] = fmaf(y[t].x, y[t].x, y[t].y * y[t].y);
#pragma unroll
        for (int s2 = 16; s2 >= 2; s2 >>= 1) {
          const bool up = lane & s2;
#pragma unroll
          for (int i = 0; i < s2 / 2; ++i) {
            const float send = up ? ss[i] : ss[i + s2 / 2];
            const float keep = up ? ss[i + s2 / 2] : ss[i];
            ss[i] = keep + __shfl_xor_sync(0xffffffffu, send, s2);
          }
        }
        ss[0] += __shfl_xor_sync(0xffffffffu, ss[0], 1);
        if (!(lane & 1)) S.nrm[isq][warp & 1][GDN_S(tk + (lane >> 1), kC)] = ss[0];
      }
      {
        const auto xv = GDN_SV(&S.ru.in.raw[2][0][0], kRawRows * kD) + (tk * kD + lrow);
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
    }
    // the raw rows and gate logits are read: the feature rows take region U
    if (__syncthreads_or(bad)) break;
    {
      const int tk = 16 * qq;
      const auto yd = GDN_SV(isq ? &S.ru.y.yq[0][0] : &S.ru.y.yk[0][0], kC * kYS);
#pragma unroll
      for (int t = 0; t < 16; ++t) vec_at<float2>(yd, (tk + t) * kYS + 2 * cp) = y[t];
      umma::tmem_st16(tlane + TM_V + tk, vv);
      // the norms: rk_t = 1 / sqrt(|y_k,t|^2 + eps), rq_t = dk^-1/2 / sqrt(|y_q,t|^2 + eps)
      if (tid < 2 * kC) {
        const int t = tid & (kC - 1), iq = tid >> 6;
        const float r = rsqrtf(S.nrm[iq][0][t] + S.nrm[iq][1][t] + kNormEps);
        if (iq) S.rq[t] = r * rsqrtf((float)kD); else S.rk[t] = r;
      }
    }
    __syncthreads();
    // ---- the 8 x 8 diagonal blocks of A' and M --------------------------------
    if (warp & 1)
      diag_block<1>(S, warp >> 1);
    else
      diag_block<0>(S, warp >> 1);

    // ---- A' and M below the diagonal blocks: levels 3 and 2 (rows: ax, columns:
    //      bx; N = 64) and level 1 (ay, by; N = 32) on the tensor core, issued
    //      by two threads (one product each: a thread issuing products waits
    //      for the tensor core to take each one) once the transform has
    //      written their operands -------------------------------------------
    auto issue_offdiag = [&]() {
      if (tid == 0) {
        umma::fence_after();
        constexpr uint32_t ID_X = umma::idesc_f16(128, 64, false, false);
        const uint64_t dax = umma::desc(smem_addr(S.ru.ops.ax), 16, 1024);
        const uint64_t dbx = umma::desc(smem_addr(S.ru.ops.bx), 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s)  // K = 16 channels a step, 64-channel blocks
          umma::mma_bf16(tmem + TM_DX, umma::adv(dax, (s >> 2) * 16384 + (s & 3) * 32),
                         umma::adv(dbx, (s >> 2) * 8192 + (s & 3) * 32), ID_X, s > 0);
        umma::commit(&S.od_bar);
      } else if (tid == 32) {
        umma::fence_after();
        constexpr uint32_t ID_Y = umma::idesc_f16(128, 32, false, false);
        const uint64_t day = umma::desc(smem_addr(S.ru.ops.ay), 16, 1024);
        const uint64_t dby = umma::desc(smem_addr(S.rt.by), 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma::mma_bf16(tmem + TM_DY, umma::adv(day, (s >> 2) * 8192 + (s & 3) * 32),
                         umma::adv(dby, (s >> 2) * 4096 + (s & 3) * 32), ID_Y, s > 0);
        umma::commit(&S.od_bar);
      }
    };
    // ---- transform (thread: channels 2 gp, 2 gp + 1 of the 8-token block gb) --
    {
      const auto al = GDN_SV(&S.rt.g.al[0][0], kC * kYS);
      const auto yk = GDN_SV(&S.ru.y.yk[0][0], kC * kYS), yq = GDN_SV(&S.ru.y.yq[0][0], kC * kYS);
      float2 a8[8], k8[8], q8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int tt = 8 * gb + t;
        a8[t] = vec_at<const float2>(al, tt * kYS + 2 * gp);
        k8[t] = vec_at<const float2>(yk, tt * kYS + 2 * gp);
        q8[t] = vec_at<const float2>(yq, tt * kYS + 2 * gp);
      }
      // block factors (per channel, from the 8-block totals G and first-token
      // log decays f): e^{lb} at this block's first token (Eb) and e^{lb_63 -
      // lb} at its last (Ee); the off-diagonal row factors e^{lb_b(gb) -
      // lb_b(R)} (F2 for R = 2, 6; F1 for R = 4) and column factors e^{lb_b(R)
      // - lb_e(gb)} (E3 for R = gb + 1; E2 for R = 2, 6; EY for R = 4)
      float2 G[8];
#pragma unroll
      for (int K = 0; K < 8; ++K) G[K] = vec_at<const float2>(&S.G8[K][0], 2 * gp);
      auto gf = [&](int K) { return vec_at<const float2>(&S.g8f[GDN_S(K, 8)][0], 2 * gp); };
      const float2 fb = gf(gb), f4 = gf(4), fR = gf(gb < 4 ? 2 : 6);
      const float2 fn = gf(gb < 7 ? gb + 1 : 7), fp = gf(gb > 0 ? gb - 1 : 0);
      float2 pre = make_float2(0.f, 0.f), post = pre, tot = pre, f1 = pre, e2 = pre, ey = pre, f2 = pre;
#pragma unroll
      for (int K = 0; K < 8; ++K) {
        tot = make_float2(tot.x + G[K].x, tot.y + G[K].y);
        if (K < gb) pre = make_float2(pre.x + G[K].x, pre.y + G[K].y);
        if (K > gb) post = make_float2(post.x + G[K].x, post.y + G[K].y);
        if (K >= 4 && K < gb) f1 = make_float2(f1.x + G[K].x, f1.y + G[K].y);
        if (K > gb && K < (gb < 4 ? 2 : 6)) e2 = make_float2(e2.x + G[K].x, e2.y + G[K].y);
        if (K > gb && K < 4) ey = make_float2(ey.x + G[K].x, ey.y + G[K].y);
        if (K + 1 == gb) f2 = make_float2(G[K].x - fp.x, G[K].y - fp.y);
      }
      const float2 Eb = make_float2(__expf(pre.x + fb.x), __expf(pre.y + fb.y));
      const float2 Ee = make_float2(__expf(post.x), __expf(post.y));
      if (gb == 0) vec_at<float2>(S.alast, 2 * gp) = make_float2(__expf(tot.x), __expf(tot.y));
      const float2 F1 = make_float2(__expf(f1.x - f4.x + fb.x), __expf(f1.y - f4.y + fb.y));
      const float2 F2 = (gb & 1) ? make_float2(__expf(f2.x + fb.x), __expf(f2.y + fb.y)) : make_float2(1.f, 1.f);
      const float2 E3 = make_float2(__expf(fn.x), __expf(fn.y));
      const float2 E2 = make_float2(__expf(e2.x + fR.x), __expf(e2.y + fR.y));
      const float2 EY = make_float2(__expf(ey.x + f4.x), __expf(ey.y + f4.y));
      float rk8v[8], rq8v[8];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float4 r4 = *reinterpret_cast<const float4*>(&S.rk[8 * gb + 4 * i]);
        const float4 s4 = *reinterpret_cast<const float4*>(&S.rq[8 * gb + 4 * i]);
        rk8v[4 * i] = r4.x; rk8v[4 * i + 1] = r4.y; rk8v[4 * i + 2] = r4.z; rk8v[4 * i + 3] = r4.w;
        rq8v[4 * i] = s4.x; rq8v[4 * i + 1] = s4.y; rq8v[4 * i + 2] = s4.z; rq8v[4 * i + 3] = s4.w;
      }
      // alpha, the feature rows and the diagonal blocks are read: the
      // operands take regions T and U
      __syncthreads();
      // fl8_t = prod of alpha from the block's first token to t, fr8_t from t
      // to its last (exclusive of the first and of t)
      float2 fl[8], fr[8];
      fl[0] = make_float2(1.f, 1.f);
#pragma unroll
      for (int t = 1; t < 8; ++t) fl[t] = make_float2(fl[t - 1].x * a8[t].x, fl[t - 1].y * a8[t].y);
      fr[7] = make_float2(1.f, 1.f);
#pragma unroll
      for (int t = 6; t >= 0; --t) fr[t] = make_float2(fr[t + 1].x * a8[t + 1].x, fr[t + 1].y * a8[t + 1].y);
      // Rows 8 m + t of the 128B-swizzled K-major operands (row r at (r / 8)
      // 1024 + (r % 8) 128 bytes, its 16-byte chunks permuted by XOR with r %
      // 8): the thread's channel pair sits at a fixed byte of a chunk, and
      // for token t of its block at row offset t 128 + (chunk ^ t) 16.
      // fp16 operands: 64-channel blocks kb bytes apart, 8 channels a chunk.
      const uint32_t ch16 = (uint32_t)(((2 * gp) & 63) >> 3) << 4, cb16 = (uint32_t)((2 * gp) & 7) * 2;
      auto rowh = [&](uint32_t kb, int m) { return (uint32_t)(gp >> 5) * kb + (uint32_t)m * 1024u + cb16; };
      auto put_h = [&](uint8_t* tile, unsigned bytes, uint32_t ob, int t, float x, float y) {
        tile_at<__half2>(tile, bytes, ob + (uint32_t)t * 128u + (ch16 ^ ((uint32_t)t << 4))) = __floats2half2_rn(x, y);
      };
      const int m3 = gb >> 1;                                  // level-3 row / column block
      const int m2 = (gb & 1) + ((gb >> 2) << 1);              // level-2 row / column block
      const uint32_t oax3 = rowh(16384, m3), oaq3 = rowh(16384, 4 + m3), obx3 = rowh(8192, m3);
      const uint32_t oax2 = rowh(16384, 8 + m2), oaq2 = rowh(16384, 12 + m2), obx2 = rowh(8192, 4 + m2);
      const uint32_t oay = rowh(8192, gb - 4), oayq = rowh(8192, gb), oby = rowh(4096, gb);
      // fp32 (tf32) operand [K~;Q~]: 32-channel blocks 16 KB apart, 4 channels a chunk
      const uint32_t ch32 = (uint32_t)(((2 * gp) & 31) >> 2) << 4;
      const uint32_t okq = (uint32_t)(gp >> 4) * 16384u + (uint32_t)gb * 1024u + (uint32_t)((2 * gp) & 3) * 4u;
      // the off-diagonal products' operands first; the [K~;Q~] and K-^T
      // values wait in registers for the products' issue
      float km0[8], km1[8];
      float2 kqk[8], kqq[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float2 kh = make_float2(k8[t].x * rk8v[t], k8[t].y * rk8v[t]);
        const float2 qh = make_float2(q8[t].x * rq8v[t], q8[t].y * rq8v[t]);
        const float2 kl = make_float2(kh.x * fl[t].x, kh.y * fl[t].y), ql = make_float2(qh.x * fl[t].x, qh.y * fl[t].y);
        const float2 kr = make_float2(kh.x * fr[t].x, kh.y * fr[t].y);
        kqk[t] = make_float2(umma::tf32_round(kl.x * Eb.x), umma::tf32_round(kl.y * Eb.y));
        kqq[t] = make_float2(umma::tf32_round(ql.x * Eb.x), umma::tf32_round(ql.y * Eb.y));
        km0[t] = umma::tf32_round(kr.x * Ee.x);
        km1[t] = umma::tf32_round(kr.y * Ee.y);
        if (gb & 1) {  // level-3 rows (blocks 1, 3, 5, 7)
          put_h(S.ru.ops.ax, sizeof(S.ru.ops.ax), oax3, t, kl.x, kl.y);
          put_h(S.ru.ops.ax, sizeof(S.ru.ops.ax), oaq3, t, ql.x, ql.y);
        } else {       // level-3 columns (blocks 0, 2, 4, 6)
          put_h(S.ru.ops.bx, sizeof(S.ru.ops.bx), obx3, t, kr.x * E3.x, kr.y * E3.y);
        }
        if (gb & 2) {  // level-2 rows (blocks 2, 3, 6, 7)
          put_h(S.ru.ops.ax, sizeof(S.ru.ops.ax), oax2, t, kl.x * F2.x, kl.y * F2.y);
          put_h(S.ru.ops.ax, sizeof(S.ru.ops.ax), oaq2, t, ql.x * F2.x, ql.y * F2.y);
        } else {       // level-2 columns (blocks 0, 1, 4, 5)
          put_h(S.ru.ops.bx, sizeof(S.ru.ops.bx), obx2, t, kr.x * E2.x, kr.y * E2.y);
        }
        if (gb >= 4) {  // level-1 rows (blocks 4..7)
          put_h(S.ru.ops.ay, sizeof(S.ru.ops.ay), oay, t, kl.x * F1.x, kl.y * F1.y);
          put_h(S.ru.ops.ay, sizeof(S.ru.ops.ay), oayq, t, ql.x * F1.x, ql.y * F1.y);
        } else {        // level-1 columns (blocks 0..3)
          put_h(S.rt.by, sizeof(S.rt.by), oby, t, kr.x * EY.x, kr.y * EY.y);
        }
      }
      umma::fence_proxy_async();
      umma::fence_before();
      __syncthreads();
      od_pending = true;
      issue_offdiag();
      // meanwhile [K~;Q~] and K-^T (read by later products only)
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t rt32 = okq + (uint32_t)t * 128u + (ch32 ^ ((uint32_t)t << 4));
        tile_at<float2>(S.kq, sizeof(S.kq), rt32) = kqk[t];
        tile_at<float2>(S.kq, sizeof(S.kq), rt32 + 8u * 1024u) = kqq[t];  // Q~ rows: 64 rows on
      }
#pragma unroll
      for (int h4 = 0; h4 < 2; ++h4) {
        // rows 2 gp and 2 gp + 1, in an order that puts the 8 lanes of each
        // quarter-warp store on 8 distinct 16-byte chunks (row % 8 distinct)
        const bool sw = (gp >> 2) & 1;
        const float4 v0 = make_float4(km0[4 * h4], km0[4 * h4 + 1], km0[4 * h4 + 2], km0[4 * h4 + 3]);
        const float4 v1 = make_float4(km1[4 * h4], km1[4 * h4 + 1], km1[4 * h4 + 2], km1[4 * h4 + 3]);
        tile_at<float4>(S.kt, sizeof(S.kt), f32_off(2 * gp + sw, 8 * gb + 4 * h4, 128 * 128)) = sw ? v1 : v0;
        tile_at<float4>(S.kt, sizeof(S.kt), f32_off(2 * gp + !sw, 8 * gb + 4 * h4, 128 * 128)) = sw ? v0 : v1;
      }
      umma::fence_proxy_async();  // (seen by the products that read them after later barriers)
    }
    // meanwhile (neither is an operand of the products): M's diagonal blocks
    // from dgM, zeros right of them, and T2 cleared
    {
      const int t = tid >> 3, J = tid & 7, I = t >> 3, tl = t & 7;
      if (J >= I) {
        float mv[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) mv[jj] = (J == I && jj <= tl) ? umma::tf32_round(S.dgM[t][jj]) : 0.f;
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4)
          tile_at<float4>(S.rt.t.mq, sizeof(S.rt.t.mq), f32_off(t, 8 * J + 4 * h4, 64 * 128)) =
              make_float4(mv[4 * h4], mv[4 * h4 + 1], mv[4 * h4 + 2], mv[4 * h4 + 3]);
      }
      for (int e = tid; e < (int)(sizeof(S.rt.t.t2) / 16); e += kThreads)
        reinterpret_cast<uint4*>(S.rt.t.t2)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (!wait_all(&S.od_bar, c & 1)) break;
    od_pending = false;
    umma::fence_after();
    // the next chunk's gate logits (their part of region U is free from
    // here), and its raw boxes into L2 (their copies into shared memory start
    // after the solve, where they lie wholly inside the tensor)
    if (c + 1 < nch) {
      if (warp == 0) {
        issue_ga(c + 1);
        const int32_t row1 = (int32_t)(t0 + (P + kC - 3 - p0));
        if (lane == 4 && row1 >= 0 && (int64_t)row1 + kRawRows <= a.total) {
#pragma unroll
          for (int q = 0; q < 3; ++q) tma_prefetch_2d(&qmap, part_x[q], row1);
        }
      }
      ga_issued = c + 2;
    }
    // A (fp32, for the solve: beta_t A'), M below the diagonal blocks (tf32
    // operand), X and T1 (cleared: the solve writes their lower triangles)
    {
      const auto A = GDN_SV(S.ru.sv.A, kC * kAX);
      const int q4 = warp & 3, k4 = warp >> 2;
      // 8 entries of row t in block column J: k rows (even lane quarter) to A,
      // q rows (odd) to M
      auto put4 = [&](int t, int j, float x0, float x1, float x2, float x3) {
        if (!(q4 & 1)) {
          const float bt = S.beta[GDN_S(t, kC)];
          vec_at<float4>(A, t * kAX + j) = make_float4(x0 * bt, x1 * bt, x2 * bt, x3 * bt);
        } else {
          tile_at<float4>(S.rt.t.mq, sizeof(S.rt.t.mq), f32_off(t, j, 64 * 128)) =
              make_float4(umma::tf32_round(x0), umma::tf32_round(x1), umma::tf32_round(x2), umma::tf32_round(x3));
        }
      };
#define GDN_PUT8(t, J, v, o)                                                \
  do {                                                                      \
    put4((t), 8 * (J), v[(o)], v[(o) + 1], v[(o) + 2], v[(o) + 3]);         \
    put4((t), 8 * (J) + 4, v[(o) + 4], v[(o) + 5], v[(o) + 6], v[(o) + 7]); \
  } while (0)
      const int m = lane >> 3, r = lane & 7;
      if (q4 < 2) {
        // lanes 0..63: level-3 rows (block 2m + 1; its columns: block 2m, at
        // columns 8m of the first product) and level-1 rows (block 4 + m)
        if (k4 == 0) {
          float v[32], w[8];
          umma::tmem_ld32(tlane + TM_DX, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = m == 0 ? v[i] : m == 1 ? v[8 + i] : m == 2 ? v[16 + i] : v[24 + i];
          GDN_PUT8(8 * (2 * m + 1) + r, 2 * m, w, 0);
        } else if (k4 < 3) {
          float v[16];
          umma::tmem_ld16(tlane + TM_DY + 16 * (k4 - 1), v);
          GDN_PUT8(8 * (4 + m) + r, 2 * (k4 - 1), v, 0);
          GDN_PUT8(8 * (4 + m) + r, 2 * (k4 - 1) + 1, v, 8);
        }
      } else if (k4 < 2) {
        // lanes 64..127: level-2 rows (blocks 2, 3, 6, 7); columns 32..47 hold
        // blocks 0, 1 (for rows of 2, 3), 48..63 blocks 4, 5 (rows of 6, 7)
        float v[16];
        umma::tmem_ld16(tlane + TM_DX + 32 + 16 * k4, v);
        if ((m >> 1) == k4) {
          const int I = m + 2 + 2 * (m >> 1);
          GDN_PUT8(8 * I + r, 4 * k4, v, 0);
          GDN_PUT8(8 * I + r, 4 * k4 + 1, v, 8);
        }
      }
#undef GDN_PUT8
      // row t, columns 8 J .. 8 J + 7: A's diagonal block (J = t / 8) from
      // dgA, zeros right of it
      {
        const int t = tid >> 3, J = tid & 7, I = t >> 3, tl = t & 7;
        if (J >= I) {
          float av[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) av[jj] = (J == I && jj < tl) ? S.dgA[t][jj] : 0.f;
#pragma unroll
          for (int h4 = 0; h4 < 2; ++h4)
            vec_at<float4>(A, t * kAX + 8 * J + 4 * h4) =
                make_float4(av[4 * h4], av[4 * h4 + 1], av[4 * h4 + 2], av[4 * h4 + 3]);
        }
      }
      for (int e = tid; e < kC * kAX / 4; e += kThreads)
        reinterpret_cast<float4*>(S.ru.sv.X)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int e = tid; e < (int)(sizeof(S.rt.t.tm) / 16); e += kThreads)
        reinterpret_cast<uint4*>(S.rt.t.tm)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    // ---- E | O1 = S [K~;Q~]^T on the tensor core, issued by a lane of warp 10,
    //      idle in the solve's first phase (a thread issuing products waits
    //      for the tensor core to take them); runs under the solve ----------
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
    // ---- T1 = X diag(beta), T2 = -T1 ---------------------------------------------
    solve_T(S.ru.sv.A, S.ru.sv.X, S.ru.sv.Y, S.ru.sv.L0, TOut{S.rt.t.tm, S.rt.t.t2, S.beta, S.ones, S.ones});
    umma::fence_proxy_async();
    __syncthreads();
    // the next chunk's raw rows (region U is dead)
    if (c + 1 < nch) {
      if (warp == 0) issue_raw(c + 1);
      ld_issued = c + 2;
    }
    if (!wait_all(&S.eo_bar, c & 1)) break;
    eo_pending = false;
    umma::fence_after();
    // ---- Delta = V^T T1^T + E T2^T (tensor core), S <- S diag(e^{lb_63}) -----
    if (tid == 0) {
      const uint64_t dtm = umma::desc(smem_addr(S.rt.t.tm), 16, 1024);
      const uint64_t dt2 = umma::desc(smem_addr(S.rt.t.t2), 16, 1024);
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
      float v[32];
      umma::tmem_ld32(tlane + TM_S + 32 * qq, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 d = *reinterpret_cast<const float4*>(&S.alast[32 * qq + 4 * i]);
        v[4 * i] *= d.x; v[4 * i + 1] *= d.y; v[4 * i + 2] *= d.z; v[4 * i + 3] *= d.w;
      }
      umma::tmem_st32(tlane + TM_S + 32 * qq, v);
    }
    umma::fence_before();
    if (!mma_wait()) break;
    // ---- S += Delta K- ; O2 = Delta M^T ----------------------------------------
    if (tid == 0) {
      const uint64_t dkt = umma::desc(smem_addr(S.kt), 16, 1024);
      const uint64_t dmq = umma::desc(smem_addr(S.rt.t.mq), 16, 1024);
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
    // ---- output O = O1 + O2, staged [token][dv] bf16 in t2 ----------------------
    {
      float o1[16], o2[16];
      umma::tmem_ld16(tlane + TM_O1 + 16 * qq, o1);
      umma::tmem_ld16(tlane + TM_O2 + 16 * qq, o2);
      const auto ot = GDN_SV(reinterpret_cast<__nv_bfloat16*>(S.rt.t.t2), kC * kD);
#pragma unroll
      for (int i = 0; i < 16; ++i) ot[(16 * qq + i) * kD + lrow] = __float2bfloat16_rn(o1[i] + o2[i]);
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
      if (full && GDN_SPAN_G(t0 + (P - p0), kC, a.total) && GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD))
        tma_store_2d(&omap, S.rt.t.t2, h * kD, (int32_t)(t0 + (P - p0)));
      if (cid >= 0) {
        const int32_t yy = (int32_t)(((int64_t)cid * a.hv + h) * kD);
        if (GDN_SPAN_G(yy, kD, (long long)a.ck_num_slots * a.hv * kD)) {
#pragma unroll
          for (int k = 0; k < 4; ++k) tma_store_2d(&cmap, S.kq + k * 16384, 32 * k, yy);
        }
      }
      bulk_commit();
    }
    if (!full) {  // rows of the chunk's tokens inside the sequence: 16-byte stores
      const auto ot = GDN_SV(reinterpret_cast<const __nv_bfloat16*>(S.rt.t.t2), kC * kD);
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
      if (od_pending) mbar_wait(&S.od_bar, c & 1);
      for (int k = ld_done; k < ld_issued; ++k) mbar_wait(&S.ld_bar, k & 1);
      for (int k = ga_done; k < ga_issued; ++k) mbar_wait(&S.ga_bar, k & 1);
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
    mbar_inval(&S.ga_bar);
    mbar_inval(&S.mma_bar);
    mbar_inval(&S.od_bar);
    mbar_inval(&S.eo_bar);
  }
}

// grid (hv, n_seq), 512 threads, one CTA per SM: one chain each.
__global__ void __launch_bounds__(kThreads, 1)
    kda_tc32_kernel(const KdaTcArgs a, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap omap,
                    const __grid_constant__ CUtensorMap cmap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  KSmem& S = *reinterpret_cast<KSmem*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int warp = threadIdx.x >> 5;
  if (warp == 0) umma::tmem_alloc(&S.tmem_base, TM_COLS);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = S.tmem_base;
  kda_chain(a, qmap, amap, omap, cmap, S, tmem, blockIdx.x, blockIdx.y);
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side (declared in kda_tc32.cuh)
// ---------------------------------------------------------------------------
bool kda_tc32_supported(const gdn_dims& d, const void* qkv, const void* av, const void* out, const gdn_params& p) {
  if (d.dk != kD || d.dv != kD || d.conv_width != 4) return false;
  if (d.act_dtype != GDN_BF16 || d.conv_dtype != GDN_BF16) return false;
  if (!aligned(qkv, 16) || !aligned(av, 16) || !aligned(out, 16) || !aligned(p.conv_w, 16) || !aligned(p.dt_bias, 8))
    return false;
  return true;
}

cudaError_t kda_tc32_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt, const gdn_params& p,
                            const int32_t* slot_ids, const int32_t* cu_seqlens, const int64_t* start_pos,
                            int32_t n_seq, int64_t total, const int32_t* ckpt_ids, int32_t max_ckpt,
                            int32_t ckpt_block, const void* qkv, const void* av, const void* bv, void* out,
                            uint32_t* dev_err, cudaStream_t s) {
  KdaTcArgs a;
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
  a.b = reinterpret_cast<const __nv_bfloat16*>(bv);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.err = dev_err;
  a.hk = d.hk;
  a.hv = d.hv;
  a.C = (int32_t)channels(d);
  a.G = d.hv / d.hk;
  const size_t smem = sizeof(KSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kda_tc32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // qkv [total][C] in boxes of 128 channels x 67 rows; the gate logits
  // [total][hv * 128] in boxes of one V head x 64 rows; out [total][hv * 128]
  // in boxes of one V head x 64 tokens; checkpoint states as in the GDN chain
  CUtensorMap qmap, amap, omap, cmap;
  if ((e = tensor_map_2d(&qmap, qkv, total, a.C, 2, kD, kRawRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&amap, av, total, (int64_t)a.hv * kD, 2, kD, kC, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&omap, out, total, (int64_t)a.hv * kD, 2, kD, kC, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  const bool has_ck = a.ck_ssm != nullptr && a.ck_num_slots > 0;
  if ((e = tensor_map_2d(&cmap, has_ck ? a.ck_ssm : a.ssm, (int64_t)(has_ck ? a.ck_num_slots : a.num_slots) * a.hv * kD,
                         kD, 4, 32, kD, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  return launch_plain(kda_tc32_kernel, dim3((unsigned)a.hv, (unsigned)n_seq), dim3(kThreads), smem, s, dim3(1), a,
                      qmap, amap, omap, cmap);
}

}  // namespace gdn
