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
// reference token per block pair, so that every factor is a product of
// alphas over a token range (at most 1):
//   off the diagonal (t in block I > J, j in block J):
//     e^{lb_t - lb_j} = fl8_t  D8_IJ  fr8_j, fl8_t = e^{lb_t - lb_b(I)} (from the
//     block's first token), fr8_j = e^{lb_e(J) - lb_j} (to the block's last),
//     D8_IJ = e^{lb_b(I) - lb_e(J)}: one fp16 warp-level tensor-core product
//     per block pair, of Lk8 = k^ (.) fl8 and Lq8 = q^ (.) fl8 rows against
//     Rk8 = k^ (.) fr8 rows scaled by D8 (fp16 keeps the 10-bit mantissa the
//     tf32 products keep; every operand lies in [-1, 1]);
//   on the eight 8 x 8 diagonal blocks: fp32 running products of alpha down
//     each row, on the CUDA cores.
// Every within-block factor is a running product of alphas (no differences
// of large cumulative sums), and the block factors exponentials of sums of
// block totals.
//
// One CTA per (V head, sequence), 512 threads, walks the sequence's chunks in
// order; the fp32 state S lives in TMEM for the whole sequence.  Per chunk:
//   gates      thread (channel c, 16-token quarter): log alpha, alpha, the
//              8-block totals
//   features   the 67 raw rows of the head's q, k and v channels and the
//              chunk's gate logits arrive by TMA tensor copies; conv1d +
//              SiLU down the chunk; q and k rows (fp32) into shared memory,
//              V^T (tf32) into TMEM
//   norms      rk_t = 1/|y_k,t|, rq_t = dk^-1/2 / |y_q,t| (with the eps)
//   diagonal   the 8 x 8 diagonal blocks of A' and M
//   transform  thread (c, quarter): fl8, fr8 by running products; the tf32
//              operand tiles [K~;Q~] and K-^T, the fp16 Lk8, Lq8, Rk8 and D8
//   off-diag   A' and M below the diagonal blocks (mma m16n8k16 f16)
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
constexpr int kHS = kD + 8;   // row stride (halves) of the fp16 operand rows: 272 bytes
constexpr int kPairs = 28;    // 8-token block pairs I > J of a chunk

// TMEM columns (fp32; lanes are dv rows)
constexpr uint32_t TM_S = 0;     // S [dv][dk]
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
      __half d8[kPairs][kD];     // D8 per block pair and channel
    } g;
    __half rk8[kC][kHS];         // Rk8 (written over al)
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
      __half lk[kC][kHS];  // Lk8, Lq8
      __half lq[kC][kHS];
    } h;
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
  float dgA[kC][8];   // diagonal blocks: beta_t A'[t][j] (j < t, local j), and
  float dgM[kC][8];   //   M[t][j] (j <= t)
  float ones[kC];
  uint64_t ld_bar, mma_bar, eo_bar;
  uint32_t tmem_base;
};

static_assert(sizeof(KSmem) + 1024 <= 232448, "one CTA's shared memory (with the alignment slack)");

__device__ __forceinline__ bool seq_ok(const KdaTcArgs& a, int n, int64_t& t0, int64_t& len, int64_t& p0) {
  const auto cu = GDN_GV(a.cu_seqlens, a.n_seq + 1);
  t0 = cu[n];
  len = (int64_t)cu[n + 1] - t0;
  p0 = GDN_GV(a.start_pos, a.n_seq)[n];
  return !(t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0);
}

// ---- warp-level fp16 products ---------------------------------------------------
// ldmatrix: four (two) 8 x 8 matrices of 16-bit elements; lane i supplies the
// address of row i % 8 of matrix i / 8 and receives row i / 4, elements
// 2 (i % 4) and 2 (i % 4) + 1 of each matrix
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_addr(p)));
}
// D += A B (m16n8k16, fp16 operands, fp32 accumulate).  Lane = 4 g + q: A
// holds rows g and g + 8, columns 2q, 2q + 1 and 2q + 8, 2q + 9; B columns g,
// rows 2q, 2q + 1 and 2q + 8, 2q + 9; D (g, 2q), (g, 2q + 1), (g + 8, 2q),
// (g + 8, 2q + 1).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t y) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&y));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Block pairs (I > J) in order p = I (I - 1) / 2 + J
__host__ __device__ constexpr int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

// The off-diagonal block pairs of warps 0..14: up to two pairs, as 8 I + J
// (-1: none)
__device__ __forceinline__ void warp_pairs(int w, int& p0, int& p1) {
  constexpr int8_t tbl[15][2] = {{8 * 1 + 0, 8 * 7 + 6}, {8 * 2 + 0, 8 * 2 + 1}, {8 * 3 + 0, 8 * 3 + 1},
                                 {8 * 3 + 2, -1},        {8 * 4 + 0, 8 * 4 + 1}, {8 * 4 + 2, 8 * 4 + 3},
                                 {8 * 5 + 0, 8 * 5 + 1}, {8 * 5 + 2, 8 * 5 + 3}, {8 * 5 + 4, -1},
                                 {8 * 6 + 0, 8 * 6 + 1}, {8 * 6 + 2, 8 * 6 + 3}, {8 * 6 + 4, 8 * 6 + 5},
                                 {8 * 7 + 0, 8 * 7 + 1}, {8 * 7 + 2, 8 * 7 + 3}, {8 * 7 + 4, 8 * 7 + 5}};
  p0 = tbl[w][0];
  p1 = tbl[w][1];
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

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
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
        const float4 kp = mul4(kj, p[r]);
        acc[o + j] += dot4(qr[r], kp);
        if (t > j) acc[o + t + 1 + j] += dot4(kr[r], kp);
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
    mbar_init(&S.mma_bar, 1);
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
  static_assert(sizeof(KSmem::rt) == 3 * 16384 && kC * kYS * 4 + kPairs * kD * 2 <= 3 * 16384,
                "region T holds T1, T2, M or alpha and D8");
  static_assert(2 * kC * kYS * 4 <= sizeof(KSmem::ru) && 2 * kC * kAX * 4 + (2048 + 8 * 3 * 64) * 4 <= sizeof(KSmem::ru),
                "region U holds the feature rows or the solve's scratch");
  static_assert(TM_E == TM_S + 256 && TM_O1 == TM_E + 64 && TM_DL == TM_O1 + 64 && TM_V == TM_DL + 64 &&
                    TM_V + 64 <= TM_COLS && TM_O2 == TM_V,
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
  // gate channel of this thread (gates and transform: channel gc, tokens 16 gq ..)
  const int gc = tid & 127, gq = tid >> 7;
  const float eA = expf(GDN_GV(a.A_log, a.hv)[h]);
  const float dtb = GDN_GV(a.dt_bias, (long long)a.hv * kD)[(size_t)h * kD + gc];
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
  constexpr uint32_t kLoadBytes = 3u * kRawRows * kD * 2u + (uint32_t)kC * kD * 2u;
  auto issue_loads = [&](int c) {  // thread 0: chunk c's raw rows and gate logits into region U
    const int64_t P = (p0 / kC + c) * kC;
    const int32_t row0 = (int32_t)(t0 + (P - 3 - p0));  // packed row of raw row 0 (may be < 0)
    mbar_arrive_expect_tx(&S.ld_bar, kLoadBytes);
#pragma unroll
    for (int q = 0; q < 3; ++q)  // a box of 128 channels from part_x[q], 67 rows (rows outside: zeros)
      if (GDN_SPAN_G(part_x[q], kD, a.C) && GDN_SBYTES(&S.ru.in.raw[q][0][0], kRawRows * kD * 2, S))
        tma_load_2d(&S.ru.in.raw[q][0][0], &qmap, part_x[q], row0, &S.ld_bar);
    // gate logits: 128 channels of V head h, 64 rows from the chunk's first token
    if (GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD) && GDN_SBYTES(&S.ru.in.ga[0][0], kC * kD * 2, S))
      tma_load_2d(&S.ru.in.ga[0][0], &amap, h * kD, row0 + 3, &S.ld_bar);
  };
  // beta logit of chunk c's token tid (threads 0..63), loaded one chunk ahead
  auto load_beta = [&](int c) -> float {
    const int64_t pos = (p0 / kC + c) * kC + tid;
    if (tid < kC && c < nch && pos >= p0 && pos < p1)
      return __bfloat162float(gate_b[(size_t)(t0 + pos - p0) * a.hv + h]);
    return 0.f;
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
  int ld_issued = 0, ld_done = 0;
  if (tid == 0) {
    issue_loads(0);
    ld_issued = 1;
  }
  float bl = load_beta(0);

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

  bool eo_pending = false;
  int c = 0;
  for (; c < nch; ++c) {
    const int64_t P = (p0 / kC + c) * kC;
    const bool full = P >= p0 && P + kC <= p1;
    const int tlo = (int)(p0 > P ? (p0 - P < kC ? p0 - P : kC) : 0);
    const int thi = (int)(p1 > P ? (p1 - P < kC ? p1 - P : kC) : 0);
    // the previous chunk's tensor stores have read kq (checkpoint staging)
    // and t2 (output staging)
    if (tid == 0) bulk_wait_read();
    if (tid < kC) S.beta[tid] = (unsigned)(tid - tlo) < (unsigned)(thi - tlo) ? sigmoid_f(bl) : 0.f;
    bl = load_beta(c + 1);
    if (!wait_all(&S.ld_bar, c & 1)) break;
    ld_done = c + 1;
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

    // ---- gates: log alpha, alpha, 8-block totals (thread: channel gc, tokens 16 gq ..)
    {
      const auto ga = GDN_SV(&S.ru.in.ga[0][0], kC * kD);
      const auto al = GDN_SV(&S.rt.g.al[0][0], kC * kYS);
      float G0 = 0.f, G1 = 0.f, f0 = 0.f, f1 = 0.f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int tt = 16 * gq + t;
        const bool valid = (unsigned)(tt - tlo) < (unsigned)(thi - tlo);
        const float x = __bfloat162float(ga[tt * kD + gc]) + dtb;
        const float sp = x > 20.f ? x : __logf(1.f + __expf(x));
        const float g = valid ? floor_log_decay(-eA * sp) : 0.f;
        al[tt * kYS + gc] = __expf(g);
        if (t < 8) G0 += g; else G1 += g;
        if (t == 0) f0 = g;
        if (t == 8) f1 = g;
      }
      S.G8[2 * gq][gc] = G0;
      S.G8[2 * gq + 1][gc] = G1;
      S.g8f[2 * gq][gc] = f0;
      S.g8f[2 * gq + 1][gc] = f1;
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
    __syncthreads();
    {
      const int tk = 16 * qq;
      const auto yd = GDN_SV(isq ? &S.ru.y.yq[0][0] : &S.ru.y.yk[0][0], kC * kYS);
#pragma unroll
      for (int t = 0; t < 16; ++t) vec_at<float2>(yd, (tk + t) * kYS + 2 * cp) = y[t];
      umma::tmem_st16(tlane + TM_V + tk, vv);
    }
    __syncthreads();
    // ---- norms: warp w, tokens 4 w .. 4 w + 3 ---------------------------------
    {
      float sk[4], sq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * warp + i;
        const float4 k4 = vec_at<const float4>(GDN_SV(&S.ru.y.yk[0][0], kC * kYS), t * kYS + 4 * lane);
        const float4 q4 = vec_at<const float4>(GDN_SV(&S.ru.y.yq[0][0], kC * kYS), t * kYS + 4 * lane);
        sk[i] = dot4(k4, k4);
        sq[i] = dot4(q4, q4);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sk[i] += __shfl_xor_sync(0xffffffffu, sk[i], o);
          sq[i] += __shfl_xor_sync(0xffffffffu, sq[i], o);
        }
      if (lane < 4) {
        float k = sk[0], q = sq[0];
#pragma unroll
        for (int i = 1; i < 4; ++i)
          if (lane == i) {
            k = sk[i];
            q = sq[i];
          }
        S.rk[4 * warp + lane] = rsqrtf(k + kNormEps);
        S.rq[4 * warp + lane] = rsqrtf(q + kNormEps) * rsqrtf((float)kD);
      }
    }
    __syncthreads();
    // ---- the 8 x 8 diagonal blocks of A' and M --------------------------------
    if (warp & 1)
      diag_block<1>(S, warp >> 1);
    else
      diag_block<0>(S, warp >> 1);

    // ---- transform (thread: channel gc, tokens 16 gq ..) -----------------------
    {
      const auto al = GDN_SV(&S.rt.g.al[0][0], kC * kYS);
      const auto yk = GDN_SV(&S.ru.y.yk[0][0], kC * kYS), yq = GDN_SV(&S.ru.y.yq[0][0], kC * kYS);
      float a16[16], k16[16], q16[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int tt = 16 * gq + t;
        a16[t] = al[tt * kYS + gc];
        k16[t] = yk[tt * kYS + gc];
        q16[t] = yq[tt * kYS + gc];
      }
      // block factors of the thread's 8-blocks I0 = 2 gq, I1 = 2 gq + 1:
      // e^{lb} at their first tokens and e^{lb_63 - lb} at their last
      float pre = 0.f, post = 0.f, tot = 0.f;
#pragma unroll
      for (int K = 0; K < 8; ++K) {
        const float gk = S.G8[K][gc];
        tot += gk;
        if (K < 2 * gq) pre += gk;
        if (K > 2 * gq + 1) post += gk;
      }
      const float G0 = S.G8[2 * gq][gc], G1 = S.G8[2 * gq + 1][gc];
      const float Eb0 = expf(pre + S.g8f[2 * gq][gc]), Eb1 = expf(pre + G0 + S.g8f[2 * gq + 1][gc]);
      const float Ee1 = expf(post), Ee0 = expf(post + G1);
      if (gq == 0) S.alast[gc] = expf(tot);
      // D8 for every block pair: thread tid takes entries tid + 512 m
#pragma unroll
      for (int m = 0; m < kPairs * kD / kThreads; ++m) {
        const int e = tid + kThreads * m, p = e >> 7, cc = e & 127;
        int I = 1;
#pragma unroll
        for (int i = 2; i < 8; ++i)
          if (p >= pair_index(i, 0)) I = i;
        const int J = p - pair_index(I, 0);
        float s = S.g8f[I][cc];
        for (int K = J + 1; K < I; ++K) s += S.G8[K][cc];
        S.rt.g.d8[GDN_S(p, kPairs)][cc] = __float2half_rn(expf(s));
      }
      float4 rk4[4], rq4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rk4[i] = *reinterpret_cast<const float4*>(&S.rk[16 * gq + 4 * i]);
        rq4[i] = *reinterpret_cast<const float4*>(&S.rq[16 * gq + 4 * i]);
      }
      // alpha, the feature rows and the diagonal blocks are read: the
      // operands take regions T and U
      __syncthreads();
      float fl[16], fr[16];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        float f = 1.f;
        fl[8 * hb] = 1.f;
#pragma unroll
        for (int t = 1; t < 8; ++t) {
          f *= a16[8 * hb + t];
          fl[8 * hb + t] = f;
        }
        f = 1.f;
#pragma unroll
        for (int t = 7; t >= 0; --t) {
          fr[8 * hb + t] = f;
          f *= a16[8 * hb + t];
        }
      }
      const auto lk = GDN_SV(&S.ru.h.lk[0][0], kC * kHS), lq = GDN_SV(&S.ru.h.lq[0][0], kC * kHS);
      const auto rk8 = GDN_SV(&S.rt.rk8[0][0], kC * kHS);
      float km[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int tt = 16 * gq + t;
        const float rkt = reinterpret_cast<const float*>(rk4)[t], rqt = reinterpret_cast<const float*>(rq4)[t];
        const float kh = k16[t] * rkt, qh = q16[t] * rqt;
        const float Eb = t < 8 ? Eb0 : Eb1, Ee = t < 8 ? Ee0 : Ee1;
        tile_at<float>(S.kq, sizeof(S.kq), f32_off(tt, gc, 128 * 128)) = umma::tf32_round(kh * fl[t] * Eb);
        tile_at<float>(S.kq, sizeof(S.kq), f32_off(kC + tt, gc, 128 * 128)) = umma::tf32_round(qh * fl[t] * Eb);
        km[t] = umma::tf32_round(kh * fr[t] * Ee);
        lk[tt * kHS + gc] = __float2half_rn(kh * fl[t]);
        lq[tt * kHS + gc] = __float2half_rn(qh * fl[t]);
        rk8[tt * kHS + gc] = __float2half_rn(kh * fr[t]);
      }
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4)
        tile_at<float4>(S.kt, sizeof(S.kt), f32_off(gc, 16 * gq + 4 * t4, 128 * 128)) =
            make_float4(km[4 * t4], km[4 * t4 + 1], km[4 * t4 + 2], km[4 * t4 + 3]);
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    // ---- A' and M below the diagonal blocks (warps 0..14) ----------------------
    float cacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    int pr[2] = {-1, -1};
    if (warp < 15) {
      warp_pairs(warp, pr[0], pr[1]);
      const auto lk = GDN_SV(&S.ru.h.lk[0][0], kC * kHS), lq = GDN_SV(&S.ru.h.lq[0][0], kC * kHS);
      const auto rk8 = GDN_SV(&S.rt.rk8[0][0], kC * kHS);
      const auto d8 = GDN_SV(reinterpret_cast<const uint32_t*>(&S.rt.g.d8[0][0]), kPairs * kD / 2);
      const int q = lane & 3;
      const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row this lane addresses
      const int Ia = pr[0] >> 3, Ib = pr[1] >= 0 ? pr[1] >> 3 : Ia;
#pragma unroll 2
      for (int ks = 0; ks < kD / 16; ++ks) {
        const int k0 = 16 * ks;
        uint32_t fa[2][4];
        // A: rows 0..7 Lk8, rows 8..15 Lq8 of block I; columns k0 .. k0 + 15
        ldsm_x4(fa[0], (mi & 1 ? lq : lk).at((8 * Ia + ri) * kHS + k0 + 8 * (mi >> 1), 8));
        if (Ib != Ia) ldsm_x4(fa[1], (mi & 1 ? lq : lk).at((8 * Ib + ri) * kHS + k0 + 8 * (mi >> 1), 8));
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (pr[i] < 0) continue;
          const int I = pr[i] >> 3, J = pr[i] & 7, p = pair_index(I, J);
          uint32_t fb[2];
          ldsm_x2(fb, rk8.at((8 * J + ri) * kHS + k0 + 8 * (mi & 1), 8));
          fb[0] = hmul2_bits(fb[0], d8[(p * kD + k0 + 2 * q) / 2]);
          fb[1] = hmul2_bits(fb[1], d8[(p * kD + k0 + 8 + 2 * q) / 2]);
          mma_f16(cacc[i], (i == 1 && Ib != Ia) ? fa[1] : fa[0], fb[0], fb[1]);
        }
      }
    }
    // every operand read: A (fp32, for the solve), M (tf32 operand), X and T1,
    // T2 (cleared: the solve writes their lower triangles)
    __syncthreads();
    {
      const auto A = GDN_SV(S.ru.sv.A, kC * kAX);
      if (warp < 15) {
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (pr[i] < 0) continue;
          const int I = pr[i] >> 3, J = pr[i] & 7;
          const int t = 8 * I + g, j = 8 * J + 2 * q;
          const float bt = S.beta[t];
          vec_at<float2>(A, t * kAX + j) = make_float2(cacc[i][0] * bt, cacc[i][1] * bt);
          tile_at<float2>(S.rt.t.mq, sizeof(S.rt.t.mq), f32_off(t, j, 64 * 128)) =
              make_float2(umma::tf32_round(cacc[i][2]), umma::tf32_round(cacc[i][3]));
        }
      }
      // row t, columns 8 J .. 8 J + 7: the diagonal block (J = t / 8) from
      // dgA / dgM, zeros right of it
      {
        const int t = tid >> 3, J = tid & 7, I = t >> 3, tl = t & 7;
        if (J >= I) {
          float av[8], mv[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            av[jj] = (J == I && jj < tl) ? S.dgA[t][jj] : 0.f;
            mv[jj] = (J == I && jj <= tl) ? umma::tf32_round(S.dgM[t][jj]) : 0.f;
          }
#pragma unroll
          for (int h4 = 0; h4 < 2; ++h4) {
            vec_at<float4>(A, t * kAX + 8 * J + 4 * h4) =
                make_float4(av[4 * h4], av[4 * h4 + 1], av[4 * h4 + 2], av[4 * h4 + 3]);
            tile_at<float4>(S.rt.t.mq, sizeof(S.rt.t.mq), f32_off(t, 8 * J + 4 * h4, 64 * 128)) =
                make_float4(mv[4 * h4], mv[4 * h4 + 1], mv[4 * h4 + 2], mv[4 * h4 + 3]);
          }
        }
      }
      for (int e = tid; e < kC * kAX / 4; e += kThreads)
        reinterpret_cast<float4*>(S.ru.sv.X)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int e = tid; e < (int)(2 * sizeof(S.rt.t.tm) / 16); e += kThreads)
        reinterpret_cast<uint4*>(S.rt.t.tm)[e] = make_uint4(0u, 0u, 0u, 0u);  // tm and t2
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
    // the next chunk's raw rows and gate logits (region U is dead)
    if (tid == 0 && c + 1 < nch) {
      issue_loads(c + 1);
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
      for (int k = ld_done; k < ld_issued; ++k) mbar_wait(&S.ld_bar, k & 1);
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
  if (!aligned(qkv, 16) || !aligned(av, 16) || !aligned(out, 16) || !aligned(p.conv_w, 16)) return false;
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
