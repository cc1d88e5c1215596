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
//              channel runs conv1d + SiLU down the chunk; the q/k rows' L2
//              norms come from a warp reduce-scatter of the squares.  Written
//              as tf32 operands: [K^ ; Q^] (shared memory, K-major),
//              K~^T = (diag(e^{b_last - b}) K^)^T (shared memory, K-major over
//              tokens) and V^T (tensor memory).
//   P          [K^;Q^] K^T                                (tcgen05, TMEM)
//   A, M       A = strict_lower(beta (.) K K^T (.) Gamma) (fp32, for the
//              solve), M = Q K^T (.) Gamma (.) lower-incl (tf32 operand)
//   T          (I + A)^-1 diag(beta): 8 x 8 substitutions, then merges on
//              warp-level mma in split tf32 (hi/lo: fp32 accuracy); written
//              as T and T'' = -T diag(e^b) (tf32 operands)
//   Delta^T    = V^T T^T + (S^T K^T) T''^T: the WY form's U - W S with
//              W = T diag(e^b) K, regrouped so that the state meets only the
//              T-free K^ (E = S^T K^T comes with O1 = S^T Q^T in one product
//              whose A operand is the state itself, in TMEM)
//   state      S^T <- e^{b_last} S^T (in TMEM, by the threads) + Delta^T K~
//              (one product accumulating into the state; A = Delta^T in TMEM)
//   output     O = O1 diag(e^b) + Delta^T M^T, staged as a bf16 tile and
//              written by one TMA tensor store
// The fp32 state S^T (dv x dk) lives in TMEM for the whole sequence: it is
// the accumulator of its own update and the A operand of the products that
// read it.  Checkpoints are staged from TMEM into the dead [K;Q] tile and
// leave by TMA tensor stores.  The conv histories of checkpoints and of the
// final state come from the history kernel of prefill.cu.
#include "gdn_common.cuh"
#include "prefill_tc.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;                 // chunk
constexpr int kD = 128;                // dk = dv
constexpr int kThreads = 256;          // 8 warps
constexpr int kRawRows = kC + 3;       // chunk rows plus 3 rows of conv history
constexpr int kAX = 68;                // row stride (floats) of the solve's A and X

// TMEM columns (fp32, one per column).  Lanes are dv rows, except P, whose
// lanes are the [K^;Q^] rows.
constexpr uint32_t TM_S = 0;    // S^T [dv][dk], 128 columns
constexpr uint32_t TM_P = 128;  // [K;Q] K^T [128 rows][64 tokens]
constexpr uint32_t TM_E = 192;  // S^T K^T [dv][64], then O1 = S^T Q^T at TM_E + 64
constexpr uint32_t TM_O1 = 256;
constexpr uint32_t TM_DL = 320;  // Delta^T [dv][64]
constexpr uint32_t TM_O2 = 384;  // Delta^T M^T [dv][64]
constexpr uint32_t TM_V = 448;   // V^T [dv][64] (operand)
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
};

// Shared memory.  Operand tiles are fp32 in the tensor core's 128-byte
// swizzled K-major layout: a 128-byte row holds 32 elements, 8-row groups
// are 1024 bytes apart, and wider rows continue in further 32-column blocks.
struct __align__(1024) Smem32 {
  uint8_t kq[4 * 128 * 128];  // [K^ ; Q^]: rows 0..63 k^, 64..127 q^ (x dk): 4 blocks of 16 KB
  uint8_t kt[2 * 128 * 128];  // K~^T [dk][64 tokens]: 2 blocks of 16 KB
  uint8_t tm[2 * 64 * 128];   // T [i][j]: 2 blocks of 8 KB
  uint8_t t2[2 * 64 * 128];   // T'' = -T diag(e^b); after its product, the output staging tile
  uint8_t mq[2 * 64 * 128];   // M [i][j]
  union {
    __nv_bfloat16 raw[3][kRawRows][kD];  // staged inputs: q, k, v parts
    struct {
      float A[kC * kAX];
      float X[kC * kAX];
      float Y[2048];
    } sv;  // the solve's scratch (after the features have read the inputs)
  };
  float g[kC], beta[kC], b[kC], eb[kC], ebl[kC];
  float part[2][4][kC];  // per-warp partial sums of squares: [k, q][warp][token]
  float rn[2][kC];       // 1 / ||k^||, dk^-1/2 / ||q^|| per token
  uint64_t ld_bar, mma_bar;
  uint32_t tmem_base;
};

__device__ __forceinline__ bool seq_ok(const Tc32Args& a, int n, int64_t& t0, int64_t& len, int64_t& p0) {
  t0 = a.cu_seqlens[n];
  len = (int64_t)a.cu_seqlens[n + 1] - t0;
  p0 = a.start_pos[n];
  return !(t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0);
}

// Byte offset of element (r, c) in a K-major swizzled fp32 tile whose
// 32-column blocks are `blk` bytes apart.
__device__ __forceinline__ uint32_t f32_off(int r, int c, uint32_t blk) {
  return (uint32_t)(c >> 5) * blk + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
         (uint32_t)((((c & 31) >> 2) ^ (r & 7)) << 4) + (uint32_t)(c & 3) * 4u;
}

__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + exp_ftz(-y)); }

// ---- the 64 x 64 solve: T = (I + A)^-1 diag(beta) ---------------------------
// Warp-level tf32 MMA (m16n8k8, fp32 accumulate).  Fragment layout: lane =
// 4 * g + t; A holds (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); B holds
// (t, g), (t + 4, g); D holds (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
// Operands are split x = hi + lo (both tf32) and each product is taken as
// lo*hi + hi*lo + hi*hi, which carries fp32 accuracy.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  const float h = umma::tf32_round(x);
  hi = __float_as_uint(h);
  lo = __float_as_uint(umma::tf32_round(x - h));
}
struct FragA {
  uint32_t h[4], l[4];
};
struct FragB {
  uint32_t h[2], l[2];
};
template <class LF>
__device__ __forceinline__ void frag_a(FragA& a, int k, LF L) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  split_tf32(L(g, k + t), a.h[0], a.l[0]);
  split_tf32(L(g + 8, k + t), a.h[1], a.l[1]);
  split_tf32(L(g, k + t + 4), a.h[2], a.l[2]);
  split_tf32(L(g + 8, k + t + 4), a.h[3], a.l[3]);
}
template <class RF>
__device__ __forceinline__ void frag_b(FragB& b, int k, RF R) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  split_tf32(R(k + t, g), b.h[0], b.l[0]);
  split_tf32(R(k + t + 4, g), b.h[1], b.l[1]);
}
__device__ __forceinline__ void mma_m16n8k8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// a 16 x 8 tile product over NK k-steps of 8 from preloaded split fragments
template <int NK>
__device__ __forceinline__ void tile_mm(float (&d)[4], const FragA (&a)[NK], const FragB (&b)[NK]) {
  d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
  for (int s = 0; s < NK; ++s) {
    mma_m16n8k8(d, a[s].l, b[s].h);
    mma_m16n8k8(d, a[s].h, b[s].l);
    mma_m16n8k8(d, a[s].h, b[s].h);
  }
}
__device__ __forceinline__ int ix(int r, int c) { return r * kAX + c; }

struct TOut {
  uint8_t* tm;        // T
  uint8_t* t2;        // T'' = -T diag(e^b)
  const float* beta;  // [64]
  const float* eb;    // [64]
};
// T entries (r, c), (r, c + 1) (c even) and their T'' counterparts, from X
// entries x0, x1 (bc: beta of the two columns, ec: their e^b)
__device__ __forceinline__ void put_t(const TOut& o, int r, int c, float x0, float x1, const float2& bc,
                                      const float2& ec) {
  const uint32_t off = f32_off(r, c, 64 * 128);
  const float t0 = x0 * bc.x, t1 = x1 * bc.y;
  *reinterpret_cast<float2*>(o.tm + off) = make_float2(umma::tf32_round(t0), umma::tf32_round(t1));
  *reinterpret_cast<float2*>(o.t2 + off) = make_float2(umma::tf32_round(-t0 * ec.x), umma::tf32_round(-t1 * ec.y));
}

// X = (I + A)^-1 for the 64 x 64 strictly lower A (fp32), written out as the
// lower triangles of T and T'' (their upper triangles are zero already).
// 8 x 8 diagonal blocks by substitution, then merged 8 -> 16 -> 32 -> 64 with
// X_ba = -X_b (A_ba X_a).  Each output column tile j of X_ba needs only column
// tile j of A_ba X_a, so a warp carries its tile through both products.
// Entries above the diagonal of X are never stored; reads mask them to zero.
// Y: 2048 floats of scratch.  256 threads; the caller synchronises before (A
// complete) and after.
__device__ __forceinline__ void solve_T(const float* A, float* X, float* Y, const TOut& to) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  auto bc_of = [&](int c) { return make_float2(to.beta[c], to.beta[c + 1]); };
  auto ec_of = [&](int c) { return make_float2(to.eb[c], to.eb[c + 1]); };
  // 8 x 8 diagonal blocks: warp w, lane l < 4 = columns 2l and 2l+1 of block w
  if (lane < 4) {
    const int o = 8 * warp, c0 = 2 * lane;
    float a[28];
#pragma unroll
    for (int r = 1, i = 0; r < 8; ++r)
#pragma unroll
      for (int m = 0; m < r; ++m, ++i) a[i] = A[ix(o + r, o + m)];
    float x0[8], x1[8];
#pragma unroll
    for (int r = 0, i = 0; r < 8; ++r) {
      float s0 = (r == c0) ? 1.f : 0.f, s1 = (r == c0 + 1) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m, ++i) {
        s0 = fmaf(-a[i], x0[m], s0);
        s1 = fmaf(-a[i], x1[m], s1);
      }
      x0[r] = s0;
      x1[r] = s1;
    }
    const float2 bc = bc_of(o + c0), ec = ec_of(o + c0);
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r >= c0) {
        *reinterpret_cast<float2*>(X + ix(o + r, o + c0)) = make_float2(x0[r], x1[r]);
        put_t(to, o + r, o + c0, x0[r], x1[r], bc, ec);
      }
  }
  __syncthreads();
  // 8 -> 16: warps 0..3, block pair p (rows/cols 16p ..); M padded to 16
  if (warp < 4) {
    const int o = 16 * warp;
    float* Ys = Y + warp * 128;
    FragA fa[1], fx[1];
    FragB fb[1], fy[1];
    frag_a(fa[0], 0, [&](int r, int k) { return r < 8 ? A[ix(o + 8 + r, o + k)] : 0.f; });
    frag_b(fb[0], 0, [&](int k, int c) { return k >= c ? X[ix(o + k, o + c)] : 0.f; });
    frag_a(fx[0], 0, [&](int r, int k) { return (r < 8 && k <= r) ? X[ix(o + 8 + r, o + 8 + k)] : 0.f; });
    float d[4];
    tile_mm<1>(d, fa, fb);
    Ys[g * 8 + 2 * t] = d[0];
    Ys[g * 8 + 2 * t + 1] = d[1];
    __syncwarp();
    frag_b(fy[0], 0, [&](int k, int c) { return Ys[k * 8 + c]; });
    tile_mm<1>(d, fx, fy);
    X[ix(o + 8 + g, o + 2 * t)] = -d[0];
    X[ix(o + 8 + g, o + 2 * t + 1)] = -d[1];
    put_t(to, o + 8 + g, o + 2 * t, -d[0], -d[1], bc_of(o + 2 * t), ec_of(o + 2 * t));
  }
  __syncthreads();
  // 16 -> 32: warps 0..3 = (pair q, column tile j)
  if (warp < 4) {
    const int o = 32 * (warp >> 1), j = warp & 1;
    float* Ys = Y + 512 + warp * 128;
    FragA fa[2], fx[2];
    FragB fb[2], fy[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      frag_a(fa[s], 8 * s, [&](int r, int k) { return A[ix(o + 16 + r, o + k)]; });
      frag_b(fb[s], 8 * s, [&](int k, int c) { return k >= 8 * j + c ? X[ix(o + k, o + 8 * j + c)] : 0.f; });
      frag_a(fx[s], 8 * s, [&](int r, int k) { return k <= r ? X[ix(o + 16 + r, o + 16 + k)] : 0.f; });
    }
    const int cc = o + 8 * j + 2 * t;
    float d[4];
    tile_mm<2>(d, fa, fb);
    Ys[g * 8 + 2 * t] = d[0];
    Ys[g * 8 + 2 * t + 1] = d[1];
    Ys[(g + 8) * 8 + 2 * t] = d[2];
    Ys[(g + 8) * 8 + 2 * t + 1] = d[3];
    __syncwarp();
#pragma unroll
    for (int s = 0; s < 2; ++s) frag_b(fy[s], 8 * s, [&](int k, int c) { return Ys[k * 8 + c]; });
    tile_mm<2>(d, fx, fy);
    X[ix(o + 16 + g, cc)] = -d[0];
    X[ix(o + 16 + g, cc + 1)] = -d[1];
    X[ix(o + 24 + g, cc)] = -d[2];
    X[ix(o + 24 + g, cc + 1)] = -d[3];
    put_t(to, o + 16 + g, cc, -d[0], -d[1], bc_of(cc), ec_of(cc));
    put_t(to, o + 24 + g, cc, -d[2], -d[3], bc_of(cc), ec_of(cc));
  }
  __syncthreads();
  // 32 -> 64: warps = (column tile j, row half mh); the two warps of a column
  // tile exchange their halves of Y_j = A_ba X_a[:, j] through a named
  // barrier.  Rows of X_a above 8j of column tile j are zero (k-steps skipped).
  {
    const int j = warp & 3, mh = warp >> 2;
    float* Ys = Y + 1024 + j * 256;  // 32 x 8
    FragA fa[4], fx[4];
    FragB fb[4], fy[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s >= j) {
        frag_a(fa[s], 8 * s, [&](int r, int k) { return A[ix(32 + 16 * mh + r, k)]; });
        frag_b(fb[s], 8 * s, [&](int k, int c) { return k >= 8 * j + c ? X[ix(k, 8 * j + c)] : 0.f; });
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) fa[s].h[e] = fa[s].l[e] = 0u;
        fb[s].h[0] = fb[s].h[1] = fb[s].l[0] = fb[s].l[1] = 0u;
      }
      frag_a(fx[s], 8 * s, [&](int r, int k) { return k <= 16 * mh + r ? X[ix(32 + 16 * mh + r, 32 + k)] : 0.f; });
    }
    const int cc = 8 * j + 2 * t;
    float d[4];
    tile_mm<4>(d, fa, fb);
    const int yr = 16 * mh + g;
    Ys[yr * 8 + 2 * t] = d[0];
    Ys[yr * 8 + 2 * t + 1] = d[1];
    Ys[(yr + 8) * 8 + 2 * t] = d[2];
    Ys[(yr + 8) * 8 + 2 * t + 1] = d[3];
    named_sync(1 + j, 64);
#pragma unroll
    for (int s = 0; s < 4; ++s) frag_b(fy[s], 8 * s, [&](int k, int c) { return Ys[k * 8 + c]; });
    tile_mm<4>(d, fx, fy);
    put_t(to, 32 + yr, cc, -d[0], -d[1], bc_of(cc), ec_of(cc));
    put_t(to, 40 + yr, cc, -d[2], -d[3], bc_of(cc), ec_of(cc));
  }
}

// ---- the kernel -------------------------------------------------------------
// grid (hv, n_seq), 256 threads, one CTA per SM.  Thread 0 issues the TMA
// copies and the tensor-core products; every wait is bounded (1 s).
template <typename Tconv>
__global__ void __launch_bounds__(kThreads, 1)
    tc32_prefill_kernel(const Tc32Args a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap cmap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem32& S = *reinterpret_cast<Smem32*>(smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, n = blockIdx.y, hq = h / a.G;
  int64_t t0, len, p0;
  if (!seq_ok(a, n, t0, len, p0)) {
    if (h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const int32_t slot = a.slot_ids[n];
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * kD; e += kThreads)
      a.out[((t0 + e / kD) * a.hv + h) * kD + (e % kD)] = __float2bfloat16_rn(0.f);
    return;
  }
  if (len == 0) return;
  const int64_t p1 = p0 + len;
  const int nch = (int)((p1 + kC - 1) / kC - p0 / kC);

  if (tid == 0) {
    mbar_init(&S.ld_bar, 1);
    mbar_init(&S.mma_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) umma::tmem_alloc(&S.tmem_base, TM_COLS);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = S.tmem_base;
  const int lrow = 32 * (warp & 3) + lane;  // TMEM lane of this thread (dv row, or [K;Q] row)
  const int half = warp >> 2;               // which column half this warp handles
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

  constexpr uint32_t ID_P = umma::idesc_tf32(128, 64, false, false);
  constexpr uint32_t ID_N64 = umma::idesc_tf32(128, 64, false, false);
  constexpr uint32_t ID_N128 = umma::idesc_tf32(128, 128, false, false);

  // feature channels of this thread: q/k channel (tid < 128: k, else q) and
  // v channel tid % 128 for token half tid / 128
  const bool isq = tid >= 128;
  const int cqk = tid & 127;
  const int gch_qk = (isq ? hq : a.hk + hq) * kD + cqk;
  const int gch_v = 2 * a.hk * kD + h * kD + cqk;
  float wqk[4], wv[4];
  {
    const float4 w4 = *reinterpret_cast<const float4*>(a.conv_w + (size_t)gch_qk * 4);
    wqk[0] = w4.x; wqk[1] = w4.y; wqk[2] = w4.z; wqk[3] = w4.w;
    const float4 v4 = *reinterpret_cast<const float4*>(a.conv_w + (size_t)gch_v * 4);
    wv[0] = v4.x; wv[1] = v4.y; wv[2] = v4.z; wv[3] = v4.w;
  }
  const float eA = expf(a.A_log[h]), dtb = a.dt_bias[h];
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
    const int32_t id = a.ckpt_ids[(size_t)n * a.max_ckpt + idx];
    return slot_class(id, a.ck_num_slots) == 0 ? id : -1;
  };
  auto issue_raw = [&](int c) {  // thread 0: chunk c's raw rows into S.raw
    const int64_t P = (p0 / kC + c) * kC;
    const int32_t row0 = (int32_t)(t0 + (P - 3 - p0));  // packed row of raw row 0 (may be < 0)
    mbar_arrive_expect_tx(&S.ld_bar, 3u * kRawRows * kD * 2u);
#pragma unroll
    for (int q = 0; q < 3; ++q) tma_load_2d(&S.raw[q][0][0], &qmap, part_x[q], row0, &S.ld_bar);
  };

  // initial state S^T rows into TMEM; the upper triangle of T stays zero
  float* gS = a.ssm + (((size_t)slot * a.hv + h) * kD + lrow) * kD + 64 * half;
  {
    float v[32];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(gS + 32 * k + 4 * i);
        v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
      }
      umma::tmem_st32(tlane + TM_S + 64 * half + 32 * k, v);
    }
  }
  for (int e = tid; e < (int)(sizeof(S.tm) / 16); e += kThreads)
    reinterpret_cast<uint4*>(S.tm)[e] = make_uint4(0u, 0u, 0u, 0u);
  int ld_issued = 0, ld_done = 0;  // raw-row loads issued (thread 0) and completed
  if (tid == 0) {
    issue_raw(0);
    ld_issued = 1;
  }

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

  int c = 0;
  for (; c < nch; ++c) {
    const int64_t P = (p0 / kC + c) * kC;
    const bool full = P >= p0 && P + kC <= p1;
    // gates of the chunk's tokens (outside the sequence: g = beta = 0)
    if (tid < kC) {
      const int64_t pos = P + tid;
      float gv = 0.f, bv = 0.f;
      if (pos >= p0 && pos < p1) {
        const size_t tok = (size_t)(t0 + pos - p0);
        const float av = __bfloat162float(a.a[tok * a.hv + h]);
        const float bb = __bfloat162float(a.b[tok * a.hv + h]);
        gv = floor_log_decay(-eA * softplus_f(av + dtb));
        bv = sigmoid_f(bb);
      }
      S.g[tid] = gv;
      S.beta[tid] = bv;
    }
    // the previous chunk's tensor stores have read the kq tile (checkpoint
    // staging) and the t2 tile (output staging)
    if (tid == 0) bulk_wait_read();
    __syncthreads();
    if (warp == 0) {  // cumulative log decay b, e^b, e^{b_last - b}
      float bv[2], carry = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v = S.g[32 * hh + lane];
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
        S.b[32 * hh + lane] = bv[hh];
        S.eb[32 * hh + lane] = expf(bv[hh]);
        S.ebl[32 * hh + lane] = expf(carry - bv[hh]);
      }
    }
    // the chunk's raw rows landed
    if (!wait_all(&S.ld_bar, c & 1)) break;
    ld_done = c + 1;
    // the up to 3 rows just before the sequence start come from the conv history
    if (P - 3 < p0) {
      const int64_t lo = (P - 3 > p0 - 3) ? P - 3 : p0 - 3;
      const int64_t hi = (P + kC < p0) ? P + kC : p0;
      const Tconv* hist = reinterpret_cast<const Tconv*>(a.conv) + (size_t)slot * 3 * a.C;
      for (int64_t pos = lo; pos < hi; ++pos) {
        const int r = (int)(pos - (P - 3));
        for (int e = tid; e < 3 * kD; e += kThreads) {
          const int q = e / kD, ch = e % kD;
          S.raw[q][r][ch] = __float2bfloat16_rn(to_f32(hist[(size_t)(3 - (p0 - pos)) * a.C + part_x[q] + ch]));
        }
      }
      __syncthreads();
    }

    // ---- features: q/k (one channel per thread, down the chunk) ------------
    {
      const __nv_bfloat16* xs = &S.raw[isq ? 0 : 1][0][cqk];
      float y[kC];
      float x0 = __bfloat162float(xs[0]), x1 = __bfloat162float(xs[kD]), x2 = __bfloat162float(xs[2 * kD]);
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        const float x3 = __bfloat162float(xs[(t + 3) * kD]);
        float acc = wqk[0] * x0;
        acc = fmaf(wqk[1], x1, acc);
        acc = fmaf(wqk[2], x2, acc);
        acc = fmaf(wqk[3], x3, acc);
        const bool valid = full || (P + t >= p0 && P + t < p1);
        y[t] = valid ? silu_fast(acc) : 0.f;
        x0 = x1;
        x1 = x2;
        x2 = x3;
      }
      // sums of squares over the warp's 32 channels: a reduce-scatter that
      // leaves lane l with tokens 2l and 2l + 1
      float s[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float lo = y[i] * y[i], hi = y[32 + i] * y[32 + i];
        const bool up = lane & 16;
        s[i] = (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool up = lane & 8;
        s[i] = (up ? s[16 + i] : s[i]) + __shfl_xor_sync(0xffffffffu, up ? s[i] : s[16 + i], 8);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool up = lane & 4;
        s[i] = (up ? s[8 + i] : s[i]) + __shfl_xor_sync(0xffffffffu, up ? s[i] : s[8 + i], 4);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool up = lane & 2;
        s[i] = (up ? s[4 + i] : s[i]) + __shfl_xor_sync(0xffffffffu, up ? s[i] : s[4 + i], 2);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool up = lane & 1;
        s[i] = (up ? s[2 + i] : s[i]) + __shfl_xor_sync(0xffffffffu, up ? s[i] : s[2 + i], 1);
      }
      *reinterpret_cast<float2*>(&S.part[isq][warp & 3][2 * lane]) = make_float2(s[0], s[1]);
      __syncthreads();
      if (tid < 2 * kC) {
        const int pq = tid >> 6, t = tid & 63;
        const float ss = S.part[pq][0][t] + S.part[pq][1][t] + S.part[pq][2][t] + S.part[pq][3][t];
        S.rn[pq][t] = rsqrtf(ss + kNormEps) * (pq ? rsqrtf((float)kD) : 1.f);
      }
      __syncthreads();
      // [K^;Q^] rows (this channel's column), and for k the scaled K~^T row
      const int R0 = isq ? kC : 0;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        y[t] *= S.rn[isq][t];
        *reinterpret_cast<float*>(S.kq + f32_off(R0 + t, cqk, 128 * 128)) = umma::tf32_round(y[t]);
      }
      if (!isq) {
#pragma unroll
        for (int t4 = 0; t4 < kC / 4; ++t4) {
          const float4 e4 = *reinterpret_cast<const float4*>(&S.ebl[4 * t4]);
          *reinterpret_cast<float4*>(S.kt + f32_off(cqk, 4 * t4, 128 * 128)) =
              make_float4(umma::tf32_round(y[4 * t4] * e4.x), umma::tf32_round(y[4 * t4 + 1] * e4.y),
                          umma::tf32_round(y[4 * t4 + 2] * e4.z), umma::tf32_round(y[4 * t4 + 3] * e4.w));
        }
      }
    }
    // ---- features: v (channel tid % 128, tokens 32 * (tid / 128) ..), into TMEM
    {
      const int t0v = 32 * half;
      const __nv_bfloat16* xs = &S.raw[2][t0v][cqk];
      float vv[32];
      float x0 = __bfloat162float(xs[0]), x1 = __bfloat162float(xs[kD]), x2 = __bfloat162float(xs[2 * kD]);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float x3 = __bfloat162float(xs[(t + 3) * kD]);
        float acc = wv[0] * x0;
        acc = fmaf(wv[1], x1, acc);
        acc = fmaf(wv[2], x2, acc);
        acc = fmaf(wv[3], x3, acc);
        const bool valid = full || (P + t0v + t >= p0 && P + t0v + t < p1);
        vv[t] = valid ? umma::tf32_round(silu_fast(acc)) : 0.f;
        x0 = x1;
        x1 = x2;
        x2 = x3;
      }
      umma::tmem_st32(tlane + TM_V + t0v, vv);
    }
    // operands visible to the tensor core, then P = [K;Q] K^T
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    if (tid == 0) {
      umma::fence_after();
      const uint64_t dkq = umma::desc(smem_addr(S.kq), 16, 1024);
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
        umma::mma_tf32(tmem + TM_P, umma::adv(dkq, ko), umma::adv(dkq, ko), ID_P, s > 0);
      }
      umma::commit(&S.mma_bar);
    }
    if (!mma_wait()) break;
    // ---- A (fp32, for the solve) and M (tf32 operand) from P ----------------
    {
      float v[32];
      umma::tmem_ld32(tlane + TM_P + 32 * half, v);
      const int c0 = 32 * half;
      float bc[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 b4 = *reinterpret_cast<const float4*>(&S.b[c0 + 4 * i]);
        bc[4 * i] = b4.x; bc[4 * i + 1] = b4.y; bc[4 * i + 2] = b4.z; bc[4 * i + 3] = b4.w;
      }
      if (lrow < kC) {
        const int r = lrow;
        const float br = S.b[r], betar = S.beta[r];
        float av[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) av[i] = (c0 + i < r) ? betar * v[i] * exp_ftz(br - bc[i]) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(S.sv.A + ix(r, c0 + 4 * q)) = make_float4(av[4 * q], av[4 * q + 1], av[4 * q + 2], av[4 * q + 3]);
      } else {
        const int r = lrow - kC;
        const float br = S.b[r];
        float m[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) m[i] = (c0 + i <= r) ? umma::tf32_round(v[i] * exp_ftz(br - bc[i])) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(S.mq + f32_off(r, c0 + 4 * q, 64 * 128)) =
              make_float4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
      }
    }
    // T'' is rewritten (its tile held the previous chunk's output staging)
    for (int e = tid; e < (int)(sizeof(S.t2) / 16); e += kThreads)
      reinterpret_cast<uint4*>(S.t2)[e] = make_uint4(0u, 0u, 0u, 0u);
    umma::fence_before();
    __syncthreads();
    solve_T(S.sv.A, S.sv.X, S.sv.Y, TOut{S.tm, S.t2, S.beta, S.eb});
    umma::fence_proxy_async();
    __syncthreads();
    // the next chunk's raw rows (the solve's scratch is dead)
    if (tid == 0 && c + 1 < nch) {
      issue_raw(c + 1);
      ld_issued = c + 2;
    }
    // ---- Delta^T = V^T T^T, and [E | O1] = S^T [K;Q]^T -----------------------
    if (tid == 0) {
      umma::fence_after();
      const uint64_t dtm = umma::desc(smem_addr(S.tm), 16, 1024);
      const uint64_t dkq = umma::desc(smem_addr(S.kq), 16, 1024);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_DL, tmem + TM_V + 8 * s, umma::adv(dtm, (s >> 2) * 8192 + (s & 3) * 32), ID_N64,
                          s > 0);
#pragma unroll
      for (int s = 0; s < 16; ++s)
        umma::mma_tf32_ta(tmem + TM_E, tmem + TM_S + 8 * s, umma::adv(dkq, (s >> 2) * 16384 + (s & 3) * 32),
                          ID_N128, s > 0);
      umma::commit(&S.mma_bar);
    }
    if (!mma_wait()) break;
    // ---- Delta^T += E T''^T (tensor core), S^T <- e^{b_last} S^T (threads) ----
    if (tid == 0) {
      const uint64_t dt2 = umma::desc(smem_addr(S.t2), 16, 1024);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma::mma_tf32_ta(tmem + TM_DL, tmem + TM_E + 8 * s, umma::adv(dt2, (s >> 2) * 8192 + (s & 3) * 32), ID_N64,
                          true);
      umma::commit(&S.mma_bar);
    }
    {
      const float dec = S.eb[kC - 1];
      float v[32];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        umma::tmem_ld32(tlane + TM_S + 64 * half + 32 * k, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= dec;
        umma::tmem_st32(tlane + TM_S + 64 * half + 32 * k, v);
      }
    }
    umma::fence_before();
    if (!mma_wait()) break;
    // ---- S^T += Delta^T K~ ; O2 = Delta^T M^T --------------------------------
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
    // ---- output O = O1 diag(e^b) + O2, staged [token][dv] bf16 in t2 ---------
    {
      float o1[32], o2[32];
      umma::tmem_ld32(tlane + TM_O1 + 32 * half, o1);
      umma::tmem_ld32(tlane + TM_O2 + 32 * half, o2);
      __nv_bfloat16* ot = reinterpret_cast<__nv_bfloat16*>(S.t2);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        ot[(32 * half + i) * kD + lrow] = __float2bfloat16_rn(fmaf(o1[i], S.eb[32 * half + i], o2[i]));
    }
    // checkpoint: the state rows, 128B-swizzled, into four 16 KB boxes (32
    // columns x 128 rows) in the dead [K;Q] tile, for four tensor stores
    const int32_t cid = ckpt_slot(c);
    if (cid >= 0) {
      float v[32];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        umma::tmem_ld32(tlane + TM_S + 64 * half + 32 * k, v);
        uint8_t* box = S.kq + (2 * half + k) * 16384;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(box + lrow * 128 + ((j ^ (lrow & 7)) << 4)) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();
    if (tid == 0) {
      if (full) tma_store_2d(&omap, S.t2, h * kD, (int32_t)(t0 + (P - p0)));
      if (cid >= 0) {
        const int32_t y = (int32_t)(((int64_t)cid * a.hv + h) * kD);
#pragma unroll
        for (int k = 0; k < 4; ++k) tma_store_2d(&cmap, S.kq + k * 16384, 32 * k, y);
      }
      bulk_commit();
    }
    if (!full) {  // rows of the chunk's tokens inside the sequence: 16-byte stores
      const __nv_bfloat16* ot = reinterpret_cast<const __nv_bfloat16*>(S.t2);
      for (int e = tid; e < kC * (kD / 8); e += kThreads) {
        const int r = e / (kD / 8), ch = e % (kD / 8);
        const int64_t pos = P + r;
        if (pos >= p0 && pos < p1)
          *reinterpret_cast<uint4*>(a.out + ((t0 + pos - p0) * a.hv + h) * kD + ch * 8) =
              *reinterpret_cast<const uint4*>(ot + r * kD + ch * 8);
      }
    }
  }
  if (c < nch) {
    // a wait expired: let the copies and products in flight land first
    if (tid == 0) {
      report(a.err, GDN_DEV_ERR_TIMEOUT);
      umma::commit(&S.mma_bar);
      mbar_wait(&S.mma_bar, mph);
      for (int k = ld_done; k < ld_issued; ++k) mbar_wait(&S.ld_bar, k & 1);
    }
  } else {
    // the final state
    float v[32];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      umma::tmem_ld32(tlane + TM_S + 64 * half + 32 * k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float4*>(gS + 32 * k + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  if (tid == 0) bulk_wait_all();
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, TM_COLS);
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
                                uint32_t* dev_err, cudaStream_t s) {
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
  auto k = tc32_prefill_kernel<__nv_bfloat16>;
  const size_t smem = sizeof(Smem32) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // qkv [total][C] in boxes of 128 channels x 67 rows; out [total][hv * 128]
  // in boxes of one V head x 64 tokens; checkpoint states [slots * hv * 128
  // rows][128] fp32 in 128B-swizzled boxes of 32 x 128 (over the working pool
  // when there is no checkpoint pool: never written then)
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
  return launch_plain(k, dim3((unsigned)a.hv, (unsigned)n_seq), dim3(kThreads), smem, s, dim3(1), a, qmap, omap,
                      cmap);
}

}  // namespace gdn
