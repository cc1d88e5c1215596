// Chunked GDN prefill on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// Same contract and chunk form as prefill.cu (TokenSpeed Qwen3.5 page, "Ciclo
// de vida de slots": block-aligned checkpoints; chunkwise WY/UT form of the
// gated delta rule), specialised for dk = dv = 128, conv width 4.
//
//   plan:     per-sequence offsets of its 64-token chunks (absolute-aligned).
//   features: one CTA per (chunk, QK head): the input tile arrives by TMA
//             tensor copies; conv1d + SiLU + L2 norm + gates
//             for the chunk's 64 tokens, written as bf16 operand images in the
//             tensor core's 128B-swizzled shared-memory layout, so the chain
//             kernel fetches each with a single bulk copy:
//               KQ image [K^ rows 0..63 ; Q^ rows 64..127] x dk (K-major),
//               V image per V head (read as the MN-major A operand of V^T),
//               g and beta per V head (fp32; rows outside the sequence get
//               zero features and g = beta = 0, which makes every chunk a
//               full 64-row chunk without changing the result).
//   chain:    one CTA per (sequence, V head) walks its chunks in order.  The
//             fp32 state S^T (dv x dk) lives in registers (one dv row per TMEM
//             lane, 64 columns per thread); a bf16 copy in shared memory is the
//             MMA operand.  Per chunk (transposed so that M = 128 throughout):
//               [K;Q] K^T             -> K K^T (A), Q K^T (masked, decayed)
//               S^T [K;Q]^T           -> S^T K^T, O1 = S^T Q^T (before T)
//               T = (I + A)^-1 diag(beta)   (fp32, CUDA cores, blocked)
//               Delta^T = (V^T - S^T K^T diag(e^b)) T^T
//                 (the WY form's U - W S with W = T diag(e^b) K, regrouped
//                 so that only T-free operands meet the state)
//               D2 = (Delta^T diag(e^{b_last - b})) K,  O2 = Delta^T (QK^T (.) Gamma)^T
//               S^T <- e^{b_last} S^T + D2,  O = O1 diag(e^b) + O2
//             Every product is one tcgen05.mma chain (bf16 in, fp32 TMEM
//             accumulators; 6 groups, 32 MMA instructions per chunk), issued
//             by one thread and completed through tcgen05.commit -> mbarrier.
//   The conv histories of checkpoints and of the final state come from the
//   history kernel of prefill.cu.
#include "gdn_common.cuh"
#include "tma.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;        // chunk
constexpr int kD = 128;       // dk = dv
constexpr int kTh = 256;      // chain / features CTA size
constexpr uint32_t kKQBytes = 2 * 128 * 128;  // [K;Q] image: 2 blocks x 128 rows x 128 B
constexpr uint32_t kVBytes = 2 * 64 * 128;    // V image: 2 atoms x 64 rows x 128 B
constexpr uint32_t kGateBytes = 2 * kC * 4;   // g[64], beta[64]

// TMEM columns.  [K;Q] K^T is double-buffered by chunk parity (TM_KQ + 64
// for odd chunks, so the next chunk's product can run while this one is
// read); S^T [K;Q]^T is one 128-column product: S^T K^T, then O1 = S^T Q^T.
constexpr uint32_t TM_KQ = 0, TM_KQ_ODD = 64, TM_SK = 128, TM_O1 = 192, TM_DL = 256, TM_O2 = 320, TM_D2 = 384,
                   TM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_kq(int c) { return (c & 1) ? TM_KQ_ODD : TM_KQ; }

struct TcArgs {
  float* ssm;
  int32_t num_slots;
  float* ck_ssm;
  int32_t ck_num_slots;
  const void* conv;
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
  const void* qkv;
  const void* a;
  const void* b;
  void* out;
  uint32_t* err;
  int32_t* chunk_base;  // [n_seq + 1]
  uint8_t* ws_kq;       // [n_chunks][hk][kKQBytes]
  uint8_t* ws_v;        // [n_chunks][hv][kVBytes]
  float* ws_gate;       // [n_chunks][hv][2][64]
  int32_t n_chunks_max;
  int32_t hk, hv, C, G;
};

__device__ __forceinline__ bool seq_ok(const TcArgs& a, int n, int64_t& t0, int64_t& len, int64_t& p0) {
  const auto cu = GDN_GV(a.cu_seqlens, a.n_seq + 1);
  t0 = cu[n];
  len = (int64_t)cu[n + 1] - t0;
  p0 = GDN_GV(a.start_pos, a.n_seq)[n];
  return !(t0 < 0 || len < 0 || t0 + len > a.total || p0 < 0);
}

__device__ __forceinline__ int n_chunks_of(int64_t p0, int64_t len) {
  if (len <= 0) return 0;
  return (int)((p0 + len + kC - 1) / kC - p0 / kC);
}

// ---------------------------------------------------------------------------
// plan: chunk_base[n] = chunks of sequences 0..n-1 (one CTA, 1024 threads)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(const TcArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.n_seq + 1023) / 1024;
  const int lo = tid * per, hi = min(a.n_seq, lo + per);
  int sum = 0;
  for (int n = lo; n < hi; ++n) {
    int64_t t0, len, p0;
    if (seq_ok(a, n, t0, len, p0)) sum += n_chunks_of(p0, len);
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  int run = (warp ? warp_sums[warp - 1] : 0) + incl - sum;  // exclusive prefix of this thread
  const auto chunk_base = GDN_GV(a.chunk_base, a.n_seq + 1);
  for (int n = lo; n < hi; ++n) {
    chunk_base[n] = run;
    int64_t t0, len, p0;
    if (seq_ok(a, n, t0, len, p0)) run += n_chunks_of(p0, len);
  }
  if (tid == 1023) chunk_base[a.n_seq] = warp_sums[31];
}

template <typename V>
__device__ __forceinline__ int seq_of_chunk(const V& base, int n_seq, int gc) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= gc) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// features: grid (n_chunks_max, hk), 256 threads, one CTA per (chunk, QK head):
// q and k of QK head hq and v of the G V heads reading it.  The CTA stages its
// input tile (3 rows before the chunk + its 64 rows) as 2 + G parts of 128
// channels (q, k, then each V head), each brought by one TMA tensor copy of
// 128 channels x 67 packed token rows; rows outside the tensor arrive as
// zeros, and the up to 3 rows just before the sequence start are then
// overwritten from the conv history (rows further out, or past the sequence
// end, only feed outputs that are zeroed).  Then each lane walks 8 consecutive
// rows of one 8-channel group (a sliding window of 4 staged rows): conv1d,
// SiLU, for q/k the row's L2 norm by a 16-lane shuffle reduction (a warp holds
// one row's 16 q groups and 16 k groups), and one 16-byte store into the
// swizzled operand image.
// ---------------------------------------------------------------------------
constexpr int kTileRows = kC + 3;
template <typename V>  // a view of bf16 elements, 8 from i on
__device__ __forceinline__ void load8(const V& xs, size_t i, const __nv_bfloat16*, float (&v)[8]) {
  const uint4 u = vec_at<const uint4>(xs, i);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <typename V>  // a view of fp32 elements, 8 from i on
__device__ __forceinline__ void load8(const V& xs, size_t i, const float*, float (&v)[8]) {
  const float4 a = vec_at<const float4>(xs, i), b = vec_at<const float4>(xs, i + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// conv1d (width 4) + SiLU of 8 channels walking 8 rows r0 .. r0+7 (tile rows
// r .. r+3 = positions P+r-3 .. P+r); zero outside the sequence.  The fast
// exponential and division are far finer than the bf16 operands they feed.
// emit(r, y) receives each row's 8 results.
template <bool kFull, typename Tact, class Emit, typename V>
__device__ __forceinline__ void conv_walk8(const V& xs, int nch, int r0, int lc, const float (&w)[8][4],
                                           int64_t P, int64_t p0, int64_t p1, Emit emit) {
  float x[4][8];
  const Tact* tag = nullptr;  // selects the element type's load8
#pragma unroll
  for (int j = 0; j < 3; ++j) load8(xs, (size_t)(r0 + j) * nch + lc, tag, x[j]);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = r0 + k;
    load8(xs, (size_t)(r + 3) * nch + lc, tag, x[(k + 3) & 3]);
    const bool valid = kFull || (P + r >= p0 && P + r < p1);  // kFull: the chunk is inside
    float y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float acc = w[c][0] * x[k & 3][c];
      acc = fmaf(w[c][1], x[(k + 1) & 3][c], acc);
      acc = fmaf(w[c][2], x[(k + 2) & 3][c], acc);
      acc = fmaf(w[c][3], x[(k + 3) & 3][c], acc);
      y[c] = valid ? __fdividef(acc, 1.f + exp_ftz(-acc)) : 0.f;
    }
    emit(r, y);
  }
}

template <typename Tact, typename Tconv>
__global__ void __launch_bounds__(kTh, 3) tc_features_kernel(const TcArgs a, const __grid_constant__ CUtensorMap qmap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char fsm_raw[];
  const int gc = blockIdx.x, hq = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const auto chunk_base = GDN_GV(a.chunk_base, a.n_seq + 1);
  if (gc >= chunk_base[a.n_seq]) return;
  const int n = seq_of_chunk(chunk_base, a.n_seq, gc);
  int64_t t0, len, p0;
  if (!seq_ok(a, n, t0, len, p0)) return;
  const int32_t slot = GDN_GV(a.slot_ids, a.n_seq)[n];
  if (slot_class(slot, a.num_slots)) return;
  const int64_t P = (p0 / kC + (gc - chunk_base[n])) * kC;  // absolute position of row 0
  const int64_t p1 = p0 + len;
  const int nparts = 2 + a.G;
  // part p: [67 rows][128 channels]; 128-byte aligned for the tensor copies
  Tact* xs = reinterpret_cast<Tact*>(fsm_raw + ((128u - (smem_addr(fsm_raw) & 127u)) & 127u));
  const auto xsv = GDN_SV(xs, (size_t)nparts * kTileRows * kD);
  uint64_t* bar = reinterpret_cast<uint64_t*>(xs + (size_t)nparts * kTileRows * kD);
  auto part = [&](int q) { return xsv + (size_t)q * kTileRows * kD; };
  auto part_chan = [&](int q) -> int {  // first global channel of part q
    return q < 2 ? (q * a.hk + hq) * kD : (2 * a.hk + hq * a.G + (q - 2)) * kD;
  };
  const auto hist = GDN_GV(reinterpret_cast<const Tconv*>(a.conv), (long long)a.num_slots * 3 * a.C) +
                    (size_t)slot * 3 * a.C;
  const auto conv_w = GDN_GV(a.conv_w, (long long)a.C * 4);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)(nparts * kTileRows * kD * sizeof(Tact)));
    const int32_t row0 = (int32_t)(t0 + (P - 3 - p0));  // packed row of tile row 0 (may be < 0)
    for (int q = 0; q < nparts; ++q)  // a box of 128 channels x 67 rows
      if (xsv.has((size_t)q * kTileRows * kD, kTileRows * kD) && GDN_SPAN_G(part_chan(q), kD, a.C))
        tma_load_2d(xs + (size_t)q * kTileRows * kD, &qmap, part_chan(q), row0, bar);
  }
  // this lane's q/k conv weights (lane l < 16: q channels 8l .. 8l+7, lane
  // 16 + l the same k channels) and the gates, while the tile lands
  const bool isq = lane < 16;
  const int lc = 8 * (lane & 15);  // channel within the part
  float w[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 w4 = vec_at<const float4>(conv_w, (size_t)(part_chan(isq ? 0 : 1) + lc + c) * 4);
    w[c][0] = w4.x; w[c][1] = w4.y; w[c][2] = w4.z; w[c][3] = w4.w;
  }
  // gates (rows outside the sequence: g = beta = 0)
  for (int e = tid; e < kC * a.G; e += kTh) {
    const int r = e % kC, gi = e / kC;
    const int h = hq * a.G + gi;
    const int64_t pos = P + r;
    float gv = 0.f, bv = 0.f;
    if (pos >= p0 && pos < p1) {
      const size_t tok = (size_t)(t0 + pos - p0);
      const float av = to_f32(GDN_GV(reinterpret_cast<const Tact*>(a.a), a.total * a.hv)[tok * a.hv + h]);
      const float bb = to_f32(GDN_GV(reinterpret_cast<const Tact*>(a.b), a.total * a.hv)[tok * a.hv + h]);
      gv = floor_log_decay(-expf(GDN_GV(a.A_log, a.hv)[h]) * softplus_f(av + GDN_GV(a.dt_bias, a.hv)[h]));
      bv = sigmoid_f(bb);
    }
    const auto gt = GDN_GV(a.ws_gate, (long long)a.n_chunks_max * a.hv * 2 * kC) + ((size_t)gc * a.hv + h) * (2 * kC);
    gt[r] = gv;
    gt[kC + r] = bv;
  }
  const bool late = !mbar_wait(bar, 0);
  if (__syncthreads_or(late)) {
    // leave only once the copies into this CTA's shared memory have landed
    if (tid == 0) {
      report(a.err, GDN_DEV_ERR_TIMEOUT);
      mbar_wait(bar, 0);
    }
    return;
  }
  // the up to 3 rows just before the sequence start come from the conv history
  {
    const int64_t lo = (P - 3 > p0 - 3) ? P - 3 : p0 - 3;
    const int64_t hi = (P + kC < p0) ? P + kC : p0;
    if (lo < hi) {
      const int per_row = nparts * (kD / 8);  // 8-channel pieces
      const int nh = (int)(hi - lo);
      for (int e = tid; e < nh * per_row; e += kTh) {
        const int64_t pos = lo + e / per_row;
        const int q = (e % per_row) / (kD / 8), c = 8 * (e % (kD / 8));
        const auto src = hist + ((size_t)(3 - (p0 - pos)) * a.C + part_chan(q) + c);
        const auto dst = part(q) + (size_t)(pos - (P - 3)) * kD + c;
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = from_f32<Tact>(to_f32(src[k]));
      }
      __syncthreads();
    }
  }
  const bool full = P >= p0 && P + kC <= p1;  // every row of the chunk is in the sequence

  // q and k: warp w walks rows 8w .. 8w+7
  {
    const auto xp = part(isq ? 0 : 1);
    const float qscale = isq ? rsqrtf((float)kD) : 1.f;
    const auto kq = GDN_GV(a.ws_kq, (long long)a.n_chunks_max * a.hk * kKQBytes) + ((size_t)gc * a.hk + hq) * kKQBytes;
    auto emit = [&](int r, float (&y)[8]) {
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(y[c], y[c], ss);
#pragma unroll
      for (int o = 8; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float sc = rsqrtf(ss + kNormEps) * qscale;
#pragma unroll
      for (int c = 0; c < 8; ++c) y[c] *= sc;
      const int R = isq ? kC + r : r;  // image rows: k^ 0..63, q^ 64..127
      vec_at<uint4>(kq, umma::sw128_off(R, lc, 128 * 128)) = umma::pack8_bf16(y);
    };
    if (full)
      conv_walk8<true, Tact>(xp, kD, 8 * warp, lc, w, P, p0, p1, emit);
    else
      conv_walk8<false, Tact>(xp, kD, 8 * warp, lc, w, P, p0, p1, emit);
  }
  // v: (8-channel group, 8-row block) items, G*16 groups per row
  {
    const int gpr = a.G * (kD / 8);
    for (int e = tid; e < 8 * gpr; e += kTh) {
      const int ch = e % gpr, rb = e / gpr;
      const int gi = ch / (kD / 8), d = 8 * (ch % (kD / 8));
      float wv[8][4];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 w4 = vec_at<const float4>(conv_w, (size_t)(part_chan(2 + gi) + d + c) * 4);
        wv[c][0] = w4.x; wv[c][1] = w4.y; wv[c][2] = w4.z; wv[c][3] = w4.w;
      }
      const auto vimg = GDN_GV(a.ws_v, (long long)a.n_chunks_max * a.hv * kVBytes) +
                        ((size_t)gc * a.hv + hq * a.G + gi) * kVBytes;
      auto emit = [&](int r, float (&y)[8]) {
        vec_at<uint4>(vimg, umma::sw128_off(r, d, 64 * 128)) = umma::pack8_bf16(y);
      };
      if (full)
        conv_walk8<true, Tact>(part(2 + gi), kD, 8 * rb, d, wv, P, p0, p1, emit);
      else
        conv_walk8<false, Tact>(part(2 + gi), kD, 8 * rb, d, wv, P, p0, p1, emit);
    }
  }
}

// ---------------------------------------------------------------------------
// chain: grid (hv, n_seq), 256 threads, one CTA per SM
// ---------------------------------------------------------------------------
constexpr int kAXStride = 68;  // row stride (floats) of the solve's A and X
struct __align__(1024) ChainSmem {
  uint8_t kq[2][kKQBytes];
  uint8_t v[2][kVBytes];
  uint8_t st[2 * 128 * 128];  // S^T bf16 operand (K-major, 2 blocks of 64 dk)
  uint8_t wt[128 * 128];      // solve scratch; -S^T K^T diag(e^b) (K-major A); O staging
  union {
    struct {
      uint8_t dt[128 * 128];   // Delta^T (K-major A: 128 dv rows x 64 tokens)
      uint8_t dtt[128 * 128];  // Delta^T diag(e^{b_last - b})
    };
    float ax[2][64 * kAXStride];  // A and X (fp32) in the solve
  };
  uint8_t tm[64 * 128];       // T (K-major B: 64 rows x 64)
  uint8_t qk[64 * 128];       // QK^T (.) Gamma (.) lower-incl
  float gates[2][2][kC];
  float b[2][kC], eb[2][kC], ebl[2][kC];  // by chunk parity
  uint64_t ld_full[2], mma_bar, kq_bar;
  uint64_t p_bar;    // Delta of the current chunk complete (its [K;Q] K^T buffer long read)
  uint64_t st_bar;   // compute warps wrote the state image and read O1 (one arrival per warp)
  uint64_t ck_bar;   // a checkpoint's tensor stores have read the Delta tiles
  uint32_t tmem_base;
};

// The chain CTA is 8 compute warps and one issue warp (warp 8: TMA loads and
// the tensor-core products that do not depend on the running state).  The
// compute warps synchronise among themselves on named barrier kCompBar.
constexpr int kIssueWarp = 8;
constexpr int kChainThreads = kTh + 32;
constexpr int kCompBar = 5;  // 1..4 are the solve's column-tile barriers
__device__ __forceinline__ void compute_sync() { named_sync(kCompBar, kTh); }

// compute threads wait (bounded) on a barrier phase, then synchronise; the
// result (no compute thread has seen a wait expire, now or before) is the
// same in every compute thread, so they all leave the chunk loop together
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, bool& bad) {
  if (!mbar_wait(bar, parity)) bad = true;
  return !named_sync_or(kCompBar, kTh, bad);
}

// Warp-level tf32 MMA (m16n8k8, fp32 accumulate).  Fragment layout: lane =
// 4 * g + t; A holds (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); B holds
// (t, g), (t + 4, g); D holds (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
// tf32 operands are the fp32 bit patterns: the MMA reads the top 19 bits
// (truncation, relative error below 2^-10, far under T's bf16 rounding).
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x); }
// Fragments of one m16n8k8 step: A = L[0..16)[k..k+8), B = R[k..k+8)[0..8).
template <class LF>
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], int k, LF L) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  a[0] = to_tf32(L(g, k + t));
  a[1] = to_tf32(L(g + 8, k + t));
  a[2] = to_tf32(L(g, k + t + 4));
  a[3] = to_tf32(L(g + 8, k + t + 4));
}
template <class RF>
__device__ __forceinline__ void frag_b(uint32_t (&b)[2], int k, RF R) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  b[0] = to_tf32(R(k + t, g));
  b[1] = to_tf32(R(k + t + 4, g));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A 16 x 8 tile product over NK k-steps of 8 from preloaded fragments.
template <int NK>
__device__ __forceinline__ void tile_mm(float (&d)[4], const uint32_t (&a)[NK][4], const uint32_t (&b)[NK][2]) {
  d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
  for (int s = 0; s < NK; ++s) mma_tf32(d, a[s], b[s]);
}

// Element (r, c) of the 64 x 64 fp32 matrices A and X: rows 68 floats apart,
// so the m16n8k8 fragment loads (lanes (g, t) at rows g, columns t, or the
// transpose) and 16-byte row stores by consecutive rows are conflict-free.
__device__ __forceinline__ int ix(int r, int c) { return r * kAXStride + c; }

// Byte offset of element (r, c) in a 64 x 64 bf16 K-major 128B-swizzled tile.
__device__ __forceinline__ uint32_t t_off(int r, int c) {
  return (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u + (uint32_t)((((c >> 3) ^ (r & 7))) << 4) +
         (uint32_t)(c & 7) * 2u;
}

struct TOut {
  uint8_t* tm;        // T = X diag(beta)
  const float* beta;  // [64]
};

// T entries (r, c), (r, c + 1) (c even) as a bf16 pair; bc is beta of the
// two columns (loaded once per lane by the caller)
__device__ __forceinline__ void put_t_pair(const TOut& o, int r, int c, float x0, float x1, const float2& bc,
                                           int line = __builtin_LINE()) {
  tile_at<__nv_bfloat162>(o.tm, 64 * 128, t_off(r, c), line) = __floats2bfloat162_rn(x0 * bc.x, x1 * bc.y);
}

// X = (I + A)^-1 for the 64 x 64 strictly lower A (fp32), written out as the
// lower triangle of T = X diag(beta) (its upper triangle stays zero).  8 x 8 diagonal blocks by substitution, then merged
// 8 -> 16 -> 32 -> 64 with X_ba = -X_b (A_ba X_a), the products on warp-level
// tf32 MMAs (T is rounded to bf16 afterwards, far coarser than tf32).  Each
// output column tile j of X_ba needs only column tile j of A_ba X_a, so a warp
// carries its tile through both products; every operand fragment is loaded
// before the warp's first product, so a phase waits on one load latency.
// Entries above the diagonal of X are never stored; reads mask them to zero.
// Y: 2048 floats of scratch.  256 threads; the caller synchronises before (A
// complete) and after.
__device__ __forceinline__ void solve_T(const float* A_, float* X_, float* Y_, const TOut& to) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const auto A = GDN_SV(A_, 64 * kAXStride);
  const auto X = GDN_SV(X_, 64 * kAXStride);
  const auto Y = GDN_SV(Y_, 2048);
  // 8 x 8 diagonal blocks: warp w, lane l < 4 = columns 2l and 2l+1 of block
  // w (two independent substitutions), written as fp32 pairs to X and bf16
  // pairs to T
  if (lane < 4) {
    const int o = 8 * warp, c0 = 2 * lane;
    float a[28];
#pragma unroll
    for (int r = 1, i = 0; r < 8; ++r)
#pragma unroll
      for (int m = 0; m < r; ++m, ++i) a[i] = A[ix(o + r, o + m)];
    const float2 bc = make_float2(to.beta[o + c0], to.beta[o + c0 + 1]);
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
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r >= c0) {
        vec_at<float2>(X, ix(o + r, o + c0)) = make_float2(x0[r], x1[r]);
        put_t_pair(to, o + r, o + c0, x0[r], x1[r], bc);
      }
  }
  compute_sync();
  // 8 -> 16: warps 0..3, block pair p (rows/cols 16p ..); M padded to 16
  if (warp < 4) {
    const int o = 16 * warp;
    const auto Ys = Y + warp * 128;
    uint32_t fa[1][4], fb[1][2], fx[1][4], fy[1][2];
    frag_a(fa[0], 0, [&](int r, int k) { return r < 8 ? A[ix(o + 8 + r, o + k)] : 0.f; });
    frag_b(fb[0], 0, [&](int k, int c) { return k >= c ? X[ix(o + k, o + c)] : 0.f; });
    frag_a(fx[0], 0, [&](int r, int k) { return (r < 8 && k <= r) ? X[ix(o + 8 + r, o + 8 + k)] : 0.f; });
    const float2 bc = make_float2(to.beta[o + 2 * t], to.beta[o + 2 * t + 1]);
    float d[4];
    tile_mm<1>(d, fa, fb);
    Ys[g * 8 + 2 * t] = d[0];
    Ys[g * 8 + 2 * t + 1] = d[1];
    __syncwarp();
    frag_b(fy[0], 0, [&](int k, int c) { return Ys[k * 8 + c]; });
    tile_mm<1>(d, fx, fy);
    X[ix(o + 8 + g, o + 2 * t)] = -d[0];
    X[ix(o + 8 + g, o + 2 * t + 1)] = -d[1];
    put_t_pair(to, o + 8 + g, o + 2 * t, -d[0], -d[1], bc);
  }
  compute_sync();
  // 16 -> 32: warps 0..3 = (pair q, column tile j)
  if (warp < 4) {
    const int o = 32 * (warp >> 1), j = warp & 1;
    const auto Ys = Y + (512 + warp * 128);
    uint32_t fa[2][4], fb[2][2], fx[2][4], fy[2][2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      frag_a(fa[s], 8 * s, [&](int r, int k) { return A[ix(o + 16 + r, o + k)]; });
      frag_b(fb[s], 8 * s, [&](int k, int c) { return k >= 8 * j + c ? X[ix(o + k, o + 8 * j + c)] : 0.f; });
      frag_a(fx[s], 8 * s, [&](int r, int k) { return k <= r ? X[ix(o + 16 + r, o + 16 + k)] : 0.f; });
    }
    const int cc = o + 8 * j + 2 * t;
    const float2 bc = make_float2(to.beta[cc], to.beta[cc + 1]);
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
    put_t_pair(to, o + 16 + g, cc, -d[0], -d[1], bc);
    put_t_pair(to, o + 24 + g, cc, -d[2], -d[3], bc);
  }
  compute_sync();
  // 32 -> 64: warps = (column tile j, row half mh); the two warps of a column
  // tile exchange their halves of Y_j = A_ba X_a[:, j] through a named
  // barrier.  Rows of X_a above 8j of column tile j are zero (k-steps skipped).
  {
    const int j = warp & 3, mh = warp >> 2;
    const auto Ys = Y + (1024 + j * 256);  // 32 x 8
    uint32_t fa[4][4], fb[4][2], fx[4][4], fy[4][2];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      if (s >= j) {
        frag_a(fa[s], 8 * s, [&](int r, int k) { return A[ix(32 + 16 * mh + r, k)]; });
        frag_b(fb[s], 8 * s, [&](int k, int c) { return k >= 8 * j + c ? X[ix(k, 8 * j + c)] : 0.f; });
      } else {
        fa[s][0] = fa[s][1] = fa[s][2] = fa[s][3] = 0u;
        fb[s][0] = fb[s][1] = 0u;
      }
      frag_a(fx[s], 8 * s, [&](int r, int k) { return k <= 16 * mh + r ? X[ix(32 + 16 * mh + r, 32 + k)] : 0.f; });
    }
    const int cc = 8 * j + 2 * t;
    const float2 bc = make_float2(to.beta[cc], to.beta[cc + 1]);
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
    put_t_pair(to, 32 + yr, cc, -d[0], -d[1], bc);
    put_t_pair(to, 40 + yr, cc, -d[2], -d[3], bc);
  }
}

template <typename Tact>
__global__ void __launch_bounds__(kChainThreads, 1)
    tc_chain_kernel(const TcArgs a, const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap cmap) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the swizzled operand tiles need 1024-byte aligned bases
  ChainSmem& S = *reinterpret_cast<ChainSmem*>(
      smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, n = blockIdx.y, hq = h / a.G;
  int64_t t0, len, p0;
  if (!seq_ok(a, n, t0, len, p0)) {
    if (h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SEQLENS);
    return;
  }
  const int32_t slot = GDN_GV(a.slot_ids, a.n_seq)[n];
  const auto out = GDN_GV(reinterpret_cast<Tact*>(a.out), a.total * a.hv * kD);
  const auto ckpt_ids = GDN_GV(a.ckpt_ids, (long long)a.n_seq * a.max_ckpt);
  const int cls = slot_class(slot, a.num_slots);
  if (cls) {
    if (cls == 2 && h == 0 && tid == 0) report(a.err, GDN_DEV_ERR_SLOT_OOB);
    for (int64_t e = tid; e < len * kD; e += kChainThreads)
      out[((t0 + e / kD) * a.hv + h) * kD + (e % kD)] = from_f32<Tact>(0.f);
    return;
  }
  const int nch = n_chunks_of(p0, len);
  const int gc0 = GDN_GV(a.chunk_base, a.n_seq + 1)[n];
  const int64_t p1 = p0 + len;

  if (tid == 0) {
    mbar_init(&S.ld_full[0], 1);
    mbar_init(&S.ld_full[1], 1);
    mbar_init(&S.mma_bar, 1);
    mbar_init(&S.kq_bar, 1);
    mbar_init(&S.p_bar, 1);
    mbar_init(&S.st_bar, kTh / 32);
    mbar_init(&S.ck_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) umma::tmem_alloc(&S.tmem_base, TM_COLS);
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = S.tmem_base;
  const int lrow = 32 * (warp & 3) + lane;  // TMEM lane = dv (or dk / token) row
  const int half = warp >> 2;               // which 64-column half this warp handles
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

  constexpr uint32_t ID_64_KK = umma::idesc_bf16(128, 64, false, false);
  constexpr uint32_t ID_64_MK = umma::idesc_bf16(128, 64, true, false);
  constexpr uint32_t ID_128_KM = umma::idesc_bf16(128, 128, false, true);
  constexpr uint32_t ID_128_KK = umma::idesc_bf16(128, 128, false, false);
  // operand extents of the products below: [K;Q] and S^T 2 blocks of 128 rows
  // x 128 bytes, V 2 atoms of 64 rows, the 64-token tiles 128 or 64 rows
  static_assert(sizeof(ChainSmem::kq[0]) == kKQBytes && sizeof(ChainSmem::v[0]) == kVBytes, "operand tiles");
  static_assert(sizeof(ChainSmem::st) == 2 * 16384 && sizeof(ChainSmem::wt) == 16384, "operand tiles");
  static_assert(sizeof(ChainSmem::tm) == 8192 && sizeof(ChainSmem::qk) == 8192, "operand tiles");
  static_assert(TM_D2 + 128 <= TM_COLS && TM_O2 + 64 <= TM_D2, "TMEM regions");
  // bf16 outputs: the output tiles and checkpoints leave by TMA tensor stores
  // (fp32 outputs stage 32 KB, which overlaps the checkpoint boxes)
  constexpr bool kTmaStores = sizeof(Tact) == 2;
  // checkpoint slot of a block boundary at the end of chunk c (-1: none).
  // The block is kpc chunks (the host checks it is a multiple of 64 tokens);
  // chunk c ends at the absolute chunk boundary p0 / 64 + c + 1, a block
  // boundary when q = (p0 / 64) mod kpc + c + 1 is a multiple of kpc, with
  // checkpoint index q / kpc - 1; a last chunk cut short ends on none.
  const int kpc = a.ckpt_block / kC;
  const bool kpc_pow2 = (kpc & (kpc - 1)) == 0;
  const int kpc_sh = __ffs(kpc) - 1;
  const int q0 = (int)((p0 / kC) % kpc);
  const bool last_full = (p1 & (kC - 1)) == 0;
  auto ckpt_slot = [&](int c) -> int32_t {
    if (c == nch - 1 && !last_full) return -1;
    const int q = q0 + c + 1;
    const int rem = kpc_pow2 ? (q & (kpc - 1)) : q % kpc;
    if (rem != 0) return -1;
    const int idx = (kpc_pow2 ? (q >> kpc_sh) : q / kpc) - 1;
    if (idx >= a.max_ckpt) return -1;
    const int32_t id = ckpt_ids[(size_t)n * a.max_ckpt + idx];
    return slot_class(id, a.ck_num_slots) == 0 ? id : -1;
  };
  // the four tensor stores of a checkpoint staged by the compute warps (state
  // columns 0..63 in the Delta tiles, 64..127 in the chunk's [K;Q] tile) as
  // two bulk groups, the Delta tiles' first
  auto store_ckpt = [&](int32_t cid, int buf) {
    const int32_t y = (int32_t)(((int64_t)cid * a.hv + h) * kD);
    if (!GDN_SPAN_G(y, kD, (long long)a.ck_num_slots * a.hv * kD)) return;
    tma_store_2d(&cmap, S.dt, 0, y);
    tma_store_2d(&cmap, S.dtt, 32, y);
    bulk_commit();
    tma_store_2d(&cmap, S.kq[buf], 64, y);
    tma_store_2d(&cmap, S.kq[buf] + 16384, 96, y);
    bulk_commit();
  };

  if (warp == kIssueWarp) {
    // Issue warp, one lane: operand loads one chunk ahead; [K;Q] K^T of chunk
    // c + 1 into its TMEM buffer once chunk c's Delta products are done (it
    // runs on the tensor core during chunk c's Delta conversion, which uses no
    // tensor core) and S^T [K;Q]^T of chunk c + 1 once the state leaving
    // chunk c is in its image (it runs under chunk c's output stores); each
    // chunk's pair completes on kq_bar.
    if (lane == 0 && nch > 0) {
      auto issue_load = [&](int c) {
        const int gc = gc0 + c, buf = c & 1;
        mbar_arrive_expect_tx(&S.ld_full[buf], kKQBytes + kVBytes + kGateBytes);
        const size_t okq = ((size_t)gc * a.hk + hq) * kKQBytes, ov = ((size_t)gc * a.hv + h) * kVBytes,
                     og = ((size_t)gc * a.hv + h) * (2 * kC);
        if (GDN_SPAN_G(okq, kKQBytes, (long long)a.n_chunks_max * a.hk * kKQBytes))
          bulk_g2s(S.kq[buf], a.ws_kq + okq, kKQBytes, &S.ld_full[buf]);
        if (GDN_SPAN_G(ov, kVBytes, (long long)a.n_chunks_max * a.hv * kVBytes))
          bulk_g2s(S.v[buf], a.ws_v + ov, kVBytes, &S.ld_full[buf]);
        if (GDN_SPAN_G(og, 2 * kC, (long long)a.n_chunks_max * a.hv * 2 * kC))
          bulk_g2s(S.gates[buf], a.ws_gate + og, kGateBytes, &S.ld_full[buf]);
      };
      auto issue_kq = [&](int c) {
        const uint64_t dkq = umma::desc(smem_addr(S.kq[c & 1]), 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          umma::mma_bf16(tmem + tm_kq(c), umma::adv(dkq, ko), umma::adv(dkq, ko), ID_64_KK, s > 0);
        }
      };
      int issued = 1, kq_issued = 0;
      bool ok = true;
      issue_load(0);
      ok = mbar_wait(&S.ld_full[0], 0);
      if (ok) {
        umma::fence_after();
        issue_kq(0);
      }
      for (int c = 0; c < nch && ok; ++c) {
        // O1 of chunk c, after the state entering it reached its image (and,
        // at a checkpoint, was staged for its tensor stores)
        ok = mbar_wait(&S.st_bar, c & 1);
        if (!ok) break;
        umma::fence_after();
        // S^T [K;Q]^T: S^T K^T (for this chunk's Delta) and O1 = S^T Q^T
        const uint64_t dkq = umma::desc(smem_addr(S.kq[c & 1]), 16, 1024);
        const uint64_t dst = umma::desc(smem_addr(S.st), 16, 1024);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          umma::mma_bf16(tmem + TM_SK, umma::adv(dst, ko), umma::adv(dkq, ko), ID_128_KK, s > 0);
        }
        umma::commit(&S.kq_bar);
        kq_issued = c + 1;
        const int32_t ck_prev = (kTmaStores && c > 0) ? ckpt_slot(c - 1) : -1;
        if (ck_prev >= 0) {
          store_ckpt(ck_prev, (c - 1) & 1);
          // the Delta tiles are free for chunk c's extraction ...
          bulk_wait_read_1();
          mbar_arrive(&S.ck_bar);
        }
        if (c + 1 >= nch) break;
        // ... and the [K;Q] tile for chunk c + 1's operands
        if (ck_prev >= 0) bulk_wait_read();
        // chunk c+1 into the buffer of chunk c-1, whose last reader (its state
        // update) finished before st_bar completed
        issue_load(c + 1);
        issued = c + 2;
        // [K;Q] K^T of chunk c + 1, after chunk c's Delta (its TMEM buffer was last
        // read by chunk c - 1's extraction)
        ok = mbar_wait(&S.p_bar, c & 1) && mbar_wait(&S.ld_full[(c + 1) & 1], ((c + 1) >> 1) & 1);
        if (!ok) break;
        umma::fence_after();
        issue_kq(c + 1);
      }
      // the last chunk's checkpoint
      if (ok && kTmaStores) {
        const int32_t ck_last = ckpt_slot(nch - 1);
        if (ck_last >= 0) {
          ok = mbar_wait(&S.st_bar, nch & 1);
          if (ok) store_ckpt(ck_last, (nch - 1) & 1);
        }
      }
      if (kTmaStores) bulk_wait_all();
      if (!ok) {
        report(a.err, GDN_DEV_ERR_TIMEOUT);
        // let issued loads and products land before shared memory and TMEM go away
        for (int c = (issued > 2 ? issued - 2 : 0); c < issued; ++c) mbar_wait(&S.ld_full[c & 1], (c >> 1) & 1);
        umma::commit(&S.kq_bar);
        mbar_wait(&S.kq_bar, kq_issued & 1);
      }
    }
    __syncwarp();
  } else {
    // state rows: S^T[lrow][64*half .. +64) in registers, bf16 copy as operand
    const auto gS = GDN_GV(a.ssm, (long long)a.num_slots * a.hv * kD * kD) +
                    ((((size_t)slot * a.hv + h) * kD + lrow) * kD + 64 * half);
    float sreg[64];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 v = vec_at<const float4>(gS, 4 * i);
      sreg[4 * i] = v.x;
      sreg[4 * i + 1] = v.y;
      sreg[4 * i + 2] = v.z;
      sreg[4 * i + 3] = v.w;
    }
    umma::store_row64(S.st + half * (128 * 128), 128 * 128, lrow, sreg);
    // T is lower triangular: its upper triangle is written only here
    for (int e = tid; e < 64 * 128 / 16; e += kTh) reinterpret_cast<uint4*>(S.tm)[e] = make_uint4(0u, 0u, 0u, 0u);

    // the state image and the T tiles reach the tensor core's proxy; then
    // the issue warp may read the image
    umma::fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.st_bar);
    uint32_t mph = 0, ckph = 0;
    bool prev_ck = false;  // the previous chunk wrote a checkpoint
    bool bad = false;  // this thread saw a bounded wait expire
    float* Af = S.ax[0];
    float* Xf = S.ax[1];
    const auto Av = GDN_SV(Af, 64 * kAXStride);
    float* Yf = reinterpret_cast<float*>(S.wt);

    // one warp, gates of chunk c resident: cumulative log-decay b, e^b, e^{b_last - b}
    auto chunk_decays = [&](int c) {
      const int buf = c & 1;
      float bv[2], carry = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v = S.gates[buf][0][32 * hh + lane];
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
    };
    bool alive = nch == 0 || cta_wait(&S.ld_full[0], 0, bad);
    if (nch > 0 && alive && warp == 0) chunk_decays(0);

    // Per chunk c (compute warps): the decays of chunk c + 1 are computed while
    // chunk c's state update runs; [K;Q] K^T and O1 come from the issue warp.
    for (int c = 0; c < nch && alive; ++c) {
      const int buf = c & 1;
      const int64_t P = (p0 / kC + c) * kC;
      const float* eb = S.eb[buf];
      // chunk c's operands landed (warp 0 saw it already; each thread observes
      // the copy's completion itself before reading the gates)
      if (!mbar_wait(&S.ld_full[buf], (c >> 1) & 1)) bad = true;
      if (!(alive = cta_wait(&S.kq_bar, c & 1, bad))) break;
      if (kTmaStores && prev_ck) {
        // the previous chunk's checkpoint stores have read the Delta tiles
        if (!(alive = cta_wait(&S.ck_bar, ckph, bad))) break;
        ckph ^= 1;
      }
      umma::fence_after();
      const uint32_t kq = smem_addr(S.kq[buf]), vv = smem_addr(S.v[buf]);
      const uint32_t st = smem_addr(S.st);
      // A = strict_lower(beta (.) K K^T (.) Gamma) (fp32) and the decayed,
      // masked Q K^T operand; lanes 0-63 hold K K^T rows, 64-127 Q K^T rows
      {
        const float* b = S.b[buf];
        float v[32], bc[32];
        const int c0 = 32 * half;
        // the column decays, loaded before any store so none waits on one
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 b4 = *reinterpret_cast<const float4*>(b + c0 + 4 * i);
          bc[4 * i] = b4.x;
          bc[4 * i + 1] = b4.y;
          bc[4 * i + 2] = b4.z;
          bc[4 * i + 3] = b4.w;
        }
        umma::tmem_ld32(tlane + tm_kq(c) + 32 * half, v);
        if (lrow < kC) {
          const int r = lrow;
          const float br = b[r], betar = S.gates[buf][1][r];
          float av[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int cc = c0 + i;
            av[i] = cc < r ? betar * v[i] * exp_ftz(br - bc[i]) : 0.f;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            vec_at<float4>(Av, ix(r, c0 + 4 * q)) = make_float4(av[4 * q], av[4 * q + 1], av[4 * q + 2], av[4 * q + 3]);
        } else {
          const int t = lrow - kC;
          const float bt = b[t];
          float m[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int cc = c0 + i;
            m[i] = cc <= t ? v[i] * exp_ftz(bt - bc[i]) : 0.f;
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int cch = 4 * half + ch;
            tile_at<uint4>(S.qk, sizeof(S.qk), (t >> 3) * 1024 + (t & 7) * 128 + ((cch ^ (t & 7)) << 4)) =
                umma::pack8_bf16(m + 8 * ch);
          }
        }
      }
      // the previous chunk's output tile (its tensor store's source is the
      // solve's scratch) has been read
      if (kTmaStores && tid == 0) bulk_wait_read();
      umma::fence_before();
      compute_sync();
      // T = X diag(beta) as a bf16 K-major tile
      solve_T(Af, Xf, Yf, TOut{S.tm, S.gates[buf][1]});
      umma::fence_proxy_async();
      compute_sync();
      // Delta^T = (V^T - S^T K^T diag(e^b)) T^T, as two products into one
      // accumulator: V^T T^T now, and (-S^T K^T diag(e^b)) T^T once its bf16
      // K-major image (128 dv rows x 64 tokens, in the solve's scratch tile)
      // is written; S^T K^T came with O1
      if (tid == 0) {
        umma::fence_after();
        const uint64_t dv = umma::desc(vv, 64 * 128, 1024), dtm = umma::desc(smem_addr(S.tm), 16, 1024);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          umma::mma_bf16(tmem + TM_DL, umma::adv(dv, s * 2048), umma::adv(dtm, s * 32), ID_64_MK, s > 0);
      }
      {
        float v[32];
        umma::tmem_ld32(tlane + TM_SK + 32 * half, v);
        float e[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 e4 = *reinterpret_cast<const float4*>(eb + 32 * half + 4 * i);
          e[4 * i] = e4.x;
          e[4 * i + 1] = e4.y;
          e[4 * i + 2] = e4.z;
          e[4 * i + 3] = e4.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = -v[i] * e[i];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int cch = 4 * half + ch;
          tile_at<uint4>(S.wt, sizeof(S.wt), (lrow >> 3) * 1024 + (lrow & 7) * 128 + ((cch ^ (lrow & 7)) << 4)) =
              umma::pack8_bf16(v + 8 * ch);
        }
      }
      umma::fence_proxy_async();
      umma::fence_before();
      compute_sync();
      if (tid == 0) {
        umma::fence_after();
        const uint64_t dsk = umma::desc(smem_addr(S.wt), 16, 1024), dtm = umma::desc(smem_addr(S.tm), 16, 1024);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          umma::mma_bf16(tmem + TM_DL, umma::adv(dsk, s * 32), umma::adv(dtm, s * 32), ID_64_KK, true);
        umma::commit(&S.mma_bar);
        umma::commit(&S.p_bar);
      }
      if (!(alive = cta_wait(&S.mma_bar, mph, bad))) break;
      mph ^= 1;
      umma::fence_after();
      // Delta^T to bf16, and its columns scaled by e^{b_last - b}
      {
        const float* ebl = S.ebl[buf];
        float d[32], dd[32];
        umma::tmem_ld32(tlane + TM_DL + 32 * half, d);
#pragma unroll
        for (int i = 0; i < 32; ++i) dd[i] = d[i] * ebl[32 * half + i];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int cch = 4 * half + ch;
          const uint32_t off = (lrow >> 3) * 1024 + (lrow & 7) * 128 + ((cch ^ (lrow & 7)) << 4);
          tile_at<uint4>(S.dt, sizeof(S.dt), off) = umma::pack8_bf16(d + 8 * ch);
          tile_at<uint4>(S.dtt, sizeof(S.dtt), off) = umma::pack8_bf16(dd + 8 * ch);
        }
      }
      umma::fence_proxy_async();
      umma::fence_before();
      compute_sync();
      // D2 = Delta~^T K ; O2 = Delta^T (QK^T Gamma)^T ; chunk c + 1's decays
      // (warp 4) meanwhile
      if (tid == 0) {
        umma::fence_after();
        const uint64_t ddt = umma::desc(smem_addr(S.dt), 16, 1024), ddtt = umma::desc(smem_addr(S.dtt), 16, 1024);
        const uint64_t dqk = umma::desc(smem_addr(S.qk), 16, 1024), dkm = umma::desc(kq, 16384, 1024);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          umma::mma_bf16(tmem + TM_D2, umma::adv(ddtt, s * 32), umma::adv(dkm, s * 2048), ID_128_KM, s > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          umma::mma_bf16(tmem + TM_O2, umma::adv(ddt, s * 32), umma::adv(dqk, s * 32), ID_64_KK, s > 0);
        umma::commit(&S.mma_bar);
      } else if (warp == 4 && c + 1 < nch) {
        if (__all_sync(0xffffffffu, mbar_wait(&S.ld_full[(c + 1) & 1], ((c + 1) >> 1) & 1)))
          chunk_decays(c + 1);
        else
          bad = true;
      }
      if (!(alive = cta_wait(&S.mma_bar, mph, bad))) break;
      mph ^= 1;
      umma::fence_after();
      // S^T <- e^{b_last} S^T + D2; O1 read (the next chunk's S^T [K;Q]^T
      // overwrites it); the state image and any checkpoint staging; then
      // st_bar, so that the issue warp's next product runs under the output
      // staging O = O1 diag(e^b) + O2
      float o1[32];
      {
        const float dec = eb[kC - 1];
        float d2[32];
        umma::tmem_ld32(tlane + TM_D2 + 64 * half, d2);
#pragma unroll
        for (int i = 0; i < 32; ++i) sreg[i] = fmaf(dec, sreg[i], d2[i]);
        umma::tmem_ld32(tlane + TM_D2 + 64 * half + 32, d2);
#pragma unroll
        for (int i = 0; i < 32; ++i) sreg[32 + i] = fmaf(dec, sreg[32 + i], d2[i]);
        umma::tmem_ld32(tlane + TM_O1 + 32 * half, o1);
      }
      umma::store_row64(S.st + half * (128 * 128), 128 * 128, lrow, sreg);
      // checkpoint slot of a block boundary at this chunk's end (-1: none)
      const int32_t cid = ckpt_slot(c);
      prev_ck = cid >= 0;
      if (cid >= 0) {
        if (kTmaStores) {
          // the fp32 rows, 128B-swizzled, into four 16 KB boxes (32 columns x
          // 128 rows): columns 0..63 in the Delta tiles, 64..127 in chunk c's
          // [K;Q] tile, both dead now; the issue warp writes them out with
          // four tensor stores after st_bar (instead of 512-byte-strided row
          // stores) and holds both tiles until the stores have read them
          // (the dt and dtt tiles are adjacent: two 16 KB boxes from dt)
          static_assert(offsetof(ChainSmem, dtt) == offsetof(ChainSmem, dt) + 16384, "adjacent Delta tiles");
          uint8_t* box = half ? S.kq[buf] : S.dt;
#pragma unroll
          for (int bl = 0; bl < 2; ++bl)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              tile_at<float4>(box, 2 * 16384, bl * 16384 + lrow * 128 + ((j ^ (lrow & 7)) << 4)) =
                  make_float4(sreg[32 * bl + 4 * j], sreg[32 * bl + 4 * j + 1], sreg[32 * bl + 4 * j + 2],
                              sreg[32 * bl + 4 * j + 3]);
        } else {
          const auto cS = GDN_GV(a.ck_ssm, (long long)a.ck_num_slots * a.hv * kD * kD) +
                          ((((size_t)cid * a.hv + h) * kD + lrow) * kD + 64 * half);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            vec_at<float4>(cS, 4 * i) = make_float4(sreg[4 * i], sreg[4 * i + 1], sreg[4 * i + 2], sreg[4 * i + 3]);
        }
      }
      // state image (and checkpoint) written, O1 read: the issue warp may
      // start chunk c + 1's O1
      umma::fence_proxy_async();
      umma::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.st_bar);
      {
        float o2[32];
        umma::tmem_ld32(tlane + TM_O2 + 32 * half, o2);
        float ebr[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 e4 = *reinterpret_cast<const float4*>(eb + 32 * half + 4 * i);
          ebr[4 * i] = e4.x;
          ebr[4 * i + 1] = e4.y;
          ebr[4 * i + 2] = e4.z;
          ebr[4 * i + 3] = e4.w;
        }
        // stage O as [token][dv] in the (now free) scratch tile; fp32 outputs
        // run on into the Delta tiles after it
        const auto ot = GDN_SV(reinterpret_cast<Tact*>(S.wt), (offsetof(ChainSmem, tm) - offsetof(ChainSmem, wt)) / sizeof(Tact));
#pragma unroll
        for (int i = 0; i < 32; ++i) ot[(32 * half + i) * kD + lrow] = from_f32<Tact>(fmaf(o1[i], ebr[i], o2[i]));
      }
      // the staged tile reaches the tensor store's proxy
      umma::fence_proxy_async();
      compute_sync();
      // a chunk inside the sequence leaves as one tensor store of its staged
      // 64 x 128 output tile
      const bool full = P >= p0 && P + kC <= p1;
      if (kTmaStores && full && tid == 0) {
        if (GDN_SPAN_G(t0 + (P - p0), kC, a.total) && GDN_SPAN_G(h * kD, kD, (long long)a.hv * kD))
          tma_store_2d(&omap, S.wt, h * kD, (int32_t)(t0 + (P - p0)));
        bulk_commit();
      }
      // otherwise output rows of the chunk's tokens: 16-byte stores of whole
      // rows (the staging tile is next written after the following chunk's
      // first barrier)
      if (!(kTmaStores && full)) {
        constexpr int EPC = 16 / sizeof(Tact), CPR = kD / EPC;
        const auto ot = GDN_SV(reinterpret_cast<const Tact*>(S.wt),
                               (offsetof(ChainSmem, tm) - offsetof(ChainSmem, wt)) / sizeof(Tact));
        for (int e = tid; e < kC * CPR; e += kTh) {
          const int r = e / CPR, ch = e % CPR;
          const int64_t pos = P + r;
          if (pos >= p0 && pos < p1)
            vec_at<uint4>(out, ((t0 + pos - p0) * a.hv + h) * kD + ch * EPC) = vec_at<const uint4>(ot, r * kD + ch * EPC);
        }
      }
    }
    if (!alive) {
      if (tid == 0) report(a.err, GDN_DEV_ERR_TIMEOUT);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        vec_at<float4>(gS, 4 * i) = make_float4(sreg[4 * i], sreg[4 * i + 1], sreg[4 * i + 2], sreg[4 * i + 3]);
    }
  }
  // the tensor stores have landed before the CTA's shared memory goes away
  if (kTmaStores && tid == 0) bulk_wait_all();
  umma::fence_before();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, TM_COLS);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// ---------------------------------------------------------------------------
// host side (declared in prefill_tc.cuh)
// ---------------------------------------------------------------------------
struct TcLayout {
  size_t base, kq, v, gate, total;
  int32_t n_chunks_max;
};

static TcLayout tc_layout(const gdn_dims& d, int32_t n_seq, int64_t total) {
  TcLayout L;
  L.n_chunks_max = (int32_t)(total / kC + 2 * (int64_t)n_seq);
  size_t off = 0;
  L.base = off; off += align256(sizeof(int32_t) * ((size_t)n_seq + 1));
  L.kq = off; off += align256((size_t)L.n_chunks_max * d.hk * kKQBytes);
  L.v = off; off += align256((size_t)L.n_chunks_max * d.hv * kVBytes);
  L.gate = off; off += align256((size_t)L.n_chunks_max * d.hv * kGateBytes);
  L.total = off;
  return L;
}

static size_t features_smem(int G, size_t esz) {
  return (size_t)(2 + G) * kTileRows * kD * esz + 128 /* alignment */ + 16 /* mbarrier */;
}

bool prefill_tc_supported(const gdn_dims& d, const void* qkv, const void* out, const gdn_params& p) {
  if (d.dk != kD || d.dv != kD || d.conv_width != 4) return false;
  if (d.hv / d.hk > 8) return false;
  // the features kernel stages (64 + 3) rows of the CTA's 256 + G*128 channels
  if (features_smem(d.hv / d.hk, dtype_size(d.act_dtype)) > 227u * 1024u) return false;
  if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(p.conv_w, 16)) return false;
  return true;
}

size_t prefill_tc_workspace(const gdn_dims& d, int32_t n_seq, int64_t total) {
  return tc_layout(d, n_seq, total).total;
}

template <typename Tact, typename Tconv>
static cudaError_t launch_tc_t(const TcArgs& a, cudaStream_t s) {
  cudaError_t e = launch_plain(plan_kernel, dim3(1), dim3(1024), 0, s, dim3(1), a);
  if (e != cudaSuccess) return e;
  auto fk = tc_features_kernel<Tact, Tconv>;
  const size_t fsm = features_smem(a.G, sizeof(Tact));
  if ((e = cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm)) != cudaSuccess)
    return e;
  // qkv [total][C], boxes of 128 channels x 67 rows
  CUtensorMap qmap;
  if ((e = tensor_map_2d(&qmap, a.qkv, a.total, a.C, sizeof(Tact), kD, kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      cudaSuccess)
    return e;
  e = launch_plain(fk, dim3((unsigned)a.n_chunks_max, (unsigned)a.hk), dim3(kTh), fsm, s, dim3(1), a, qmap);
  if (e != cudaSuccess) return e;
  auto ck = tc_chain_kernel<Tact>;
  const size_t csm = sizeof(ChainSmem) + 1024;
  if ((e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm)) != cudaSuccess)
    return e;
  // out [total][hv * 128] in boxes of one V head x 64 tokens; checkpoint
  // states [slots * hv * 128 rows][128] fp32 in 128B-swizzled boxes of 32 x 128
  // (over the working pool when there is no checkpoint pool: never used then)
  CUtensorMap omap, cmap;
  if ((e = tensor_map_2d(&omap, a.out, a.total, (int64_t)a.hv * kD, sizeof(Tact), kD, kC,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  const bool has_ck = a.ck_ssm != nullptr && a.ck_num_slots > 0;
  if ((e = tensor_map_2d(&cmap, has_ck ? a.ck_ssm : a.ssm,
                         (int64_t)(has_ck ? a.ck_num_slots : a.num_slots) * a.hv * kD, kD, 4, 32, kD,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  return launch_plain(ck, dim3((unsigned)a.hv, (unsigned)a.n_seq), dim3(kChainThreads), csm, s, dim3(1), a, omap,
                      cmap);
}

cudaError_t prefill_tc_launch(const gdn_dims& d, const gdn_pool& pool, const gdn_pool& ckpt,
                              const gdn_params& p, const int32_t* slot_ids, const int32_t* cu_seqlens,
                              const int64_t* start_pos, int32_t n_seq, int64_t total,
                              const int32_t* ckpt_ids, int32_t max_ckpt, int32_t ckpt_block,
                              const void* qkv, const void* av, const void* bv, void* out,
                              void* workspace, uint32_t* dev_err, cudaStream_t s) {
  const TcLayout L = tc_layout(d, n_seq, total);
  TcArgs a;
  a.ssm = pool.ssm;
  a.num_slots = pool.num_slots;
  a.ck_ssm = ckpt.ssm;
  a.ck_num_slots = max_ckpt > 0 ? ckpt.num_slots : 0;
  a.conv = pool.conv;
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
  a.qkv = qkv;
  a.a = av;
  a.b = bv;
  a.out = out;
  a.err = dev_err;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  a.chunk_base = reinterpret_cast<int32_t*>(ws + L.base);
  a.ws_kq = ws + L.kq;
  a.ws_v = ws + L.v;
  a.ws_gate = reinterpret_cast<float*>(ws + L.gate);
  a.n_chunks_max = L.n_chunks_max;
  a.hk = d.hk;
  a.hv = d.hv;
  a.C = (int32_t)channels(d);
  a.G = d.hv / d.hk;
  if (d.act_dtype == GDN_BF16 && d.conv_dtype == GDN_BF16)
    return launch_tc_t<__nv_bfloat16, __nv_bfloat16>(a, s);
  if (d.act_dtype == GDN_BF16) return launch_tc_t<__nv_bfloat16, float>(a, s);
  return launch_tc_t<float, float>(a, s);
}

}  // namespace gdn
