// Pieces shared by the chunked prefills on the 5th-generation tensor cores
// in tf32 (the GDN chain of prefill_tc32.cu and the KDA chain of
// kda_tc32.cu): the chunk geometry, the 128-byte swizzled K-major fp32
// operand layout, SiLU by one tanh.approx, warp-level tf32 products with fp32
// accuracy (split operands) and the 64 x 64 unit-lower-triangular solve of
// the chunkwise WY/UT form (Yang et al., NeurIPS 2024; Gated Delta Networks,
// ICLR 2025).  Included by one .cu file each, inside their own anonymous
// namespace, after gdn_common.cuh and umma.cuh.
#pragma once

constexpr int kC = 64;                 // chunk
constexpr int kD = 128;                // dk = dv
constexpr int kThreads = 512;          // 16 warps
constexpr int kRawRows = kC + 3;       // chunk rows plus 3 rows of conv history
constexpr int kAX = 68;                // row stride (floats) of the solve's A and X

// Byte offset of element (r, c) in a K-major swizzled fp32 tile whose
// 32-column blocks are `blk` bytes apart.
__device__ __forceinline__ uint32_t f32_off(int r, int c, uint32_t blk) {
  return (uint32_t)(c >> 5) * blk + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
         (uint32_t)((((c & 31) >> 2) ^ (r & 7)) << 4) + (uint32_t)(c & 3) * 4u;
}

__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + exp_ftz(-y)); }
// SiLU of the features by one special-function operation: sigmoid(y) =
// (1 + tanh(y / 2)) / 2 with tanh.approx.f32 (relative error about 2^-11, so
// the sigmoid's absolute error is at most about 2^-12 |tanh|, the size of the
// tf32 rounding the features take next; a float64 model of the chunk form
// shows no change in the output, row and state errors).  The features'
// SiLUs are half the special-function work of a chunk, and that unit bounds
// the features phase.
__device__ __forceinline__ float silu_tanh(float y) {
  float t;
  asm("tanh.approx.f32 %0, %1;\n" : "=f"(t) : "f"(0.5f * y));
  return y * fmaf(0.5f, t, 0.5f);
}

// element (r, c) of the solve's 64 x 64 fp32 matrices A and X
__device__ __forceinline__ int ix(int r, int c) { return r * kAX + c; }

// ---- warp-level tf32 products with fp32 accuracy -------------------------------
// mma m16n8k8 (row.col, fp32 accumulate).  Lane = 4 g + q: A holds (g, q),
// (g + 8, q), (g, q + 4), (g + 8, q + 4); B holds (q, g), (q + 4, g); C and D
// hold (g, 2q), (g, 2q + 1), (g + 8, 2q), (g + 8, 2q + 1).  Each operand is
// split x = hi + lo, both tf32 rounded to nearest, and a product is the three
// products hi hi + hi lo + lo hi: the lo lo term lies below fp32's rounding,
// so the sum carries an fp32 product.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(umma::tf32_round(x));
  lo = __float_as_uint(umma::tf32_round(x - __uint_as_float(hi)));
}
__device__ __forceinline__ void mma_m16n8k8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// one k-step D += L R: L (16 x 8) element (r, k) from la(r, k0 + k), R (8 x 8)
// element (k, c) from lb(k0 + k, c)
template <class LA, class LB>
__device__ __forceinline__ void step3(float (&d)[4], int k0, LA la, LB lb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const float a[4] = {la(g, k0 + q), la(g + 8, k0 + q), la(g, k0 + q + 4), la(g + 8, k0 + q + 4)};
  const float b[2] = {lb(k0 + q, g), lb(k0 + q + 4, g)};
  uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
  split_tf32(b[0], bh[0], bl[0]);
  split_tf32(b[1], bh[1], bl[1]);
  mma_m16n8k8(d, al, bh[0], bh[1]);
  mma_m16n8k8(d, ah, bl[0], bl[1]);
  mma_m16n8k8(d, ah, bh[0], bh[1]);
}

// ---- the 64 x 64 solve ---------------------------------------------------------
// X = (I + A)^-1 for the strictly lower 64 x 64 A (fp32, rows kAX apart),
// blockwise: the eight 8 x 8 diagonal blocks by substitution on the CUDA
// cores, then merged 8 -> 16 -> 32 -> 64 with X_ba = -X_b (A_ba X_a) on
// fp32-accurate warp-level tensor-core products; every entry of X above the
// diagonal is zero (X is cleared first), so the sums run over whole rows and
// columns.  Each entry of X is written out as T1 = rk_i X_ij beta_j and
// T2 = -rk_i X_ij beta_j e^{b_j} rk_j (tf32).  Y: 2048 floats of scratch,
// L0: 8 x 3 x 64.  512 threads (warps 8..15 wait at the first barrier while
// warps 0..7 invert the diagonal blocks; named barriers 2..5 in the last
// merge); the caller synchronises before (A complete, X cleared) and after.
struct TOut {
  uint8_t* t1;
  uint8_t* t2;
  const float* beta;
  const float* eb;
  const float* rk;
};
constexpr unsigned kTileT = 2 * 64 * 128;  // bytes of a 64 x 64 fp32 operand tile (T1, T2, M')
__device__ __forceinline__ void put_t(const TOut& o, int r, int c, float x, int line = __builtin_LINE()) {
  const uint32_t off = f32_off(r, c, 64 * 128);
  const float t = o.rk[GDN_S(r, kC)] * x * o.beta[GDN_S(c, kC)];
  tile_at<float>(o.t1, kTileT, off, line) = umma::tf32_round(t);
  tile_at<float>(o.t2, kTileT, off, line) = umma::tf32_round(-t * o.eb[c] * o.rk[c]);
}

__device__ __forceinline__ void solve_T(const float* A_, float* X_, float* Y_, float (*L0)[3][64], const TOut& to) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const auto A = GDN_SV(A_, kC * kAX);
  const auto X = GDN_SV(X_, kC * kAX);
  const auto Y = GDN_SV(Y_, 2048);
  // 8 x 8 diagonal blocks: warp w < 8 inverts block w, L = A_ww (strictly
  // lower, so L^8 = 0), as (I + L)^-1 = (I - L)(I + L^2)(I + L^4); lane l
  // holds entries (l / 4, 2 (l % 4)) and (l / 4, 2 (l % 4) + 1)
  if (warp < 8) {
    const int o = 8 * warp, i = lane >> 2, j = 2 * (lane & 3);
    const auto L2 = GDN_SV(L0[warp][0], 64);
    const auto L4 = GDN_SV(L0[warp][1], 64);
    const auto B = GDN_SV(L0[warp][2], 64);
    auto Lw = [&](int r, int c) { return A[ix(o + r, o + c)]; };
    float s0 = 0.f, s1 = 0.f;  // L^2
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float lik = Lw(i, k);
      s0 = fmaf(lik, Lw(k, j), s0);
      s1 = fmaf(lik, Lw(k, j + 1), s1);
    }
    L2[8 * i + j] = s0;
    L2[8 * i + j + 1] = s1;
    __syncwarp();
    float q0 = 0.f, q1 = 0.f, c0 = 0.f, c1 = 0.f;  // L^4 and L^3 = L L^2
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float l2 = L2[8 * i + k], l1 = Lw(i, k);
      q0 = fmaf(l2, L2[8 * k + j], q0);
      q1 = fmaf(l2, L2[8 * k + j + 1], q1);
      c0 = fmaf(l1, L2[8 * k + j], c0);
      c1 = fmaf(l1, L2[8 * k + j + 1], c1);
    }
    L4[8 * i + j] = q0;
    L4[8 * i + j + 1] = q1;
    // B = (I - L)(I + L^2) = I - L + L^2 - L^3
    B[8 * i + j] = (i == j ? 1.f : 0.f) - Lw(i, j) + s0 - c0;
    B[8 * i + j + 1] = (i == j + 1 ? 1.f : 0.f) - Lw(i, j + 1) + s1 - c1;
    __syncwarp();
    float x0 = B[8 * i + j], x1 = B[8 * i + j + 1];  // X = B + B L^4
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float bk = B[8 * i + k];
      x0 = fmaf(bk, L4[8 * k + j], x0);
      x1 = fmaf(bk, L4[8 * k + j + 1], x1);
    }
    X[ix(o + i, o + j)] = x0;
    X[ix(o + i, o + j + 1)] = x1;
    if (j <= i) put_t(to, o + i, o + j, x0);
    if (j + 1 <= i) put_t(to, o + i, o + j + 1, x1);
  }
  __syncthreads();
  // 8 -> 16 and 16 -> 32 on the CUDA cores (the tensor-core form measured
  // slower at these sizes: each product is a short chain of dependent steps)
  // 8 -> 16: pair p (rows 16p + 8 .., columns 16p ..), entry (i, j) per thread
  {
    const int p = (tid >> 6) & 3, i = (tid >> 3) & 7, j = tid & 7, o = 16 * p;
    if (tid < 256) {
      float y = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) y = fmaf(A[ix(o + 8 + i, o + k)], X[ix(o + k, o + j)], y);
      Y[tid] = y;  // Y_p[i][j] at 64 p + 8 i + j
    }
    __syncthreads();
    if (tid < 256) {
      float x = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) x = fmaf(X[ix(o + 8 + i, o + 8 + k)], Y[64 * p + 8 * k + j], x);
      X[ix(o + 8 + i, o + j)] = -x;
      put_t(to, o + 8 + i, o + j, -x);
    }
  }
  __syncthreads();
  // 16 -> 32: pair q (rows 32q + 16 .., columns 32q ..), entry (i, j) per thread
  {
    const int q = tid >> 8, i = (tid >> 4) & 15, j = tid & 15, o = 32 * q;
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) y = fmaf(A[ix(o + 16 + i, o + k)], X[ix(o + k, o + j)], y);
    Y[256 * q + 16 * i + j] = y;
    __syncthreads();
    float x = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) x = fmaf(X[ix(o + 16 + i, o + 16 + k)], Y[256 * q + 16 * k + j], x);
    X[ix(o + 16 + i, o + j)] = -x;
    put_t(to, o + 16 + i, o + j, -x);
  }
  __syncthreads();
  // 32 -> 64 on fp32-accurate warp-level tensor-core products (step3): a
  // warp carries one column tile j of X_ba through both products, since column
  // tile j of X_ba needs only column tile j of Y = A_ba X_a.
  const int g = lane >> 2, q = lane & 3;
  // 32 -> 64: warps 0..7 = (column tile j = warp % 4, row half mh = warp / 4);
  // the two warps of a column tile share Y[:, 8j ..] through a named barrier.
  // k-steps whose X_a rows lie above the tile's columns (s < j), or whose
  // X_b columns lie right of the warp's rows (s > 2 mh + 1), are zero.
  if (warp < 8) {
    const int j = warp & 3, mh = warp >> 2;
    const auto Ys = Y + (1024 + j * 256);  // Y[:, 8j ..] [32][8]
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (s >= j)
        step3(d, 8 * s, [&](int r, int k) { return A[ix(32 + 16 * mh + r, k)]; },
              [&](int k, int c) { return X[ix(k, 8 * j + c)]; });
    const int yr = 16 * mh + g;
    Ys[yr * 8 + 2 * q] = d[0];
    Ys[yr * 8 + 2 * q + 1] = d[1];
    Ys[(yr + 8) * 8 + 2 * q] = d[2];
    Ys[(yr + 8) * 8 + 2 * q + 1] = d[3];
    named_sync(2 + j, 64);
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (s <= 2 * mh + 1)
        step3(e, 8 * s, [&](int r, int k) { return X[ix(32 + 16 * mh + r, 32 + k)]; },
              [&](int k, int c) { return Ys[k * 8 + c]; });
    const int cc = 8 * j + 2 * q;
    put_t(to, 32 + yr, cc, -e[0]);
    put_t(to, 32 + yr, cc + 1, -e[1]);
    put_t(to, 40 + yr, cc, -e[2]);
    put_t(to, 40 + yr, cc + 1, -e[3]);
  }
}
