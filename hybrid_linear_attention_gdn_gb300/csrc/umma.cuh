// tcgen05 (5th-generation tensor core) helpers: shared-memory matrix
// descriptors, the kind::f16 and kind::tf32 instruction descriptors, MMA
// issue/commit (operand A from shared memory or from TMEM), TMEM allocation,
// loads and stores.  Inline PTX only.
//
// Shared-memory operand layouts used here (bf16, 128-byte swizzle):
//  * K-major tile, R rows x 64 K: row r at (r/8)*1024 + (r%8)*128 bytes, its
//    16-byte chunk k/8 stored at chunk (k/8) ^ (r%8); a wider K is stored as
//    consecutive such 64-wide blocks.  One MMA k-step (16 elements) advances
//    the descriptor start by 32 bytes inside a block.
//  * MN-major tile, K rows x MN: the same 128-byte rows, each holding 64 MN
//    elements of one k; wider MN uses further 64-wide atoms at the descriptor's
//    leading byte offset.  One MMA k-step (16 rows) advances the start by 2048.
// Both forms (and M = 128, N = 64..256) were checked against a CPU GEMM.
// An fp32 (tf32) tile uses the same bytes: a 128-byte row holds 32 elements,
// and one tf32 k-step (8 elements) is the same 32 bytes.
#pragma once
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {
namespace umma {

constexpr uint32_t kSwizzle128 = 2;
constexpr uint32_t kTmemCols = 512;  // TMEM columns of an SM

// Checked build: a TMEM access of `ncols` columns from taddr stays inside the
// SM's 512 columns, and (warp-level loads and stores, 32x32b shape) touches
// the lanes of its warp's quarter.  A failure is recorded against the
// caller's line and the access is skipped.  Always true in the normal build.
__device__ __forceinline__ bool tmem_ok([[maybe_unused]] uint32_t taddr, [[maybe_unused]] uint32_t ncols,
                                        [[maybe_unused]] bool warp_lanes, [[maybe_unused]] int line) {
#ifdef GDN_DEBUG_BOUNDS
  const uint32_t col = taddr & 0xFFFFu, lane = taddr >> 16;
  if (col + ncols > kTmemCols) {
    bounds_fail(line, 2, (long long)col + ncols - 1, kTmemCols);
    return false;
  }
  const uint32_t quarter = 32u * ((threadIdx.x >> 5) & 3u);
  if (warp_lanes ? lane != quarter : lane >= 128u) {
    bounds_fail(line, 2, lane, warp_lanes ? quarter : 128);
    return false;
  }
#endif
  return true;
}
// columns an MMA of instruction descriptor `idesc` writes (N)
__host__ __device__ constexpr uint32_t idesc_n(uint32_t idesc) { return ((idesc >> 17) & 0x3Fu) << 3; }

__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)kSwizzle128 << 61;
  return d;
}

// The descriptor of a tile `bytes` further on (a multiple of 16): only the
// start-address field changes, and it cannot carry out for shared-memory
// addresses below 256 KB.
__device__ __forceinline__ uint64_t adv(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// kind::f16 instruction descriptor: bf16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate, int line = __builtin_LINE()) {
  if (!tmem_ok(tmem_d, idesc_n(idesc), false, line)) return;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// kind::f16 instruction descriptor: fp16 A and B, fp32 D (issued by mma_bf16,
// the same instruction).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// kind::tf32 instruction descriptor: tf32 A and B (fp32 containers; the
// tensor core reads their top 19 bits), fp32 D.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) (+)= A B, A and B from shared-memory descriptors, kind::tf32 (K = 8)
__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate, int line = __builtin_LINE()) {
  if (!tmem_ok(tmem_d, idesc_n(idesc), false, line)) return;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// D (TMEM) (+)= A B with A in TMEM (M rows = lanes, K = 8 consecutive fp32
// columns from tmem_a) and B from a shared-memory descriptor, kind::tf32
__device__ __forceinline__ void mma_tf32_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            bool accumulate, int line = __builtin_LINE()) {
  if (!tmem_ok(tmem_d, idesc_n(idesc), false, line) || !tmem_ok(tmem_a, 8, false, line)) return;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// fp32 rounded to tf32 (10 explicit mantissa bits, nearest, ties away from
// zero), as an fp32 bit pattern whose low 13 bits are zero
__device__ __forceinline__ float tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the tensor core / TMA
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// whole warp: allocate ncols TMEM columns, address written to *slot
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. +31; taddr already carries the lane base in bits 16..31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32], int line = __builtin_LINE()) {
  if (!tmem_ok(taddr, 32, true, line)) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    return;
  }
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of this thread's TMEM lane, written; returns
// once the writes are done (the caller still fences before other threads or
// the tensor core read them)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32], int line = __builtin_LINE()) {
  if (!tmem_ok(taddr, 32, true, line)) return;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (as tmem_ld32)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16], int line = __builtin_LINE()) {
  if (!tmem_ok(taddr, 16, true, line)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
    return;
  }
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive fp32 columns of this thread's TMEM lane, written (as tmem_st32)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16], int line = __builtin_LINE()) {
  if (!tmem_ok(taddr, 16, true, line)) return;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// byte offset of element (row, col) in a K-major / MN-major 128B-swizzled tile
// whose 64-wide column blocks are `block_bytes` apart
__device__ __forceinline__ uint32_t sw128_off(int row, int col, uint32_t block_bytes) {
  return (uint32_t)(col >> 6) * block_bytes + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u +
         (uint32_t)((((col & 63) >> 3) ^ (row & 7)) << 4) + (uint32_t)(col & 7) * 2u;
}

// pack 8 floats to 8 bf16 (round to nearest even) in one 16-byte value
__device__ __forceinline__ uint4 pack8_bf16(const float* f) {
  uint4 u;
  __nv_bfloat162 p0 = __floats2bfloat162_rn(f[0], f[1]);
  __nv_bfloat162 p1 = __floats2bfloat162_rn(f[2], f[3]);
  __nv_bfloat162 p2 = __floats2bfloat162_rn(f[4], f[5]);
  __nv_bfloat162 p3 = __floats2bfloat162_rn(f[6], f[7]);
  u.x = *reinterpret_cast<uint32_t*>(&p0);
  u.y = *reinterpret_cast<uint32_t*>(&p1);
  u.z = *reinterpret_cast<uint32_t*>(&p2);
  u.w = *reinterpret_cast<uint32_t*>(&p3);
  return u;
}

// store one 64-element row (8 x 16-byte chunks) of a swizzled tile of
// tile_bytes bytes
__device__ __forceinline__ void store_row64(uint8_t* tile, unsigned tile_bytes, int row, const float* v64,
                                            int line = __builtin_LINE()) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const uint32_t off = (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u +
                         (uint32_t)((ch ^ (row & 7)) << 4);
    tile_at<uint4>(tile, tile_bytes, off, line) = pack8_bf16(v64 + ch * 8);
  }
}

}  // namespace umma
}  // namespace gdn
