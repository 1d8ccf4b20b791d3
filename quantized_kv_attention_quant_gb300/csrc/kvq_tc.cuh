// Blackwell tensor-core (tcgen05) building blocks for the prompt-chunk and
// training-read paths:
// tensor-memory allocation, shared-memory matrix descriptors, the f16 MMA with
// its commit to an mbarrier, and tensor-memory loads/stores.  Written from the
// PTX ISA's description of tcgen05 (sm_100 family).
#pragma once
#include <cstdint>

namespace kvq {
namespace tc {

// ---- tensor memory allocation (one warp, all lanes) ----
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering of tcgen05 operations around thread synchronisation ----
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- shared-memory matrix descriptor: K-major operand, 128-byte swizzle ----
// Rows of 128 bytes (64 16-bit elements of K), eight rows per 1024-byte
// swizzle atom (16-byte chunk i of row r stored at chunk i ^ (r % 8)), atoms
// stacked along M/N every `sbo` bytes.  The start address advances by 32
// bytes per 16-element step of K inside the atom.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)1 << 16;                                // leading byte offset (unused with this swizzle)
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;           // stride byte offset
  d |= (uint64_t)1 << 46;                                // descriptor version
  d |= (uint64_t)2 << 61;                                // 128-byte swizzle
  return d;
}

// ---- instruction descriptor: kind::f16, f16 A and B, f32 accumulator, both K-major ----
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                            // D format: f32
         | (0u << 7) | (0u << 10)             // A, B format: f16
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// the same with bf16 A and B (both operands must share their type)
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                            // D format: f32
         | (1u << 7) | (1u << 10)             // A, B format: bf16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A's row i in lane i, K elements 2j and
// 2j+1 of a 16-bit type packed in column j (8 columns per K step of 16)
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// the mbarrier receives one arrival when every MMA issued so far by this thread is complete
__device__ __forceinline__ void commit(uint64_t* mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar))) : "memory");
}

// ---- tensor memory <-> registers: warp w reaches lanes 32*(w % 4) .. +31 ----
__device__ __forceinline__ void ld_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
               "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st_x16(uint32_t taddr, const float (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
               "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                  "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                  "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                  "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                  "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                  "r"(__float_as_uint(v[15]))
               : "memory");
}
__device__ __forceinline__ void ld_x4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st_x1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" :: "r"(taddr), "r"(__float_as_uint(v)) : "memory");
}
__device__ __forceinline__ void st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- shared-memory store of four 8x8 16-bit matrices, transposed ----
// Register j of lane t holds elements (t / 4, 2 (t % 4) .. +1) of matrix j;
// lane 8 j + i gives the address of stored row i of matrix j, which receives
// column i of the matrix.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t smem_row_addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                                  uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
               :: "r"(smem_row_addr), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

// ---- tensor memory accelerator: a 3-D tile global -> shared ----
// `map` is the address of a CUtensorMap kernel parameter; coordinates are
// elements, innermost first; completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const void* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(smem_dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
               : "memory");
}

// 16-byte chunk `chunk` of row `r` of a K-major 128-byte-swizzled tile whose
// rows are 128 bytes (byte offset from the tile's 1024-aligned base)
__host__ __device__ constexpr uint32_t sw128_off(int r, int chunk) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4));
}

}  // namespace tc
}  // namespace kvq
