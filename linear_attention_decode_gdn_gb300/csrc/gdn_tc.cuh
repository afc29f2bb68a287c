// gdn_tc.cuh -- fifth-generation tensor-core helpers (sm_100 family): TMEM allocation,
// tcgen05.mma of kind::tf32 with shared-memory operand descriptors, commits to mbarriers,
// TMEM loads and stores, and the fences that order them with ordinary thread code.
//
// Operand tiles in shared memory use the no-swizzle K-major layout: the tile is made of
// "core matrices" of 8 rows x 16 bytes (8 x 4 fp32 values), each 128 contiguous bytes.
// Element (r, k) of a tile with row stride sbo (between groups of 8 rows) and k stride lbo
// (between groups of 4 columns) sits at  (r / 8) * sbo + (k / 4) * lbo + (r % 8) * 16 + (k % 4) * 4.
// One kind::tf32 MMA consumes K = 8 columns, i.e. two core matrices along k, so the next
// instruction starts 2 * lbo bytes further.
#pragma once

#include <cstdint>

#include "gdn_device.cuh"

namespace gdn {
namespace tc {

// ---- TMEM allocation (one warp, .sync.aligned) ------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering ----------------------------------------------------------------------------
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// ordinary shared-memory stores -> visible to the tensor core's operand reads
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- descriptors -------------------------------------------------------------------------
// Shared-memory operand descriptor, no swizzle: start address, k-direction stride (lbo) and
// 8-row-group stride (sbo), all in bytes (multiples of 16), and the fixed version bit.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::tf32 with an fp32 accumulator, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool negate_a = false) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (negate_a ? (1u << 13) : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- MMA ----------------------------------------------------------------------------------
// Called by every lane of one warp with the same (warp-uniform) operands: one elected lane
// (the lowest, so always the same one) issues the instruction. Keeping the descriptor
// arithmetic uniform lets it live in the uniform datapath, which the MMA reads its operands
// from; a single divergent thread would move every operand across per instruction.
// D[tmem] (+)= A[smem] * B[smem]^T
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T  (A: row m in lane m, column k in TMEM column k)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every MMA the elected lane issued so far has completed (same
// calling convention: the whole warp, one lane elected).
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          smem_addr(bar))
      : "memory");
}

// ---- TMA bulk loads counted on an mbarrier (whole warp, warp-uniform operands) -------------
// One elected lane announces `bytes` on `bar` (arrival + expected transaction count)...
__device__ __forceinline__ void expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .pred e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n"
      " @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}
// ... and issues the copies: global -> shared, contiguous, 16-byte aligned, a multiple of 16
// bytes, completion counted on `bar`, with an L2 cache policy.
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "{\n .reg .pred e;\n .reg .b32 l;\n elect.sync l|e, 0xffffffff;\n"
      " @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n}\n" ::"r"(
          smem_addr(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ---- TMEM <-> registers (warp w reaches lanes 32 (w % 4) .. + 31) --------------------------
__device__ __forceinline__ uint32_t lane_base(int warp) { return static_cast<uint32_t>(32 * (warp & 3)) << 16; }

// 32 lanes x 16 consecutive columns: v[i] = column col + i of this thread's lane. The load
// is asynchronous, so its wait sits in the same statement: the registers are only defined
// (for the compiler too) once it has completed.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- TF32 splitting -----------------------------------------------------------------------
// x = hi + lo exactly, hi with the low 13 mantissa bits cleared (a TF32 value), lo the rest
// (|lo| < 2^-10 |x|; the tensor core reads lo as TF32 too, leaving an error below 2^-20 |x|).
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

}  // namespace tc
}  // namespace gdn
