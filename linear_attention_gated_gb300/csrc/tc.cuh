// tc.cuh -- thin inline-PTX helpers for the sm_103a tensor-core path:
// TMEM allocation, tcgen05.mma (kind::tf32, FP32 accumulate), commit to an
// mbarrier, bounded mbarrier waits, TMEM loads, and the shared-memory operand
// layout the MMAs read.
//
// Operand layout (canonical "no swizzle" K-major form): a tile of R rows by C
// 4-byte elements along K is stored as 8-row x 16-byte core matrices; element
// (r, c) sits at  (r / 8) * SBO + (c / 4) * 128 + (r % 8) * 16 + (c % 4) * 4
// with SBO = (C / 4) * 128 bytes (8-row groups) and LBO = 128 bytes (the
// K-adjacent core matrix). One MMA K-step of 8 TF32 elements covers two core
// matrices, so step s starts 256 bytes further along.
// The tensor core reads TF32 by dropping the low 13 mantissa bits of an FP32
// operand; operands are therefore rounded to nearest (cvt.rna.tf32.f32) when
// they are written.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {
namespace tc {

// True in exactly one lane of the calling (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .b32 rx;\n .reg .pred px;\n elect.sync rx|px, 0xffffffff;\n selp.u32 %0, 1, 0, px;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ float round_tf32(float x) {
  uint32_t u;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
  return __uint_as_float(u);
}

// Byte offset of element (r, c) in a K-major operand tile with kcols elements along K.
__device__ __forceinline__ uint32_t kmaj(int r, int c, int kcols) {
  return (uint32_t)((r >> 3) * (kcols >> 2) * 128 + (c >> 2) * 128 + (r & 7) * 16 + (c & 3) * 4);
}

// Shared-memory matrix descriptor (no swizzle, sm_100 family version bits).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Descriptor of K-step s (8 TF32 elements) of a K-major tile with kcols along K.
__device__ __forceinline__ uint64_t kdesc(uint32_t tile_saddr, int s, int kcols) {
  return sdesc(tile_saddr + (uint32_t)s * 256u, 128u, (uint32_t)(kcols >> 2) * 128u);
}

// Instruction descriptor: kind::tf32, FP32 accumulator, K-major A and B.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool negA = false) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((negA ? 1u : 0u) << 13) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// A operand read from tensor memory (128 lanes x K columns at a_tmem).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;");
}

// Arrive on an mbarrier and raise its expected transaction count by `bytes`:
// the phase completes once the arrivals are in and that many bytes have landed.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}

// Copy engine bulk copy, global -> shared, of `bytes` bytes (a multiple of 16;
// both addresses 16-byte aligned); completion is counted on the mbarrier in
// transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

// Plain arrive (release at CTA scope) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

// Bounded wait for the phase with the given parity: gives up (returns false)
// after `limit` SM clock cycles, ~2 s at the default.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, long long limit = 1ll << 32) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// The same wait for a whole (converged) warp: lane 0 polls and the result is
// shared, so the other 31 lanes put no traffic on the mbarrier while it spins.
// Lane 0's acquire is passed on to the warp by the shuffle's warp barrier.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t mbar, uint32_t parity, long long limit = 1ll << 32) {
  uint32_t ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(mbar, parity, limit) ? 1u : 0u;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Asynchronous 16-byte global -> shared copy (bypassing L1); src_bytes < 16
// zero-fills the rest (0 copies nothing and writes zeros).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Wait until at most N of this thread's most recent cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Issue a 16-column TMEM load without waiting; tmem_wait_ld() completes it.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Wait for this thread's outstanding TMEM loads; v names the destination
// registers so the compiler does not read them before the wait.
__device__ __forceinline__ void tmem_wait_ld(float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
}

// Completes two outstanding 16-column loads (the empty statement orders the
// second array's registers after the wait).
__device__ __forceinline__ void tmem_wait_ld2(float* a, float* b) {
  tmem_wait_ld(a);
  uint32_t* r = reinterpret_cast<uint32_t*>(b);
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 16 consecutive 32-bit columns of this thread's TMEM lane (caller
// issues tcgen05.wait::st before the values are consumed by an MMA).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shape .16x128b, four repeats along the columns (16 columns of 16 lanes): register
// 2 i + j of lane l holds lane (taddr lane) + 8 j + l / 4, column (taddr column) + 4 i + l % 4.
__device__ __forceinline__ void tmem_ld16x128_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.ld.sync.aligned.16x128b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld8x2(float* a, float* b) {
  uint32_t* r = reinterpret_cast<uint32_t*>(a);
  uint32_t* s = reinterpret_cast<uint32_t*>(b);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(s[0]), "+r"(s[1]), "+r"(s[2]), "+r"(s[3]), "+r"(s[4]), "+r"(s[5]), "+r"(s[6]), "+r"(s[7])
               :: "memory");
}
// Shape .16x128b, two repeats (8 columns of 16 lanes): register 2 i + j of lane l holds lane
// (taddr lane) + 8 j + l / 4, column (taddr column) + 4 i + l % 4.
__device__ __forceinline__ void tmem_ld16x128x2_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile("tcgen05.ld.sync.aligned.16x128b.x2.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld4x2(float* a, float* b) {
  uint32_t* r = reinterpret_cast<uint32_t*>(a);
  uint32_t* s = reinterpret_cast<uint32_t*>(b);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(s[0]), "+r"(s[1]), "+r"(s[2]), "+r"(s[3])
               :: "memory");
}
__device__ __forceinline__ void tmem_st16x128(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])));
}

// 4x4 transpose among the four lanes of an aligned lane quad: on entry lane (quad base + j) holds
// row j of the block, on exit it holds column j (four shuffles; the whole warp takes part).
__device__ __forceinline__ void quad_transpose(float x[4], int lane) {
  const bool odd = lane & 1;
  float a = odd ? x[0] : x[1];
  float b = odd ? x[2] : x[3];
  a = __shfl_xor_sync(0xffffffffu, a, 1);
  b = __shfl_xor_sync(0xffffffffu, b, 1);
  if (odd) { x[0] = a; x[2] = b; } else { x[1] = a; x[3] = b; }
  const bool hi = lane & 2;
  float c = hi ? x[0] : x[2];
  float d = hi ? x[1] : x[3];
  c = __shfl_xor_sync(0xffffffffu, c, 2);
  d = __shfl_xor_sync(0xffffffffu, d, 2);
  if (hi) { x[0] = c; x[1] = d; } else { x[2] = c; x[3] = d; }
}

}  // namespace tc
}  // namespace kda
