// Building blocks of the W4A16 kernels (the decode linear and the small-batch
// MoE): e2m1 codes times their E4M3 block scale become f16 weights, which
// enter mma.sync.m16n8k16 as the A operand (16 weight rows) against up to 8
// activation rows as B; activations are staged as f16 after a power-of-two
// rescale that puts the largest magnitude of the rescaled group in
// [2^14, 2^15).  e2m1 * E4M3 has at most 6 significant bits and lies in
// [2^-10, 2688], so the weights are exact in f16; an activation within 2^31 of
// its group's largest magnitude converts exactly (smaller ones round on the
// f16 subnormal grid, an error below 2^-39 of that magnitude); and products of
// f16 values are exact in the fp32 accumulators.
#pragma once
#include <cuda_fp16.h>

#include "nvfp4_common.cuh"

namespace nvfp4 {

__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 scale bytes -> (S_lo, S_lo) and (S_hi, S_hi) as f16x2.
__device__ __forceinline__ void scale_pair_f16(uint32_t two_bytes, uint32_t& lo, uint32_t& hi) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  lo = __byte_perm(h2, 0, 0x1010);
  hi = __byte_perm(h2, 0, 0x3232);
}

// Activation chunk (8 f16, 16 bytes) c of a 128-k block sits at chunk
// c ^ (((c >> 3) & 1) << 1): with a row stride of 16 (mod 32) bytes the four
// chunks a quarter-warp reads together fall on distinct bank groups.
__device__ __forceinline__ int xchunk(int c) { return c ^ (((c >> 3) & 1) << 1); }

__device__ __forceinline__ void cp_async_16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// Power-of-two exponent that puts a token's largest magnitude (fp32 bits) in
// [2^14, 2^15), clamped so that 2^shift and 2^-shift stay normal floats.
__device__ __forceinline__ int token_shift(unsigned int amax_bits) {
  const int sh = amax_bits ? static_cast<int>((amax_bits >> 23) & 0xFF) - 127 - 14 : 0;
  return sh < -110 ? -110 : (sh > 113 ? 113 : sh);
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// A consumer that read a ring slot with ordinary shared-memory loads releases
// it to a TMA refill (async proxy) only after this fence: without it the
// refill was seen to overwrite data that the loads had not yet returned.
__device__ __forceinline__ void fence_proxy_async_smem_read() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block clusters and named barriers.

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace nvfp4
