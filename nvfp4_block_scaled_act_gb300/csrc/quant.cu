// NVFP4 quantisation kernels (the activation quant kernel of "run nvfp4 linears
// on nvfp4 activations on sm_120", section "Changes"; the global g = 448 * 6 /
// amax of "Add BF16_FP4 GEMM ... for W4A16 workloads", section "API").
//
// quant_act: HBM-bound.  Each lane owns one 16-element block: two 16-byte
// loads, the block amax on packed bf16 magnitudes, one E4M3 scale, sixteen
// conversions to e2m1 (hardware cvt), one 8-byte code store and the scale byte
// at its swizzled position.  A warp covers 512 consecutive elements of a row
// (1 KB, coalesced); rows are split into such chunks, so long rows spread over
// many warps.  (Two lanes per block computed every per-block step twice.)
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kQuantUnroll = 2;  // 512-element chunks per warp and iteration, loads issued together

// Work item = kQuantUnroll consecutive 512-element chunks of one row (padded
// rows and columns included), so one 32-bit division per item finds its row.
// The grid is persistent; each warp loads its next item while it converts
// the current one.
struct QuantItem {
  uint4 raw[kQuantUnroll][2];
};

__device__ __forceinline__ void quant_load_item(QuantItem& it, uint32_t item, uint32_t total, uint32_t groups,
                                                uint32_t chunks, const uint16_t* __restrict__ x, int64_t M,
                                                int64_t ldx, int64_t C, int lane) {
  const uint32_t r32 = item / groups;
  const uint32_t ch0 = (item - r32 * groups) * kQuantUnroll;
  const bool row_real = item < total && static_cast<int64_t>(r32) < M;
  const uint16_t* xrow = x + static_cast<int64_t>(r32) * ldx;
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) {
    const uint32_t cc = (ch0 + u) * 32 + lane;  // this lane's block
    const bool in = row_real && ch0 + u < chunks && cc < C;
    const uint4* src = reinterpret_cast<const uint4*>(xrow + static_cast<int64_t>(cc) * 16);
    it.raw[u][0] = in ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
    it.raw[u][1] = in ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Eight fp32 -> four bytes of e2m1 codes (element 2j in the low nibble of byte j).
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float (&v)[8], float r) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(__fmul_rn(v[0], r)), "f"(__fmul_rn(v[1], r)), "f"(__fmul_rn(v[2], r)), "f"(__fmul_rn(v[3], r)),
        "f"(__fmul_rn(v[4], r)), "f"(__fmul_rn(v[5], r)), "f"(__fmul_rn(v[6], r)), "f"(__fmul_rn(v[7], r)));
  return out;
}

// amax / 6 rounded to nearest even, the value an IEEE division gives, by
// Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34, 1990):
// q0 = RN(a * y) with y = RN(1/6), the remainder r = a - 6 q0 exact through one
// FMA, then RN(q0 + r y).  Checked against the oracle's IEEE division for every
// non-negative bf16 a by the quantiser tests.
__device__ __forceinline__ float div6_rn(float a) {
  const float y = 0.16666667f;  // RN(1/6)
  const float q0 = __fmul_rn(a, y);
  const float r = __fmaf_rn(-q0, 6.0f, a);
  return __fmaf_rn(r, y, q0);
}

__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, const float* __restrict__ d_global,
                                                        uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales, int64_t Mp, int64_t C,
                                                        int64_t Cp) {
  // a GEMM launched after this kernel with programmatic dependent launch may
  // set up while this one runs; it reads the codes only after this grid ends
  pdl_launch_dependents();
  // r = g / S for every E4M3 scale byte S (IEEE division, as in the block rule)
  __shared__ float r_of_s8[256];
  const float g = __ldg(d_global);
  {
    const float S = e4m3_to_f32(threadIdx.x);
    r_of_s8[threadIdx.x] = (S != 0.0f && S == S) ? __fdiv_rn(g, S) : 0.0f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint64_t pol = act_policy();  // the codes are read next by the GEMM
  const uint32_t chunks = static_cast<uint32_t>((Cp + 31) / 32);       // 512-element chunks per row
  const uint32_t groups = (chunks + kQuantUnroll - 1) / kQuantUnroll;  // items per row
  const uint32_t total = static_cast<uint32_t>(Mp) * groups;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const int64_t cpad4 = Cp / 4;
  uint32_t item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  QuantItem cur;
  quant_load_item(cur, item, total, groups, chunks, x, M, ldx, C, lane);
  for (; item < total; item += nwarps) {
    QuantItem nxt;
    quant_load_item(nxt, item + nwarps, total, groups, chunks, x, M, ldx, C, lane);
    const uint32_t r32 = item / groups;
    const uint32_t ch0 = (item - r32 * groups) * kQuantUnroll;
    const int64_t r = r32;
    const bool row_real = r < M;
    uint8_t* crow = codes + r * (K / 2);
    uint8_t* srow = scales + ((r >> 7) * cpad4) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      if (ch0 + u >= chunks) break;  // warp-uniform
      const uint32_t cc = (ch0 + u) * 32 + lane;  // scale column of this lane's block
      const bool real = row_real && cc < C;
      const uint32_t w[8] = {cur.raw[u][0].x, cur.raw[u][0].y, cur.raw[u][0].z, cur.raw[u][0].w,
                             cur.raw[u][1].x, cur.raw[u][1].y, cur.raw[u][1].z, cur.raw[u][1].w};
      // block amax on packed bf16 magnitudes (the max of bf16 values is exact;
      // like fmaxf, __hmax2 returns the other operand when one is NaN)
      __nv_bfloat162 m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t a = w[j] & 0x7FFF7FFFu;
        m[j] = *reinterpret_cast<const __nv_bfloat162*>(&a);
      }
      const __nv_bfloat162 xm =
          __hmax2(__hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3])), __hmax2(__hmax2(m[4], m[5]), __hmax2(m[6], m[7])));
      const uint32_t a01 = *reinterpret_cast<const uint32_t*>(&xm);
      const float amax = fmaxf(bf16_bits_to_f32(a01 & 0xFFFFu), bf16_bits_to_f32(a01 >> 16));
      const uint32_t s8 = f32_to_e4m3(__fmul_rn(div6_rn(amax), g));
      const float rr = r_of_s8[s8];
      if (real) {
        uint32_t packed[2] = {0u, 0u};
        if (rr != 0.0f) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              v[2 * j] = bf16_bits_to_f32(w[4 * h + j] & 0xFFFFu);
              v[2 * j + 1] = bf16_bits_to_f32(w[4 * h + j] >> 16);
            }
            packed[h] = f32x8_to_e2m1x8(v, rr);
          }
        }
        stg_v2_hint(crow + static_cast<int64_t>(cc) * 8, packed[0], packed[1], pol);
      }
      if (cc < Cp) srow[(cc >> 2) * 512 + (cc & 3)] = real ? static_cast<uint8_t>(s8) : 0;
    }
    cur = nxt;
  }
}

// amax over a bf16 matrix, folded into *bits (fp32 bit pattern; non-negative
// floats order like their bit patterns).
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ldx, unsigned int* __restrict__ bits) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gpr = cols / 8;
  for (int64_t i = tid; i < rows * gpr; i += stride) {
    const int64_t r = i / gpr, gi = i - r * gpr;
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + r * ldx + gi * 8));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(bf16_bits_to_f32(w[j] & 0xFFFFu)));
      m = fmaxf(m, fabsf(bf16_bits_to_f32(w[j] >> 16)));
    }
  }
  const int64_t rem = cols - gpr * 8;
  for (int64_t i = tid; i < rows * rem; i += stride) {
    const int64_t r = i / rem, cc = gpr * 8 + (i - r * rem);
    m = fmaxf(m, fabsf(bf16_bits_to_f32(x[r * ldx + cc])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) b = fmaxf(b, wmax[i]);
    atomicMax(bits, __float_as_uint(b));
  }
}

// In place: amax bits -> g = 2688 / amax (1 for an all-zero tensor).
__global__ void global_from_amax_kernel(float* g) {
  const float a = *g;  // holds the amax bit pattern written by amax_kernel
  *g = (a > 0.0f) ? __fdiv_rn(2688.0f, a) : 1.0f;
}

__global__ void make_alpha_kernel(const float* __restrict__ g_a, const float* __restrict__ g_w, int64_t n,
                                  float* __restrict__ alpha) {
  const float ga = g_a ? *g_a : 1.0f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    alpha[i] = __fdiv_rn(1.0f, g_a ? __fmul_rn(ga, g_w[i]) : g_w[i]);
}

__global__ void __launch_bounds__(256) reduce_max_kernel(const float* __restrict__ in, int64_t n,
                                                         float* __restrict__ out) {
  float m = -INFINITY;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, in[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) b = fmaxf(b, wmax[i]);
    *out = b;
  }
}

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, const float* d_global,
                             uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t stream) {
  const int64_t C = K / 16, Cp = (C + 3) / 4 * 4, Mp = (M + 127) / 128 * 128;
  const int64_t chunks = (Cp + 31) / 32;
  const int64_t items = Mp * ((chunks + kQuantUnroll - 1) / kQuantUnroll);  // warp work items
  if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  // persistent: 4 blocks of 8 warps per SM (the register limit at 256 threads)
  const int64_t want = (items + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  const int blocks = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
  quant_act_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(x), M, K, ldx, d_global, codes, scales,
                                               Mp, C, Cp);
  return cudaGetLastError();
}

cudaError_t launch_compute_global(const void* x, int64_t rows, int64_t cols, int64_t ldx, float* d_global,
                                  cudaStream_t stream, int num_sms) {
  cudaError_t e = cudaMemsetAsync(d_global, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t work = rows * (cols / 8 + 1);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  amax_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const uint16_t*>(x), rows, cols, ldx,
                                                           reinterpret_cast<unsigned int*>(d_global));
  global_from_amax_kernel<<<1, 1, 0, stream>>>(d_global);
  return cudaGetLastError();
}

cudaError_t launch_make_alpha(const float* d_g_a, const float* d_g_w, int64_t n, float* d_alpha,
                              cudaStream_t stream) {
  const int64_t blocks = (n + 255) / 256;
  make_alpha_kernel<<<static_cast<int>(blocks > 1024 ? 1024 : blocks), 256, 0, stream>>>(d_g_a, d_g_w, n, d_alpha);
  return cudaGetLastError();
}

cudaError_t launch_reduce_max(const float* d_in, int64_t n, float* d_out, cudaStream_t stream) {
  reduce_max_kernel<<<1, 256, 0, stream>>>(d_in, n, d_out);
  return cudaGetLastError();
}

}  // namespace nvfp4
