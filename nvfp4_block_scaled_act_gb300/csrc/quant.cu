// NVFP4 quantisation kernels (the activation quant kernel of "run nvfp4 linears
// on nvfp4 activations on sm_120", section "Changes"; the global g = 448 * 6 /
// amax of "Add BF16_FP4 GEMM ... for W4A16 workloads", section "API").
//
// quant_act: HBM-bound.  One warp handles a 256-element chunk of a row: each
// lane loads 8 bf16 with one 16-byte load, two lanes form a 16-element block
// and exchange their partial amax with a warp shuffle, both derive the same
// E4M3 scale, each converts its 8 values to e2m1 with the hardware cvt and
// stores 4 code bytes; the even lane stores the scale byte at its swizzled
// position.  Rows are split into chunks, so long rows spread over many warps.
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kQuantUnroll = 4;  // chunks per warp, loads issued together

__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, const float* __restrict__ d_global,
                                                        uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales, int64_t Mp, int64_t C,
                                                        int64_t Cp) {
  const float g = __ldg(d_global);
  const int lane = threadIdx.x & 31;
  const int64_t chunks = (Cp * 16 + 255) / 256;  // per row, padded columns included
  const int64_t total = Mp * chunks;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t cpad4 = Cp / 4;
  for (int64_t base = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kQuantUnroll;
       base < total; base += nwarps * kQuantUnroll) {
    uint4 raw[kQuantUnroll];
    int64_t rr[kQuantUnroll], cc[kQuantUnroll], kk[kQuantUnroll];
    bool real[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t item = base + u;
      const int64_t r = item / chunks;
      const int64_t ch = item - r * chunks;
      rr[u] = r;
      cc[u] = ch * 16 + (lane >> 1);
      kk[u] = ch * 256 + lane * 8;
      real[u] = (item < total) && (r < M) && (cc[u] < C);
      raw[u] = real[u] ? __ldg(reinterpret_cast<const uint4*>(x + r * ldx + kk[u])) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      float v[8];
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu);
        v[2 * j + 1] = bf16_bits_to_f32(w[j] >> 16);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const BlockScale bs = block_scale(amax, g);
      if (real[u]) {
        uint32_t packed = 0;
        if (bs.r != 0.0f) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            packed |= f32x2_to_e2m1x2(__fmul_rn(v[2 * j], bs.r), __fmul_rn(v[2 * j + 1], bs.r)) << (8 * j);
        }
        *reinterpret_cast<uint32_t*>(codes + rr[u] * (K / 2) + kk[u] / 2) = packed;
      }
      if ((lane & 1) == 0 && base + u < total && rr[u] < Mp && cc[u] < Cp)
        scales[sf_offset(rr[u], cc[u], cpad4)] = real[u] ? static_cast<uint8_t>(bs.s8) : 0;
    }
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
                             uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t C = K / 16, Cp = (C + 3) / 4 * 4, Mp = (M + 127) / 128 * 128;
  const int64_t items = Mp * ((Cp * 16 + 255) / 256);
  const int64_t want = (items + 8 * kQuantUnroll - 1) / (8 * kQuantUnroll);
  const int blocks = static_cast<int>(want < 1 ? 1 : (want > 65535 ? 65535 : want));
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
