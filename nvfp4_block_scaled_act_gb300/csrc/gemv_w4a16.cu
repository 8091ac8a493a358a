// W4A16 decode GEMM: bf16 activations (T <= 16 tokens) x NVFP4 weight read in
// place from its row-major [N, K/2] codes and 128x4-swizzled scales
// ("Add BF16_FP4 GEMM ... for W4A16 workloads", section "Summary":
// out = (a @ dequant(b, b_sf).T) * alpha; the small-batch W4A16 kernels of
// "run nvfp4 linears on nvfp4 activations on sm_120", section "Changes":
// one MMA operand carries weight rows and the other the tokens, and k is
// reordered inside 128-element blocks until a single 16-byte load of codes
// already is an MMA operand fragment;
// split-K with a fixed-order reduce, as in the FlashInfer follow-up).
//
// HBM-bound: every weight byte is read once, with 16-byte non-allocating loads.
// Tile: a CTA owns 256 weight rows x kc k-elements (grid = row blocks x k
// splits); each of its 8 warps owns 32 rows as four n8 tiles of
// mma.sync.m16n8k16 (A = tokens, B = weights).  Lane (g, t) loads 16 code bytes
// (k = 32t .. 32t+31 of a 128-k block) of row 8j + g; nibble pairs 16 bits
// apart in a code word become one bf16x2 B register exactly:
//   bits = (sign << 15) | (e1 e0 m << 6)   ==  e2m1 * 2^-126  (bf16, exact)
//   w'   = bits * bf16(S * 2^117)          ==  e2m1 * S * 2^-9 (exact)
// and the 2^-9 is undone on the fp32 accumulator.  The activations of the
// CTA's k-range are staged once in shared memory in the same k order.
#include "nvfp4_common.cuh"
#include "nvfp4_moe.h"

namespace nvfp4 {

constexpr int kGemvWarps = 8;
constexpr int kGemvRows = 32 * kGemvWarps;  // weight rows per CTA

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t e2m1x2_bits(uint32_t x) {
  return ((x & 0x00070007u) << 6) | ((x & 0x00080008u) << 12);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t scale_mult(uint32_t s8) {
  const float m = __fmul_rn(e4m3_to_f32(s8), 0x1p117f);
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(m));
  return (b << 16) | b;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// kTok16: tokens 8..15 present (T > 8).
template <bool kTok16>
__global__ void __launch_bounds__(256) gemv_w4a16_kernel(const uint16_t* __restrict__ x, int T, int64_t ldx,
                                                         const uint8_t* __restrict__ w_codes,
                                                         const uint8_t* __restrict__ w_sf, int N, int K, int kc,
                                                         const float* __restrict__ d_alpha,
                                                         uint16_t* __restrict__ out, int64_t ldo,
                                                         float* __restrict__ ws) {
  constexpr int kTokRows = kTok16 ? 16 : 8;
  extern __shared__ __align__(16) uint8_t sm[];
  const int rb = blockIdx.x;
  const int split = blockIdx.y;
  const int k_begin = split * kc;
  const int k_len = min(kc, K - k_begin);
  const int xs_stride = kc * 2 + 64;  // bytes per token row; +64 spreads rows over banks
  uint8_t* xs = sm;
  uint8_t* sfs = sm + kTokRows * xs_stride;

  // stage the scale atoms of this row block and k-range (contiguous in the 128x4 layout)
  {
    const int sf_atoms_row = K / 64;
    const int nbytes = (k_len / 64) * 512;
    const int rb128 = rb * 2;  // first 128-row block of this CTA
    for (int h = 0; h < 2; ++h) {
      if ((rb128 + h) * 128 >= ((N + 127) / 128) * 128) break;
      const uint4* src = reinterpret_cast<const uint4*>(w_sf + (static_cast<int64_t>(rb128 + h) * sf_atoms_row +
                                                                k_begin / 64) * 512);
      uint4* dst = reinterpret_cast<uint4*>(sfs + h * nbytes);
      for (int i = threadIdx.x; i < nbytes / 16; i += blockDim.x) dst[i] = __ldg(src + i);
    }
  }
  // stage the activations, permuted inside each 128-k block: element
  // 32t + 8i + r (r = 0..7) of a block goes to unit (i, t) at byte 64i + 16t,
  // position [0,4,1,5,2,6,3,7][r]
  {
    const int units = k_len / 8;
    for (int u = threadIdx.x; u < kTokRows * units; u += blockDim.x) {
      const int tok = u / units;
      const int k8 = (u - tok * units) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (tok < T) v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * ldx + k_begin + k8));
      uint4 o;
      o.x = __byte_perm(v.x, v.z, 0x5410);
      o.y = __byte_perm(v.x, v.z, 0x7632);
      o.z = __byte_perm(v.y, v.w, 0x5410);
      o.w = __byte_perm(v.y, v.w, 0x7632);
      const int kb = k8 >> 7, tt = (k8 & 127) >> 5, i = (k8 & 31) >> 3;
      *reinterpret_cast<uint4*>(xs + tok * xs_stride + kb * 256 + i * 64 + tt * 16) = o;
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int lr0 = warp * 32;  // local row of tile 0 (row lr0 + 8j + g)
  const int row0 = rb * kGemvRows + lr0;
  const uint8_t* wp[4];
  bool rv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = row0 + 8 * j + g;
    rv[j] = row < N;
    wp[j] = w_codes + static_cast<int64_t>(rv[j] ? row : 0) * (K / 2) + k_begin / 2 + 16 * t;
  }
  // scale bytes of row (lr, block c): atom c/4 of this k-range at (lr/128) * nbytes
  const int nbytes = (k_len / 64) * 512;
  int sf_off[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int lr = lr0 + 8 * j + g;
    sf_off[j] = (lr >> 7) * nbytes + (lr & 31) * 16 + ((lr & 127) >> 5) * 4 + 2 * (t & 1) + (t >> 1) * 512;
  }
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[j][c] = 0.0f;

  const int nkb = k_len / 128;
  uint4 cur[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) cur[j] = rv[j] ? ldg_stream(wp[j]) : make_uint4(0u, 0u, 0u, 0u);
  for (int kb = 0; kb < nkb; ++kb) {
    uint4 nxt[4];
    if (kb + 1 < nkb) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        nxt[j] = rv[j] ? ldg_stream(wp[j] + (kb + 1) * 64) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t mlo[4], mhi[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint16_t s2 = *reinterpret_cast<const uint16_t*>(sfs + sf_off[j] + kb * 1024);
      mlo[j] = scale_mult(s2 & 0xFFu);
      mhi[j] = scale_mult(s2 >> 8);
    }
    const uint8_t* xrow = xs + g * xs_stride + kb * 256 + t * 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 alo = *reinterpret_cast<const uint4*>(xrow + i * 64);
      uint4 ahi = make_uint4(0u, 0u, 0u, 0u);
      if (kTok16) ahi = *reinterpret_cast<const uint4*>(xrow + 8 * xs_stride + i * 64);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t a0 = h ? alo.z : alo.x;
        const uint32_t a2 = h ? alo.w : alo.y;
        const uint32_t a1 = h ? ahi.z : ahi.x;
        const uint32_t a3 = h ? ahi.w : ahi.y;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t word = (i == 0) ? cur[j].x : (i == 1) ? cur[j].y : (i == 2) ? cur[j].z : cur[j].w;
          const uint32_t m = (i < 2) ? mlo[j] : mhi[j];
          const uint32_t b0 = bf16x2_mul(e2m1x2_bits(word >> (8 * h)), m);
          const uint32_t b1 = bf16x2_mul(e2m1x2_bits(word >> (8 * h + 4)), m);
          mma_bf16_16816(acc[j], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    if (kb + 1 < nkb) {
#pragma unroll
      for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
    }
  }

  // acc[j][0..1]: token g, rows 2t, 2t+1 of tile j; acc[j][2..3]: token g + 8
  const bool direct = (gridDim.y == 1);
  const float alpha = direct ? __ldg(d_alpha) : 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = row0 + 8 * j + 2 * t;
    if (n >= N) continue;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int tok = g + 8 * hh;
      if (tok >= T) continue;
      const float v0 = acc[j][2 * hh] * 512.0f, v1 = acc[j][2 * hh + 1] * 512.0f;
      if (direct) {
        const __nv_bfloat162 o = __floats2bfloat162_rn(v0 * alpha, v1 * alpha);
        *reinterpret_cast<__nv_bfloat162*>(out + static_cast<int64_t>(tok) * ldo + n) = o;
      } else {
        *reinterpret_cast<float2*>(ws + (static_cast<int64_t>(split) * T + tok) * N + n) = make_float2(v0, v1);
      }
    }
  }
}

// out[t, n] = bf16(alpha * sum_s ws[s, t, n]), s in ascending order.
__global__ void __launch_bounds__(256) gemv_reduce_kernel(const float* __restrict__ ws, int S, int T, int N,
                                                          const float* __restrict__ d_alpha,
                                                          uint16_t* __restrict__ out, int64_t ldo) {
  const float alpha = __ldg(d_alpha);
  const int64_t total = static_cast<int64_t>(T) * N / 2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 2;
    const int tok = static_cast<int>(e / N);
    const int n = static_cast<int>(e - static_cast<int64_t>(tok) * N);
    float2 s = make_float2(0.f, 0.f);
    for (int k = 0; k < S; ++k) {
      const float2 v = *reinterpret_cast<const float2*>(ws + (static_cast<int64_t>(k) * T + tok) * N + n);
      s.x += v.x;
      s.y += v.y;
    }
    *reinterpret_cast<__nv_bfloat162*>(out + static_cast<int64_t>(tok) * ldo + n) =
        __floats2bfloat162_rn(s.x * alpha, s.y * alpha);
  }
}

GemvPlan gemv_plan(int64_t T, int64_t N, int64_t K, int num_sms) {
  GemvPlan p;
  p.row_blocks = static_cast<int>((N + kGemvRows - 1) / kGemvRows);
  const int kblocks = static_cast<int>(K / 128);
  int want = (2 * num_sms + p.row_blocks - 1) / p.row_blocks;
  if (want < 1) want = 1;
  if (want > kblocks) want = kblocks;
  const int kcb = (kblocks + want - 1) / want;
  p.kc = kcb * 128;
  p.splits = (kblocks + kcb - 1) / kcb;
  p.ws_bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * T * N * sizeof(float) : 0;
  return p;
}

template <bool kTok16>
static cudaError_t launch_gemv_t(const void* x, int64_t T, int64_t ldx, const uint8_t* w_codes, const uint8_t* w_sf,
                                 int64_t N, int64_t K, const float* d_alpha, void* out, int64_t ldo, float* ws,
                                 const GemvPlan& plan, cudaStream_t stream) {
  constexpr int kTokRows = kTok16 ? 16 : 8;
  const size_t smem = static_cast<size_t>(kTokRows) * (plan.kc * 2 + 64) + 2 * (plan.kc / 64) * 512;
  static size_t attr = 0;
  if (smem > 48 * 1024 && smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(gemv_w4a16_kernel<kTok16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  dim3 grid(plan.row_blocks, plan.splits);
  gemv_w4a16_kernel<kTok16><<<grid, 256, smem, stream>>>(static_cast<const uint16_t*>(x), static_cast<int>(T), ldx,
                                                         w_codes, w_sf, static_cast<int>(N), static_cast<int>(K),
                                                         plan.kc, d_alpha, static_cast<uint16_t*>(out), ldo, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || plan.splits == 1) return e;
  const int64_t pairs = T * N / 2;
  int64_t blocks = (pairs + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  gemv_reduce_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(ws, plan.splits, static_cast<int>(T),
                                                                   static_cast<int>(N), d_alpha,
                                                                   static_cast<uint16_t*>(out), ldo);
  return cudaGetLastError();
}

cudaError_t launch_gemv_w4a16(const void* x, int64_t T, int64_t ldx, const uint8_t* w_codes, const uint8_t* w_sf,
                              int64_t N, int64_t K, const float* d_alpha, void* out, int64_t ldo, float* ws,
                              const GemvPlan& plan, cudaStream_t stream) {
  if (T > 8) return launch_gemv_t<true>(x, T, ldx, w_codes, w_sf, N, K, d_alpha, out, ldo, ws, plan, stream);
  return launch_gemv_t<false>(x, T, ldx, w_codes, w_sf, N, K, d_alpha, out, ldo, ws, plan, stream);
}

}  // namespace nvfp4

// ---------------------------------------------------------------------------
// Allocation-free variant of the W4A16 decode GEMM.
//
// Some callers cannot allocate device memory when they run a decode GEMM: a
// runtime that owns every byte of the GPU through its own pool and forbids
// side allocations, code already running inside stream capture of a CUDA
// graph where a cudaMalloc would break the capture, or a plugin host that
// hands out only its inputs and outputs.  For them this entry point keeps the
// split-K partial sums in a fixed array compiled into the library instead of
// a caller-sized workspace.  The array lives in every GPU that loads the
// library until the process exits.  In host code its name is only a stand-in
// for the device array, so the device address is looked up once per device
// (with that device current) and passed to the kernels.
// ---------------------------------------------------------------------------
#include <mutex>

#include "nvfp4.h"

namespace nvfp4 {

constexpr size_t kStaticScratchBytes = size_t(6) << 20;  // 6 MiB of fp32 partials
static __device__ __align__(256) float g_w4a16_static_scratch[kStaticScratchBytes / sizeof(float)];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_static_mu;
float* g_static_ptr[kMaxScratchDevices] = {};
int g_static_sms[kMaxScratchDevices] = {};

// Device address of the static scratch on the current device (looked up on
// the first call per device) and that device's SM count.
nvfp4_status static_scratch(float** ptr, int* sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return NVFP4_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    if (major != 10 || minor != 3) return NVFP4_ERR_NO_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_w4a16_static_scratch) != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
    g_static_ptr[dev] = static_cast<float*>(p);
    g_static_sms[dev] = count;
  }
  *ptr = g_static_ptr[dev];
  *sms = g_static_sms[dev];
  return NVFP4_OK;
}
}  // namespace

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_linear_w4a16_noalloc(const void* x, int64_t T, int64_t ldx, const uint8_t* w_codes,
                                                   const uint8_t* w_sf, int64_t N, int64_t K, const float* d_alpha,
                                                   void* out, int64_t ldo, nvfp4_stream_t stream) {
  using namespace nvfp4;
  if (T < 0 || N <= 0 || K <= 0 || ldx < K || ldo < N) return NVFP4_ERR_INVALID_ARG;
  if (T > 16 || N % 8 != 0 || K % 128 != 0 || N > (1LL << 30) || K > (1LL << 24))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return NVFP4_OK;
  if (!x || !w_codes || !w_sf || !d_alpha || !out) return NVFP4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_codes) & 15u) ||
      (reinterpret_cast<uintptr_t>(w_sf) & 15u) || (ldx % 8) != 0 || (ldo % 2) != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 3u))
    return NVFP4_ERR_MISALIGNED;
  float* scratch = nullptr;
  int sms = 0;
  const nvfp4_status st = static_scratch(&scratch, &sms);
  if (st != NVFP4_OK) return st;
  const GemvPlan plan = gemv_plan(T, N, K, sms);
  if (plan.ws_bytes > kStaticScratchBytes) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
  return launch_gemv_w4a16(x, T, ldx, w_codes, w_sf, N, K, d_alpha, out, ldo, plan.ws_bytes ? scratch : nullptr,
                           plan, stream) == cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}
