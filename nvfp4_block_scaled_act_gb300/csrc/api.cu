// C ABI of the NVFP4 library (include/nvfp4.h): argument checks, TMA
// descriptor encoding, workspace carving and kernel launches.  No call
// allocates device memory or synchronises the host (except
// nvfp4_device_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "nvfp4.h"
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_moe.h"

// Device status word: set by kernels (pipeline timeout, bad expert id), read
// and cleared by nvfp4_device_status.  One per device context.
__device__ int g_nvfp4_device_status;

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool ok = false;
  int sms = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

const DeviceInfo* device_info() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    d.probed = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess && prop.major == 10 && prop.minor == 3) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_nvfp4_device_status) == cudaSuccess) {
        d.status = static_cast<int*>(p);
        d.sms = prop.multiProcessorCount;
        d.ok = true;
      }
    }
  }
  return d.ok ? &d : nullptr;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline nvfp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

// Codes of a W4A16 weight: boxes of 64 bytes (one 128-k block) x box_rows
// rows, no swizzle; rows past the end read as zero codes.
bool make_gemv_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

MoELayoutBytes moe_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk) {
  MoELayoutBytes L{};
  const int64_t R = T * topk;
  const int bm = moe_row_block(T, H, E, topk);
  const int64_t p_max = (R + E * (bm - 1) + bm - 1) / bm * bm;
  const int64_t chunk = nvfp4::moe_align_chunk(R);
  const int64_t nchunks = (R + chunk - 1) / chunk;
  L.p_max = p_max;
  L.bm = bm;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.n_tiles = take(sizeof(int32_t));
  L.row_map = take(sizeof(int32_t) * p_max);
  L.tile_expert = take(sizeof(int32_t) * (p_max / 128));
  L.pos = take(sizeof(int32_t) * (R > 0 ? R : 1));
  L.hist = take(sizeof(int32_t) * (nchunks > 0 ? nchunks : 1) * E);
  L.ids = take(sizeof(int32_t) * (R > 0 ? R : 1));
  L.amax = take(sizeof(unsigned int) * E);
  L.a1_codes = take(static_cast<size_t>(p_max) * (H / 2));
  L.a1_sf = take(static_cast<size_t>(p_max) * ((H / 16 + 3) / 4 * 4));
  L.h_codes = take(static_cast<size_t>(p_max) * (I / 2));
  L.h_sf = take(static_cast<size_t>(p_max) * ((I / 16 + 3) / 4 * 4));
  L.y = take(sizeof(float) * static_cast<size_t>(T) * H);
  L.total = off;
  return L;
}

MoEWorkspace moe_carve(void* base, const MoELayoutBytes& L) {
  uint8_t* b = static_cast<uint8_t*>(base);
  MoEWorkspace w;
  w.counts = reinterpret_cast<int32_t*>(b + L.counts);
  w.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  w.n_tiles = reinterpret_cast<int32_t*>(b + L.n_tiles);
  w.row_map = reinterpret_cast<int32_t*>(b + L.row_map);
  w.tile_expert = reinterpret_cast<int32_t*>(b + L.tile_expert);
  w.pos = reinterpret_cast<int32_t*>(b + L.pos);
  w.hist = reinterpret_cast<int32_t*>(b + L.hist);
  w.ids = reinterpret_cast<int32_t*>(b + L.ids);
  w.amax = reinterpret_cast<unsigned int*>(b + L.amax);
  w.a1_codes = b + L.a1_codes;
  w.a1_sf = b + L.a1_sf;
  w.h_codes = b + L.h_codes;
  w.h_sf = b + L.h_sf;
  w.y = reinterpret_cast<float*>(b + L.y);
  w.p_max = L.p_max;
  w.bm = L.bm;
  return w;
}

// Up to this many routes per expert on average, MoE down adds its rows into y
// with vector reductions from registers (kEpiDownDirect) instead of staged
// 512-byte bulk reduce-adds (kEpiDownSum).
constexpr int64_t kDirectDownRoutesPerExpert = 32;

// grouped GEMM launch over the permuted rows of the MoE workspace; with 256-row
// segments (w.bm) gate_up and down run on CTA pairs
static nvfp4_status launch_grouped(int mode, const uint8_t* a_codes, const uint8_t* a_sf, int64_t p_max, int64_t K,
                                   const uint8_t* b_codes, const uint8_t* b_sf, int64_t b_rows_per_expert, int64_t E,
                                   int64_t n_tiles, const MoEWorkspace& w, GemmParams p, const DeviceInfo* dev,
                                   cudaStream_t stream) {
  GemmMaps maps = {};
  if (!make_codes_map(&maps.a, a_codes, p_max, K / 2)) return NVFP4_ERR_CUDA;
  if (!make_codes_map(&maps.b, b_codes, E * b_rows_per_expert, K / 2)) return NVFP4_ERR_CUDA;
  p.sfa = a_sf;
  p.sfb = b_sf;
  p.K = static_cast<int>(K);
  p.kblocks = static_cast<int>((K + 255) / 256);
  p.sf_atoms = static_cast<int>(K / 64);
  p.n_tiles = static_cast<int>(n_tiles);
  p.d_m_tiles = w.n_tiles;
  p.tile_expert = w.tile_expert;
  p.row_map = w.row_map;
  p.b_rows_per_expert = static_cast<int>(b_rows_per_expert);
  p.b_rows_total = static_cast<int>(E * b_rows_per_expert);
  p.status = dev->status;
  if (w.bm == 256 && (mode == kEpiGatedQuant || mode == kEpiDownSum)) {
    // CTA pairs on 256-row tiles of one expert; down then covers 256 columns
    // per tile (H % 256 == 0 when the layout pads to 256)
    if (mode == kEpiDownSum) p.n_tiles = static_cast<int>(n_tiles / 2);
    const int64_t pair_tiles = (p_max / 256) * p.n_tiles;
    const int64_t pairs = pair_tiles < dev->sms / 2 ? (pair_tiles < 1 ? 1 : pair_tiles) : dev->sms / 2;
    return cuda_status(launch_gemm(mode == kEpiGatedQuant ? kLaunchPairGated : kLaunchPairDown, maps, p,
                                   static_cast<int>(2 * pairs), stream));
  }
  const int64_t tiles_max = (p_max / 128) * n_tiles;
  const int grid = static_cast<int>(tiles_max < dev->sms ? (tiles_max < 1 ? 1 : tiles_max) : dev->sms);
  return cuda_status(launch_gemm(mode, maps, p, grid, stream));
}

// One CTA whose pipeline wait nobody completes: the bounded mbarrier wait of
// the kernels gives up after kWaitLimitCycles (about a second) and records
// kStatusTimeout; the CTA then returns normally.
__global__ void selftest_wait_timeout_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, status);
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(int s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case NVFP4_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4_ERR_BAD_EXPERT_ID: return "expert id out of range";
    case NVFP4_ERR_NO_DEVICE: return "no sm_103 device is current";
    default: return "unknown status";
  }
}

int nvfp4_version(void) { return 100; }

size_t nvfp4_scale_bytes(int64_t rows, int64_t k) {
  if (rows <= 0 || k <= 0) return 0;
  const int64_t C = k / 16;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((C + 3) / 4 * 4);
}

nvfp4_status nvfp4_compute_global(const void* x, int64_t rows, int64_t cols, int64_t ldx, float* d_global,
                                  nvfp4_stream_t stream) {
  if (!x || !d_global || rows < 0 || cols <= 0 || ldx < cols) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx % 8) != 0) return NVFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  return cuda_status(launch_compute_global(x, rows, cols, ldx, d_global, stream, dev->sms));
}

nvfp4_status nvfp4_make_alpha(const float* d_g_a, const float* d_g_w, int64_t n, float* d_alpha,
                              nvfp4_stream_t stream) {
  if (!d_g_w || !d_alpha || n < 0) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  if (!device_info()) return NVFP4_ERR_NO_DEVICE;
  return cuda_status(launch_make_alpha(d_g_a, d_g_w, n, d_alpha, stream));
}

nvfp4_status nvfp4_reduce_max(const float* d_in, int64_t n, float* d_out, nvfp4_stream_t stream) {
  if (!d_in || !d_out || n <= 0) return NVFP4_ERR_INVALID_ARG;
  if (!device_info()) return NVFP4_ERR_NO_DEVICE;
  return cuda_status(launch_reduce_max(d_in, n, d_out, stream));
}

nvfp4_status nvfp4_quantize_act(const void* x, int64_t M, int64_t K, int64_t ldx, const float* d_global,
                                uint8_t* codes, uint8_t* scales, nvfp4_stream_t stream) {
  if (M < 0 || K <= 0 || ldx < K) return NVFP4_ERR_INVALID_ARG;
  if (M == 0) return NVFP4_OK;
  if (!x || !d_global || !codes || !scales) return NVFP4_ERR_INVALID_ARG;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (ldx % 8) != 0) return NVFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  return cuda_status(launch_quant_act(x, M, K, ldx, d_global, codes, scales, dev->sms, stream));
}

// Up to this many rows the dense W4A4 linear runs on 128 x 128 tiles.
constexpr int64_t kSmallM = 128;

nvfp4_status nvfp4_linear_w4a4(const uint8_t* a_codes, const uint8_t* a_sf, int64_t M, const uint8_t* w_codes,
                               const uint8_t* w_sf, int64_t N, int64_t K, const float* d_alpha, void* out,
                               int64_t ldo, nvfp4_stream_t stream) {
  if (M < 0 || N <= 0 || K <= 0 || ldo < N) return NVFP4_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 24)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!a_codes || !a_sf || !w_codes || !w_sf || !d_alpha || !out) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a_codes) || !aligned16(a_sf) || !aligned16(w_codes) || !aligned16(w_sf) || !aligned16(out) ||
      (ldo % 8) != 0)
    return NVFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  const int64_t m_tiles = (M + 127) / 128;
  GemmMaps maps;
  if (!make_codes_map(&maps.a, a_codes, M, K / 2) || !make_codes_map(&maps.b, w_codes, N, K / 2) ||
      !make_out_map(&maps.out, out, M, N, ldo))
    return NVFP4_ERR_CUDA;
  GemmParams p{};
  p.sfa = a_sf;
  p.sfb = w_sf;
  p.K = static_cast<int>(K);
  p.kblocks = static_cast<int>((K + 255) / 256);
  p.sf_atoms = static_cast<int>(K / 64);
  p.n_tiles = static_cast<int>((N + 255) / 256);
  p.m_tiles = static_cast<int>(m_tiles);
  p.b_rows_total = static_cast<int>(N);
  p.alpha = d_alpha;
  p.out = static_cast<uint16_t*>(out);
  p.ldo = ldo;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.status = dev->status;
  if (M <= kSmallM) {
    // few tokens: 128 x 128 tiles on single CTAs, one per SM at most
    p.n_tiles = static_cast<int>((N + 127) / 128);
    const int64_t tiles = m_tiles * p.n_tiles;
    const int64_t grid = tiles < dev->sms ? tiles : dev->sms;
    return cuda_status(launch_gemm(kLaunchDenseSmall, maps, p, static_cast<int>(grid), stream));
  }
  // one CTA pair per 256 x 256 tile, at most one pair per two SMs
  const int64_t units = ((m_tiles + 1) / 2) * p.n_tiles;
  const int64_t pairs = units < dev->sms / 2 ? units : dev->sms / 2;
  return cuda_status(launch_gemm(kEpiDense, maps, p, static_cast<int>(2 * pairs), stream));
}

size_t nvfp4_linear_w4a16_workspace(int64_t T, int64_t N, int64_t K) {
  if (T <= 0 || N <= 0 || K <= 0 || K % 128 != 0) return 0;
  const DeviceInfo* dev = device_info();
  const int sms = dev ? dev->sms : 152;
  if (T <= 16 && gemv_ring_plan(T, N, K, sms).ok) return 0;  // partials stay on chip
  return gemv_plan(T, N, K, sms).ws_bytes;
}

nvfp4_status nvfp4_linear_w4a16(const void* x, int64_t T, int64_t ldx, const uint8_t* w_codes, const uint8_t* w_sf,
                                int64_t N, int64_t K, const float* d_alpha, void* out, int64_t ldo, void* workspace,
                                size_t ws_bytes, nvfp4_stream_t stream) {
  if (T < 0 || N <= 0 || K <= 0 || ldx < K || ldo < N) return NVFP4_ERR_INVALID_ARG;
  if (T > 16 || N % 8 != 0 || K % 128 != 0 || N > (1LL << 30) || K > (1LL << 24))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return NVFP4_OK;
  if (!x || !w_codes || !w_sf || !d_alpha || !out) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_codes) || !aligned16(w_sf) || (ldx % 8) != 0 || (ldo % 2) != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 3u) != 0)
    return NVFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  const GemvRingPlan ring = gemv_ring_plan(T, N, K, dev->sms);
  if (ring.ok) {
    CUtensorMap cmap;
    if (!make_gemv_codes_map(&cmap, w_codes, N, K / 2)) return NVFP4_ERR_CUDA;
    return cuda_status(launch_gemv_w4a16_ring(cmap, x, T, ldx, w_sf, N, K, d_alpha, out, ldo, ring, dev->status,
                                              stream));
  }
  const GemvPlan plan = gemv_plan(T, N, K, dev->sms);
  if (plan.ws_bytes > 0) {
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    if (ws_bytes < plan.ws_bytes) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return NVFP4_ERR_MISALIGNED;
  }
  return cuda_status(launch_gemv_w4a16(x, T, ldx, w_codes, w_sf, N, K, d_alpha, out, ldo,
                                       static_cast<float*>(workspace), plan, stream));
}

size_t nvfp4_moe_workspace(int64_t T, int64_t H, int64_t I, int64_t E, int topk) {
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return 0;
  return moe_layout(T, H, I, E, topk).total;
}

nvfp4_status nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                        nvfp4_moe_layout* out) {
  if (!out || T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return NVFP4_ERR_INVALID_ARG;
  const MoELayoutBytes L = moe_layout(T, H, I, E, topk);
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->n_tiles = L.n_tiles;
  out->row_map = L.row_map;
  out->tile_expert = L.tile_expert;
  out->pos = L.pos;
  out->a1_codes = L.a1_codes;
  out->a1_sf = L.a1_sf;
  out->h_codes = L.h_codes;
  out->h_sf = L.h_sf;
  out->y = L.y;
  out->hist = L.hist;
  out->total = L.total;
  out->p_max = L.p_max;
  out->row_block = L.bm;
  return NVFP4_OK;
}

static nvfp4_status moe_check(int64_t T, int64_t H, int64_t I, int64_t E, int topk, int64_t topk_max) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return NVFP4_ERR_INVALID_ARG;
  if (H % 128 != 0 || I % 128 != 0 || E > 1024 || topk > topk_max) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (H > (1 << 16) || I > (1 << 16) || T * topk + E * 128 > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (E * 2 * I > (1LL << 30) || E * H > (1LL << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_w4a4(const void* x, int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                            const int32_t* topk_ids, const float* topk_w, const float* d_g_a1,
                            const uint8_t* w13_codes, const uint8_t* w13_sf, const float* d_alpha13,
                            const float* d_g_a2, const uint8_t* w2_codes, const uint8_t* w2_sf,
                            const float* d_alpha2, void* out, void* workspace, size_t ws_bytes,
                            nvfp4_stream_t stream) {
  nvfp4_status st = moe_check(T, H, I, E, topk, 32);
  if (st != NVFP4_OK) return st;
  if (T == 0) return NVFP4_OK;
  if (!x || !topk_ids || !topk_w || !d_g_a1 || !w13_codes || !w13_sf || !d_alpha13 || !d_g_a2 || !w2_codes ||
      !w2_sf || !d_alpha2 || !out || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13_codes) || !aligned16(w13_sf) || !aligned16(w2_codes) || !aligned16(w2_sf) ||
      !aligned16(out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return NVFP4_ERR_MISALIGNED;
  const MoELayoutBytes L = moe_layout(T, H, I, E, topk);
  if (ws_bytes < L.total) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  const MoEWorkspace w = moe_carve(workspace, L);
  cudaError_t e = launch_moe_align(topk_ids, T, topk, static_cast<int>(E), L.bm, w, dev->status, stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  e = launch_moe_quant_permute(x, T, H, topk, d_g_a1, w, dev->sms, stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  {  // gate_up: SiLU(gate) * up, re-quantised with g_a2
    GemmParams p{};
    p.up_offset = static_cast<int>(I);
    p.alpha = d_alpha13;
    p.g_out = d_g_a2;
    p.q_codes = w.h_codes;
    p.q_sf = w.h_sf;
    p.q_row_bytes = I / 2;
    p.q_cpad4 = (I / 16 + 3) / 4;
    st = launch_grouped(kEpiGatedQuant, w.a1_codes, w.a1_sf, w.p_max, H, w13_codes, w13_sf, 2 * I, E, I / 128, w, p,
                        dev, stream);
    if (st != NVFP4_OK) return st;
  }
  {  // down: routing weight, fp32 top-k sum
    GemmParams p{};
    p.alpha = d_alpha2;
    p.y = w.y;
    p.ldy = H;
    p.topk_w = topk_w;
    p.topk = topk;
    // few routes per expert: the tile loop is bound by the weight stream, and
    // the register-direct top-k adds free the staging memory for 6 stages
    const int down = T * topk <= kDirectDownRoutesPerExpert * E ? kEpiDownDirect : kEpiDownSum;
    st = launch_grouped(down, w.h_codes, w.h_sf, w.p_max, I, w2_codes, w2_sf, H, E, H / 128, w, p, dev, stream);
    if (st != NVFP4_OK) return st;
  }
  return cuda_status(launch_moe_finalize(w.y, T * H, out, dev->sms, stream));
}

namespace {
struct MoeW16Layout {
  size_t h, dn, total;
};
// bf16 h of every route, then the fp32 down rows of every route.
MoeW16Layout moe_w16_layout(int64_t T, int64_t H, int64_t I, int topk) {
  MoeW16Layout L{};
  const int64_t R = T * topk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.h = take(static_cast<size_t>(R * I) * sizeof(uint16_t));
  L.dn = take(static_cast<size_t>(R * H) * sizeof(float));
  L.total = off;
  return L;
}
nvfp4_status moe_w16_check(int64_t T, int64_t H, int64_t I, int64_t E, int topk) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0) return NVFP4_ERR_INVALID_ARG;
  if (T > 64 || topk > 8 || H % 128 != 0 || I % 128 != 0 || E > 1024) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (H > (1 << 14) || I > (1 << 14) || E * 2 * I > (1LL << 30) || E * H > (1LL << 30))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!moe16_plan(0, H, T, E, topk, I / 64, 1).ok || !moe16_plan(1, I, T, E, topk, H / 128, 1).ok))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}
}  // namespace

size_t nvfp4_moe_w4a16_workspace(int64_t T, int64_t H, int64_t I, int64_t E, int topk) {
  if (moe_w16_check(T, H, I, E, topk) != NVFP4_OK) return 0;
  return moe_w16_layout(T, H, I, topk).total;
}

nvfp4_status nvfp4_moe_w4a16(const void* x, int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                             const int32_t* topk_ids, const float* topk_w, const uint8_t* w13_codes,
                             const uint8_t* w13_sf, const float* d_alpha13, const uint8_t* w2_codes,
                             const uint8_t* w2_sf, const float* d_alpha2, void* out, void* workspace,
                             size_t ws_bytes, nvfp4_stream_t stream) {
  nvfp4_status st = moe_w16_check(T, H, I, E, topk);
  if (st != NVFP4_OK) return st;
  if (T == 0) return NVFP4_OK;
  if (!x || !topk_ids || !topk_w || !w13_codes || !w13_sf || !d_alpha13 || !w2_codes || !w2_sf || !d_alpha2 ||
      !out || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13_codes) || !aligned16(w13_sf) || !aligned16(w2_codes) || !aligned16(w2_sf) ||
      !aligned16(out) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) || (reinterpret_cast<uintptr_t>(d_alpha13) & 3u) ||
      (reinterpret_cast<uintptr_t>(d_alpha2) & 3u))
    return NVFP4_ERR_MISALIGNED;
  const MoeW16Layout L = moe_w16_layout(T, H, I, topk);
  if (ws_bytes < L.total) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  MoeW16Params p{};
  p.x = static_cast<const uint16_t*>(x);
  p.T = static_cast<int>(T);
  p.H = static_cast<int>(H);
  p.I = static_cast<int>(I);
  p.E = static_cast<int>(E);
  p.topk = topk;
  p.ids = topk_ids;
  p.topk_w = topk_w;
  p.w13_sf = w13_sf;
  p.alpha13 = d_alpha13;
  p.w2_sf = w2_sf;
  p.alpha2 = d_alpha2;
  p.out = static_cast<uint16_t*>(out);
  p.h = reinterpret_cast<uint16_t*>(b + L.h);
  p.dn = reinterpret_cast<float*>(b + L.dn);
  p.status = dev->status;
  CUtensorMap m13, m2;
  if (!make_gemv_codes_map(&m13, w13_codes, E * 2 * I, H / 2, 64) || !make_gemv_codes_map(&m2, w2_codes, E * H, I / 2))
    return NVFP4_ERR_CUDA;
  return cuda_status(launch_moe_w4a16(m13, m2, p, dev->sms, stream));
}

nvfp4_status nvfp4_moe_calibrate(const void* x_calib, int64_t Tc, int64_t H, int64_t I, int64_t E,
                                 const float* d_g_a1, const uint8_t* w13_codes, const uint8_t* w13_sf,
                                 const float* d_alpha13, float* d_amax, float* d_g_a2, void* workspace,
                                 size_t ws_bytes, nvfp4_stream_t stream) {
  nvfp4_status st = moe_check(Tc, H, I, E, static_cast<int>(E), 1024);
  if (st != NVFP4_OK) return st;
  if (Tc == 0) return NVFP4_ERR_INVALID_ARG;
  if (!x_calib || !d_g_a1 || !w13_codes || !w13_sf || !d_alpha13 || !d_g_a2 || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x_calib) || !aligned16(w13_codes) || !aligned16(w13_sf) || !aligned16(workspace))
    return NVFP4_ERR_MISALIGNED;
  const MoELayoutBytes L = moe_layout(Tc, H, I, E, E);
  if (ws_bytes < L.total) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  const MoEWorkspace w = moe_carve(workspace, L);
  cudaError_t e = launch_moe_dense_ids(w.ids, Tc, static_cast<int>(E), stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  // 128-row segments: the calibration GEMM runs on single CTAs
  e = launch_moe_align(w.ids, Tc, static_cast<int>(E), static_cast<int>(E), 128, w, dev->status, stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  e = launch_moe_quant_permute(x_calib, Tc, H, static_cast<int>(E), d_g_a1, w, dev->sms, stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaMemsetAsync(w.amax, 0, sizeof(unsigned int) * E, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  GemmParams p{};
  p.up_offset = static_cast<int>(I);
  p.alpha = d_alpha13;
  p.amax = w.amax;
  st = launch_grouped(kEpiGatedAmax, w.a1_codes, w.a1_sf, w.p_max, H, w13_codes, w13_sf, 2 * I, E, I / 128, w, p,
                      dev, stream);
  if (st != NVFP4_OK) return st;
  e = launch_moe_calib_finish(w.amax, static_cast<int>(E), d_g_a2, stream);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  if (d_amax && cudaMemcpyAsync(d_amax, w.amax, sizeof(float) * E, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_wait_timeout(nvfp4_stream_t stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(dev->status);
  return cuda_status(cudaGetLastError());
}

nvfp4_status nvfp4_device_status(nvfp4_stream_t stream, int32_t* host_out) {
  if (!host_out) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return NVFP4_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return NVFP4_ERR_CUDA;
  *host_out = v;
  return NVFP4_OK;
}

}  // extern "C"
