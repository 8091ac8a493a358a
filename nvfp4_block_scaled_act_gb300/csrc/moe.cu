// MoE routing kernels around the grouped GEMMs (layer flow "align -> gate_up ->
// act -> down -> sum" of "speed up the nvfp4 moe prefill gemm on rtx gpus",
// section "Changes"; static input scales and top-k sum of the W4A4 MoE prefill
// page, section "Changes").
//
// align: a stable counting sort of the T * topk routes by expert, each
// expert's segment padded to a multiple of bm rows (128: one GEMM tile; 256: a
// CTA-pair tile, both halves of one expert).  tile_expert and n_tiles count
// 128-row tiles either way.  Up to
// 4096 routes one block does it all (moe_align_block_kernel); above that:
//   moe_hist_kernel     per chunk of routes (256, doubled while there are
//                       over 512 chunks), routes per expert
//   moe_scan_kernel     one block: expert offsets, padded tile table,
//                       per-chunk bases, padding rows of row_map
//   moe_scatter_kernel  one warp per chunk, in route order: row_map / pos
// The order inside a segment is the route order, so the layout is the same on
// every run.  Nothing leaves the device: the tile count is read by the GEMMs.
//
// quant_permute: the NVFP4 quantisation of x with the static global g_a1, one
// warp per 256-element chunk of a token row, written to each of the token's
// permuted rows (codes as one 128-byte row segment per warp, scales as 4-byte
// words of four blocks); it also clears the fp32 top-k accumulator y.
// finalize: y (fp32) -> bf16.
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_moe.h"

namespace nvfp4 {

constexpr int kIdBatch = 8;  // global loads a thread keeps in flight in the align kernels

// Per chunk of `chunk` routes: routes per expert.
__global__ void __launch_bounds__(256) moe_hist_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int chunk,
                                                       int32_t* __restrict__ hist, int* status) {
  pdl_wait();  // the routes, tables or buffers of the preceding kernels
  pdl_launch_dependents();
  extern __shared__ int32_t sh[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  for (int i = threadIdx.x; i < chunk; i += blockDim.x) {
    const int64_t r = base + i;
    if (r < R) {
      const int e = ids[r];
      if (e >= 0 && e < E)
        atomicAdd(&sh[e], 1);
      else
        record_status(status, kStatusBadExpert);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = sh[e];
}

// One block of 1024 threads.  Each expert's column of the chunk histogram is
// split into P = 1024 / E contiguous runs of chunks, one thread per run
// (thread t: expert t % E, run t / E, so a warp reads consecutive experts of
// one chunk).  The run sums give the expert counts; one thread per expert scans
// the padded counts; each run thread then rewrites its chunks as the expert's
// base for that chunk (in chunk order) and writes its share of the padding
// rows and tile entries.
__global__ void __launch_bounds__(1024) moe_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E, int bm,
                                                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                        int32_t* __restrict__ n_tiles, int32_t* __restrict__ row_map,
                                                        int32_t* __restrict__ tile_expert) {
  pdl_wait();  // the routes, tables or buffers of the preceding kernels
  pdl_launch_dependents();
  __shared__ int32_t part_s[1024];  // [run][expert] chunk sums
  __shared__ int32_t off_s[1024];   // [expert] padded segment start
  __shared__ int32_t cnt_s[1024];   // [expert] routes
  __shared__ int32_t warp_sums[32];
  const int t = threadIdx.x;
  const int P = static_cast<int>(blockDim.x) / E;
  const int e = t % E, run = t / E;
  const bool active = run < P;
  const int per = (nchunks + P - 1) / P;
  const int c_begin = min(run * per, nchunks), c_end = min(c_begin + per, nchunks);
  int32_t part = 0;
  if (active) {
    for (int c0 = c_begin; c0 < c_end; c0 += kIdBatch) {
      int32_t h[kIdBatch];
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) h[q] = c0 + q < c_end ? hist[static_cast<int64_t>(c0 + q) * E + e] : 0;
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) part += h[q];
    }
  }
  part_s[t] = part;
  __syncthreads();
  int32_t cnt = 0;
  if (t < E)
    for (int q = 0; q < P; ++q) cnt += part_s[q * E + t];
  const int32_t padded = (cnt + bm - 1) / bm * bm;
  // exclusive scan of padded over experts (block-wide)
  int32_t v = padded;
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t s = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += s;
  }
  if (lane == 31) warp_sums[w] = v;
  __syncthreads();
  if (w == 0) {
    int32_t s = (lane < static_cast<int>(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += u;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int32_t incl = v + (w > 0 ? warp_sums[w - 1] : 0);
  if (t < E) {
    const int32_t off = incl - padded;
    counts[t] = cnt;
    offsets[t] = off;
    off_s[t] = off;
    cnt_s[t] = cnt;
  }
  if (t == E - 1) {
    offsets[E] = incl;
    *n_tiles = incl / 128;
  }
  __syncthreads();
  if (active) {
    const int32_t off = off_s[e], ce = cnt_s[e], pe = (ce + bm - 1) / bm * bm;
    int32_t base = off;
    for (int q = 0; q < run; ++q) base += part_s[q * E + e];
    for (int c0 = c_begin; c0 < c_end; c0 += kIdBatch) {
      int32_t h[kIdBatch];
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) h[q] = c0 + q < c_end ? hist[static_cast<int64_t>(c0 + q) * E + e] : 0;
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) {
        if (c0 + q < c_end) hist[static_cast<int64_t>(c0 + q) * E + e] = base;
        base += h[q];
      }
    }
    for (int32_t p = off + ce + run; p < off + pe; p += P) row_map[p] = -1;
    for (int32_t p = off / 128 + run; p < (off + pe) / 128; p += P) tile_expert[p] = e;
  }
}

// One warp per chunk; routes in order, 32 at a time.  The ids of a chunk are
// loaded in batches of kIdBatch per lane before they are ranked, so the loads
// of a batch are in flight together.
__global__ void __launch_bounds__(32) moe_scatter_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int chunk,
                                                         const int32_t* __restrict__ hist,
                                                         int32_t* __restrict__ row_map, int32_t* __restrict__ pos) {
  pdl_wait();  // the routes, tables or buffers of the preceding kernels
  pdl_launch_dependents();
  extern __shared__ int32_t run[];
  for (int e = threadIdx.x; e < E; e += 32) run[e] = hist[static_cast<int64_t>(blockIdx.x) * E + e];
  __syncwarp();
  const int lane = threadIdx.x;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  for (int i0 = 0; i0 < chunk; i0 += 32 * kIdBatch) {
    int ev[kIdBatch];
#pragma unroll
    for (int q = 0; q < kIdBatch; ++q) {
      const int64_t r = base + i0 + q * 32 + lane;
      ev[q] = r < R ? __ldg(ids + r) : -1;
    }
#pragma unroll
    for (int q = 0; q < kIdBatch; ++q) {
      const int64_t r = base + i0 + q * 32 + lane;
      const bool in = r < R;
      const int e = ev[q];
      const bool valid = in && e >= 0 && e < E;
      const unsigned key = valid ? static_cast<unsigned>(e) : 0xFFFFFFFFu;
      const unsigned same = __match_any_sync(0xFFFFFFFFu, key);
      const int rank = __popc(same & ((1u << lane) - 1u));
      int32_t p = -1;
      if (valid) {
        p = run[e] + rank;
        row_map[p] = static_cast<int32_t>(r);
      }
      if (in) pos[r] = p;
      __syncwarp();
      if (valid && rank == 0) run[e] += __popc(same);
      __syncwarp();
    }
  }
}

// The whole alignment in one block of 32 warps, for up to kAlignOneBlock
// routes: warp w counts its contiguous share of the routes per expert into
// its own shared-memory histogram, one thread per expert scans the padded
// counts and turns the warp histograms into per-warp bases (in warp order),
// and each warp places its routes in order.  The layout is the stable counting
// sort of the multi-block path.
constexpr int64_t kAlignOneBlock = 4096;  // above this, one SM's rank matching is the bound

__global__ void __launch_bounds__(1024) moe_align_block_kernel(const int32_t* __restrict__ ids, int64_t R, int E,
                                                               int bm,
                                                               int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ n_tiles,
                                                               int32_t* __restrict__ row_map,
                                                               int32_t* __restrict__ tile_expert,
                                                               int32_t* __restrict__ pos, int* status) {
  pdl_wait();  // the routes, tables or buffers of the preceding kernels
  pdl_launch_dependents();
  extern __shared__ int32_t wh[];  // [32][E]
  __shared__ int32_t warp_sums[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int64_t share = (R + 32 * 32 - 1) / (32 * 32) * 32;  // routes per warp, a multiple of 32
  const int64_t begin = warp * share, end = begin + share < R ? begin + share : R;
  int32_t* mine = wh + warp * E;
  bool bad = false;
  for (int pass = 0; pass < 2; ++pass) {
    for (int64_t i0 = begin; i0 < end; i0 += 32 * kIdBatch) {
      int ev[kIdBatch];
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) {
        const int64_t r = i0 + q * 32 + lane;
        ev[q] = r < end ? __ldg(ids + r) : -1;
      }
#pragma unroll
      for (int q = 0; q < kIdBatch; ++q) {
        const int64_t r = i0 + q * 32 + lane;
        if (i0 + q * 32 >= end) break;  // warp-uniform
        const bool in = r < end;
        const int e = ev[q];
        const bool valid = in && e >= 0 && e < E;
        if (in && !valid) bad = true;
        const unsigned key = valid ? static_cast<unsigned>(e) : 0xFFFFFFFFu;
        const unsigned same = __match_any_sync(0xFFFFFFFFu, key);
        const int rank = __popc(same & ((1u << lane) - 1u));
        if (pass == 1) {
          int32_t p = -1;
          if (valid) {
            p = mine[e] + rank;
            row_map[p] = static_cast<int32_t>(r);
          }
          if (in) pos[r] = p;
        }
        __syncwarp();
        if (valid && rank == 0) mine[e] += __popc(same);
        __syncwarp();
      }
    }
    __syncthreads();
    if (pass == 1) break;
    // one thread per expert (E <= 1024): counts, padded offsets, per-warp bases
    const int e = threadIdx.x;
    int32_t cnt = 0;
    if (e < E)
      for (int w = 0; w < 32; ++w) cnt += wh[w * E + e];
    const int32_t padded = (cnt + bm - 1) / bm * bm;
    int32_t v = padded;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int32_t s2 = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xFFFFFFFFu, s2, o);
        if (lane >= o) s2 += t;
      }
      warp_sums[lane] = s2;
    }
    __syncthreads();
    const int32_t incl = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    const int32_t off = incl - padded;
    if (e < E) {
      counts[e] = cnt;
      offsets[e] = off;
      int32_t run = off;
      for (int w = 0; w < 32; ++w) {
        const int32_t h = wh[w * E + e];
        wh[w * E + e] = run;
        run += h;
      }
      for (int32_t p = off + cnt; p < off + padded; ++p) row_map[p] = -1;
      for (int32_t p = off; p < off + padded; p += 128) tile_expert[p / 128] = e;
    }
    if (e == E - 1) {
      offsets[E] = incl;
      *n_tiles = incl / 128;
    }
    __syncthreads();
  }
  if (bad) record_status(status, kStatusBadExpert);
}

// x [T, H] bf16 -> NVFP4 rows of a1 at pos[t * topk + s]; clears y [T, H].
__global__ void __launch_bounds__(256) moe_quant_permute_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H,
                                                                int topk, const float* __restrict__ d_g,
                                                                const int32_t* __restrict__ pos,
                                                                uint8_t* __restrict__ a_codes,
                                                                uint8_t* __restrict__ a_sf, int64_t cpad4,
                                                                float* __restrict__ y) {
  pdl_wait();  // the routes, tables or buffers of the preceding kernels
  pdl_launch_dependents();
  const float g = __ldg(d_g);
  const int lane = threadIdx.x & 31;
  // T * chunks < 2^31 (checked by the launcher): 32-bit index arithmetic
  const uint32_t chunks = static_cast<uint32_t>((H + 255) / 256);
  const uint32_t total = static_cast<uint32_t>(T) * chunks;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < total; item += nwarps) {
    const int64_t t = item / chunks;
    const int64_t ch = item - static_cast<uint32_t>(t) * chunks;
    const int64_t k0 = ch * 256 + lane * 8;
    const bool real = k0 < H;
    float v[8];
    float amax = 0.0f;
    if (real) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(x + t * H + k0));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu);
        v[2 * j + 1] = bf16_bits_to_f32(w[j] >> 16);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
      float4* yz = reinterpret_cast<float4*>(y + t * H + k0);
      yz[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      yz[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    const BlockScale bs = block_scale(amax, g);
    uint32_t packed = 0;
    if (bs.r != 0.0f) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        packed |= f32x2_to_e2m1x2(__fmul_rn(v[2 * j], bs.r), __fmul_rn(v[2 * j + 1], bs.r)) << (8 * j);
    }
    if (real) {
      for (int s = 0; s < topk; ++s) {
        const int32_t p = pos[t * topk + s];
        if (p >= 0) *reinterpret_cast<uint32_t*>(a_codes + static_cast<int64_t>(p) * (H / 2) + k0 / 2) = packed;
      }
    }
    // scale bytes: block j of the chunk sits on lanes 2j and 2j + 1.  Four
    // consecutive blocks are four consecutive bytes of the 128x4 layout, so
    // lane 8w packs blocks 4w .. 4w+3 into a word, and lane l stores word
    // l % 4 for routes l / 4, l / 4 + 8, ...
    const uint32_t sv = static_cast<uint32_t>(bs.s8) & 0xFFu;
    const uint32_t packed_sf = sv | (__shfl_down_sync(0xFFFFFFFFu, sv, 2) << 8) |
                               (__shfl_down_sync(0xFFFFFFFFu, sv, 4) << 16) |
                               (__shfl_down_sync(0xFFFFFFFFu, sv, 6) << 24);
    const int wq = lane & 3;
    const uint32_t word = __shfl_sync(0xFFFFFFFFu, packed_sf, 8 * wq);
    const int64_t c = ch * 16 + 4 * wq;
    if (c * 16 < H) {
      for (int s = lane >> 2; s < topk; s += 8) {
        const int32_t p = pos[t * topk + s];
        if (p >= 0) *reinterpret_cast<uint32_t*>(a_sf + sf_offset(p, c, cpad4)) = word;
      }
    }
  }
}

__global__ void __launch_bounds__(256) moe_finalize_kernel(const float* __restrict__ y, int64_t n,
                                                           uint16_t* __restrict__ out) {
  pdl_wait();  // y of the down GEMM
  pdl_launch_dependents();
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x * 8) {
    const float4 a = reinterpret_cast<const float4*>(y + i)[0];
    const float4 b = reinterpret_cast<const float4*>(y + i)[1];
    __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t*>(&h0);
    o.y = *reinterpret_cast<uint32_t*>(&h1);
    o.z = *reinterpret_cast<uint32_t*>(&h2);
    o.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(out + i) = o;
  }
}

// Dense calibration routing: route (t, e) for every row t and expert e.
__global__ void moe_dense_ids_kernel(int32_t* __restrict__ ids, int64_t Tc, int E) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < Tc * E;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    ids[i] = static_cast<int32_t>(i % E);
}

// amax bits [E] -> g_e = 2688 / amax_e (1 when zero); *g_max = max_e g_e; the
// amax values are rewritten as floats for the caller.
__global__ void __launch_bounds__(1024) moe_calib_finish_kernel(unsigned int* __restrict__ amax_bits, int E,
                                                                float* __restrict__ g_max) {
  __shared__ float wm[32];
  float g = -INFINITY;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float a = __uint_as_float(amax_bits[e]);
    g = fmaxf(g, a > 0.0f ? __fdiv_rn(2688.0f, a) : 1.0f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) g = fmaxf(g, __shfl_xor_sync(0xFFFFFFFFu, g, o));
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = g;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, wm[i]);
    *g_max = m;
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_moe_align(const int32_t* ids, int64_t T, int topk, int E, int bm, const MoEWorkspace& w,
                             int* status, cudaStream_t stream) {
  const int64_t R = T * topk;
  if (R <= kAlignOneBlock && E <= 1024) {
    const size_t smem = 32 * static_cast<size_t>(E) * sizeof(int32_t);
    if (smem > 48 * 1024) {  // per device: set on every launch
      const cudaError_t e = cudaFuncSetAttribute(moe_align_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_pdl(moe_align_block_kernel, dim3(1), dim3(1024), smem, stream, ids, R, E, bm, w.counts,
                      w.offsets, w.n_tiles, w.row_map, w.tile_expert, w.pos, status);
  }
  const int64_t chunk = moe_align_chunk(R);
  const int nchunks = static_cast<int>((R + chunk - 1) / chunk);
  const int ci = static_cast<int>(chunk);
  cudaError_t e = launch_pdl(moe_hist_kernel, dim3(nchunks), dim3(256), E * sizeof(int32_t), stream, ids, R, E, ci,
                             w.hist, status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(moe_scan_kernel, dim3(1), dim3(1024), 0, stream, w.hist, nchunks, E, bm, w.counts, w.offsets,
                 w.n_tiles, w.row_map, w.tile_expert);
  if (e != cudaSuccess) return e;
  return launch_pdl(moe_scatter_kernel, dim3(nchunks), dim3(32), E * sizeof(int32_t), stream, ids, R, E, ci,
                    static_cast<const int32_t*>(w.hist), w.row_map, w.pos);
}

cudaError_t launch_moe_quant_permute(const void* x, int64_t T, int64_t H, int topk, const float* d_g,
                                     const MoEWorkspace& w, int num_sms, cudaStream_t stream) {
  const int64_t items = T * ((H + 255) / 256);
  if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  int64_t blocks = (items + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(moe_quant_permute_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    static_cast<const uint16_t*>(x), T, H, topk, d_g, static_cast<const int32_t*>(w.pos), w.a1_codes,
                    w.a1_sf, static_cast<int64_t>((H / 16 + 3) / 4), w.y);
}

cudaError_t launch_moe_finalize(const float* y, int64_t n, void* out, int num_sms, cudaStream_t stream) {
  int64_t blocks = (n / 8 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(moe_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, y, n,
                    static_cast<uint16_t*>(out));
}

cudaError_t launch_moe_dense_ids(int32_t* ids, int64_t Tc, int E, cudaStream_t stream) {
  const int64_t n = Tc * E;
  const int blocks = static_cast<int>((n + 255) / 256 > 4096 ? 4096 : (n + 255) / 256);
  moe_dense_ids_kernel<<<blocks < 1 ? 1 : blocks, 256, 0, stream>>>(ids, Tc, E);
  return cudaGetLastError();
}

cudaError_t launch_moe_calib_finish(unsigned int* amax_bits, int E, float* g_max, cudaStream_t stream) {
  moe_calib_finish_kernel<<<1, 1024, 0, stream>>>(amax_bits, E, g_max);
  return cudaGetLastError();
}

}  // namespace nvfp4
