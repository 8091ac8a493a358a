// W4A16 MoE for small batches: decode and prefills with few tokens per expert
// run with bf16 activations against the same NVFP4 expert banks as the W4A4
// path (the W4A4 MoE prefill page, section "Changes": W4A4 from 4 tokens per
// expert, W4A16 below; no repack).
//
//   route     one CTA: per-expert route lists in route order, one slot per
//             expert in use, and the power-of-two shift of every token row
//   gate_up   grouped GEMV: CTA (slot, column block j of 64) streams gate rows
//             64j .. 64j+63 and up rows I+64j .. of W13[e] over H and emits
//             h = bf16(silu(a13 G) * (a13 U)) for the slot's routes, with the
//             per-route max |h| (the shift of the down stage's input rows)
//   down      grouped GEMV: CTA (slot, row block b of 128) streams rows of W2[e]
//             over I and writes w_route * a2 * acc (fp32) for each route
//   finalize  out[t] = bf16(sum over the token's slots, in slot order)
//
// The GEMVs stream weights through a per-thread cp.async ring (kW16Stages 128-k
// blocks in flight) and multiply on mma.sync with the W4A16 arithmetic of
// nvfp4_decode.cuh (f16 weights, activations staged as f16 after a per-row
// power-of-two rescale).
#include "nvfp4_common.cuh"
#include "nvfp4_decode.cuh"
#include "nvfp4_moe.h"

namespace nvfp4 {

constexpr int kW16Threads = 128;                 // 4 warps x 32 weight rows
constexpr int kW16Stages = 6;                    // 128-k weight blocks in flight per thread
constexpr int kW16Lane = 80;                     // per thread and block: 4 x 16 B codes + 4 x 4 B scales
constexpr int kW16StageBytes = kW16Threads * kW16Lane;
constexpr int kW16Tok = 16;                      // input rows per pass
constexpr int kW16XStride = 256 + 16;            // f16 row of a 128-k block, padded
constexpr int kW16Smem = kW16Stages * kW16StageBytes + 2 * kW16Tok * kW16XStride + 128 * kW16Tok * 4;

__device__ __forceinline__ void cp_async_4(uint32_t sdst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sdst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_16s(uint32_t sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sdst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// silu(v) = v / (1 + e^-v) with the hardware exp2 and fast division (as the W4A4
// gate_up epilogue).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// ---------------------------------------------------------------------------
// route
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe16_route_kernel(MoeW16Params p) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;            // [E]
  int32_t* slot_of = sh + p.E;  // [E]
  __shared__ float red[8];
  const int R = p.T * p.topk;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int e = p.ids[r];
    if (e >= 0 && e < p.E)
      atomicAdd(&cnt[e], 1);
    else
      record_status(p.status, kStatusBadExpert);
    p.h_amax[r] = 0u;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // one slot per expert in use, in expert order; routes in route order
    int s = 0, start = 0;
    for (int e = 0; e < p.E; ++e) {
      if (cnt[e] > 0) {
        slot_of[e] = start;
        p.slot_expert[s] = e;
        p.slot_start[s] = start;
        p.slot_count[s] = cnt[e];
        start += cnt[e];
        ++s;
      }
    }
    *p.n_slots = s;
    for (int r = 0; r < R; ++r) {
      const int e = p.ids[r];
      if (e >= 0 && e < p.E) p.route_list[slot_of[e]++] = r;
    }
  }
  // per-token shift: the row's largest magnitude -> [2^14, 2^15) in f16
  for (int t = 0; t < p.T; ++t) {
    float m = 0.0f;
    const uint16_t* xr = p.x + static_cast<int64_t>(t) * p.H;
    for (int k = threadIdx.x * 8; k < p.H; k += blockDim.x * 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] & 0xFFFFu)));
        m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] >> 16)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = 0.0f;
      for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) b = fmaxf(b, red[i]);
      p.tok_shift[t] = token_shift(__float_as_uint(b));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// grouped GEMV (MODE 0: gate_up, 1: down)
// ---------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(kW16Threads) moe16_gemv_kernel(MoeW16Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int in_row[kW16Tok];     // route of each input row of the pass
  __shared__ int in_shift[kW16Tok];   // its power-of-two shift
  const int slot = blockIdx.x;
  if (slot >= *p.n_slots) return;     // uniform for the CTA
  const int e = p.slot_expert[slot];
  const int c_all = p.slot_count[slot];
  const int start = p.slot_start[slot];
  const int K = MODE == 0 ? p.H : p.I;
  const int nkb = K / 128;
  const int sf_atoms = K / 64;
  const uint8_t* wc = MODE == 0 ? p.w13_codes : p.w2_codes;
  const uint8_t* ws = MODE == 0 ? p.w13_sf : p.w2_sf;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  uint8_t* ring = smem;
  uint8_t* xs = smem + kW16Stages * kW16StageBytes;           // [2][kW16Tok][kW16XStride]
  float* part = reinterpret_cast<float*>(xs + 2 * kW16Tok * kW16XStride);  // [128][kW16Tok]
  const uint32_t my_ring = smem_u32(ring) + threadIdx.x * kW16Lane;

  // this thread's 4 weight rows: CTA rows 32 warp + 8 j + g
  const uint8_t* cptr[4];
  const uint8_t* sptr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 32 * warp + 8 * j + g;
    int64_t R;
    if (MODE == 0)
      R = static_cast<int64_t>(e) * 2 * p.I + (r < 64 ? 64 * blockIdx.y + r : p.I + 64 * blockIdx.y + (r - 64));
    else
      R = static_cast<int64_t>(e) * p.H + 128 * blockIdx.y + r;
    cptr[j] = wc + R * (K / 2) + 16 * t;
    sptr[j] = ws + ((R >> 7) * sf_atoms + (t >> 1)) * 512 + (R & 31) * 16 + ((R & 127) >> 5) * 4;
  }
  auto issue = [&](int kb) {
    const uint32_t dst = my_ring + (kb % kW16Stages) * kW16StageBytes;
#pragma unroll
    for (int j = 0; j < 4; ++j) cp_async_16s(dst + 16 * j, cptr[j] + kb * 64);
#pragma unroll
    for (int j = 0; j < 4; ++j) cp_async_4(dst + 64 + 4 * j, sptr[j] + kb * 1024);
  };

  int xofs[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) xofs[i] = g * kW16XStride + xchunk(4 * t + i) * 16;

  for (int tok0 = 0; tok0 < c_all; tok0 += kW16Tok) {
    const int c = min(kW16Tok, c_all - tok0);
    if (threadIdx.x < kW16Tok) {
      const int i = threadIdx.x;
      const int route = i < c ? p.route_list[start + tok0 + i] : 0;
      in_row[i] = route;
      in_shift[i] = i < c ? (MODE == 0 ? p.tok_shift[route / p.topk] : token_shift(p.h_amax[route])) : 0;
    }
    __syncthreads();
    // input unit u = (row, 8-element chunk) of block kb: bf16 -> f16 * 2^-shift
    auto load_units = [&](int kb, uint4 (&v)[2]) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * kW16Threads;
        v[q] = make_uint4(0u, 0u, 0u, 0u);
        if (u < c * 16 && kb < nkb) {
          const int row = u >> 4, ch = u & 15;
          const uint16_t* src = MODE == 0 ? p.x + static_cast<int64_t>(in_row[row] / p.topk) * p.H
                                          : p.h + static_cast<int64_t>(in_row[row]) * p.I;
          v[q] = *reinterpret_cast<const uint4*>(src + kb * 128 + ch * 8);
        }
      }
    };
    auto store_units = [&](int buf, const uint4 (&v)[2]) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * kW16Threads;
        if (u < kW16Tok * 16) {
          const int row = u >> 4, ch = u & 15;
          const float f = pow2f(-in_shift[row]);
          const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __half2 h =
                __floats2half2_rn(bf16_bits_to_f32(w4[j] & 0xFFFFu) * f, bf16_bits_to_f32(w4[j] >> 16) * f);
            o[j] = *reinterpret_cast<const uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(xs + buf * (kW16Tok * kW16XStride) + row * kW16XStride + xchunk(ch) * 16) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    };

    // prime: weight blocks 0 .. S-2 in flight, inputs of block 0 staged
#pragma unroll
    for (int s = 0; s < kW16Stages - 1; ++s) {
      if (s < nkb) issue(s);
      cp_async_commit_group();
    }
    {
      uint4 v[2];
      load_units(0, v);
      store_units(0, v);
    }
    __syncthreads();

    float acc[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][h][q] = 0.0f;
    const bool tok_lo = g < c, tok_hi = g + 8 < c;

    for (int kb = 0; kb < nkb; ++kb) {
      if (kb + kW16Stages - 1 < nkb) issue(kb + kW16Stages - 1);
      cp_async_commit_group();
      uint4 nv[2];
      load_units(kb + 1, nv);  // next block's inputs, stored after this block's MMAs
      cp_async_wait_group<kW16Stages - 1>();  // block kb of this thread landed
      const uint8_t* st = ring + (kb % kW16Stages) * kW16StageBytes + threadIdx.x * kW16Lane;
      uint4 cw[4];
      uint32_t slo[4], shi[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        cw[j] = *reinterpret_cast<const uint4*>(st + 16 * j);
        const uint32_t word = *reinterpret_cast<const uint32_t*>(st + 64 + 4 * j);
        scale_pair_f16(word >> (16 * (t & 1)), slo[j], shi[j]);
      }
      const uint8_t* xb = xs + (kb & 1) * (kW16Tok * kW16XStride);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 blo = make_uint4(0u, 0u, 0u, 0u), bhi = make_uint4(0u, 0u, 0u, 0u);
        if (tok_lo) blo = *reinterpret_cast<const uint4*>(xb + xofs[i]);
        if (tok_hi) bhi = *reinterpret_cast<const uint4*>(xb + xofs[i] + 8 * kW16XStride);
        uint32_t wf[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t word = (i == 0) ? cw[j].x : (i == 1) ? cw[j].y : (i == 2) ? cw[j].z : cw[j].w;
          const uint32_t m = (i < 2) ? slo[j] : shi[j];
          e2m1x4_to_f16x2(word, wf[j]);
#pragma unroll
          for (int q = 0; q < 4; ++q) wf[j][q] = f16x2_mul(wf[j][q], m);
        }
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          mma_f16_16816(acc[a][0], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1], wf[2 * a + 1][1], blo.x, blo.y);
          mma_f16_16816(acc[a][0], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3], wf[2 * a + 1][3], blo.z, blo.w);
          if (c > 8) {
            mma_f16_16816(acc[a][1], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1], wf[2 * a + 1][1], bhi.x, bhi.y);
            mma_f16_16816(acc[a][1], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3], wf[2 * a + 1][3], bhi.z, bhi.w);
          }
        }
      }
      store_units((kb + 1) & 1, nv);
      __syncthreads();  // next block's inputs staged; this block's buffer free
    }
    cp_async_wait_group<0>();

    // acc[a][h][q]: CTA row 32 warp + 16 a + g (+8 for q >= 2), input 8 h + 2 t (+1 for odd q)
    if (MODE == 1) {
      const float a2 = __ldg(p.alpha2 + e);
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = 8 * h + 2 * t + (q & 1);
            if (i < c) {
              const int row = 32 * warp + 16 * a + g + 8 * (q >> 1);
              const int route = in_row[i];
              const float v = acc[a][h][q] * pow2f(in_shift[i]);
              p.partial[static_cast<int64_t>(route) * p.H + 128 * blockIdx.y + row] =
                  __fmul_rn(__fmul_rn(__ldg(p.topk_w + route), a2), v);
            }
          }
    } else {
      const float a13 = __ldg(p.alpha13 + e);
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = 8 * h + 2 * t + (q & 1);
            const int row = 32 * warp + 16 * a + g + 8 * (q >> 1);
            part[row * kW16Tok + i] = i < c ? acc[a][h][q] * pow2f(in_shift[i]) : 0.0f;
          }
      __syncthreads();
      // gate row jj pairs with up row 64 + jj
      for (int u = threadIdx.x; u < 64 * c; u += kW16Threads) {
        const int i = u / 64, jj = u - i * 64;
        const float G = part[jj * kW16Tok + i], U = part[(64 + jj) * kW16Tok + i];
        const float hv = silu_fast(__fmul_rn(a13, G)) * __fmul_rn(a13, U);
        const uint16_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        const int route = in_row[i];
        p.h[static_cast<int64_t>(route) * p.I + 64 * blockIdx.y + jj] = hb;
        atomicMax(p.h_amax + route, __float_as_uint(fabsf(bf16_bits_to_f32(hb))));
      }
    }
    __syncthreads();  // the pass's smem (inputs, partials) is free
  }
}

// ---------------------------------------------------------------------------
// finalize: out[t][n] = bf16(sum over slots in order of the route partials)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe16_finalize_kernel(MoeW16Params p) {
  const int64_t total = static_cast<int64_t>(p.T) * p.H;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tkn = idx / p.H, n = idx - tkn * p.H;
    float y = 0.0f;
    for (int s = 0; s < p.topk; ++s) {
      const int64_t r = tkn * p.topk + s;
      const int e = p.ids[r];
      if (e < 0 || e >= p.E) continue;
      y += p.partial[r * p.H + n];
    }
    p.out[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

cudaError_t launch_moe_w4a16(const MoeW16Params& p, int num_sms, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe16_gemv_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kW16Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(moe16_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kW16Smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int R = p.T * p.topk;
  const int S = R < p.E ? R : p.E;  // slots at most
  moe16_route_kernel<<<1, 256, 2 * p.E * sizeof(int32_t), stream>>>(p);
  moe16_gemv_kernel<0><<<dim3(S, p.I / 64), kW16Threads, kW16Smem, stream>>>(p);
  moe16_gemv_kernel<1><<<dim3(S, p.H / 128), kW16Threads, kW16Smem, stream>>>(p);
  const int64_t total = static_cast<int64_t>(p.T) * p.H;
  int64_t blocks = (total + 255) / 256;
  if (blocks > num_sms * 4) blocks = num_sms * 4;
  moe16_finalize_kernel<<<static_cast<int>(blocks < 1 ? 1 : blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4
