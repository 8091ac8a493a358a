// W4A16 MoE for small batches: decode and prefills with few tokens per expert
// run with bf16 activations against the same NVFP4 expert banks as the W4A4
// path (the W4A4 MoE prefill page, section "Changes": W4A4 from 4 tokens per
// expert, W4A16 below; no repack).
//
//   gate_up   grouped GEMV: CTA (slot, 128-row block of W13[e], k-split)
//             streams its rows over its k-range of H and writes the fp32
//             sums G (rows < I) or U (rows >= I) of every route of the slot
//   down      grouped GEMV: CTA (slot, 128-row block of W2[e], k-split) stages
//             h = bf16(silu(a13 G) * (a13 U)) of its routes over its k-range
//             of I, streams its rows and writes w_route * a2 * acc (fp32)
//   finalize  out[t] = bf16(sum over the token's top-k routes, in slot order)
//
// There is no routing kernel: a slot is the s-th expert in use (ascending
// expert id), and every CTA derives its expert and its routes (in route order)
// from the top-k ids itself.  The GEMVs are the decode kernel's weight ring
// per CTA: TMA boxes of 128 rows x one 128-k block and its two scale atoms,
// the whole ring filled up front, split-K inside a thread-block cluster with
// a fixed-order reduction through distributed shared memory, and the W4A16
// arithmetic of nvfp4_decode.cuh (f16 weights, activations staged as f16
// after a power-of-two rescale per route row and k-range).  The three
// kernels are chained by programmatic dependent launch: the down kernel
// fills its weight ring while gate_up still runs.
#include "nvfp4_common.cuh"
#include "nvfp4_decode.cuh"
#include "nvfp4_moe.h"

namespace nvfp4 {

constexpr int kM16Groups = 2;                       // k-groups (128-k blocks dealt round-robin)
constexpr int kM16CompWarps = 4 * kM16Groups;       // 4 row groups of 32 x 2 k-groups
constexpr int kM16Comp = kM16CompWarps * 32;
constexpr int kM16Threads = kM16Comp + 32;          // + one producer warp
constexpr int kM16Rows = 128;                       // weight rows per CTA
constexpr int kM16Chunk = kM16Rows * 64;            // codes of one 128-k block
constexpr int kM16ChunkSf = 1024;                   // its two scale atoms
constexpr int kM16Slot = kM16Chunk + kM16ChunkSf;
constexpr int kM16MaxSlots = 24;
constexpr int kM16MaxCluster = 8;
constexpr int kM16MaxRoutes = 64 * 8;               // T <= 64, top-k <= 8
constexpr int kM16MaxKBlocks = 16;                  // k elements per CTA <= 2048
constexpr size_t kM16SmemBudget = 104 * 1024;       // two CTAs per SM with the static shared memory

// silu(v) = v / (1 + e^-v) with the hardware exp2 and fast division (as the W4A4
// gate_up epilogue).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// ---------------------------------------------------------------------------
// grouped GEMV (MODE 0: gate_up over H, 1: down over I)
// ---------------------------------------------------------------------------
template <int MODE, bool kTok16>
__global__ void __launch_bounds__(kM16Threads, kTok16 ? 2 : 3)
    moe16_ring_kernel(const __grid_constant__ CUtensorMap cmap, const MoeW16Params p, const Moe16Plan pl) {
  constexpr int kP = kTok16 ? 16 : 8;  // route rows per pass
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kM16MaxSlots];
  __shared__ __align__(8) uint64_t empty[kM16MaxSlots];
  __shared__ unsigned int row_amax[kP];
  __shared__ uint32_t present[32];
  __shared__ int s_ids[kM16MaxRoutes];
  __shared__ int routes[kM16MaxRoutes];
  __shared__ int s_expert, s_count;
  __shared__ volatile int abort_flag;

  // gate_up reads the top-k ids and x of the preceding kernel; the down kernel
  // is released only after that wait, so its own reads of the ids (below,
  // before its wait) see the final values.
  if (MODE == 0) pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = (warp == kM16CompWarps) && lane == 0;
  const int ncl = pl.cl;
  const uint32_t rank = cluster_ctarank();
  const int unit = static_cast<int>(blockIdx.x) / ncl;
  const int slot = unit / pl.nrb;
  const int rb = unit - slot * pl.nrb;
  const int R = p.T * p.topk;
  const int K = MODE == 0 ? p.H : p.I;
  const int rows_e = MODE == 0 ? 2 * p.I : p.H;
  const int k_begin = static_cast<int>(rank) * pl.kc;
  const int k_len = max(0, min(pl.kc, K - k_begin));
  const int nkb = k_len / 128;
  const int Rs = pl.R;

  // --- the slot's expert and routes -----------------------------------------
  if (threadIdx.x < 32) present[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < Rs; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    fence_barrier_init();
  }
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int e = MODE == 0 ? p.ids[r] : __ldcg(p.ids + r);
    s_ids[r] = e;
    if (e >= 0 && e < p.E)
      atomicOr(&present[e >> 5], 1u << (e & 31));
    else if (MODE == 0 && blockIdx.x == 0)
      record_status(p.status, kStatusBadExpert);
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t word = present[lane];
    const int pc = __popc(word);
    int incl = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    int e = -1;
    if (slot < total) {
      const int L = __ffs(__ballot_sync(0xFFFFFFFFu, incl > slot)) - 1;
      uint32_t w = __shfl_sync(0xFFFFFFFFu, word, L);
      for (int n = slot - __shfl_sync(0xFFFFFFFFu, incl - pc, L); n > 0; --n) w &= w - 1;
      e = 32 * L + __ffs(w) - 1;
    }
    int cnt = 0;
    if (e >= 0) {
      for (int r0 = 0; r0 < R; r0 += 32) {
        const bool m = r0 + lane < R && s_ids[r0 + lane] == e;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, m);
        if (m) routes[cnt + __popc(b & ((1u << lane) - 1u))] = r0 + lane;
        cnt += __popc(b);
      }
    }
    if (lane == 0) {
      s_expert = e;
      s_count = cnt;
    }
  }
  __syncthreads();
  const int e = s_expert;
  if (e < 0) return;  // no expert for this slot: the same for the whole cluster
  const int count = s_count;
  const int passes = (count + kP - 1) / kP;
  const int nq = passes * nkb;  // ring chunks of this CTA over all passes

  uint8_t* ring = sm;
  uint8_t* ring_sf = ring + Rs * kM16Chunk;
  const int xs_stride = pl.kc * 2 + 16;
  uint8_t* xs = ring_sf + Rs * kM16ChunkSf;                      // [kP][kc*2+16] f16 inputs
  float* part = reinterpret_cast<float*>(xs + kP * xs_stride);   // [kP][128] partial sums
  const int grow = e * rows_e + rb * kM16Rows;                   // first weight row (< 2^30)
  const uint8_t* sf_src =
      (MODE == 0 ? p.w13_sf : p.w2_sf) + (static_cast<int64_t>(grow >> 7) * (K / 64) + k_begin / 64) * 512;
  auto issue = [&](int q) {
    const int s = q % Rs, kb = q % nkb;
    mbar_arrive_expect_tx(&full[s], kM16Slot);
    tma_load_2d(ring + s * kM16Chunk, &cmap, &full[s], k_begin / 2 + kb * 64, grow);
    bulk_load(ring_sf + s * kM16ChunkSf, sf_src + kb * kM16ChunkSf, kM16ChunkSf, &full[s]);
  };
  int issued = 0;
  if (producer) {
    // the weights do not depend on the preceding kernel: fill the ring now
    prefetch_tmap(&cmap);
    const int pre = min(Rs, nq);
    for (int q = 0; q < pre; ++q) issue(q);
    issued = pre;
  }
  if (MODE == 1) pdl_wait();  // G / U of the gate_up kernel

  const float a13 = __ldg(p.alpha13 + e);
  const int units = k_len / 8;  // 16-byte input units per route row
  for (int pass = 0; pass < passes; ++pass) {
    const int tok0 = pass * kP;
    const int c = min(kP, count - tok0);
    if (warp < kM16CompWarps) {
      // --- stage the pass's inputs: raw bf16, row amax, then f16 in place ----
      if (threadIdx.x < kP) row_amax[threadIdx.x] = 0u;
      named_barrier_sync(1, kM16Comp);
      const int nunits = c * units;
      constexpr int kXB = MODE == 0 ? 4 : 2;
      for (int ub0 = threadIdx.x - lane; ub0 < nunits; ub0 += kXB * kM16Comp) {
        uint4 v[kXB];
#pragma unroll
        for (int q = 0; q < kXB; ++q) {
          const int u = ub0 + q * kM16Comp + lane;
          v[q] = make_uint4(0u, 0u, 0u, 0u);
          if (u < nunits) {
            const int i = u / units;
            const int k = k_begin + (u - i * units) * 8;
            const int route = routes[tok0 + i];
            if (MODE == 0) {
              v[q] = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(route / p.topk) * p.H + k));
            } else {
              const float* gr = p.gu + static_cast<int64_t>(route) * 2 * p.I + k;
              const float4 g0 = __ldcg(reinterpret_cast<const float4*>(gr));
              const float4 g1 = __ldcg(reinterpret_cast<const float4*>(gr + 4));
              const float4 u0 = __ldcg(reinterpret_cast<const float4*>(gr + p.I));
              const float4 u1 = __ldcg(reinterpret_cast<const float4*>(gr + p.I + 4));
              const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
              const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
              float hv[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) hv[j] = silu_fast(__fmul_rn(a13, gg[j])) * __fmul_rn(a13, uu[j]);
              v[q] = make_uint4(bf16x2_bits(hv[0], hv[1]), bf16x2_bits(hv[2], hv[3]), bf16x2_bits(hv[4], hv[5]),
                                bf16x2_bits(hv[6], hv[7]));
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kXB; ++q) {
          const int ubase = ub0 + q * kM16Comp;
          if (ubase >= nunits) break;  // warp-uniform
          const int u = ubase + lane;
          const bool in = u < nunits;
          const int i = in ? u / units : kP;
          float m = 0.0f;
          const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] & 0xFFFFu)));
            m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] >> 16)));
          }
          // units per row >= 16: the warp's 32 units span at most three rows
          const int i0 = ubase / units, i1 = min(c - 1, (ubase + 31) / units);
          for (int ii = i0; ii <= i1; ++ii) {
            const unsigned int mb = __reduce_max_sync(0xFFFFFFFFu, (in && i == ii) ? __float_as_uint(m) : 0u);
            if (lane == 0 && mb != 0u) atomicMax(&row_amax[ii], mb);
          }
          if (in) {
            const int k8 = (u - i * units) * 8;
            *reinterpret_cast<uint4*>(xs + i * xs_stride + (k8 >> 7) * 256 + xchunk((k8 & 127) >> 3) * 16) = v[q];
          }
        }
      }
      named_barrier_sync(1, kM16Comp);
      for (int u = threadIdx.x; u < nunits; u += kM16Comp) {
        const int i = u / units;
        const float f = pow2f(-token_shift(row_amax[i]));
        const int k8 = (u - i * units) * 8;
        uint4* sl = reinterpret_cast<uint4*>(xs + i * xs_stride + (k8 >> 7) * 256 + xchunk((k8 & 127) >> 3) * 16);
        const uint4 v = *sl;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 h =
              __floats2half2_rn(bf16_bits_to_f32(w4[j] & 0xFFFFu) * f, bf16_bits_to_f32(w4[j] >> 16) * f);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *sl = make_uint4(o[0], o[1], o[2], o[3]);
      }
      named_barrier_sync(1, kM16Comp);

      // --- stream the weight rows of the pass --------------------------------
      const int g = lane >> 2, t = lane & 3;
      const int kp = warp >> 2;
      const int lr0 = (warp & 3) * 32;
      int sf_off[4], cofs[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int lr = lr0 + 8 * j + g;
        sf_off[j] = (lr & 31) * 16 + (lr >> 5) * 4 + 2 * (t & 1) + (t >> 1) * 512;
        cofs[j] = lr * 64 + 16 * t;
      }
      int xofs[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xofs[i] = g * xs_stride + xchunk(4 * t + i) * 16;
      const bool tok_lo = g < c, tok_hi = g + 8 < c;
      // acc[a][h][q]: rows lr0 + 16a + g (+8 for q >= 2) x route rows 8h + 2t (+1 for odd q)
      float acc[2][kTok16 ? 2 : 1][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[a][h][q] = 0.0f;
      for (int kb = kp; kb < nkb; kb += kM16Groups) {
        const int q = pass * nkb + kb;
        const int s = q % Rs;
        if (!mbar_wait(&full[s], (q / Rs) & 1, &abort_flag, p.status)) break;
        const uint8_t* cs = ring + s * kM16Chunk;
        const uint8_t* ss = ring_sf + s * kM16ChunkSf;
        uint4 cw[4];
        uint32_t slo[4], shi[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cw[j] = *reinterpret_cast<const uint4*>(cs + cofs[j]);
          scale_pair_f16(*reinterpret_cast<const uint16_t*>(ss + sf_off[j]), slo[j], shi[j]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const uint8_t* xb = xs + kb * 256;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 blo = make_uint4(0u, 0u, 0u, 0u), bhi = make_uint4(0u, 0u, 0u, 0u);
          if (tok_lo) blo = *reinterpret_cast<const uint4*>(xb + xofs[i]);
          if (kTok16 && tok_hi) bhi = *reinterpret_cast<const uint4*>(xb + xofs[i] + 8 * xs_stride);
          uint32_t wf[4][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t word = (i == 0) ? cw[j].x : (i == 1) ? cw[j].y : (i == 2) ? cw[j].z : cw[j].w;
            const uint32_t m = (i < 2) ? slo[j] : shi[j];
            e2m1x4_to_f16x2(word, wf[j]);
#pragma unroll
            for (int x = 0; x < 4; ++x) wf[j][x] = f16x2_mul(wf[j][x], m);
          }
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_f16_16816(acc[a][0], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1], wf[2 * a + 1][1], blo.x, blo.y);
            mma_f16_16816(acc[a][0], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3], wf[2 * a + 1][3], blo.z, blo.w);
            if (kTok16 && c > 8) {
              mma_f16_16816(acc[a][kTok16 ? 1 : 0], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1], wf[2 * a + 1][1],
                            bhi.x, bhi.y);
              mma_f16_16816(acc[a][kTok16 ? 1 : 0], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3], wf[2 * a + 1][3],
                            bhi.z, bhi.w);
            }
          }
        }
      }
      // partials with the rescale undone, summed over the k-groups in a fixed
      // order: the last group writes part[i][row], each lower one adds its own
      for (int grp = kM16Groups - 1; grp >= 0; --grp) {
        if (kp == grp) {
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int row = lr0 + a * 16 + g + 8 * (q >> 1);
                const int i = h * 8 + 2 * t + (q & 1);
                if (i < c) {
                  float* pp = part + i * kM16Rows + row;
                  const float v = acc[a][h][q] * pow2f(token_shift(row_amax[i]));
                  *pp = (grp == kM16Groups - 1) ? v : __fadd_rn(v, *pp);
                }
              }
        }
        if (grp > 0) named_barrier_sync(1, kM16Comp);
      }
    } else if (producer) {
      // the rest of the pass's chunks, into slots as the compute warps free them
      for (int q = max(issued, pass * nkb); q < (pass + 1) * nkb; ++q) {
        const int s = q % Rs;
        if (!mbar_wait(&empty[s], ((q / Rs) - 1) & 1, &abort_flag, p.status)) break;
        issue(q);
        issued = q + 1;
      }
    }

    // --- split-K reduction over the cluster, in rank order --------------------
    __syncwarp();  // the producer warp reconverges before the aligned barrier
    cluster_arrive();
    cluster_wait();
    const int rows_per = (kM16Rows + ncl - 1) / ncl;
    for (int idx = threadIdx.x; idx < c * rows_per; idx += blockDim.x) {
      const int i = idx / rows_per;
      const int row = static_cast<int>(rank) * rows_per + (idx - i * rows_per);
      if (row >= kM16Rows) continue;
      float v[kM16MaxCluster];
#pragma unroll
      for (int q = 0; q < kM16MaxCluster; ++q) v[q] = q < ncl ? ld_cluster_f32(part + i * kM16Rows + row, q) : 0.0f;
      float sum = 0.0f;
#pragma unroll
      for (int q = 0; q < kM16MaxCluster; ++q) sum += v[q];
      const int route = routes[tok0 + i];
      if (MODE == 0) {
        p.gu[static_cast<int64_t>(route) * rows_e + rb * kM16Rows + row] = sum;
      } else {
        const float w = __fmul_rn(__ldg(p.topk_w + route), __ldg(p.alpha2 + e));
        p.partial[static_cast<int64_t>(route) * p.H + rb * kM16Rows + row] = __fmul_rn(w, sum);
      }
    }
    cluster_arrive();  // every rank has read the partials: they may be overwritten
    cluster_wait();
  }

  if (abort_flag && producer) {
    // wind down after a timed-out wait: let this CTA's copies still in flight
    // land (bounded) before its shared memory is released
    const long long t0 = clock64();
    for (int i = 0; i < Rs && i < issued; ++i) {
      const int last = i + ((issued - 1 - i) / Rs) * Rs;  // last chunk issued into slot i
      while (!mbar_try_wait(smem_u32(&full[i]), (last / Rs) & 1) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  }
}

// ---------------------------------------------------------------------------
// finalize: out[t][n] = bf16(sum over the token's routes in slot order)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe16_finalize_kernel(const MoeW16Params p) {
  pdl_wait();
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

Moe16Plan moe16_plan(int64_t K, int64_t rows_per_expert, int64_t slots, int64_t T, int num_sms) {
  Moe16Plan pl{};
  pl.tok16 = T > 16;
  const int64_t kP = pl.tok16 ? 16 : 8;
  pl.nrb = static_cast<int>(rows_per_expert / kM16Rows);
  const int64_t nkb = K / 128;
  const int64_t units = (slots < 1 ? 1 : slots) * pl.nrb;
  int64_t cl = (2 * static_cast<int64_t>(num_sms) + units - 1) / units;
  const int64_t cl_min = (nkb + kM16MaxKBlocks - 1) / kM16MaxKBlocks;
  if (cl < cl_min) cl = cl_min;
  if (cl > kM16MaxCluster) cl = kM16MaxCluster;
  if (cl > nkb) cl = nkb;
  if (cl < 1) cl = 1;
  const int64_t kcb = (nkb + cl - 1) / cl;
  cl = (nkb + kcb - 1) / kcb;  // no rank without k-blocks
  pl.cl = static_cast<int>(cl);
  pl.kc = static_cast<int>(kcb * 128);
  const size_t fixed = static_cast<size_t>(kP) * (kcb * 256 + 16) + static_cast<size_t>(kP * kM16Rows * 4);
  int64_t R = fixed < kM16SmemBudget ? static_cast<int64_t>((kM16SmemBudget - fixed) / kM16Slot) : 0;
  if (R > kcb) R = kcb;
  if (R > kM16MaxSlots) R = kM16MaxSlots;
  pl.R = static_cast<int>(R);
  pl.ok = kcb <= kM16MaxKBlocks && (R >= 2 || (R >= 1 && kcb == 1)) && rows_per_expert % kM16Rows == 0;
  pl.smem = fixed + static_cast<size_t>(R) * kM16Slot + 1024;  // + alignment slack
  return pl;
}

template <int MODE, bool kTok16>
static cudaError_t launch_stage(const CUtensorMap& map, const MoeW16Params& p, const Moe16Plan& pl, int64_t slots,
                                cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe16_ring_kernel<MODE, kTok16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kM16SmemBudget + 1024));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(slots * pl.nrb * pl.cl));
  cfg.blockDim = dim3(kM16Threads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, moe16_ring_kernel<MODE, kTok16>, map, p, pl);
}

cudaError_t launch_moe_w4a16(const CUtensorMap& w13_map, const CUtensorMap& w2_map, const MoeW16Params& p,
                             int num_sms, cudaStream_t stream) {
  const int64_t R = static_cast<int64_t>(p.T) * p.topk;
  const int64_t S = R < p.E ? R : p.E;  // slots at most
  const Moe16Plan up = moe16_plan(p.H, 2 * static_cast<int64_t>(p.I), S, p.T, num_sms);
  const Moe16Plan dn = moe16_plan(p.I, p.H, S, p.T, num_sms);
  if (!up.ok || !dn.ok) return cudaErrorInvalidValue;
  cudaError_t e = up.tok16 ? launch_stage<0, true>(w13_map, p, up, S, stream)
                           : launch_stage<0, false>(w13_map, p, up, S, stream);
  if (e != cudaSuccess) return e;
  e = dn.tok16 ? launch_stage<1, true>(w2_map, p, dn, S, stream) : launch_stage<1, false>(w2_map, p, dn, S, stream);
  if (e != cudaSuccess) return e;
  const int64_t total = static_cast<int64_t>(p.T) * p.H;
  int64_t blocks = (total + 255) / 256;
  if (blocks > num_sms * 4) blocks = num_sms * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < 1 ? 1 : blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe16_finalize_kernel, p);
}

}  // namespace nvfp4
