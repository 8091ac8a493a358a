// W4A16 MoE for small batches: decode and prefills with few tokens per expert
// run with bf16 activations against the same NVFP4 expert banks as the W4A4
// path (the W4A4 MoE prefill page, section "Changes": W4A4 from 4 tokens per
// expert, W4A16 below; no repack).
//
//   gate_up   grouped GEMV over H; item = (slot, 64 gate rows 64j.. with the
//             64 up rows I+64j..): h = bf16(silu(a13 G) * (a13 U)) of the
//             slot's routes for h columns 64j .. 64j+63
//   down      grouped GEMV over I; item = (slot, 128 rows of W2[e]):
//             w * a2 * (h @ W2[e].T) per route, fp32
//   finalize  out[t] = bf16(sum over the token's top-k routes, in slot order)
//
// A slot is an expert in use (ascending expert id); its routes are taken in
// route order, in passes of 8 (or 16) route rows.  Every CTA derives the slot
// table from the top-k ids itself (no routing kernel).  Items are dealt
// round-robin to persistent CTAs; two producer lanes (codes, scales) stream
// the weights of the CTA's items through one ring of 128-k blocks (TMA boxes
// of 64 code bytes per row plus the 128-k block's scale atoms) without
// stopping between items.
// The compute warps stage the route rows (x or h) in windows of up to 1024 k
// as f16 after a power-of-two rescale per row and window, multiply with the
// W4A16 arithmetic of nvfp4_decode.cuh (f16 weights on mma.sync), undo the
// rescale on each window's fp32 sums and add them in window order.  Every sum
// has a fixed order: the result is deterministic.  The three kernels are
// chained by programmatic dependent launch.
#include "nvfp4_common.cuh"
#include "nvfp4_decode.cuh"
#include "nvfp4_moe.h"

namespace nvfp4 {

constexpr int kM16Groups = 2;                       // k-groups (128-k blocks dealt by parity)
constexpr int kM16CompWarps = 4 * kM16Groups;       // 4 row groups of 32 x 2 k-groups
constexpr int kM16Comp = kM16CompWarps * 32;
constexpr int kM16Threads = kM16Comp + 64;          // + a code and a scale producer warp
constexpr int kM16Rows = 128;                       // weight rows per item
constexpr int kM16Chunk = kM16Rows * 64;            // codes of one 128-k block
constexpr int kM16MaxSlots = 24;
constexpr int kM16MaxRoutes = 64 * 8;               // T <= 64, top-k <= 8
constexpr int kM16MaxExpSlots = 512;                // experts in use <= routes
constexpr int kM16WinBlocks = 8;                    // 128-k blocks per staging window
constexpr size_t kM16SmemBudget = 100 * 1024;       // two CTAs per SM with the static shared memory

// Scale bytes per ring slot: the two scale atoms of the 128-k block for each
// 128-row atom block the item's rows come from (gate and up: two).
template <int MODE>
constexpr int m16_sf_bytes() {
  return MODE == 0 ? 2048 : 1024;
}

// silu(v) = v / (1 + e^-v) with the hardware exp2 and fast division (as the W4A4
// gate_up epilogue).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// ---------------------------------------------------------------------------
// grouped GEMV (MODE 0: gate_up over H, 1: down over I)
// ---------------------------------------------------------------------------
template <int MODE, bool kTok16>
__global__ void __launch_bounds__(kM16Threads, 2)
    moe16_gemv_kernel(const __grid_constant__ CUtensorMap cmap, const MoeW16Params p, const Moe16Plan pl) {
  constexpr int kP = kTok16 ? 16 : 8;  // route rows per pass
  constexpr int kSf = m16_sf_bytes<MODE>();
  constexpr int kSlot = kM16Chunk + kSf;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kM16MaxSlots];
  __shared__ __align__(8) uint64_t empty[kM16MaxSlots];
  __shared__ unsigned int row_amax[kP];
  __shared__ uint32_t present[32];
  __shared__ int word_pre[32];
  __shared__ int s_ids[kM16MaxRoutes];       // expert of every route, -1 if dropped
  __shared__ int slot_exp[kM16MaxExpSlots];  // expert of every slot
  __shared__ int routes[kM16MaxRoutes];      // the current item's routes, in route order
  __shared__ int s_nslots, s_count;
  __shared__ volatile int abort_flag;

  // gate_up reads the top-k ids and x of the preceding kernel; the down kernel
  // is released only after that wait, so its own reads of the ids (below,
  // before its wait) see the final values.
  if (MODE == 0) pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.T * p.topk;
  const int K = MODE == 0 ? p.H : p.I;
  const int nkb = K / 128;
  const int units = MODE == 0 ? p.I / 64 : p.H / kM16Rows;  // items per slot
  const int Rs = pl.R;
  const int wb = pl.win / 128;                              // 128-k blocks per window

  uint8_t* ring = sm;
  uint8_t* ring_sf = ring + Rs * kM16Chunk;
  const int xs_stride = pl.win * 2 + 16;
  uint8_t* xs = ring_sf + Rs * kSf;                              // [kP][win*2+16] f16 inputs
  float* part = reinterpret_cast<float*>(xs + kP * xs_stride);   // [kP][128] k-group 1 sums
  float* tot = part + kP * kM16Rows;                             // [kP][128] totals (gate_up)

  // --- slots from the top-k ids ---------------------------------------------
  if (threadIdx.x < 32) present[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < Rs; ++i) {
      mbar_init(&full[i], 2);  // the code and the scale producer
      mbar_init(&empty[i], 4);
    }
    fence_barrier_init();
  }
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int e = MODE == 0 ? p.ids[r] : __ldcg(p.ids + r);
    const bool ok = e >= 0 && e < p.E;
    s_ids[r] = ok ? e : -1;
    if (ok)
      atomicOr(&present[e >> 5], 1u << (e & 31));
    else if (MODE == 0 && blockIdx.x == 0)
      record_status(p.status, kStatusBadExpert);
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t word = present[lane];
    int incl = __popc(word);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const int pre = incl - __popc(word);
    word_pre[lane] = pre;
    int k = 0;
    for (uint32_t w = word; w; w &= w - 1, ++k) slot_exp[pre + k] = 32 * lane + __ffs(w) - 1;
    if (lane == 31) s_nslots = incl;
  }
  __syncthreads();
  const int nitems = s_nslots * units;
  // routes of expert e in route order (warp-wide: every lane gets the count;
  // with `list`, the routes go to routes[])
  auto scan_routes = [&](int e, bool list) {
    int cnt = 0;
    for (int r0 = 0; r0 < R; r0 += 32) {
      const bool m = r0 + lane < R && s_ids[r0 + lane] == e;
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, m);
      if (list && m) routes[cnt + __popc(b & ((1u << lane) - 1u))] = r0 + lane;
      cnt += __popc(b);
    }
    return cnt;
  };
  // first weight row of the item (for gate_up: the gate half; the up half
  // starts I rows further)
  auto item_row = [&](int e, int unit) {
    return MODE == 0 ? e * 2 * p.I + 64 * unit : e * p.H + kM16Rows * unit;
  };

  if (warp >= kM16CompWarps) {
    // --- producer warps: lane 0 of the first streams the codes, of the second
    // the scales (every copy costs its issuing lane a few hundred cycles, so
    // two lanes keep the ring full at twice the rate); the warps count the
    // routes of every item
    const bool codes = warp == kM16CompWarps;
    if (codes && lane == 0) prefetch_tmap(&cmap);
    const uint8_t* wsf = MODE == 0 ? p.w13_sf : p.w2_sf;
    int q = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x) {
      const int e = slot_exp[it / units];
      const int unit = it - (it / units) * units;
      const int passes = (scan_routes(e, false) + kP - 1) / kP;
      if (lane == 0) {
        const int g0 = item_row(e, unit);
        const uint8_t* sf0 = wsf + static_cast<int64_t>(g0 >> 7) * (K / 64) * 512;
        const uint8_t* sf1 = wsf + static_cast<int64_t>((g0 + p.I) >> 7) * (K / 64) * 512;
        for (int pass = 0; ok && pass < passes; ++pass) {
          for (int kb = 0; kb < nkb; ++kb, ++q) {
            const int s = q % Rs;
            if (q >= Rs && !mbar_wait(&empty[s], ((q / Rs) - 1) & 1, &abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (codes) {
              mbar_arrive_expect_tx(&full[s], kM16Chunk);
              tma_load_2d(ring + s * kM16Chunk, &cmap, &full[s], kb * 64, g0);
              if (MODE == 0) tma_load_2d(ring + s * kM16Chunk + kM16Chunk / 2, &cmap, &full[s], kb * 64, g0 + p.I);
            } else {
              mbar_arrive_expect_tx(&full[s], kSf);
              bulk_load(ring_sf + s * kSf, sf0 + kb * 1024, 1024, &full[s]);
              if (MODE == 0) bulk_load(ring_sf + s * kSf + 1024, sf1 + kb * 1024, 1024, &full[s]);
            }
          }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    }
    if (lane == 0) {
      // every copy this lane issued lands before the CTA can leave (the
      // compute warps have waited for them unless a wait timed out; then
      // this wait is bounded too)
      const long long t0 = clock64();
      for (int i = 0; i < Rs && i < q; ++i) {
        const int last = i + ((q - 1 - i) / Rs) * Rs;  // last chunk issued into slot i
        while (!mbar_try_wait(smem_u32(&full[i]), (last / Rs) & 1) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
    }
    return;
  }

  // --- compute warps ----------------------------------------------------------
  if (MODE == 1) pdl_wait();  // h of the gate_up kernel
  const int g = lane >> 2, t = lane & 3;
  const int kp = warp >> 2;
  const int lr0 = (warp & 3) * 32;
  int cofs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) cofs[j] = (lr0 + 8 * j + g) * 64 + 16 * t;
  int xofs[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) xofs[i] = g * xs_stride + xchunk(4 * t + i) * 16;

  int qb = 0;  // ring chunk of the item's first 128-k block
  for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
    const int slot = it / units;
    const int unit = it - slot * units;
    const int e = slot_exp[slot];
    named_barrier_sync(1, kM16Comp);  // the previous item is done with routes[]
    if (warp == 0) {
      const int cnt = scan_routes(e, true);
      if (lane == 0) s_count = cnt;
    }
    named_barrier_sync(1, kM16Comp);
    const int count = s_count;
    const int passes = (count + kP - 1) / kP;
    // scale offsets of this thread's rows (gate_up: rows 0-63 gate, 64-127 up,
    // each half in its own pair of atoms, at row quadrant (64 unit mod 128)/32)
    int sf_off[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int lr = lr0 + 8 * j + g;
      const int quad = MODE == 0 ? (((64 * unit) & 127) >> 5) + ((lr & 63) >> 5) : lr >> 5;
      sf_off[j] = (MODE == 0 ? (lr >> 6) * 1024 : 0) + (lr & 31) * 16 + quad * 4 + 2 * (t & 1) + (t >> 1) * 512;
    }
    for (int pass = 0; pass < passes; ++pass) {
      const int tok0 = pass * kP;
      const int c = min(kP, count - tok0);
      const int qp = qb + pass * nkb;
      const bool tok_lo = g < c, tok_hi = g + 8 < c;
      // acc[a][h][q]: rows lr0 + 16a + g (+8 for q >= 2) x route rows 8h + 2t (+1 for odd q)
      float acc[2][kTok16 ? 2 : 1][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[a][h][q] = 0.0f;

      for (int w0 = 0; w0 < nkb; w0 += wb) {
        const int wn = min(wb, nkb - w0);
        // --- stage the window: raw bf16, row amax, then f16 in place ----------
        named_barrier_sync(1, kM16Comp);  // the previous window is done with xs
        if (threadIdx.x < kP) row_amax[threadIdx.x] = 0u;
        named_barrier_sync(1, kM16Comp);
        const int wunits = wn * 16;  // 16-byte units per row
        const int nunits = c * wunits;
        constexpr int kXB = kTok16 ? 2 : 4;
        for (int ub0 = threadIdx.x - lane; ub0 < nunits; ub0 += kXB * kM16Comp) {
          uint4 v[kXB];
#pragma unroll
          for (int q = 0; q < kXB; ++q) {
            const int u = ub0 + q * kM16Comp + lane;
            v[q] = make_uint4(0u, 0u, 0u, 0u);
            if (u < nunits) {
              const int i = u / wunits;
              const int k = w0 * 128 + (u - i * wunits) * 8;
              const int route = routes[tok0 + i];
              const uint16_t* src = MODE == 0 ? p.x + static_cast<int64_t>(route / p.topk) * p.H
                                              : p.h + static_cast<int64_t>(route) * p.I;
              v[q] = __ldcg(reinterpret_cast<const uint4*>(src + k));
            }
          }
#pragma unroll
          for (int q = 0; q < kXB; ++q) {
            const int ubase = ub0 + q * kM16Comp;
            if (ubase >= nunits) break;  // warp-uniform
            const int u = ubase + lane;
            const bool in = u < nunits;
            const int i = in ? u / wunits : kP;
            float m = 0.0f;
            const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] & 0xFFFFu)));
              m = fmaxf(m, fabsf(bf16_bits_to_f32(w4[j] >> 16)));
            }
            // units per row >= 16: the warp's 32 units span at most three rows
            const int i0 = ubase / wunits, i1 = min(c - 1, (ubase + 31) / wunits);
            for (int ii = i0; ii <= i1; ++ii) {
              const unsigned int mb = __reduce_max_sync(0xFFFFFFFFu, (in && i == ii) ? __float_as_uint(m) : 0u);
              if (lane == 0 && mb != 0u) atomicMax(&row_amax[ii], mb);
            }
            if (in) {
              const int k8 = (u - i * wunits) * 8;
              *reinterpret_cast<uint4*>(xs + i * xs_stride + (k8 >> 7) * 256 + xchunk((k8 & 127) >> 3) * 16) = v[q];
            }
          }
        }
        named_barrier_sync(1, kM16Comp);
        for (int u = threadIdx.x; u < nunits; u += kM16Comp) {
          const int i = u / wunits;
          const float f = pow2f(-token_shift(row_amax[i]));
          const int k8 = (u - i * wunits) * 8;
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

        // --- the window's weight blocks ---------------------------------------
        // k-group kp takes the ring chunks q with q % 2 == kp: with an even
        // ring a slot always serves the same four warps, so none of them can
        // wait on a slot two phases ahead (the parity test would pass on a
        // stale phase)
        float wacc[2][kTok16 ? 2 : 1][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) wacc[a][h][q] = 0.0f;
        for (int kb = w0 + ((kp - qp - w0) & 1); kb < w0 + wn; kb += kM16Groups) {
          const int q = qp + kb;
          const int s = q % Rs;
          if (!mbar_wait(&full[s], (q / Rs) & 1, &abort_flag, p.status)) break;
          const uint8_t* cs = ring + s * kM16Chunk;
          const uint8_t* ss = ring_sf + s * kSf;
          uint4 cw[4];
          uint32_t slo[4], shi[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            cw[j] = *reinterpret_cast<const uint4*>(cs + cofs[j]);
            scale_pair_f16(*reinterpret_cast<const uint16_t*>(ss + sf_off[j]), slo[j], shi[j]);
          }
          fence_proxy_async_smem_read();
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          const uint8_t* xb = xs + (kb - w0) * 256;
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
              mma_f16_16816(wacc[a][0], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1], wf[2 * a + 1][1], blo.x,
                            blo.y);
              mma_f16_16816(wacc[a][0], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3], wf[2 * a + 1][3], blo.z,
                            blo.w);
              if (kTok16 && c > 8) {
                mma_f16_16816(wacc[a][kTok16 ? 1 : 0], wf[2 * a][0], wf[2 * a + 1][0], wf[2 * a][1],
                              wf[2 * a + 1][1], bhi.x, bhi.y);
                mma_f16_16816(wacc[a][kTok16 ? 1 : 0], wf[2 * a][2], wf[2 * a + 1][2], wf[2 * a][3],
                              wf[2 * a + 1][3], bhi.z, bhi.w);
              }
            }
          }
        }
        // the window's sums with the rescale undone, added in window order
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              acc[a][h][q] =
                  __fmaf_rn(wacc[a][h][q], pow2f(token_shift(row_amax[h * 8 + 2 * t + (q & 1)])), acc[a][h][q]);
      }

      // --- the pass's sums: k-group 1 into shared memory, k-group 0 adds --------
      if (kp == 1) {
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = h * 8 + 2 * t + (q & 1);
              if (i < c) part[i * kM16Rows + lr0 + a * 16 + g + 8 * (q >> 1)] = acc[a][h][q];
            }
      }
      named_barrier_sync(1, kM16Comp);
      if (kp == 0) {
        const float wa = MODE == 1 ? __ldg(p.alpha2 + e) : 0.0f;
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int h = 0; h < (kTok16 ? 2 : 1); ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = h * 8 + 2 * t + (q & 1);
              if (i < c) {
                const int row = lr0 + a * 16 + g + 8 * (q >> 1);
                const float v = __fadd_rn(acc[a][h][q], part[i * kM16Rows + row]);
                if (MODE == 0) {
                  tot[i * kM16Rows + row] = v;
                } else {
                  const int route = routes[tok0 + i];
                  __stcg(p.dn + static_cast<int64_t>(route) * p.H + kM16Rows * unit + row,
                         __fmul_rn(__fmul_rn(__ldg(p.topk_w + route), wa), v));
                }
              }
            }
      }
      if (MODE == 0) {
        // h = bf16(silu(a13 G) * (a13 U)) for gate row jj and up row 64 + jj
        named_barrier_sync(1, kM16Comp);
        const float a13 = __ldg(p.alpha13 + e);
        for (int u = threadIdx.x; u < c * 64; u += kM16Comp) {
          const int i = u >> 6, jj = u & 63;
          const float G = tot[i * kM16Rows + jj], U = tot[i * kM16Rows + 64 + jj];
          const float hv = silu_fast(__fmul_rn(a13, G)) * __fmul_rn(a13, U);
          p.h[static_cast<int64_t>(routes[tok0 + i]) * p.I + 64 * unit + jj] =
              __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        }
      }
    }
    qb += passes * nkb;
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
    // all loads of the token's routes in flight at once, then the sum in order
    bool ok[8];
    float v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int e = s < p.topk ? p.ids[tkn * p.topk + s] : -1;
      ok[s] = e >= 0 && e < p.E;
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) v[s] = ok[s] ? __ldcg(p.dn + (tkn * p.topk + s) * p.H + n) : 0.0f;
    float y = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (ok[s]) y += v[s];
    p.out[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
Moe16Plan moe16_plan(int mode, int64_t K, int64_t T, int64_t E, int topk, int64_t units, int num_sms) {
  Moe16Plan pl{};
  pl.tok16 = T > 16;
  const int64_t kP = pl.tok16 ? 16 : 8;
  const int64_t nkb = K / 128;
  const int64_t wb = nkb < kM16WinBlocks ? nkb : kM16WinBlocks;
  pl.win = static_cast<int>(wb * 128);
  const int64_t slot = kM16Chunk + (mode == 0 ? m16_sf_bytes<0>() : m16_sf_bytes<1>());
  const size_t fixed =
      static_cast<size_t>(kP) * (wb * 256 + 16) + static_cast<size_t>((mode == 0 ? 2 : 1) * kP * kM16Rows * 4);
  int64_t slots = fixed < kM16SmemBudget ? static_cast<int64_t>((kM16SmemBudget - fixed) / slot) : 0;
  if (slots > kM16MaxSlots) slots = kM16MaxSlots;
  slots &= ~int64_t{1};  // even: each slot belongs to one k-group
  pl.R = static_cast<int>(slots);
  const int64_t R = T * topk;
  pl.ok = slots >= 2 && nkb >= 1 && K % 128 == 0 && R <= kM16MaxRoutes && E <= 1024;
  pl.smem = fixed + static_cast<size_t>(slots) * slot + 1024;  // + alignment slack
  // persistent CTAs: two per SM, no more than the items can use
  const int64_t max_items = (E < R ? E : R) * units;
  const int64_t ctas = 2 * static_cast<int64_t>(num_sms);
  pl.ctas = static_cast<int>(ctas < max_items ? ctas : max_items);
  return pl;
}

template <int MODE, bool kTok16>
static cudaError_t launch_stage(const CUtensorMap& map, const MoeW16Params& p, const Moe16Plan& pl,
                                cudaStream_t stream) {
  // the attribute belongs to the current device: set it on every launch
  cudaError_t e = cudaFuncSetAttribute(moe16_gemv_kernel<MODE, kTok16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kM16SmemBudget + 1024));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas));
  cfg.blockDim = dim3(kM16Threads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe16_gemv_kernel<MODE, kTok16>, map, p, pl);
}

cudaError_t launch_moe_w4a16(const CUtensorMap& w13_map, const CUtensorMap& w2_map, const MoeW16Params& p,
                             int num_sms, cudaStream_t stream) {
  const Moe16Plan up = moe16_plan(0, p.H, p.T, p.E, p.topk, p.I / 64, num_sms);
  const Moe16Plan dn = moe16_plan(1, p.I, p.T, p.E, p.topk, p.H / kM16Rows, num_sms);
  if (!up.ok || !dn.ok) return cudaErrorInvalidValue;
  cudaError_t e = up.tok16 ? launch_stage<0, true>(w13_map, p, up, stream)
                           : launch_stage<0, false>(w13_map, p, up, stream);
  if (e != cudaSuccess) return e;
  e = dn.tok16 ? launch_stage<1, true>(w2_map, p, dn, stream) : launch_stage<1, false>(w2_map, p, dn, stream);
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
