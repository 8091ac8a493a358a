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
#include "nvfp4_decode.cuh"
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

// ---------------------------------------------------------------------------
// Default decode path.
//
// A CTA owns one 128-row block of the weight and a k-range of kc elements; the
// k-ranges of a row block form one thread-block cluster (at most 8 CTAs).
//
// Weight stream.  One producer lane copies the CTA's slice into a ring of
// shared-memory slots: per 128-k block one TMA tile of codes (64 bytes x 128
// rows) and its two scale atoms (1 KB, contiguous in the swizzled layout).  As
// many slots as fit are filled, and the blocks beyond them are prefetched into
// L2, before the kernel waits for the preceding kernel on the stream
// (programmatic dependent launch); the producer refills slots as the compute
// warps release them.  A call has one CTA per SM at most (the cluster size is
// the number of SMs over the row blocks).  Below four tokens a CTA takes
// under half of an SM's shared memory and registers, so the next call's CTAs
// are resident while this call computes and their weight copies overlap it;
// from four tokens a CTA takes the whole SM (see RingShape).
//
// Activations.  After the dependency wait the compute warps stage the CTA's
// k-range of the T tokens as f16: each (token, 128-k block) is rescaled by its
// own power of two, which puts its largest magnitude in [2^14, 2^15), so one
// half-warp finds the block maximum and converts the block with no exchange
// beyond its own lanes.  A bf16 value within 2^31 of that maximum converts
// exactly; smaller values round on the f16 subnormal grid, an error below
// 2^-39 of the maximum.
//
// Arithmetic.  Sixteen or twenty-four compute warps: eight 16-row tiles x two
// or three k-groups (the 128-k blocks are dealt to the groups round-robin).  mma.sync.m16n8k16 with
// 16 weight rows as A and 8 tokens as B (tokens 8..15 in a second MMA), each
// 128-k block into a fresh fp32 accumulator that is then added, times the
// block's inverse rescale (a power of two, exact), to the running sums.
// Inside a 128-k block the k order is permuted so that one 16-byte code load
// of row r (k = 32t .. 32t+31 for lane t) feeds A of that row directly; the
// activations are staged in the same order.  A code byte becomes an f16x2
// pair with one hardware conversion, times the block scale: e2m1 * E4M3 has
// at most 6 significant bits and lies in [2^-10, 2688], so it is exact in
// f16, and products of f16 values are exact in fp32.
//
// Split-K sum.  The k-groups add their partials in shared memory in a fixed
// order.  Rank r of the cluster owns rows [r * rows_per, ...) of the
// row block: every CTA pushes its partials of those rows into the owner's
// shared memory with st.async, which counts the bytes on the owner's
// mbarrier; the owner adds the cluster's partials in rank order and writes
// bf16.  Nobody waits for anything but the bytes it needs, and the result is
// the same from run to run.
// ---------------------------------------------------------------------------
constexpr int kRingRows = 128;             // weight rows per CTA (one scale-atom row block)
constexpr int kRingTiles = kRingRows / 16;  // 16-row MMA tiles per CTA
// Two layouts.  Below kRingWideFromT tokens: two k-groups (16 compute warps),
// two CTAs per SM, so that the next call's CTAs are resident beside this
// call's and copy their weights while it computes.  From kRingWideFromT
// tokens the k-loop has more work per weight byte: three k-groups (24 compute
// warps, up to 80 registers) and one CTA per SM, whose ring then usually holds
// the CTA's whole weight slice.
template <bool kTok16, int kG> struct RingShape {
  static constexpr int kGroups = kG;                        // k-groups
  static constexpr int kCompWarps = kRingTiles * kGroups;   // one tile per warp
  static constexpr int kThreads = (kCompWarps + 1) * 32;    // + one producer warp
  static constexpr int kMinBlocks = kG == 2 ? 2 : 1;
};
constexpr int kRingWideFromT = 4;
__host__ __device__ constexpr int ring_groups(int64_t T) { return T >= kRingWideFromT ? 3 : 2; }
constexpr int kRingMaxSlots = 24;
constexpr int kRingChunk = kRingRows * 64;            // codes of one 128-k block
constexpr int kRingChunkSf = 1024;                    // its two scale atoms
constexpr int kRingSlot = kRingChunk + kRingChunkSf;
constexpr int kRingMaxCluster = 8;
// dynamic shared memory per CTA: two CTAs per SM with their static shared
// memory, or one
constexpr size_t ring_smem_budget(int groups) { return groups == 2 ? 109 * 1024 : 220 * 1024; }
constexpr int kStageLoads = 4;                        // activation units in flight per lane while staging

__device__ __forceinline__ uint32_t mapa_u32(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Store one fp32 into another CTA's shared memory and count its 4 bytes on
// that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
               "r"(__float_as_uint(v)), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

template <bool kTok16, int kG>
__global__ void __launch_bounds__(RingShape<kTok16, kG>::kThreads, RingShape<kTok16, kG>::kMinBlocks) gemv_ring_kernel(
    const __grid_constant__ CUtensorMap cmap, const uint16_t* __restrict__ x, int T, int64_t ldx,
    const uint8_t* __restrict__ w_sf, int N, int K, int kc, int R, const float* __restrict__ d_alpha,
    uint16_t* __restrict__ out, int64_t ldo, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ __align__(8) uint64_t full[kRingMaxSlots];
  __shared__ __align__(8) uint64_t empty[kRingMaxSlots];
  __shared__ __align__(8) uint64_t red_bar;
  __shared__ volatile int abort_flag;

  constexpr int kGroups = RingShape<kTok16, kG>::kGroups;
  constexpr int kCompWarps = RingShape<kTok16, kG>::kCompWarps;
  constexpr int kComp = kCompWarps * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = (warp == kCompWarps) && lane == 0;
  if (producer) prefetch_tmap(&cmap);
  const uint32_t ncl = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int rb = static_cast<int>(blockIdx.x / ncl);
  const int k_begin = static_cast<int>(rank) * kc;
  const int k_len = max(0, min(kc, K - k_begin));
  const int nkb = k_len / 128;
  const int kcb = kc / 128;
  const int rows_per = (kRingRows + static_cast<int>(ncl) - 1) / static_cast<int>(ncl);
  const int my_rows = min(rows_per, kRingRows - static_cast<int>(rank) * rows_per);
  uint8_t* ring = sm;                                                // R x codes
  uint8_t* ring_sf = ring + R * kRingChunk;                          // R x scales
  const int xs_stride = kc * 2 + 16;
  uint8_t* xs = ring_sf + R * kRingChunkSf;                          // [T][kc] f16 activations, permuted
  float* xmul = reinterpret_cast<float*>(xs + T * xs_stride);        // [kcb][16] inverse rescales
  float* part = xmul + kcb * 16;                                     // [T][128] this CTA's partials
  float* recv = part + T * kRingRows;                                // [ncl][T][rows_per] partials of my rows
  const uint8_t* sf_src = w_sf + (static_cast<int64_t>(rb) * (K / 64) + k_begin / 64) * 512;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRingTiles);
    }
    mbar_init(&red_bar, 1);
    // the cluster's pushes of my rows: (ncl - 1) CTAs x T tokens x my_rows fp32
    mbar_arrive_expect_tx(&red_bar, (ncl - 1) * static_cast<uint32_t>(T * my_rows) * 4u);
    fence_barrier_init();
  }
  __syncthreads();
  // every CTA's red_bar is initialised before anyone pushes (the matching wait
  // comes after the k-loop)
  cluster_arrive_relaxed();
  int issued = 0;  // producer: fills issued so far (chunk c goes to slot c % R, phase c / R)
  if (producer) {
    // the weight does not depend on the preceding kernel: fill the ring now
    const int pre = min(R, nkb);
    issued = pre;
    for (int c = 0; c < pre; ++c) {
      mbar_arrive_expect_tx(&full[c], kRingSlot);
      tma_load_2d(ring + c * kRingChunk, &cmap, &full[c], k_begin / 2 + c * 64, rb * kRingRows);
      bulk_load(ring_sf + c * kRingChunkSf, sf_src + c * kRingChunkSf, kRingChunkSf, &full[c]);
    }
    // the blocks the ring cannot hold yet go to L2, so that the refills after
    // the dependency wait read them from there
    for (int c = pre; c < nkb; ++c) {
      tma_prefetch_2d(&cmap, k_begin / 2 + c * 64, rb * kRingRows);
      bulk_prefetch_l2(sf_src + c * kRingChunkSf, kRingChunkSf);
    }
  }

  // activations, alpha and the output follow the preceding kernel
  pdl_wait();
  // the next call may start now: its CTAs fit beside this call's and copy their
  // weights while this call computes.  Released only here, after the wait, so
  // that no more than two calls are in flight and the prefetched weights of
  // the next one are not pushed out of L2 by calls further ahead.
  pdl_launch_dependents();
  if (producer) {
    // refill slots as the compute warps release them
    int s = 0, round = 1;
    for (int c = R; c < nkb; ++c) {
      if (!mbar_wait(&empty[s], (round - 1) & 1, &abort_flag, status)) break;
      mbar_arrive_expect_tx(&full[s], kRingSlot);
      tma_load_2d(ring + s * kRingChunk, &cmap, &full[s], k_begin / 2 + c * 64, rb * kRingRows);
      bulk_load(ring_sf + s * kRingChunkSf, sf_src + c * kRingChunkSf, kRingChunkSf, &full[s]);
      ++issued;
      if (++s == R) {
        s = 0;
        ++round;
      }
    }
  } else if (warp < kCompWarps) {
    // stage the activations: half-warp h of warp w takes the (token, block)
    // pairs p = 2w + h, 2w + h + 2 * kCompWarps, ...; lane l16 holds the
    // 16-byte unit l16 (k = 8 l16 .. 8 l16 + 7) of the block
    {
      const int npairs = T * nkb;
      const int l16 = lane & 15;
      for (int p0 = warp * 2 + (lane >> 4); p0 - (lane >> 4) < npairs; p0 += kStageLoads * 2 * kCompWarps) {
        uint4 v[kStageLoads];
#pragma unroll
        for (int q = 0; q < kStageLoads; ++q) {
          const int p = p0 + q * 2 * kCompWarps;
          v[q] = make_uint4(0u, 0u, 0u, 0u);
          if (p < npairs) {
            const int tok = p / nkb, kb = p - (p / nkb) * nkb;
            v[q] = ldg_v4_hint(x + static_cast<int64_t>(tok) * ldx + k_begin + kb * 128 + l16 * 8, act_policy());
          }
        }
#pragma unroll
        for (int q = 0; q < kStageLoads; ++q) {
          const int p = p0 + q * 2 * kCompWarps;
          if (p - (lane >> 4) >= npairs) break;  // warp-uniform
          const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
          // largest magnitude: bf16 bit patterns of |x| order like the values
          uint32_t m = 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e) m = max(m, max(w4[e] & 0x7FFFu, (w4[e] >> 16) & 0x7FFFu));
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
          if (p < npairs) {
            const int tok = p / nkb, kb = p - (p / nkb) * nkb;
            const int sh = token_shift(m << 16);
            const float f = pow2f(-sh);
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 h =
                  __floats2half2_rn(bf16_bits_to_f32(w4[e] & 0xFFFFu) * f, bf16_bits_to_f32(w4[e] >> 16) * f);
              o[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(xs + tok * xs_stride + kb * 256 + xchunk(l16) * 16) =
                make_uint4(o[0], o[1], o[2], o[3]);
            if (l16 == 0) xmul[kb * 16 + tok] = pow2f(sh);
          }
        }
      }
    }
    named_barrier_sync(1, kComp);

    const int g = lane >> 2, t = lane & 3;
    const int kp = warp / kRingTiles;
    const int r0 = (warp % kRingTiles) * 16 + g, r1 = r0 + 8;
    const int cofs0 = r0 * 64 + 16 * t, cofs1 = r1 * 64 + 16 * t;
    const int sf0 = (r0 & 31) * 16 + (r0 >> 5) * 4 + 2 * (t & 1) + (t >> 1) * 512;
    const int sf1 = (r1 & 31) * 16 + (r1 >> 5) * 4 + 2 * (t & 1) + (t >> 1) * 512;
    int xofs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xofs[i] = g * xs_stride + xchunk(4 * t + i) * 16;
    const bool tok_lo = g < T, tok_hi = g + 8 < T;
    constexpr int kH = kTok16 ? 2 : 1;
    // acc[h][c]: row r0 (c < 2) or r1 (c >= 2) x token 8h + 2t + (c & 1)
    float acc[kH][4];
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[h][c] = 0.0f;
    // chunk kb sits in slot kb % R, phase (kb / R) & 1; R >= kGroups
    int s = kp;
    uint32_t ph = 0;
    const bool refilled = nkb > R;  // slots are released to the producer only then
    for (int kb = kp; kb < nkb; kb += kGroups) {
      if (!mbar_test_wait(smem_u32(&full[s]), ph) && !mbar_wait_slow(&full[s], ph, &abort_flag, status)) break;
      const uint8_t* cs = ring + s * kRingChunk;
      const uint8_t* ss = ring_sf + s * kRingChunkSf;
      const uint4 c0 = *reinterpret_cast<const uint4*>(cs + cofs0);
      const uint4 c1 = *reinterpret_cast<const uint4*>(cs + cofs1);
      uint32_t slo0, shi0, slo1, shi1;
      scale_pair_f16(*reinterpret_cast<const uint16_t*>(ss + sf0), slo0, shi0);
      scale_pair_f16(*reinterpret_cast<const uint16_t*>(ss + sf1), slo1, shi1);
      if (refilled) {
        fence_proxy_async_smem_read();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      s += kGroups;
      if (s >= R) {
        s -= R;
        ph ^= 1u;
      }
      // in the two-group layout the two MMAs of a code word go to separate
      // accumulators (two chains of four dependent MMAs per block instead of
      // one of eight: 1-2 % per call at 1-2 tokens); the three-group layouts
      // keep one chain, where the extra registers bought nothing
      constexpr int kS = (kTok16 || kG == 3) ? 1 : 2;
      float blk[kH][4], blk2[kS == 2 ? kH : 1][4];
#pragma unroll
      for (int h = 0; h < kH; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) blk[h][c] = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) blk2[0][c] = 0.0f;
      const uint8_t* xb = xs + kb * 256;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w0 = (i == 0) ? c0.x : (i == 1) ? c0.y : (i == 2) ? c0.z : c0.w;
        const uint32_t w1 = (i == 0) ? c1.x : (i == 1) ? c1.y : (i == 2) ? c1.z : c1.w;
        uint32_t a[4], b[4];
        e2m1x4_to_f16x2(w0, a);
        e2m1x4_to_f16x2(w1, b);
        const uint32_t m0 = (i < 2) ? slo0 : shi0, m1 = (i < 2) ? slo1 : shi1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          a[e] = f16x2_mul(a[e], m0);
          b[e] = f16x2_mul(b[e], m1);
        }
        uint4 xl = make_uint4(0u, 0u, 0u, 0u);
        if (tok_lo) xl = *reinterpret_cast<const uint4*>(xb + xofs[i]);
        // A: rows r0 / r1, k pairs (0,1) then (2,3) of code word i
        mma_f16_16816(blk[0], a[0], b[0], a[1], b[1], xl.x, xl.y);
        mma_f16_16816(kS == 2 ? blk2[0] : blk[0], a[2], b[2], a[3], b[3], xl.z, xl.w);
        if constexpr (kTok16) {
          uint4 xh = make_uint4(0u, 0u, 0u, 0u);
          if (tok_hi) xh = *reinterpret_cast<const uint4*>(xb + xofs[i] + 8 * xs_stride);
          mma_f16_16816(blk[kH - 1], a[0], b[0], a[1], b[1], xh.x, xh.y);
          mma_f16_16816(blk[kH - 1], a[2], b[2], a[3], b[3], xh.z, xh.w);
        }
      }
      // undo the block's rescale (exact) and add to the running sums
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        const float2 mu = *reinterpret_cast<const float2*>(xmul + kb * 16 + 8 * h + 2 * t);
        if constexpr (kS == 2) {
#pragma unroll
          for (int c = 0; c < 4; ++c) blk[h][c] += blk2[h][c];
        }
        acc[h][0] = fmaf(blk[h][0], mu.x, acc[h][0]);
        acc[h][1] = fmaf(blk[h][1], mu.y, acc[h][1]);
        acc[h][2] = fmaf(blk[h][2], mu.x, acc[h][2]);
        acc[h][3] = fmaf(blk[h][3], mu.y, acc[h][3]);
      }
    }
    // the k-groups' partials, added in a fixed order: group 0 + (group 1 + (...))
    for (int grp = kGroups - 1; grp >= 0; --grp) {
      if (kp == grp) {
#pragma unroll
        for (int h = 0; h < kH; ++h)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int row = (c < 2) ? r0 : r1;
            const int tok = h * 8 + 2 * t + (c & 1);
            if (tok < T) {
              float* pp = part + tok * kRingRows + row;
              *pp = (grp == kGroups - 1) ? acc[h][c] : __fadd_rn(acc[h][c], *pp);
            }
          }
      }
      if (grp > 0) named_barrier_sync(2, kComp);
    }
  }
  __syncthreads();
  if (abort_flag && producer) {
    // wind down after a timed-out wait: let this CTA's copies still in flight
    // land (bounded) before its shared memory is released
    const long long t0 = clock64();
    for (int i = 0; i < R && i < issued; ++i) {
      const int last = i + ((issued - 1 - i) / R) * R;  // last chunk issued into slot i
      while (!mbar_try_wait(smem_u32(&full[i]), (last / R) & 1) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  }
  // split-K sum: push the partials of every owner's rows to it, in place
  // [rank][tok][row - owner's first row] of its receive buffer
  cluster_wait();
  const uint32_t recv_local = smem_u32(recv);
  const uint32_t bar_local = smem_u32(&red_bar);
  for (int e = threadIdx.x; e < T * kRingRows; e += blockDim.x) {
    const int tok = e / kRingRows, row = e - (e / kRingRows) * kRingRows;
    const int owner = row / rows_per;
    const int idx = (static_cast<int>(rank) * T + tok) * rows_per + (row - owner * rows_per);
    const float v = part[e];
    if (owner == static_cast<int>(rank))
      recv[idx] = v;
    else
      st_async_f32(mapa_u32(recv_local + idx * 4, owner), v, mapa_u32(bar_local, owner));
  }
  __syncthreads();  // my own contribution is in recv
  // wait for the cluster's pushes of my rows, not cut short by an abort, so
  // that no push lands after this CTA has exited
  bool got = false;
  {
    const long long t0 = clock64();
    while (!(got = mbar_try_wait(bar_local, 0)) && clock64() - t0 < 2 * kWaitLimitCycles) {
    }
    if (!got && threadIdx.x == 0) record_status(status, kStatusTimeout);
  }
  if (got) {
    const float alpha = __ldg(d_alpha);
    for (int e = threadIdx.x; e < T * my_rows; e += blockDim.x) {
      const int tok = e / my_rows, rl = e - (e / my_rows) * my_rows;
      float sum = 0.0f;
      for (int q = 0; q < static_cast<int>(ncl); ++q) sum += recv[(q * T + tok) * rows_per + rl];
      const int n = rb * kRingRows + static_cast<int>(rank) * rows_per + rl;
      if (n < N)
        stg_u16_hint(out + static_cast<int64_t>(tok) * ldo + n, __bfloat16_as_ushort(__float2bfloat16_rn(sum * alpha)),
                     act_policy());  // the next layer's input
    }
  }
}

GemvRingPlan gemv_ring_plan(int64_t T, int64_t N, int64_t K, int num_sms) {
  GemvRingPlan p{};
  const int64_t row_blocks = (N + kRingRows - 1) / kRingRows;
  const int64_t kblocks = K / 128;
  // one CTA per SM: the next call's CTAs fit beside this call's and start
  // their weight copies while this call computes.  More k-splits only when
  // the activations of a CTA leave too little room for the ring.
  int64_t cl = static_cast<int64_t>(num_sms) / row_blocks;
  cl = cl < 1 ? 1 : (cl > kRingMaxCluster ? kRingMaxCluster : cl);
  if (cl > kblocks) cl = kblocks;
  for (;; ++cl) {
    const int64_t kcb = (kblocks + cl - 1) / cl;
    const int64_t ncl = (kblocks + kcb - 1) / kcb;  // no CTA without k-blocks
    const int64_t rows_per = (kRingRows + ncl - 1) / ncl;
    // activations, inverse rescales, partials and the receive buffer
    const size_t fixed = static_cast<size_t>(T) * (kcb * 256 + 16) + static_cast<size_t>(kcb * 16 * 4) +
                         static_cast<size_t>(T * kRingRows * 4) + static_cast<size_t>(ncl * T * rows_per * 4);
    const int64_t groups = ring_groups(T);
    const size_t budget = ring_smem_budget(static_cast<int>(groups));
    int64_t slots = fixed < budget ? static_cast<int64_t>((budget - fixed) / kRingSlot) : 0;
    if (slots > kcb) slots = kcb;
    if (slots > kRingMaxSlots) slots = kRingMaxSlots;
    // a ring that is refilled holds a multiple of the k-groups: each slot then
    // stays with one k-group (kb and kb + R are dealt to the same group), so
    // no warp waits on a slot two phases ahead of the last one it read, where
    // the mbarrier parity test would pass on a stale phase
    if (slots < kcb && slots > 1) slots -= slots % groups;
    const bool ok = slots >= groups || (slots >= 1 && slots >= kcb);
    const bool roomy = slots >= kcb || slots >= 4;
    if ((ok && roomy) || cl >= kRingMaxCluster || cl >= kblocks) {
      p.cl = static_cast<int>(ncl);
      p.kc = static_cast<int>(kcb * 128);
      p.row_blocks = row_blocks;
      p.R = static_cast<int>(slots);
      p.ok = ok;
      p.smem = fixed + static_cast<size_t>(slots) * kRingSlot + 1024;  // + alignment slack
      return p;
    }
  }
}

template <bool kTok16, int kG>
static cudaError_t launch_ring_t(const CUtensorMap& cmap, const void* x, int64_t T, int64_t ldx, const uint8_t* w_sf,
                                 int64_t N, int64_t K, const float* d_alpha, void* out, int64_t ldo,
                                 const GemvRingPlan& plan, int* status, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(gemv_ring_kernel<kTok16, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(ring_smem_budget(kG) + 1024));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.row_blocks * plan.cl));
  cfg.blockDim = dim3(RingShape<kTok16, kG>::kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(plan.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemv_ring_kernel<kTok16, kG>, cmap, static_cast<const uint16_t*>(x),
                            static_cast<int>(T), ldx, w_sf, static_cast<int>(N), static_cast<int>(K), plan.kc, plan.R,
                            d_alpha, static_cast<uint16_t*>(out), ldo, status);
}

cudaError_t launch_gemv_w4a16_ring(const CUtensorMap& cmap, const void* x, int64_t T, int64_t ldx,
                                   const uint8_t* w_sf, int64_t N, int64_t K, const float* d_alpha, void* out,
                                   int64_t ldo, const GemvRingPlan& plan, int* status, cudaStream_t stream) {
  static_assert(kRingWideFromT <= 8, "T > 8 runs the three-group layout");
  if (T > 8) return launch_ring_t<true, 3>(cmap, x, T, ldx, w_sf, N, K, d_alpha, out, ldo, plan, status, stream);
  if (ring_groups(T) == 3)
    return launch_ring_t<false, 3>(cmap, x, T, ldx, w_sf, N, K, d_alpha, out, ldo, plan, status, stream);
  return launch_ring_t<false, 2>(cmap, x, T, ldx, w_sf, N, K, d_alpha, out, ldo, plan, status, stream);
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
  if (smem > 48 * 1024) {  // the attribute belongs to the current device: set it on every launch
    cudaError_t e = cudaFuncSetAttribute(gemv_w4a16_kernel<kTok16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
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
