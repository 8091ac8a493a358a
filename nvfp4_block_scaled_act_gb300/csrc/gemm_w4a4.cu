// Block-scaled NVFP4 x NVFP4 GEMM on the sm_103a tensor cores
// (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: e2m1 operands, one UE4M3 scale per
// 16 k-elements, fp32 accumulation in TMEM).
//
// Computes, for 128-row tiles of A and column tiles of B (both K-major NVFP4):
//   acc[m, n] = sum_k e2m1(A[m,k]) s_A[m,k/16] * e2m1(B[n,k]) s_B[n,k/16]
// and hands acc to one of four epilogues:
//   kEpiDense      out = bf16(alpha * acc)                       (W4A4 linear)
//   kEpiGatedQuant h = silu(alpha_e * G) * (alpha_e * U) -> NVFP4 codes/scales
//                  (MoE gate_up: B tile = 128 gate rows then 128 up rows)
//   kEpiGatedAmax  per-expert max |h| (calibration of the second input global)
//   kEpiDownSum    y[t] += w_route * alpha_e * acc with fp32 bulk reductions
//                  (MoE down and top-k sum); kEpiDownDirect the same with
//                  vector reductions from registers, for few routes per expert
// The W4A4 linear of "run nvfp4 linears on nvfp4 activations on sm_120" and the
// warp-specialised gate_up / down GEMMs of the W4A4 MoE prefill page (both
// section "Changes") were written for mma.sync on sm_120; this kernel keeps
// their dataflow and epilogue fusion and maps it onto tcgen05 and TMEM.
//
// Two kernels.  gemm_nvfp4_kernel (below) runs one CTA per SM on 128 x BN tiles
// and serves the grouped MoE GEMMs; gemm_pair_kernel (further down) runs the
// dense W4A4 linear on CTA pairs and 256 x 256 tiles.
//
// gemm_nvfp4_kernel structure (one CTA of 16 warps per SM, persistent over
// tiles n-fastest):
//   warp 0      operand producer: a 128x128-byte A box and the B tile (one
//               BN-row box, or one 128-row box per block for the MoE gate
//               and up blocks; 128-byte swizzle) into a STAGES-deep smem ring.
//   warp 2      scale producer: the stage's 512-byte scale atoms of A and B
//               (bulk copies, contiguous in the 128x4 layout).  Splitting the
//               copies over two warps halves the serial issue work per stage
//               (each TMA or bulk copy costs its issuing lane about 100 cycles).
//   warp 1      allocates TMEM; one lane issues 4 MMAs of K = 64 per 256-k
//               stage once the stage's scales are in TMEM; tcgen05.commit
//               releases smem stages and publishes finished accumulators.
//   warps 4-7   scale writers: warp q copies the stage's scale atoms from smem
//               into TMEM lane quadrant q with tcgen05.st (the replicated
//               layout the block-scaled MMA reads), so the MMA lane issues
//               nothing but MMAs.
//   warps 8-15  epilogue: tcgen05.ld of the accumulator, fused epilogue math,
//               global stores; an accumulator is released as soon as it has
//               been read, so the next tile's MMAs overlap the epilogue math.
// setmaxnreg moves registers from the producer/MMA/scale warps (64) to the
// epilogue warps (192).
// Every mbarrier wait is bounded; a timeout sets the device status word and
// every role winds down (waiting for its own copies and MMAs) before TMEM is freed.
#include "nvfp4_common.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

template <int BN_, int NUM_ACC_, int STAGES_, int MODE_>
struct GemmCfg {
  static constexpr int BN = BN_;           // MMA N (B rows per tile)
  static constexpr int NUM_ACC = NUM_ACC_;
  static constexpr int STAGES = STAGES_;
  static constexpr int MODE = MODE_;
  static constexpr int BM = 128;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int NBLK = BN / 128;    // 128-row B boxes per stage
  static constexpr int SFA_BYTES = 2048;   // 4 atoms = 256 k of 128 rows
  static constexpr int SFB_BYTES = NBLK * 2048;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // MoE down: fp32 staging of the 128 rows x BN columns of a tile (row pitch
  // padded by 16 bytes) for the bulk reduce-adds into y
  static constexpr int EPI_PITCH = BN * 4 + 16;
  static constexpr int EPI_BYTES = MODE_ == kEpiDownSum ? 128 * EPI_PITCH : 0;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024;
  static constexpr int SF_COLS = 16 + 4 * (BN / 32);  // TMEM scale columns per stage
  static constexpr int SF_BASE = NUM_ACC * BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr bool GROUPED = MODE != kEpiDense;
  static_assert(SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "smem budget");
};

// ---------------------------------------------------------------------------
// epilogue helpers
// ---------------------------------------------------------------------------
// silu(v) = v / (1 + e^-v) with the hardware exp2 and fast division (a few ulp
// from the correctly rounded value; both the calibration and the quantising
// epilogue use it).
__device__ __forceinline__ float silu_f32(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1,%2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}

// 32 fp32 accumulator values * alpha -> bf16, stored as four 16-byte vectors;
// `remaining` = valid columns from dst on (a multiple of 8).
__device__ __forceinline__ void store_bf16_32(uint16_t* dst, const uint32_t (&r)[32], float alpha, int remaining) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    if (8 * v < remaining) {
      uint4 o;
      o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * alpha, __uint_as_float(r[8 * v + 1]) * alpha);
      o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * alpha, __uint_as_float(r[8 * v + 3]) * alpha);
      o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * alpha, __uint_as_float(r[8 * v + 5]) * alpha);
      o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * alpha, __uint_as_float(r[8 * v + 7]) * alpha);
      *reinterpret_cast<uint4*>(dst + 8 * v) = o;
    }
  }
}


// Bulk reduce-add of `bytes` fp32 from shared memory into global memory
// (both 16-byte aligned, bytes % 16 == 0), in this thread's bulk group.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const float* ssrc, uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n\t"
      "cp.async.bulk.commit_group;" ::"l"(gdst),
      "r"(smem_u32(ssrc)), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Quantise 64 consecutive h values (four 16-blocks) of one row: 32 code bytes
// and 4 scale bytes.  r_of_s8[s] = g / S(s) (IEEE division, per E4M3 byte).
__device__ __forceinline__ void quant64(const float (&h)[64], float g, const float* r_of_s8, uint4& c0, uint4& c1,
                                        uint32_t& s4) {
  uint32_t words[8];
  s4 = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = h[16 * b + i];
      amax = fmaxf(amax, fabsf(v[i]));
    }
    BlockScale bs;
    bs.s8 = f32_to_e4m3(__fmul_rn(__fdiv_rn(amax, 6.0f), g));
    bs.r = r_of_s8[bs.s8];
    const uint2 w = encode_block16(v, bs.r, bs.r == 0.0f);
    words[2 * b] = w.x;
    words[2 * b + 1] = w.y;
    s4 |= bs.s8 << (8 * b);
  }
  c0 = make_uint4(words[0], words[1], words[2], words[3]);
  c1 = make_uint4(words[4], words[5], words[6], words[7]);
}

// Gated epilogue of one row and 64 h columns: h = silu(a * G) * (a * U) from
// the gate and up accumulator columns (g0 g1 | u0 u1), then either the NVFP4
// codes and scales of h at permuted row prow, h columns 64 * hcb .. (quant),
// or the row's max |h| folded into the expert's amax (calibration).
template <int MODE>
__device__ __forceinline__ void gated_row64(const uint32_t (&g0)[32], const uint32_t (&g1)[32],
                                            const uint32_t (&u0)[32], const uint32_t (&u1)[32], float a, int rm,
                                            int e, int prow, int hcb, const GemmParams& p, const float* r_of_s8,
                                            float g_out) {
  float h[64];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    h[i] = __fmul_rn(silu_f32(__fmul_rn(a, __uint_as_float(g0[i]))), __fmul_rn(a, __uint_as_float(u0[i])));
    h[32 + i] = __fmul_rn(silu_f32(__fmul_rn(a, __uint_as_float(g1[i]))), __fmul_rn(a, __uint_as_float(u1[i])));
  }
  if constexpr (MODE == kEpiGatedQuant) {
    if (rm >= 0) {
      uint4 c0, c1;
      uint32_t s4;
      quant64(h, g_out, r_of_s8, c0, c1, s4);
      uint8_t* dst = p.q_codes + static_cast<int64_t>(prow) * p.q_row_bytes + hcb * 32;
      reinterpret_cast<uint4*>(dst)[0] = c0;
      reinterpret_cast<uint4*>(dst)[1] = c1;
      *reinterpret_cast<uint32_t*>(p.q_sf + sf_offset(prow, static_cast<int64_t>(hcb) * 4, p.q_cpad4)) = s4;
    }
  } else {
    float m = 0.0f;
    if (rm >= 0) {
#pragma unroll
      for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(h[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(p.amax + e, __float_as_uint(m));
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
constexpr int kThreads = 512;   // four warpgroups
constexpr int kNumEpi = 8;      // epilogue warps (warpgroups 2 and 3)
constexpr int kRegsLow = 64;    // producer / MMA / scale-writer warpgroups
constexpr int kRegsHigh = 192;  // epilogue warpgroups; 2*128*64 + 2*128*192 = 65536

__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow)); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh)); }

// Read COLS accumulator columns of this warp's 32 lanes into registers.
template <int COLS>
__device__ __forceinline__ void drain(uint32_t taddr, uint32_t (&r)[COLS / 32][32]) {
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) tmem_ld_32x32b_x32(taddr + 32 * c, r[c]);
  tmem_ld_wait();
}

template <class Cfg>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const GemmParams p) {
  constexpr int STAGES = Cfg::STAGES;
  constexpr int NUM_ACC = Cfg::NUM_ACC;
  constexpr int BN = Cfg::BN;
  constexpr int MODE = Cfg::MODE;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[STAGES];   // TMA data landed
  __shared__ __align__(8) uint64_t sf_bar[STAGES];     // scales written to TMEM
  __shared__ __align__(8) uint64_t empty_bar[STAGES];  // MMAs of the stage done
  __shared__ __align__(8) uint64_t accf_bar[NUM_ACC];
  __shared__ __align__(8) uint64_t acce_bar[NUM_ACC];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ __align__(8) uint64_t quad_bar[4];  // MoE down: the two epilogue warps of a lane quadrant
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float r_of_s8[MODE == kEpiGatedQuant ? 256 : 1];  // g_out / S for every E4M3 scale byte

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 2);  // the operand and the scale producer
      mbar_init(&sf_bar[s], 4);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], kNumEpi);
    }
    mbar_init(&done_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&quad_bar[i], 2);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // Launched with programmatic serialization: the setup above (barriers, TMEM,
  // descriptor prefetch) touches no global memory and overlaps the preceding
  // kernel; tile counts, tables, operands and outputs are accessed only after
  // this wait.
  pdl_wait();
  pdl_launch_dependents();
  if constexpr (MODE == kEpiGatedQuant) {
    if (threadIdx.x < 256) {
      const float S = e4m3_to_f32(threadIdx.x);
      r_of_s8[threadIdx.x] = (S != 0.0f && S == S) ? __fdiv_rn(__ldg(p.g_out), S) : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;

  // Work units: a 128-row tile times a column tile, column-fastest.
  const int m_tiles = Cfg::GROUPED ? *p.d_m_tiles : p.m_tiles;
  const int total = m_tiles * p.n_tiles;
  const int unit0 = blockIdx.x;
  const int unit_step = gridDim.x;
  const int wg = warp >> 2;

  if (wg == 0) {
    regs_dec();
    if (warp == 0 || warp == 2) {
      // ---------------------------------------------------------- producers
      // Warp 0 copies the operand tiles (TMA boxes), warp 2 the scale atoms
      // (bulk copies); each arrives on the stage's full barrier with its own
      // byte count, so a stage costs each issuing lane two or three copies.
      // The whole warp runs the loop, so every address and coordinate is
      // warp-uniform; lane 0 issues.
      const bool scale_role = warp == 2;
      uint32_t it = 0;  // stages issued so far: stage it % STAGES, round it / STAGES
      bool ok = true;
      for (int tile = unit0; ok && tile < total; tile += unit_step) {
        const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
        const int e = Cfg::GROUPED ? p.tile_expert[mt] : 0;
        int b_row[Cfg::NBLK];
        if (MODE == kEpiDense) {
#pragma unroll
          for (int j = 0; j < Cfg::NBLK; ++j) b_row[j] = nt * BN + 128 * j;
        } else {
          b_row[0] = e * p.b_rows_per_expert + nt * 128;
          if (Cfg::NBLK > 1) b_row[Cfg::NBLK - 1] = b_row[0] + p.up_offset;
        }
        const bool mvalid = mt < m_tiles;
        for (int kb = 0; kb < p.kblocks; ++kb) {
          const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
          if (!mbar_wait_warp(&empty_bar[stage], phase ^ 1, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int ks = min(4, (p.K - kb * 256) / 64);
          uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sB = sA + Cfg::A_BYTES;
          uint8_t* sSFA = sB + Cfg::B_BYTES;
          uint8_t* sSFB = sSFA + Cfg::SFA_BYTES;
          if (lane == 0) {
            if (!scale_role) {
              // A box; B as one BN-row box (dense: consecutive rows) or one
              // 128-row box per block (gate and up blocks of an expert)
              uint32_t bytes = mvalid ? Cfg::A_BYTES : 0;
              if (MODE == kEpiDense) {
                if (b_row[0] < p.b_rows_total) bytes += Cfg::B_BYTES;
              } else {
#pragma unroll
                for (int j = 0; j < Cfg::NBLK; ++j)
                  if (b_row[j] < p.b_rows_total) bytes += 128 * 128;
              }
              mbar_arrive_expect_tx(&full_bar[stage], bytes);
              if (mvalid) tma_load_2d_hint(sA, &tmA, &full_bar[stage], kb * 128, mt * 128, act_policy());
              if (MODE == kEpiDense) {
                if (b_row[0] < p.b_rows_total) tma_load_2d(sB, &tmB, &full_bar[stage], kb * 128, b_row[0]);
              } else {
#pragma unroll
                for (int j = 0; j < Cfg::NBLK; ++j)
                  if (b_row[j] < p.b_rows_total) tma_load_2d(sB + j * 128 * 128, &tmB, &full_bar[stage], kb * 128, b_row[j]);
              }
            } else {
              uint32_t bytes = mvalid ? ks * 512 : 0;
#pragma unroll
              for (int j = 0; j < Cfg::NBLK; ++j)
                if (b_row[j] < p.b_rows_total) bytes += ks * 512;
              mbar_arrive_expect_tx(&full_bar[stage], bytes);
              if (mvalid)
                bulk_load(sSFA, p.sfa + (static_cast<int64_t>(mt) * p.sf_atoms + kb * 4) * 512, ks * 512,
                          &full_bar[stage]);
#pragma unroll
              for (int j = 0; j < Cfg::NBLK; ++j)
                if (b_row[j] < p.b_rows_total)
                  bulk_load(sSFB + j * 2048, p.sfb + (static_cast<int64_t>(b_row[j] >> 7) * p.sf_atoms + kb * 4) * 512,
                            ks * 512, &full_bar[stage]);
            }
          }
          __syncwarp();
          ++it;
        }
      }
      // every copy this warp started lands before the CTA can exit and every
      // release of its stages has arrived: the last issue of each stage is
      // among the last STAGES issues
      int drain_abort = 0;
      for (uint32_t i = it > STAGES ? it - STAGES : 0u; i < it; ++i) {
        mbar_wait_warp(&full_bar[i % STAGES], (i / STAGES) & 1u, reinterpret_cast<volatile int*>(&drain_abort),
                       p.status);
        mbar_wait_warp(&empty_bar[i % STAGES], (i / STAGES) & 1u, reinterpret_cast<volatile int*>(&drain_abort),
                       p.status);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs the loop (descriptors and TMEM addresses are
      // warp-uniform); lane 0 issues every MMA and commit, since a commit
      // tracks the MMAs of the thread that issues it.
      {
        const uint32_t idesc = idesc_nvfp4(128, BN);
        // Descriptors of stage 0; stage s adds s * STAGE_BYTES / 16 to the
        // 14-bit address field (all of shared memory stays below 256 KB).
        const uint32_t sbase = smem_u32(smem);
        const uint64_t da0 = desc_kmajor_sw128(sbase);
        const uint64_t db0 = desc_kmajor_sw128(sbase + Cfg::A_BYTES);
        const uint32_t tsf0 = tmem_base + Cfg::SF_BASE;
        constexpr uint32_t kStageUnits = Cfg::STAGE_BYTES >> 4;
        uint32_t it = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        for (int tile = unit0; ok && tile < total; tile += unit_step) {
          if (!mbar_wait_warp(&acce_bar[acc], acc_phase ^ 1, &abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          // two 256-k stages per pass: the waits, the fence and the loop are
          // paid once per eight MMAs, so the lane keeps the tensor pipe fed
          for (int kb = 0; kb < p.kblocks; kb += 2) {
            const bool two = kb + 1 < p.kblocks;
            const uint32_t st0 = it % STAGES, ph0 = (it / STAGES) & 1u;
            const uint32_t st1 = (it + 1) % STAGES, ph1 = ((it + 1) / STAGES) & 1u;
            if (!mbar_wait_warp(&sf_bar[st0], ph0, &abort_flag, p.status) ||
                (two && !mbar_wait_warp(&sf_bar[st1], ph1, &abort_flag, p.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (h == 1 && !two) break;
                const uint32_t stage = h ? st1 : st0;
                const int ks = min(4, (p.K - (kb + h) * 256) >> 6);
                const uint64_t off = static_cast<uint64_t>(stage * kStageUnits);
                const uint64_t da = da0 + off, db = db0 + off;
                const uint32_t t_sfa = tsf0 + stage * Cfg::SF_COLS;
                const uint32_t t_sfb = t_sfa + 16;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                  if (s < ks)
                    umma_nvfp4(d_tmem, da + 2 * s, db + 2 * s, idesc, t_sfa + 4 * s, t_sfb + (BN / 32) * s,
                               (kb + h > 0 || s > 0) ? 1u : 0u);
                }
                umma_commit(&empty_bar[stage]);
              }
            }
            __syncwarp();
            it += two ? 2u : 1u;
          }
          if (!ok) break;
          if (lane == 0) umma_commit(&accf_bar[acc]);
          __syncwarp();
          if (++acc == NUM_ACC) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
        // wait until every MMA issued above has completed
        if (lane == 0) umma_commit(&done_bar);
        __syncwarp();
        int drain_abort = 0;
        mbar_wait_warp(&done_bar, 0, reinterpret_cast<volatile int*>(&drain_abort), p.status);
      }
    }
  } else if (wg == 1) {
    // ------------------------------------------------------------ scale writers
    // Warp q writes the scale atoms of each landed stage into its own TMEM lane
    // quadrant: atom row `lane` (16 bytes) -> 4 consecutive columns, the same
    // replicated layout a 32x128b.warpx4 copy produces, which the block-scaled
    // MMA reads (column base + row / 32, lane row % 32).
    regs_dec();
    const int q = warp & 3;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < total; tile += unit_step) {
      for (int kb = 0; kb < p.kblocks; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* sSFA = smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES + Cfg::B_BYTES;
        const uint8_t* sSFB = sSFA + Cfg::SFA_BYTES;
        const uint32_t t_sf = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + Cfg::SF_BASE + stage * Cfg::SF_COLS;
        uint32_t va[16];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint4 x = *reinterpret_cast<const uint4*>(sSFA + 512 * s + 16 * lane);
          va[4 * s] = x.x;
          va[4 * s + 1] = x.y;
          va[4 * s + 2] = x.z;
          va[4 * s + 3] = x.w;
        }
        tmem_st_32x32b_x16(t_sf, va);
#pragma unroll
        for (int h = 0; h < Cfg::NBLK; ++h) {  // 16 columns at a time
          uint32_t vb[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // columns 16 h + 4 i of the SFB region: k-step s, 128-row block j
            const int col = 16 * h + 4 * i;
            const int s = col / (BN / 32);
            const int j = (col % (BN / 32)) / 4;
            const uint4 x = *reinterpret_cast<const uint4*>(sSFB + j * 2048 + 512 * s + 16 * lane);
            vb[4 * i] = x.x;
            vb[4 * i + 1] = x.y;
            vb[4 * i + 2] = x.z;
            vb[4 * i + 3] = x.w;
          }
          tmem_st_32x32b_x16(t_sf + 16 + 16 * h, vb);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_bar[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    regs_inc();
    const int ew = warp - 8;
    const int q = warp & 3;      // TMEM lane quadrant of this warp
    const int part = ew >> 2;    // column half of this warp within its quadrant
    uint32_t acc = 0, acc_phase = 0, quad_phase = 0;
    const float alpha_dense = (MODE == kEpiDense) ? __ldg(p.alpha) : 0.0f;
    const float g_out = (MODE == kEpiGatedQuant) ? __ldg(p.g_out) : 0.0f;
    for (int tile = unit0; tile < total; tile += unit_step) {
      const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
      const int row = 32 * q + lane;
      // per-row routing data of a grouped tile, loaded while the MMAs run
      int rm = -1, e = 0;
      float row_scale = 0.0f;
      // kEpiDownDirect: the four rows this thread adds (16x256b layout, below)
      int drm[4] = {-1, -1, -1, -1};
      float dsc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (MODE == kEpiDownDirect) {
        e = p.tile_expert[mt];
        const float ae = __ldg(p.alpha + e);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          drm[i] = p.row_map[mt * 128 + 32 * q + 16 * (i >> 1) + (lane >> 2) + 8 * (i & 1)];
          dsc[i] = drm[i] >= 0 ? __fmul_rn(__ldg(p.topk_w + drm[i]), ae) : 0.0f;
        }
      } else if constexpr (Cfg::GROUPED) {
        rm = p.row_map[mt * 128 + row];
        e = p.tile_expert[mt];
        const float ae = __ldg(p.alpha + e);
        row_scale = (MODE == kEpiDownSum && rm >= 0) ? __fmul_rn(__ldg(p.topk_w + rm), ae) : ae;
      }
      if (!mbar_wait(&accf_bar[acc], acc_phase, &abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN;

      if constexpr (MODE == kEpiDownDirect) {
        // w * alpha_e * acc of this warp's 32 rows x 64 columns, added into
        // the tokens' rows of y straight from registers: with the 16x256b
        // layout four consecutive lanes hold 32 contiguous bytes of one row,
        // so each red.v2 of the warp covers eight whole 32-byte sectors.
        // Half hh holds TMEM lanes 32q + 16hh ..; thread t adds rows
        // 16hh + t/4 (i = 2hh) and 16hh + t/4 + 8 (i = 2hh + 1) of the quadrant.
        static_assert(BN == 128, "64 columns per epilogue warp");
        uint32_t v[2][32];
        tmem_ld_16x256b_x8(t_row + part * 64, v[0]);
        tmem_ld_16x256b_x8(t_row + (16u << 16) + part * 64, v[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
        const int c0 = nt * BN + part * 64 + 2 * (lane & 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (drm[i] >= 0) {
            float* yrow = p.y + static_cast<int64_t>(drm[i] / p.topk) * p.ldy + c0;
            const float sc = dsc[i];
            const uint32_t* vv = v[i >> 1];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v2(yrow + 8 * j, __uint_as_float(vv[4 * j + 2 * (i & 1)]) * sc,
                         __uint_as_float(vv[4 * j + 2 * (i & 1) + 1]) * sc);
          }
        }
      } else if constexpr (MODE == kEpiDense || MODE == kEpiDownSum) {
        // this warp owns COLS accumulator columns: read them all, release the
        // accumulator, then finish from registers
        constexpr int COLS = BN / 2;
        uint32_t r[COLS / 32][32];
        drain<COLS>(t_row + part * COLS, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
        if constexpr (MODE == kEpiDense) {
          const int m = mt * 128 + row;
          if (m < p.M) {
            const int nbase = nt * BN + part * COLS;
            uint16_t* dst = p.out + static_cast<int64_t>(m) * p.ldo + nbase;
#pragma unroll
            for (int c = 0; c < COLS / 32; ++c) store_bf16_32(dst + 32 * c, r[c], alpha_dense, p.N - nbase - 32 * c);
          }
        } else {
          // The two warps of a lane quadrant hold the same 32 rows (one per
          // lane) and split the columns.  Each stages w * alpha_e * acc of its
          // columns into the quadrant's full-width rows; then lanes 0-15 of
          // each warp add one whole row (BN fp32) into its token's row of y
          // with one bulk reduce-add.
          // The two warps meet on the quadrant's mbarrier (bounded waits).
          float* stg_q = reinterpret_cast<float*>(smem + STAGES * Cfg::STAGE_BYTES + q * 32 * Cfg::EPI_PITCH);
          bulk_wait_read_all();  // this lane's reduce of the last tile has read its row ...
          __syncwarp();
          if (lane == 0) mbar_arrive(&quad_bar[q]);
          if (!mbar_wait(&quad_bar[q], quad_phase, &abort_flag, p.status)) break;  // ... and so has the partner's
          quad_phase ^= 1;
          if (rm >= 0) {
            const float scale = row_scale;
            float* stg = stg_q + lane * (Cfg::EPI_PITCH / 4) + part * COLS;
#pragma unroll
            for (int c = 0; c < COLS / 32; ++c)
#pragma unroll
              for (int v = 0; v < 8; ++v)
                reinterpret_cast<float4*>(stg + 32 * c)[v] =
                    make_float4(__uint_as_float(r[c][4 * v]) * scale, __uint_as_float(r[c][4 * v + 1]) * scale,
                                __uint_as_float(r[c][4 * v + 2]) * scale, __uint_as_float(r[c][4 * v + 3]) * scale);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&quad_bar[q]);
          if (!mbar_wait(&quad_bar[q], quad_phase, &abort_flag, p.status)) break;  // both halves are staged
          quad_phase ^= 1;
          const int rr = 16 * part + (lane & 15);
          const int rm_r = __shfl_sync(0xFFFFFFFFu, rm, rr);
          if (lane < 16 && rm_r >= 0)
            bulk_reduce_add_f32(p.y + static_cast<int64_t>(rm_r / p.topk) * p.ldy + nt * BN,
                                stg_q + rr * (Cfg::EPI_PITCH / 4), BN * 4);
        }
      } else {
        // accumulator columns [0, 128) = gate, [128, 256) = up; this warp owns
        // h columns [64 * part, 64 * part + 64)
        uint32_t g0[32], g1[32], u0[32], u1[32];
        tmem_ld_32x32b_x32(t_row + 64 * part, g0);
        tmem_ld_32x32b_x32(t_row + 64 * part + 32, g1);
        tmem_ld_32x32b_x32(t_row + 128 + 64 * part, u0);
        tmem_ld_32x32b_x32(t_row + 128 + 64 * part + 32, u1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
        gated_row64<MODE>(g0, g1, u0, u1, row_scale, rm, e, mt * 128 + row, 2 * nt + part, p, r_of_s8, g_out);
      }
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  if constexpr (MODE == kEpiDownSum) bulk_wait_all();  // this thread's reduce-adds into y are complete
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// dense W4A4 GEMM on CTA pairs
// ---------------------------------------------------------------------------
// A cluster of two CTAs computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 64 per instruction) issued by
// CTA 0.  CTA r holds rows 128r.. of the A tile and rows 128r.. of the B tile in
// its shared memory (the MMA reads the peer's halves at the same offsets), its
// 128 x 256 fp32 accumulator, the scales of its A rows and the scales of all 256
// B rows in its TMEM.  Against one CTA on a 128 x 256 tile this halves the B
// bytes an SM brings in per stage (each SM's TMA ingest is what bounds the
// single-CTA tile), and leaves room to stage the bf16 output tile for TMA stores
// (row-per-lane global stores scatter 16-byte pieces over 32 rows).
//
// Roles per CTA (16 warps):
//   warp 0      A box and this CTA's 128-row B box of each 256-k stage
//   warp 2      scale atoms: this CTA's A rows, all 256 B rows
//   warp 1      TMEM allocation (both CTAs); MMA issue (CTA 0 only)
//   warps 4-7   scale writers: smem -> own TMEM, then arrive on CTA 0's
//               scale-ready barrier (8 arrivals: both CTAs)
//   warps 8-15  epilogue: TMEM -> alpha -> bf16 -> swizzled smem -> TMA store;
//               the accumulator is released to CTA 0 (16 arrivals) as soon as
//               it has been read
// Each CTA's copies complete on its own full barrier; CTA 0's MMA commits are
// multicast to the stage-empty and accumulator-full barriers of both CTAs.
//
// The grouped MoE GEMMs run on the same pairs when every expert's segment is
// padded to 256 rows, so that both 128-row halves of a pair tile belong to one
// expert and share its B tile:
//   gate_up  N = 256 = 128 gate rows (CTA 0's B half) + the 128 matching up
//            rows (CTA 1's), so each CTA's accumulator holds G and U of its
//            rows and runs the gated epilogue of gemm_nvfp4_kernel;
//   down     N = 256 weight rows; each epilogue warp adds its 32 rows x 128
//            columns into y in four 32-column slabs (two staging buffers per
//            warp, one 128-byte bulk reduce-add per row and slab).
template <int MODE>
struct PairCfgT {
  static constexpr bool GROUPED = MODE != kEpiDense;
  static constexpr int STAGES = MODE == kEpiDownSum ? 4 : 5;
  static constexpr int BN = 256;
  static constexpr int A_BYTES = 128 * 128;   // 128 rows x 256 k
  static constexpr int B_BYTES = 128 * 128;   // this CTA's 128 B rows
  static constexpr int SFA_BYTES = 2048;
  static constexpr int SFB_BYTES = 4096;      // scale atoms of all 256 B rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // dense: one box of 32 rows x 64 bf16 at a time; down: two fp32 slabs of
  // 32 rows x 32 columns (row pitch 144 bytes: the row-per-lane stores of a
  // quarter-warp fall on distinct banks)
  static constexpr int DOWN_PITCH = 32 * 4 + 16;
  static constexpr int EPI_WARP_BYTES =
      MODE == kEpiDense ? 32 * 128 : (MODE == kEpiDownSum ? 2 * 32 * DOWN_PITCH : 0);
  static constexpr int EPI_BYTES = kNumEpi * EPI_WARP_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024;
  static constexpr int SF_COLS = 48;          // TMEM scale columns per stage: 16 (A) + 32 (B)
  static constexpr int SF_BASE = BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(STAGE_BYTES % 1024 == 0 && EPI_WARP_BYTES % 128 == 0, "alignment");
  static_assert(SMEM_BYTES <= 232448, "smem budget");
};
using PairCfg = PairCfgT<kEpiDense>;

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  using Cfg = PairCfgT<MODE>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int BN = Cfg::BN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[STAGES];   // this CTA's copies landed
  __shared__ __align__(8) uint64_t sf_bar[STAGES];     // CTA 0: scales of both CTAs in TMEM
  __shared__ __align__(8) uint64_t empty_bar[STAGES];  // the stage's MMAs completed
  __shared__ __align__(8) uint64_t accf_bar;           // the tile's MMAs completed
  __shared__ __align__(8) uint64_t acce_bar;           // CTA 0: both accumulators read
  __shared__ __align__(8) uint64_t done_bar;           // CTA 0: every MMA completed
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float r_of_s8[MODE == kEpiGatedQuant ? 256 : 1];  // g_out / S for every E4M3 scale byte

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 2);  // operand and scale producer
      mbar_init(&sf_bar[s], 8);    // four scale writers in each CTA
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&acce_bar, 2 * kNumEpi);
    mbar_init(&done_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if constexpr (MODE == kEpiDense) prefetch_tmap(&tmOut);  // grouped modes pass no output map
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if constexpr (Cfg::GROUPED) {
    // launched with programmatic serialization: the tile count, the tables
    // and the operands come from the preceding kernels
    pdl_wait();
    pdl_launch_dependents();
    if constexpr (MODE == kEpiGatedQuant) {
      if (threadIdx.x < 256) {
        const float S = e4m3_to_f32(threadIdx.x);
        r_of_s8[threadIdx.x] = (S != 0.0f && S == S) ? __fdiv_rn(__ldg(p.g_out), S) : 0.0f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;

  // work units: 256-row tile pairs x 256-column tiles, column-fastest
  // (grouped: an even number of 128-row tiles, two per expert pair tile)
  const int m_tiles = Cfg::GROUPED ? *p.d_m_tiles : p.m_tiles;
  const int total = ((m_tiles + 1) / 2) * p.n_tiles;
  const int unit0 = blockIdx.x >> 1;
  const int unit_step = gridDim.x >> 1;
  const int wg = warp >> 2;

  if (wg == 0) {
    regs_dec();
    if (warp == 0 || warp == 2) {
      // ---------------------------------------------------------- producers
      // The kernel starts under programmatic dependent launch: everything above
      // (barriers, TMEM, descriptors) overlaps the preceding kernel's tail; the
      // activations and their scales are read only after it has finished.
      pdl_wait();
      const bool scale_role = warp == 2;
      uint32_t it = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < total; tile += unit_step) {
        const int mp = tile / p.n_tiles, nt = tile - mp * p.n_tiles;
        const int mt = 2 * mp + static_cast<int>(rank);
        const bool mvalid = mt < m_tiles;
        // first B row of block j of the pair tile; this CTA copies block `rank`
        int bj[2];
        if constexpr (MODE == kEpiDense) {
          bj[0] = nt * BN;
          bj[1] = nt * BN + 128;
        } else {
          const int e = p.tile_expert[2 * mp];
          const int base = e * p.b_rows_per_expert;
          bj[0] = MODE == kEpiDownSum ? base + nt * BN : base + nt * 128;
          bj[1] = MODE == kEpiDownSum ? base + nt * BN + 128 : base + p.up_offset + nt * 128;
        }
        const int b_row = bj[rank];
        for (int kb = 0; kb < p.kblocks; ++kb) {
          const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
          if (!mbar_wait_warp(&empty_bar[stage], phase ^ 1, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int ks = min(4, (p.K - kb * 256) / 64);
          uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sB = sA + Cfg::A_BYTES;
          uint8_t* sSFA = sB + Cfg::B_BYTES;
          uint8_t* sSFB = sSFA + Cfg::SFA_BYTES;
          if (lane == 0) {
            if (!scale_role) {
              const bool bvalid = b_row < p.b_rows_total;
              mbar_arrive_expect_tx(&full_bar[stage], (mvalid ? Cfg::A_BYTES : 0) + (bvalid ? Cfg::B_BYTES : 0));
              if (mvalid) tma_load_2d_hint(sA, &tmA, &full_bar[stage], kb * 128, mt * 128, act_policy());
              if (bvalid) tma_load_2d(sB, &tmB, &full_bar[stage], kb * 128, b_row);
            } else {
              uint32_t bytes = mvalid ? ks * 512 : 0;
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (bj[j] < p.b_rows_total) bytes += ks * 512;
              mbar_arrive_expect_tx(&full_bar[stage], bytes);
              if (mvalid)
                bulk_load(sSFA, p.sfa + (static_cast<int64_t>(mt) * p.sf_atoms + kb * 4) * 512, ks * 512,
                          &full_bar[stage]);
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (bj[j] < p.b_rows_total)
                  bulk_load(sSFB + j * 2048, p.sfb + (static_cast<int64_t>(bj[j] >> 7) * p.sf_atoms + kb * 4) * 512,
                            ks * 512, &full_bar[stage]);
            }
          }
          __syncwarp();
          ++it;
        }
      }
      int drain_abort = 0;
      for (uint32_t i = it > STAGES ? it - STAGES : 0u; i < it; ++i) {
        mbar_wait_warp(&full_bar[i % STAGES], (i / STAGES) & 1u, reinterpret_cast<volatile int*>(&drain_abort),
                       p.status);
        mbar_wait_warp(&empty_bar[i % STAGES], (i / STAGES) & 1u, reinterpret_cast<volatile int*>(&drain_abort),
                       p.status);
      }
    } else if (warp == 1 && rank == 0 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // One lane, and as little work between MMAs as possible: the tensor pipe
      // queues only a few MMAs, so every cycle the lane spends on waits and
      // bookkeeping beyond that is idle pipe.  Two stages per pass share one
      // wait (the writers complete stages in order, so the second stage's
      // scale-ready phase implies the first's); stage, phase and operand
      // addresses advance incrementally.
      const uint32_t idesc = idesc_nvfp4(256, BN);
      const uint32_t sbase = smem_u32(smem);
      const uint64_t da0 = desc_kmajor_sw128(sbase);
      const uint64_t db0 = desc_kmajor_sw128(sbase + Cfg::A_BYTES);
      const uint32_t tsf0 = tmem_base + Cfg::SF_BASE;
      constexpr uint32_t kStageUnits = Cfg::STAGE_BYTES >> 4;
      const bool kfull = (p.K & 255) == 0;
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      uint64_t da = da0, db = db0;
      uint32_t t_sfa = tsf0;
      auto advance = [&]() {
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
          da = da0;
          db = db0;
          t_sfa = tsf0;
        } else {
          da += kStageUnits;
          db += kStageUnits;
          t_sfa += Cfg::SF_COLS;
        }
      };
      auto issue_stage = [&](int kb) {
        const uint32_t t_sfb = t_sfa + 16;
        if (kfull || (p.K - kb * 256) >= 256) {
          umma_nvfp4_pair(tmem_base, da, db, idesc, t_sfa, t_sfb, kb > 0 ? 1u : 0u);
#pragma unroll
          for (int s = 1; s < 4; ++s)
            umma_nvfp4_pair(tmem_base, da + 2 * s, db + 2 * s, idesc, t_sfa + 4 * s, t_sfb + (BN / 32) * s, 1u);
        } else {
          const int ks = (p.K - kb * 256) >> 6;
#pragma unroll
          for (int s = 0; s < 4; ++s)
            if (s < ks)
              umma_nvfp4_pair(tmem_base, da + 2 * s, db + 2 * s, idesc, t_sfa + 4 * s, t_sfb + (BN / 32) * s,
                              (kb > 0 || s > 0) ? 1u : 0u);
        }
        umma_commit_pair(&empty_bar[stage], 0x3);
      };
      bool ok = true;
      for (int tile = unit0; ok && tile < total; tile += unit_step) {
        if (!mbar_wait(&acce_bar, acc_phase ^ 1, &abort_flag, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < p.kblocks; kb += 2) {
          const bool two = kb + 1 < p.kblocks;
          const uint32_t wst = two ? (stage + 1 == STAGES ? 0u : stage + 1) : stage;
          const uint32_t wph = (two && stage + 1 == STAGES) ? phase ^ 1 : phase;
          if (!mbar_wait(&sf_bar[wst], wph, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_stage(kb);
          advance();
          if (two) {
            issue_stage(kb + 1);
            advance();
          }
        }
        if (!ok) break;
        umma_commit_pair(&accf_bar, 0x3);
        acc_phase ^= 1;
      }
      // wait until every MMA issued above has completed
      umma_commit_pair(&done_bar, 0x1);
      int drain_abort = 0;
      mbar_wait(&done_bar, 0, reinterpret_cast<volatile int*>(&drain_abort), p.status);
    }
  } else if (wg == 1) {
    // ------------------------------------------------------------ scale writers
    // as in gemm_nvfp4_kernel: warp q writes its TMEM lane quadrant; then one
    // arrival per warp on CTA 0's scale-ready barrier of the stage
    regs_dec();
    const int q = warp & 3;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < total; tile += unit_step) {
      for (int kb = 0; kb < p.kblocks; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* sSFA = smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES + Cfg::B_BYTES;
        const uint8_t* sSFB = sSFA + Cfg::SFA_BYTES;
        const uint32_t t_sf = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + Cfg::SF_BASE + stage * Cfg::SF_COLS;
        uint32_t va[16];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint4 x = *reinterpret_cast<const uint4*>(sSFA + 512 * s + 16 * lane);
          va[4 * s] = x.x;
          va[4 * s + 1] = x.y;
          va[4 * s + 2] = x.z;
          va[4 * s + 3] = x.w;
        }
        tmem_st_32x32b_x16(t_sf, va);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t vb[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = 16 * h + 4 * i;
            const int s = col / (BN / 32);
            const int j = (col % (BN / 32)) / 4;
            const uint4 x = *reinterpret_cast<const uint4*>(sSFB + j * 2048 + 512 * s + 16 * lane);
            vb[4 * i] = x.x;
            vb[4 * i + 1] = x.y;
            vb[4 * i + 2] = x.z;
            vb[4 * i + 3] = x.w;
          }
          tmem_st_32x32b_x16(t_sf + 16 + 16 * h, vb);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(&sf_bar[stage], 0));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    regs_inc();
    const int ew = warp - 8;
    const int q = warp & 3;      // TMEM lane quadrant: output rows 32q ..
    const int part = ew >> 2;    // column half: 128 part ..
    uint8_t* stg = smem + STAGES * Cfg::STAGE_BYTES + ew * Cfg::EPI_WARP_BYTES;
    const uint32_t acce_lead = mapa_shared(&acce_bar, 0);
    pdl_wait();  // alpha (and the output buffer) may belong to the preceding kernel
    const float alpha = MODE == kEpiDense ? __ldg(p.alpha) : 0.0f;
    const float g_out = MODE == kEpiGatedQuant ? __ldg(p.g_out) : 0.0f;
    uint32_t acc_phase = 0;
    for (int tile = unit0; tile < total; tile += unit_step) {
      const int mp = tile / p.n_tiles, nt = tile - mp * p.n_tiles;
      const int mt = 2 * mp + static_cast<int>(rank);
      const int row = 32 * q + lane;
      // routing data of a grouped tile, loaded while the MMAs run
      int rm = -1, e = 0;
      float row_scale = 0.0f;
      if constexpr (Cfg::GROUPED) {
        rm = p.row_map[mt * 128 + row];
        e = p.tile_expert[mt];
        const float ae = __ldg(p.alpha + e);
        row_scale = (MODE == kEpiDownSum && rm >= 0) ? __fmul_rn(__ldg(p.topk_w + rm), ae) : ae;
      }
      if (!mbar_wait(&accf_bar, acc_phase, &abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
      if constexpr (MODE == kEpiDense) {
        constexpr int COLS = BN / 2;
        uint32_t r[COLS / 32][32];
        drain<COLS>(t_row + part * COLS, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_lead);
        acc_phase ^= 1;
        if (mt >= m_tiles) continue;  // rows past M (the second half of the last pair)
        // row `lane` of a 32 x 64 box, 128-byte rows with the 128-byte swizzle
        // (16-byte chunk j of row r at chunk j ^ (r % 8)); two boxes per tile
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          // this warp's previous box has been read out of the staging buffer
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          uint8_t* srow = stg + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t* v = r[2 * g + j / 4] + 8 * (j % 4);
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[0]) * alpha, __uint_as_float(v[1]) * alpha);
            o.y = pack_bf16x2(__uint_as_float(v[2]) * alpha, __uint_as_float(v[3]) * alpha);
            o.z = pack_bf16x2(__uint_as_float(v[4]) * alpha, __uint_as_float(v[5]) * alpha);
            o.w = pack_bf16x2(__uint_as_float(v[6]) * alpha, __uint_as_float(v[7]) * alpha);
            *reinterpret_cast<uint4*>(srow + ((j ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x = nt * BN + part * COLS + 64 * g, y = mt * 128 + 32 * q;
            if (x < p.N && y < p.M) tma_store_2d(&tmOut, stg, x, y);
          }
          __syncwarp();
        }
      } else if constexpr (MODE == kEpiDownSum) {
        // w * alpha_e * acc of this row, columns 128 part .. 128 part + 127, in
        // four 32-column slabs; slab j stages in buffer j % 2, reused once the
        // reduce-add two slabs back has read it
        uint32_t r[4][32];
        drain<128>(t_row + part * 128, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_lead);
        acc_phase ^= 1;
        float* ydst = p.y + static_cast<int64_t>(rm >= 0 ? rm / p.topk : 0) * p.ldy + nt * BN + part * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bulk_wait_read_1();
          float* srow = reinterpret_cast<float*>(stg + (j & 1) * 32 * Cfg::DOWN_PITCH + lane * Cfg::DOWN_PITCH);
          if (rm >= 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(srow)[v] =
                  make_float4(__uint_as_float(r[j][4 * v]) * row_scale, __uint_as_float(r[j][4 * v + 1]) * row_scale,
                              __uint_as_float(r[j][4 * v + 2]) * row_scale,
                              __uint_as_float(r[j][4 * v + 3]) * row_scale);
            fence_proxy_async_smem();
            bulk_reduce_add_f32(ydst + 32 * j, srow, 32 * 4);
          }
        }
      } else {
        // accumulator columns [0, 128) = gate, [128, 256) = up; this warp owns
        // h columns [64 * part, 64 * part + 64) of the tile
        uint32_t g0[32], g1[32], u0[32], u1[32];
        tmem_ld_32x32b_x32(t_row + 64 * part, g0);
        tmem_ld_32x32b_x32(t_row + 64 * part + 32, g1);
        tmem_ld_32x32b_x32(t_row + 128 + 64 * part, u0);
        tmem_ld_32x32b_x32(t_row + 128 + 64 * part + 32, u1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acce_lead);
        acc_phase ^= 1;
        gated_row64<MODE>(g0, g1, u0, u1, row_scale, rm, e, mt * 128 + row, 2 * nt + part, p, r_of_s8, g_out);
      }
    }
    // this warp's stores (dense: lane 0) and reduce-adds (down: every lane) are complete
    if (MODE == kEpiDownSum || lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no MMA, copy or arrival of the pair touches this CTA after this point
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using GatedCfg = GemmCfg<256, 1, 4, kEpiGatedQuant>;
using AmaxCfg = GemmCfg<256, 1, 4, kEpiGatedAmax>;
using DownCfg = GemmCfg<128, 2, 4, kEpiDownSum>;
using DownDirectCfg = GemmCfg<128, 2, 6, kEpiDownDirect>;  // 6 x 36 KB stages, no staging
using DenseSmallCfg = GemmCfg<128, 2, 6, kEpiDense>;  // 6 x 36 KB stages, 2 x 128 + 6 x 32 TMEM columns

template <class Cfg>
static cudaError_t launch_cfg(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t stream) {
  // set on every launch: the attribute belongs to the current device, and a
  // process may launch on several
  cudaError_t e = cudaFuncSetAttribute(gemm_nvfp4_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_nvfp4_kernel<Cfg>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), Cfg::SMEM_BYTES,
                    stream, maps.a, maps.b, p);
}

template <int MODE>
static cudaError_t launch_pair(const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t stream) {
  using Cfg = PairCfgT<MODE>;
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;  // whole CTA pairs
  return launch_pdl(gemm_pair_kernel<MODE>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), Cfg::SMEM_BYTES,
                    stream, maps.a, maps.b, maps.out, p);
}

cudaError_t launch_gemm(int mode, const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t stream) {
  switch (mode) {
    case kEpiDense: return launch_pair<kEpiDense>(maps, p, grid, stream);
    case kEpiGatedQuant: return launch_cfg<GatedCfg>(maps, p, grid, stream);
    case kEpiGatedAmax: return launch_cfg<AmaxCfg>(maps, p, grid, stream);
    case kEpiDownSum: return launch_cfg<DownCfg>(maps, p, grid, stream);
    case kEpiDownDirect: return launch_cfg<DownDirectCfg>(maps, p, grid, stream);
    case kLaunchDenseSmall: return launch_cfg<DenseSmallCfg>(maps, p, grid, stream);
    case kLaunchPairGated: return launch_pair<kEpiGatedQuant>(maps, p, grid, stream);
    case kLaunchPairDown: return launch_pair<kEpiDownSum>(maps, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4
