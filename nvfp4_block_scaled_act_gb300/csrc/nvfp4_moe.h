// MoE workspace carving and launchers (moe.cu), shared with api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace nvfp4 {

struct MoEWorkspace {
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E + 1]
  int32_t* n_tiles;      // [1]
  int32_t* row_map;      // [P_max]
  int32_t* tile_expert;  // [P_max / 128]
  int32_t* pos;          // [T * topk]
  int32_t* hist;         // [nchunks * E]
  int32_t* ids;          // [T * topk] (calibration routes)
  uint8_t* a1_codes;     // [P_max, H/2]
  uint8_t* a1_sf;        // swizzled over P_max rows, H/16 columns
  uint8_t* h_codes;      // [P_max, I/2]
  uint8_t* h_sf;         // swizzled over P_max rows, I/16 columns
  float* y;              // [T, H]
  unsigned int* amax;    // [E] (calibration)
  int64_t p_max;
  int bm;  // row block the segments are padded to (256: the grouped GEMMs run on CTA pairs)
};

struct MoELayoutBytes {
  size_t counts, offsets, n_tiles, row_map, tile_expert, pos, hist, ids, a1_codes, a1_sf, h_codes, h_sf, y, amax,
      total;
  int64_t p_max;
  int bm;  // row block of the alignment for nvfp4_moe_w4a4 (moe_row_block)
};

// Row block the W4A4 MoE pads every expert segment to: 256 (the grouped GEMMs
// then run on CTA pairs, 256-row tiles of one expert) once the experts average
// at least kPairRoutesPerExpert routes and the hidden size splits into
// 256-column down tiles; else 128 (one CTA per 128-row tile).  Per padded row
// the pairs are about 15 % faster, but 256-row padding adds about 64 rows per
// expert on average: at 256 routes per expert that is 20 % more rows and the
// pairs lose, at 1024 it is about 6 % and they win.
constexpr int64_t kPairRoutesPerExpert = 1024;
inline int moe_row_block(int64_t T, int64_t H, int64_t E, int64_t topk) {
  return (T * topk >= kPairRoutesPerExpert * E && H % 256 == 0) ? 256 : 128;
}

// Routes per histogram / scatter chunk of the multi-block align: 256, doubled
// until there are at most 512 chunks, so the scatter has a warp per 256-512
// routes and the scan's per-expert column stays short.  The workspace sizes the
// chunk histogram with the same rule.
inline int64_t moe_align_chunk(int64_t R) {
  int64_t c = 256;
  while ((R + c - 1) / c > 512) c *= 2;
  return c;
}

MoELayoutBytes moe_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
MoEWorkspace moe_carve(void* base, const MoELayoutBytes& L);

// bm: 128 or 256, the row block every expert segment is padded to
cudaError_t launch_moe_align(const int32_t* ids, int64_t T, int topk, int E, int bm, const MoEWorkspace& w,
                             int* status, cudaStream_t stream);
cudaError_t launch_moe_quant_permute(const void* x, int64_t T, int64_t H, int topk, const float* d_g,
                                     const MoEWorkspace& w, int num_sms, cudaStream_t stream);
cudaError_t launch_moe_finalize(const float* y, int64_t n, void* out, int num_sms, cudaStream_t stream);
cudaError_t launch_moe_dense_ids(int32_t* ids, int64_t Tc, int E, cudaStream_t stream);
cudaError_t launch_moe_calib_finish(unsigned int* amax_bits, int E, float* g_max, cudaStream_t stream);

// ---- W4A16 decode (gemv_w4a16.cu) -------------------------------------------
// W4A16 MoE for small batches (moe_w4a16.cu).  Workspace (device) fields are
// carved by the API from the caller's workspace.
struct MoeW16Params {
  const uint16_t* x;  // [T, H] bf16, contiguous
  int T, H, I, E, topk;
  const int32_t* ids;     // [T * topk]
  const float* topk_w;    // [T * topk]
  const uint8_t* w13_sf;  // codes are read through the tensor maps
  const float* alpha13;   // [E]
  const uint8_t* w2_sf;
  const float* alpha2;    // [E]
  uint16_t* out;          // [T, H] bf16
  uint16_t* h;            // [R, I]  bf16 silu(a13 G) * (a13 U) of every route
  float* dn;              // [R, H]  w * a2 * (h @ W2[e].T) of every route
  int* status;
};

// Launch shape of one grouped GEMV stage.  Work items are (slot, row block);
// `ctas` persistent CTAs take items round-robin and stream their weights
// through a ring of R 128-k blocks; activations are staged in windows of
// `win` k elements, 16 route rows at a time if tok16, else 8.
struct Moe16Plan {
  int win, R, ctas;
  bool tok16;
  size_t smem;  // dynamic shared memory per CTA
  bool ok;
};
Moe16Plan moe16_plan(int mode, int64_t K, int64_t T, int64_t E, int topk, int64_t units, int num_sms);
// w13_map: the stacked gate/up codes [E*2I, H/2] as boxes of 64 bytes x 64
// rows; w2_map: the down codes [E*H, I/2] as boxes of 64 bytes x 128 rows.
cudaError_t launch_moe_w4a16(const CUtensorMap& w13_map, const CUtensorMap& w2_map, const MoeW16Params& p,
                             int num_sms, cudaStream_t stream);

struct GemvPlan {
  int splits;      // k-splits (1 = no workspace)
  int kc;          // k elements per split (multiple of 128)
  int row_blocks;  // ceil(N / 128)
  size_t ws_bytes;
};
GemvPlan gemv_plan(int64_t T, int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemv_w4a16(const void* x, int64_t T, int64_t ldx, const uint8_t* w_codes, const uint8_t* w_sf,
                              int64_t N, int64_t K, const float* d_alpha, void* out, int64_t ldo, float* ws,
                              const GemvPlan& plan, cudaStream_t stream);

// Default decode path: weight ring in shared memory, split-K inside a
// thread-block cluster, programmatic dependent launch; no workspace.
struct GemvRingPlan {
  int cl;              // CTAs per cluster (k-splits of a row block)
  int kc;              // k elements per CTA
  int R;               // ring slots (128-k blocks resident at once)
  int64_t row_blocks;  // ceil(N / 128)
  size_t smem;         // dynamic shared memory per CTA
  bool ok;             // false: the activations of a CTA do not fit; use the split-K path
};
GemvRingPlan gemv_ring_plan(int64_t T, int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemv_w4a16_ring(const CUtensorMap& cmap, const void* x, int64_t T, int64_t ldx,
                                   const uint8_t* w_sf, int64_t N, int64_t K, const float* d_alpha, void* out,
                                   int64_t ldo, const GemvRingPlan& plan, int* status, cudaStream_t stream);

}  // namespace nvfp4
