// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
// Every launcher enqueues on `stream` and returns cudaGetLastError().
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace nvfp4 {

// ---- quantisation (quant.cu) ----------------------------------------------
cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, int64_t ldx, const float* d_global,
                             uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t stream);
cudaError_t launch_compute_global(const void* x, int64_t rows, int64_t cols, int64_t ldx, float* d_global,
                                  cudaStream_t stream, int num_sms);
cudaError_t launch_make_alpha(const float* d_g_a, const float* d_g_w, int64_t n, float* d_alpha,
                              cudaStream_t stream);
cudaError_t launch_reduce_max(const float* d_in, int64_t n, float* d_out, cudaStream_t stream);

// ---- block-scaled tcgen05 GEMM (gemm_w4a4.cu) ------------------------------
enum EpiMode : int {
  kEpiDense = 0,
  kEpiGatedQuant = 1,
  kEpiGatedAmax = 2,
  kEpiDownSum = 3,     // MoE down: rows staged in shared memory, 512-byte bulk reduce-adds into y
  kEpiDownDirect = 7,  // MoE down for few routes per expert: vector reductions straight from TMEM reads
};
// Launch mode of the dense W4A4 linear for small M: the single-CTA kernel on
// 128 x 128 tiles (twice the CTAs of the pair kernel's 256 x 256 tiles, a
// deeper stage ring), dense epilogue.
constexpr int kLaunchDenseSmall = 4;
// MoE gate_up / down on CTA pairs (expert segments padded to 256 rows)
constexpr int kLaunchPairGated = 5;
constexpr int kLaunchPairDown = 6;

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream is still running, and every such kernel
// executes pdl_wait (griddepcontrol.wait) before it reads or writes memory the
// predecessors use.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct GemmParams {
  const uint8_t* sfa;      // swizzled scales of A (over all A rows)
  const uint8_t* sfb;      // swizzled scales of B (over all B rows)
  int K;                   // reduction length (multiple of 64)
  int kblocks;             // ceil(K / 256)
  int sf_atoms;            // K / 64: 512-byte scale atoms per 128-row block
  int n_tiles;             // output column tiles
  int m_tiles;             // dense: ceil(M / 128)
  const int* d_m_tiles;    // grouped: device count of 128-row tiles
  const int* tile_expert;  // grouped: expert of each 128-row tile
  const int* row_map;      // grouped: route id of each permuted row, -1 = padding
  int b_rows_per_expert;   // grouped: B rows per expert (2I or H)
  int up_offset;           // gated: row offset of the up half (I)
  int b_rows_total;        // rows of B
  const float* alpha;      // dense: [1]; grouped: [E]
  // dense output
  uint16_t* out;
  int64_t ldo;
  int M;
  int N;
  // gated output (NVFP4 of SiLU(gate) * up)
  const float* g_out;
  uint8_t* q_codes;
  uint8_t* q_sf;
  int64_t q_row_bytes;     // I / 2
  int64_t q_cpad4;         // padded scale columns / 4 of the intermediate
  unsigned int* amax;      // calibration: per-expert amax bits
  // routed down output
  float* y;
  int64_t ldy;
  const float* topk_w;
  int topk;
  int* status;
};

struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b;
  CUtensorMap out;  // dense mode: the bf16 output (boxes of 32 rows x 64 columns, 128-byte swizzle)
};

// Build a 2D TMA map over a [rows, row_bytes] byte matrix, box box_rows x 128
// bytes, 128-byte swizzle.
bool make_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows = 128);

// Build the TMA map of a [rows, cols] bf16 output with a row pitch of ld
// elements: boxes of 32 rows x 64 columns, 128-byte swizzle (TMA stores).
bool make_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld);

// B boxes are 128 rows in every mode.  The dense mode runs on CTA pairs (the
// grid counts CTAs and must be even: one pair per 256 x 256 output tile).
cudaError_t launch_gemm(int mode, const GemmMaps& maps, const GemmParams& p, int grid, cudaStream_t stream);

}  // namespace nvfp4
