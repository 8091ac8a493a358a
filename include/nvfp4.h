/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 weight-GEMM library.
 *
 * Formats (the pages "run nvfp4 linears on nvfp4 activations on sm_120",
 * section "Changes", and "Add BF16_FP4 GEMM ... for W4A16 workloads",
 * sections "Summary" and "API"):
 *   codes   e2m1 values, two per byte, row-major [rows, K/2]; element 2j in the
 *           low nibble, 2j+1 in the high nibble; low 3 bits magnitude, bit 3
 *           sign.
 *   scales  one FP8-E4M3 (unsigned use) scale per 16 consecutive k-elements,
 *           stored in the 128x4-swizzled layout: the rows x C scale matrix
 *           (C = K/16) is cut into 128-row x 4-column atoms of 512 bytes,
 *           ordered row-block major, and inside an atom row r, column c sits
 *           at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.  The buffer
 *           holds nvfp4_scale_bytes(rows, K) bytes; padding bytes are zero.
 *   global  one fp32 per tensor, g = 448 * 6 / amax (quantisation direction).
 *   alpha   fp32 dequantisation factor applied to the fp32 accumulator:
 *           1 / (g_a * g_w) for W4A4, 1 / g_w for W4A16.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers unless the name says host; the caller
 *     owns every buffer.  The library allocates no device memory; calls that
 *     need scratch take a caller-sized workspace.
 *   - Scalars that depend on data (globals, alphas) are device pointers, so a
 *     sequence of calls can be captured in a CUDA graph.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and is asynchronous: no call synchronises the host except
 *     nvfp4_device_status.
 *   - Argument errors are returned before anything is launched.  M, T or rows
 *     equal to 0 return NVFP4_OK and launch nothing.  A failed launch returns
 *     NVFP4_ERR_CUDA.  Errors found on the device (a pipeline wait that timed
 *     out, an expert id out of range) set a device status word that
 *     nvfp4_device_status reads.
 *   - Alignment: every codes, scales, bf16 and workspace pointer must be
 *     16-byte aligned (TMA and 16-byte vector loads), else
 *     NVFP4_ERR_MISALIGNED.
 *   - The library runs on the current CUDA device, which must be an sm_103
 *     GPU (GB300); otherwise NVFP4_ERR_NO_DEVICE.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4_stream_t; /* same type as cudaStream_t */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad stride   */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2,   /* N % 8, K % 64, topk, sizes past the limits */
  NVFP4_ERR_MISALIGNED = 3,          /* a pointer or leading dimension is misaligned */
  NVFP4_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the *_workspace() figure   */
  NVFP4_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed      */
  NVFP4_ERR_DEVICE_TIMEOUT = 6,      /* device word: a pipeline wait gave up      */
  NVFP4_ERR_BAD_EXPERT_ID = 7,       /* device word: a route named an expert outside [0, E) */
  NVFP4_ERR_NO_DEVICE = 8            /* no current CUDA device of compute capability 10.3 */
} nvfp4_status;

/* Text of a status code (static storage). */
const char* nvfp4_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int nvfp4_version(void);

/* Bytes of the swizzled scale buffer of a [rows, k] NVFP4 tensor:
 * ceil(rows / 128) * 128 * ceil((k / 16) / 4) * 4. */
size_t nvfp4_scale_bytes(int64_t rows, int64_t k);

/* Per-tensor global of a bf16 [rows, cols] tensor (row stride ldx elements):
 * *d_global = 2688 / amax(|x|) in fp32, or 1 for an all-zero tensor.
 * ("Add BF16_FP4 GEMM ...", section API: g_w = (448 * 6) / amax(w); also the
 * static activation global of "run nvfp4 linears ...", taken from a
 * calibration batch.)  d_global: one fp32 on the device, overwritten. */
nvfp4_status nvfp4_compute_global(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                                  float* d_global, nvfp4_stream_t stream);

/* Dequantisation factors: d_alpha[i] = 1 / (g_a * d_g_w[i]) for i < n, all
 * fp32, where g_a = *d_g_a, or g_a = 1 when d_g_a is NULL (W4A16: alpha =
 * 1 / g_w, "Add BF16_FP4 GEMM ...", section API). */
nvfp4_status nvfp4_make_alpha(const float* d_g_a, const float* d_g_w, int64_t n, float* d_alpha,
                              nvfp4_stream_t stream);

/* *d_out = max over i < n of d_in[i] (fp32).  Used for the fused-weight global
 * (a fused weight takes the largest of its parts' globals: "run nvfp4 linears
 * ...", Changes) and the MoE input globals (the largest per-expert input
 * global feeds each GEMM: the W4A4 MoE prefill page, Changes). */
nvfp4_status nvfp4_reduce_max(const float* d_in, int64_t n, float* d_out, nvfp4_stream_t stream);

/* NVFP4 quantisation of bf16 activations (or weights) with a static global
 * ("run nvfp4 linears ...", Changes: the activation quantiser, which cuts long
 * rows into chunks and writes 128x4-swizzled scales).  Per 16-element block of a row:
 * amax -> s = E4M3_satfinite((amax / 6) * g) -> codes = e2m1_satfinite(x * (g / s)),
 * all codes +0 when s == 0.
 *   x_bf16  [M, K] bf16, row stride ldx >= K elements, ldx % 8 == 0
 *   K       multiple of 16
 *   d_global one fp32 (g), 0 < g <= 6.6e35 so that g / s stays finite for
 *           every E4M3 scale s (the smallest is 2^-9)
 *   codes   [M, K/2] bytes, written
 *   scales  nvfp4_scale_bytes(M, K) bytes, written in full (padding zeroed)
 * Codes and scales are bit-identical to the reference rule for any finite input. */
nvfp4_status nvfp4_quantize_act(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                const float* d_global, uint8_t* codes, uint8_t* scales,
                                nvfp4_stream_t stream);

/* W4A4 block-scaled GEMM ("run nvfp4 linears ...", Changes: W4A4 GEMM on NVFP4
 * activations with one weight global per tensor; the W4A16 form
 * out = (a @ dequant(b, b_sf).T) * alpha of "Add BF16_FP4 GEMM ...", Summary,
 * with a dequantised too):
 *   out[m, n] = bf16( alpha * sum_k e2m1(a[m,k]) s_a[m,k/16] * e2m1(w[n,k]) s_w[n,k/16] )
 *   a_codes [M, K/2], a_sf swizzled over M rows (from nvfp4_quantize_act)
 *   w_codes [N, K/2], w_sf swizzled over N rows (row-major weight, no repack)
 *   d_alpha one fp32 = 1 / (g_a * g_w)
 *   out     bf16 [M, N] with row stride ldo >= N, ldo % 8 == 0
 * Requires N % 8 == 0 (N = 12 is refused, as the pages' b12x route does) and
 * K % 64 == 0.  fp32 accumulation on the tcgen05 tensor cores. */
nvfp4_status nvfp4_linear_w4a4(const uint8_t* a_codes, const uint8_t* a_sf, int64_t M,
                               const uint8_t* w_codes, const uint8_t* w_sf, int64_t N, int64_t K,
                               const float* d_alpha, void* out_bf16, int64_t ldo,
                               nvfp4_stream_t stream);

/* Workspace bytes of nvfp4_linear_w4a16 for this shape (0 when no split-K
 * partials are needed). */
size_t nvfp4_linear_w4a16_workspace(int64_t T, int64_t N, int64_t K);

/* W4A16 decode GEMM ("Add BF16_FP4 GEMM ...", Summary: out = (a @ dequant(b,
 * b_sf).T) * alpha with a bf16; "run nvfp4 linears ...", Changes: W4A16
 * kernels for small batches on the same row-major weight, no repack):
 *   out[t, n] = bf16( alpha * sum_k a[t,k] * e2m1(w[n,k]) s_w[n,k/16] ), fp32 accumulation
 *   x_bf16  [T, K] bf16, row stride ldx >= K, ldx % 8 == 0; 1 <= T <= 16
 *   w_codes/w_sf as for nvfp4_linear_w4a4; N % 8 == 0, K % 128 == 0
 *   d_alpha one fp32 = 1 / g_w
 *   out     bf16 [T, N], row stride ldo >= N
 *   workspace of nvfp4_linear_w4a16_workspace(T, N, K) bytes (may be NULL when
 *   that is 0).  The k-split partial sums of a 128-row block are summed on
 *   chip, inside a thread-block cluster, so the query returns 0, unless the
 *   activations of one k-split do not fit in shared memory next to the weight
 *   (long K at large T: on 152 SMs from K = 44160 at T = 16 and from
 *   K = 91264 at T = 8, whatever N); those shapes keep fp32
 *   partials in the workspace and sum them with a second kernel.  Either way
 *   the partials are summed in a fixed order, so the result is the same from
 *   run to run.
 * The call is launched as a programmatic dependent launch: it starts copying
 * its weight into shared memory while the preceding kernel on the stream
 * finishes, if that kernel allows it (this library's decode kernel does, and
 * writes no weight); it reads x and alpha and writes out only after the
 * preceding kernel has completed.  Back-to-back decode calls (a layer stack in
 * a CUDA graph) overlap this way. */
nvfp4_status nvfp4_linear_w4a16(const void* x_bf16, int64_t T, int64_t ldx,
                                const uint8_t* w_codes, const uint8_t* w_sf, int64_t N, int64_t K,
                                const float* d_alpha, void* out_bf16, int64_t ldo,
                                void* workspace, size_t ws_bytes, nvfp4_stream_t stream);

/* The same W4A16 decode GEMM for callers that cannot allocate device memory
 * (a runtime that owns the whole GPU through its own pool, code already inside
 * CUDA stream capture, a plugin host that hands out only inputs and outputs).
 * The pages have no counterpart of this call; it is an addition of this
 * library.  Instead of a caller-sized workspace it keeps the split-K partial
 * sums in one 6 MiB array compiled into the library, which every GPU that
 * loads the library holds until the process exits.  It allocates nothing.
 *   - Arguments, layouts and results are those of nvfp4_linear_w4a16.
 *   - Shapes whose partials need more than 6 MiB (split-K partials of
 *     splits * T * N fp32; e.g. T = 16, N = 25600, K = 4096) are refused with
 *     NVFP4_ERR_WORKSPACE_TOO_SMALL; both decode shapes of the workloads fit.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: a cudaDeviceReset
 *     after that first call is not supported.
 *   - Every call shares the one array and it keeps the last call's partials;
 *     nothing in it needs to start at zero (each partial is written before it
 *     is read).  Calls that overlap on the GPU (other streams, other threads)
 *     race on the array: serialise them. */
nvfp4_status nvfp4_linear_w4a16_noalloc(const void* x_bf16, int64_t T, int64_t ldx,
                                        const uint8_t* w_codes, const uint8_t* w_sf, int64_t N,
                                        int64_t K, const float* d_alpha, void* out_bf16,
                                        int64_t ldo, nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Mixture of experts, W4A4 (the W4A4 MoE prefill page, Changes; layer flow
 * align -> gate_up -> act -> down -> sum of "speed up the nvfp4 moe prefill
 * gemm on rtx gpus", Changes).
 *
 * Weights (one NVFP4 tensor per expert, experts concatenated, no repack):
 *   w13_codes [E, 2I, H/2], w13_sf = E consecutive nvfp4_scale_bytes(2I, H)
 *             blocks; rows [0, I) of an expert are gate, rows [I, 2I) are up.
 *   w2_codes  [E, H, I/2],  w2_sf = E consecutive nvfp4_scale_bytes(H, I) blocks.
 *   d_alpha13[e] = 1 / (g_a1 * g_w13[e]), d_alpha2[e] = 1 / (g_a2 * g_w2[e]).
 *   d_g_a1, d_g_a2: the static input globals of the two GEMMs (one fp32 each).
 * Routes: topk_ids int32 [T, topk], topk_w fp32 [T, topk].  Ids outside [0, E)
 * set NVFP4_ERR_BAD_EXPERT_ID in the device word and the route is dropped.
 * Shapes: H % 128 == 0, I % 128 == 0, 1 <= topk <= 32 (nvfp4_moe_calibrate
 * routes every row to every expert, so there topk = E <= 1024).
 * Result: out bf16 [T, H] = sum over routes of w * alpha2[e] * (h_q @ W2[e].T),
 * h = silu(alpha13[e] * G) * (alpha13[e] * U) re-quantised to NVFP4 with g_a2;
 * the top-k sum is accumulated in fp32 and rounded to bf16 once.
 * --------------------------------------------------------------------------- */

/* Workspace bytes of nvfp4_moe_w4a4 (and of its stages) for T tokens. */
size_t nvfp4_moe_workspace(int64_t T, int64_t H, int64_t I, int64_t E, int topk);

/* The whole layer: align -> quantise and permute x -> gate_up (SiLU * up, NVFP4
 * re-quantisation in the epilogue) -> down (routing weight, fp32 top-k sum)
 * -> bf16.  No host synchronisation: tile counts stay on the device. */
nvfp4_status nvfp4_moe_w4a4(const void* x_bf16, int64_t T, int64_t H, int64_t I, int64_t E,
                            int topk, const int32_t* topk_ids, const float* topk_w,
                            const float* d_g_a1, const uint8_t* w13_codes, const uint8_t* w13_sf,
                            const float* d_alpha13, const float* d_g_a2,
                            const uint8_t* w2_codes, const uint8_t* w2_sf, const float* d_alpha2,
                            void* out_bf16, void* workspace, size_t ws_bytes,
                            nvfp4_stream_t stream);

/* Calibration of the second GEMM's input global: every one of the Tc rows of
 * x_calib goes through every expert; d_amax[e] (optional, [E]) receives
 * max |h| of expert e and *d_g_a2 = max_e 2688 / amax_e.  Workspace:
 * nvfp4_moe_workspace(Tc, H, I, E, E). */
nvfp4_status nvfp4_moe_calibrate(const void* x_calib_bf16, int64_t Tc, int64_t H, int64_t I,
                                 int64_t E, const float* d_g_a1, const uint8_t* w13_codes,
                                 const uint8_t* w13_sf, const float* d_alpha13, float* d_amax,
                                 float* d_g_a2, void* workspace, size_t ws_bytes,
                                 nvfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * W4A16 MoE for small batches: decode and prefills with few tokens per expert
 * (the W4A4 MoE prefill page, section "Changes", keeps W4A16 below 4 tokens
 * per expert).  Same weight banks as nvfp4_moe_w4a4, no repack; activations
 * are never quantised:
 *   G, U = x @ W13[e][0:I].T, x @ W13[e][I:2I].T          (fp32 accumulation)
 *   h    = bf16(silu(alpha13[e] * G) * (alpha13[e] * U))
 *   out  = bf16(sum over the token's slots, in slot order, of
 *               w * alpha2[e] * (h @ W2[e].T))              (fp32 sum)
 * with d_alpha13[e] = 1 / g_w13[e] and d_alpha2[e] = 1 / g_w2[e] (no
 * activation global).  x: bf16 [T, H], contiguous, 16-byte aligned.  Routes
 * and weights as nvfp4_moe_w4a4; ids outside [0, E) set
 * NVFP4_ERR_BAD_EXPERT_ID in the device word and are dropped.
 * Shapes: 1 <= T <= 64, 1 <= topk <= 8, H % 128 == 0, I % 128 == 0,
 * H <= 16384, I <= 16384, E <= 1024; T = 0 returns NVFP4_OK with no launch.
 * w13_codes, w13_sf, w2_codes, w2_sf, out and workspace 16-byte aligned;
 * ids, weights and alphas 4-byte aligned (else NVFP4_ERR_MISALIGNED).  The
 * result is deterministic (no atomics in the sums).
 * --------------------------------------------------------------------------- */

/* Workspace bytes of nvfp4_moe_w4a16 for T tokens: the bf16 h of every route
 * [T*topk, I] and its fp32 weighted down row [T*topk, H]; 0 for an
 * unsupported shape. */
size_t nvfp4_moe_w4a16_workspace(int64_t T, int64_t H, int64_t I, int64_t E, int topk);

/* gate_up (64 gate rows with the matching 64 up rows per work item, h
 * written in its epilogue) -> down (w * alpha2 * h @ W2[e].T per route) ->
 * slot sum -> bf16:
 * three kernels chained by programmatic dependent launch.  No host
 * synchronisation. */
nvfp4_status nvfp4_moe_w4a16(const void* x_bf16, int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                             const int32_t* topk_ids, const float* topk_w, const uint8_t* w13_codes,
                             const uint8_t* w13_sf, const float* d_alpha13, const uint8_t* w2_codes,
                             const uint8_t* w2_sf, const float* d_alpha2, void* out_bf16, void* workspace,
                             size_t ws_bytes, nvfp4_stream_t stream);

/* Layout of the MoE workspace, for inspection of the intermediate stages
 * (all offsets in bytes from the workspace pointer, 256-byte aligned).  The
 * composite call fills:
 *   counts      int32 [E]         routes per expert
 *   offsets     int32 [E + 1]     first padded row of each expert; offsets[E] = P
 *   n_tiles     int32 [1]         P / 128
 *   row_map     int32 [P_max]     t * topk + slot of each permuted row, -1 for padding
 *   tile_expert int32 [P_max/128] expert of each 128-row tile
 *   pos         int32 [T*topk]    permuted row of each route, -1 if dropped
 *   hist        int32 [chunks, E] routes per expert in each chunk of routes
 *                                 (align's working space above 4096 routes)
 *   a1_codes    u8 [P_max, H/2]   quantised x at the permuted rows
 *   a1_sf       swizzled over P_max rows
 *   h_codes     u8 [P_max, I/2]   quantised SiLU(gate) * up
 *   h_sf        swizzled over P_max rows
 *   y           fp32 [T, H]       top-k sum before the bf16 rounding
 * row_block: the multiple of rows nvfp4_moe_w4a4 pads each expert's segment
 * to: 256 when T * topk >= 1024 * E and H % 256 == 0 (the grouped GEMMs then
 * run on CTA pairs whose 256-row tiles belong to one expert), else 128.
 * P_max = T * topk + E * (row_block - 1), rounded up to row_block.
 * nvfp4_moe_calibrate pads to 128 rows in a workspace of this layout. */
typedef struct {
  size_t counts, offsets, n_tiles, row_map, tile_expert, pos;
  size_t a1_codes, a1_sf, h_codes, h_sf, y, hist, total;
  int64_t p_max;
  int64_t row_block;
} nvfp4_moe_layout;

nvfp4_status nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                        nvfp4_moe_layout* host_layout);

/* Self-test of the device timeout path: launches one CTA whose pipeline wait
 * (the bounded mbarrier wait every kernel uses) has nobody to complete it.
 * The wait gives up after about a second and records NVFP4_ERR_DEVICE_TIMEOUT
 * in the device status word; the CTA then exits normally and the context
 * stays usable.  No fault, trap or unbounded wait is involved. */
nvfp4_status nvfp4_selftest_wait_timeout(nvfp4_stream_t stream);

/* Synchronises `stream`, copies the device status word to *host_out (an
 * nvfp4_status value, NVFP4_OK if nothing was flagged) and clears it. */
nvfp4_status nvfp4_device_status(nvfp4_stream_t stream, int32_t* host_out);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
