/*
 * NVFP4 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of
 * __graft_entry__ and the cpu_baseline leg of bench.py may build, load or call
 * this file.  The CUDA library never does: it shares no code, header, table or
 * helper with this oracle.
 *
 * Plain, slow and meant to be read against the pages:
 *   [linear]  "run nvfp4 linears on nvfp4 activations on sm_120" (FreeToken PR 737),
 *             section "Changes" (row-major [N, K/2] codes, 128x4-swizzled block
 *             scales, one global per tensor, largest per-part global for fused
 *             weights, static activation global).
 *   [moe]     the W4A4 MoE prefill page (FreeToken PR 736), section "Changes"
 *             (gate_up with gated activation and NVFP4 quantisation of its output,
 *             down with routing weight and top-k sum, static per-expert input
 *             scales, max over experts).
 *   [flow]    "speed up the nvfp4 moe prefill gemm on rtx gpus" (FreeToken PR 733),
 *             section "Changes" (layer flow align -> gate_up -> act -> down -> sum).
 *   [mmbf16]  "Add BF16_FP4 GEMM ... for W4A16 workloads" (FlashInfer PR 3597),
 *             sections "Summary" (out = (a @ dequant(b, b_sf).T) * alpha, per-16
 *             FP8-E4M3 block scales) and "API" (g_w = 448*6/amax(w),
 *             alpha = 1/g_w, SfLayout.layout_128x4) and the review excerpt that
 *             gives the E2M1 nibble table (low 3 bits magnitude, bit 3 sign).
 *
 * Arithmetic is IEEE fp32 with round-to-nearest-even, evaluated exactly in the
 * order written (build with -ffp-contract=off, never -ffast-math).  Readings of
 * points the pages leave open are marked READING.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* threads                                                                   */
/* ------------------------------------------------------------------------- */

void nvo_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int nvo_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* bf16                                                                      */
/* ------------------------------------------------------------------------- */

float nvo_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round an fp32 value to the nearest bf16, ties to the even code.  The two
 * candidates are the truncation and the next code away from zero; the one
 * past the largest finite bf16 stands for 2^128 (which rounds to infinity). */
uint16_t nvo_f32_to_bf16(float f) {
  if (isnan(f)) return 0x7FC0;
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t lo = (uint16_t)(u >> 16);
  float flo = nvo_bf16_to_f32(lo);
  if (flo == f) return lo;
  uint16_t hi = (uint16_t)(lo + 1);
  double vlo = (double)flo;
  double vhi = isinf(nvo_bf16_to_f32(hi)) ? copysign(ldexp(1.0, 128), (double)f)
                                          : (double)nvo_bf16_to_f32(hi);
  double dlo = fabs((double)f - vlo), dhi = fabs(vhi - (double)f);
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo & 1) ? hi : lo;
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 (block scale): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; */
/* exponent field 0 is subnormal; 0x7F / 0xFF are NaN; no infinity.          */
/* ------------------------------------------------------------------------- */

float nvo_e4m3_to_f32(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9)            /* (m/8) * 2^-6      */
                      : ldexp((double)(8 + m), e - 10); /* (1+m/8) * 2^(e-7) */
  return (float)(s ? -v : v);
}

/* Nearest finite E4M3 value, ties to the even code; magnitudes above 448
 * saturate to 448 ("satfinite").  The sign of the input is kept. */
uint8_t nvo_f32_to_e4m3_satfinite(float f) {
  double a = fabs((double)f);
  uint8_t sign = signbit(f) ? 0x80 : 0x00;
  /* satfinite: a magnitude at or beyond the largest finite value (448) maps to
   * it; said explicitly because the distances below stop telling candidates
   * apart once a is huge (or infinite) */
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(a - (double)nvo_e4m3_to_f32((uint8_t)c));
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------- */
/* E2M1 codes: low 3 bits magnitude, bit 3 sign ([mmbf16], review excerpt).   */
/* Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.                                     */
/* ------------------------------------------------------------------------- */

static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float nvo_e2m1_to_f32(uint8_t code) {
  double v = kE2M1Mag[code & 7];
  return (float)((code & 8) ? -v : v);
}

/* Nearest e2m1 value, ties to the even code, magnitudes above 6 give 6.
 * READING: a negative value that rounds to zero keeps its sign (code 0x8),
 * as an IEEE conversion does. */
uint8_t nvo_f32_to_e2m1_satfinite(float f) {
  double a = fabs((double)f);
  uint8_t sign = signbit(f) ? 0x8 : 0x0;
  /* satfinite: a magnitude at or beyond the largest finite value (6) maps to
   * it; said explicitly because the distances below stop telling candidates
   * apart once a is huge (or infinite) */
  if (a >= 6.0) return (uint8_t)(sign | 7);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - kE2M1Mag[c]);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------- */
/* 128x4-swizzled block-scale layout ([linear] Changes: the block scales of  */
/* the weight are stored 128x4-swizzled;                                      */
/* [mmbf16] SfLayout.layout_128x4).  READING: the pages name the layout but    */
/* print no formula; this is the block-scaling layout scaled_mm consumes: the  */
/* scale matrix (rows x C) is cut into 128-row x 4-column atoms of 512 bytes,  */
/* atoms ordered row-block major; inside an atom, row r and column c sit at    */
/* (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.  Rows and columns are padded  */
/* to multiples of 128 and 4 with zero bytes.                                  */
/* ------------------------------------------------------------------------- */

int64_t nvo_scale_cols_padded(int64_t C) { return (C + 3) / 4 * 4; }

size_t nvo_scale_bytes(int64_t rows, int64_t k) {
  int64_t C = k / 16;
  return (size_t)(((rows + 127) / 128) * 128) * (size_t)nvo_scale_cols_padded(C);
}

int64_t nvo_scale_offset(int64_t r, int64_t c, int64_t C) {
  int64_t Cp = nvo_scale_cols_padded(C);
  return ((r / 128) * (Cp / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* ------------------------------------------------------------------------- */
/* global scale: g = 448 * 6 / amax ([mmbf16] "API", the g_w line).           */
/* READING: an all-zero tensor has no amax; it gets g = 1 (any finite g gives */
/* the same all-zero codes).                                                   */
/* ------------------------------------------------------------------------- */

float nvo_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float v = fabsf(nvo_bf16_to_f32(x[r * ld + c]));
      if (v > amax) amax = v;
    }
  return amax;
}

float nvo_global_from_amax(float amax) { return amax > 0.0f ? 2688.0f / amax : 1.0f; }

float nvo_global_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld) {
  return nvo_global_from_amax(nvo_amax_bf16(x, rows, cols, ld));
}

/* ------------------------------------------------------------------------- */
/* quantisation of one row of K fp32 values with global g                     */
/* ([linear] activation quant; [mmbf16] nvfp4_quantize with a global):        */
/* per 16-element block b                                                      */
/*   amax_b = max |x_i|                                                        */
/*   s_f    = (amax_b / 6) * g            two fp32 operations in this order    */
/*   s8     = E4M3 satfinite(s_f),  S = value of s8                            */
/*   S == 0 -> every code of the block is +0                                   */
/*   else r = g / S and code_i = e2m1 satfinite(x_i * r)                       */
/* element 2j goes to the low nibble of byte j, 2j+1 to the high nibble.       */
/* READING: the order of these fp32 operations is not on the pages; this is  */
/* the plainest one.                                                           */
/* ------------------------------------------------------------------------- */

static void quant_row_f32(const float* x, int64_t K, float g, uint8_t* codes_row,
                          uint8_t* sf, int64_t row, int64_t C) {
  for (int64_t b = 0; b < K / 16; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float v = fabsf(x[16 * b + i]);
      if (v > amax) amax = v;
    }
    float s_f = (amax / 6.0f) * g;
    uint8_t s8 = nvo_f32_to_e4m3_satfinite(s_f);
    float S = nvo_e4m3_to_f32(s8);
    sf[nvo_scale_offset(row, b, C)] = s8;
    for (int i = 0; i < 16; ++i) {
      uint8_t code = 0;
      if (S != 0.0f) {
        float r = g / S;
        float y = x[16 * b + i] * r;
        code = nvo_f32_to_e2m1_satfinite(y);
      }
      int64_t k = 16 * b + i;
      if (k & 1)
        codes_row[k / 2] = (uint8_t)(codes_row[k / 2] | (code << 4));
      else
        codes_row[k / 2] = (uint8_t)(code & 0xF);
    }
  }
}

/* bf16 [M, K] (row stride ldx) -> codes [M, K/2] and scales (sw(M, K/16) bytes,
 * padding zero).  K must be a multiple of 16. */
void nvo_quantize_bf16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                       uint8_t* codes, uint8_t* scales) {
  int64_t C = K / 16;
  memset(scales, 0, nvo_scale_bytes(M, K));
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    float* row = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t k = 0; k < K; ++k) row[k] = nvo_bf16_to_f32(x[m * ldx + k]);
    quant_row_f32(row, K, g, codes + m * (K / 2), scales, m, C);
    free(row);
  }
}

/* fp32 [M, K] variant (the MoE intermediate is quantised from fp32). */
void nvo_quantize_f32(const float* x, int64_t M, int64_t K, int64_t ldx, float g,
                      uint8_t* codes, uint8_t* scales) {
  int64_t C = K / 16;
  memset(scales, 0, nvo_scale_bytes(M, K));
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) quant_row_f32(x + m * ldx, K, g, codes + m * (K / 2), scales, m, C);
}

/* dequantise without the global: value = e2m1(code) * S (exact in fp32) */
void nvo_dequant(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t K, float* out) {
  int64_t C = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
      float S = nvo_e4m3_to_f32(scales[nvo_scale_offset(r, k / 16, C)]);
      out[r * K + k] = nvo_e2m1_to_f32(code) * S;
    }
}

/* ------------------------------------------------------------------------- */
/* W4A4 linear ([linear] W4A4 GEMM on NVFP4 activations; the W4A16 form of     */
/* [mmbf16] "Summary" read with both operands dequantised):                    */
/*   acc = sum_k A^[m,k] * W^[n,k]     one fp32 sum, ascending k                */
/*   out = bf16(acc * alpha),  alpha = 1 / (g_a * g_w)                          */
/* A^ = e2m1 * S_a and W^ = e2m1 * S_w carry no global; every product is exact */
/* in fp32.                                                                    */
/* ------------------------------------------------------------------------- */

void nvo_linear_w4a4(const uint8_t* a_codes, const uint8_t* a_sf, int64_t M,
                     const uint8_t* w_codes, const uint8_t* w_sf, int64_t N, int64_t K,
                     float alpha, uint16_t* out, int64_t ldo) {
  float* A = (float*)malloc(sizeof(float) * (size_t)(M * K + 1));
  float* W = (float*)malloc(sizeof(float) * (size_t)(N * K + 1));
  nvo_dequant(a_codes, a_sf, M, K, A);
  nvo_dequant(w_codes, w_sf, N, K, W);
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      for (int64_t k = 0; k < K; ++k) acc += A[m * K + k] * W[n * K + k];
      out[m * ldo + n] = nvo_f32_to_bf16(acc * alpha);
    }
  free(A);
  free(W);
}

/* ------------------------------------------------------------------------- */
/* W4A16 linear ([mmbf16] "Summary": out = (a @ dequant(b, b_sf).T) * alpha;   */
/* alpha = 1 / g_w from "API"):                                                */
/*   acc = sum_k float(a[t,k]) * W^[n,k]   fp32, ascending k                    */
/*   out = bf16(acc * alpha)                                                   */
/* ------------------------------------------------------------------------- */

void nvo_linear_w4a16(const uint16_t* x, int64_t T, int64_t ldx, const uint8_t* w_codes,
                      const uint8_t* w_sf, int64_t N, int64_t K, float alpha, uint16_t* out,
                      int64_t ldo) {
  float* W = (float*)malloc(sizeof(float) * (size_t)(N * K + 1));
  nvo_dequant(w_codes, w_sf, N, K, W);
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t t = 0; t < T; ++t) {
      float acc = 0.0f;
      for (int64_t k = 0; k < K; ++k) acc += nvo_bf16_to_f32(x[t * ldx + k]) * W[n * K + k];
      out[t * ldo + n] = nvo_f32_to_bf16(acc * alpha);
    }
  free(W);
}

/* ------------------------------------------------------------------------- */
/* MoE token alignment ([flow] "align"): a stable counting sort of the        */
/* (token, slot) routes by expert; each expert's segment is padded to a       */
/* multiple of BM rows.  Outputs                                               */
/*   counts[e]      routes of expert e (valid ids only)                         */
/*   offsets[e]     first padded row of expert e; offsets[E] = P               */
/*   row_map[p]     t * topk + slot for a real row, -1 for a padding row        */
/*   tile_expert[i] expert of rows [i*BM, (i+1)*BM)                            */
/* Routes with an id outside [0, E) are dropped.  Returns P, or -1 if P would  */
/* exceed cap.                                                                 */
/* ------------------------------------------------------------------------- */

int64_t nvo_moe_align(const int32_t* ids, int64_t T, int64_t topk, int64_t E, int64_t BM,
                      int32_t* counts, int32_t* offsets, int32_t* row_map,
                      int32_t* tile_expert, int64_t cap) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * topk; ++i)
    if (ids[i] >= 0 && ids[i] < E) counts[ids[i]]++;
  int64_t P = 0;
  for (int64_t e = 0; e < E; ++e) {
    offsets[e] = (int32_t)P;
    P += (counts[e] + BM - 1) / BM * BM;
  }
  offsets[E] = (int32_t)P;
  if (P > cap) return -1;
  for (int64_t p = 0; p < P; ++p) row_map[p] = -1;
  int64_t* fill = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
  for (int64_t i = 0; i < T * topk; ++i) {
    int32_t e = ids[i];
    if (e < 0 || e >= E) continue;
    row_map[offsets[e] + fill[e]] = (int32_t)i;
    fill[e]++;
  }
  free(fill);
  for (int64_t e = 0; e < E; ++e)
    for (int64_t p = offsets[e]; p < offsets[e + 1]; p += BM) tile_expert[p / BM] = (int32_t)e;
  return P;
}

/* ------------------------------------------------------------------------- */
/* MoE layer, W4A4 ([moe] "Changes"; [flow] align -> gate_up -> act -> down   */
/* -> sum):                                                                    */
/*  1. x -> NVFP4 with the static input global g_a1 (the quantisation above)   */
/*  2. per route (t, slot), e = topk_ids[t, slot]:                             */
/*       G_j = sum_k x^[t,k] W13^[e][j][k],  U_j = sum_k x^[t,k] W13^[e][I+j][k] */
/*       (rows [0, I) gate, rows [I, 2I) up: READING, the pages do not say)      */
/*  3. h_j = silu(alpha13[e] * G_j) * (alpha13[e] * U_j),                       */
/*       silu(v) = v / (1 + expf(-v))                                           */
/*  4. h -> NVFP4 with the static global g_a2                                  */
/*  5. d_n = alpha2[e] * sum_k h^[k] W2^[e][n][k]                               */
/*  6. y[t,n] = sum over slots in order 0..topk-1 of (w[t,slot] * d_n), fp32;   */
/*     out = bf16(y).  READING: the pages add the top-k routes with bf16       */
/*     atomics in a varying order; the oracle adds in fp32 in slot order.      */
/*  Routes with an id outside [0, E) contribute nothing.                       */
/* Optional h_codes [T*topk, I/2] and h_sf (sw(T*topk, I/16)) receive step 4's  */
/* codes and scales for row t * topk + slot (zero for dropped routes).         */
/* Experts are visited one at a time, so only one expert's dequantised weights */
/* are held in memory.                                                         */
/* ------------------------------------------------------------------------- */

static float silu_f32(float v) { return v / (1.0f + expf(-v)); }

void nvo_moe_w4a4(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                  const int32_t* topk_ids, const float* topk_w, float g_a1,
                  const uint8_t* w13_codes, const uint8_t* w13_sf, const float* alpha13,
                  float g_a2, const uint8_t* w2_codes, const uint8_t* w2_sf,
                  const float* alpha2, uint16_t* out, uint8_t* h_codes, uint8_t* h_sf) {
  const int64_t R = T * topk;
  uint8_t* xq = (uint8_t*)malloc((size_t)(T * (H / 2) + 1));
  uint8_t* xs = (uint8_t*)malloc(nvo_scale_bytes(T, H) + 1);
  float* X = (float*)malloc(sizeof(float) * (size_t)(T * H + 1));
  nvo_quantize_bf16(x, T, H, H, g_a1, xq, xs);
  nvo_dequant(xq, xs, T, H, X);

  float* D = (float*)calloc((size_t)(R * H + 1), sizeof(float)); /* d per route */
  uint8_t* hq_all = (uint8_t*)calloc((size_t)(R * (I / 2) + 1), 1);
  uint8_t* hs_all = (uint8_t*)calloc(nvo_scale_bytes(R, I) + 1, 1);
  float* W13 = (float*)malloc(sizeof(float) * (size_t)(2 * I * H + 1));
  float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I + 1));
  const size_t w13_bytes = (size_t)(2 * I) * (size_t)(H / 2), w13_sfb = nvo_scale_bytes(2 * I, H);
  const size_t w2_bytes = (size_t)H * (size_t)(I / 2), w2_sfb = nvo_scale_bytes(H, I);
  int64_t* routes = (int64_t*)malloc(sizeof(int64_t) * (size_t)(R + 1));

  for (int64_t e = 0; e < E; ++e) {
    int64_t nr = 0;
    for (int64_t i = 0; i < R; ++i)
      if (topk_ids[i] == e) routes[nr++] = i;
    if (nr == 0) continue;
    nvo_dequant(w13_codes + (size_t)e * w13_bytes, w13_sf + (size_t)e * w13_sfb, 2 * I, H, W13);
    nvo_dequant(w2_codes + (size_t)e * w2_bytes, w2_sf + (size_t)e * w2_sfb, H, I, W2);
#pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < nr; ++q) {
      int64_t i = routes[q], t = i / topk;
      float* h = (float*)malloc(sizeof(float) * (size_t)I);
      float* hd = (float*)malloc(sizeof(float) * (size_t)I);
      uint8_t* hq = hq_all + i * (I / 2);
      uint8_t* hs1 = (uint8_t*)calloc(nvo_scale_bytes(1, I), 1);
      for (int64_t j = 0; j < I; ++j) {
        float G = 0.0f, U = 0.0f;
        for (int64_t k = 0; k < H; ++k) G += X[t * H + k] * W13[j * H + k];
        for (int64_t k = 0; k < H; ++k) U += X[t * H + k] * W13[(I + j) * H + k];
        h[j] = silu_f32(alpha13[e] * G) * (alpha13[e] * U);
      }
      /* step 4 on this one row; its scales are moved to row i of the shared
       * swizzled array below */
      quant_row_f32(h, I, g_a2, hq, hs1, 0, I / 16);
      for (int64_t c = 0; c < I / 16; ++c) {
        uint8_t s8 = hs1[nvo_scale_offset(0, c, I / 16)];
        hs_all[nvo_scale_offset(i, c, I / 16)] = s8;
        float S = nvo_e4m3_to_f32(s8);
        for (int64_t u = 0; u < 16; ++u) {
          int64_t k = 16 * c + u;
          uint8_t code = (k & 1) ? (hq[k / 2] >> 4) : (hq[k / 2] & 0xF);
          hd[k] = nvo_e2m1_to_f32(code) * S;
        }
      }
      for (int64_t n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int64_t k = 0; k < I; ++k) acc += hd[k] * W2[n * I + k];
        D[i * H + n] = alpha2[e] * acc;
      }
      free(h);
      free(hd);
      free(hs1);
    }
  }
  /* step 6: fp32 sum over the slots in order */
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < H; ++n) {
      float y = 0.0f;
      for (int64_t s = 0; s < topk; ++s) {
        int64_t i = t * topk + s;
        int32_t e = topk_ids[i];
        if (e < 0 || e >= E) continue;
        y += topk_w[i] * D[i * H + n];
      }
      out[t * H + n] = nvo_f32_to_bf16(y);
    }
  if (h_codes) memcpy(h_codes, hq_all, (size_t)(R * (I / 2)));
  if (h_sf) memcpy(h_sf, hs_all, nvo_scale_bytes(R, I));
  free(routes);
  free(W13);
  free(W2);
  free(hq_all);
  free(hs_all);
  free(D);
  free(X);
  free(xs);
  free(xq);
}

/* ------------------------------------------------------------------------- */
/* MoE down projection on a given NVFP4 intermediate ([moe] "Changes": the     */
/* routed down GEMM applies the routing weight and sums the top-k outputs).    */
/* Steps 5 and 6 of the layer above, taken on their own so that a caller can   */
/* hand in another implementation's h:                                         */
/*   d[n]   = alpha2[e] * sum_k h^[i,k] * W2^[e][n,k]   fp32, ascending k       */
/*   y[t,n] = sum over slots s in order of w[t,s] * d[n] (fp32), out = bf16(y)  */
/* h_codes [T*topk, I/2] and h_sf (swizzled over T*topk rows) hold route       */
/* i = t * topk + s; routes with an id outside [0, E) are dropped.              */
/* ------------------------------------------------------------------------- */

void nvo_moe_down(const uint8_t* h_codes, const uint8_t* h_sf, int64_t T, int64_t H, int64_t I,
                  int64_t E, int64_t topk, const int32_t* topk_ids, const float* topk_w,
                  const uint8_t* w2_codes, const uint8_t* w2_sf, const float* alpha2, uint16_t* out) {
  const int64_t R = T * topk;
  float* Hd = (float*)malloc(sizeof(float) * (size_t)(R * I + 1));
  nvo_dequant(h_codes, h_sf, R, I, Hd);
  float* D = (float*)calloc((size_t)(R * H + 1), sizeof(float));
  float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I + 1));
  const size_t w2_bytes = (size_t)H * (size_t)(I / 2), w2_sfb = nvo_scale_bytes(H, I);
  int64_t* routes = (int64_t*)malloc(sizeof(int64_t) * (size_t)(R + 1));
  for (int64_t e = 0; e < E; ++e) {
    int64_t nr = 0;
    for (int64_t i = 0; i < R; ++i)
      if (topk_ids[i] == e) routes[nr++] = i;
    if (nr == 0) continue;
    nvo_dequant(w2_codes + (size_t)e * w2_bytes, w2_sf + (size_t)e * w2_sfb, H, I, W2);
#pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < nr; ++q) {
      const int64_t i = routes[q];
      for (int64_t n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int64_t k = 0; k < I; ++k) acc += Hd[i * I + k] * W2[n * I + k];
        D[i * H + n] = alpha2[e] * acc;
      }
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < H; ++n) {
      float y = 0.0f;
      for (int64_t s = 0; s < topk; ++s) {
        const int64_t i = t * topk + s;
        const int32_t e = topk_ids[i];
        if (e < 0 || e >= E) continue;
        y += topk_w[i] * D[i * H + n];
      }
      out[t * H + n] = nvo_f32_to_bf16(y);
    }
  free(routes);
  free(W2);
  free(D);
  free(Hd);
}

/* ------------------------------------------------------------------------- */
/* W4A16 MoE for small batches ([moe] "Changes": prefill runs W4A4 from 4     */
/* tokens per expert and W4A16 below; "Decode ... and W4A16 prefill are       */
/* untouched").  READING: [moe]'s layer with the activations never quantised   */
/* (the W4A16 linear of [mmbf16] applied per expert):                          */
/*   G = sum_k x[t,k] W13^[j,k],  U = sum_k x[t,k] W13^[I+j,k]   fp32, asc. k   */
/*   h[j] = bf16(silu(alpha13[e] * G) * (alpha13[e] * U))   the intermediate is */
/*          an activation of a W4A16 layer, so it is rounded to bf16            */
/*   d[n] = alpha2[e] * sum_k h[k] W2^[n,k]                  fp32, asc. k       */
/*   y[t,n] = sum over slots s in order of w[t,s] * d[n] (fp32), out = bf16(y)  */
/* alpha13[e] = 1 / g13[e], alpha2[e] = 1 / g2[e].  Routes with an id outside  */
/* [0, E) are dropped.                                                          */
/* ------------------------------------------------------------------------- */

void nvo_moe_w4a16(const uint16_t* x, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                   const int32_t* topk_ids, const float* topk_w, const uint8_t* w13_codes,
                   const uint8_t* w13_sf, const float* alpha13, const uint8_t* w2_codes,
                   const uint8_t* w2_sf, const float* alpha2, uint16_t* out, uint16_t* h_out) {
  const int64_t R = T * topk;
  float* D = (float*)calloc((size_t)(R * H + 1), sizeof(float)); /* d per route */
  float* W13 = (float*)malloc(sizeof(float) * (size_t)(2 * I * H + 1));
  float* W2 = (float*)malloc(sizeof(float) * (size_t)(H * I + 1));
  const size_t w13_bytes = (size_t)(2 * I) * (size_t)(H / 2), w13_sfb = nvo_scale_bytes(2 * I, H);
  const size_t w2_bytes = (size_t)H * (size_t)(I / 2), w2_sfb = nvo_scale_bytes(H, I);
  int64_t* routes = (int64_t*)malloc(sizeof(int64_t) * (size_t)(R + 1));

  for (int64_t e = 0; e < E; ++e) {
    int64_t nr = 0;
    for (int64_t i = 0; i < R; ++i)
      if (topk_ids[i] == e) routes[nr++] = i;
    if (nr == 0) continue;
    nvo_dequant(w13_codes + (size_t)e * w13_bytes, w13_sf + (size_t)e * w13_sfb, 2 * I, H, W13);
    nvo_dequant(w2_codes + (size_t)e * w2_bytes, w2_sf + (size_t)e * w2_sfb, H, I, W2);
#pragma omp parallel for schedule(dynamic)
    for (int64_t q = 0; q < nr; ++q) {
      int64_t i = routes[q], t = i / topk;
      float* h = (float*)malloc(sizeof(float) * (size_t)I);
      for (int64_t j = 0; j < I; ++j) {
        float G = 0.0f, U = 0.0f;
        for (int64_t k = 0; k < H; ++k) G += nvo_bf16_to_f32(x[t * H + k]) * W13[j * H + k];
        for (int64_t k = 0; k < H; ++k) U += nvo_bf16_to_f32(x[t * H + k]) * W13[(I + j) * H + k];
        const uint16_t hb = nvo_f32_to_bf16(silu_f32(alpha13[e] * G) * (alpha13[e] * U));
        if (h_out) h_out[i * I + j] = hb;
        h[j] = nvo_bf16_to_f32(hb);
      }
      for (int64_t n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int64_t k = 0; k < I; ++k) acc += h[k] * W2[n * I + k];
        D[i * H + n] = alpha2[e] * acc;
      }
      free(h);
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t n = 0; n < H; ++n) {
      float y = 0.0f;
      for (int64_t s = 0; s < topk; ++s) {
        int64_t i = t * topk + s;
        int32_t e = topk_ids[i];
        if (e < 0 || e >= E) continue;
        y += topk_w[i] * D[i * H + n];
      }
      out[t * H + n] = nvo_f32_to_bf16(y);
    }
  free(routes);
  free(W13);
  free(W2);
  free(D);
}

/* ------------------------------------------------------------------------- */
/* MoE calibration of the second GEMM's input ([moe] "Static activation        */
/* scales": the largest per-expert input global feeds each GEMM).  READING:   */
/* every calibration row goes through every expert (steps 1-3 above), so each  */
/* expert has a finite amax; amax_out[e] = max |h| over the rows and the I     */
/* columns.  The caller forms g_a2,e = 2688 / amax_out[e] and takes the max.   */
/* ------------------------------------------------------------------------- */

void nvo_moe_h_amax(const uint16_t* x, int64_t Tc, int64_t H, int64_t I, int64_t E, float g_a1,
                    const uint8_t* w13_codes, const uint8_t* w13_sf, const float* alpha13,
                    float* amax_out) {
  uint8_t* xq = (uint8_t*)malloc((size_t)(Tc * (H / 2) + 1));
  uint8_t* xs = (uint8_t*)malloc(nvo_scale_bytes(Tc, H) + 1);
  float* X = (float*)malloc(sizeof(float) * (size_t)(Tc * H + 1));
  nvo_quantize_bf16(x, Tc, H, H, g_a1, xq, xs);
  nvo_dequant(xq, xs, Tc, H, X);
  float* W13 = (float*)malloc(sizeof(float) * (size_t)(2 * I * H + 1));
  const size_t w13_bytes = (size_t)(2 * I) * (size_t)(H / 2), w13_sfb = nvo_scale_bytes(2 * I, H);
  float* rowmax = (float*)malloc(sizeof(float) * (size_t)(Tc + 1));
  for (int64_t e = 0; e < E; ++e) {
    nvo_dequant(w13_codes + (size_t)e * w13_bytes, w13_sf + (size_t)e * w13_sfb, 2 * I, H, W13);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < Tc; ++t) {
      float m = 0.0f;
      for (int64_t j = 0; j < I; ++j) {
        float G = 0.0f, U = 0.0f;
        for (int64_t k = 0; k < H; ++k) G += X[t * H + k] * W13[j * H + k];
        for (int64_t k = 0; k < H; ++k) U += X[t * H + k] * W13[(I + j) * H + k];
        float h = fabsf(silu_f32(alpha13[e] * G) * (alpha13[e] * U));
        if (h > m) m = h;
      }
      rowmax[t] = m;
    }
    float m = 0.0f;
    for (int64_t t = 0; t < Tc; ++t)
      if (rowmax[t] > m) m = rowmax[t];
    amax_out[e] = m;
  }
  free(rowmax);
  free(W13);
  free(X);
  free(xs);
  free(xq);
}
