/*
 * CPU oracle for the Attention -> FFN MoE token dispatch and combine.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call this code. The library never does,
 * and this code shares nothing (types, headers, helpers, tables) with it.
 *
 * It is a plain, sequential, single-threaded restatement of what the
 * afdEP-comm "API contract" page defines (sections "Roles and tensors" and
 * "Graphs, streams and lifetime") for one exchange: validate the top-k IDs,
 * count routes per expert, lay experts out with the ends[] convention and
 * align_up(expert_alignment) padding, place every valid route's row in an
 * expert-major receive buffer, and sum the reply rows back per token with the
 * routing weight applied once.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared orc.c -lm
 * (-ffp-contract=off keeps every a*b+c a separate multiply and add; the only
 * fused operation is the explicit fmaf() of the combine step.)
 */
#ifndef ORC_H
#define ORC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ROUTE_RANGE = 1, ORC_ROUTE_DUP = 2 };
enum { ORC_BF16 = 0, ORC_FP8 = 1 };
enum { ORC_EXPERT_IDENTITY = 0, ORC_EXPERT_SCALE = 1 };

/* One exchange. Every per-source array is padded to `bucket` tokens:
 * index (s, t, k) lives at (s*bucket + t)*K + k; only t < T[s] is read. */
typedef struct orc_problem {
  int32_t A;      /* Attention sources */
  int32_t F;      /* FFN workers; worker f owns experts [f*E/F, (f+1)*E/F) */
  int32_t E;      /* experts */
  int32_t K;      /* top-k */
  int32_t H;      /* hidden size */
  int32_t alpha;  /* expert_alignment */
  int32_t bucket; /* padded tokens per source */
  int32_t dtype;  /* ORC_BF16 or ORC_FP8 */
  const int32_t* T; /* [A] live tokens per source */
} orc_problem;

/* ---- number formats (written from the format definitions) ---- */
float orc_bf16_to_float(uint16_t b);
uint16_t orc_float_to_bf16(float f);   /* round to nearest, ties to even */
float orc_e4m3_to_float(uint8_t q);    /* OCP FP8 E4M3 (bias 7, no inf) */
void orc_bf16_to_float_n(const uint16_t* in, float* out, int64_t n);
void orc_float_to_bf16_n(const float* in, uint16_t* out, int64_t n);
void orc_e4m3_to_float_n(const uint8_t* in, float* out, int64_t n);

/* ---- the exchange ---- */

/* First invalid route in (s, t, k) order. Returns ORC_OK, ORC_ROUTE_RANGE or
 * ORC_ROUTE_DUP and, when not OK, its (s, t, k). */
int32_t orc_validate(const orc_problem* p, const int64_t* ids,
                     int32_t* err_s, int32_t* err_t, int32_t* err_k);

/* Per worker f and local expert l (arrays [F][E/F]): raw route count,
 * aligned start, end (ends[]), aligned host count; r_exact[f] is the exact
 * receive row count. Invalid routes (see orc_validate) are not counted. */
void orc_layout(const orc_problem* p, const int64_t* ids, int32_t* count,
                int32_t* start, int32_t* ends, int32_t* host_counts,
                int64_t* r_exact);

/* Places every valid route. slot [A][bucket][K] gets the row inside the
 * owning worker (-1 when skipped). row_src and row_w are [F][r_stride];
 * rows are [F][r_stride][row_bytes] with row_bytes = 2H (BF16) or H (FP8);
 * row_scales is [F][r_stride][H/128] (FP8 only, else may be NULL).
 * x is [A][bucket][row_bytes] bytes and x_scales [A][bucket][H/128].
 * Rows in [0, r_exact) that no route fills get row_src -1 and row_w +0. */
void orc_dispatch(const orc_problem* p, const int64_t* ids, const float* w,
                  const uint8_t* x, const float* x_scales, const int32_t* start,
                  const int64_t* r_exact, int64_t r_stride, int32_t* slot,
                  int32_t* row_src, float* row_w, uint8_t* rows,
                  float* row_scales);

/* Stand-in FFN expert (not part of the exchange; it produces BF16 replies
 * from received rows). Identity: reply = row (BF16 only). Scale: reply =
 * bf16(value * c_e), c_e = 2^((e mod 4) - 1), value = the BF16 row value or,
 * for FP8, e4m3(q) * scale of its 128-block. reply is [F][r_stride][H]. */
void orc_expert(const orc_problem* p, int32_t mode, const int32_t* start,
                const int32_t* ends, int64_t r_stride, const uint8_t* rows,
                const float* row_scales, uint16_t* reply);

/* OCP E4M3 encoding, round to nearest even, saturating: finite values beyond
 * 448 and infinities become +-448; NaN becomes S.1111.111. */
uint8_t orc_float_to_e4m3(float f);
void orc_float_to_e4m3_n(const float* in, uint8_t* out, int64_t n);

/* Power-of-two scale exponent of one 128-element group (design page,
 * "19. FP8 combine replies"): the smallest integer e with amax <= 448 * 2^e,
 * compared in FP32, and at least -117. */
int32_t orc_group_exponent(float amax);
void orc_group_exponent_n(const float* amax, int32_t* out, int64_t n);

/* Two-stage combine (design page, sections 6 and 19): for every token, each
 * worker's routes give a BF16 partial (FP32 fused multiply-adds in ascending
 * k from +0, one rounding); with fp8 != 0 each partial is quantized to E4M3
 * with one power-of-two factor shared by each block of 128 values, and dequantized; the partials
 * are added in FP32 in the order of each worker's last route (ascending k),
 * from +0, and the sum is rounded once to BF16. */
void orc_combine_two_stage(const orc_problem* p, const int64_t* ids, const float* w,
                           const int32_t* slot, int64_t r_stride, const uint16_t* reply,
                           int32_t fp8, uint16_t* out);

/* out[s][t][h] = bf16( fma chain over k ascending of w[s][t][k] *
 * reply[f][slot][h] ), starting from +0.0f; skipped routes add nothing.
 * out is [A][bucket][H]; rows t >= T[s] are left untouched. */
void orc_combine(const orc_problem* p, const int64_t* ids, const float* w,
                 const int32_t* slot, int64_t r_stride, const uint16_t* reply,
                 uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
