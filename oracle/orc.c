/*
 * CPU oracle for the Attention -> FFN MoE token dispatch and combine.
 * TEST INFRASTRUCTURE ONLY (see orc.h). Sequential on purpose: every step is
 * the plain definition, so a reader can check it against the pages by eye.
 *
 * Sources: afdEP-comm "API contract" (Roles and tensors; Graphs, streams and
 * lifetime); afdEP-comm design page, "10. Single-FFN reduction" and
 * "13. Single-FFN collect view"; "DeepEP V2 ElasticBuffer first principles",
 * section 3 (per-route slot and expert-major placement) and section 7 (FP8
 * dispatch with per-block scales, BF16 combine).
 */
#include "orc.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* BF16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7
 * fraction bits. Widening is exact. */
float orc_bf16_to_float(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

/* Narrowing drops the low 16 bits of the binary32 pattern, rounding to
 * nearest with ties to even. Because binary32 and BF16 share the exponent
 * field, incrementing the kept pattern carries correctly into the exponent
 * (and into infinity on overflow). NaN stays NaN (quiet, sign kept). */
uint16_t orc_float_to_bf16(float f) {
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu) != 0)
    return (uint16_t)((bits >> 16) | 0x0040u);
  uint32_t kept = bits >> 16;
  uint32_t dropped = bits & 0xffffu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
    kept += 1u;
  return (uint16_t)kept;
}

/* OCP 8-bit E4M3: 1 sign, 4 exponent (bias 7), 3 fraction bits. Exponent
 * field 0 is subnormal (value = fraction/8 * 2^-6); S.1111.111 is NaN; there
 * is no infinity, so S.1111.110 = 448 is the largest finite value. */
float orc_e4m3_to_float(uint8_t q) {
  int sign = (q >> 7) & 1;
  int e = (q >> 3) & 0xf;
  int m = q & 7;
  float v;
  if (e == 0xf && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexpf((float)m, -9); /* m/8 * 2^(1-7) */
  else
    v = ldexpf((float)(8 + m), e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Routes                                                                    */
/* ------------------------------------------------------------------------ */

static int64_t route_index(const orc_problem* p, int s, int t, int k) {
  return ((int64_t)s * p->bucket + t) * p->K + k;
}

/* Classifies route (s,t,k). "API contract", Roles and tensors: an ID is
 * either -1 (skip) or an expert number in [0, num_experts), and no expert
 * repeats within a token; anything else is an invalid route. A duplicate is the second (or later) occurrence of an
 * in-range ID inside one token. Returns 1 (valid), 0 (skip, -1) or
 * -ORC_ROUTE_RANGE / -ORC_ROUTE_DUP. */
static int classify(const orc_problem* p, const int64_t* ids, int s, int t,
                    int k) {
  int64_t id = ids[route_index(p, s, t, k)];
  if (id == -1) return 0;
  if (id < -1 || id >= p->E) return -ORC_ROUTE_RANGE;
  for (int j = 0; j < k; ++j)
    if (ids[route_index(p, s, t, j)] == id) return -ORC_ROUTE_DUP;
  return 1;
}

int32_t orc_validate(const orc_problem* p, const int64_t* ids, int32_t* err_s,
                     int32_t* err_t, int32_t* err_k) {
  for (int s = 0; s < p->A; ++s)
    for (int t = 0; t < p->T[s]; ++t)
      for (int k = 0; k < p->K; ++k) {
        int c = classify(p, ids, s, t, k);
        if (c < 0) {
          *err_s = s;
          *err_t = t;
          *err_k = k;
          return -c;
        }
      }
  *err_s = *err_t = *err_k = -1;
  return ORC_OK;
}

static int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

/* "API contract", Roles and tensors: worker f owns the E/F consecutive
 * experts starting at f*E/F. Receive prefix sum: expert e occupies
 * [align_up(ends[e-1], alpha), ends[e]) with ends[-1] = 0, numbered locally
 * per worker; host counts report aligned per-expert counts. */
void orc_layout(const orc_problem* p, const int64_t* ids, int32_t* count,
                int32_t* start, int32_t* ends, int32_t* host_counts,
                int64_t* r_exact) {
  const int Ef = p->E / p->F;
  for (int i = 0; i < p->E; ++i) count[i] = 0;

  for (int s = 0; s < p->A; ++s)
    for (int t = 0; t < p->T[s]; ++t)
      for (int k = 0; k < p->K; ++k)
        if (classify(p, ids, s, t, k) == 1) {
          int64_t e = ids[route_index(p, s, t, k)];
          count[e] += 1; /* [f][l] flattened is exactly [e] */
        }

  for (int f = 0; f < p->F; ++f) {
    int64_t prev_end = 0; /* ends[-1] = 0 */
    for (int l = 0; l < Ef; ++l) {
      int i = f * Ef + l;
      start[i] = (int32_t)align_up(prev_end, p->alpha);
      ends[i] = start[i] + count[i];
      host_counts[i] = (int32_t)align_up(count[i], p->alpha);
      prev_end = ends[i];
    }
    r_exact[f] = align_up(prev_end, p->alpha);
  }
}

/* Expert-major placement. Within one expert, rows follow (source ascending,
 * token ascending); each valid route takes the next free row of its expert
 * ("DeepEP V2 ElasticBuffer first principles" section 3 assigns these slots
 * in arrival order with an atomic counter per destination; this oracle fixes
 * the order so that the result is unique). The row is a byte copy of the
 * source row and, for FP8, of its FP32 block-128 scales. */
void orc_dispatch(const orc_problem* p, const int64_t* ids, const float* w,
                  const uint8_t* x, const float* x_scales, const int32_t* start,
                  const int64_t* r_exact, int64_t r_stride, int32_t* slot,
                  int32_t* row_src, float* row_w, uint8_t* rows,
                  float* row_scales) {
  const int Ef = p->E / p->F;
  const int64_t row_bytes = p->dtype == ORC_FP8 ? p->H : 2 * (int64_t)p->H;
  const int nb = p->H / 128;
  int64_t* cursor = (int64_t*)malloc(sizeof(int64_t) * (size_t)p->E);

  for (int f = 0; f < p->F; ++f)
    for (int64_t r = 0; r < r_exact[f]; ++r) {
      row_src[f * r_stride + r] = -1;
      row_w[f * r_stride + r] = 0.0f;
    }
  for (int e = 0; e < p->E; ++e) cursor[e] = start[e];

  for (int s = 0; s < p->A; ++s)
    for (int t = 0; t < p->bucket; ++t)
      for (int k = 0; k < p->K; ++k) {
        int64_t ri = route_index(p, s, t, k);
        if (t >= p->T[s] || classify(p, ids, s, t, k) != 1) {
          slot[ri] = -1;
          continue;
        }
        int64_t e = ids[ri];
        int f = (int)(e / Ef);
        int64_t row = cursor[e]++;
        slot[ri] = (int32_t)row;
        row_src[f * r_stride + row] = (int32_t)ri;
        row_w[f * r_stride + row] = w[ri];
        memcpy(rows + (f * r_stride + row) * row_bytes,
               x + ((int64_t)s * p->bucket + t) * row_bytes, (size_t)row_bytes);
        if (p->dtype == ORC_FP8)
          for (int b = 0; b < nb; ++b)
            row_scales[(f * r_stride + row) * nb + b] =
                x_scales[((int64_t)s * p->bucket + t) * nb + b];
      }
  free(cursor);
}

/* Harness expert: turns each live received row into a BF16 reply. */
void orc_expert(const orc_problem* p, int32_t mode, const int32_t* start,
                const int32_t* ends, int64_t r_stride, const uint8_t* rows,
                const float* row_scales, uint16_t* reply) {
  const int Ef = p->E / p->F;
  const int64_t row_bytes = p->dtype == ORC_FP8 ? p->H : 2 * (int64_t)p->H;
  const int nb = p->H / 128;
  for (int f = 0; f < p->F; ++f)
    for (int l = 0; l < Ef; ++l) {
      int e = f * Ef + l;
      float c = mode == ORC_EXPERT_SCALE ? ldexpf(1.0f, (e % 4) - 1) : 1.0f;
      for (int64_t r = start[e]; r < ends[e]; ++r) {
        const uint8_t* row = rows + (f * r_stride + r) * row_bytes;
        uint16_t* out = reply + (f * r_stride + r) * p->H;
        for (int h = 0; h < p->H; ++h) {
          float v;
          if (p->dtype == ORC_FP8) {
            v = orc_e4m3_to_float(row[h]);
            v = v * row_scales[(f * r_stride + r) * nb + h / 128];
          } else {
            uint16_t b = (uint16_t)(row[2 * h] | (row[2 * h + 1] << 8));
            v = orc_bf16_to_float(b);
          }
          v = v * c;
          out[h] = orc_float_to_bf16(v);
        }
      }
    }
}

/* "API contract": source_collect returns BF16 [T,H] summed over the selected
 * experts in original token order, the routing weight applied exactly once.
 * Design page, "19. FP8 combine replies": sum in FP32 in slot order and round
 * once to BF16. Reading used here: one FP32 accumulator per element, +0.0f
 * to start, one fused multiply-add per valid route in ascending k, one
 * round-to-nearest-even at the end; a token with no valid route gives +0
 * (design page, "13. Single-FFN collect view": such rows are zeroed). */
void orc_combine(const orc_problem* p, const int64_t* ids, const float* w,
                 const int32_t* slot, int64_t r_stride, const uint16_t* reply,
                 uint16_t* out) {
  const int Ef = p->E / p->F;
  for (int s = 0; s < p->A; ++s)
    for (int t = 0; t < p->T[s]; ++t)
      for (int h = 0; h < p->H; ++h) {
        float acc = 0.0f;
        for (int k = 0; k < p->K; ++k) {
          int64_t ri = route_index(p, s, t, k);
          if (slot[ri] < 0) continue;
          int f = (int)(ids[ri] / Ef);
          float r = orc_bf16_to_float(reply[(f * r_stride + slot[ri]) * p->H + h]);
          acc = fmaf(w[ri], r, acc);
        }
        out[((int64_t)s * p->bucket + t) * p->H + h] = orc_float_to_bf16(acc);
      }
}

/* Array forms of the format conversions, for tests that sweep many values. */
void orc_bf16_to_float_n(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_float(in[i]);
}
void orc_float_to_bf16_n(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_float_to_bf16(in[i]);
}
void orc_e4m3_to_float_n(const uint8_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_float(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Two-stage combine with optional FP8 partials                              */
/* ------------------------------------------------------------------------ */

/* E4M3 from the format definition: codes 0..7 are the subnormals m * 2^-9,
 * code (e+7)*8 + m for e in [-6, 8] is (1 + m/8) * 2^e, 0x7e = 448 is the
 * largest finite value and 0x7f is NaN. Rounding is to the nearest value,
 * ties to the even code; anything at or beyond 448 after rounding saturates
 * to 448. */
uint8_t orc_float_to_e4m3(float f) {
  if (isnan(f)) return 0x7f;
  uint8_t sign = signbit(f) ? 0x80 : 0x00;
  double a = fabs((double)f); /* exact: float -> double */
  if (a >= 448.0) return sign | 0x7e;
  int code;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9, codes 0..8 (8 = smallest normal) */
    double q = a / ldexp(1.0, -9);
    double n = floor(q);
    double r = q - n;
    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) == 1.0)) n += 1.0;
    code = (int)n;
  } else {
    int e;
    frexp(a, &e); /* a = m * 2^e with m in [0.5, 1) */
    e -= 1;       /* now a = (1 + f) * 2^e */
    double q = a / ldexp(1.0, e - 3); /* in [8, 16) */
    double n = floor(q);
    double r = q - n;
    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) == 1.0)) n += 1.0;
    if (n == 16.0) {
      n = 8.0;
      e += 1;
    }
    code = (e + 7) * 8 + ((int)n - 8);
    if (code > 0x7e) code = 0x7e; /* the NaN pattern is not a value: saturate */
  }
  return (uint8_t)(sign | code);
}

void orc_float_to_e4m3_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_float_to_e4m3(in[i]);
}

int32_t orc_group_exponent(float amax) {
  /* the page's definition, searched directly: the first e from -117 up with
   * amax <= 448 * 2^e evaluated in FP32 (2^e scales exactly; 448 * 2^121 and
   * above overflow to infinity, so an infinite amax stops at 120) */
  for (int e = -117; e <= 128; ++e)
    if (amax <= ldexpf(448.0f, e)) return e;
  return 128; /* NaN: no e satisfies the comparison */
}

void orc_group_exponent_n(const float* amax, int32_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_group_exponent(amax[i]);
}

void orc_combine_two_stage(const orc_problem* p, const int64_t* ids, const float* w,
                           const int32_t* slot, int64_t r_stride, const uint16_t* reply,
                           int32_t fp8, uint16_t* out) {
  const int Ef = p->E / p->F;
  const int H = p->H;
  float* acc = (float*)malloc(sizeof(float) * (size_t)H);
  float* part = (float*)malloc(sizeof(float) * (size_t)H);
  for (int s = 0; s < p->A; ++s)
    for (int t = 0; t < p->T[s]; ++t) {
      for (int h = 0; h < H; ++h) acc[h] = 0.0f;
      for (int k = 0; k < p->K; ++k) {
        int64_t rk = route_index(p, s, t, k);
        if (slot[rk] < 0) continue;
        int f = (int)(ids[rk] / Ef);
        /* is k this worker's last route of the token? */
        int last = 1;
        for (int j = k + 1; j < p->K; ++j) {
          int64_t rj = route_index(p, s, t, j);
          if (slot[rj] >= 0 && (int)(ids[rj] / Ef) == f) last = 0;
        }
        if (!last) continue;
        /* the worker's BF16 partial */
        for (int h = 0; h < H; ++h) {
          float a = 0.0f;
          for (int j = 0; j <= k; ++j) {
            int64_t rj = route_index(p, s, t, j);
            if (slot[rj] < 0 || (int)(ids[rj] / Ef) != f) continue;
            a = fmaf(w[rj], orc_bf16_to_float(reply[(f * r_stride + slot[rj]) * H + h]), a);
          }
          part[h] = orc_bf16_to_float(orc_float_to_bf16(a));
        }
        if (fp8) {
          for (int g = 0; g < H / 128; ++g) {
            float amax = 0.0f;
            for (int h = g * 128; h < (g + 1) * 128; ++h) amax = fmaxf(amax, fabsf(part[h]));
            int e = orc_group_exponent(amax);
            for (int h = g * 128; h < (g + 1) * 128; ++h) {
              uint8_t q = orc_float_to_e4m3(ldexpf(part[h], -e));
              part[h] = ldexpf(orc_e4m3_to_float(q), e);
            }
          }
        }
        for (int h = 0; h < H; ++h) acc[h] = acc[h] + part[h];
      }
      for (int h = 0; h < H; ++h)
        out[((int64_t)s * p->bucket + t) * H + h] = orc_float_to_bf16(acc[h]);
    }
  free(acc);
  free(part);
}
