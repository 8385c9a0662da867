/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
 * CUDA library is checked against.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.  It
 * shares no code, header, table or constant generator with the CUDA sources.
 *
 * Sources (web pages on NVFP4 KV-cache quantisation):
 *  - "nvfp4-kv-cache-memory-wall" (grer.cn blog), section 2 (two-level
 *    scaling): E2M1 data values +-{0,0.5,1,1.5,2,3,4,6}; one FP8 E4M3 scale per
 *    16 consecutive values; one FP32 scale for the whole tensor; the demo maps
 *    each block's amax onto 6 and snaps every value to the nearest E2M1 value.
 *  - same page, section 1: 16 E2M1 values pack into 8 bytes plus 1 scale byte,
 *    i.e. 9/16 byte per value.
 *  - same page, section 3 (three data flows): new K/V are quantised to NVFP4 on
 *    the way into the paged cache; decode dequantises inside the attention
 *    kernel; chunked prefill/extend dequantises the cached prefix into one FP8
 *    E4M3 workspace shared by all layers.
 *  - "NVFP4: breaking the memory wall" (cloud.tencent.com), technical
 *    breakdown: E2M1 is 1 sign, 2 exponent and 1 mantissa bit; the micro-block
 *    scale is E4M3; the tensor-level scale is FP32.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - E2M1 and E4M3 encoders round to nearest, ties to the even code, and
 *    saturate at the largest finite value (+-6, +-448).  The sign of the input
 *    is kept, so a small negative value encodes as -0.
 *  - Block scale: sb = E4M3(amax / (6*g)); value code: E2M1(x / (E4M3val(sb)*g)).
 *    Every step is one IEEE binary32 operation rounded to nearest (this file
 *    is compiled with -ffp-contract=off, so no multiply-add is fused).
 *  - If E4M3val(sb)*g is 0 the block stores signed zeros.
 *  - Blocks run along head_dim; element 2i is the low nibble of byte i.
 *  - Attention is evaluated in binary64 over the dequantised cache.
 *  - FP8 workspace: w = E4M3(fp32(fp32(e2m1*E4M3val(sb)) * g) / s_ws), signed.
 *
 * Cache layout (a proposal the pages leave open): data pages
 * [num_pages][num_kv_heads][page_size][head_dim/2] bytes, scale pages
 * [num_pages][num_kv_heads][page_size][head_dim/16] E4M3 bytes; a slot s names
 * page s / page_size, row s % page_size.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "nvfp4_oracle.h"

/* ------------------------------------------------------------------------- */
/* Formats, from their bit-field definitions.                                */
/* ------------------------------------------------------------------------- */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.  Exponent 0
 * is subnormal: value = m * 0.5.  Otherwise value = 2^(e-1) * (1 + m/2). */
double nvfp4_oracle_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E4M3 ("fn" flavour: no infinities, 0x7F/0xFF are NaN): bit 7 sign, bits
 * 6..3 exponent (bias 7), bits 2..0 mantissa.  Exponent 0 is subnormal:
 * value = m/8 * 2^-6. */
double nvfp4_oracle_e4m3_value(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp(m / 8.0, -6);
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Non-negative values of each format by code, filled once from the decoders
 * above so that the searches below are table lookups. */
static double e2m1_mag[8];
static double e4m3_mag[0x7F];
static int tables_ready = 0;

static void init_tables(void) {
  if (tables_ready) return;
  for (int c = 0; c < 8; ++c) e2m1_mag[c] = nvfp4_oracle_e2m1_value((uint8_t)c);
  for (int c = 0; c < 0x7F; ++c) e4m3_mag[c] = nvfp4_oracle_e4m3_value((uint8_t)c);
  tables_ready = 1;
}

/* Nearest-value search over the non-negative codes 0..max_code of a format
 * whose values increase with the code (value[c] for code c).  Ties pick the
 * even code (the one whose mantissa LSB, which is the code LSB, is zero).
 * Saturating: anything at or beyond the largest finite value maps to it. */
static uint8_t nearest_code(double mag, int max_code, const double* value) {
  /* at or beyond the largest finite value: saturate (distances to the
   * candidates would also lose their differences for huge inputs) */
  if (mag >= value[max_code]) return (uint8_t)max_code;
  int best = 0;
  double best_d = fabs(mag - value[0]);
  for (int c = 1; c <= max_code; ++c) {
    double d = fabs(mag - value[c]);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)best;
}

uint8_t nvfp4_oracle_e2m1_encode(float y) {
  init_tables();
  uint8_t mag = nearest_code(fabs((double)y), 7, e2m1_mag);
  return (uint8_t)(mag | (signbit(y) ? 0x8 : 0x0));
}

uint8_t nvfp4_oracle_e4m3_encode(float z) {
  init_tables();
  uint8_t mag = nearest_code(fabs((double)z), 0x7E, e4m3_mag);
  return (uint8_t)(mag | (signbit(z) ? 0x80 : 0x00));
}

/* bf16 is the top half of a binary32 bit pattern. */
float nvfp4_oracle_bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------- */
/* One 16-value block: two-level scaling.                                    */
/* ------------------------------------------------------------------------- */

void nvfp4_oracle_quantize_block(const float x[NVFP4_ORACLE_BLOCK], float g,
                                 uint8_t packed[NVFP4_ORACLE_BLOCK / 2], uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < NVFP4_ORACLE_BLOCK; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float t = 6.0f * g;          /* the block's amax lands on E2M1's largest value */
  float ratio = amax / t;
  uint8_t sb = nvfp4_oracle_e4m3_encode(ratio);
  float den = (float)nvfp4_oracle_e4m3_value(sb) * g;
  uint8_t codes[NVFP4_ORACLE_BLOCK];
  for (int i = 0; i < NVFP4_ORACLE_BLOCK; ++i) {
    if (den == 0.0f) {
      codes[i] = signbit(x[i]) ? 0x8 : 0x0;
    } else {
      float y = x[i] / den;
      codes[i] = nvfp4_oracle_e2m1_encode(y);
    }
  }
  for (int i = 0; i < NVFP4_ORACLE_BLOCK / 2; ++i)
    packed[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
  *scale = sb;
}

double nvfp4_oracle_dequant_value(uint8_t code, uint8_t scale, float g) {
  return nvfp4_oracle_e2m1_value(code) * nvfp4_oracle_e4m3_value(scale) * (double)g;
}

/* ------------------------------------------------------------------------- */
/* The page demo's arithmetic (binary64, unrounded block scale, global scale */
/* 1, ties to the first entry of the value list in ascending order).         */
/* ------------------------------------------------------------------------- */

void nvfp4_oracle_demo_fake_quant(const double* x, int64_t n, int64_t block, double* out) {
  /* the 16 E2M1 values in ascending order, -0 before +0 */
  double list[16];
  int k = 0;
  for (int c = 7; c >= 0; --c) list[k++] = nvfp4_oracle_e2m1_value((uint8_t)(c | 8));
  for (int c = 0; c <= 7; ++c) list[k++] = nvfp4_oracle_e2m1_value((uint8_t)c);
  for (int64_t b0 = 0; b0 < n; b0 += block) {
    int64_t b1 = b0 + block < n ? b0 + block : n;
    double amax = 0.0;
    for (int64_t i = b0; i < b1; ++i)
      if (fabs(x[i]) > amax) amax = fabs(x[i]);
    double scale = amax > 1e-12 ? amax / 6.0 : 1.0;
    for (int64_t i = b0; i < b1; ++i) {
      double y = x[i] / scale;
      int best = 0;
      for (int j = 1; j < 16; ++j)
        if (fabs(list[j] - y) < fabs(list[best] - y)) best = j;
      out[i] = list[best] * scale;
    }
  }
}

/* ------------------------------------------------------------------------- */
/* Paged cache: sizes and addressing.                                        */
/* ------------------------------------------------------------------------- */

int64_t nvfp4_oracle_row_bytes(int head_dim) { return head_dim / 2; }
int64_t nvfp4_oracle_row_scale_bytes(int head_dim) { return head_dim / NVFP4_ORACLE_BLOCK; }

static int64_t row_index(int64_t page, int h, int off, int num_kv_heads, int page_size) {
  return (page * num_kv_heads + h) * page_size + off;
}

/* ------------------------------------------------------------------------- */
/* Quantize-append: every new token's K and V rows into their slots.         */
/* ------------------------------------------------------------------------- */

int nvfp4_oracle_quantize_append(const nvfp4_oracle_cache* c, const uint16_t* k_bf16,
                                 const uint16_t* v_bf16, const int64_t* slot_mapping,
                                 int64_t num_tokens) {
  int bad = 0;
  const int d = c->head_dim, H = c->num_kv_heads, P = c->page_size;
  const int64_t rb = nvfp4_oracle_row_bytes(d), sbk = nvfp4_oracle_row_scale_bytes(d);
  float x[NVFP4_ORACLE_BLOCK];
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;                      /* padding token */
    if (s >= c->num_pages * P) { bad = 1; continue; }
    int64_t page = s / P;
    int off = (int)(s % P);
    for (int h = 0; h < H; ++h) {
      int64_t r = row_index(page, h, off, H, P);
      for (int which = 0; which < 2; ++which) {
        const uint16_t* src = (which == 0 ? k_bf16 : v_bf16) + (t * H + h) * d;
        uint8_t* data = (which == 0 ? c->k_data : c->v_data) + r * rb;
        uint8_t* scl = (which == 0 ? c->k_scale : c->v_scale) + r * sbk;
        float g = which == 0 ? c->k_global_scale : c->v_global_scale;
        for (int j = 0; j < d / NVFP4_ORACLE_BLOCK; ++j) {
          for (int i = 0; i < NVFP4_ORACLE_BLOCK; ++i)
            x[i] = nvfp4_oracle_bf16_to_float(src[j * NVFP4_ORACLE_BLOCK + i]);
          nvfp4_oracle_quantize_block(x, g, data + j * (NVFP4_ORACLE_BLOCK / 2), scl + j);
        }
      }
    }
  }
  return bad;
}

/* Value tables built once per call from the format definitions above (the
 * same numbers nvfp4_oracle_e2m1_value / nvfp4_oracle_e4m3_value return). */
typedef struct {
  double e2m1[16];
  double e4m3[256];
} value_tables;

static void build_tables(value_tables* vt) {
  for (int c = 0; c < 16; ++c) vt->e2m1[c] = nvfp4_oracle_e2m1_value((uint8_t)c);
  for (int c = 0; c < 256; ++c) vt->e4m3[c] = nvfp4_oracle_e4m3_value((uint8_t)c);
}

/* Dequantised row (all head_dim elements) of the cached (page, kv head, row). */
static void cached_row(const nvfp4_oracle_cache* c, const value_tables* vt, int which, int64_t page,
                       int h, int off, double* dst) {
  const int d = c->head_dim;
  int64_t r = row_index(page, h, off, c->num_kv_heads, c->page_size);
  const uint8_t* data = (which == 0 ? c->k_data : c->v_data) + r * nvfp4_oracle_row_bytes(d);
  const uint8_t* scl = (which == 0 ? c->k_scale : c->v_scale) + r * nvfp4_oracle_row_scale_bytes(d);
  double g = (double)(which == 0 ? c->k_global_scale : c->v_global_scale);
  for (int dd = 0; dd < d; ++dd) {
    uint8_t byte = data[dd / 2];
    uint8_t code = (dd & 1) ? (byte >> 4) : (byte & 0xF);
    dst[dd] = vt->e2m1[code] * vt->e4m3[scl[dd / NVFP4_ORACLE_BLOCK]] * g;
  }
}

/* ------------------------------------------------------------------------- */
/* Decode attention: one query token per sequence, softmax over all cached   */
/* tokens of that sequence, GQA (query head h reads KV head h / G).  Query   */
/* heads [head_begin, head_end) are computed; other rows of out are left as  */
/* they are.                                                                 */
/* ------------------------------------------------------------------------- */

int nvfp4_oracle_decode_attention_heads(const nvfp4_oracle_cache* c, const uint16_t* q_bf16,
                                        const int32_t* page_table, int32_t max_pages,
                                        const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                        double softmax_scale, int32_t head_begin, int32_t head_end,
                                        double* out) {
  const int d = c->head_dim, H = c->num_kv_heads, P = c->page_size;
  int bad = 0;
  if (d > 512 || d % NVFP4_ORACLE_BLOCK != 0 || H <= 0 || num_q_heads % H != 0) return -1;
  const int G = num_q_heads / H;
  value_tables vt;
  build_tables(&vt);
  double row[512];
  for (int32_t b = 0; b < batch; ++b) {
    int64_t L = seq_lens[b];
    if (L < 0 || L > (int64_t)max_pages * P) { bad = 1; L = L < 0 ? 0 : (int64_t)max_pages * P; }
    for (int hq = head_begin; hq < head_end; ++hq) {
      double* o = out + ((int64_t)b * num_q_heads + hq) * d;
      for (int dd = 0; dd < d; ++dd) o[dd] = 0.0;
      if (L == 0) continue;
      const int hk = hq / G;
      double q[512];
      for (int dd = 0; dd < d; ++dd)
        q[dd] = nvfp4_oracle_bf16_to_float(q_bf16[((int64_t)b * num_q_heads + hq) * d + dd]);
      double* s = (double*)malloc(sizeof(double) * (size_t)L);
      int* valid = (int*)malloc(sizeof(int) * (size_t)L);
      double m = -INFINITY;
      for (int64_t t = 0; t < L; ++t) {
        int32_t page = page_table[(int64_t)b * max_pages + t / P];
        valid[t] = page >= 0 && page < c->num_pages;
        if (!valid[t]) { bad = 1; continue; }
        cached_row(c, &vt, 0, page, hk, (int)(t % P), row);
        double acc = 0.0;
        for (int dd = 0; dd < d; ++dd) acc += q[dd] * row[dd];
        s[t] = softmax_scale * acc;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int64_t t = 0; t < L; ++t) {
        if (!valid[t]) continue;
        double w = exp(s[t] - m);
        l += w;
        int32_t page = page_table[(int64_t)b * max_pages + t / P];
        cached_row(c, &vt, 1, page, hk, (int)(t % P), row);
        for (int dd = 0; dd < d; ++dd) o[dd] += w * row[dd];
      }
      if (l > 0.0)
        for (int dd = 0; dd < d; ++dd) o[dd] /= l;
      free(s);
      free(valid);
    }
  }
  return bad;
}

int nvfp4_oracle_decode_attention(const nvfp4_oracle_cache* c, const uint16_t* q_bf16,
                                  const int32_t* page_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                  double softmax_scale, double* out) {
  return nvfp4_oracle_decode_attention_heads(c, q_bf16, page_table, max_pages, seq_lens, batch,
                                             num_q_heads, softmax_scale, 0, num_q_heads, out);
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 workspace for chunked prefill / extend.                          */
/* ------------------------------------------------------------------------- */

int nvfp4_oracle_dequant_to_fp8_workspace(const nvfp4_oracle_cache* c, const int32_t* page_table,
                                          int32_t max_pages, const int32_t* prefix_lens,
                                          const int64_t* cu_prefix, int32_t batch,
                                          float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                          uint8_t* ws_v) {
  const int d = c->head_dim, H = c->num_kv_heads, P = c->page_size;
  int bad = 0;
  for (int32_t b = 0; b < batch; ++b) {
    int64_t L = prefix_lens[b];
    if (L < 0 || L > (int64_t)max_pages * P) { bad = 1; L = L < 0 ? 0 : (int64_t)max_pages * P; }
    for (int64_t t = 0; t < L; ++t) {
      int64_t row = cu_prefix[b] + t;
      int32_t page = page_table[(int64_t)b * max_pages + t / P];
      int ok = page >= 0 && page < c->num_pages;
      if (!ok) bad = 1;
      for (int h = 0; h < H; ++h) {
        for (int which = 0; which < 2; ++which) {
          uint8_t* w = (which == 0 ? ws_k : ws_v) + (row * H + h) * d;
          float g = which == 0 ? c->k_global_scale : c->v_global_scale;
          float sws = which == 0 ? k_ws_scale : v_ws_scale;
          for (int dd = 0; dd < d; ++dd) {
            if (!ok) { w[dd] = 0; continue; }
            int64_t r = row_index(page, h, (int)(t % P), H, P);
            const uint8_t* data = (which == 0 ? c->k_data : c->v_data) + r * nvfp4_oracle_row_bytes(d);
            const uint8_t* scl =
                (which == 0 ? c->k_scale : c->v_scale) + r * nvfp4_oracle_row_scale_bytes(d);
            uint8_t byte = data[dd / 2];
            uint8_t code = (dd & 1) ? (byte >> 4) : (byte & 0xF);
            float v = (float)(nvfp4_oracle_e2m1_value(code) *
                              nvfp4_oracle_e4m3_value(scl[dd / NVFP4_ORACLE_BLOCK]));
            float vg = v * g;
            float z = vg / sws;
            w[dd] = nvfp4_oracle_e4m3_encode(z);
          }
        }
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Decode attention over a cache written by a format variant (the decode side */
/* of the comparison the pages draw between NVFP4 and its variants).          */
/*   format 0: NVFP4, as nvfp4_oracle_decode_attention;                       */
/*   format 1: NVFP4 of Hadamard-rotated rows: each dequantised row is        */
/*             rotated back (the orthonormal transform is its own inverse;    */
/*             binary64 butterflies) before the attention;                    */
/*   format 2: MXFP4: head_dim/32 E8M0 scale bytes per row, value =           */
/*             E2M1(code) * 2^(scale - 127); the global scales are not used.   */
/* ------------------------------------------------------------------------- */

static void variant_row(const nvfp4_oracle_cache* c, const value_tables* vt, int format, int which,
                        int64_t page, int h, int off, double* dst) {
  const int d = c->head_dim;
  if (format == 2) {
    const int64_t r = row_index(page, h, off, c->num_kv_heads, c->page_size);
    const uint8_t* data = (which == 0 ? c->k_data : c->v_data) + r * nvfp4_oracle_row_bytes(d);
    const uint8_t* scl = (which == 0 ? c->k_scale : c->v_scale) + r * (d / 32);
    for (int dd = 0; dd < d; ++dd) {
      const uint8_t byte = data[dd / 2];
      const uint8_t code = (dd & 1) ? (byte >> 4) : (byte & 0xF);
      dst[dd] = vt->e2m1[code] * nvfp4_oracle_e8m0_value(scl[dd / 32]);
    }
    return;
  }
  cached_row(c, vt, which, page, h, off, dst);
  if (format == 1) {
    for (int hh = 1; hh < d; hh *= 2)
      for (int i = 0; i < d; i += 2 * hh)
        for (int j = i; j < i + hh; ++j) {
          const double a = dst[j], b = dst[j + hh];
          dst[j] = a + b;
          dst[j + hh] = a - b;
        }
    const double sc = 1.0 / sqrt((double)d);
    for (int dd = 0; dd < d; ++dd) dst[dd] *= sc;
  }
}

int nvfp4_oracle_decode_attention_format(const nvfp4_oracle_cache* c, int format, const uint16_t* q_bf16,
                                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                                         int32_t batch, int32_t num_q_heads, double softmax_scale, double* out) {
  const int d = c->head_dim, H = c->num_kv_heads, P = c->page_size;
  if (format < 0 || format > 2 || d > 512 || d % 32 != 0 || (d & (d - 1)) != 0 || H <= 0 ||
      num_q_heads % H != 0)
    return -1;
  const int G = num_q_heads / H;
  int bad = 0;
  value_tables vt;
  build_tables(&vt);
  double row[512];
  for (int32_t b = 0; b < batch; ++b) {
    int64_t L = seq_lens[b];
    if (L < 0 || L > (int64_t)max_pages * P) { bad = 1; L = L < 0 ? 0 : (int64_t)max_pages * P; }
    for (int hq = 0; hq < num_q_heads; ++hq) {
      double* o = out + ((int64_t)b * num_q_heads + hq) * d;
      for (int dd = 0; dd < d; ++dd) o[dd] = 0.0;
      if (L == 0) continue;
      const int hk = hq / G;
      double q[512];
      for (int dd = 0; dd < d; ++dd)
        q[dd] = nvfp4_oracle_bf16_to_float(q_bf16[((int64_t)b * num_q_heads + hq) * d + dd]);
      double* s = (double*)malloc(sizeof(double) * (size_t)L);
      int* valid = (int*)malloc(sizeof(int) * (size_t)L);
      double m = -INFINITY;
      for (int64_t t = 0; t < L; ++t) {
        const int32_t page = page_table[(int64_t)b * max_pages + t / P];
        valid[t] = page >= 0 && page < c->num_pages;
        if (!valid[t]) { bad = 1; continue; }
        variant_row(c, &vt, format, 0, page, hk, (int)(t % P), row);
        double acc = 0.0;
        for (int dd = 0; dd < d; ++dd) acc += q[dd] * row[dd];
        s[t] = softmax_scale * acc;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int64_t t = 0; t < L; ++t) {
        if (!valid[t]) continue;
        const double w = exp(s[t] - m);
        l += w;
        const int32_t page = page_table[(int64_t)b * max_pages + t / P];
        variant_row(c, &vt, format, 1, page, hk, (int)(t % P), row);
        for (int dd = 0; dd < d; ++dd) o[dd] += w * row[dd];
      }
      if (l > 0.0)
        for (int dd = 0; dd < d; ++dd) o[dd] /= l;
      free(s);
      free(valid);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Extend (chunked prefill) over the FP8 workspace ("nvfp4-kv-cache-memory-  */
/* wall", section 3, item 2 and the data-flow figure: the chunk attends over */
/* its cached prefix, dequantised into the FP8 workspace, and over itself;   */
/* the current tokens' own K/V take part as FP8).                            */
/*                                                                           */
/* Readings: the chunk's K/V rows enter the workspace straight from bf16,    */
/* w = E4M3(fp32(x) / s_ws) with the sign kept; sequence b's rows are        */
/* cu_prefix[b] + j for its key j, the prefix (j < prefix_lens[b]) first and */
/* chunk token t at j = prefix_lens[b] + t; token t sees keys 0 .. P_b + t   */
/* (causal).  Attention is evaluated in binary64 over E4M3val(w) * s_ws.     */
/* ------------------------------------------------------------------------- */

int nvfp4_oracle_bf16_to_fp8_workspace(const uint16_t* k_bf16, const uint16_t* v_bf16,
                                       const int64_t* ws_rows, int64_t num_tokens,
                                       int32_t num_kv_heads, int32_t head_dim, int64_t total_rows,
                                       float k_ws_scale, float v_ws_scale, uint8_t* ws_k,
                                       uint8_t* ws_v) {
  const int64_t row_vals = (int64_t)num_kv_heads * head_dim;
  int bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t row = ws_rows[t];
    if (row < 0) continue; /* padding */
    if (row >= total_rows) { bad = 1; continue; }
    for (int which = 0; which < 2; ++which) {
      const uint16_t* x = (which == 0 ? k_bf16 : v_bf16) + t * row_vals;
      uint8_t* w = (which == 0 ? ws_k : ws_v) + row * row_vals;
      const float sws = which == 0 ? k_ws_scale : v_ws_scale;
      for (int64_t i = 0; i < row_vals; ++i) {
        const float z = nvfp4_oracle_bf16_to_float(x[i]) / sws;
        w[i] = nvfp4_oracle_e4m3_encode(z);
      }
    }
  }
  return bad;
}

/* The sequence holding global query token i (cu_q non-decreasing), or -1. */
static int32_t sequence_of(const int64_t* cu_q, int32_t batch, int64_t i) {
  for (int32_t b = 0; b < batch; ++b)
    if (i >= cu_q[b] && i < cu_q[b + 1]) return b;
  return -1;
}

int nvfp4_oracle_extend_attention_rows(const uint8_t* ws_k, const uint8_t* ws_v, int64_t total_rows,
                                       int32_t num_kv_heads, int32_t head_dim, float k_ws_scale,
                                       float v_ws_scale, const uint16_t* q_bf16, int32_t num_q_heads,
                                       const int64_t* cu_q, const int64_t* cu_prefix,
                                       const int32_t* prefix_lens, int32_t batch,
                                       double softmax_scale, const int64_t* pairs, int64_t num_pairs,
                                       double* out) {
  const int d = head_dim, H = num_kv_heads;
  if (d > 512 || H <= 0 || num_q_heads % H != 0) return -1;
  const int G = num_q_heads / H;
  int bad = 0;
  value_tables vt;
  build_tables(&vt);
  for (int64_t n = 0; n < num_pairs; ++n) {
    const int64_t i = pairs[2 * n];
    const int hq = (int)pairs[2 * n + 1];
    double* o = out + n * d;
    for (int dd = 0; dd < d; ++dd) o[dd] = 0.0;
    const int32_t b = sequence_of(cu_q, batch, i);
    if (b < 0 || hq < 0 || hq >= num_q_heads) { bad = 1; continue; }
    const int64_t t = i - cu_q[b];
    const int64_t L = (int64_t)prefix_lens[b] + t + 1; /* keys 0 .. P_b + t */
    const int hk = hq / G;
    double q[512];
    for (int dd = 0; dd < d; ++dd)
      q[dd] = nvfp4_oracle_bf16_to_float(q_bf16[(i * num_q_heads + hq) * d + dd]);
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    double m = -INFINITY;
    int ok = 1;
    for (int64_t j = 0; j < L; ++j) {
      const int64_t row = cu_prefix[b] + j;
      if (row < 0 || row >= total_rows) { ok = 0; break; }
      const uint8_t* kr = ws_k + (row * H + hk) * d;
      double acc = 0.0;
      for (int dd = 0; dd < d; ++dd)
        acc += q[dd] * (vt.e4m3[kr[dd]] * (double)k_ws_scale);
      s[j] = softmax_scale * acc;
      if (s[j] > m) m = s[j];
    }
    if (!ok) { bad = 1; free(s); continue; }
    double l = 0.0;
    for (int64_t j = 0; j < L; ++j) {
      const double w = exp(s[j] - m);
      l += w;
      const uint8_t* vr = ws_v + ((cu_prefix[b] + j) * H + hk) * d;
      for (int dd = 0; dd < d; ++dd) o[dd] += w * (vt.e4m3[vr[dd]] * (double)v_ws_scale);
    }
    for (int dd = 0; dd < d; ++dd) o[dd] /= l;
    free(s);
  }
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Format variants the pages compare with NVFP4.                             */
/* ------------------------------------------------------------------------- */

/* MXFP4 ("NVIDIA NVFP4: LLM memory doubled, inference 3x" (nmedialink),
 * figure 6 and its text: NVFP4's finer blocks and more precise E4M3 scale beat
 * MXFP4; "NVFP4: breaking the memory wall" (cloud.tencent.com), technical
 * breakdown: MXFP4 shares one scale among 32 values, NVFP4 among 16).
 * Reading: the public microscaling layout -- a power-of-two scale stored as an
 * E8M0 byte (exponent + 127), X = 2^(floor(log2 amax) - 2), 2 being E2M1's
 * largest exponent; elements E2M1(x / X), nearest even, saturating; an all-zero
 * block takes the smallest scale, 2^-127. */
double nvfp4_oracle_e8m0_value(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

void nvfp4_oracle_mxfp4_quantize_block(const float x[32], uint8_t packed[16], uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  int e = -127;
  if (amax > 0.0f) {
    int ex;
    frexpf(amax, &ex); /* amax = m * 2^ex with m in [0.5, 1): floor(log2 amax) = ex - 1 */
    e = ex - 1 - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  *scale = (uint8_t)(e + 127);
  for (int i = 0; i < 16; ++i) {
    /* division by a power of two: exact unless the quotient is subnormal */
    const uint8_t lo = nvfp4_oracle_e2m1_encode((float)((double)x[2 * i] / ldexp(1.0, e)));
    const uint8_t hi = nvfp4_oracle_e2m1_encode((float)((double)x[2 * i + 1] / ldexp(1.0, e)));
    packed[i] = (uint8_t)(lo | (hi << 4));
  }
}

double nvfp4_oracle_mxfp4_dequant_value(uint8_t code, uint8_t scale) {
  return nvfp4_oracle_e2m1_value(code) * nvfp4_oracle_e8m0_value(scale);
}

/* Stochastic rounding ("NVFP4: breaking the memory wall" (cloud.tencent.com),
 * the quantisation techniques and the two engineering tricks: a value between
 * two grid points goes up with probability equal to its distance past the
 * lower point, 2.3 -> 2 with 70 %, -> 3 with 30 %, so the errors cancel on
 * average).  Reading: applied to the E2M1 element codes (the block scale stays
 * nearest-even); the random number is an input byte r, read as the uniform
 * (r + 0.5) / 256: |y| rounds up iff (r + 0.5) / 256 < (|y| - a) / (b - a) for
 * the grid neighbours a <= |y| < b.  Every E2M1 gap is a power of two, so that
 * fraction is exact in binary32 and so is the decision.  Sign kept; |y| >= 6
 * gives 6. */
uint8_t nvfp4_oracle_e2m1_encode_sr(float y, uint8_t r) {
  init_tables();
  const float m = fabsf(y);
  uint8_t code;
  if (m >= 6.0f) {
    code = 7;
  } else {
    int c = 0; /* largest code with value <= m */
    while (c < 7 && e2m1_mag[c + 1] <= (double)m) ++c;
    const double a = e2m1_mag[c], b = e2m1_mag[c + 1];
    const double frac = ((double)m - a) / (b - a); /* exact: the gap is a power of two */
    code = (uint8_t)(((double)r + 0.5) / 256.0 < frac ? c + 1 : c);
  }
  return (uint8_t)(code | (signbit(y) ? 0x8 : 0x0));
}

void nvfp4_oracle_quantize_block_sr(const float x[NVFP4_ORACLE_BLOCK], float g, const uint8_t r[NVFP4_ORACLE_BLOCK],
                                    uint8_t packed[NVFP4_ORACLE_BLOCK / 2], uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < NVFP4_ORACLE_BLOCK; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  const float t = 6.0f * g;
  const uint8_t sb = nvfp4_oracle_e4m3_encode(amax / t);
  const float den = (float)nvfp4_oracle_e4m3_value(sb) * g;
  *scale = sb;
  for (int i = 0; i < NVFP4_ORACLE_BLOCK / 2; ++i) {
    uint8_t c[2];
    for (int h = 0; h < 2; ++h) {
      const float xv = x[2 * i + h];
      if (den == 0.0f)
        c[h] = (uint8_t)(signbit(xv) ? 0x8 : 0x0);
      else
        c[h] = nvfp4_oracle_e2m1_encode_sr(xv / den, r[2 * i + h]);
    }
    packed[i] = (uint8_t)(c[0] | (c[1] << 4));
  }
}

/* Hadamard rotation before quantisation (the same page, same two passages: an
 * orthogonal transform spreads a local outlier over the whole vector; its
 * worked numbers are garbled and not used).  Reading: the
 * orthonormal Walsh-Hadamard transform of order n (a power of two; the head
 * vector, n = 128), Sylvester ordering (H_2n = [[H_n, H_n], [H_n, -H_n]]),
 * evaluated in binary32 as log2(n) butterfly passes y_j, y_(j+h) <- y_j + y_(j+h),
 * y_j - y_(j+h) for h = 1, 2, 4, ... followed by one multiplication by
 * RN(1 / sqrt(n)).  The transform is its own inverse. */
int nvfp4_oracle_hadamard(const float* x, int n, float* y) {
  if (n <= 0 || (n & (n - 1)) != 0) return -1;
  for (int i = 0; i < n; ++i) y[i] = x[i];
  for (int h = 1; h < n; h *= 2)
    for (int i = 0; i < n; i += 2 * h)
      for (int j = i; j < i + h; ++j) {
        const float a = y[j], b = y[j + h];
        y[j] = a + b;
        y[j + h] = a - b;
      }
  const float c = (float)(1.0 / sqrt((double)n));
  for (int i = 0; i < n; ++i) y[i] = y[i] * c;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Global-scale calibration ("nvfp4-kv-cache-memory-wall", section 2: the FP32
 * per-tensor scale is left at 1 by the uncalibrated public setting, and a
 * calibrated one reduces overflow and underflow of the two-level range; the
 * calibrated value maps the tensor's largest magnitude onto 6 x 448).        */

float nvfp4_oracle_tensor_amax(const uint16_t* x_bf16, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    const float a = fabsf(nvfp4_oracle_bf16_to_float(x_bf16[i]));
    if (a > m) m = a;
  }
  return m;
}

float nvfp4_oracle_calibrated_global_scale(float amax) {
  const float top = 6.0f * 448.0f; /* 2688, exact */
  if (amax == 0.0f) return 1.0f;
  return amax / top;
}
