/*
 * moe_oracle.c -- plain, slow CPU reference ("the oracle") for the forward pass of a
 * mixture-of-experts layer whose expert weights are stored quantized.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU-baseline
 * leg of bench.py may load this library.  It shares no code with the CUDA library
 * (nvfp4_expert_gemms_gb300/csrc) and includes none of its headers.
 *
 * Arithmetic rules: every quantizer step is one IEEE fp32 operation rounded to nearest
 * even (compiled with -ffp-contract=off, no fast-math); dot products and the layer
 * itself accumulate in fp64.
 *
 * Sources (model-card pages; the citation names the page and its section):
 *   [fp8]   clef-omni-fp8, "What was quantized" and "Recipe": E4M3 weights, one FP32 scale
 *           per 128x128 block, scale = 448/amax per tile, round-to-nearest cast, stored as
 *           weight + weight_scale_inv.
 *   [int4]  clef-omni-int4, "What was quantized" and the page header: INT4, group size 128,
 *           symmetric, auto_gptq packing (8 codes per int32 along K).
 *   [nvfp4] clef-omni-NVFP4, "How it was made": E2M1 codes two per byte, one E4M3 scale per
 *           16 weights, one fp32 global scale 448*6/amax per expert matrix (gate+up fused as
 *           one matrix), codes rounded to the nearest FP4 value with ties to even, scales from
 *           the plain block maxima.
 *   [w4a4]  clef-flash-NVFP4-Hybrid, layer table: NVFP4 for weights and activations, an E4M3
 *           scale per 16 elements and one fp32 global scale; here computed at run time per
 *           activation row.
 *   [bf16]  clef-omni-fp8, "Which Clef-Omni quant should I use?": the BF16 original is the
 *           reference every quant is compared with; its weights are used as stored.
 *   [w8a8]  clef-omni-fp8, "What was quantized": the same FP8 block weights with activations
 *           quantized to FP8 at run time, one scale per 1x128 group of a row.
 *
 * Readings where the pages are silent:
 *   - E4M3 is the OCP "e4m3fn" variant (max 448, no infinities); encode saturates at 448.
 *   - E2M1 and E4M3 encodes keep the sign of a negative value that rounds to zero.
 *   - A zero tile / matrix / row amax is clamped to 1e-12 before dividing.
 *   - INT4 rounds w / fp16(amax/7) with rint (RNE) -- AutoRound's tuned rounding needs
 *     calibration data and is replaced by round-to-nearest.
 *   - NVFP4 stores the quantize multiplier gs = 2688/amax and dequantizes by dividing.
 *   - Top-k keeps the k largest logits (ties to the lower expert index) and renormalises
 *     the softmax over them; permuted rows are ordered by (expert, token, slot).
 *   - W4A4 quantizes each activation row with its own global scale 2688/amax(row); the
 *     gated intermediate h is rounded to bf16 first and quantized the same way.
 *   - W8A8 quantizes each 1x128 activation group with the [fp8] weight recipe applied to that
 *     group (s = 448/amax, E4M3 round-to-nearest, 1/s stored); h is rounded to bf16 first and
 *     quantized the same way.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_FP8 = 1, ORC_INT4 = 2, ORC_NVFP4_W4A16 = 3, ORC_NVFP4_W4A4 = 4, ORC_BF16 = 5, ORC_FP8_W8A8 = 6 };

/* ------------------------------------------------------------------------------------ */
/* Scalar formats: a sign-magnitude minifloat with `mbits` mantissa bits and exponent   */
/* bias `bias`, with subnormals and no infinities.  E4M3 = (3, 7), E2M1 = (1, 1),       */
/* fp16 = (10, 15), bf16 = (7, 127).                                                    */
/* ------------------------------------------------------------------------------------ */

static double mf_value(unsigned mag, int mbits, int bias) {
  unsigned e = mag >> mbits, m = mag & ((1u << mbits) - 1u);
  if (e == 0) return ldexp((double)m, 1 - bias - mbits);
  return ldexp((double)((1u << mbits) | m), (int)e - bias - mbits);
}

/* Nearest representable magnitude to a >= 0, ties to the even code, saturating at max_mag. */
static unsigned mf_encode_mag(double a, int mbits, int bias, unsigned max_mag) {
  if (!(a > 0.0)) return 0;
  int E;
  frexp(a, &E);              /* a = f * 2^E, f in [0.5, 1): unbiased exponent E-1 */
  int ue = E - 1;
  if (ue < 1 - bias) ue = 1 - bias;   /* subnormal binade shares the smallest normal spacing */
  double step = ldexp(1.0, ue - mbits);
  double q = nearbyint(a / step);     /* exact power-of-two scaling, then round half even */
  if (q >= (double)(2u << mbits)) { ue += 1; q = (double)(1u << mbits); }
  unsigned long long code;
  if (q < (double)(1u << mbits)) code = (unsigned long long)q;
  else code = ((unsigned long long)(ue + bias) << mbits) | ((unsigned long long)q - (1u << mbits));
  if (code > max_mag) code = max_mag;
  return (unsigned)code;
}

static unsigned mf_encode(double v, int ebits, int mbits, int bias, unsigned max_mag) {
  unsigned mag = mf_encode_mag(fabs(v), mbits, bias, max_mag);
  return (signbit(v) ? (1u << (ebits + mbits)) : 0u) | mag;
}

static double mf_decode(unsigned code, int ebits, int mbits, int bias) {
  unsigned mag = code & ((1u << (ebits + mbits)) - 1u);
  double v = mf_value(mag, mbits, bias);
  return (code >> (ebits + mbits)) & 1u ? -v : v;
}

/* E4M3 (OCP e4m3fn): codes 0x7F / 0xFF are NaN. */
double orc_e4m3_decode(uint8_t c) {
  if ((c & 0x7F) == 0x7F) return NAN;
  return mf_decode(c, 4, 3, 7);
}
uint8_t orc_e4m3_encode(float v) { return (uint8_t)mf_encode(v, 4, 3, 7, 0x7E); }

/* E2M1: magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign. */
double orc_e2m1_decode(uint8_t c) { return mf_decode(c & 0xF, 2, 1, 1); }
uint8_t orc_e2m1_encode(float v) { return (uint8_t)mf_encode(v, 2, 1, 1, 0x7); }

/* IEEE binary16 and bfloat16 (round to nearest even from any double). */
uint16_t orc_f16_encode(double v) { return (uint16_t)mf_encode(v, 5, 10, 15, 0x7BFF); }
double orc_f16_decode(uint16_t h) { return mf_decode(h, 5, 10, 15); }
uint16_t orc_bf16_encode(double v) { return (uint16_t)mf_encode(v, 8, 7, 127, 0x7F7F); }
static float bf16f(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------------------ */
/* Weight quantizers.  W is [N, K] bf16 bits in torch Linear orientation ([out, in]).   */
/* ------------------------------------------------------------------------------------ */

/* [fp8]: per 128x128 tile, s = 448/amax, code = E4M3(w*s), store 1/s.
   codes [N, K]; scale_inv [N/128, K/128]. */
void orc_pack_fp8(const uint16_t* w, int N, int K, uint8_t* codes, float* scale_inv) {
  for (int tn = 0; tn < N / 128; ++tn)
    for (int tk = 0; tk < K / 128; ++tk) {
      float amax = 0.0f;
      for (int r = 0; r < 128; ++r)
        for (int c = 0; c < 128; ++c) {
          float a = fabsf(bf16f(w[(size_t)(tn * 128 + r) * K + tk * 128 + c]));
          if (a > amax) amax = a;
        }
      if (amax < 1e-12f) amax = 1e-12f;
      float s = 448.0f / amax;
      for (int r = 0; r < 128; ++r)
        for (int c = 0; c < 128; ++c) {
          size_t i = (size_t)(tn * 128 + r) * K + tk * 128 + c;
          float v = bf16f(w[i]) * s;
          codes[i] = orc_e4m3_encode(v);
        }
      scale_inv[tn * (K / 128) + tk] = 1.0f / s;
    }
}

void orc_dequant_fp8(const uint8_t* codes, const float* scale_inv, int N, int K, float* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      size_t i = (size_t)n * K + k;
      float c = (float)orc_e4m3_decode(codes[i]);
      out[i] = c * scale_inv[(n / 128) * (K / 128) + k / 128];
    }
}

/* [int4]: per output row n and K-group g of 128: s16 = fp16(amax/7),
   q = clamp(rint(w / s16), -8, 7), code = q + 8.
   auto_gptq packing: qweight [K/8, N] int32, nibble j of word (kr, n) holds k = 8*kr + j.
   scales [K/128, N] fp16 bits. */
void orc_pack_int4(const uint16_t* w, int N, int K, int32_t* qweight, uint16_t* scales) {
  memset(qweight, 0, sizeof(int32_t) * (size_t)(K / 8) * N);
  for (int n = 0; n < N; ++n)
    for (int g = 0; g < K / 128; ++g) {
      float amax = 0.0f;
      for (int c = 0; c < 128; ++c) {
        float a = fabsf(bf16f(w[(size_t)n * K + g * 128 + c]));
        if (a > amax) amax = a;
      }
      float s = amax / 7.0f;
      uint16_t s16 = orc_f16_encode(s);
      float sf = (float)orc_f16_decode(s16);
      scales[(size_t)g * N + n] = s16;
      for (int c = 0; c < 128; ++c) {
        int k = g * 128 + c;
        int code = 8;
        if (sf != 0.0f) {
          float qf = rintf(bf16f(w[(size_t)n * K + k]) / sf);
          if (qf < -8.0f) qf = -8.0f;
          if (qf > 7.0f) qf = 7.0f;
          code = (int)qf + 8;
        }
        uint32_t* word = (uint32_t*)&qweight[(size_t)(k / 8) * N + n];
        *word |= (uint32_t)code << (4 * (k % 8));
      }
    }
}

void orc_dequant_int4(const int32_t* qweight, const uint16_t* scales, int N, int K, float* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      uint32_t word = (uint32_t)qweight[(size_t)(k / 8) * N + n];
      int code = (int)((word >> (4 * (k % 8))) & 0xF);
      float sf = (float)orc_f16_decode(scales[(size_t)(k / 128) * N + n]);
      out[(size_t)n * K + k] = (float)(code - 8) * sf;
    }
}

/* One NVFP4 block-scaled row segment with a given global scale gs ([nvfp4]):
   bs = E4M3((amax_b/6)*gs); eff = bs/gs; q = E2M1(w/eff) (q = 0 when bs == 0). */
static void nvfp4_row(const float* v, int K, float gs, uint8_t* packed_row, uint8_t* scale_row) {
  for (int b = 0; b < K / 16; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(v[b * 16 + i]);
      if (a > amax) amax = a;
    }
    float t = amax / 6.0f;
    float t2 = t * gs;
    uint8_t bsc = orc_e4m3_encode(t2);
    float bs = (float)orc_e4m3_decode(bsc);
    scale_row[b] = bsc;
    for (int i = 0; i < 16; ++i) {
      uint8_t q = 0;
      if (bs != 0.0f) {
        float eff = bs / gs;
        q = orc_e2m1_encode(v[b * 16 + i] / eff);
      }
      int k = b * 16 + i;
      if ((k & 1) == 0) packed_row[k / 2] = q;
      else packed_row[k / 2] |= (uint8_t)(q << 4);
    }
  }
}

/* [nvfp4]: one global scale per matrix, gs = 2688/amax(W).
   weight_packed [N, K/2] (element 2i in the low nibble), weight_scale [N, K/16] E4M3 codes. */
void orc_pack_nvfp4(const uint16_t* w, int N, int K, uint8_t* packed, uint8_t* scales, float* gs_out) {
  float amax = 0.0f;
  for (size_t i = 0; i < (size_t)N * K; ++i) {
    float a = fabsf(bf16f(w[i]));
    if (a > amax) amax = a;
  }
  if (amax < 1e-12f) amax = 1e-12f;
  float gs = 2688.0f / amax;
  *gs_out = gs;
  float* row = (float*)malloc(sizeof(float) * K);
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < K; ++k) row[k] = bf16f(w[(size_t)n * K + k]);
    nvfp4_row(row, K, gs, packed + (size_t)n * (K / 2), scales + (size_t)n * (K / 16));
  }
  free(row);
}

/* value = (E2M1(q) * E4M3(bs)) / gs, one fp32 rounding. */
void orc_dequant_nvfp4(const uint8_t* packed, const uint8_t* scales, float gs, int N, int K, float* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      uint8_t byte = packed[(size_t)n * (K / 2) + k / 2];
      uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
      float bs = (float)orc_e4m3_decode(scales[(size_t)n * (K / 16) + k / 16]);
      float p = (float)orc_e2m1_decode(q) * bs;
      out[(size_t)n * K + k] = p / gs;
    }
}

/* [w4a4], dynamic: each row of a [T, H] bf16 activation gets gs_t = 2688/max(amax_t, 1e-12)
   and is block-quantized like a weight row.  codes [T, H/2], scales [T, H/16], gs [T]. */
/* The same with one static global scale gs for every row (calibrated ahead of time; the
   clef-flash-NVFP4-Hybrid layer table calibrates the activations' global scales): block scales
   saturate at 448 and codes at 6 where a block exceeds the calibrated range. */
void orc_quant_act_nvfp4_static(const uint16_t* x, int T, int H, float gs, uint8_t* codes, uint8_t* scales) {
  float* row = (float*)malloc(sizeof(float) * H);
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < H; ++k) row[k] = bf16f(x[(size_t)t * H + k]);
    nvfp4_row(row, H, gs, codes + (size_t)t * (H / 2), scales + (size_t)t * (H / 16));
  }
  free(row);
}

void orc_quant_act_nvfp4(const uint16_t* x, int T, int H, uint8_t* codes, uint8_t* scales, float* gs) {
  float* row = (float*)malloc(sizeof(float) * H);
  for (int t = 0; t < T; ++t) {
    float amax = 0.0f;
    for (int k = 0; k < H; ++k) {
      row[k] = bf16f(x[(size_t)t * H + k]);
      float a = fabsf(row[k]);
      if (a > amax) amax = a;
    }
    if (amax < 1e-12f) amax = 1e-12f;
    gs[t] = 2688.0f / amax;
    nvfp4_row(row, H, gs[t], codes + (size_t)t * (H / 2), scales + (size_t)t * (H / 16));
  }
  free(row);
}

/* [w8a8]: each group of 128 consecutive elements of a [T, H] bf16 row is quantized like one
   [fp8] weight tile: s = 448/max(amax, 1e-12), code = E4M3(v*s), 1/s stored.
   codes [T, H] E4M3; scale_inv [T, H/128]. */
void orc_quant_act_fp8(const uint16_t* x, int T, int H, uint8_t* codes, float* scale_inv) {
  for (int t = 0; t < T; ++t)
    for (int g = 0; g < H / 128; ++g) {
      const uint16_t* v = x + (size_t)t * H + g * 128;
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i) {
        float a = fabsf(bf16f(v[i]));
        if (a > amax) amax = a;
      }
      if (amax < 1e-12f) amax = 1e-12f;
      float s = 448.0f / amax;
      for (int i = 0; i < 128; ++i) codes[(size_t)t * H + g * 128 + i] = orc_e4m3_encode(bf16f(v[i]) * s);
      scale_inv[(size_t)t * (H / 128) + g] = 1.0f / s;
    }
}

/* value = E4M3(code) * scale_inv(group), one fp32 rounding (as the weights' dequantization). */
void orc_dequant_act_fp8(const uint8_t* codes, const float* scale_inv, int T, int H, float* out) {
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < H; ++k) {
      size_t i = (size_t)t * H + k;
      out[i] = (float)orc_e4m3_decode(codes[i]) * scale_inv[(size_t)t * (H / 128) + k / 128];
    }
}

/* ------------------------------------------------------------------------------------ */
/* Routing: top-k of the router logits, renormalised softmax, permutation by expert.    */
/* ------------------------------------------------------------------------------------ */

/* Per token: the k largest logits in descending order (ties to the lower expert index);
   w_j = exp(l_j - l_max) / sum over the selected of exp(l - l_max), in fp64. */
void orc_route(const float* logits, int T, int E, int k, int32_t* idx, double* w) {
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    double lmax = (double)l[idx[(size_t)t * k]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[idx[(size_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j)
      w[(size_t)t * k + j] = exp((double)l[idx[(size_t)t * k + j]] - lmax) / den;
  }
  free(taken);
}

/* Rows r = 0..T*k-1 sorted by (expert, token, slot).  offsets [E+1] (exclusive prefix of the
   per-expert counts), perm [T*k] = t*k + j of row r, inv [T*k] = row of (t, j). */
void orc_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets, int32_t* perm, int32_t* inv) {
  int pos = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = pos;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) {
          perm[pos] = t * k + j;
          inv[(size_t)t * k + j] = pos;
          ++pos;
        }
  }
  offsets[E] = pos;
}

/* ------------------------------------------------------------------------------------ */
/* The layer.                                                                            */
/* ------------------------------------------------------------------------------------ */

/* Dequantize expert e's matrix (which = 0: fused gate/up [2I, H]; 1: down [H, I]). */
static void dequant_expert(int fmt, int which, int e, int H, int I, const void* a, const void* b,
                           const float* gs, float* out) {
  int N = which == 0 ? 2 * I : H, K = which == 0 ? H : I;
  size_t NK = (size_t)N * K;
  if (fmt == ORC_FP8 || fmt == ORC_FP8_W8A8) {
    orc_dequant_fp8((const uint8_t*)a + NK * e, (const float*)b + (size_t)(N / 128) * (K / 128) * e, N, K, out);
  } else if (fmt == ORC_INT4) {
    orc_dequant_int4((const int32_t*)a + NK / 8 * e, (const uint16_t*)b + (size_t)(K / 128) * N * e, N, K, out);
  } else if (fmt == ORC_BF16) {  /* the stored bf16 value itself */
    const uint16_t* w = (const uint16_t*)a + NK * e;
    for (size_t i = 0; i < NK; ++i) out[i] = bf16f(w[i]);
  } else {
    orc_dequant_nvfp4((const uint8_t*)a + NK / 2 * e, (const uint8_t*)b + NK / 16 * e, gs[e], N, K, out);
  }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* y = Wd * act(Wgu * a) for one (token, expert) pair; h per the format's rules. */
static void expert_mlp(int fmt, int H, int I, const float* wgu, const float* wd, const double* a,
                       const float* act_gs, double* h, uint16_t* hb, uint8_t* hq, uint8_t* hs, uint8_t* hq8,
                       float* hdq, double* y) {
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    const float* wg = wgu + (size_t)n * H;
    const float* wu = wgu + (size_t)(I + n) * H;
    for (int k = 0; k < H; ++k) {
      g += (double)wg[k] * a[k];
      u += (double)wu[k] * a[k];
    }
    h[n] = silu(g) * u;
  }
  if (fmt == ORC_NVFP4_W4A4) {
    float gsr;
    for (int n = 0; n < I; ++n) hb[n] = orc_bf16_encode(h[n]);
    if (act_gs) {
      gsr = act_gs[1];
      orc_quant_act_nvfp4_static(hb, 1, I, gsr, hq, hs);
    } else {
      orc_quant_act_nvfp4(hb, 1, I, hq, hs, &gsr);
    }
    orc_dequant_nvfp4(hq, hs, gsr, 1, I, hdq);
    for (int n = 0; n < I; ++n) h[n] = (double)hdq[n];
  } else if (fmt == ORC_FP8_W8A8) {
    float* hsi = (float*)malloc(sizeof(float) * (I / 128));
    for (int n = 0; n < I; ++n) hb[n] = orc_bf16_encode(h[n]);
    orc_quant_act_fp8(hb, 1, I, hq8, hsi);
    orc_dequant_act_fp8(hq8, hsi, 1, I, hdq);
    for (int n = 0; n < I; ++n) h[n] = (double)hdq[n];
    free(hsi);
  }
  for (int c = 0; c < H; ++c) {
    double acc = 0.0;
    const float* wr = wd + (size_t)c * I;
    for (int n = 0; n < I; ++n) acc += (double)wr[n] * h[n];
    y[c] = acc;
  }
}

/* Activation row a_t: bf16 x (W8A16, W4A16) or the dequantized NVFP4 (W4A4) or FP8 (W8A8) row. */
static void act_row(int fmt, const uint16_t* xrow, int H, const float* act_gs, double* a) {
  if (fmt == ORC_FP8_W8A8) {
    uint8_t* q = (uint8_t*)malloc((size_t)H);
    float* si = (float*)malloc(sizeof(float) * (H / 128));
    float* d = (float*)malloc(sizeof(float) * H);
    orc_quant_act_fp8(xrow, 1, H, q, si);
    orc_dequant_act_fp8(q, si, 1, H, d);
    for (int k = 0; k < H; ++k) a[k] = (double)d[k];
    free(q);
    free(si);
    free(d);
  } else if (fmt == ORC_NVFP4_W4A4) {
    uint8_t* q = (uint8_t*)malloc((size_t)H / 2);
    uint8_t* s = (uint8_t*)malloc((size_t)H / 16);
    float* d = (float*)malloc(sizeof(float) * H);
    float gs;
    if (act_gs) {
      gs = act_gs[0];
      orc_quant_act_nvfp4_static(xrow, 1, H, gs, q, s);
    } else {
      orc_quant_act_nvfp4(xrow, 1, H, q, s, &gs);
    }
    orc_dequant_nvfp4(q, s, gs, 1, H, d);
    for (int k = 0; k < H; ++k) a[k] = (double)d[k];
    free(q);
    free(s);
    free(d);
  } else {
    for (int k = 0; k < H; ++k) a[k] = (double)bf16f(xrow[k]);
  }
}

/* Forward pass for the tokens tok[0..n_tok-1] (all T tokens when tok == NULL):
   route, then for every (token, slot): y = Wd_e * (silu(Wg_e a) * (Wu_e a)), and
   out_t = sum_j w_j y_j summed in slot order; everything accumulated in fp64.
   dense != 0 runs the dense masked definition instead: every token through all E experts,
   weighted by the routing weights scattered over experts (zero for unselected ones).
   Weights are passed per format: fp8 and fp8 W8A8 (codes, scale_inv, -), int4 (qweight, scales, -),
   nvfp4 (packed, block scales, global scales), bf16 (weights, -, -).  act_gs (W4A4 only): NULL
   quantizes x and h rows with their own dynamic global scales, else with the static scales
   act_gs[0] (x) and act_gs[1] (h).  Returns 0 on success. */
int orc_moe_layer(int fmt, int T, int H, int I, int E, int k, const uint16_t* x, const float* logits,
                  const void* gu_a, const void* gu_b, const float* gu_gs, const void* d_a, const void* d_b,
                  const float* d_gs, const int32_t* tok, int n_tok, int dense, int nthreads, const float* act_gs,
                  double* out) {
  if (H % 128 || I % 128 || k < 1 || k > E) return 1;
  if (tok == NULL) n_tok = T;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_tok * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)n_tok * k);
  double* acts = (double*)malloc(sizeof(double) * (size_t)n_tok * H);
  for (int i = 0; i < n_tok; ++i) {
    int t = tok ? tok[i] : i;
    orc_route(logits + (size_t)t * E, 1, E, k, idx + (size_t)i * k, w + (size_t)i * k);
    act_row(fmt, x + (size_t)t * H, H, act_gs, acts + (size_t)i * H);
  }
  int slots = dense ? E : k;
  double* ybuf = (double*)calloc((size_t)n_tok * slots * H, sizeof(double));
  char* used = (char*)calloc((size_t)n_tok * slots, 1);

#pragma omp parallel
  {
    float* wgu = (float*)malloc(sizeof(float) * (size_t)2 * I * H);
    float* wd = (float*)malloc(sizeof(float) * (size_t)H * I);
    double* h = (double*)malloc(sizeof(double) * I);
    uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * I);
    uint8_t* hq = (uint8_t*)malloc((size_t)I / 2);
    uint8_t* hs = (uint8_t*)malloc((size_t)I / 16);
    uint8_t* hq8 = (uint8_t*)malloc((size_t)I);
    float* hdq = (float*)malloc(sizeof(float) * I);
#pragma omp for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
      int any = 0;
      for (int i = 0; i < n_tok * k && !any; ++i) any = idx[i] == e;
      if (!any && !dense) continue;
      dequant_expert(fmt, 0, e, H, I, gu_a, gu_b, gu_gs, wgu);
      dequant_expert(fmt, 1, e, H, I, d_a, d_b, d_gs, wd);
      for (int i = 0; i < n_tok; ++i) {
        int slot = -1;
        if (dense) slot = e;
        else
          for (int j = 0; j < k; ++j)
            if (idx[(size_t)i * k + j] == e) slot = j;
        if (slot < 0) continue;
        expert_mlp(fmt, H, I, wgu, wd, acts + (size_t)i * H, act_gs, h, hb, hq, hs, hq8, hdq,
                   ybuf + ((size_t)i * slots + slot) * H);
        used[(size_t)i * slots + slot] = 1;
      }
    }
    free(wgu);
    free(wd);
    free(h);
    free(hb);
    free(hq);
    free(hs);
    free(hq8);
    free(hdq);
  }

  for (int i = 0; i < n_tok; ++i)
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      if (dense) {
        for (int e = 0; e < E; ++e) {
          double m = 0.0;
          for (int j = 0; j < k; ++j)
            if (idx[(size_t)i * k + j] == e) m = w[(size_t)i * k + j];
          acc += m * ybuf[((size_t)i * E + e) * H + c];
        }
      } else {
        for (int j = 0; j < k; ++j) acc += w[(size_t)i * k + j] * ybuf[((size_t)i * k + j) * H + c];
      }
      out[(size_t)i * H + c] = acc;
    }
  free(idx);
  free(w);
  free(acts);
  free(ybuf);
  free(used);
  return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
