/*
 * Oracle for the DSA attention layer group with IndexShare.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously correct CPU
 * restatement of what the hot path computes, used by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg.  The product path never
 * calls it, and it shares no code, header, table or constant with the CUDA
 * sources.
 *
 * Arithmetic is fp64 on the exact values of the inputs (bf16 -> double,
 * E4M3 code * fp32 scale -> double).  The FP8 quantisers follow their
 * definition in fp64 as well: rotate (indexer) by the normalised Hadamard
 * matrix, scale = the fp32 number nearest to amax / 448 (the scale is stored
 * as fp32), code = the E4M3 value nearest to x / scale.  The one rounding
 * this restatement adds is fp64's own (2^-53 relative), far below the fp32
 * error of any single-precision quantiser, so GPU codes are compared with
 * these by a rule that allows a code step only within the GPU arithmetic's
 * error bound of an E4M3 rounding boundary.
 *
 * Sources (GLM-5.2 pages):
 *  - "GLM-5.2 / 总览", config table (@tbl-glm52-config): 64 heads, QK head dim
 *    256 (NoPE 192 + RoPE 64), KV latent 512, per-token KV = 512 latent +
 *    64 RoPE key (1152 B in bf16), IndexShare indexer 32 heads x 128, top-K
 *    2048; sub-doc index row 02: lightning indexer with ReLU and an
 *    "FP8 per-block + Hadamard" variant.
 *  - "GLM-5.2 架构深度拆解" CH 2.2: an F layer scores every earlier token with
 *    32 heads x 128 dims and keeps the top 2048 as the sparse set; S layers
 *    skip the indexer and reuse the nearest F layer's indices; CH 2.4: the
 *    indices are written at F and read at S through an outer buffer.
 *  - "GLM-5 -> 5.1 -> 5.2" section 10: run the indexer once per group, write
 *    the shared indices to a buffer reused within the group, each layer
 *    gathers from its own K/V cache, then runs sparse attention.
 *  - "GLM-5.2架构与基准" Q&A: the indexer selects the top-k tokens per query
 *    among earlier positions (causal), turning O(L^2) attention into O(Lk).
 * The indexer formula I[t,s] = sum_j w[t,j] * ReLU(q[t,j] . k[s]) and the
 * tie-break on the lower position are the readings this build takes where
 * the pages give only the ingredients.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------ conversions */

/* bf16 bit pattern -> exact double. */
static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 flavour: 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; S.1111.111
 * is NaN; no infinities; largest finite magnitude 1.75 * 2^8 = 448. */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round-to-nearest-even encode with saturation to +-448, from a double: the
 * value is scaled by a power of two (exact) so that the E4M3 grid of its
 * binade becomes the integers, rounded with nearbyint (default rounding
 * mode: nearest, ties to even) and decoded back into a code.  No E4M3
 * infinity exists, so every magnitude from 448 up (and +-inf) saturates to
 * the largest finite code; NaN maps to 0x7F. */
uint8_t oracle_e4m3_encode_f64(double x) {
  uint8_t sign = (signbit(x) ? 0x80 : 0x00);
  double a = fabs(x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid: multiples of 2^-9; q == 8 is the smallest normal */
    double q = nearbyint(a / ldexp(1.0, -9)); /* exact scaling; ties to even */
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
  e -= 1;
  double quantum = ldexp(1.0, e - 3);
  double q = nearbyint(a / quantum); /* in [8, 16] */
  if (q >= 16.0) {
    q = 8.0;
    e += 1;
  }
  int field = e + 7;
  int code = (field << 3) | ((int)q - 8);
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

/* The same for an fp32 input (its value is exact in a double). */
uint8_t oracle_e4m3_encode(float xf) { return oracle_e4m3_encode_f64((double)xf); }

/* Element-wise forms for arrays (test bookkeeping). */
void oracle_e4m3_encode_array(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode_f64(x[i]);
}
void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* The fp32 number nearest to a / 448 for a finite a >= 0 (ties to the even
 * significand): the fp32 rounding of the fp64 quotient is a candidate, and
 * it and its two fp32 neighbours are compared by their exact distance to
 * a / 448, i.e. |a - 448 c| (448 c is exact in a double, and so is the
 * difference of two doubles this close). */
static float f32_nearest_quotient_448(double a) {
  const float r = (float)(a / 448.0);
  float best = r;
  double bd = fabs(a - 448.0 * (double)r);
  const float cand[2] = {nextafterf(r, -INFINITY), nextafterf(r, INFINITY)};
  for (int i = 0; i < 2; ++i) {
    const float c = cand[i];
    if (!(c >= 0.0f) || isinf(c)) continue;
    const double d = fabs(a - 448.0 * (double)c);
    uint32_t ub, uc;
    memcpy(&ub, &best, 4);
    memcpy(&uc, &c, 4);
    if (d < bd || (d == bd && (uc & 1u) == 0 && (ub & 1u) == 1)) {
      best = c;
      bd = d;
    }
  }
  return best;
}

/* Per-block FP8 scale of a block whose largest magnitude is amax: amax / 448
 * stored as fp32, 1 for an all-zero block. */
float oracle_fp8_block_scale(double amax) {
  return amax > 0.0 ? f32_nearest_quotient_448(amax) : 1.0f;
}

/* ------------------------------------------------------------ Hadamard */

/* Exact definition, fp64: out = H_128 * in / sqrt(128) where H is built by
 * Sylvester's recursion H_2n = [[H_n, H_n], [H_n, -H_n]], H_1 = [1]; the
 * entry (i, j) of H is (-1)^popcount(i & j). */
void oracle_hadamard128_f64(const double* in, double* out) {
  for (int i = 0; i < 128; ++i) {
    double s = 0.0;
    for (int j = 0; j < 128; ++j) s += (__builtin_popcount((unsigned)(i & j)) & 1) ? -in[j] : in[j];
    out[i] = s / sqrt(128.0);
  }
}

/* The rotated rows H_128 x / sqrt(128) of bf16 rows x [rows, 128], in fp64
 * (test bookkeeping: the values the quantiser below encodes). */
void oracle_fp8_rotate_rows(const uint16_t* x, int64_t rows, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double v[128];
    for (int j = 0; j < 128; ++j) v[j] = bf16_value(x[r * 128 + j]);
    oracle_hadamard128_f64(v, y + r * 128);
  }
}

/* FP8 per-block quantiser for indexer vectors ("GLM-5.2 / 总览" sub-doc
 * index row 02: "FP8 per-block + Hadamard"; one block = one 128-vector):
 *   y     = H_128 x / sqrt(128)                       (fp64, definition above)
 *   scale = amax / 448 as fp32, amax = max_j |y_j|    (1 for an all-zero block)
 *   q_j   = E4M3(y_j / scale), nearest, ties to even, saturating
 * The quotient is formed in fp64 (one rounding of 2^-53 relative) and
 * encoded from that double.  x is bf16 [rows, 128]; q is [rows, 128] codes;
 * scale is [rows]. */
void oracle_fp8_quantize_rows(const uint16_t* x, int64_t rows, uint8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double v[128], y[128];
    for (int j = 0; j < 128; ++j) v[j] = bf16_value(x[r * 128 + j]);
    oracle_hadamard128_f64(v, y);
    double amax = 0.0;
    for (int j = 0; j < 128; ++j)
      if (fabs(y[j]) > amax) amax = fabs(y[j]);
    const float sc = oracle_fp8_block_scale(amax);
    scale[r] = sc;
    for (int j = 0; j < 128; ++j) q[r * 128 + j] = oracle_e4m3_encode_f64(y[j] / (double)sc);
  }
}

/* ------------------------------------------------------------ RoPE */

/* fp64 -> bf16 bit pattern, rounded once to nearest with ties to even: |x|
 * is scaled by a power of two (exact) so that the bf16 grid of its binade
 * becomes the integers (bf16 keeps 8 significant bits; below the normal
 * range the grid spacing stays 2^-133), rounded with rint (default rounding
 * mode: nearest, ties to even) and scaled back (exact).  Results beyond the
 * largest finite bf16 become infinity. */
uint16_t oracle_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  const uint16_t sign = signbit(x) ? 0x8000 : 0;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
  int es = e - 8;
  if (es < -133) es = -133;
  const double y = ldexp(rint(ldexp(a, -es)), es);
  if (y > 3.3895313892515355e38) return sign | 0x7F80;
  const float f = (float)y; /* exact: y lies on the bf16 grid */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/* Interleaved rotary embedding ("GLM-5.2 架构深度拆解" CH 7.1 table: indexer
 * 32 heads x 128 with indexer_rope_interleave; partial RoPE on a 64-d
 * subspace, interleaved): each vector of width `dim` at position pos[v] has
 * its entries (2i, 2i+1), i < rope_dims / 2, rotated by the angle
 * pos[v] * inv_freq[i]:
 *   y[2i]   = x[2i] cos a - x[2i+1] sin a
 *   y[2i+1] = x[2i] sin a + x[2i+1] cos a
 * in fp64 on the exact bf16 inputs, each result rounded once to bf16; the
 * entries from rope_dims on are copied.  inv_freq[i] = theta^(-2i/rope_dims)
 * for the model's base theta, given by the caller. */
void oracle_rope_bf16(const uint16_t* x, const int32_t* pos, int64_t n, int dim, int rope_dims,
                      const double* inv_freq, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t v = 0; v < n; ++v) {
    const uint16_t* xv = x + v * dim;
    uint16_t* yv = out + v * dim;
    for (int i = 0; i < rope_dims / 2; ++i) {
      const double a = (double)pos[v] * inv_freq[i];
      const double c = cos(a), s = sin(a);
      const double x0 = bf16_value(xv[2 * i]), x1 = bf16_value(xv[2 * i + 1]);
      yv[2 * i] = oracle_f64_to_bf16(x0 * c - x1 * s);
      yv[2 * i + 1] = oracle_f64_to_bf16(x0 * s + x1 * c);
    }
    for (int k = rope_dims; k < dim; ++k) yv[k] = xv[k];
  }
}

/* ------------------------------------------------------------ FP8 KV latent */

/* FP8 KV cache row (656 bytes per position; "GLM-5.2 / 总览" config table:
 * per-token per-layer KV cache BF16 = 1152 B, FP8 ~656 B per-group): the
 * 512-d latent as E4M3 codes in four groups of 128 dims, each with its own
 * scale amax/448 stored as fp32 (1 for an all-zero group), then the 64-d
 * RoPE key kept in bf16:  bytes [0, 512) codes, [512, 528) four fp32 scales,
 * [528, 656) 64 bf16.  Code = the E4M3 value nearest to x / scale (ties to
 * even, saturating).  The quotient of a bf16 value by an fp32 scale is
 * formed in fp64; it can lie no closer than about 2^-30 relative to an
 * E4M3 rounding boundary without being on it, far more than fp64's 2^-53,
 * so each code is the exact quotient's. */
void oracle_kv_fp8_quantize(const uint16_t* kv, int64_t rows, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* x = kv + r * 576;
    uint8_t* o = out + r * 656;
    for (int g = 0; g < 4; ++g) {
      double amax = 0.0;
      for (int j = 0; j < 128; ++j) {
        const double m = fabs(bf16_value(x[128 * g + j]));
        if (m > amax) amax = m;
      }
      const float sc = oracle_fp8_block_scale(amax);
      memcpy(o + 512 + 4 * g, &sc, 4);
      for (int j = 0; j < 128; ++j)
        o[128 * g + j] = oracle_e4m3_encode_f64(bf16_value(x[128 * g + j]) / (double)sc);
    }
    memcpy(o + 528, x + 512, 128);
  }
}

/* The bf16 row the attention reads from an FP8 KV row: latent value =
 * code * scale formed as an fp32 product (round to nearest even), then
 * rounded to the bf16 the attention multiplies; the RoPE key as stored.  The
 * pages fix no rounding for this step; two roundings (fp32, then bf16)
 * rather than one of the exact product is the reading taken because it is
 * the cheaper one to widen inside the attention kernel. */
void oracle_kv_fp8_dequantize(const uint8_t* in, int64_t rows, uint16_t* kv) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t* o = in + r * 656;
    uint16_t* x = kv + r * 576;
    for (int g = 0; g < 4; ++g) {
      float sc;
      memcpy(&sc, o + 512 + 4 * g, 4);
      for (int j = 0; j < 128; ++j) {
        volatile float prod = (float)oracle_e4m3_decode(o[128 * g + j]) * sc;
        x[128 * g + j] = oracle_f64_to_bf16((double)prod);
      }
    }
    memcpy(x + 512, o + 528, 128);
  }
}

/* ------------------------------------------------------------ indexer */

/* Lightning-indexer scores for the listed query rows.
 *   I[t, s] = sum_{j < Hi} w[t, j] * ReLU( q[t, j, :] . k[s, :] ),  0 <= s <= pos[t]
 *   I[t, s] = -inf                                                pos[t] < s < max_len
 * dtype 0: q_idx [num_q, Hi, Di] and k_idx [rows, Di] are bf16 bit patterns.
 * dtype 1: they are E4M3 codes; the value of a q element is code * q_scale[t, j]
 *          and of a k element code * k_scale[row].
 * Listed row i is query t = rows[i] at position row_pos[i]; its key for
 * position s is cache row row_key0[i] + s.  scores is [nrows, max_len]. */
void oracle_indexer_scores(int Hi, int Di, int dtype, const void* q_idx, const float* q_scale,
                           const float* w, const void* k_idx, const float* k_scale,
                           const int32_t* rows, const int32_t* row_pos, const int64_t* row_key0,
                           int nrows, int64_t max_len, double* scores) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < nrows; ++i) {
    const int64_t t = rows[i];
    double* out = scores + (int64_t)i * max_len;
    double* qv = (double*)malloc(sizeof(double) * (size_t)Hi * (size_t)Di);
    double* kv = (double*)malloc(sizeof(double) * (size_t)Di);
    for (int j = 0; j < Hi; ++j)
      for (int d = 0; d < Di; ++d) {
        int64_t e = (t * Hi + j) * Di + d;
        qv[j * Di + d] = dtype == 0 ? bf16_value(((const uint16_t*)q_idx)[e])
                                    : oracle_e4m3_decode(((const uint8_t*)q_idx)[e]) *
                                          (double)q_scale[t * Hi + j];
      }
    for (int64_t s = 0; s < max_len; ++s) {
      if (s > row_pos[i]) {
        out[s] = -INFINITY;
        continue;
      }
      int64_t kr = row_key0[i] + s;
      for (int d = 0; d < Di; ++d)
        kv[d] = dtype == 0 ? bf16_value(((const uint16_t*)k_idx)[kr * Di + d])
                           : oracle_e4m3_decode(((const uint8_t*)k_idx)[kr * Di + d]) *
                                 (double)k_scale[kr];
      double acc = 0.0;
      for (int j = 0; j < Hi; ++j) {
        double dot = 0.0;
        for (int d = 0; d < Di; ++d) dot += qv[j * Di + d] * kv[d];
        acc += (double)w[t * Hi + j] * (dot > 0.0 ? dot : 0.0);
      }
      out[s] = acc;
    }
    free(qv);
    free(kv);
  }
}

/* ------------------------------------------------------------ top-K */

typedef struct {
  double v;
  int32_t s;
} scored_t;

/* Larger score first; equal scores: lower position first. */
static int by_score_then_pos(const void* a, const void* b) {
  const scored_t* x = (const scored_t*)a;
  const scored_t* y = (const scored_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->s > y->s) - (x->s < y->s);
}
static int by_int(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* For each row i, the K positions s in [0, len[i]) with the largest
 * scores[i, s] (ties: lower s), written to idx[i, :] in ascending position
 * order; when len[i] < K every visible position is taken and the remaining
 * slots hold -1. */
void oracle_topk(const double* scores, int64_t ld, const int32_t* len, int nrows, int K,
                 int32_t* idx) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < nrows; ++i) {
    int n = len[i];
    scored_t* buf = (scored_t*)malloc(sizeof(scored_t) * (size_t)(n > 0 ? n : 1));
    for (int s = 0; s < n; ++s) {
      buf[s].v = scores[(int64_t)i * ld + s];
      buf[s].s = s;
    }
    qsort(buf, (size_t)n, sizeof(scored_t), by_score_then_pos);
    int take = n < K ? n : K;
    int32_t* row = idx + (int64_t)i * K;
    for (int j = 0; j < take; ++j) row[j] = buf[j].s;
    qsort(row, (size_t)take, sizeof(int32_t), by_int);
    for (int j = take; j < K; ++j) row[j] = -1;
    free(buf);
  }
}

/* ------------------------------------------------------------ sparse MLA */

/* Absorbed-MLA attention over the selected positions only.  For listed row
 * i (query t = rows[i]), head h and selected position s = idx[i, j] >= 0:
 *   z_s = scale * ( q_lat[t,h,:] . C[s, :Dl] + q_rope[t,h,:] . C[s, Dl:] )
 *   p_s = exp(z_s - max z) / sum exp(z - max z)
 *   out[i,h,:] = sum_s p_s C[s, :Dl],   lse[i,h] = log sum_s exp(z_s)
 * where C[s] is kv row row_key0[i] + s (latent Dl, then rope key Dr).
 * Entries equal to -1 are skipped; a row with no selected position gives
 * out = 0 and lse = -inf. */
void oracle_sparse_mla(int H, int Dl, int Dr, const uint16_t* q_lat, const uint16_t* q_rope,
                       const uint16_t* kv, const int32_t* rows, const int64_t* row_key0,
                       int nrows, const int32_t* idx, int K, double scale, double* out,
                       double* lse) {
  const int Dk = Dl + Dr;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < nrows; ++i) {
    const int64_t t = rows[i];
    const int32_t* sel = idx + (int64_t)i * K;
    double* z = (double*)malloc(sizeof(double) * (size_t)K);
    for (int h = 0; h < H; ++h) {
      double m = -INFINITY;
      for (int j = 0; j < K; ++j) {
        if (sel[j] < 0) continue;
        const uint16_t* c = kv + (row_key0[i] + sel[j]) * Dk;
        double dot = 0.0;
        for (int d = 0; d < Dl; ++d) dot += bf16_value(q_lat[(t * H + h) * Dl + d]) * bf16_value(c[d]);
        for (int d = 0; d < Dr; ++d)
          dot += bf16_value(q_rope[(t * H + h) * Dr + d]) * bf16_value(c[Dl + d]);
        z[j] = dot * scale;
        if (z[j] > m) m = z[j];
      }
      double* o = out + ((int64_t)i * H + h) * Dl;
      for (int d = 0; d < Dl; ++d) o[d] = 0.0;
      if (m == -INFINITY) {
        lse[(int64_t)i * H + h] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int j = 0; j < K; ++j) {
        if (sel[j] < 0) continue;
        double p = exp(z[j] - m);
        l += p;
        const uint16_t* c = kv + (row_key0[i] + sel[j]) * Dk;
        for (int d = 0; d < Dl; ++d) o[d] += p * bf16_value(c[d]);
      }
      for (int d = 0; d < Dl; ++d) o[d] /= l;
      lse[(int64_t)i * H + h] = m + log(l);
    }
    free(z);
  }
}

/* Dense causal attention for the same row, over every position 0..pos:
 * used only to pin the sparse routine (equal when K covers all positions). */
void oracle_dense_mla(int H, int Dl, int Dr, const uint16_t* q_lat, const uint16_t* q_rope,
                      const uint16_t* kv, const int32_t* rows, const int32_t* row_pos,
                      const int64_t* row_key0, int nrows, double scale, double* out, double* lse) {
  const int Dk = Dl + Dr;
  for (int i = 0; i < nrows; ++i) {
    const int64_t t = rows[i];
    const int n = row_pos[i] + 1;
    double* z = (double*)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < H; ++h) {
      double m = -INFINITY;
      for (int s = 0; s < n; ++s) {
        const uint16_t* c = kv + (row_key0[i] + s) * Dk;
        double dot = 0.0;
        for (int d = 0; d < Dl; ++d) dot += bf16_value(q_lat[(t * H + h) * Dl + d]) * bf16_value(c[d]);
        for (int d = 0; d < Dr; ++d)
          dot += bf16_value(q_rope[(t * H + h) * Dr + d]) * bf16_value(c[Dl + d]);
        z[s] = dot * scale;
        if (z[s] > m) m = z[s];
      }
      double l = 0.0;
      double* o = out + ((int64_t)i * H + h) * Dl;
      for (int d = 0; d < Dl; ++d) o[d] = 0.0;
      for (int s = 0; s < n; ++s) {
        double p = exp(z[s] - m);
        l += p;
        const uint16_t* c = kv + (row_key0[i] + s) * Dk;
        for (int d = 0; d < Dl; ++d) o[d] += p * bf16_value(c[d]);
      }
      for (int d = 0; d < Dl; ++d) o[d] /= l;
      lse[(int64_t)i * H + h] = m + log(l);
    }
    free(z);
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
