/*
 * Oracle for the low-bit dual-path MLA KV cache: a plain, slow, fp64 CPU restatement of
 * what the fused cache writer and the decode attention compute.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU-baseline
 * / reference legs may load this library. It shares no code, header, table or helper with
 * the CUDA library; it follows the method as the pages state it:
 *   - RAQ-MLA page (Role-Aware Quantization for Multi-Head Latent Attention Caches),
 *     appendix Table 5: latent INT2/INT4 per token in groups of 128 channels with an FP16
 *     scale and minimum per group and a per-token 0.94-quantile clip of |x|; k_R INT4 per
 *     channel within a cache page, FP16 scale and minimum per channel and page, no clip.
 *   - QuantMLA page, appendix Figure 8 caption: a packed copy of every incoming token, BF16
 *     pre-quantization values kept for sink and recent tokens, the switch to the existing
 *     packed copy when a token leaves the recent window, one global softmax over all tokens.
 *   - RAQ-MLA page, Figures 3-4: the cached latent serves as key and value, the score is
 *     q_lat . c + q_rope . k_R, the readout stays in latent space.
 * Readings where the pages are silent (the exact roundings, the quantile definition, the
 * byte layout) are those documented with the C ABI; the byte layout is re-derived here from
 * its written description, independently of the CUDA code.
 *
 * Everything is computed in double precision. Every FP16/BF16 value is exactly a double,
 * and every threshold formed below (an FP16 minimum plus a half-integer multiple of an FP16
 * scale) is exact in double (at most 46 significant bits), so each rounding decision is made
 * exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LATENT 512
#define ROPE 64
#define ROW 576
#define GROUP 128

#define ERR_BAD_PAGE 1
#define ERR_SEQ_OVERFLOW 2
#define ERR_NONFINITE 4
#define ERR_RANGE 8
#define ERR_ROWS 16

#define F16_MAX 65504.0

typedef struct {
  int32_t bits_c;
  int32_t bits_r;
  int32_t page_size;
  int32_t n_sink;
  int32_t n_recent;
  float clip_q;
} oracle_config;

/* ---------------------------------------------------------------- number formats */

/* BF16 bit pattern -> value (the upper half of an IEEE binary32). */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP16 bit pattern -> value, from the binary16 definition. */
double oracle_f16_to_double(uint16_t bits) {
  int sign = bits >> 15;
  int e = (bits >> 10) & 31;
  int m = bits & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* Bit pattern of a value that is exactly a finite FP16 number (zero encodes as +0). */
uint16_t oracle_f16_bits(double v) {
  if (v == 0.0) return 0;
  uint16_t sign = v < 0 ? 0x8000 : 0;
  double a = fabs(v);
  if (a < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(a, 24); /* subnormal: a = m * 2^-24 */
  int E;
  frexp(a, &E);                 /* a = f * 2^E, f in [0.5, 1) -> binary16 exponent E-1 */
  int e = E - 1 + 15;           /* biased exponent */
  int m = (int)ldexp(a, 11 - E) - 1024; /* a = (1024 + m) * 2^(E-11) */
  return sign | (uint16_t)(e << 10) | (uint16_t)m;
}

/* Largest FP16 value <= a, for finite a >= 0 (at most F16_MAX). */
static double f16_floor_nonneg(double a) {
  if (a >= F16_MAX) return F16_MAX;
  if (a < ldexp(1.0, -14)) return ldexp(floor(ldexp(a, 24)), -24);
  int E;
  frexp(a, &E); /* a = f * 2^E with f in [0.5, 1): the FP16 grid step there is 2^(E-11) */
  return ldexp(floor(ldexp(a, 11 - E)), E - 11);
}

/* Smallest FP16 value >= a, for finite a >= 0 (may exceed F16_MAX: callers check). */
static double f16_ceil_nonneg(double a) {
  if (a < ldexp(1.0, -14)) return ldexp(ceil(ldexp(a, 24)), -24);
  int E;
  frexp(a, &E);
  return ldexp(ceil(ldexp(a, 11 - E)), E - 11);
}

/* Largest finite FP16 value <= x (zero as +0). Sets *range if none exists (x < -65504). */
double oracle_f16_round_down(double x, int* range) {
  if (x >= 0) return f16_floor_nonneg(x) + 0.0;
  double c = f16_ceil_nonneg(-x);
  if (c > F16_MAX) {
    if (range) *range = 1;
    return -F16_MAX;
  }
  return -c;
}

/* Smallest finite FP16 value >= x (zero as +0). Sets *range if none exists (x > 65504). */
double oracle_f16_round_up(double x, int* range) {
  if (x <= 0) {
    double f = f16_floor_nonneg(-x);
    return f == 0.0 ? 0.0 : -f;
  }
  double c = f16_ceil_nonneg(x);
  if (c > F16_MAX) {
    if (range) *range = 1;
    return F16_MAX;
  }
  return c;
}

/* Neighbours of a non-negative finite FP16 value, by stepping its bit pattern. */
static double f16_next_up(double v) { return oracle_f16_to_double((uint16_t)(oracle_f16_bits(v) + 1)); }
static double f16_next_down(double v) {
  uint16_t b = oracle_f16_bits(v);
  return b == 0 ? 0.0 : oracle_f16_to_double((uint16_t)(b - 1));
}

/* ---------------------------------------------------------------- quantizer (Table 5) */

/*
 * Asymmetric uniform quantizer with FP16 minimum and scale, L = 2^bits - 1 levels above the
 * minimum (RAQ-MLA page, appendix Table 5: "FP16 scale and minimum"; rounding directions and
 * ties are the documented reading):
 *   min   = largest FP16 <= min(x)
 *   scale = smallest FP16 >= 0 such that min + L*scale >= max(x)
 *   code  = nearest level index in [0, L], an exact tie going to the even index
 * Returns ERR_* flags (0 when fine).
 */
int oracle_quantize(const double* x, int n, int bits, uint8_t* codes, uint16_t* scale_bits,
                    uint16_t* min_bits) {
  const int L = (1 << bits) - 1;
  int flags = 0, range = 0;
  double lo = x[0], hi = x[0];
  for (int i = 0; i < n; ++i) {
    if (!isfinite(x[i])) flags |= ERR_NONFINITE;
    if (x[i] < lo) lo = x[i];
    if (x[i] > hi) hi = x[i];
  }
  if (flags) { /* unspecified output; keep it deterministic */
    memset(codes, 0, (size_t)n);
    *scale_bits = 0;
    *min_bits = 0;
    return flags;
  }
  double mn = oracle_f16_round_down(lo, &range);
  /* scale: start from the smallest FP16 >= (hi - mn)/L computed in double, then settle it
     with exact tests of the defining inequality mn + L*scale >= hi. */
  double s = oracle_f16_round_up((hi - mn) / L, &range);
  if (s < 0) s = 0;
  while (s > 0 && mn + L * f16_next_down(s) >= hi) s = f16_next_down(s);
  while (mn + L * s < hi && s < F16_MAX) s = f16_next_up(s);
  if (mn + L * s < hi) range = 1;
  if (hi > F16_MAX) range = 1;
  if (range) flags |= ERR_RANGE;
  *min_bits = oracle_f16_bits(mn);
  *scale_bits = oracle_f16_bits(s);
  for (int i = 0; i < n; ++i) {
    int k = 0;
    if (s > 0) {
      /* midpoint between levels j and j+1: T_j = mn + (j + 1/2) * s (exact in double) */
      for (int j = 0; j < L; ++j) {
        double T = mn + (j + 0.5) * s;
        if (x[i] > T || (x[i] == T && ((j + 1) % 2 == 0))) k = j + 1;
      }
    }
    codes[i] = (uint8_t)k;
  }
  return flags;
}

/*
 * Per-token clip of the latent (RAQ-MLA page, appendix Table 5: clip at the 0.94 quantile of
 * |x|, per token). Reading: tau is the nearest-rank order statistic, the k-th smallest |x_i|
 * with k = ceil(q * n) (1-based), and every x_i is clamped to [-tau, tau].
 */
static int cmp_double(const void* a, const void* b) {
  double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

double oracle_clip_tau(const double* x, int n, float clip_q) {
  double* a = (double*)malloc(sizeof(double) * (size_t)n);
  for (int i = 0; i < n; ++i) a[i] = fabs(x[i]);
  qsort(a, (size_t)n, sizeof(double), cmp_double);
  int k = (int)ceil((double)clip_q * n);
  if (k < 1) k = 1;
  if (k > n) k = n;
  double tau = a[k - 1];
  free(a);
  return tau;
}

/* ---------------------------------------------------------------- page layout */

size_t oracle_page_bytes(const oracle_config* cfg) {
  size_t P = (size_t)cfg->page_size;
  return P * (64u * (size_t)cfg->bits_c + 32u + 16u) + 256u;
}

/* Position of latent code (token t of the page, channel c): byte offset in the page and bit shift.
   Region A holds one row of 64*bits_c bytes per token. Byte k of the row carries channels in
   order (c = 2k low nibble, 2k+1 high nibble for INT4; c = 4k+i at bits 2i for INT2); the
   row's 16-byte chunks are stored permuted, logical chunk k/16 at chunk (k/16) XOR (t mod 8). */
void oracle_latent_code_pos(int bits_c, int t, int c, size_t* byte, int* shift) {
  int row = 64 * bits_c;
  int k = c * bits_c / 8;
  int chunk = (k / 16) ^ (t % 8);
  *byte = (size_t)t * (size_t)row + (size_t)chunk * 16u + (size_t)(k % 16);
  *shift = (c * bits_c) % 8;
}

/* Position of k_R code (token t of the page, channel j). */
void oracle_rope_code_pos(int bits_c, int page_size, int t, int j, size_t* byte, int* shift) {
  int e = j % 16, q = (e % 8) / 2, h = e / 8, o = e % 2, n = (t % 16) / 8;
  int lane = 4 * (t % 8) + q;
  int pos = (2 * n + h) + 4 * o;
  int bit = 4 * pos;
  size_t base = (size_t)page_size * 64u * (size_t)bits_c;
  size_t block = ((size_t)(t / 16) * 4 + (size_t)(j / 16)) * 128u;
  *byte = base + block + (size_t)lane * 4u + (size_t)(bit / 8);
  *shift = bit % 8;
}

static size_t latent_meta_off(const oracle_config* cfg, int t, int g) {
  return (size_t)cfg->page_size * (64u * (size_t)cfg->bits_c + 32u) + ((size_t)t * 4 + (size_t)g) * 4u;
}

static size_t rope_meta_off(const oracle_config* cfg, int j) {
  return (size_t)cfg->page_size * (64u * (size_t)cfg->bits_c + 48u) + (size_t)j * 4u;
}

static void put_code(uint8_t* page, size_t byte, int shift, int width, int code) {
  uint8_t mask = (uint8_t)(((1 << width) - 1) << shift);
  page[byte] = (uint8_t)((page[byte] & ~mask) | ((code << shift) & mask));
}

static int get_code(const uint8_t* page, size_t byte, int shift, int width) {
  return (page[byte] >> shift) & ((1 << width) - 1);
}

static void put_u16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xff);
  p[1] = (uint8_t)(v >> 8);
}

static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------- writer (Figure 8) */

int oracle_config_ok(const oracle_config* c) {
  if (!c) return 0;
  if (c->bits_c != 2 && c->bits_c != 4) return 0;
  if (c->bits_r != 4) return 0;
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128) return 0;
  if (c->n_sink < 0 || c->n_sink > 16) return 0;
  if (c->n_recent < c->page_size || c->n_recent > 1024) return 0;
  if (!(c->clip_q >= 0.0f && c->clip_q <= 1.0f)) return 0;
  return 1;
}

/* Quantize token (c, k_R are double[512] / the BF16 row) into its page slot: latent only. */
static int pack_latent(const oracle_config* cfg, uint8_t* page, int t, const double* c_in) {
  double c[LATENT];
  int flags = 0;
  memcpy(c, c_in, sizeof c);
  if (cfg->clip_q > 0.0f) {
    double tau = oracle_clip_tau(c, LATENT, cfg->clip_q);
    for (int i = 0; i < LATENT; ++i) c[i] = c[i] < -tau ? -tau : (c[i] > tau ? tau : c[i]);
  }
  for (int g = 0; g < LATENT / GROUP; ++g) {
    uint8_t codes[GROUP];
    uint16_t sb, mb;
    flags |= oracle_quantize(c + g * GROUP, GROUP, cfg->bits_c, codes, &sb, &mb);
    for (int i = 0; i < GROUP; ++i) {
      size_t byte;
      int shift;
      oracle_latent_code_pos(cfg->bits_c, t, g * GROUP + i, &byte, &shift);
      put_code(page, byte, shift, cfg->bits_c, codes[i]);
    }
    size_t mo = latent_meta_off(cfg, t, g);
    put_u16(page + mo, sb);
    put_u16(page + mo + 2, mb);
  }
  return flags;
}

/* Quantize the k_R of a full page, per channel over its P tokens (values[t*64 + j]). */
static int pack_rope_page(const oracle_config* cfg, uint8_t* page, const double* values) {
  const int P = cfg->page_size;
  int flags = 0;
  double* col = (double*)malloc(sizeof(double) * (size_t)P);
  uint8_t* codes = (uint8_t*)malloc((size_t)P);
  for (int j = 0; j < ROPE; ++j) {
    uint16_t sb, mb;
    for (int t = 0; t < P; ++t) col[t] = values[(size_t)t * ROPE + (size_t)j];
    flags |= oracle_quantize(col, P, cfg->bits_r, codes, &sb, &mb);
    for (int t = 0; t < P; ++t) {
      size_t byte;
      int shift;
      oracle_rope_code_pos(cfg->bits_c, P, t, j, &byte, &shift);
      put_code(page, byte, shift, 4, codes[t]);
    }
    size_t mo = rope_meta_off(cfg, j);
    put_u16(page + mo, sb);
    put_u16(page + mo + 2, mb);
  }
  free(col);
  free(codes);
  return flags;
}

/*
 * Sequential cache writer. Tokens are processed one at a time in position order, as a plain
 * state machine: pack the latent, store the BF16 row in the ring (and the sink buffer for
 * t < S), and when a page becomes full quantize its k_R from the ring (P <= W keeps every
 * token of that page in the ring). Returns ERR_* flags.
 */
int oracle_write(const oracle_config* cfg, int B, int n_rows, const uint16_t* c_new,
                 const uint16_t* kr_new, const int32_t* cu_new, const int32_t* seq_lens,
                 int max_new, const int32_t* page_table, int max_pages, uint8_t* pool,
                 int64_t n_pages, uint16_t* sink, uint16_t* ring) {
  const int P = cfg->page_size, S = cfg->n_sink, W = cfg->n_recent;
  const size_t pb = oracle_page_bytes(cfg);
  int flags = 0;
  if (cu_new[0] != 0 || cu_new[B] != n_rows) flags |= ERR_ROWS;
  double* page_vals = (double*)malloc(sizeof(double) * (size_t)P * ROPE);
  for (int b = 0; b < B; ++b) {
    int n = cu_new[b + 1] - cu_new[b];
    if (n < 0 || n > max_new) {
      flags |= ERR_ROWS;
      continue;
    }
    if (seq_lens[b] < 0) {
      flags |= ERR_SEQ_OVERFLOW;
      continue;
    }
    for (int i = 0; i < n; ++i) {
      int64_t t = (int64_t)seq_lens[b] + i;
      size_t row = (size_t)cu_new[b] + (size_t)i;
      int64_t p = t / P;
      if (p >= max_pages) {
        flags |= ERR_SEQ_OVERFLOW;
        continue;
      }
      int32_t pid = page_table[(size_t)b * (size_t)max_pages + (size_t)p];
      int page_ok = pid >= 0 && pid < n_pages;
      if (!page_ok) flags |= ERR_BAD_PAGE;
      uint8_t* page = page_ok ? pool + (size_t)pid * pb : NULL;

      uint16_t rowbits[ROW];
      memcpy(rowbits, c_new + row * LATENT, sizeof(uint16_t) * LATENT);
      memcpy(rowbits + LATENT, kr_new + row * ROPE, sizeof(uint16_t) * ROPE);
      if (page_ok) {
        double c[LATENT];
        for (int k = 0; k < LATENT; ++k) c[k] = oracle_bf16_to_double(rowbits[k]);
        flags |= pack_latent(cfg, page, (int)(t % P), c);
      }
      if (t < S) memcpy(sink + ((size_t)b * S + (size_t)t) * ROW, rowbits, sizeof rowbits);
      memcpy(ring + ((size_t)b * W + (size_t)(t % W)) * ROW, rowbits, sizeof rowbits);

      if ((t + 1) % P == 0 && page_ok) {
        for (int u = 0; u < P; ++u) {
          int64_t tu = p * P + u;
          const uint16_t* r = ring + ((size_t)b * W + (size_t)(tu % W)) * ROW;
          for (int j = 0; j < ROPE; ++j) page_vals[(size_t)u * ROPE + j] = oracle_bf16_to_double(r[LATENT + j]);
        }
        flags |= pack_rope_page(cfg, page, page_vals);
      }
    }
  }
  free(page_vals);
  return flags;
}

/* ---------------------------------------------------------------- reading the cache back */

/*
 * The 576 values attention uses for token t of sequence b with T cached tokens: the BF16
 * row if the token is protected (t < S or t >= T - W), otherwise the dequantized packed copy
 * min + code * scale of its latent group and of its page's k_R channel.
 * Returns 1 if the token was protected, 0 if read from its packed copy, -1 on a bad page.
 */
int oracle_token_values(const oracle_config* cfg, int b, int t, int T, const int32_t* page_table,
                        int max_pages, const uint8_t* pool, int64_t n_pages, const uint16_t* sink,
                        const uint16_t* ring, double* v) {
  const int P = cfg->page_size, S = cfg->n_sink, W = cfg->n_recent;
  if (t < S || t >= T - W) {
    const uint16_t* r = t < S ? sink + ((size_t)b * S + (size_t)t) * ROW
                              : ring + ((size_t)b * W + (size_t)(t % W)) * ROW;
    for (int k = 0; k < ROW; ++k) v[k] = oracle_bf16_to_double(r[k]);
    return 1;
  }
  int p = t / P, tp = t % P;
  if (p >= max_pages) return -1;
  int32_t pid = page_table[(size_t)b * (size_t)max_pages + (size_t)p];
  if (pid < 0 || pid >= n_pages) return -1;
  const uint8_t* page = pool + (size_t)pid * oracle_page_bytes(cfg);
  for (int c = 0; c < LATENT; ++c) {
    size_t byte;
    int shift;
    oracle_latent_code_pos(cfg->bits_c, tp, c, &byte, &shift);
    int code = get_code(page, byte, shift, cfg->bits_c);
    size_t mo = latent_meta_off(cfg, tp, c / GROUP);
    double sc = oracle_f16_to_double(get_u16(page + mo));
    double mn = oracle_f16_to_double(get_u16(page + mo + 2));
    v[c] = mn + code * sc;
  }
  for (int j = 0; j < ROPE; ++j) {
    size_t byte;
    int shift;
    oracle_rope_code_pos(cfg->bits_c, P, tp, j, &byte, &shift);
    int code = get_code(page, byte, shift, 4);
    size_t mo = rope_meta_off(cfg, j);
    double sc = oracle_f16_to_double(get_u16(page + mo));
    double mn = oracle_f16_to_double(get_u16(page + mo + 2));
    v[LATENT + j] = mn + code * sc;
  }
  return 0;
}

/* ---------------------------------------------------------------- decode attention */

/*
 * Single-token decode attention with one global softmax (QuantMLA page, Figure 8; RAQ-MLA
 * page, Figures 3-4), written as the two-pass definition:
 *   s_t = scale * (q_lat . v_t[0:512] + q_rope . v_t[512:576])
 *   m = max_t s_t,  l = sum_t exp(s_t - m)
 *   out = sum_t exp(s_t - m) v_t[0:512] / l,  lse = m + ln l
 * T = 0 gives out = 0 and lse = -inf. Returns ERR_* flags (bad pages are skipped).
 */
/* Exact attention of one sequence over its gathered token rows V[T][576] (ok[t] = row usable):
 * scores s_t = scale * (q . v_t), one softmax over all usable tokens, O = sum_t p_t v_t[0:512],
 * LSE natural log (QuantMLA page, appendix Figure 8: one global softmax, latent readout). */
static void attend_rows(int H, const uint16_t* q_lat_b, const uint16_t* q_rope_b, const double* V,
                        const char* ok, int T, float softmax_scale, double* out_b, double* lse_b) {
#pragma omp parallel for schedule(dynamic)
  for (int h = 0; h < H; ++h) {
    double q[ROW];
    for (int k = 0; k < LATENT; ++k) q[k] = oracle_bf16_to_double(q_lat_b[(size_t)h * LATENT + k]);
    for (int j = 0; j < ROPE; ++j) q[LATENT + j] = oracle_bf16_to_double(q_rope_b[(size_t)h * ROPE + j]);
    double* o = out_b + (size_t)h * LATENT;
    for (int k = 0; k < LATENT; ++k) o[k] = 0.0;
    double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double m = -INFINITY;
    int any = 0;
    for (int t = 0; t < T; ++t) {
      if (!ok[t]) continue;
      const double* v = V + (size_t)t * ROW;
      double dot = 0.0;
      for (int k = 0; k < ROW; ++k) dot += q[k] * v[k];
      s[t] = (double)softmax_scale * dot;
      if (!any || s[t] > m) m = s[t];
      any = 1;
    }
    if (!any) {
      lse_b[h] = -INFINITY;
    } else {
      double l = 0.0;
      for (int t = 0; t < T; ++t) {
        if (!ok[t]) continue;
        double w = exp(s[t] - m);
        l += w;
        const double* v = V + (size_t)t * ROW;
        for (int k = 0; k < LATENT; ++k) o[k] += w * v[k];
      }
      for (int k = 0; k < LATENT; ++k) o[k] /= l;
      lse_b[h] = m + log(l);
    }
    free(s);
  }
}

int oracle_decode(const oracle_config* cfg, int B, int H, const uint16_t* q_lat,
                  const uint16_t* q_rope, const int32_t* page_table, int max_pages,
                  const int32_t* seq_lens, const uint8_t* pool, int64_t n_pages,
                  const uint16_t* sink, const uint16_t* ring, float softmax_scale, double* out,
                  double* lse) {
  int flags = 0;
  for (int b = 0; b < B; ++b) {
    int T = seq_lens[b];
    if (T < 0 || (int64_t)T > (int64_t)max_pages * cfg->page_size) {
      flags |= ERR_SEQ_OVERFLOW;
      T = 0;
    }
    double* V = (double*)malloc(sizeof(double) * ((size_t)(T > 0 ? T : 1)) * ROW);
    char* ok = (char*)malloc((size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) {
      int r = oracle_token_values(cfg, b, t, T, page_table, max_pages, pool, n_pages, sink, ring,
                                  V + (size_t)t * ROW);
      ok[t] = r >= 0;
      if (r < 0) flags |= ERR_BAD_PAGE;
    }
    attend_rows(H, q_lat + (size_t)b * H * LATENT, q_rope + (size_t)b * H * ROPE, V, ok, T, softmax_scale,
                out + (size_t)b * H * LATENT, lse + (size_t)b * H);
    free(V);
    free(ok);
  }
  return flags;
}

/* The unquantized comparator: the same attention over a paged BF16 cache, token t of sequence
 * b in row t % P of page page_table[b][t / P] of kv_pool [n_pages][P][576] (c then k_R). */
int oracle_decode_bf16(int B, int H, const uint16_t* q_lat, const uint16_t* q_rope,
                       const int32_t* page_table, int max_pages, int page_size, const int32_t* seq_lens,
                       const uint16_t* kv_pool, int64_t n_pages, float softmax_scale, double* out,
                       double* lse) {
  int flags = 0;
  for (int b = 0; b < B; ++b) {
    int T = seq_lens[b];
    if (T < 0 || (int64_t)T > (int64_t)max_pages * page_size) {
      flags |= ERR_SEQ_OVERFLOW;
      T = 0;
    }
    double* V = (double*)malloc(sizeof(double) * ((size_t)(T > 0 ? T : 1)) * ROW);
    char* ok = (char*)malloc((size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) {
      const int32_t pid = page_table[(size_t)b * max_pages + t / page_size];
      ok[t] = pid >= 0 && pid < n_pages;
      if (!ok[t]) {
        flags |= ERR_BAD_PAGE;
        continue;
      }
      const uint16_t* row = kv_pool + ((size_t)pid * page_size + (size_t)(t % page_size)) * ROW;
      for (int k = 0; k < ROW; ++k) V[(size_t)t * ROW + k] = oracle_bf16_to_double(row[k]);
    }
    attend_rows(H, q_lat + (size_t)b * H * LATENT, q_rope + (size_t)b * H * ROPE, V, ok, T, softmax_scale,
                out + (size_t)b * H * LATENT, lse + (size_t)b * H);
    free(V);
    free(ok);
  }
  return flags;
}

/* ---------------------------------------------------------------- cached-tensor transforms */

/* Round a float to BF16, to nearest with ties to even (the upper 16 bits of binary32 after
   adding half of the dropped part's unit, biased towards the even result); NaN stays NaN. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* RAQ-MLA page, Figure 4: before a token is cached, its latent is mapped to c A_c (after the
   RMSNorm) and its positional key to k_R A_R (after RoPE); the read path compensates with the
   inverses on the weights / query side, so the cache simply holds the transformed rows.
   Reading taken (the page fixes no arithmetic): the transform is a BF16 matrix A [dim][dim]
   applied to a BF16 row x as x'_j = sum_i x_i A[i][j], the sum accumulated in float32 in the
   order i = 0, 1, ..., dim-1 starting from +0 (a BF16 x BF16 product is exact in float32, so
   each step rounds once), then rounded to BF16 to nearest-even. acc_out (nullable) receives
   the float32 sums before that rounding. */
void oracle_row_transform(int n_rows, int dim, const uint16_t* x, const uint16_t* a, float* acc_out,
                          uint16_t* out) {
  for (int r = 0; r < n_rows; ++r) {
    const uint16_t* xr = x + (size_t)r * dim;
    for (int j = 0; j < dim; ++j) {
      float acc = 0.0f;
      for (int i = 0; i < dim; ++i) {
        const float prod = bf16_to_f32(xr[i]) * bf16_to_f32(a[(size_t)i * dim + j]);
        acc = acc + prod;
      }
      if (acc_out) acc_out[(size_t)r * dim + j] = acc;
      out[(size_t)r * dim + j] = f32_to_bf16_rne(acc);
    }
  }
}

/* Threads of the parallel loops over heads (timing of the oracle only: every head's result is
 * computed by one thread in the same order whatever the count). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
