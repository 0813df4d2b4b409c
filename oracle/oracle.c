/*
 * CPU ORACLE for the H3 attention step -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg load this
 * file.  The CUDA library never links, includes or calls it, and it shares no
 * code with the CUDA library.  It is plain, slow and written to be checked
 * by eye against the method's definition:
 *
 *   1. Q/K RMSNorm per (token, head) row of D channels (FastVideo PR #1832,
 *      "Preserve H3-specific attention behavior": H3 applies Q/K RMSNorm
 *      before attention; TeleFuser PR #37 section 2.2 step 1).
 *   2. A bf16 rounding boundary after the norm (TeleFuser PR #37 section 2.2
 *      step 2, "BF16-compatible rounding"; section 2.5: BF16 store/load
 *      rounding boundaries are preserved).
 *   3. Partial rotate-half RoPE over the first rotary_dim of D channels
 *      (FastVideo PR #1832, "Preserve H3-specific attention behavior": 96 of
 *      128 channels rotated; TeleFuser PR #37 section 2.2 step 3).
 *   4. Dense prefill attention softmax(Q K^T * scale) V on BSHD tensors with
 *      GQA, cross-attention, causal, key-padding and boolean [Q, K] mask
 *      variants (FastVideo PR #1832, "Summary"; FastVideo PR #1799,
 *      "Implementation").
 *   5. RMSNorm of a DiT hidden row followed by indexed AdaLN scale/shift
 *      modulation, keeping the bf16 store/load boundaries of the unfused
 *      norm-then-modulate path (TeleFuser PR #37 section 2.5).
 *
 * Precision: every step of the definition runs in double precision (fp64);
 * bf16 inputs widen exactly.  The one exception is
 * oracle_qk_norm_rope_emulate_bf16, a float32 emulation of the norm/RoPE
 * step in a fixed operation order; its rounding behaviour is the contract a
 * CUDA kernel has to reproduce bit for bit.
 *
 * Build with -ffp-contract=off so that no multiply-add is fused behind the
 * source's back; every fused multiply-add below is an explicit fma/fmaf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ */
/* bf16 helpers                                                        */
/* ------------------------------------------------------------------ */
static inline double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* float -> bf16, round to nearest, ties to even (IEEE 754 default rounding
   applied to an 8-bit significand).  NaN -> canonical quiet NaN. */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* double -> bf16 value, rounded once (no intermediate float), ties to even.
   bf16: 8 significant bits, exponent range of float (normal >= 2^-126,
   subnormal quantum 2^-133, largest finite (2 - 2^-7) * 2^127). */
static double round_f64_to_bf16(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double ax = fabs(x);
  int e;
  frexp(ax, &e); /* ax = m * 2^e, m in [0.5, 1) */
  int q_exp = e - 8; /* quantum 2^(e-8): 8 significant bits */
  if (q_exp < -133) q_exp = -133;
  double r = ldexp(nearbyint(ldexp(ax, -q_exp)), q_exp); /* nearbyint: ties to even */
  double maxf = ldexp(2.0 - ldexp(1.0, -7), 127);
  if (r > maxf) r = INFINITY;
  return x < 0 ? -r : r;
}

static uint16_t f64_to_bf16_bits(double x) {
  double r = round_f64_to_bf16(x);
  float f = (float)r; /* exact: r is representable in bf16, hence in float */
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(r)) return 0x7FC0;
  return (uint16_t)(u >> 16);
}

void oracle_round_f64_to_bf16(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f64_to_bf16_bits(in[i]);
}

static int auto_threads(int n) {
  if (n > 0) return n;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  if (c < 1) c = 1;
  if (c > 64) c = 64;
  return (int)c;
}

typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct {
  range_fn fn;
  void* ctx;
  int64_t begin, end;
} range_job;

static void* range_worker(void* a) {
  range_job* j = (range_job*)a;
  j->fn(j->ctx, j->begin, j->end);
  return NULL;
}

/* Split [0, n) into contiguous ranges, one per thread. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
  int nt = auto_threads(nthreads);
  if (nt > n) nt = n > 0 ? (int)n : 1;
  pthread_t th[64];
  range_job jobs[64];
  for (int t = 0; t < nt; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].begin = n * t / nt;
    jobs[t].end = n * (t + 1) / nt;
  }
  for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, range_worker, &jobs[t]);
  range_worker(&jobs[0]);
  for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* 1-3. Q/K RMSNorm -> bf16 boundary -> partial rotate-half RoPE, fp64  */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint16_t* x;
  double* y;
  int S, H, D;
  const float* w;
  const float* cos_t;
  const float* sin_t;
  int rotary_dim;
  double eps;
  int round_boundary;
} nr64_ctx;

static void nr64_rows(void* p, int64_t r0, int64_t r1) {
  const nr64_ctx* c = (const nr64_ctx*)p;
  int D = c->D, half = c->rotary_dim / 2;
  double* n = (double*)malloc(sizeof(double) * (size_t)D);
  for (int64_t r = r0; r < r1; ++r) {
    const uint16_t* xr = c->x + r * D;
    double* yr = c->y + r * D;
    int64_t pos = (r / c->H) % c->S; /* row r = ((b * S + s) * H + h) */
    /* RMSNorm: ms = mean of squares over the row; r = 1/sqrt(ms + eps). */
    double ss = 0.0;
    for (int d = 0; d < D; ++d) {
      double xd = bf16_to_f64(xr[d]);
      ss += xd * xd;
    }
    double ms = ss / (double)D;
    double rinv = 1.0 / sqrt(ms + c->eps);
    for (int d = 0; d < D; ++d) {
      double v = bf16_to_f64(xr[d]) * rinv * (double)c->w[d];
      n[d] = c->round_boundary ? round_f64_to_bf16(v) : v; /* bf16 boundary */
    }
    /* Rotate-half RoPE on pairs (i, i + half), i < half: rotation of the
       point (n_i, n_{i+half}) by the angle whose cosine/sine the table holds. */
    for (int i = 0; i < half; ++i) {
      double a = n[i], b = n[i + half];
      double cs = (double)c->cos_t[pos * half + i];
      double sn = (double)c->sin_t[pos * half + i];
      yr[i] = a * cs - b * sn;
      yr[i + half] = b * cs + a * sn;
    }
    for (int d = 2 * half; d < D; ++d) yr[d] = n[d]; /* channels past rotary_dim pass through */
  }
  free(n);
}

/* x: bf16 [rows, D] with rows = B*S*H in BSHD order; w: [D]; cos/sin:
   [S, rotary_dim/2] (row = position s).  y: fp64 [rows, D], the value before
   the final bf16 store.  round_boundary = 1 applies the bf16 boundary between
   norm and RoPE (the method); 0 skips it (used by exact-math checks). */
void oracle_qk_norm_rope_f64(const uint16_t* x, double* y, int64_t rows, int S, int H, int D,
                             const float* w, const float* cos_t, const float* sin_t, int rotary_dim,
                             double eps, int round_boundary, int nthreads) {
  nr64_ctx c = {x, y, S, H, D, w, cos_t, sin_t, rotary_dim, eps, round_boundary};
  parallel_for(rows, nthreads, nr64_rows, &c);
}

/* ------------------------------------------------------------------ */
/* The same step in float32 with a fixed operation order (the bit-exact  */
/* contract for a CUDA implementation):                                  */
/*   8-channel groups g = 0 .. D/8-1; h8 = floor(rotary_dim/16);         */
/*   L = D/16 lanes, each holding two groups: first group g0 = l (l < h8) */
/*   or L + l (l >= h8), second group g1 = l + h8 (every group exactly     */
/*   once for any h8 in 0..L; when 16 divides rotary_dim a lane l < h8    */
/*   holds the rotation pair (l, l + h8));                                */
/*   per lane acc = 0; acc = fmaf(x, x, acc) over the 8 channels of g0 in */
/*   order, then those of g1;                                             */
/*   butterfly over lanes: for off = L/2 .. 1: p[l] = p[l] + p[l ^ off];   */
/*   ms = sum * (1/D) (exact power-of-two scaling);                       */
/*   r = 1 / sqrtf(ms + eps), each operation IEEE correctly rounded;      */
/*   n = (x * r) * w, two rounded multiplies; n^ = bf16(n);               */
/*   y_i = fmaf(a, c, -(b * s)), y_{i+half} = fmaf(b, c, a * s);          */
/*   output bf16(y) with round to nearest even.                           */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint16_t* x;
  uint16_t* out;
  int S, H, D;
  const float* w;
  const float* cos_t;
  const float* sin_t;
  int rotary_dim;
  float eps;
} nr32_ctx;

static void nr32_rows(void* p, int64_t r0, int64_t r1) {
  const nr32_ctx* c = (const nr32_ctx*)p;
  int D = c->D, half = c->rotary_dim / 2, L = D / 16, h8 = c->rotary_dim / 16;
  float part[32];
  float nh[256];
  float y[256];
  for (int64_t r = r0; r < r1; ++r) {
    const uint16_t* xr = c->x + r * D;
    int64_t pos = (r / c->H) % c->S;
    for (int l = 0; l < L; ++l) {
      int g0 = l < h8 ? l : L + l;
      int g1 = l + h8;
      float acc = 0.0f;
      for (int e = 0; e < 8; ++e) {
        float xv = bf16_to_f32(xr[8 * g0 + e]);
        acc = fmaf(xv, xv, acc);
      }
      for (int e = 0; e < 8; ++e) {
        float xv = bf16_to_f32(xr[8 * g1 + e]);
        acc = fmaf(xv, xv, acc);
      }
      part[l] = acc;
    }
    for (int off = L / 2; off >= 1; off /= 2) {
      float nxt[32];
      for (int l = 0; l < L; ++l) nxt[l] = part[l] + part[l ^ off];
      memcpy(part, nxt, sizeof(float) * (size_t)L);
    }
    float ms = part[0] * (1.0f / (float)D);
    float rinv = 1.0f / sqrtf(ms + c->eps);
    for (int d = 0; d < D; ++d) {
      float t = bf16_to_f32(xr[d]) * rinv;
      float v = t * c->w[d];
      nh[d] = bf16_to_f32(f32_to_bf16_rne(v));
    }
    for (int d = 0; d < D; ++d) y[d] = nh[d];
    for (int i = 0; i < half; ++i) {
      float a = nh[i], b = nh[i + half];
      float cs = c->cos_t[pos * half + i], sn = c->sin_t[pos * half + i];
      float bs = b * sn;
      float as = a * sn;
      y[i] = fmaf(a, cs, -bs);
      y[i + half] = fmaf(b, cs, as);
    }
    for (int d = 0; d < D; ++d) c->out[r * D + d] = f32_to_bf16_rne(y[d]);
  }
}

void oracle_qk_norm_rope_emulate_bf16(const uint16_t* x, uint16_t* out, int64_t rows, int S, int H,
                                      int D, const float* w, const float* cos_t, const float* sin_t,
                                      int rotary_dim, float eps, int nthreads) {
  nr32_ctx c = {x, out, S, H, D, w, cos_t, sin_t, rotary_dim, eps};
  parallel_for(rows, nthreads, nr32_rows, &c);
}

/* ------------------------------------------------------------------ */
/* 5. RMSNorm -> indexed AdaLN scale/shift modulation                   */
/*                                                                      */
/* The unfused path it replaces, with a bf16 store after every step:    */
/*   n = bf16(x * r * w)          r = 1/sqrt(mean_c(x_c^2) + eps)        */
/*   a = bf16(1 + scale[idx[t]])  m = bf16(n * a)                        */
/*   y = bf16(m + shift[idx[t]])                                         */
/* w is optional (absent = 1).  Rows whose index is outside [0, N) are   */
/* written as zeros.                                                     */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint16_t* x;
  uint16_t* y;
  int C, N;
  const float* w;
  const uint16_t* scale;
  const uint16_t* shift;
  const int32_t* idx;
  double eps;
  float epsf;
} mod_ctx;

/* Definition in fp64: every bf16 boundary rounds the exact value once. */
static void mod64_rows(void* p, int64_t r0, int64_t r1) {
  const mod_ctx* c = (const mod_ctx*)p;
  int C = c->C;
  for (int64_t t = r0; t < r1; ++t) {
    const uint16_t* xr = c->x + t * C;
    uint16_t* yr = c->y + t * C;
    int32_t ix = c->idx ? c->idx[t] : 0;
    if (ix < 0 || ix >= c->N) {
      for (int ch = 0; ch < C; ++ch) yr[ch] = 0;
      continue;
    }
    double ss = 0.0;
    for (int ch = 0; ch < C; ++ch) {
      double v = bf16_to_f64(xr[ch]);
      ss += v * v;
    }
    double rinv = 1.0 / sqrt(ss / (double)C + c->eps);
    const uint16_t* sc = c->scale + (int64_t)ix * C;
    const uint16_t* sh = c->shift + (int64_t)ix * C;
    for (int ch = 0; ch < C; ++ch) {
      double n = round_f64_to_bf16(bf16_to_f64(xr[ch]) * rinv * (c->w ? (double)c->w[ch] : 1.0));
      double a = round_f64_to_bf16(1.0 + bf16_to_f64(sc[ch]));
      double m = round_f64_to_bf16(n * a);
      yr[ch] = f64_to_bf16_bits(m + bf16_to_f64(sh[ch]));
    }
  }
}

void oracle_rmsnorm_modulate_f64(const uint16_t* x, uint16_t* y, int64_t T, int C, const float* w,
                                 const uint16_t* scale, const uint16_t* shift, const int32_t* idx, int N,
                                 double eps, int nthreads) {
  mod_ctx c = {x, y, C, N, w, scale, shift, idx, eps, (float)eps};
  parallel_for(T, nthreads, mod64_rows, &c);
}

/* The same step in float32 with a fixed operation order (the bit-exact    */
/* contract for a CUDA implementation):                                    */
/*   8-channel groups g = 0 .. C/8-1; group g belongs to lane g mod 32;    */
/*   per lane acc = 0; acc = fmaf(x, x, acc) over its groups in increasing */
/*   g, channels in order; butterfly over the 32 lanes: for off = 16 .. 1: */
/*   p[l] = p[l] + p[l ^ off];  ms = sum / C;  r = 1 / sqrtf(ms + eps)     */
/*   (each operation IEEE correctly rounded);  n = bf16((x * r) * w)       */
/*   (n = bf16(x * r) without w);  a = bf16(1 + s);  m = bf16(n * a);       */
/*   y = bf16(m + sh), every rounding to nearest even.                     */
static void mod32_rows(void* p, int64_t r0, int64_t r1) {
  const mod_ctx* c = (const mod_ctx*)p;
  int C = c->C, G = C / 8;
  float part[32];
  for (int64_t t = r0; t < r1; ++t) {
    const uint16_t* xr = c->x + t * C;
    uint16_t* yr = c->y + t * C;
    int32_t ix = c->idx ? c->idx[t] : 0;
    if (ix < 0 || ix >= c->N) {
      for (int ch = 0; ch < C; ++ch) yr[ch] = 0;
      continue;
    }
    for (int l = 0; l < 32; ++l) {
      float acc = 0.0f;
      for (int g = l; g < G; g += 32)
        for (int e = 0; e < 8; ++e) {
          float xv = bf16_to_f32(xr[8 * g + e]);
          acc = fmaf(xv, xv, acc);
        }
      part[l] = acc;
    }
    for (int off = 16; off >= 1; off /= 2) {
      float nxt[32];
      for (int l = 0; l < 32; ++l) nxt[l] = part[l] + part[l ^ off];
      memcpy(part, nxt, sizeof(part));
    }
    float ms = part[0] / (float)C;
    float rinv = 1.0f / sqrtf(ms + c->epsf);
    const uint16_t* sc = c->scale + (int64_t)ix * C;
    const uint16_t* sh = c->shift + (int64_t)ix * C;
    for (int ch = 0; ch < C; ++ch) {
      float v = bf16_to_f32(xr[ch]) * rinv;
      if (c->w) v = v * c->w[ch];
      float n = bf16_to_f32(f32_to_bf16_rne(v));
      float a = bf16_to_f32(f32_to_bf16_rne(1.0f + bf16_to_f32(sc[ch])));
      float m = bf16_to_f32(f32_to_bf16_rne(n * a));
      yr[ch] = f32_to_bf16_rne(m + bf16_to_f32(sh[ch]));
    }
  }
}

void oracle_rmsnorm_modulate_emulate_bf16(const uint16_t* x, uint16_t* y, int64_t T, int C, const float* w,
                                          const uint16_t* scale, const uint16_t* shift, const int32_t* idx,
                                          int N, float eps, int nthreads) {
  mod_ctx c = {x, y, C, N, w, scale, shift, idx, (double)eps, eps};
  parallel_for(T, nthreads, mod32_rows, &c);
}

/* ------------------------------------------------------------------ */
/* 4. Dense prefill attention, fp64, one output row at a time          */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint16_t *q, *k, *v;
  int B, Sq, Sk, Hq, Hkv, D;
  double scale;
  int causal;
  const int32_t* kv_len;   /* [B] or NULL */
  const int32_t* q_len;    /* [B] or NULL */
  const uint8_t* causal_b; /* [B] or NULL */
  const uint32_t* bits;    /* [B, Sq, ceil(Sk/32)] or NULL */
  const int64_t* row_ids;  /* flat BSHD row ids ((b*Sq + i)*Hq + h), or NULL for all rows */
  double* out;             /* [nrows, D] */
  /* chunked window (self-attention): 0 tokens per chunk = no window */
  int64_t win_af;          /* anchor tokens: anchor_frames * frame_tokens */
  int64_t win_ct;          /* tokens per chunk: chunk_frames * frame_tokens */
  int64_t win_r;           /* radius in chunks */
} att_ctx;

/* Chunked window with anchor frames (SGLang PR #37903, "Modifications",
   hybrid_window_attn_h3: chunk-5 / radius-1 window with anchor frames,
   dense-query rows against all keys; "Accuracy Tests": the anchor frames
   shift the chunk grid).  Rows and keys of the anchor frames are dense; any
   other query in chunk c = (i - af) / ct attends the keys of chunks
   c - r .. c + r. */
static int window_allows(int64_t af, int64_t ct, int64_t r, int64_t i, int64_t j) {
  if (ct <= 0 || i < af || j < af) return 1;
  int64_t d = (i - af) / ct - (j - af) / ct;
  return d <= r && d >= -r;
}

/* Whether query row i of sample b may attend key j. */
static int allowed(const att_ctx* c, int b, int64_t i, int64_t j) {
  if (j >= c->Sk) return 0;
  if (c->kv_len && j >= (int64_t)c->kv_len[b]) return 0;
  int causal = c->causal || (c->causal_b && c->causal_b[b]);
  if (causal && j > i) return 0;
  if (c->bits) {
    int64_t W = (c->Sk + 31) / 32;
    uint32_t word = c->bits[((int64_t)b * c->Sq + i) * W + (j >> 5)];
    if (!((word >> (j & 31)) & 1u)) return 0;
  }
  if (!window_allows(c->win_af, c->win_ct, c->win_r, i, j)) return 0;
  return 1;
}

static void att_rows(void* p, int64_t r0, int64_t r1) {
  const att_ctx* c = (const att_ctx*)p;
  int D = c->D, g = c->Hq / c->Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)c->Sk);
  int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)c->Sk);
  double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
  for (int64_t r = r0; r < r1; ++r) {
    int64_t row = c->row_ids ? c->row_ids[r] : r;
    int h = (int)(row % c->Hq);
    int64_t i = (row / c->Hq) % c->Sq;
    int b = (int)(row / ((int64_t)c->Hq * c->Sq));
    int kvh = h / g; /* GQA: query heads [kvh*g, (kvh+1)*g) share kv head kvh */
    double* o = c->out + r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (c->q_len && i >= (int64_t)c->q_len[b]) continue; /* zero tail */
    const uint16_t* qr = c->q + row * D;
    for (int d = 0; d < D; ++d) qrow[d] = bf16_to_f64(qr[d]);
    /* Scores over the allowed keys only: a disallowed key is skipped, never
       multiplied by zero, so its K/V contents cannot reach the output. */
    int64_t n = 0;
    for (int64_t j = 0; j < c->Sk; ++j) {
      if (!allowed(c, b, i, j)) continue;
      const uint16_t* kr = c->k + (((int64_t)b * c->Sk + j) * c->Hkv + kvh) * D;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qrow[d] * bf16_to_f64(kr[d]);
      s[n] = c->scale * dot;
      idx[n] = j;
      ++n;
    }
    if (n == 0) continue; /* fully masked row -> 0 */
    double m = s[0];
    for (int64_t t = 1; t < n; ++t)
      if (s[t] > m) m = s[t];
    double denom = 0.0;
    for (int64_t t = 0; t < n; ++t) {
      s[t] = exp(s[t] - m);
      denom += s[t];
    }
    for (int64_t t = 0; t < n; ++t) {
      const uint16_t* vr = c->v + (((int64_t)b * c->Sk + idx[t]) * c->Hkv + kvh) * D;
      double pw = s[t] / denom;
      for (int d = 0; d < D; ++d) o[d] += pw * bf16_to_f64(vr[d]);
    }
  }
  free(s);
  free(idx);
  free(qrow);
}

/* q: bf16 [B, Sq, Hq, D]; k, v: bf16 [B, Sk, Hkv, D]; out: fp64 [nrows, D]
   for the rows listed in row_ids (flat ids into the BSHD output), or for all
   B*Sq*Hq rows in order when row_ids is NULL. */
void oracle_attention_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Sq,
                          int Sk, int Hq, int Hkv, int D, double scale, int causal,
                          const int32_t* kv_len, const int32_t* q_len, const uint8_t* causal_b,
                          const uint32_t* bits, const int64_t* row_ids, int64_t nrows, double* out,
                          int nthreads) {
  att_ctx c = {q, k, v, B, Sq, Sk, Hq, Hkv, D, scale, causal, kv_len, q_len, causal_b, bits, row_ids, out, 0, 0, 0};
  int64_t n = row_ids ? nrows : (int64_t)B * Sq * Hq;
  parallel_for(n, nthreads, att_rows, &c);
}

/* Self-attention under the chunked window (plus optional key padding and
   zero tail): frame_tokens F, anchor_frames A, chunk_frames K, radius r. */
void oracle_attention_window_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int S,
                                 int Hq, int Hkv, int D, double scale, int frame_tokens, int anchor_frames,
                                 int chunk_frames, int radius, const int32_t* kv_len, const int32_t* q_len,
                                 const int64_t* row_ids, int64_t nrows, double* out, int nthreads) {
  att_ctx c = {q, k, v, B, S, S, Hq, Hkv, D, scale, 0, kv_len, q_len, NULL, NULL, row_ids, out,
               (int64_t)anchor_frames * frame_tokens, (int64_t)chunk_frames * frame_tokens, radius};
  int64_t n = row_ids ? nrows : (int64_t)B * S * Hq;
  parallel_for(n, nthreads, att_rows, &c);
}

/* Allowed (query row, key) pairs of one sample under the window and key
   padding L: per row, the anchor keys plus the keys of the row's chunk
   window, counted by intervals. */
int64_t oracle_window_allowed_pairs(int S, int L, int frame_tokens, int anchor_frames, int chunk_frames,
                                    int radius) {
  int64_t af = (int64_t)anchor_frames * frame_tokens, ct = (int64_t)chunk_frames * frame_tokens;
  int64_t total = 0;
  if (L > S) L = S;
  if (L < 0) L = 0;
  for (int64_t i = 0; i < S; ++i) {
    if (i < af) {
      total += L;
      continue;
    }
    int64_t ci = (i - af) / ct;
    int64_t lo = af + (ci - radius) * ct, hi = af + (ci + radius + 1) * ct;
    if (lo < af) lo = af;
    if (hi > L) hi = L;
    total += (af < L ? af : L) + (hi > lo ? hi - lo : 0);
  }
  return total;
}

/* Number of allowed (i, j) pairs, summed over samples and query rows (times
   nothing per head): the algorithmic work count of the attention step is
   4 * D * Hq * pairs flops. */
int64_t oracle_allowed_pairs(int B, int Sq, int Sk, int causal, const int32_t* kv_len,
                             const int32_t* q_len, const uint8_t* causal_b) {
  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    int64_t L = Sk;
    if (kv_len && kv_len[b] < L) L = kv_len[b];
    if (L < 0) L = 0;
    int64_t rows = Sq;
    if (q_len && q_len[b] < rows) rows = q_len[b] < 0 ? 0 : q_len[b];
    int cz = causal || (causal_b && causal_b[b]);
    for (int64_t i = 0; i < rows; ++i) {
      int64_t lim = L;
      if (cz && i + 1 < lim) lim = i + 1;
      total += lim;
    }
  }
  return total;
}
