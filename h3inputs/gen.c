/*
 * Seeded synthetic inputs for the H3 attention step (QK-norm + partial RoPE,
 * then dense prefill attention).  Both sides of every comparison -- the CUDA
 * library and the CPU oracle -- are fed from here, so this file holds none of
 * the method's arithmetic: it only draws numbers and lays them out.
 *
 * Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; the finaliser
 * constants are the published "mix13" variant).  Draw k of stream
 * (seed, stream) is mix(base + (k + 1) * GAMMA), so any slice of a tensor can
 * be produced independently and in parallel.  Normal deviates come from the
 * Box-Muller transform (Box and Muller, Ann. Math. Statist. 1958) in double
 * precision, then round to float and to bf16 (round to nearest even).
 *
 * Build: plain C11 + pthreads, no architecture flags, so the x86 container and
 * the aarch64 GPU host build the same thing.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Base state of a stream: the seed and the stream id are mixed separately so
   that (seed, stream) pairs do not collide for small integers. */
static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return mix64(seed * GAMMA + 0x632BE59BD9B4E019ULL) ^ mix64(stream + 0x2545F4914F6CDD1DULL);
}

static inline uint64_t draw(uint64_t base, uint64_t k) { return mix64(base + (k + 1) * GAMMA); }

/* Uniform in the open interval (0, 1): 53 random bits, centred in the cell. */
static inline double u01(uint64_t base, uint64_t k) {
  return ((double)(draw(base, k) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal deviate k of the stream.  Pair p = k / 2 uses draws 2p and
   2p + 1; even k takes the cosine branch, odd k the sine branch. */
static inline double normal_at(uint64_t base, uint64_t k) {
  uint64_t p = k >> 1;
  double u1 = u01(base, 2 * p), u2 = u01(base, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (k & 1) ? r * sin(t) : r * cos(t);
}

/* float -> bf16 bits, round to nearest even; NaN -> canonical quiet NaN. */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int auto_threads(int n) {
  if (n > 0) return n;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  if (c < 1) c = 1;
  if (c > 64) c = 64;
  return (int)c;
}

/* ---- BSHD tensor of N(0, std) + optional per-(head, channel) offset ---- */
typedef struct {
  uint16_t* out;
  int64_t begin, end;
  int H, D;
  uint64_t base, off_base;
  double std, off_std;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  int64_t hd = (int64_t)j->H * j->D;
  for (int64_t e = j->begin; e < j->end; ++e) {
    double z = j->std * normal_at(j->base, (uint64_t)e);
    if (j->off_std != 0.0) {
      int64_t c = e % hd; /* (head, channel) index */
      z += j->off_std * normal_at(j->off_base, (uint64_t)c);
    }
    j->out[e] = f32_to_bf16((float)z);
  }
  return NULL;
}

/* out[b, s, h, d] = bf16( std * N_k + off_std * M_{h,d} ), k = flat index.
   M is one normal vector per (head, channel), drawn from stream + 2^32, shared
   by every token: the "per-head offset" of the long-sequence workload. */
void h3in_fill_bshd(uint16_t* out, int64_t B, int64_t S, int H, int D, uint64_t seed,
                    uint64_t stream, double std, double off_std, int nthreads) {
  int64_t n = B * S * (int64_t)H * D;
  int nt = auto_threads(nthreads);
  if (n < (1 << 16)) nt = 1;
  pthread_t th[64];
  fill_job jobs[64];
  for (int t = 0; t < nt; ++t) {
    jobs[t].out = out;
    jobs[t].begin = n * t / nt;
    jobs[t].end = n * (t + 1) / nt;
    jobs[t].H = H;
    jobs[t].D = D;
    jobs[t].base = stream_base(seed, stream);
    jobs[t].off_base = stream_base(seed, stream + (1ULL << 32));
    jobs[t].std = std;
    jobs[t].off_std = off_std;
  }
  for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
  fill_worker(&jobs[0]);
  for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
}

/* Uniform floats in [lo, hi): lo + (hi - lo) * u, computed in double, rounded once. */
void h3in_uniform_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, double lo, double hi) {
  uint64_t base = stream_base(seed, stream);
  for (int64_t k = 0; k < n; ++k) out[k] = (float)(lo + (hi - lo) * u01(base, (uint64_t)k));
}

/* Uniform integers in the closed range [lo, hi] (modulo reduction of 64 random
   bits; the bias is below 2^-40 for the ranges used here). */
void h3in_uniform_int(int32_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t lo, int64_t hi) {
  uint64_t base = stream_base(seed, stream);
  uint64_t span = (uint64_t)(hi - lo + 1);
  for (int64_t k = 0; k < n; ++k) out[k] = (int32_t)(lo + (int64_t)(draw(base, (uint64_t)k) % span));
}

/* Random boolean [Q, K] mask packed 32 keys per word: bit (j & 31) of word
   (row, j >> 5) is 1 with probability p (1 = the key may be attended).  Bits
   for j >= Sk are 0.  rows = B * Sq; words = ceil(Sk / 32). */
void h3in_bernoulli_bits(uint32_t* out, int64_t rows, int Sk, uint64_t seed, uint64_t stream, double p) {
  uint64_t base = stream_base(seed, stream);
  int64_t W = (Sk + 31) / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t w = 0; w < W; ++w) {
      uint32_t word = 0;
      for (int b = 0; b < 32; ++b) {
        int64_t j = w * 32 + b;
        if (j >= Sk) break;
        if (u01(base, (uint64_t)(r * (int64_t)Sk + j)) < p) word |= 1u << b;
      }
      out[r * W + w] = word;
    }
}

/* RoPE cache: cos/sin tables of shape [S, rotary_dim / 2] (row = position),
   angle(pos, i) = pos * theta^(-2 i / rotary_dim), evaluated in double with the
   host libm and rounded once to float.  The tables are an input of both the
   kernel and the oracle, exactly as a model hands its RoPE cache to the fused
   norm/RoPE kernel. */
void h3in_rope_tables(float* cos_out, float* sin_out, int64_t S, int rotary_dim, double theta) {
  int half = rotary_dim / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)rotary_dim);
    for (int64_t s = 0; s < S; ++s) {
      double a = (double)s * inv_freq;
      cos_out[s * half + i] = (float)cos(a);
      sin_out[s * half + i] = (float)sin(a);
    }
  }
}
