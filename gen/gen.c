/*
 * Seeded synthetic inputs for the MoE-layer forward pass.
 *
 * This file draws the layer's inputs (token activations x, router weights,
 * expert weights, router bias) and nothing else: it holds none of the layer's
 * arithmetic.  The same values feed the CUDA path and the CPU oracle.
 *
 * Generator definition (counter based, so any element can be drawn on its own
 * and any thread split gives the same bits):
 *   mix64(z)      : the splitmix64 finaliser
 *                   z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                   z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(seed,tid) = mix64(seed ^ (tid * 0xD1B54A32D192ED03))
 *   u64(seed,tid,i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 *   uniform(..)   = ((u64 >> 11) + 1) * 2^-53            in (0, 1]
 * Normal deviates come from Box-Muller on pair p = i/2:
 *   u1 = uniform(seed, tid, 2p), u2 = uniform(seed, tid, 2p+1)
 *   r  = sqrt(-2 ln u1); element 2p = r cos(2 pi u2), element 2p+1 = r sin(2 pi u2)
 * ln, sin and cos are evaluated here with fixed series in plain IEEE double
 * arithmetic (no libm, no contraction) so that x86-64 and AArch64 hosts draw
 * identical bits.  Values are scaled by the requested standard deviation and
 * rounded to bfloat16 (round to nearest, ties to even; |v| < 2^-126 flushes to
 * a signed zero, which a N(0, s^2) draw at these scales never reaches).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(seed ^ (tid * 0xD1B54A32D192ED03ull));
}

static inline double uniform01(uint64_t key, uint64_t i) {
  uint64_t z = mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
  return (double)((z >> 11) + 1) * (1.0 / 9007199254740992.0);
}

/* ln(u) for u in (0, 1]: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(s), s = (m-1)/(m+1), |s| < 0.172, 12 odd terms. */
static double LOG_C[12];  /* 1/(2n+1), n = 0..11 */
static double SIN_C[10];  /* -1/((2n+2)(2n+3)) */
static double COS_C[10];  /* -1/((2n+1)(2n+2)) */
static pthread_once_t coef_once = PTHREAD_ONCE_INIT;

static void init_coefficients(void) {
  for (int n = 0; n < 12; ++n) LOG_C[n] = 1.0 / (double)(2 * n + 1);
  for (int n = 0; n < 10; ++n) {
    SIN_C[n] = -1.0 / (double)((2 * n + 2) * (2 * n + 3));
    COS_C[n] = -1.0 / (double)((2 * n + 1) * (2 * n + 2));
  }
}

static double series_log(double u) {
  int e = 0;
  double m = frexp(u, &e); /* m in [0.5, 1), exact */
  if (m < 0.70710678118654752) {
    m *= 2.0;
    e -= 1;
  }
  double s = (m - 1.0) / (m + 1.0);
  double s2 = s * s;
  double acc = LOG_C[11];
  for (int n = 10; n >= 0; --n) acc = acc * s2 + LOG_C[n];
  return 2.0 * s * acc + (double)e * 0.69314718055994530942;
}

/* sin and cos of 2*pi*x for x in [0, 1). Reduce to phi in [-pi/4, pi/4] by
 * quarter turns, then Taylor series to phi^19 / phi^18 (coefficients
 * 1/((2n+2)(2n+3)) and 1/((2n+1)(2n+2)) computed once at start-up). */
static void series_sincos_turns(double x, double* s_out, double* c_out) {
  double q = floor(4.0 * x + 0.5); /* 0..4 */
  double r = x - 0.25 * q;         /* [-1/8, 1/8] turns, exact */
  double phi = r * 6.28318530717958647692;
  double p2 = phi * phi;
  double sn = 0.0, cs = 0.0, ts = phi, tc = 1.0;
  for (int n = 0; n < 10; ++n) {
    sn += ts;
    cs += tc;
    ts *= p2 * SIN_C[n];
    tc *= p2 * COS_C[n];
  }
  int quad = ((int)q) & 3;
  switch (quad) {
    case 0: *s_out = sn; *c_out = cs; break;
    case 1: *s_out = cs; *c_out = -sn; break;
    case 2: *s_out = -sn; *c_out = -cs; break;
    default: *s_out = -cs; *c_out = sn; break;
  }
}

static inline uint16_t to_bf16(double v) {
  uint64_t b;
  memcpy(&b, &v, 8);
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  int exp = (int)((b >> 52) & 0x7FF) - 1023;
  if (exp < -126) return sign; /* below the normal bf16 range */
  uint64_t man = b & ((1ull << 52) - 1);
  uint64_t keep = man >> 45;          /* top 7 mantissa bits */
  uint64_t rest = man & ((1ull << 45) - 1);
  uint64_t half = 1ull << 44;
  if (rest > half || (rest == half && (keep & 1))) {
    keep += 1;
    if (keep == 128) {
      keep = 0;
      exp += 1;
    }
  }
  return (uint16_t)(sign | ((uint16_t)(exp + 127) << 7) | (uint16_t)keep);
}

static void normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
  double u1 = uniform01(key, 2 * p);
  double u2 = uniform01(key, 2 * p + 1);
  double r = sqrt(-2.0 * series_log(u1));
  double s, c;
  series_sincos_turns(u2, &s, &c);
  *z0 = r * c;
  *z1 = r * s;
}

typedef struct {
  uint64_t key;
  uint64_t first;   /* tensor index of out[0] */
  uint64_t n;
  double scale;
  uint16_t* out_bf16;
  float* out_f32;
} job_t;

static void run_job(const job_t* j) {
  uint64_t i = 0;
  while (i < j->n) {
    uint64_t gi = j->first + i;
    uint64_t p = gi >> 1;
    double z0, z1;
    normal_pair(j->key, p, &z0, &z1);
    if ((gi & 1) == 0) {
      if (j->out_bf16) j->out_bf16[i] = to_bf16(z0 * j->scale);
      else j->out_f32[i] = (float)(z0 * j->scale);
      ++i;
      if (i >= j->n) break;
    }
    if (j->out_bf16) j->out_bf16[i] = to_bf16(z1 * j->scale);
    else j->out_f32[i] = (float)(z1 * j->scale);
    ++i;
  }
}

static void* job_thread(void* arg) {
  run_job((const job_t*)arg);
  return NULL;
}

static void fill(uint64_t seed, uint64_t tid, uint64_t first, uint64_t n, double scale,
                 uint16_t* ob, float* of, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < (1ull << 16)) threads = 1;
  job_t jobs[256];
  pthread_t th[256];
  pthread_once(&coef_once, init_coefficients);
  uint64_t key = stream_key(seed, tid);
  uint64_t chunk = (n + (uint64_t)threads - 1) / (uint64_t)threads;
  chunk = (chunk + 1) & ~1ull; /* even split points keep pairs whole */
  int used = 0;
  for (int t = 0; t < threads; ++t) {
    uint64_t a = (uint64_t)t * chunk;
    if (a >= n) break;
    uint64_t b = a + chunk < n ? a + chunk : n;
    jobs[t].key = key;
    jobs[t].first = first + a;
    jobs[t].n = b - a;
    jobs[t].scale = scale;
    jobs[t].out_bf16 = ob ? ob + a : NULL;
    jobs[t].out_f32 = of ? of + a : NULL;
    ++used;
  }
  if (used == 1) {
    run_job(&jobs[0]);
    return;
  }
  int started = 0;
  for (int t = 0; t < used; ++t) {
    if (pthread_create(&th[t], NULL, job_thread, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = started; t < used; ++t) run_job(&jobs[t]);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* out[i] = bf16(std * N_i) for tensor indices first .. first+n-1 of stream (seed, tid). */
void gen_normal_bf16(uint64_t seed, uint64_t tid, uint64_t first, uint64_t n, double std_dev,
                     uint16_t* out, int threads) {
  fill(seed, tid, first, n, std_dev, out, NULL, threads);
}

/* Same draw, kept in float32 (used for the router bias). */
void gen_normal_f32(uint64_t seed, uint64_t tid, uint64_t first, uint64_t n, double std_dev,
                    float* out, int threads) {
  fill(seed, tid, first, n, std_dev, NULL, out, threads);
}

/* Raw uniforms in (0, 1] (used for seeded permutations and shuffles). */
void gen_uniform_f64(uint64_t seed, uint64_t tid, uint64_t first, uint64_t n, double* out) {
  uint64_t key = stream_key(seed, tid);
  for (uint64_t i = 0; i < n; ++i) out[i] = uniform01(key, first + i);
}

/* Token rows of x: row t is drawn from stream (seed, TID_X + (retry[t] << 16))
 * at indices t*d .. t*d+d-1, so redrawing one row leaves the others intact. */
void gen_x_rows(uint64_t seed, uint64_t tid_x, int T, int d, const int32_t* retry, uint16_t* out,
                int threads) {
  if (retry == NULL) {
    fill(seed, tid_x, 0, (uint64_t)T * (uint64_t)d, 1.0, out, NULL, threads);
    return;
  }
  for (int t = 0; t < T; ++t) {
    uint64_t tid = tid_x + ((uint64_t)(uint32_t)retry[t] << 16);
    fill(seed, tid, (uint64_t)t * (uint64_t)d, (uint64_t)d, 1.0, out + (size_t)t * (size_t)d, NULL,
         1);
  }
}
