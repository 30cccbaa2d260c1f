/*
 * Seeded synthetic inputs for the asymmetric KV-cache workloads.
 *
 * This file generates random numbers and nothing else: it holds none of the
 * quantization or attention arithmetic.  Both the CPU oracle and the CUDA
 * library consume the host arrays it fills, so they always see the same bytes.
 *
 * Generator: a counter-based SplitMix64 stream per (seed, tensor, b, h).  The
 * k-th draw of a stream is the SplitMix64 output finaliser applied to
 * base + (k+1)*gamma, which is exactly the k-th output of the sequential
 * SplitMix64 generator started at `base`, so any element can be generated
 * independently of the others.  Element i = t*D + c of a stream takes pair
 * p = i/2 of Box-Muller normals (cos branch for even i, sin branch for odd i)
 * drawn from outputs 2p and 2p+1.  The value mean + std*z is formed in double
 * and rounded once to IEEE binary16 (round to nearest even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_stream_base(uint64_t seed, uint64_t tensor, uint64_t b, uint64_t h) {
  uint64_t a = mix64(seed * SYNTH_GAMMA + 0x632BE59BD9B4E019ULL);
  uint64_t k = mix64((tensor << 40) ^ (b << 20) ^ h ^ 0xA0761D6478BD642FULL);
  return mix64(a ^ k);
}

uint64_t synth_draw(uint64_t base, uint64_t k) { return mix64(base + (k + 1) * SYNTH_GAMMA); }

static inline double unit_open(uint64_t r) { return ((double)(r >> 11) + 0.5) * 0x1.0p-53; }

static inline void normal_pair(uint64_t base, uint64_t p, double* z0, double* z1) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = unit_open(synth_draw(base, 2 * p));
  double u2 = unit_open(synth_draw(base, 2 * p + 1));
  double rad = sqrt(-2.0 * log(u1));
  double ang = two_pi * u2;
  *z0 = rad * cos(ang);
  *z1 = rad * sin(ang);
}

static inline uint16_t to_half_bits(double x) {
  _Float16 h = (_Float16)x;
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

/* One standard normal for element i of a stream (exported for tests). */
double synth_normal(uint64_t base, uint64_t i) {
  double z0, z1;
  normal_pair(base, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

typedef struct {
  uint64_t seed, tensor;
  int64_t b0, nb, h0, nh, t0, nt, D;
  const double* mean; /* [nh][D] for heads h0..h0+nh-1 */
  const double* stdv; /* [nh][D] */
  uint16_t* out;      /* [nb][nh][nt][D] */
  int64_t row_begin, row_end; /* rows are (b, h, t) triples in output order */
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  const int64_t D = j->D;
  for (int64_t row = j->row_begin; row < j->row_end; ++row) {
    int64_t t = row % j->nt;
    int64_t bh = row / j->nt;
    int64_t h = bh % j->nh;
    int64_t b = bh / j->nh;
    uint64_t base = synth_stream_base(j->seed, j->tensor, (uint64_t)(j->b0 + b), (uint64_t)(j->h0 + h));
    const double* mu = j->mean + h * D;
    const double* sd = j->stdv + h * D;
    uint16_t* o = j->out + row * D;
    uint64_t i0 = (uint64_t)(j->t0 + t) * (uint64_t)D;
    for (int64_t c = 0; c < D; c += 2) {
      double z0, z1;
      normal_pair(base, (i0 + (uint64_t)c) >> 1, &z0, &z1);
      o[c] = to_half_bits(mu[c] + sd[c] * z0);
      o[c + 1] = to_half_bits(mu[c + 1] + sd[c + 1] * z1);
    }
  }
  return 0;
}

/*
 * Fill out[nb][nh][nt][D] (fp16 bits) with element (b, h, t, c) =
 * fp16(mean[h][c] + stdv[h][c] * z(seed, tensor, b0+b, h0+h, t0+t, c)).
 * D must be even.  Returns 0 on success, -1 on a bad argument.
 */
int synth_fill_f16(uint64_t seed, uint64_t tensor, int64_t b0, int64_t nb, int64_t h0, int64_t nh,
                   int64_t t0, int64_t nt, int64_t D, const double* mean, const double* stdv,
                   uint16_t* out, int threads) {
  if (D <= 0 || (D & 1) || nb < 0 || nh < 0 || nt < 0 || !mean || !stdv || !out) return -1;
  int64_t rows = nb * nh * nt;
  if (rows == 0) return 0;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if ((int64_t)threads > rows) threads = (int)rows;
  fill_job jobs[256];
  pthread_t tid[256];
  for (int k = 0; k < threads; ++k) {
    fill_job* j = &jobs[k];
    j->seed = seed; j->tensor = tensor;
    j->b0 = b0; j->nb = nb; j->h0 = h0; j->nh = nh; j->t0 = t0; j->nt = nt; j->D = D;
    j->mean = mean; j->stdv = stdv; j->out = out;
    j->row_begin = rows * k / threads;
    j->row_end = rows * (k + 1) / threads;
  }
  int started = 0;
  for (int k = 1; k < threads; ++k) {
    if (pthread_create(&tid[k], 0, fill_worker, &jobs[k]) != 0) break;
    started = k;
  }
  /* any job whose thread could not start runs on the calling thread */
  for (int k = started + 1; k < threads; ++k) fill_worker(&jobs[k]);
  fill_worker(&jobs[0]);
  for (int k = 1; k <= started; ++k) pthread_join(tid[k], 0);
  return 0;
}
