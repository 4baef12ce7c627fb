/* Seeded synthetic input generator (host C, multithreaded).
 *
 * Draws random numbers only; it contains none of the attention arithmetic.
 * splitmix64 used as a counter-based generator: word i of stream (seed, tag)
 * is mix(base + (i + 1) * GOLDEN) with base = mix(seed * GOLDEN + tag) and mix
 * the splitmix64 finaliser.  Uniforms u = ((w >> 11) + 0.5) * 2^-53; normals by
 * Box-Muller, two per pair of uniforms; each normal times sigma is rounded to
 * float (nearest-even) and then to bf16 (nearest-even on the bit pattern).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static uint64_t stream_base(uint64_t seed, uint64_t tag) { return mix64(seed * GOLDEN + tag); }

static inline uint64_t word_at(uint64_t base, uint64_t i) { return mix64(base + (i + 1) * GOLDEN); }

static inline double uniform_of(uint64_t w) { return ((double)(w >> 11) + 0.5) * 0x1.0p-53; }

static inline uint16_t f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b = (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;
  return (uint16_t)b;
}

/* normal number k of the stream (pairs 2*(k/2), 2*(k/2)+1 of uniforms) */
static inline double normal_at(uint64_t base, int64_t k) {
  int64_t p = k / 2;
  double u1 = uniform_of(word_at(base, (uint64_t)(2 * p)));
  double u2 = uniform_of(word_at(base, (uint64_t)(2 * p + 1)));
  double r = sqrt(-2.0 * log(u1));
  double th = 2.0 * M_PI * u2;
  return (k & 1) ? r * sin(th) : r * cos(th);
}

void synth_words(uint64_t seed, uint64_t tag, uint64_t offset, int64_t n, uint64_t* out) {
  uint64_t base = stream_base(seed, tag);
  for (int64_t i = 0; i < n; ++i) out[i] = word_at(base, offset + (uint64_t)i);
}

void synth_normals_f64(uint64_t seed, uint64_t tag, int64_t start, int64_t n, double sigma, double* out) {
  uint64_t base = stream_base(seed, tag);
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(base, start + i) * sigma;
}

typedef struct {
  uint64_t base;
  int64_t start, lo, hi;
  double sigma;
  uint16_t* out;
} job_t;

static void* bf16_worker(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    double z = normal_at(j->base, j->start + i) * j->sigma;
    j->out[i] = f32_to_bf16((float)z);
  }
  return NULL;
}

void synth_bf16_normals(uint64_t seed, uint64_t tag, int64_t start, int64_t n, double sigma, uint16_t* out,
                        int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < 65536) threads = 1;
  pthread_t th[256];
  job_t jobs[256];
  uint64_t base = stream_base(seed, tag);
  int64_t per = (n + threads - 1) / threads;
  per = (per + 1) & ~(int64_t)1;
  int used = 0;
  for (int t = 0; t < threads; ++t) {
    int64_t lo = (int64_t)t * per, hi = lo + per;
    if (lo >= n) break;
    if (hi > n) hi = n;
    jobs[t] = (job_t){base, start, lo, hi, sigma, out};
    if (threads == 1) {
      bf16_worker(&jobs[t]);
    } else {
      pthread_create(&th[t], NULL, bf16_worker, &jobs[t]);
    }
    ++used;
  }
  if (threads > 1)
    for (int t = 0; t < used; ++t) pthread_join(th[t], NULL);
}
