/*
 * Seeded, counter-based generator of synthetic inputs (Q, K, V rows).
 *
 * This module holds no arithmetic of the method itself: it only produces the
 * numbers that both the CPU oracle and the GPU path take as input. Any element
 * can be regenerated on its own from (seed, stream, index), so a large
 * workload never has to exist whole on the host just to check a few outputs.
 *
 * Definition
 *   splitmix64(x): z = x + 0x9E3779B97F4A7C15;
 *                  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                  z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                  return z ^ (z >> 31)             (all mod 2^64)
 *   base(seed, stream) = splitmix64(splitmix64(seed) ^ stream)
 *   words w_j = splitmix64(base + 3 i + j), j = 0, 1, 2, for element i
 *   u_0..u_11 = the twelve 16-bit fields of w_0, w_1, w_2
 *   n_i = (u_0 + ... + u_11 - 393210) / 65536
 * n_i is the Irwin-Hall sum of twelve uniforms minus its mean: mean 0,
 * variance 1 (to within 2^-32), range [-6, 6]. It uses integer arithmetic and
 * one exact power-of-two scaling only, so every platform yields the same bits.
 *   value_i = float(n_i * scale * chan_scale[i % period])   (double -> float RNE)
 * and the stored element is value_i rounded to binary16 or bfloat16 (RNE).
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GEN_F32 0
#define GEN_F16 1
#define GEN_BF16 2

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t kvqgen_splitmix64(uint64_t x) { return splitmix64(x); }

uint64_t kvqgen_base(uint64_t seed, uint64_t stream) {
  return splitmix64(splitmix64(seed) ^ stream);
}

/* Numerator of n_i (n_i = numerator / 65536). */
static inline int32_t ih12_numerator(uint64_t base, uint64_t i) {
  int64_t s = 0;
  for (uint64_t j = 0; j < 3; ++j) {
    const uint64_t w = splitmix64(base + 3 * i + j);
    s += (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) +
         (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
  }
  return (int32_t)(s - 393210);
}

static inline uint16_t to_f16(float f) {
  _Float16 h = (_Float16)f; /* IEEE conversion, round to nearest even */
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

static inline uint16_t to_bf16(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x40); /* NaN */
  x += 0x7FFFu + ((x >> 16) & 1u); /* round to nearest, ties to even */
  return (uint16_t)(x >> 16);
}

typedef struct {
  uint64_t base, start, count;
  double scale;
  const float* chan_scale;
  uint64_t period;
  int dtype;
  void* out;
} gen_job;

static void run_job(const gen_job* J) {
  for (uint64_t k = 0; k < J->count; ++k) {
    const uint64_t i = J->start + k;
    double v = (double)ih12_numerator(J->base, i) / 65536.0 * J->scale;
    if (J->chan_scale) v *= (double)J->chan_scale[i % J->period];
    const float f = (float)v;
    if (J->dtype == GEN_F32) {
      ((float*)J->out)[k] = f;
    } else if (J->dtype == GEN_F16) {
      ((uint16_t*)J->out)[k] = to_f16(f);
    } else {
      ((uint16_t*)J->out)[k] = to_bf16(f);
    }
  }
}

static void* job_thread(void* arg) {
  run_job((const gen_job*)arg);
  return NULL;
}

/*
 * Fill out[0..count) with elements start..start+count of stream `stream`.
 * chan_scale (may be NULL) multiplies element i by chan_scale[i % period].
 * dtype: 0 = float32, 1 = binary16 bits, 2 = bfloat16 bits.
 * nthreads > 1 splits the range over POSIX threads; the bits do not depend
 * on it. Returns 0, or -1 on a bad argument.
 */
int kvqgen_normal(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                  double scale, const float* chan_scale, uint64_t period, int dtype,
                  void* out, int nthreads) {
  if (dtype < 0 || dtype > 2 || (chan_scale && period == 0) || (count && !out)) return -1;
  const uint64_t base = kvqgen_base(seed, stream);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (count < (uint64_t)nthreads * 65536) nthreads = 1;
  gen_job jobs[64];
  pthread_t tids[64];
  int started[64] = {0};
  const size_t esz = dtype == GEN_F32 ? 4 : 2;
  const uint64_t per = (count + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const uint64_t s = (uint64_t)t * per;
    if (s >= count) break;
    const uint64_t c = (s + per > count) ? count - s : per;
    jobs[t] = (gen_job){base, start + s, c, scale, chan_scale, period, dtype,
                        (char*)out + s * esz};
    if (nthreads == 1) {
      run_job(&jobs[t]);
    } else if (pthread_create(&tids[t], NULL, job_thread, &jobs[t]) == 0) {
      started[t] = 1;
    } else {
      run_job(&jobs[t]); /* no thread available: do this share inline */
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (started[t]) pthread_join(tids[t], NULL);
  return 0;
}
