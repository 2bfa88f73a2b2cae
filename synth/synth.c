/*
 * synth.c -- seeded synthetic input generator (counter-based, threaded).
 *
 * Holds no quantization, dequantization or GEMV arithmetic: it only draws
 * random numbers. Both the CPU oracle and the CUDA path consume its output.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used counter-style: draw i of stream key is
 *   z = key * 2^32 + (i + 1) * 0x9E3779B97F4A7C15   (mod 2^64)
 * passed through the SplitMix64 output mix. Uniforms in (0, 1] take the top
 * 53 bits: (z >> 11 + 1) * 2^-53. Normal deviates use the Box-Muller
 * transform: element 2p = r cos(2 pi u2), element 2p+1 = r sin(2 pi u2) with
 * r = sqrt(-2 ln u1), u1 = uniform 2p, u2 = uniform 2p+1, computed in binary64
 * and rounded once to binary32.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t sm_draw(uint64_t key, int64_t i) {
  return sm_mix(key * 4294967296ull + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull);
}

static inline double sm_uniform(uint64_t key, int64_t i) {
  return ((double)(sm_draw(key, i) >> 11) + 1.0) * 0x1p-53;
}

static const double kTwoPi = 6.283185307179586476925286766559;

typedef struct {
  uint64_t key;
  int64_t begin, end; /* element range */
  double std;
  float* out_f32;
  uint16_t* out_bf16;
  uint64_t* out_u64;
} job_t;

static void normal_range(const job_t* j) {
  for (int64_t e = j->begin; e < j->end; ++e) {
    const int64_t p = e >> 1;
    const double u1 = sm_uniform(j->key, 2 * p);
    const double u2 = sm_uniform(j->key, 2 * p + 1);
    const double r = sqrt(-2.0 * log(u1)) * j->std;
    const double t = kTwoPi * u2;
    const double z = (e & 1) ? r * sin(t) : r * cos(t);
    const float f = (float)z;
    if (j->out_f32) j->out_f32[e - j->begin + 0] = f;
    if (j->out_bf16) {
      uint32_t u;
      memcpy(&u, &f, 4);
      const uint32_t lsb = (u >> 16) & 1u;
      j->out_bf16[e - j->begin] = (uint16_t)((u + 0x7fffu + lsb) >> 16);
    }
  }
}

static void draws_range(const job_t* j) {
  for (int64_t e = j->begin; e < j->end; ++e) j->out_u64[e - j->begin] = sm_draw(j->key, e);
}

typedef struct {
  job_t job;
  int kind;
} task_t;

static void* worker(void* arg) {
  task_t* t = (task_t*)arg;
  if (t->kind == 0)
    normal_range(&t->job);
  else
    draws_range(&t->job);
  return NULL;
}

static void run(int kind, uint64_t key, int64_t start, int64_t n, double std, float* f32,
                uint16_t* bf16, uint64_t* u64, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < (int64_t)nthreads * 65536) nthreads = 1;
  pthread_t th[64];
  task_t tasks[64];
  const int64_t per = (n + nthreads - 1) / nthreads;
  int launched = 0;
  for (int i = 0; i < nthreads; ++i) {
    const int64_t b = start + (int64_t)i * per;
    int64_t e = b + per;
    if (e > start + n) e = start + n;
    if (b >= e) break;
    tasks[i].kind = kind;
    tasks[i].job.key = key;
    tasks[i].job.begin = b;
    tasks[i].job.end = e;
    tasks[i].job.std = std;
    tasks[i].job.out_f32 = f32 ? f32 + (b - start) : NULL;
    tasks[i].job.out_bf16 = bf16 ? bf16 + (b - start) : NULL;
    tasks[i].job.out_u64 = u64 ? u64 + (b - start) : NULL;
    if (nthreads == 1) {
      worker(&tasks[i]);
    } else {
      pthread_create(&th[i], NULL, worker, &tasks[i]);
      ++launched;
    }
  }
  for (int i = 0; i < launched; ++i) pthread_join(th[i], NULL);
}

/* Elements [start, start+n) of the N(0, std^2) stream `key`, as binary32. */
void synth_normal_f32(uint64_t key, int64_t start, int64_t n, double std, float* out,
                      int nthreads) {
  run(0, key, start, n, std, out, NULL, NULL, nthreads);
}

/* Same stream with std 1, rounded to bfloat16 (nearest even) bit patterns. */
void synth_normal_bf16(uint64_t key, int64_t start, int64_t n, uint16_t* out, int nthreads) {
  run(0, key, start, n, 1.0, NULL, out, NULL, nthreads);
}

/* Raw 64-bit draws [start, start+n) of stream `key`. */
void synth_draws(uint64_t key, int64_t start, int64_t n, uint64_t* out, int nthreads) {
  run(1, key, start, n, 0.0, NULL, NULL, out, nthreads);
}
