/* Host-side fast path of the seeded synthetic input generator (workloads.py).
 *
 * Holds no part of the SDM method: it only draws the counter-based random numbers
 * workloads.py defines (Philox4x32-10, Salmon et al., SC'11; Box-Muller with fixed
 * fp32 series), for contiguous ranges of element indices, using threads.  Every
 * fp32 operation is a separately rounded IEEE operation (built with
 * -ffp-contract=off), so the bits equal those of the numpy definition and of the
 * CUDA library's device generator.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline float bitsf(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}
static inline uint32_t fbits(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  return b;
}

static void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = (uint32_t)p1;
    c[2] = n2;
    c[3] = (uint32_t)p0;
  }
}

static inline void draw(uint64_t seed, int field, uint64_t e, uint32_t* x0, uint32_t* x1) {
  uint32_t c[4] = {(uint32_t)e, (uint32_t)(e >> 32), (uint32_t)field, 0u};
  philox(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  *x0 = c[0];
  *x1 = c[1];
}

static inline float uniform_open(uint32_t x0) {
  return ((float)(x0 >> 8) + 1.0f) * bitsf(0x33800000u);
}

static float fixed_ln(float u) {
  const uint32_t bits = fbits(u);
  int e = (int)(bits >> 23) - 127;
  float f = bitsf((bits & 0x7FFFFFu) | 0x3F800000u);
  if (f > bitsf(0x3FB504F3u)) {
    f = f * 0.5f;
    e += 1;
  }
  const float z = (f - 1.0f) / (f + 1.0f);
  const float z2 = z * z;
  float p = bitsf(0x3DE38E39u);
  p = p * z2 + bitsf(0x3E124925u);
  p = p * z2 + bitsf(0x3E4CCCCDu);
  p = p * z2 + bitsf(0x3EAAAAABu);
  p = p * z2 + 1.0f;
  const float t = z * p;
  return (float)e * bitsf(0x3F317218u) + (t + t);
}

static float fixed_cos_turn(uint32_t k24) {
  const uint32_t quad = k24 >> 22;
  const float phi = (float)(k24 & 0x3FFFFFu) * bitsf(0x34C90FDBu);
  const float p2 = phi * phi;
  float s = bitsf(0x2F309231u);
  s = s * p2 + bitsf(0xB2D7322Bu);
  s = s * p2 + bitsf(0x3638EF1Du);
  s = s * p2 + bitsf(0xB9500D01u);
  s = s * p2 + bitsf(0x3C088889u);
  s = s * p2 + bitsf(0xBE2AAAABu);
  s = phi * (s * p2 + 1.0f);
  float c = bitsf(0xAD49CBA5u);
  c = c * p2 + bitsf(0x310F76C7u);
  c = c * p2 + bitsf(0xB493F27Eu);
  c = c * p2 + bitsf(0x37D00D01u);
  c = c * p2 + bitsf(0xBAB60B61u);
  c = c * p2 + bitsf(0x3D2AAAABu);
  c = c * p2 + bitsf(0xBF000000u);
  c = c * p2 + 1.0f;
  return quad == 0 ? c : (quad == 1 ? -s : (quad == 2 ? -c : s));
}

static inline float normal_at(uint64_t seed, int field, uint64_t e) {
  uint32_t x0, x1;
  draw(seed, field, e, &x0, &x1);
  const float r = sqrtf(-2.0f * fixed_ln(uniform_open(x0)));
  return r * fixed_cos_turn(x1 >> 8);
}

typedef struct {
  uint64_t seed, e0;
  int field, kind;  /* kind 0: normal, 1: uniform in (0, 1] */
  float* out;
  int64_t lo, hi;
} Job;

static void* run(void* arg) {
  const Job* j = (const Job*)arg;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    const uint64_t e = j->e0 + (uint64_t)i;
    if (j->kind == 0) {
      j->out[i] = normal_at(j->seed, j->field, e);
    } else {
      uint32_t x0, x1;
      draw(j->seed, j->field, e, &x0, &x1);
      j->out[i] = uniform_open(x0);
    }
  }
  return 0;
}

/* out[i] = draw for element index e0 + i, i in [0, n); kind 0 normal, 1 uniform. */
int sdm_workloads_fill(uint64_t seed, int field, uint64_t e0, int64_t n, int kind, float* out,
                       int n_threads) {
  if (n <= 0) return 0;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n < 65536) n_threads = 1;
  Job jobs[256];
  pthread_t th[256];
  const int64_t per = (n + n_threads - 1) / n_threads;
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    jobs[t] = (Job){seed, e0, field, kind, out, t * per, (t + 1) * per < n ? (t + 1) * per : n};
    if (jobs[t].lo >= jobs[t].hi) break;
    if (t == 0) continue;
    if (pthread_create(&th[t], 0, run, &jobs[t]) != 0) {
      run(&jobs[t]);
      th[t] = 0;
    }
    started = t;
  }
  run(&jobs[0]);
  for (int t = 1; t <= started; ++t)
    if (th[t]) pthread_join(th[t], 0);
  return 0;
}
