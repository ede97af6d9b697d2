/* Host generator (test and benchmark infrastructure; none of the layer's arithmetic): the
 * same splitmix64 + Box-Muller recipe as synth/__init__.py and synth/gen.cu, in C with
 * OpenMP for large draws. Built with -ffp-contract=off. */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static float round_bf16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  u = (u + (((u >> 16) & 1u) + 0x7FFFu)) & 0xFFFF0000u;
  memcpy(&v, &u, 4);
  return v;
}

/* out[i] = value of flat element idx[i] (idx NULL: offset + i). */
void synth_normal_host(float* out, int64_t n, const int64_t* idx, int64_t offset, int bf16,
                       uint32_t seed, uint32_t tid, double std_) {
  const uint64_t key = mix64(((uint64_t)seed << 32) | tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t e = (uint64_t)(idx ? idx[i] : offset + i);
    const uint64_t b = mix64(key + (e + 1) * 0x9E3779B97F4A7C15ull);
    const double hi = (double)(b >> 32), lo = (double)(b & 0xffffffffull);
    const double u1 = (hi + 0.5) * 0x1p-32, u2 = lo * 0x1p-32;
    const double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    const float v = (float)(z * std_);
    out[i] = bf16 ? round_bf16(v) : v;
  }
}
