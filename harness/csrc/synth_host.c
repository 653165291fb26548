/* Host (CPU) implementation of the harness's counter-based weight generator: the same
 * definition as harness/inputs.py and harness/csrc/synth.cu, bit for bit.  SplitMix64
 * output function over the counter (Steele, Lea and Flood, OOPSLA 2014), four 22-bit
 * fields summed (Irwin-Hall(4)), one fp32 multiply, optional round-to-nearest-even to
 * bf16 (returned as the fp32 value of that bf16).  Input generation only: no method
 * arithmetic.  Threads split the range with OpenMP when the compiler provides it. */
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1ull) * 0x9E3779B97F4A7C15ull); }

/* out[i] = weight element (start + i) of stream key, i < count, as fp32 (bf16-rounded if as_bf16). */
int synth_weights_host(uint64_t key, uint64_t start, uint64_t count, float scale, int as_bf16, float* out) {
  const uint64_t mask = (1ull << 22) - 1ull;
  const int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t e = start + (uint64_t)i;
    const uint64_t w0 = draw(key, 2ull * e), w1 = draw(key, 2ull * e + 1ull);
    const uint64_t s = (w0 & mask) + ((w0 >> 22) & mask) + (w1 & mask) + ((w1 >> 22) & mask);
    const int64_t z = (int64_t)s - ((1ll << 23) - 2);
    float w = (float)z * scale; /* (float)z is exact (|z| < 2^24); one correctly rounded fp32 multiply */
    if (as_bf16) {
      uint32_t u;
      memcpy(&u, &w, 4);
      u = u + 0x7FFFu + ((u >> 16) & 1u);
      u &= 0xFFFF0000u;
      memcpy(&w, &u, 4);
    }
    out[i] = w;
  }
  return 0;
}
