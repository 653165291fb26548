// Device implementation of the harness's counter-based weight generator (the same
// definition as harness/inputs.py, bit for bit): SplitMix64 output function over the
// counter, four 22-bit fields summed (Irwin-Hall(4)), one fp32 multiply, optional
// round-to-nearest-even to bf16.  Input generation only: no method arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1ull) * 0x9E3779B97F4A7C15ull); }

__global__ void synth_kernel(uint64_t key, uint64_t start, uint64_t count, float scale, int as_bf16, void* out) {
  const uint64_t mask = (1ull << 22) - 1ull;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t e = start + i;
    const uint64_t w0 = draw(key, 2ull * e), w1 = draw(key, 2ull * e + 1ull);
    const uint64_t s = (w0 & mask) + ((w0 >> 22) & mask) + (w1 & mask) + ((w1 >> 22) & mask);
    const long long z = static_cast<long long>(s) - ((1ll << 23) - 2);
    const float w = __fmul_rn(static_cast<float>(z), scale);
    if (as_bf16) {
      uint32_t u = __float_as_uint(w);
      u = u + 0x7FFFu + ((u >> 16) & 1u);
      static_cast<uint16_t*>(out)[i] = static_cast<uint16_t>(u >> 16);
    } else {
      static_cast<float*>(out)[i] = w;
    }
  }
}

}  // namespace

extern "C" int synth_weights(uint64_t key, uint64_t start, uint64_t count, float scale, int as_bf16, void* out,
                             void* stream) {
  if (count == 0) return 0;
  uint64_t blocks = (count + 255) / 256;
  if (blocks > 152ull * 64) blocks = 152ull * 64;
  synth_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(key, start, count, scale,
                                                                                            as_bf16, out);
  return static_cast<int>(cudaGetLastError());
}
