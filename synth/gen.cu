// Device twin of the seeded input generator in synth/__init__.py (test and benchmark
// infrastructure; none of the layer's arithmetic). Element i of tensor `tid` under `seed`:
//   key  = mix64((seed << 32) | tid)
//   bits = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
//   z    = sqrt(-2 ln((hi + 0.5) 2^-32)) * cos(2 pi lo 2^-32)     (Box-Muller, fp64)
//   v    = fp32(z * std), then bf16 (nearest-even) for bf16 tensors.
// mix64 is the splitmix64 finaliser (Steele, Lea, Flood 2014). Built with -fmad=false so
// no multiply-add is contracted.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void normal_kernel(void* out, int64_t n, int bf16, uint64_t key, double std_,
                              int64_t offset) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint64_t b = mix64(key + (uint64_t)(offset + i + 1) * 0x9E3779B97F4A7C15ull);
    const double hi = (double)(b >> 32), lo = (double)(b & 0xffffffffull);
    const double u1 = (hi + 0.5) * 0x1p-32, u2 = lo * 0x1p-32;
    const double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    const float v = __double2float_rn(z * std_);
    if (bf16) reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<float*>(out)[i] = v;
  }
}

}  // namespace

extern "C" int synth_normal(void* out, int64_t n, int bf16, uint32_t seed, uint32_t tid,
                            double std_, int64_t offset, void* stream) {
  if (n <= 0) return 0;
  const uint64_t key = mix64(((uint64_t)seed << 32) | tid);
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  normal_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, n, bf16, key, std_, offset);
  return (int)cudaGetLastError();
}
