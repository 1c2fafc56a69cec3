// CUDA version of the counter-based input generator defined in duo_synth/__init__.py.
// It fills device buffers with the same bf16 bits the numpy version produces on the
// host; it holds no attention or cache arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  // SplitMix64 output function (Steele, Lea and Flood, OOPSLA 2014).
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_kernel(__nv_bfloat16* __restrict__ out, uint64_t seed, uint64_t stream,
                            int B, int64_t pos0, int64_t T, int H, int D, float scale) {
  const int64_t total = (int64_t)B * T * H * D;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = idx;
    const uint64_t d = r % D; r /= D;
    const uint64_t h = r % H; r /= H;
    const uint64_t t = r % T; r /= T;
    const uint64_t b = r;
    const uint64_t key = (seed << 51) | (stream << 47) | (b << 39) | ((uint64_t)(pos0 + t) << 15) |
                         (h << 8) | d;
    const uint64_t z = mix64(key + 0x9E3779B97F4A7C15ull);
    const uint64_t s2 = (z & 0x00FF00FF00FF00FFull) + ((z >> 8) & 0x00FF00FF00FF00FFull);
    const int u = (int)((s2 * 0x0001000100010001ull) >> 48);
    const float x = __fmul_rn((float)(u - 1020), scale);
    out[idx] = __float2bfloat16_rn(x);
  }
}

}  // namespace

extern "C" int synth_fill_bf16(void* out, int seed, int stream, int B, int64_t pos0, int64_t T, int H,
                               int D, float scale, void* cuda_stream) {
  const int64_t total = (int64_t)B * T * H * D;
  if (total <= 0) return 0;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(
      (__nv_bfloat16*)out, (uint64_t)seed, (uint64_t)stream, B, pos0, T, H, D, scale);
  return (int)cudaGetLastError();
}
