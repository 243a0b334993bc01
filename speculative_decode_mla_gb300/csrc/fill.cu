// Device generator of the seeded synthetic inputs (not part of the method).
//
// dst[i] = bf16_rne( (sum of the four 16-bit fields of h - 131070) * float32(0x37DDB3D7) ),
// h = SplitMix64 output for the counter state seed + (start + i + 1) * 0x9E3779B97F4A7C15.
// SplitMix64 is the published generator of Steele, Lea and Flood (OOPSLA 2014).
// Every step is integer work or one correctly rounded float32 multiply, so the
// host generator reproduces these bits exactly. HBM-bound: 2 bytes written per element.
#include "mla_workload.h"
#include "common.cuh"

namespace mla {
namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t draw(uint64_t seed, uint64_t i) {
  const uint64_t h = splitmix64(seed, i);
  const int32_t sum = (int32_t)(h & 0xFFFF) + (int32_t)((h >> 16) & 0xFFFF) + (int32_t)((h >> 32) & 0xFFFF) +
                      (int32_t)(h >> 48);
  const float x = __fmul_rn((float)(sum - 131070), __uint_as_float(0x37DDB3D7u));
  // float32 -> bf16, round to nearest even on the bit pattern (x is finite)
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__global__ void fill_kernel(uint16_t* __restrict__ dst, int64_t count, uint64_t seed, uint64_t start) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; base < count; base += stride) {
    if (base + 4 <= count && (reinterpret_cast<uintptr_t>(dst + base) & 7) == 0) {
      ushort4 v = make_ushort4(draw(seed, start + base), draw(seed, start + base + 1),
                               draw(seed, start + base + 2), draw(seed, start + base + 3));
      *reinterpret_cast<ushort4*>(dst + base) = v;
    } else {
      for (int64_t k = base; k < min(count, base + 4); ++k) dst[k] = draw(seed, start + k);
    }
  }
}

}  // namespace
}  // namespace mla

extern "C" int mla_fill_normal_bf16(void* dst, int64_t count, uint64_t seed, uint64_t start,
                                    mla_stream_t stream) {
  if (count < 0 || (count > 0 && dst == nullptr)) return MLA_ERR_INVALID_ARGUMENT;
  if (count == 0) return MLA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  int64_t blocks = (count + 4 * 256 - 1) / (4 * 256);
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  mla::fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(static_cast<uint16_t*>(dst), count, seed,
                                                                        start);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
