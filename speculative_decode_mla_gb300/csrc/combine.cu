// LSE-weighted merge of split-KV partials (flash-decoding combine).
//
// Each partial (o_s, lse_s) is attention normalised over its own part of a row's
// visible set. The exact result over the union is
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s,
// with parts of lse_s = -inf (nothing visible there) carrying no weight.
//
// HBM-bound: per row it reads splits * (4 + 4*d_v) bytes and writes one output
// row. One CTA of d_v/4 threads per row; each thread owns four consecutive
// columns (16-byte loads of the partial rows, which sit contiguously per split).
#include "common.cuh"

namespace mla {
namespace {

constexpr int kMaxCombineThreads = 256;  // d_v up to 1024

__global__ void __launch_bounds__(kMaxCombineThreads)
combine_kernel(int32_t splits, int64_t rows, int32_t d_v, const float* __restrict__ part_o,
               const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
               int32_t out_dtype) {
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  __shared__ float s_w[32];
  __shared__ float s_red[32];
  // pass 1: max and sum of exp over the splits (a warp-strided loop, then a block reduction)
  float m = -INFINITY;
  for (int s = threadIdx.x; s < splits; s += blockDim.x) m = fmaxf(m, part_lse[(int64_t)s * rows + r]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  const int nwarps = (blockDim.x + 31) >> 5;
  m = -INFINITY;
  for (int w = 0; w < nwarps; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();
  float z = 0.f;
  if (m != -INFINITY)
    for (int s = threadIdx.x; s < splits; s += blockDim.x) z += expf(part_lse[(int64_t)s * rows + r] - m);
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = z;
  __syncthreads();
  z = 0.f;
  for (int w = 0; w < nwarps; ++w) z += s_w[w];
  const float total = (m == -INFINITY) ? -INFINITY : m + logf(z);

  // pass 2: weighted sum of the partial rows, four columns per thread
  const int c = threadIdx.x * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < d_v && total != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ls = part_lse[(int64_t)s * rows + r];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - total);
      const float4 v = *reinterpret_cast<const float4*>(part_o + ((int64_t)s * rows + r) * d_v + c);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  if (c < d_v) {
    if (out_dtype == MLA_DTYPE_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + r * d_v + c) = acc;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + r * d_v + c) = packed;
    }
  }
  if (threadIdx.x == 0 && lse) lse[r] = total;
}

}  // namespace

cudaError_t launch_combine(int32_t splits, int64_t rows, int32_t d_v, const float* part_o,
                           const float* part_lse, void* out, float* lse, int32_t out_dtype,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int threads = ((d_v / 4 + 31) / 32) * 32;
  combine_kernel<<<dim3((unsigned)rows), threads, 0, stream>>>(splits, rows, d_v, part_o, part_lse, out,
                                                               lse, out_dtype);
  return cudaGetLastError();
}

}  // namespace mla
