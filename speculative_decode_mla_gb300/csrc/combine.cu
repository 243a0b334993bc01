// LSE-weighted merge of split-KV partials (flash-decoding combine).
//
// Each partial (o_s, lse_s) is attention normalised over its own part of a row's
// visible set. The exact result over the union is
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s,
// with parts of lse_s = -inf (nothing visible there) carrying no weight.
//
// Bandwidth-bound on the partials (which normally still sit in L2): per row it
// reads splits * (4 + 4*d_v) bytes and writes one output row. To keep enough
// loads in flight, one CTA handles one row and 128 columns; its 8 warps stride
// over the splits (lane = 4 consecutive columns, 16-byte loads, 4 splits in
// flight per lane) and are reduced through shared memory at the end.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kCols = 128;   // columns per CTA (32 lanes x 4)
constexpr int kWarps = 8;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(int32_t splits, int64_t rows, int32_t d_v, const float* __restrict__ part_o,
               const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
               int32_t out_dtype) {
  const int64_t r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float s_red[kWarps];
  __shared__ float4 s_acc[kWarps][32];

  // 1. max over the splits, then the sum of exp: total = ln sum_s exp(lse_s)
  float m = -INFINITY;
  for (int s = threadIdx.x; s < splits; s += blockDim.x) m = fmaxf(m, part_lse[(int64_t)s * rows + r]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  m = s_red[0];
  for (int w = 1; w < kWarps; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();
  float z = 0.f;
  if (m != -INFINITY)
    for (int s = threadIdx.x; s < splits; s += blockDim.x) z += expf(part_lse[(int64_t)s * rows + r] - m);
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) s_red[warp] = z;
  __syncthreads();
  z = 0.f;
  for (int w = 0; w < kWarps; ++w) z += s_red[w];
  const float total = (m == -INFINITY) ? -INFINITY : m + logf(z);

  // 2. weighted sum of this CTA's 128 columns; warp w takes splits w, w + 8, ...
  const int c = blockIdx.y * kCols + lane * 4;
  const bool col_ok = c < d_v;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (total != -INFINITY && col_ok) {
    for (int s0 = warp; s0 < splits; s0 += kWarps * kUnroll) {
      float w[kUnroll];
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int s = s0 + u * kWarps;
        const float ls = s < splits ? part_lse[(int64_t)s * rows + r] : -INFINITY;
        w[u] = ls == -INFINITY ? 0.f : expf(ls - total);
        v[u] = ls == -INFINITY ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : __ldg(reinterpret_cast<const float4*>(part_o + ((int64_t)s * rows + r) * d_v + c));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
      }
    }
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = s_acc[0][lane];
    for (int w = 1; w < kWarps; ++w) {
      const float4 x = s_acc[w][lane];
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
    if (col_ok) {
      if (out_dtype == MLA_DTYPE_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + r * d_v + c) = t;
      } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + r * d_v + c) = packed;
      }
    }
    if (lane == 0 && blockIdx.y == 0 && lse) lse[r] = total;
  }
}

}  // namespace

cudaError_t launch_combine(int32_t splits, int64_t rows, int32_t d_v, const float* part_o,
                           const float* part_lse, void* out, float* lse, int32_t out_dtype,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid((unsigned)rows, (unsigned)((d_v + kCols - 1) / kCols));
  combine_kernel<<<grid, kWarps * 32, 0, stream>>>(splits, rows, d_v, part_o, part_lse, out, lse, out_dtype);
  return cudaGetLastError();
}

}  // namespace mla
