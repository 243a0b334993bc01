// LSE-weighted merge of split-KV partials (flash-decoding combine).
//
// Each partial (o_s, lse_s) is attention normalised over its own part of a row's
// visible set. The exact result over the union is
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s,
// with parts of lse_s = -inf (nothing visible there) carrying no weight.
//
// Bandwidth-bound on the partials (which normally still sit in L2): per row it
// reads splits * (4 + d_v * sizeof(partial)) bytes and writes one output row. To
// keep enough loads in flight, one CTA handles one row and 128 columns; its 8 warps
// stride over the splits in one pass (lane = 4 consecutive columns, 10 splits in flight
// per lane, an online max per warp) and are merged through shared memory at the end.
// Partials are fp32 or fp16.
// Launched after the attention kernel with programmatic dependent launch: the
// kernel waits for the primary grid's results before its first read.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kCols = 128;   // columns per CTA (32 lanes x 4)
constexpr int kWarps = 8;
constexpr int kBatch = 10;  // splits per warp whose loads are in flight together

__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename PT>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(int32_t splits, int64_t rows, int32_t d_v, const PT* __restrict__ part_o,
               const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
               int32_t out_dtype) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // no-op unless launched as a dependent
  const int64_t r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float s_m[kWarps], s_z[kWarps];
  __shared__ float4 s_acc[kWarps][32];

  // One pass: warp w folds splits w, w + 8, ... into its own running max m, sum z and
  // weighted sum acc (all loads of a batch issued before any is used); warps merge below.
  const int c = blockIdx.y * kCols + lane * 4;
  const bool col_ok = c < d_v;
  float m = -INFINITY, z = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < splits; s0 += kWarps * kBatch) {
    float ls[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int s = s0 + u * kWarps;
      ls[u] = s < splits ? part_lse[(int64_t)s * rows + r] : -INFINITY;
      v[u] = (s < splits && col_ok) ? load4(part_o + ((int64_t)s * rows + r) * d_v + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (ls[u] == -INFINITY) continue;  // nothing visible in that part (its partial is not read)
      if (ls[u] > m) {
        const float f = expf(m - ls[u]);  // 0 while m = -inf
        z *= f;
        acc.x *= f;
        acc.y *= f;
        acc.z *= f;
        acc.w *= f;
        m = ls[u];
      }
      const float w = expf(ls[u] - m);
      z += w;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_z[warp] = z;
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
    float Z = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        if (s_m[w] == -INFINITY) continue;
        const float f = expf(s_m[w] - M);
        Z = fmaf(s_z[w], f, Z);
        const float4 x = s_acc[w][lane];
        t.x = fmaf(x.x, f, t.x);
        t.y = fmaf(x.y, f, t.y);
        t.z = fmaf(x.z, f, t.z);
        t.w = fmaf(x.w, f, t.w);
      }
      const float inv = 1.f / Z;
      t.x *= inv;
      t.y *= inv;
      t.z *= inv;
      t.w *= inv;
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
    if (lane == 0 && blockIdx.y == 0 && lse) lse[r] = (M == -INFINITY) ? -INFINITY : M + logf(Z);
  }
}

}  // namespace

cudaError_t launch_combine(int32_t splits, int64_t rows, int32_t d_v, const void* part_o, int32_t part_dtype,
                           const float* part_lse, void* out, float* lse, int32_t out_dtype, bool dependent,
                           cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows, (unsigned)((d_v + kCols - 1) / kCols));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  if (part_dtype == MLA_DTYPE_F16)
    return cudaLaunchKernelEx(&cfg, combine_kernel<__half>, splits, rows, d_v, static_cast<const __half*>(part_o),
                              part_lse, out, lse, out_dtype);
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, splits, rows, d_v, static_cast<const float*>(part_o),
                            part_lse, out, lse, out_dtype);
}

}  // namespace mla
