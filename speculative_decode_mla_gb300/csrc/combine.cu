// LSE-weighted merge of split-KV partials (flash-decoding combine).
//
// Each partial (o_s, lse_s) is attention normalised over its own part of a row's
// visible set. The exact result over the union is
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s,
// with parts of lse_s = -inf (nothing visible there) carrying no weight.
//
// Work per row is tiny (splits * d_v multiply-adds), so the kernel is shaped to keep
// the instruction count low and the loads few and wide. One CTA handles one row and
// 128 columns (lane = 4 consecutive columns). Every warp first takes the row's largest
// lse_s M with a warp-shuffle max; each split then weighs w_s = 2^((lse_s - M) log2 e)
// (one ex2, no running-max rescale), and the 8 warps, each folding every 8th split,
// are summed through shared memory:
//   out = (sum_s w_s o_s) / (sum_s w_s),  lse = M + ln sum_s w_s.
// fp16 partials with d_v a multiple of 128 arrive by one TMA tensor load per CTA (a box
// of 128 columns x 1 row x up to 128 splits), which also keeps them off the per-SM limit
// on outstanding LSU requests; fp32 partials are read with plain vector loads.
// Calls with many rows (batches, wide head counts) use one warp per (row, 128 columns)
// instead, which folds in the same order (combine_warp_kernel).
// Launched after the attention kernel with programmatic dependent launch: the kernel
// waits for the primary grid's results before its first read.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kCols = 128;       // columns per CTA (32 lanes x 4)
constexpr int kWarps = 8;
constexpr int kBatch = 10;       // splits per warp whose loads are in flight together (plain kernel)
constexpr int kTmaSplits = 128;  // splits per TMA box (32 KB of shared memory)
// From this many (row, 128-column) items on, one warp per item instead of one CTA (more than
// one wave of 8-warp CTAs on this part's SMs).
constexpr int64_t kWarpKernelItems = 2048;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kTimeoutCycles = 4000000000ll;  // ~2 s at 2 GHz

__device__ __forceinline__ float ex2(float x) {  // 2^x on the MUFU unit; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// The row's largest split lse (every lane of the warp receives it); NaN entries are ignored here
// and poison the output through their own weight.
__device__ __forceinline__ float row_lse_max(const float* part_lse, int32_t splits, int64_t rows, int64_t r, int lane) {
  float M = -INFINITY;
  for (int s = lane; s < splits; s += 32) M = fmaxf(M, part_lse[(int64_t)s * rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  return M;
}

__device__ __forceinline__ void fold(float ls, float M, float4 v, float& z, float4& acc) {
  const float w = ex2((ls - M) * kLog2e);
  z += w;
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

// Writes a row's 4 columns at c, O = acc / Z, and (write_lse) its lse = M + ln Z.
__device__ __forceinline__ void store_row(float M, float Z, float4 t, int64_t r, int c, int32_t d_v, void* out,
                                          float* lse, int32_t out_dtype, bool write_lse) {
  const float inv = Z > 0.f ? 1.f / Z : 0.f;  // all parts empty: out = 0, lse = -inf
  t.x *= inv;
  t.y *= inv;
  t.z *= inv;
  t.w *= inv;
  if (c < d_v) {
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
  if (write_lse && lse) lse[r] = (Z > 0.f || Z != Z) ? M + logf(Z) : -INFINITY;
}

// Sums the warps' (z, acc) and writes the row's 128 columns and its lse (warp 0 does the writing).
__device__ __forceinline__ void finish(float M, float z, float4 acc, int64_t r, int c, int32_t d_v, void* out,
                                       float* lse, int32_t out_dtype, int warp, int lane) {
  __shared__ float s_z[kWarps];
  __shared__ float4 s_acc[kWarps][32];
  if (lane == 0) s_z[warp] = z;
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp != 0) return;
  float Z = 0.f;
  float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    Z += s_z[w];
    const float4 x = s_acc[w][lane];
    t.x += x.x;
    t.y += x.y;
    t.z += x.z;
    t.w += x.w;
  }
  store_row(M, Z, t, r, c, d_v, out, lse, out_dtype, lane == 0 && blockIdx.y == 0);
}

template <typename PT>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(int32_t splits, int64_t rows, int32_t d_v, const PT* __restrict__ part_o,
               const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
               int32_t out_dtype) {
  // the next kernel in the stream (e.g. the next layer's attention) may be scheduled now; it waits
  // for this grid to finish before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // no-op unless launched as a dependent
  const int64_t r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.y * kCols + lane * 4;
  const bool col_ok = c < d_v;
  const float M = row_lse_max(part_lse, splits, rows, r, lane);
  float z = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < splits; s0 += kWarps * kBatch) {
    float ls[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int sp = s0 + u * kWarps;
      ls[u] = sp < splits ? part_lse[(int64_t)sp * rows + r] : -INFINITY;
      v[u] = (sp < splits && col_ok && ls[u] != -INFINITY) ? load4(part_o + ((int64_t)sp * rows + r) * d_v + c)
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (ls[u] != -INFINITY) fold(ls[u], M, v[u], z, acc);  // an empty part's partial is not used
  }
  finish(M, z, acc, r, c, d_v, out, lse, out_dtype, warp, lane);
}

__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok)
               : "r"(bar), "r"(parity)
               : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  const long long start = clock64();
  while (!bar_test(bar, parity))
    if (clock64() - start > kTimeoutCycles) return false;
  return true;
}

// fp16 partials through one TMA tensor load per CTA and chunk of up to 128 splits.
__global__ void __launch_bounds__(kWarps * 32)
combine_tma_kernel(const __grid_constant__ CUtensorMap tm, int32_t splits, int32_t box_splits, int64_t rows,
                   int32_t d_v, const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
                   int32_t out_dtype) {
  // the next kernel in the stream (e.g. the next layer's attention) may be scheduled now; it waits
  // for this grid to finish before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // no-op unless launched as a dependent
  extern __shared__ __align__(128) uint8_t sm[];      // [box_splits][kCols] fp16
  __shared__ __align__(8) uint64_t bar;
  const int64_t r = blockIdx.x;
  const int c0 = blockIdx.y * kCols;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar_a = (uint32_t)__cvta_generic_to_shared(&bar);
  const uint32_t sm_a = (uint32_t)__cvta_generic_to_shared(sm);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int nchunks = (splits + box_splits - 1) / box_splits;
  __shared__ float s_ls[kTmaSplits];
  float M = -INFINITY;
  if (nchunks > 1) M = row_lse_max(part_lse, splits, rows, r, lane);  // else taken from s_ls below
  float z = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool ok = true;
  int failed = 0;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int s0 = ch * box_splits;
    if (threadIdx.x == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_a), "r"(box_splits * kCols * 2)
                   : "memory");
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
          "%4}], [%5];" ::"r"(sm_a),
          "l"(&tm), "r"(c0), "r"((int)r), "r"(s0), "r"(bar_a)
          : "memory");
    }
    // the chunk's lse values, one per thread, while the box is in flight
    for (int i = threadIdx.x; i < box_splits; i += kWarps * 32)
      s_ls[i] = s0 + i < splits ? part_lse[(int64_t)(s0 + i) * rows + r] : -INFINITY;
    __syncthreads();
    if (nchunks == 1) {
      for (int i = lane; i < box_splits; i += 32) M = fmaxf(M, s_ls[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    if (!bar_wait(bar_a, ch & 1)) {
      ok = false;
      failed = ch;
      break;
    }
    const uint8_t* colp = sm + lane * 8;
    for (int sl = warp; sl < box_splits; sl += kWarps) {
      const float ls = s_ls[sl];
      if (ls == -INFINITY) continue;  // empty part or past the last split: not read
      const uint2 raw = *reinterpret_cast<const uint2*>(colp + sl * (kCols * 2));
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      fold(ls, M, make_float4(a.x, a.y, b.x, b.y), z, acc);
    }
    __syncthreads();  // every warp is done with the box and s_ls before the next chunk overwrites them
  }
  if (!ok) {  // a copy that never completed: let it land (bounded) before the CTA exits; mark the row
    bar_wait(bar_a, failed & 1);
    z = __int_as_float(0x7fc00000);
  }
  finish(M, z, acc, r, c0 + lane * 4, d_v, out, lse, out_dtype, warp, lane);
}

// Many rows (batches of sequences, wide head counts): one warp per (row, 128 columns), eight per
// CTA. A CTA per row would spend its time on launch and load latency, wave after wave, for the
// few splits a row of a batch has; here a warp reads the row's lse values, then only the splits
// up to the last non-empty one, eight loads in flight per lane. The folds keep one (z, acc) per
// residue of the split index mod 8 and add them in that order, the order in which the CTA
// kernels' eight warps fold and are summed, so every combine kernel gives the same bits.
template <typename PT>
__global__ void __launch_bounds__(kWarps * 32)
combine_warp_kernel(int32_t splits, int64_t rows, int32_t d_v, int32_t col_blocks, const PT* __restrict__ part_o,
                    const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
                    int32_t out_dtype) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // no-op unless launched as a dependent
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kWarps + warp;
  if (item >= rows * col_blocks) return;  // (no block-wide synchronisation below)
  const int64_t r = item / col_blocks;
  const int cb = (int)(item % col_blocks);
  const int c = cb * kCols + lane * 4;
  const bool col_ok = c < d_v;
  float M = -INFINITY;
  int last = -1;
  for (int s = lane; s < splits; s += 32) {
    const float l = part_lse[(int64_t)s * rows + r];
    M = fmaxf(M, l);
    if (l != -INFINITY) last = s;  // (a NaN counts: it must reach the output)
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  float z[kWarps];
  float4 acc[kWarps];
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    z[w] = 0.f;
    acc[w] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s0 = 0; s0 <= last; s0 += kWarps) {
    float ls[kWarps];
    float4 v[kWarps];
#pragma unroll
    for (int u = 0; u < kWarps; ++u) ls[u] = s0 + u <= last ? part_lse[(int64_t)(s0 + u) * rows + r] : -INFINITY;
#pragma unroll
    for (int u = 0; u < kWarps; ++u)
      v[u] = (col_ok && ls[u] != -INFINITY) ? load4(part_o + ((int64_t)(s0 + u) * rows + r) * d_v + c)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kWarps; ++u)
      if (ls[u] != -INFINITY) fold(ls[u], M, v[u], z[u], acc[u]);
  }
  float Z = 0.f;
  float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    Z += z[w];
    t.x += acc[w].x;
    t.y += acc[w].y;
    t.z += acc[w].z;
    t.w += acc[w].w;
  }
  store_row(M, Z, t, r, c, d_v, out, lse, out_dtype, lane == 0 && cb == 0);
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
  const int32_t col_blocks = (d_v + kCols - 1) / kCols;
  if ((int64_t)rows * col_blocks >= kWarpKernelItems) {
    cfg.gridDim = dim3((unsigned)(((int64_t)rows * col_blocks + kWarps - 1) / kWarps));
    if (part_dtype == MLA_DTYPE_F16)
      return cudaLaunchKernelEx(&cfg, combine_warp_kernel<__half>, splits, rows, d_v, col_blocks,
                                static_cast<const __half*>(part_o), part_lse, out, lse, out_dtype);
    return cudaLaunchKernelEx(&cfg, combine_warp_kernel<float>, splits, rows, d_v, col_blocks,
                              static_cast<const float*>(part_o), part_lse, out, lse, out_dtype);
  }
  EncodeTiledFn enc = tensor_map_encoder();
  if (part_dtype == MLA_DTYPE_F16 && d_v % kCols == 0 && enc != nullptr &&
      (reinterpret_cast<uintptr_t>(part_o) & 15) == 0 && rows <= 0x7fffffff && splits <= 0x7fffffff) {
    // fp16 partials viewed as [splits][rows][d_v]; one box = 128 columns of one row, box_splits splits
    const int32_t box_splits = splits < kTmaSplits ? splits : kTmaSplits;
    CUtensorMap tm;
    const cuuint64_t dims[3] = {(cuuint64_t)d_v, (cuuint64_t)rows, (cuuint64_t)splits};
    const cuuint64_t strides[2] = {(cuuint64_t)d_v * 2, (cuuint64_t)rows * (cuuint64_t)d_v * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kCols, 1, (cuuint32_t)box_splits};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(part_o), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      cfg.gridDim = dim3((unsigned)rows, (unsigned)(d_v / kCols));
      cfg.dynamicSmemBytes = (size_t)box_splits * kCols * 2;
      return cudaLaunchKernelEx(&cfg, combine_tma_kernel, tm, splits, box_splits, rows, d_v, part_lse, out, lse,
                                out_dtype);
    }
  }
  if (part_dtype == MLA_DTYPE_F16)
    return cudaLaunchKernelEx(&cfg, combine_kernel<__half>, splits, rows, d_v, static_cast<const __half*>(part_o),
                              part_lse, out, lse, out_dtype);
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, splits, rows, d_v, static_cast<const float*>(part_o),
                            part_lse, out, lse, out_dtype);
}

}  // namespace mla
