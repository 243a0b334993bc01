// Plain SIMT reference kernel for split-KV tree-verify attention (fp32 FMA, no tensor cores).
//
// The same work decomposition and partial layout as the tcgen05 kernel, in the
// plainest form: one warp per query row, one KV position at a time.
//   grid.x = (sequence b, 8-row tile), grid.y = split index s; 8 warps per CTA.
//   For each position t of the chunk [s*chunk, (s+1)*chunk) that row r can see
//   (prefix t < L_b, or tree position L_b + j with j in anc*(i)), the warp
//   gathers the 1152-byte latent row kv[slot_table[b][t]] (page_size=1; or, with hybrid
//   addressing, the contiguous prefix row kv[prefix_base[b] + t] / the tree node's own slot),
//   computes s_t = scale * <q_r, k_t> with a shuffle reduction, and folds it into
//   an online softmax (running max m, running sum l, o += p * v_t).
//   The partial o/l and lse = m + ln l go to the workspace; the combine merges.
// Lane l holds bf16 pairs p = l + 32*j of the row (j < 9 for keys, j < 8 for
// values), so every gather instruction of a warp reads 128 contiguous bytes.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kKeyPairsPerLane = kDK / 2 / 32;       // 9
constexpr int kValPairsPerLane = kDLatent / 2 / 32;  // 8

__global__ void __launch_bounds__(kWarps * 32) verify_simt_kernel(VerifyArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.y;
  const int b = blockIdx.x / a.row_tiles;
  const int tile = blockIdx.x % a.row_tiles;
  const int R = a.T * a.H;
  const int local_row = tile * a.rows_per_tile + warp;
  if (local_row >= R) return;
  const int i = local_row / a.H;
  const int64_t row = (int64_t)b * R + local_row;

  const int32_t L = load_len(a, b);
  const int32_t Tb = load_tree_size(a, b);
  const int64_t N = (int64_t)L + Tb;
  const int64_t t0 = (int64_t)s * a.chunk;
  const int64_t t1 = min(N, t0 + a.chunk);
  __half* po = a.part_o + ((int64_t)s * a.rows + row) * kDLatent;
  if (t0 >= t1 || i >= Tb) {  // nothing in this chunk, or a padding row of a smaller tree
    if (lane == 0) a.part_lse[(int64_t)s * a.rows + row] = -INFINITY;
    return;
  }
  const uint64_t anc = ancestor_mask(a, b, i);

  float2 qf[kKeyPairsPerLane];
  const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(a.q + row * kDK);
#pragma unroll
  for (int j = 0; j < kKeyPairsPerLane; ++j) qf[j] = __bfloat1622float2(q2[lane + 32 * j]);

  float m = -INFINITY, l = 0.f;
  float2 o[kValPairsPerLane];
#pragma unroll
  for (int j = 0; j < kValPairsPerLane; ++j) o[j] = make_float2(0.f, 0.f);

  for (int64_t t = t0; t < t1; ++t) {
    if (t >= L && !((anc >> (t - L)) & 1ull)) continue;
    const int64_t slot = load_slot(a, b, L, t);
    const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(a.kv + slot * kDK);
    float2 kf[kKeyPairsPerLane];
#pragma unroll
    for (int j = 0; j < kKeyPairsPerLane; ++j) kf[j] = __bfloat1622float2(k2[lane + 32 * j]);
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kKeyPairsPerLane; ++j) dot = fmaf(qf[j].x, kf[j].x, fmaf(qf[j].y, kf[j].y, dot));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * a.scale;
    const float m_new = fmaxf(m, sc);
    const float alpha = expf(m - m_new);  // 0 on the first visible position (m = -inf)
    const float p = expf(sc - m_new);
    l = l * alpha + p;
#pragma unroll
    for (int j = 0; j < kValPairsPerLane; ++j) {
      // values are the first 512 dims of the same row: pairs lane + 32*j, j < 8
      o[j].x = fmaf(p, kf[j].x, o[j].x * alpha);
      o[j].y = fmaf(p, kf[j].y, o[j].y * alpha);
    }
    m = m_new;
  }
  if (m == -INFINITY) {  // nothing visible to this row in this chunk
    if (lane == 0) a.part_lse[(int64_t)s * a.rows + row] = -INFINITY;
    return;
  }
  const float inv = 1.f / l;
  __half2* po2 = reinterpret_cast<__half2*>(po);
#pragma unroll
  for (int j = 0; j < kValPairsPerLane; ++j) po2[lane + 32 * j] = __floats2half2_rn(o[j].x * inv, o[j].y * inv);
  if (lane == 0) a.part_lse[(int64_t)s * a.rows + row] = m + logf(l);
}

}  // namespace

cudaError_t launch_verify_simt(const VerifyArgs& a, cudaStream_t stream) {
  dim3 grid((unsigned)(a.B * a.row_tiles), (unsigned)a.splits);
  verify_simt_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
