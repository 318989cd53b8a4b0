// Split-K combine: one warp per (token, head) row merges the per-split
// normalised partial outputs by their log-sum-exp weights,
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// and writes bf16 out (round-to-nearest-even) + fp32 lse.  The split count
// of a request is re-derived on the device from its key count, so splits
// past the request's end are never read ("The Final Solder Joint" -- "The
// Three-Edits Sequence": empty splits early-out).
#include <math.h>

#include "mtv_internal.cuh"

namespace mtv {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const Params P) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t tok = row / kHeads;
  if (P.bs <= 0 || tok >= P.total_q_max) return;
  const int64_t total_q = P.qo_indptr[P.bs];
  if (tok >= total_q) return;
  // request owning this token: last r with qo_indptr[r] <= tok
  int lo = 0, hi = P.bs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (P.qo_indptr[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  const int64_t p = int64_t(P.kv_indptr[lo + 1]) - P.kv_indptr[lo];
  const int64_t n = P.qo_indptr[lo + 1] - P.qo_indptr[lo];
  if (p < 0 || n < 0 || p > P.max_prefix || n > P.max_q) return;  // flagged by the partial kernel
  const int ns = splits_used(P, p + n);
  const int64_t stride_rows = P.total_q_max * kHeads;

  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, P.part_lse[s * stride_rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  float lse = -INFINITY;
  if (m != -INFINITY) {
    float sum = 0.f;
    for (int s = lane; s < ns; s += 32) sum += expf(P.part_lse[s * stride_rows + row] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse = m + logf(sum);
    for (int s = 0; s < ns; ++s) {
      const float w = expf(P.part_lse[s * stride_rows + row] - lse);
      if (w == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(P.part_o + (s * stride_rows + row) * kDLat) + lane * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4 v = src[j];
        acc[4 * j] = fmaf(w, v.x, acc[4 * j]);
        acc[4 * j + 1] = fmaf(w, v.y, acc[4 * j + 1]);
        acc[4 * j + 2] = fmaf(w, v.z, acc[4 * j + 2]);
        acc[4 * j + 3] = fmaf(w, v.w, acc[4 * j + 3]);
      }
    }
  }
  uint4 packed[2];
  uint32_t* pw = reinterpret_cast<uint32_t*>(packed);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    pw[j] = *reinterpret_cast<uint32_t*>(&b);
  }
  uint4* dst = reinterpret_cast<uint4*>(P.out + row * kDLat) + lane * 2;
  dst[0] = packed[0];
  dst[1] = packed[1];
  if (lane == 0) P.lse[row] = lse;
}

}  // namespace

cudaError_t launch_combine(const Params& P, cudaStream_t st) {
  const int64_t rows = P.total_q_max * kHeads;
  if (rows == 0 || P.bs == 0) return cudaSuccess;
  const unsigned blocks = unsigned((rows + kWarps - 1) / kWarps);
  combine_kernel<<<blocks, kWarps * 32, 0, st>>>(P);
  return cudaGetLastError();
}

}  // namespace mtv
