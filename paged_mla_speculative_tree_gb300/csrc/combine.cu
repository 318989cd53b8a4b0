// Split-K combine: merges the per-split normalised partial outputs of every
// (token, head) row by their log-sum-exp weights,
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// and writes bf16 out (round-to-nearest-even) + fp32 lse.  The split count
// of a request is re-derived on the device from its key count, so splits
// past the request's end are never read ("The Final Solder Joint" -- "The
// Three-Edits Sequence": empty splits early-out).
//
// One block per (tree token, 64-dim chunk of the output): 64 head rows x 64
// dims.  The first 64 threads reduce the rows' split LSEs; then every thread
// owns one float4 column of four rows and keeps the loads of two splits in
// flight.  The kernel is launched as a programmatic dependent of the partial
// kernel: everything before the grid-dependency wait (request geometry)
// overlaps the partial kernel's tail.
#include <math.h>

#include "mtv_internal.cuh"

namespace mtv {
namespace {

constexpr int kThreads = 256;
constexpr int kChunkDims = 64;                 // output dims per block
constexpr int kChunks = kDLat / kChunkDims;    // 8
constexpr int kF4 = kChunkDims / 4;            // float4 columns per row chunk: 16
constexpr int kRowsPerPass = kThreads / kF4;   // 16
constexpr int kPasses = kHeads / kRowsPerPass; // 4 rows per thread

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads) combine_kernel(const Params P) {
  __shared__ float lse_row[kHeads];
  const int r = int(blockIdx.x / unsigned(P.max_q));
  const int t = int(blockIdx.x % unsigned(P.max_q));
  const int chunk = int(blockIdx.y);
  const Req R = load_req(P, r);
  if (t >= R.n) return;
  const int ns = splits_used(P, R.keys);
  const int64_t stride_rows = P.total_q_max * kHeads;
  const int64_t row0 = (R.q_off + t) * kHeads;  // first (token, head) row of this block
  grid_dependency_wait();                        // partials of the preceding kernel are complete

  const int tid = threadIdx.x;
  if (tid < kHeads) {
    const float* l = P.part_lse + row0 + tid;
    float m = -INFINITY;
    for (int s = 0; s < ns; ++s) m = fmaxf(m, l[s * stride_rows]);
    float lse = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < ns; ++s) sum += expf(l[s * stride_rows] - m);
      lse = m + logf(sum);
    }
    lse_row[tid] = lse;
    if (chunk == 0) P.lse[row0 + tid] = lse;
  }
  __syncthreads();

  const int f4 = tid % kF4;
  const int rbase = tid / kF4;
  float4 acc[kPasses];
  float lr[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    lr[i] = lse_row[rbase + i * kRowsPerPass];
  }
  const int64_t col = int64_t(chunk) * kChunkDims + f4 * 4;
#pragma unroll 2
  for (int s = 0; s < ns; ++s) {
    float4 v[kPasses];
    float w[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const int64_t row = row0 + rbase + i * kRowsPerPass;
      v[i] = *reinterpret_cast<const float4*>(P.part_o + (s * stride_rows + row) * kDLat + col);
      w[i] = P.part_lse[s * stride_rows + row];
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const float wi = lr[i] == -INFINITY ? 0.f : expf(w[i] - lr[i]);
      acc[i].x = fmaf(wi, v[i].x, acc[i].x);
      acc[i].y = fmaf(wi, v[i].y, acc[i].y);
      acc[i].z = fmaf(wi, v[i].z, acc[i].z);
      acc[i].w = fmaf(wi, v[i].w, acc[i].w);
    }
  }
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int64_t row = row0 + rbase + i * kRowsPerPass;
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[i].x, acc[i].y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[i].z, acc[i].w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&a);
    o.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(P.out + row * kDLat + col) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const Params& P, cudaStream_t st, bool programmatic) {
  if (P.bs == 0 || P.max_q == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(P.bs) * unsigned(P.max_q), unsigned(kChunks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, P);
}

}  // namespace mtv
