// SIMT fp32 correctness-floor kernel for MLA tree-verify attention.
//
// One CTA = (request, tree token, split): the 64 heads of one draft-tree token
// against one contiguous range of the request's keys.  Each 32-key latent tile
// is gathered into shared memory once and shared by all 64 heads (the MLA
// latent is common to every head: "The Glue That Connects" -- "The Context").
// Online softmax over the tiles ("Design Decisions and Trade-Offs"), split-K
// partial output + LSE ("The Final Solder Joint" -- "The Three-Edits
// Sequence").  fp32 CUDA-core arithmetic; kept as a debug path beside the
// tensor-core kernel, selected only by MTV_FLAG_SIMT_FLOOR at plan time.
#include <math.h>

#include "mtv_internal.cuh"

namespace mtv {
namespace {

constexpr int KT = kSimtKeyTile;       // keys per tile
constexpr int NT = kSimtThreads;       // threads per CTA
constexpr int RS = kDQK + 2;           // padded bf16 row stride (odd word count)
constexpr size_t kSmemQ = size_t(kHeads) * RS * 2;
constexpr size_t kSmemKV = size_t(KT) * RS * 2;
constexpr size_t kSmemP = size_t(kHeads) * (KT + 1) * 4;
constexpr size_t kSmemMisc = kHeads * 4 * 3 + KT * 8 + KT * 4;
constexpr size_t kSmemTotal = kSmemQ + kSmemKV + kSmemP + kSmemMisc;

__global__ void __launch_bounds__(NT, 1) partial_simt_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* kvs = reinterpret_cast<__nv_bfloat16*>(smem + kSmemQ);
  float* ps = reinterpret_cast<float*>(smem + kSmemQ + kSmemKV);
  float* m_s = reinterpret_cast<float*>(smem + kSmemQ + kSmemKV + kSmemP);
  float* l_s = m_s + kHeads;
  float* f_s = l_s + kHeads;
  int64_t* slot_s = reinterpret_cast<int64_t*>(f_s + kHeads);
  int* vis_s = reinterpret_cast<int*>(slot_s + KT);

  const int tid = threadIdx.x;
  const int r = blockIdx.x / P.max_q;
  const int i = blockIdx.x % P.max_q;
  const int split = blockIdx.y;
  const Req R = load_req(P, r);
  if (i >= R.n) return;
  const int64_t k_begin = int64_t(split) * P.split_keys;
  if (split > 0 && k_begin >= R.keys) return;  // empty split: the combine skips it
  const int64_t k_end = min(R.keys, k_begin + P.split_keys);
  const int64_t tok = R.q_off + i;

  // q for the 64 heads of this token -> smem (bf16, padded rows)
  {
    const __nv_bfloat16* qg = P.q + tok * kHeads * kDQK;
    for (int idx = tid; idx < kHeads * (kDQK / 2); idx += NT) {
      int h = idx / (kDQK / 2), d2 = idx % (kDQK / 2);
      reinterpret_cast<__nv_bfloat162*>(qs + h * RS)[d2] =
          reinterpret_cast<const __nv_bfloat162*>(qg + h * kDQK)[d2];
    }
  }
  if (tid < kHeads) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  const int h_pv = tid >> 2;            // head owned in the PV step and scoring
  const int q4 = tid & 3;               // quarter: keys q4 + 4j / dims q4*128..
  float o[128];
#pragma unroll
  for (int j = 0; j < 128; ++j) o[j] = 0.f;

  for (int64_t kt = k_begin; kt < k_end; kt += KT) {
    __syncthreads();
    if (tid < KT) {
      int64_t k = kt + tid;
      int64_t s = -1;
      int vis = 0;
      if (k < k_end) {
        s = key_slot(P, R, k);
        vis = (s >= 0) && (k < R.p || tree_visible(P, R, i, k - R.p));
      }
      slot_s[tid] = s < 0 ? 0 : s;
      vis_s[tid] = vis;
    }
    __syncthreads();
    // gather the latent rows (1152 B each) of this tile
    for (int idx = tid; idx < KT * (kDQK / 8); idx += NT) {
      int k = idx / (kDQK / 8), c = idx % (kDQK / 8);
      const uint4* src = reinterpret_cast<const uint4*>(P.kv_pool + slot_s[k] * kDQK) + c;
      uint4 v = vis_s[k] ? __ldg(src) : make_uint4(0, 0, 0, 0);
      uint32_t* dst = reinterpret_cast<uint32_t*>(kvs + k * RS) + c * 4;
      dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
    }
    __syncthreads();
    // scores: head h_pv, keys q4 + 4j
    {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      const __nv_bfloat162* qrow = reinterpret_cast<const __nv_bfloat162*>(qs + h_pv * RS);
      for (int d2 = 0; d2 < kDQK / 2; ++d2) {
        float2 qf = __bfloat1622float2(qrow[d2]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float2 kf = __bfloat1622float2(
              reinterpret_cast<const __nv_bfloat162*>(kvs + (q4 + 4 * j) * RS)[d2]);
          acc[j] = fmaf(qf.x, kf.x, acc[j]);
          acc[j] = fmaf(qf.y, kf.y, acc[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int k = q4 + 4 * j;
        ps[h_pv * (KT + 1) + k] = vis_s[k] ? acc[j] * P.scale : -INFINITY;
      }
    }
    __syncthreads();
    // online softmax, one thread per head
    if (tid < kHeads) {
      float* row = ps + tid * (KT + 1);
      float mt = -INFINITY;
      for (int k = 0; k < KT; ++k) mt = fmaxf(mt, row[k]);
      float m_old = m_s[tid];
      float m_new = fmaxf(m_old, mt);
      float fac = 1.f, sum = 0.f;
      if (m_new != -INFINITY) {
        fac = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
        for (int k = 0; k < KT; ++k) {
          float e = (row[k] == -INFINITY) ? 0.f : expf(row[k] - m_new);
          row[k] = e;
          sum += e;
        }
      } else {
        for (int k = 0; k < KT; ++k) row[k] = 0.f;
      }
      l_s[tid] = l_s[tid] * fac + sum;
      m_s[tid] = m_new;
      f_s[tid] = fac;
    }
    __syncthreads();
    // O[h_pv, q4*128 .. +128] = fac * O + P V
    {
      float fac = f_s[h_pv];
#pragma unroll
      for (int j = 0; j < 128; ++j) o[j] *= fac;
      const float* prow = ps + h_pv * (KT + 1);
      for (int k = 0; k < KT; ++k) {
        float p = prow[k];
        if (p == 0.f) continue;
        const __nv_bfloat162* vrow =
            reinterpret_cast<const __nv_bfloat162*>(kvs + k * RS + q4 * 128);
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float2 vf = __bfloat1622float2(vrow[j]);
          o[2 * j] = fmaf(p, vf.x, o[2 * j]);
          o[2 * j + 1] = fmaf(p, vf.y, o[2 * j + 1]);
        }
      }
    }
  }
  __syncthreads();
  const float l = l_s[h_pv], m = m_s[h_pv];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? m + logf(l) : -INFINITY;
  const int64_t row = tok * kHeads + h_pv;
  if (P.nsplit == 1) {
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(P.out + row * kDLat + q4 * 128);
#pragma unroll
    for (int j = 0; j < 64; ++j) dst[j] = __floats2bfloat162_rn(o[2 * j] * inv, o[2 * j + 1] * inv);
    if (q4 == 0) P.lse[row] = lse;
  } else {
    float4* dst = reinterpret_cast<float4*>(
        P.part_o + (int64_t(split) * P.total_q_max * kHeads + row) * kDLat + q4 * 128);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      dst[j] = make_float4(o[4 * j] * inv, o[4 * j + 1] * inv, o[4 * j + 2] * inv, o[4 * j + 3] * inv);
    if (q4 == 0) P.part_lse[int64_t(split) * P.total_q_max * kHeads + row] = lse;
  }
}

}  // namespace

cudaError_t prepare_partial_simt() {
  return cudaFuncSetAttribute(partial_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(kSmemTotal));
}

cudaError_t launch_partial_simt(const Params& P, cudaStream_t st) {
  dim3 grid(unsigned(P.bs) * unsigned(P.max_q), unsigned(P.nsplit));
  if (grid.x == 0) return cudaSuccess;
  partial_simt_kernel<<<grid, NT, kSmemTotal, st>>>(P);
  return cudaGetLastError();
}

}  // namespace mtv
