// Test-only probes of the tcgen05 building blocks used by the tensor-core
// kernel (descriptors, TMEM A operand, MN-major B, 64-byte swizzle, tcgen05.ld
// layout).  One CTA computes D[128 x N] = A[128 x K] * B[N x K]^T with the
// operand layout selected by `variant` and writes D to global memory.
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

using namespace mtv::ptx;

namespace {

constexpr int kM = 128;

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return uint32_t(__bfloat16_as_ushort(lo)) | (uint32_t(__bfloat16_as_ushort(hi)) << 16);
}

// variant: 0 A smem SW128 / B K-major SW128 (K=64)
//          1 A tmem / B K-major SW128 (K=64)
//          2 A smem SW128 / B MN-major SW128 (K=32), LBO = MN-atom stride, SBO = K-group stride
//          3 A tmem / B K-major SW64 (K=32)
//          4 A tmem / B = K-major SW128 chunk (64) + K-major SW64 chunk (32)  (K=96)
//          5 as 2 with LBO and SBO exchanged
__global__ void __launch_bounds__(128) probe_kernel(int variant, int N, int K, const __nv_bfloat16* A,
                                                    const __nv_bfloat16* B, float* D, int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint32_t tmem_base_s;
  __shared__ __align__(8) uint64_t bar;
  const uint32_t base = (smem_u32(smem_raw) + 1023) & ~1023u;
  const uint32_t a_s = base;              // 16 KB: A K-major SW128 (K <= 64)
  const uint32_t b_s = base + 16384;      // up to 48 KB for B
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_s), 512);
    tmem_relinquish();
  }
  if (tid == 0) mbar_init(smem_u32(&bar), 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t a_tmem = tmem + 256;

  const bool a_in_tmem = (variant == 1 || variant == 3 || variant == 4);
  // ---- A: row m = tid
  {
    const int m = tid;
    if (!a_in_tmem) {
      for (int c = 0; c < K / 8; ++c) {  // 16-byte units of the row
        const uint4 v = *reinterpret_cast<const uint4*>(A + m * K + c * 8);
        st_shared_v4(a_s + m * 128 + ((c ^ (m & 7)) << 4), v.x, v.y, v.z, v.w);
      }
    } else {
      for (int c0 = 0; c0 < K / 2; c0 += 16) {
        uint32_t r[16];
        for (int j = 0; j < 16; ++j) r[j] = pack2(A[m * K + 2 * (c0 + j)], A[m * K + 2 * (c0 + j) + 1]);
        tmem_st16_sync(a_tmem + (uint32_t(warp * 32) << 16) + c0, r);
      }
    }
  }
  // ---- B
  for (int n = tid; n < N; n += 128) {
    if (variant == 0 || variant == 1) {
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(B + n * K + c * 8);
        st_shared_v4(b_s + n * 128 + ((c ^ (n & 7)) << 4), v.x, v.y, v.z, v.w);
      }
    } else if (variant == 3) {
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(B + n * K + c * 8);
        st_shared_v4(b_s + n * 64 + ((c ^ ((n >> 1) & 3)) << 4), v.x, v.y, v.z, v.w);
      }
    } else if (variant == 4) {
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(B + n * K + c * 8);
        st_shared_v4(b_s + n * 128 + ((c ^ (n & 7)) << 4), v.x, v.y, v.z, v.w);
      }
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(B + n * K + 64 + c * 8);
        st_shared_v4(b_s + 16384 + n * 64 + ((c ^ ((n >> 1) & 3)) << 4), v.x, v.y, v.z, v.w);
      }
    } else {  // MN-major: element (k, n) at chunk n/64, row k, 16-byte unit (n%64)/8
      for (int k = 0; k < K; ++k) {
        const uint32_t addr = b_s + (n >> 6) * (K * 128) + k * 128 + ((((n & 63) >> 3) ^ (k & 7)) << 4) + (n & 7) * 2;
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(__bfloat16_as_ushort(B[n * K + k])) : "memory");
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    if (variant == 0) {
      const uint32_t id = idesc_bf16_f32(kM, N, 0, 0);
      for (int kk = 0; kk < K / 16; ++kk)
        mma_ss(tmem, smem_desc(a_s + kk * 32, 16, 1024, kSwizzle128B), smem_desc(b_s + kk * 32, 16, 1024, kSwizzle128B),
               id, kk > 0);
    } else if (variant == 1) {
      const uint32_t id = idesc_bf16_f32(kM, N, 0, 0);
      for (int kk = 0; kk < K / 16; ++kk)
        mma_ts(tmem, a_tmem + kk * 8, smem_desc(b_s + kk * 32, 16, 1024, kSwizzle128B), id, kk > 0);
    } else if (variant == 2 || variant == 5) {
      const uint32_t id = idesc_bf16_f32(kM, N, 0, 1);
      const uint32_t lbo = variant == 2 ? K * 128 : 1024, sbo = variant == 2 ? 1024 : K * 128;
      for (int kk = 0; kk < K / 16; ++kk)
        mma_ss(tmem, smem_desc(a_s + kk * 32, 16, 1024, kSwizzle128B),
               smem_desc(b_s + kk * 2048, lbo, sbo, kSwizzle128B), id, kk > 0);
    } else if (variant == 3) {
      const uint32_t id = idesc_bf16_f32(kM, N, 0, 0);
      for (int kk = 0; kk < K / 16; ++kk)
        mma_ts(tmem, a_tmem + kk * 8, smem_desc(b_s + kk * 32, 16, 512, kSwizzle64B), id, kk > 0);
    } else if (variant == 4) {
      const uint32_t id = idesc_bf16_f32(kM, N, 0, 0);
      for (int kk = 0; kk < 6; ++kk) {
        const uint64_t bd = kk < 4 ? smem_desc(b_s + kk * 32, 16, 1024, kSwizzle128B)
                                   : smem_desc(b_s + 16384 + (kk - 4) * 32, 16, 512, kSwizzle64B);
        mma_ts(tmem, a_tmem + kk * 8, bd, id, kk > 0);
      }
    }
    mma_commit(smem_u32(&bar));
  }
  // wait for completion (bounded)
  bool ok = mbar_try_wait(smem_u32(&bar), 0);
  long long t0 = clock64();
  while (!ok) {
    ok = mbar_try_wait(smem_u32(&bar), 0);
    if (!ok && clock64() - t0 > (1ll << 31)) break;
  }
  if (!ok && tid == 0) atomicExch(status, 1);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t v[32];
      tmem_ld32_sync(tmem + (uint32_t(warp * 32) << 16) + c0, v);
      for (int j = 0; j < 32; ++j) D[tid * N + c0 + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int tc_probe_run(int variant, int N, int K, const void* A, const void* B, void* D, int* status,
                            void* stream) {
  if (N % 64 || N > 256 || K % 16 || K > 96) return -3;
  const size_t smem = 1024 + 16384 + 49152;
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  probe_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      variant, N, K, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
      static_cast<float*>(D), status);
  return cudaGetLastError() == cudaSuccess ? 0 : -7;
}
