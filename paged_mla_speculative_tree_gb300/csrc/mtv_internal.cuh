// Internal declarations shared by the kernels and the C-ABI shim of the
// MLA tree-verify library (not installed, not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_tree_verify.h"

namespace mtv {

constexpr int kHeads = 64;
constexpr int kDLat = 512;
constexpr int kDRope = 64;
constexpr int kDQK = kDLat + kDRope;  // 576
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Everything a kernel needs, passed by value (no host data is read by kernels).
struct Params {
  const __nv_bfloat16* q;        // [total_q, 64, 576]
  const __nv_bfloat16* kv_pool;  // [num_slots, 576]
  int64_t num_slots;
  const int64_t* kv_indices;
  const int32_t* kv_indptr;
  const int64_t* out_cache_loc;
  const int64_t* qo_indptr;
  const uint8_t* custom_mask;
  const int64_t* mask_indptr;
  int64_t kv_indices_len, out_cache_loc_len, custom_mask_len;  // elements readable at each buffer
  float scale;       // natural-log domain score scale
  float scale_log2;  // scale * log2(e)
  __nv_bfloat16* out;  // [total_q, 64, 512]
  float* lse;          // [total_q, 64]
  float* part_o;       // [nsplit, total_q_max*64, 512] (nsplit > 1)
  float* part_lse;     // [nsplit, total_q_max*64]
  unsigned* err;       // sticky device error word
  int bs, max_q, mask_layout, nsplit, grid_rows, key_tile;
  int64_t total_q_max, max_prefix, split_keys;
  long long wait_cycles;  // bound of one pipeline wait before the kernel gives up
};

// Per-request geometry read from the device CSR buffers and validated before
// any of it is used as an offset: the plan bounds, monotone offsets, and every
// range the request will index (kv_indices, out_cache_loc and q rows, its mask
// block) inside the buffer lengths given to the run.  ok == false: the request
// is skipped (error bit set, p = n = 0, nothing of it is read or written).
struct Req {
  int64_t p, n, kv_off, q_off, mask_off, keys;
  bool ok;
};

__device__ __forceinline__ Req load_req(const Params& P, int r) {
  Req R;
  const int64_t k0 = P.kv_indptr[r], k1 = P.kv_indptr[r + 1];
  const int64_t q0 = P.qo_indptr[r], q1 = P.qo_indptr[r + 1];
  R.kv_off = k0;
  R.q_off = q0;
  R.mask_off = P.mask_indptr[r];
  R.p = k1 - k0;
  R.n = q1 - q0;
  R.keys = R.p + R.n;
  bool ok = R.p >= 0 && R.n >= 0 && R.p <= P.max_prefix && R.n <= P.max_q && q0 >= 0 &&
            q1 <= P.total_q_max && q1 <= P.out_cache_loc_len && k0 >= 0 && k1 <= P.kv_indices_len &&
            R.mask_off >= 0 && R.mask_off <= P.custom_mask_len;
  if (ok && R.n > 0) {
    // mask block of n rows x (p + n) (FULL_ROW) or n (TREE_ONLY) bytes; the
    // division keeps the product from overflowing
    const int64_t row = (P.mask_layout == MTV_MASK_FULL_ROW) ? R.keys : R.n;
    ok = row <= (P.custom_mask_len - R.mask_off) / R.n;
  }
  R.ok = ok;
  if (!R.ok) {
    atomicOr(P.err, MTV_DEVERR_INDPTR);
    R.p = R.n = R.keys = 0;
  }
  return R;
}

// Slot of key k (prefix keys first, then the tree tokens); -1 if out of range.
__device__ __forceinline__ int64_t key_slot(const Params& P, const Req& R, int64_t k) {
  int64_t s = (k < R.p) ? P.kv_indices[R.kv_off + k] : P.out_cache_loc[R.q_off + (k - R.p)];
  if (s < 0 || s >= P.num_slots) {
    atomicOr(P.err, MTV_DEVERR_SLOT_RANGE);
    return -1;
  }
  return s;
}

// May tree token i see tree token t?  (prefix keys are always visible)
__device__ __forceinline__ bool tree_visible(const Params& P, const Req& R, int64_t i, int64_t t) {
  const int64_t off = (P.mask_layout == MTV_MASK_FULL_ROW) ? R.mask_off + i * R.keys + R.p + t
                                                            : R.mask_off + i * R.n + t;
  return P.custom_mask[off] != 0;
}

// Number of splits that carry keys for a request with `keys` keys (>= 1 so
// that split 0 always writes a result, even for an empty request).
__device__ __forceinline__ int splits_used(const Params& P, int64_t keys) {
  int64_t s = (keys + P.split_keys - 1) / P.split_keys;
  if (s < 1) s = 1;
  if (s > P.nsplit) s = P.nsplit;
  return (int)s;
}

// Launchers (return cudaGetLastError()).
cudaError_t launch_partial_simt(const Params& P, cudaStream_t st);
cudaError_t prepare_partial_simt();
cudaError_t launch_partial_tc(const Params& P, cudaStream_t st);
cudaError_t prepare_partial_tc();
cudaError_t launch_combine(const Params& P, cudaStream_t st, bool programmatic);

// Kernel geometry constants shared by plan and launch.
constexpr int kSimtKeyTile = 32;
constexpr int kSimtThreads = 256;

}  // namespace mtv
