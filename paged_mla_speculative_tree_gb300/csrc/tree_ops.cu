// The steps around verify attention: the visibility mask rebuilt from the
// draft tree's parent array ("The Glue That Binds" -- "The Thinking
// Process"), the greedy acceptance of the verified tree ("The Glue That
// Connects" -- "What the Edit Actually Does": tree building and acceptance
// sit behind the same C ABI as verify attention), and the defragmentation of
// a request's prefix rows into one contiguous run of slots ("The Final Solder
// Joint" -- "The Mandate: Three Priorities"); and the merge of requests that
// share a prefix into one (not on the pages: the plainest extension).
#include <stdint.h>

#include "mla_tree_ops.h"
#include "mtv_internal.cuh"

namespace mtv {
namespace {

constexpr int kMaskThreads = 256;
constexpr int kMaxTreeForMask = 32768;  // dynamic shared memory holds one flag per tree node

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// Size in bytes of request r's mask block (0 for a request whose geometry is
// invalid; that request is flagged by the block that owns its row 0).
__device__ __forceinline__ int64_t mask_block_bytes(const int64_t* qo_indptr, const int32_t* kv_indptr, int r,
                                                    int max_q, int layout, bool* ok) {
  const int64_t n = qo_indptr[r + 1] - qo_indptr[r];
  const int64_t p = layout == MTV_MASK_FULL_ROW ? int64_t(kv_indptr[r + 1]) - kv_indptr[r] : 0;
  *ok = n >= 0 && n <= max_q && p >= 0 && qo_indptr[r] >= 0;
  return *ok ? n * (p + n) : 0;
}

// Block (i, r) writes row i of request r; block (0, r) also writes
// mask_indptr[r + 1] (and block (0, 0) mask_indptr[0]).
__global__ void __launch_bounds__(kMaskThreads) tree_mask_kernel(const int32_t* parents, const int64_t* qo_indptr,
                                                                 const int32_t* kv_indptr, int bs, int max_q,
                                                                 int layout, uint8_t* mask, uint64_t capacity,
                                                                 int64_t* mask_indptr, uint32_t* err) {
  extern __shared__ unsigned char vis[];  // [max_q]: tree column t visible from row i
  __shared__ long long part[kMaskThreads / 32];
  const int i = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;

  // offset of request r = sum of the earlier requests' block sizes
  long long acc = 0;
  for (int rr = tid; rr < r; rr += kMaskThreads) {
    bool ok_rr;
    acc += mask_block_bytes(qo_indptr, kv_indptr, rr, max_q, layout, &ok_rr);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((tid & 31) == 0) part[tid >> 5] = acc;
  __syncthreads();
  long long off = 0;
#pragma unroll
  for (int w = 0; w < kMaskThreads / 32; ++w) off += part[w];

  bool ok;
  const int64_t bytes = mask_block_bytes(qo_indptr, kv_indptr, r, max_q, layout, &ok);
  const int64_t q0 = qo_indptr[r];
  const int64_t n = ok ? qo_indptr[r + 1] - q0 : 0;
  const int64_t p = (ok && layout == MTV_MASK_FULL_ROW) ? int64_t(kv_indptr[r + 1]) - kv_indptr[r] : 0;
  const bool fits = uint64_t(off) + uint64_t(bytes) <= capacity;
  if (i == 0 && tid == 0) {
    if (r == 0) mask_indptr[0] = 0;
    mask_indptr[r + 1] = off + bytes;
    if (!ok || !fits) set_err(err, MTV_DEVERR_INDPTR);
  }
  if (!ok || !fits || i >= n) return;

  const int64_t width = p + n;  // TREE_ONLY: p == 0
  uint8_t* row = mask + off + int64_t(i) * width;

  // ancestors-or-self of node i
  for (int t = tid; t < n; t += kMaskThreads) vis[t] = 0;
  __syncthreads();
  if (tid == 0) {
    int j = i;
    for (int steps = 0; j >= 0 && steps <= i; ++steps) {
      vis[j] = 1;
      const int pj = parents[q0 + j];
      if (pj < -1 || pj >= j) {  // not a tree: treat node j as hanging off the prefix
        set_err(err, MTV_DEVERR_PARENT);
        break;
      }
      j = pj;
    }
  }
  __syncthreads();

  // prefix columns: ones, 16-byte stores on the aligned middle part
  if (p > 0) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row), e = a + uintptr_t(p);
    const uintptr_t a16 = (a + 15) & ~uintptr_t(15), e16 = e & ~uintptr_t(15);
    if (a16 >= e16) {
      for (uintptr_t x = a + tid; x < e; x += kMaskThreads) *reinterpret_cast<uint8_t*>(x) = 1;
    } else {
      for (uintptr_t x = a + tid; x < a16; x += kMaskThreads) *reinterpret_cast<uint8_t*>(x) = 1;
      const uint4 ones = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
      for (uintptr_t x = a16 + 16 * uintptr_t(tid); x < e16; x += 16 * kMaskThreads)
        *reinterpret_cast<uint4*>(x) = ones;
      for (uintptr_t x = e16 + tid; x < e; x += kMaskThreads) *reinterpret_cast<uint8_t*>(x) = 1;
    }
  }
  // tree columns
  for (int t = tid; t < n; t += kMaskThreads) row[p + t] = vis[t];
}

// One warp per request walks the tree from the prefix root.
__global__ void __launch_bounds__(128) tree_accept_kernel(const int32_t* parents, const int32_t* draft,
                                                          const int32_t* target, const int32_t* target_root,
                                                          const int64_t* out_cache_loc, const int64_t* qo_indptr,
                                                          int bs, int max_q, int32_t* accept_len,
                                                          int32_t* accept_nodes, int64_t* accept_slots,
                                                          int32_t* bonus, uint32_t* err) {
  const int r = int((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= bs) return;
  const int64_t q0 = qo_indptr[r];
  int64_t n = qo_indptr[r + 1] - q0;
  if (n < 0 || n > max_q || q0 < 0) {
    if (lane == 0) set_err(err, MTV_DEVERR_INDPTR);
    n = 0;
  }
  int32_t* nodes = accept_nodes + int64_t(r) * max_q;
  int64_t* slots = accept_slots + int64_t(r) * max_q;
  int cur = -1, want = target_root[r], len = 0;
  for (;;) {
    int nxt = -1;
    for (int64_t b = 0; b < n && nxt < 0; b += 32) {
      const int64_t c = b + lane;
      bool m = false;
      if (c < n) {
        int pc = parents[q0 + c];
        if (pc < -1 || pc >= c) {
          set_err(err, MTV_DEVERR_PARENT);
          pc = -1;
        }
        m = pc == cur && draft[q0 + c] == want;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, m);
      if (hit) nxt = int(b) + __ffs(hit) - 1;  // lowest-index matching child
    }
    if (nxt < 0) break;  // children have larger indices than their parents: at most n steps
    if (lane == 0) {
      nodes[len] = nxt;
      slots[len] = out_cache_loc[q0 + nxt];
    }
    ++len;
    cur = nxt;
    want = target[q0 + nxt];
  }
  for (int k = len + lane; k < max_q; k += 32) {
    nodes[k] = -1;
    slots[k] = -1;
  }
  if (lane == 0) {
    accept_len[r] = len;
    bonus[r] = want;
  }
}

// Warp w of block (x, r) copies prefix row j = 8x + w of request r: 72
// 16-byte units of the 1152-byte row, all loads issued before the stores.
constexpr int kDefragRowsPerBlock = 8;
constexpr int kRowUnits = kDQK * 2 / 16;  // 72

__global__ void __launch_bounds__(32 * kDefragRowsPerBlock) kv_defrag_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t num_slots, const int64_t* kv_indices,
    const int32_t* kv_indptr, int64_t max_prefix, const int64_t* dst_base, int64_t* kv_indices_out,
    uint32_t* err) {
  const int r = blockIdx.y, lane = threadIdx.x & 31;
  const int64_t j = int64_t(blockIdx.x) * kDefragRowsPerBlock + (threadIdx.x >> 5);
  const int64_t k0 = kv_indptr[r];
  const int64_t p = int64_t(kv_indptr[r + 1]) - k0;
  if (p < 0 || p > max_prefix || k0 < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, MTV_DEVERR_INDPTR);
    return;
  }
  if (j >= p) return;
  const int64_t s = kv_indices[k0 + j];
  const int64_t d = dst_base[r] + j;
  if (s < 0 || s >= num_slots || d < 0 || d >= num_slots) {
    if (lane == 0) set_err(err, MTV_DEVERR_SLOT_RANGE);
    return;
  }
  const uint4* a = src + s * kRowUnits;
  uint4* b = dst + d * kRowUnits;
  uint4 v0 = a[lane], v1 = a[lane + 32], v2 = make_uint4(0u, 0u, 0u, 0u);
  if (lane + 64 < kRowUnits) v2 = a[lane + 64];
  b[lane] = v0;
  b[lane + 32] = v1;
  if (lane + 64 < kRowUnits) b[lane + 64] = v2;
  if (lane == 0) kv_indices_out[k0 + j] = d;
}

// Block (g, y) of the grouping kernel: slice y of group g's leader prefix is
// copied and compared with every follower's; block y == 0 also publishes the
// group's offsets and remaps the parents of the group's tokens.
constexpr int kGroupThreads = 256;
constexpr int kGroupSlices = 16;

__global__ void __launch_bounds__(kGroupThreads) group_prefix_kernel(
    const int32_t* group_indptr, int num_groups, int64_t max_prefix, const int64_t* kv_indices,
    const int32_t* kv_indptr, const int64_t* qo_indptr, const int32_t* parents, int32_t* kv_indptr_out,
    int64_t* kv_indices_out, int64_t* qo_indptr_out, int32_t* parents_out, uint32_t* err) {
  __shared__ long long part[kGroupThreads / 32];
  const int g = blockIdx.x, y = blockIdx.y, tid = threadIdx.x;
  const int r0 = group_indptr[g], r1 = group_indptr[g + 1];
  auto leader_len = [&](int gg) -> int64_t {
    const int a = group_indptr[gg], b = group_indptr[gg + 1];
    if (b <= a) return 0;
    const int64_t p = int64_t(kv_indptr[a + 1]) - kv_indptr[a];
    return (p < 0 || p > max_prefix) ? 0 : p;
  };
  // output offset of this group's prefix: leaders' lengths of the earlier groups
  long long acc = 0;
  for (int gg = tid; gg < g; gg += kGroupThreads) acc += leader_len(gg);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((tid & 31) == 0) part[tid >> 5] = acc;
  __syncthreads();
  long long off = 0;
#pragma unroll
  for (int w = 0; w < kGroupThreads / 32; ++w) off += part[w];
  const int64_t p = leader_len(g);
  if (y == 0 && tid == 0) {
    if (g == 0) {
      kv_indptr_out[0] = 0;
      qo_indptr_out[0] = qo_indptr[r0];
    }
    kv_indptr_out[g + 1] = int32_t(off + p);
    qo_indptr_out[g + 1] = qo_indptr[r1 > r0 ? r1 : r0];
    if (r1 > r0) {
      const int64_t p_raw = int64_t(kv_indptr[r0 + 1]) - kv_indptr[r0];
      if (p_raw < 0 || p_raw > max_prefix) set_err(err, MTV_DEVERR_INDPTR);
    }
  }
  if (r1 <= r0) return;
  // slice y of the prefix: copy the leader's slots, compare the followers'
  const int64_t lo = p * y / kGroupSlices, hi = p * (y + 1) / kGroupSlices;
  const int64_t k_lead = kv_indptr[r0];
  bool bad = false;
  for (int64_t j = lo + tid; j < hi; j += kGroupThreads) {
    const int64_t s = kv_indices[k_lead + j];
    kv_indices_out[off + j] = s;
    for (int r = r0 + 1; r < r1; ++r) {
      const int64_t pr = int64_t(kv_indptr[r + 1]) - kv_indptr[r];
      if (pr != p) bad = true;  // (only a follower of the same length is read)
      else if (kv_indices[kv_indptr[r] + j] != s) bad = true;
    }
  }
  if (y == 0 && tid < r1 - r0 - 1) {  // a follower with a different length but no slots compared above
    const int r = r0 + 1 + tid;
    if (int64_t(kv_indptr[r + 1]) - kv_indptr[r] != p) bad = true;
  }
  if (bad) set_err(err, MTV_DEVERR_PREFIX);
  // parents of the group's tokens, shifted by each request's offset in the merged tree
  const int64_t q0 = qo_indptr[r0];
  for (int r = r0; r < r1; ++r) {
    const int64_t a = qo_indptr[r], b = qo_indptr[r + 1];
    const int64_t shift = a - q0;
    for (int64_t t = a + int64_t(y) * kGroupThreads + tid; t < b; t += int64_t(kGroupSlices) * kGroupThreads) {
      const int32_t par = parents[t];
      parents_out[t] = par < 0 ? -1 : int32_t(par + shift);
    }
  }
}

}  // namespace
}  // namespace mtv

extern "C" int mla_tree_group_prefix(const int32_t* group_indptr, int num_groups, int64_t max_group_prefix,
                                     const int64_t* kv_indices, const int32_t* kv_indptr, const int64_t* qo_indptr,
                                     const int32_t* parents, int32_t* kv_indptr_out, int64_t* kv_indices_out,
                                     int64_t* qo_indptr_out, int32_t* parents_out, uint32_t* err, void* stream) {
  if (num_groups < 0 || max_group_prefix < 0 || max_group_prefix > INT32_MAX) return MTV_E_BAD_ARGUMENT;
  if (num_groups == 0) return MTV_OK;
  if (!group_indptr || !kv_indices || !kv_indptr || !qo_indptr || !parents || !kv_indptr_out || !kv_indices_out ||
      !qo_indptr_out || !parents_out)
    return MTV_E_NULL_POINTER;
  const dim3 grid(static_cast<unsigned>(num_groups), static_cast<unsigned>(mtv::kGroupSlices));
  mtv::group_prefix_kernel<<<grid, mtv::kGroupThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      group_indptr, num_groups, max_group_prefix, kv_indices, kv_indptr, qo_indptr, parents, kv_indptr_out,
      kv_indices_out, qo_indptr_out, parents_out, err);
  return cudaGetLastError() == cudaSuccess ? MTV_OK : MTV_E_CUDA;
}

extern "C" int mla_kv_defrag(const void* kv_src, void* kv_dst, int64_t num_slots, const int64_t* kv_indices,
                             const int32_t* kv_indptr, int bs, int64_t max_prefix, const int64_t* dst_base,
                             int64_t* kv_indices_out, uint32_t* err, void* stream) {
  if (bs < 0 || max_prefix < 0 || num_slots < 0) return MTV_E_BAD_ARGUMENT;
  if (bs == 0 || max_prefix == 0) return MTV_OK;
  if (!kv_src || !kv_dst || !kv_indices || !kv_indptr || !dst_base || !kv_indices_out) return MTV_E_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(kv_src) | reinterpret_cast<uintptr_t>(kv_dst)) & 15) return MTV_E_BAD_ARGUMENT;
  const int64_t gx = (max_prefix + mtv::kDefragRowsPerBlock - 1) / mtv::kDefragRowsPerBlock;
  if (gx > 0x7fffffff || bs > 65535) return MTV_E_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(bs));
  mtv::kv_defrag_kernel<<<grid, 32 * mtv::kDefragRowsPerBlock, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(kv_src), static_cast<uint4*>(kv_dst), num_slots, kv_indices, kv_indptr, max_prefix,
      dst_base, kv_indices_out, err);
  return cudaGetLastError() == cudaSuccess ? MTV_OK : MTV_E_CUDA;
}

extern "C" int mla_tree_mask_build(const int32_t* parents, const int64_t* qo_indptr, const int32_t* kv_indptr,
                                   int bs, int max_q_per_req, int mask_layout, uint8_t* custom_mask,
                                   uint64_t mask_capacity, int64_t* mask_indptr, uint32_t* err, void* stream) {
  if (bs < 0 || max_q_per_req < 0) return MTV_E_BAD_ARGUMENT;
  if (mask_layout != MTV_MASK_FULL_ROW && mask_layout != MTV_MASK_TREE_ONLY) return MTV_E_BAD_ARGUMENT;
  if (!mask_indptr) return MTV_E_NULL_POINTER;
  if (max_q_per_req > mtv::kMaxTreeForMask) return MTV_E_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bs == 0) {
    if (cudaMemsetAsync(mask_indptr, 0, sizeof(int64_t), st) != cudaSuccess) {
      cudaGetLastError();
      return MTV_E_CUDA;
    }
    return MTV_OK;
  }
  if (!qo_indptr || (!parents && max_q_per_req > 0) || (!custom_mask && mask_capacity > 0) ||
      (mask_layout == MTV_MASK_FULL_ROW && !kv_indptr))
    return MTV_E_NULL_POINTER;
  const dim3 grid(unsigned(max_q_per_req > 0 ? max_q_per_req : 1), unsigned(bs));
  mtv::tree_mask_kernel<<<grid, mtv::kMaskThreads, size_t(max_q_per_req > 0 ? max_q_per_req : 1), st>>>(
      parents, qo_indptr, kv_indptr, bs, max_q_per_req, mask_layout, custom_mask, mask_capacity, mask_indptr, err);
  return cudaGetLastError() == cudaSuccess ? MTV_OK : MTV_E_CUDA;
}

extern "C" int mla_tree_accept(const int32_t* parents, const int32_t* draft_tokens, const int32_t* target_tokens,
                               const int32_t* target_root_tokens, const int64_t* out_cache_loc,
                               const int64_t* qo_indptr, int bs, int max_q_per_req, int32_t* accept_len,
                               int32_t* accept_nodes, int64_t* accept_slots, int32_t* bonus_tokens, uint32_t* err,
                               void* stream) {
  if (bs < 0 || max_q_per_req < 0) return MTV_E_BAD_ARGUMENT;
  if (bs == 0) return MTV_OK;
  if (!qo_indptr || !target_root_tokens || !accept_len || !bonus_tokens) return MTV_E_NULL_POINTER;
  if (max_q_per_req > 0 &&
      (!parents || !draft_tokens || !target_tokens || !out_cache_loc || !accept_nodes || !accept_slots))
    return MTV_E_NULL_POINTER;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int threads = 128;
  const unsigned blocks = unsigned((int64_t(bs) * 32 + threads - 1) / threads);
  mtv::tree_accept_kernel<<<blocks, threads, 0, st>>>(parents, draft_tokens, target_tokens, target_root_tokens,
                                                      out_cache_loc, qo_indptr, bs, max_q_per_req, accept_len,
                                                      accept_nodes, accept_slots, bonus_tokens, err);
  return cudaGetLastError() == cudaSuccess ? MTV_OK : MTV_E_CUDA;
}
