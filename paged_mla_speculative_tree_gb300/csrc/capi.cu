// C-ABI shim of the MLA tree-verify library: plan (host only, from upper
// bounds) and run (argument checks + kernel launches on the caller's stream;
// no sync, no allocation, capture-safe).  The split into a small extern "C"
// surface over device pointers and a stream follows "The Glue That Makes
// Kernels Run" -- "The Decision Architecture" (C-ABI as the integration
// boundary) and "The Final Solder Joint" -- "Why the C-ABI Edit Matters".
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

#include "mtv_internal.cuh"

using namespace mtv;

namespace {

constexpr uint64_t kWsHeader = 256;

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Split-K choice for the SIMT floor: enough CTAs for ~2 waves, >= 256 keys per split.
int choose_nsplit_simt(int num_sms, int64_t ctas_per_split, int64_t max_keys) {
  if (ctas_per_split <= 0) return 1;
  int64_t want = ceil_div(2 * int64_t(num_sms), ctas_per_split);
  int64_t cap = std::max<int64_t>(1, ceil_div(max_keys, 256));
  return int(std::max<int64_t>(1, std::min<int64_t>({want, cap, 64})));
}

}  // namespace

// Defined in partial_tc.cu: picks split count for the tensor-core kernel.
namespace mtv {
int choose_nsplit_tc(int num_sms, int64_t pairs_per_split, int64_t max_keys, int64_t rows_total);
extern const int kTcRowTile;
extern const int kTcKeyTile;
}  // namespace mtv

namespace {

// Estimated partial + combine time (us) of a ragged batch split `ns` ways:
// the partial kernel's work units (one CTA pair per 128-row block and split,
// in grid order: split-major, then request, then row block) are handed to
// the first free SM pair; a unit costs a fixed set-up/epilogue time plus its
// 64-key tiles, an empty one (past its request's rows or keys) almost
// nothing.  The constants were fitted to measured split-count sweeps on a
// GB300 at 2.07 GHz (Long, Batch-4, the Stress request shape and three Mixed
// draws).  split_keys is derived from max_keys exactly as the plan does.
// With `bound` > 0 the estimate stops early (returning a value above
// `bound`) once the work divided evenly over the SM pairs already exceeds it.
double estimate_ragged_us(int slots, int bs, const int64_t* keys, const int64_t* row_blocks, int64_t max_keys,
                          int64_t max_row_blocks, int64_t rows_total, int ns, int* ns_used, double bound) {
  constexpr double kTileUs = 1.24, kUnitUs = 6.0, kEmptyUs = 0.2, kCombineUs = 8.0, kHbmBytesPerUs = 6.0e6;
  const int64_t split_keys = ceil_div(ceil_div(max_keys, ns), kTcKeyTile) * kTcKeyTile;
  const int64_t used = std::max<int64_t>(1, ceil_div(max_keys, split_keys));
  *ns_used = int(used);
  const double combine =
      used > 1 ? double(used) * double(rows_total) * kDLat * 4.0 * 2.0 / kHbmBytesPerUs + kCombineUs : 0.0;
  if (bound > 0.0) {
    double work = 0.0;
    for (int r = 0; r < bs; ++r) {
      const int64_t live = std::max<int64_t>(1, ceil_div(keys[r], split_keys));  // splits holding keys
      work += double(row_blocks[r]) * (double(live) * kUnitUs + double(ceil_div(std::max<int64_t>(1, keys[r]),
                                                                                kTcKeyTile)) * kTileUs);
    }
    if (work / slots + combine > bound) return work / slots + combine;
  }
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < slots; ++i) free_at.push(0.0);
  double makespan = 0.0;
  for (int64_t s = 0; s < used; ++s) {
    for (int r = 0; r < bs; ++r) {
      const int64_t k0 = s * split_keys;
      const bool live = s == 0 || k0 < keys[r];  // split 0 always writes a result
      const int64_t tiles = live ? ceil_div(std::max<int64_t>(1, std::min(split_keys, keys[r] - k0)), kTcKeyTile) : 0;
      for (int64_t rb = 0; rb < max_row_blocks; ++rb) {
        const double cost = (live && rb < row_blocks[r]) ? kUnitUs + double(tiles) * kTileUs : kEmptyUs;
        const double t = free_at.top() + cost;
        free_at.pop();
        free_at.push(t);
        makespan = std::max(makespan, t);
      }
    }
  }
  return makespan + combine;
}

}  // namespace

extern "C" {

const char* mla_tree_verify_strerror(int code) {
  switch (code) {
    case MTV_OK: return "ok";
    case MTV_E_NULL_POINTER: return "a required pointer is NULL";
    case MTV_E_UNSUPPORTED: return "unsupported shape (needs 64 heads, 512 latent + 64 rope dims)";
    case MTV_E_BAD_ARGUMENT: return "bad argument (negative size, unknown mask layout or flag)";
    case MTV_E_WORKSPACE_SMALL: return "workspace smaller than plan->ws_bytes";
    case MTV_E_WORKSPACE_ALIGN: return "workspace not 256-byte aligned";
    case MTV_E_BAD_PLAN: return "plan was not produced by mla_tree_verify_plan (or wrong ABI version)";
    case MTV_E_CUDA: return "CUDA runtime call or kernel launch failed";
    case MTV_E_DEVICE: return "device unusable (needs an sm_103 GPU; plan device must be current)";
    default: return "unknown error code";
  }
}

int mla_tree_verify_choose_nsplit(int num_sms, int bs, const int64_t* prefix_lens, const int32_t* tree_sizes,
                                  int flags, int* nsplit_out) {
  if (!nsplit_out) return MTV_E_NULL_POINTER;
  if (num_sms < 2 || bs < 0) return MTV_E_BAD_ARGUMENT;
  if (flags & ~(MTV_FLAG_SIMT_FLOOR | MTV_FLAG_TEST_SHORT_WAITS)) return MTV_E_BAD_ARGUMENT;
  if (bs > 0 && (!prefix_lens || !tree_sizes)) return MTV_E_NULL_POINTER;
  int64_t max_prefix = 0, max_q = 0, rows_total = 0;
  bool uniform = true;
  for (int r = 0; r < bs; ++r) {
    if (prefix_lens[r] < 0 || tree_sizes[r] < 0) return MTV_E_BAD_ARGUMENT;
    max_prefix = std::max(max_prefix, prefix_lens[r]);
    max_q = std::max<int64_t>(max_q, tree_sizes[r]);
    rows_total += int64_t(tree_sizes[r]) * kHeads;
    uniform = uniform && prefix_lens[r] == prefix_lens[0] && tree_sizes[r] == tree_sizes[0];
  }
  // the plan's key bound (a run may present max_prefix + max_q keys)
  const int64_t max_keys = std::max<int64_t>(1, max_prefix + max_q);
  if (bs == 0 || max_q == 0) {
    *nsplit_out = 1;
    return MTV_OK;
  }
  if (flags & MTV_FLAG_SIMT_FLOOR) {
    *nsplit_out = choose_nsplit_simt(num_sms, int64_t(bs) * max_q, max_keys);
    return MTV_OK;
  }
  const int64_t max_rb = ceil_div(max_q * kHeads, kTcRowTile);
  // the plan's own choice for a batch of equal requests, and for batches too
  // large to simulate cheaply (the estimate walks every work unit)
  if (uniform || int64_t(bs) * max_rb > (int64_t(1) << 16)) {
    *nsplit_out = choose_nsplit_tc(num_sms, int64_t(bs) * max_rb, max_keys, int64_t(bs) * max_q * kHeads);
    return MTV_OK;
  }
  std::vector<int64_t> keys(bs), rbs(bs);
  for (int r = 0; r < bs; ++r) {
    keys[r] = prefix_lens[r] + tree_sizes[r];
    rbs[r] = ceil_div(int64_t(tree_sizes[r]) * kHeads, kTcRowTile);
  }
  // estimate every distinct split count; keep the smallest within 2 % of the best
  std::vector<std::pair<int, double>> est;
  int prev_used = 0;
  double best_so_far = 0.0;  // estimates above 1.02x the best so far cannot be picked: bound them
  for (int ns = 1; ns <= 64; ++ns) {
    int used = 0;
    const double t = estimate_ragged_us(num_sms / 2, bs, keys.data(), rbs.data(), max_keys, max_rb, rows_total, ns,
                                        &used, best_so_far * 1.02);
    best_so_far = best_so_far > 0.0 ? std::min(best_so_far, t) : t;
    if (used == prev_used) continue;  // same split length as a smaller count
    prev_used = used;
    est.emplace_back(used, t);
    if (int64_t(used) * kTcKeyTile >= max_keys) break;  // one tile per split
  }
  double best = 1e300;
  for (const auto& e : est) best = std::min(best, e.second);
  int pick = 1;
  for (const auto& e : est) {
    if (e.second <= best * 1.02) {
      pick = e.first;
      break;
    }
  }
  *nsplit_out = pick;
  return MTV_OK;
}

int mla_tree_verify_plan(int device, int bs, int max_q_per_req, int64_t total_q_max,
                         int64_t max_prefix, int num_heads, int d_latent, int d_rope,
                         int mask_layout, int flags, int nsplit_override, mtv_plan_t* plan_out,
                         uint64_t* ws_bytes_out) {
  if (!plan_out) return MTV_E_NULL_POINTER;
  if (num_heads != kHeads || d_latent != kDLat || d_rope != kDRope) return MTV_E_UNSUPPORTED;
  if (bs < 0 || max_q_per_req < 0 || total_q_max < 0 || max_prefix < 0 || nsplit_override < 0)
    return MTV_E_BAD_ARGUMENT;
  if (mask_layout != MTV_MASK_FULL_ROW && mask_layout != MTV_MASK_TREE_ONLY) return MTV_E_BAD_ARGUMENT;
  if (flags & ~(MTV_FLAG_SIMT_FLOOR | MTV_FLAG_TEST_SHORT_WAITS)) return MTV_E_BAD_ARGUMENT;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return MTV_E_DEVICE;
  }
  int sms = 0, ccmaj = 0, ccmin = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ccmaj, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ccmin, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  if (ccmaj != 10 || ccmin != 3) return MTV_E_DEVICE;

  mtv_plan_t p;
  memset(&p, 0, sizeof p);
  p.magic = MTV_PLAN_MAGIC;
  p.version = MTV_ABI_VERSION;
  p.device = device;
  p.num_sms = sms;
  p.cc_major = ccmaj;
  p.cc_minor = ccmin;
  p.bs = bs;
  p.max_q_per_req = max_q_per_req;
  p.num_heads = num_heads;
  p.d_latent = d_latent;
  p.d_rope = d_rope;
  p.mask_layout = mask_layout;
  p.flags = flags;
  p.total_q_max = total_q_max;
  p.max_prefix = max_prefix;
  const int64_t max_keys = std::max<int64_t>(1, max_prefix + max_q_per_req);

  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MTV_E_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return MTV_E_CUDA;
  cudaError_t prep;
  if (flags & MTV_FLAG_SIMT_FLOOR) {
    p.row_tile = kHeads;
    p.key_tile = kSimtKeyTile;
    p.grid_rows = max_q_per_req;
    const int64_t ctas = int64_t(bs) * max_q_per_req;
    p.nsplit = nsplit_override ? nsplit_override : choose_nsplit_simt(sms, ctas, max_keys);
    prep = prepare_partial_simt();
  } else {
    p.row_tile = kTcRowTile;
    p.key_tile = kTcKeyTile;
    p.grid_rows = int(ceil_div(int64_t(max_q_per_req) * kHeads, kTcRowTile));
    const int64_t pairs = int64_t(bs) * p.grid_rows;
    p.nsplit = nsplit_override ? nsplit_override
                               : choose_nsplit_tc(sms, pairs, max_keys, int64_t(bs) * max_q_per_req * kHeads);
    prep = prepare_partial_tc();
  }
  if (prev != device) cudaSetDevice(prev);
  if (prep != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  p.nsplit = std::max(1, std::min(p.nsplit, 1024));
  p.split_keys = ceil_div(ceil_div(max_keys, p.nsplit), p.key_tile) * p.key_tile;
  p.nsplit = int(std::max<int64_t>(1, ceil_div(max_keys, p.split_keys)));

  uint64_t ws = kWsHeader;
  if (p.nsplit > 1) {
    const uint64_t rows = uint64_t(total_q_max) * kHeads;
    p.ws_part_o = ws;
    ws = align256(ws + uint64_t(p.nsplit) * rows * kDLat * sizeof(float));
    p.ws_part_lse = ws;
    ws = align256(ws + uint64_t(p.nsplit) * rows * sizeof(float));
  }
  p.ws_bytes = ws;
  *plan_out = p;
  if (ws_bytes_out) *ws_bytes_out = ws;
  return MTV_OK;
}

}  // extern "C"

// Host checks and kernel launches shared by run and run_steps.
static int run_impl(const mtv_plan_t* plan, const void* q, const void* kv_pool, int64_t num_slots,
                    const int64_t* kv_indices, int64_t kv_indices_len, const int32_t* kv_indptr,
                    const int64_t* out_cache_loc, int64_t out_cache_loc_len, const int64_t* qo_indptr,
                    const uint8_t* custom_mask, int64_t custom_mask_len, const int64_t* mask_indptr,
                    float scale, void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                    int steps, void* stream) {
  if ((steps & ~(MTV_STEP_PARTIAL | MTV_STEP_COMBINE)) || steps == 0) return MTV_E_BAD_ARGUMENT;
  if (!plan) return MTV_E_NULL_POINTER;
  if (plan->magic != MTV_PLAN_MAGIC || plan->version != MTV_ABI_VERSION) return MTV_E_BAD_PLAN;
  if (!workspace || !kv_indptr || !qo_indptr || !mask_indptr) return MTV_E_NULL_POINTER;
  if (kv_indices_len < 0 || out_cache_loc_len < 0 || custom_mask_len < 0) return MTV_E_BAD_ARGUMENT;
  if ((kv_indices_len > 0 && !kv_indices) || (out_cache_loc_len > 0 && !out_cache_loc) ||
      (custom_mask_len > 0 && !custom_mask))
    return MTV_E_NULL_POINTER;
  if (plan->bs > 0 && plan->total_q_max > 0 && (!q || !kv_pool || !out || !lse)) return MTV_E_NULL_POINTER;
  // The gather warps hold a checked slot in a 32-bit register.
  if (num_slots < 0 || num_slots > INT32_MAX) return MTV_E_BAD_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(kv_pool) & 15) return MTV_E_BAD_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MTV_E_WORKSPACE_ALIGN;
  if (workspace_bytes < plan->ws_bytes) return MTV_E_WORKSPACE_SMALL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  if (cur != plan->device) return MTV_E_DEVICE;
  if (plan->bs == 0 || plan->total_q_max == 0 || plan->max_q_per_req == 0) return MTV_OK;

  Params P;
  memset(&P, 0, sizeof P);
  P.q = static_cast<const __nv_bfloat16*>(q);
  P.kv_pool = static_cast<const __nv_bfloat16*>(kv_pool);
  P.num_slots = num_slots;
  P.kv_indices = kv_indices;
  P.kv_indptr = kv_indptr;
  P.out_cache_loc = out_cache_loc;
  P.qo_indptr = qo_indptr;
  P.custom_mask = custom_mask;
  P.mask_indptr = mask_indptr;
  P.kv_indices_len = kv_indices_len;
  P.out_cache_loc_len = out_cache_loc_len;
  P.custom_mask_len = custom_mask_len;
  P.scale = scale;
  P.scale_log2 = scale * kLog2e;
  P.out = static_cast<__nv_bfloat16*>(out);
  P.lse = lse;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  P.err = reinterpret_cast<unsigned*>(ws);
  P.part_o = plan->nsplit > 1 ? reinterpret_cast<float*>(ws + plan->ws_part_o) : nullptr;
  P.part_lse = plan->nsplit > 1 ? reinterpret_cast<float*>(ws + plan->ws_part_lse) : nullptr;
  P.bs = plan->bs;
  P.max_q = plan->max_q_per_req;
  P.mask_layout = plan->mask_layout;
  P.nsplit = plan->nsplit;
  P.grid_rows = plan->grid_rows;
  P.key_tile = plan->key_tile;
  P.total_q_max = plan->total_q_max;
  P.max_prefix = plan->max_prefix;
  P.split_keys = plan->split_keys;
  // ~1 s at the GB300's clock; the test flag makes any wait that has to spin give up
  P.wait_cycles = (plan->flags & MTV_FLAG_TEST_SHORT_WAITS) ? 0ll : (1ll << 31);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (steps & MTV_STEP_PARTIAL)
    e = (plan->flags & MTV_FLAG_SIMT_FLOOR) ? launch_partial_simt(P, st) : launch_partial_tc(P, st);
  // Launched right behind the partial kernel, the combine is its programmatic
  // dependent; launched alone it waits for the stream's earlier work as usual.
  if (e == cudaSuccess && plan->nsplit > 1 && (steps & MTV_STEP_COMBINE))
    e = launch_combine(P, st, (steps & MTV_STEP_PARTIAL) != 0);
  if (e != cudaSuccess) return MTV_E_CUDA;
  return MTV_OK;
}

extern "C" {

int mla_tree_verify_run(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                        int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                        const int32_t* kv_indptr, const int64_t* out_cache_loc,
                        int64_t out_cache_loc_len, const int64_t* qo_indptr,
                        const uint8_t* custom_mask, int64_t custom_mask_len,
                        const int64_t* mask_indptr, float scale, void* out, float* lse,
                        void* workspace, uint64_t workspace_bytes, void* stream) {
  return run_impl(plan, q, kv_pool, num_slots, kv_indices, kv_indices_len, kv_indptr, out_cache_loc,
                  out_cache_loc_len, qo_indptr, custom_mask, custom_mask_len, mask_indptr, scale, out, lse,
                  workspace, workspace_bytes, MTV_STEP_PARTIAL | MTV_STEP_COMBINE, stream);
}

int mla_tree_verify_run_steps(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                              int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                              const int32_t* kv_indptr, const int64_t* out_cache_loc,
                              int64_t out_cache_loc_len, const int64_t* qo_indptr,
                              const uint8_t* custom_mask, int64_t custom_mask_len,
                              const int64_t* mask_indptr, float scale, void* out, float* lse,
                              void* workspace, uint64_t workspace_bytes, int steps, void* stream) {
  return run_impl(plan, q, kv_pool, num_slots, kv_indices, kv_indices_len, kv_indptr, out_cache_loc,
                  out_cache_loc_len, qo_indptr, custom_mask, custom_mask_len, mask_indptr, scale, out, lse,
                  workspace, workspace_bytes, steps, stream);
}

int mla_tree_verify_clear_device_error(void* workspace, void* stream) {
  if (!workspace) return MTV_E_NULL_POINTER;
  if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  return MTV_OK;
}

int mla_tree_verify_read_device_error(const void* workspace, uint32_t* flags_out, void* stream) {
  if (!workspace || !flags_out) return MTV_E_NULL_POINTER;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  *flags_out = v;
  return MTV_OK;
}

}  // extern "C"
