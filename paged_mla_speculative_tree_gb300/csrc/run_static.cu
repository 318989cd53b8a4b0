// Allocation-free entry point: the same verify-attention kernels as
// mla_tree_verify_run, with the workspace (device error word + split-K
// partials) placed in a fixed, file-scope device array instead of memory the
// caller allocates.
//
// Who needs it: code that may not allocate device memory at the point where
// it runs attention -- for example a serving step that is being recorded
// into a CUDA graph (allocation calls are not allowed while a stream is
// capturing), a host framework that owns every device allocation through its
// own pool and forbids side allocations, or a latency-critical path that must
// not risk an allocator call or fragmentation.  Such callers still own and
// pass every input and output buffer; only the scratch space moves here.
#include <mutex>

#include "mtv_internal.cuh"

namespace {

// Every GPU that loads this library holds this array until the process exits.
constexpr uint64_t kStaticScratchBytes = uint64_t(64) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for `device` (which must be current).
// Resolved once per device; the host-side name of the array is not a device
// address and must never be handed to a kernel.
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return MTV_E_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MTV_E_CUDA;
    }
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return MTV_OK;
}

}  // namespace

extern "C" int mla_tree_verify_run_static(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                                          int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                                          const int32_t* kv_indptr, const int64_t* out_cache_loc,
                                          int64_t out_cache_loc_len, const int64_t* qo_indptr,
                                          const uint8_t* custom_mask, int64_t custom_mask_len,
                                          const int64_t* mask_indptr, float scale, void* out, float* lse,
                                          void* stream) {
  if (!plan) return MTV_E_NULL_POINTER;
  if (plan->magic != MTV_PLAN_MAGIC || plan->version != MTV_ABI_VERSION) return MTV_E_BAD_PLAN;
  if (plan->ws_bytes > kStaticScratchBytes) return MTV_E_WORKSPACE_SMALL;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  if (device != plan->device) return MTV_E_DEVICE;
  void* ws = nullptr;
  const int rc = scratch_address(device, &ws);
  if (rc != MTV_OK) return rc;
  // The error word is the only part of the scratch that must start at zero
  // (the partials are always written before they are read).
  if (cudaMemsetAsync(ws, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  return mla_tree_verify_run(plan, q, kv_pool, num_slots, kv_indices, kv_indices_len, kv_indptr, out_cache_loc,
                             out_cache_loc_len, qo_indptr, custom_mask, custom_mask_len, mask_indptr, scale, out,
                             lse, ws, kStaticScratchBytes, stream);
}

// The error word sits at the head of the same fixed array, so reading it
// back needs only the array's device address (no allocation either).
extern "C" int mla_tree_verify_read_static_device_error(uint32_t* flags_out, void* stream) {
  if (!flags_out) return MTV_E_NULL_POINTER;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MTV_E_CUDA;
  }
  void* ws = nullptr;
  const int rc = scratch_address(device, &ws);
  if (rc != MTV_OK) return rc;
  return mla_tree_verify_read_device_error(ws, flags_out, stream);
}
