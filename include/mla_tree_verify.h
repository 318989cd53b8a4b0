/*
 * mla_tree_verify.h -- C ABI of the GB300 (sm_103a) MLA tree-verify attention library.
 *
 * The operation (one speculative-decoding verify step of Multi-head Latent
 * Attention over a paged latent KV pool):
 *
 *   for every request r, draft-tree token i < n_r and head h < 64:
 *     keys  = the r-th prefix (slots kv_indices[kv_indptr[r] .. kv_indptr[r+1]))
 *           + the tree tokens t whose custom_mask bit for (i, t) is set
 *             (slots out_cache_loc[qo_indptr[r] + t])
 *     s_k   = scale * <q[qo_indptr[r]+i, h, 0:576], kv_pool[slot_k, 0:576]>
 *     out   = softmax(s) @ kv_pool[slot_k, 0:512]          (bf16, round-to-nearest-even)
 *     lse   = ln sum_k exp(s_k)                             (fp32)
 *
 * Where the pages define it (page title -- section):
 *   - absorbed query [num_tok, H, 576] and latent pool [num_slots, 576]:
 *     "The Glue That Binds" -- "The Broader Engineering Effort";
 *   - prefix through kv_indices/kv_indptr, tree tokens through out_cache_loc,
 *     visibility through custom_mask/mask_indptr, everything derived on the
 *     device from those buffers, fixed grid, early-out of empty splits:
 *     "The Final Solder Joint" -- "The Three-Edits Sequence", item 1;
 *   - buffer types (int64 kv_indices/qo_indptr/mask_indptr/out_cache_loc,
 *     int32 kv_indptr, uint8 custom_mask): same page -- "The Investigation";
 *   - caller-owned workspace, no host sync, no internal cudaMalloc (graph
 *     capture safety): same page -- "The Capture-Safety Constraint" and
 *     "Why the C-ABI Edit Matters";
 *   - extern "C" entry points returning error codes, called through ctypes:
 *     "The Glue That Makes Kernels Run" -- "The Subject Message".
 *
 * Conventions shared by every entry point:
 *   - every pointer argument named as a device buffer is a CUDA device pointer
 *     on the plan's device; host arguments are plain host memory;
 *   - every buffer is owned by the caller; the library never allocates, frees
 *     or synchronises inside mla_tree_verify_run, so a run may be captured in a
 *     CUDA graph (bind the same buffers; refresh their contents between replays);
 *   - the return value is MTV_OK (0) or a negative MTV_E* code; nothing is
 *     launched when a run returns an error found on the host.
 */
#ifndef MLA_TREE_VERIFY_H_
#define MLA_TREE_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */
#define MTV_OK 0
#define MTV_E_NULL_POINTER -1      /* a required pointer is NULL                   */
#define MTV_E_UNSUPPORTED -2       /* H != 64, d_latent != 512 or d_rope != 64      */
#define MTV_E_BAD_ARGUMENT -3      /* bad size, alignment, mask layout or flags     */
#define MTV_E_WORKSPACE_SMALL -4   /* workspace_bytes < plan->ws_bytes              */
#define MTV_E_WORKSPACE_ALIGN -5   /* workspace not 256-byte aligned                */
#define MTV_E_BAD_PLAN -6          /* plan not produced by mla_tree_verify_plan     */
#define MTV_E_CUDA -7              /* a CUDA runtime call or a launch failed        */
#define MTV_E_DEVICE -8            /* device not usable (not sm_103, bad ordinal)   */

/* --------------------------------------------------------- mask layouts */
/* FULL_ROW: request r's mask is row-major [n_r, p_r + n_r] uint8 at
 * custom_mask + mask_indptr[r]; tree column t is at p_r + t.  The prefix
 * columns are never read: the prefix is always visible.                      */
#define MTV_MASK_FULL_ROW 0
/* TREE_ONLY: request r's mask is row-major [n_r, n_r] at mask_indptr[r].     */
#define MTV_MASK_TREE_ONLY 1

/* ------------------------------------------------------------ plan flags */
/* Use the SIMT fp32 correctness-floor kernel instead of the tcgen05 one.     */
#define MTV_FLAG_SIMT_FLOOR 0x1
/* Test only: every pipeline wait of the kernels gives up as soon as it has to
 * spin, so that the timeout path (MTV_DEVERR_TIMEOUT, orderly wind-down, the
 * call still returns) can be exercised without a fault.  Results of a run with
 * this flag are undefined; never set it in production.                       */
#define MTV_FLAG_TEST_SHORT_WAITS 0x100

/* ------------------------------------------------ device error word bits */
/* The first 4 bytes of the workspace hold a sticky error word that kernels OR
 * into.  Offending keys are treated as masked; nothing traps.                */
#define MTV_DEVERR_SLOT_RANGE 0x1     /* a slot index outside [0, num_slots)          */
#define MTV_DEVERR_INDPTR 0x2         /* decreasing indptr, a request beyond the plan's bounds,
                                         or CSR offsets past the end of kv_indices,
                                         out_cache_loc or custom_mask (see run)  */
#define MTV_DEVERR_TIMEOUT 0x4        /* a bounded pipeline wait gave up              */

#define MTV_PLAN_MAGIC 0x4D545650u    /* 'MTVP' */
#define MTV_ABI_VERSION 2u

/* POD plan.  Produced on the host by mla_tree_verify_plan from upper bounds
 * only (never from device data), then passed unchanged to every run.  The
 * caller owns it; copying it byte-wise is allowed.                            */
typedef struct mtv_plan {
  uint32_t magic, version;
  int32_t device, num_sms, cc_major, cc_minor;
  int32_t bs, max_q_per_req, num_heads, d_latent, d_rope, mask_layout, flags;
  int32_t row_tile;    /* query rows per CTA (pair) row block                  */
  int32_t key_tile;    /* keys per pipeline step                               */
  int32_t nsplit;      /* split-K count (splits past a request's end exit)     */
  int32_t grid_rows;   /* row blocks per request in the grid                   */
  int32_t reserved0;
  int64_t total_q_max; /* capacity of q/out/lse in tokens                       */
  int64_t max_prefix;  /* longest prefix a run may present                      */
  int64_t split_keys;  /* keys per split (multiple of key_tile)                 */
  uint64_t ws_bytes;   /* workspace bytes the run needs                         */
  uint64_t ws_part_o;  /* byte offset of the fp32 partial outputs               */
  uint64_t ws_part_lse;/* byte offset of the fp32 partial LSEs                  */
  int64_t reserved[6];
} mtv_plan_t;

/*
 * mla_tree_verify_plan -- choose tiles, split count and workspace size.
 *
 * device         CUDA ordinal; must be an sm_103 device.
 * bs             number of requests a run will present (>= 0).
 * max_q_per_req  largest tree size n_r a run may present.
 * total_q_max    capacity of q/out/lse in tokens (>= sum of n_r).
 * max_prefix     largest prefix p_r a run may present.
 * num_heads / d_latent / d_rope   must be 64 / 512 / 64.
 * mask_layout    MTV_MASK_FULL_ROW or MTV_MASK_TREE_ONLY.
 * flags          0, MTV_FLAG_SIMT_FLOOR and/or MTV_FLAG_TEST_SHORT_WAITS.
 * nsplit_override 0 = automatic, else the split count to use (tuning).
 * plan_out       host memory, filled on success.
 * ws_bytes_out   host memory (may be NULL), receives plan_out->ws_bytes.
 *
 * Reads device attributes (SM count, compute capability): call it outside
 * stream capture.  Returns MTV_OK or a negative code.
 */
int mla_tree_verify_plan(int device, int bs, int max_q_per_req, int64_t total_q_max,
                         int64_t max_prefix, int num_heads, int d_latent, int d_rope,
                         int mask_layout, int flags, int nsplit_override,
                         mtv_plan_t* plan_out, uint64_t* ws_bytes_out);

/*
 * mla_tree_verify_choose_nsplit -- a split count for a batch whose request
 * lengths are known on the host, to pass as nsplit_override to
 * mla_tree_verify_plan (with max_prefix / max_q_per_req = the batch's
 * largest p_r / n_r).  The automatic choice of mla_tree_verify_plan sees only
 * upper bounds and treats every request as the largest; for a ragged batch
 * this function instead estimates the partial kernel's work units (one per
 * 128-row block and split, handed to the SM pairs in grid order; empty ones
 * cost almost nothing) plus the combine's partial traffic, for every
 * distinct split length, and returns the smallest count within 2 % of the
 * best estimate ("The Final Solder Joint" -- "The Three-Edits Sequence": a
 * fixed split grid whose empty splits exit early).  A batch of identical
 * requests, or one of more than 65,536 row blocks in all, gets the plan's
 * own choice.  Host only; reads no device.
 *
 * num_sms        SM count of the device (>= 2).
 * bs             requests (>= 0).
 * prefix_lens    host int64 [bs], p_r >= 0 (may be NULL when bs == 0).
 * tree_sizes     host int32 [bs], n_r >= 0 (may be NULL when bs == 0).
 * flags          as for mla_tree_verify_plan (MTV_FLAG_SIMT_FLOOR selects the
 *                SIMT kernel's rule).
 * nsplit_out     host, receives a count in [1, 64].
 *
 * Returns MTV_OK, MTV_E_NULL_POINTER or MTV_E_BAD_ARGUMENT (num_sms < 2,
 * a negative size, an unknown flag).
 */
int mla_tree_verify_choose_nsplit(int num_sms, int bs, const int64_t* prefix_lens, const int32_t* tree_sizes,
                                  int flags, int* nsplit_out);

/*
 * mla_tree_verify_run -- enqueue one verify-attention pass on `stream`.
 *
 * q              device, bf16 [total_q, 64, 576] row-major (token, head, dim).
 * kv_pool        device, bf16 [num_slots, 576], 16-byte aligned; V is columns
 *                0..511 of each row.
 * num_slots      rows in kv_pool, 0 <= num_slots < 2^31 (the gather keeps a
 *                slot in a 32-bit register; slot indices are checked against
 *                num_slots and an out-of-range slot is treated as masked).
 * kv_indices     device, int64 [kv_indices_len]: prefix slots, request-major.
 * kv_indices_len number of int64 elements readable at kv_indices (>= 0).
 * kv_indptr      device, int32 [bs + 1]: CSR offsets into kv_indices.
 * out_cache_loc  device, int64 [out_cache_loc_len]: slot of every tree token.
 * out_cache_loc_len  number of int64 elements readable at out_cache_loc.
 * qo_indptr      device, int64 [bs + 1]: CSR offsets of tree tokens (rows of q).
 * custom_mask    device, uint8 [custom_mask_len]: per-request visibility
 *                (see MTV_MASK_*).
 * custom_mask_len  number of bytes readable at custom_mask.
 * mask_indptr    device, int64 [bs + 1]: start of request r's mask block.
 * scale          softmax scale applied to q.k (e.g. 192^-0.5).
 * out            device, bf16 [total_q, 64, 512]; rows past qo_indptr[bs] untouched.
 * lse            device, fp32 [total_q, 64]; natural-log LSE of the scaled scores.
 * workspace      device, >= plan->ws_bytes bytes, 256-byte aligned; its first
 *                4 bytes are the sticky device error word (clear it once with
 *                mla_tree_verify_clear_device_error before the first run).
 * stream         a cudaStream_t passed as void* (NULL = legacy default stream).
 *
 * Sizes of each request come from the device buffers ("The Final Solder
 * Joint" -- "The Three-Edits Sequence": everything is derived on the device
 * from the native buffers) and are checked there before any of them is used
 * as an offset: n_r <= max_q_per_req, p_r <= max_prefix, kv_indptr and
 * qo_indptr non-decreasing from >= 0, qo_indptr[r+1] <= min(total_q_max,
 * out_cache_loc_len), kv_indptr[r+1] <= kv_indices_len, and request r's mask
 * block (n_r x (p_r + n_r) bytes for FULL_ROW, n_r x n_r for TREE_ONLY) inside
 * [0, custom_mask_len).  A request failing any check sets MTV_DEVERR_INDPTR and
 * is skipped: none of its offsets is dereferenced and its rows of out/lse are
 * left untouched.
 * A row with no visible key gets out = 0 and lse = -inf.
 * No host sync, no allocation: safe to capture in a CUDA graph.
 */
int mla_tree_verify_run(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                        int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                        const int32_t* kv_indptr, const int64_t* out_cache_loc,
                        int64_t out_cache_loc_len, const int64_t* qo_indptr,
                        const uint8_t* custom_mask, int64_t custom_mask_len,
                        const int64_t* mask_indptr, float scale, void* out, float* lse,
                        void* workspace, uint64_t workspace_bytes, void* stream);

/* Steps of one pass, for mla_tree_verify_run_steps. */
#define MTV_STEP_PARTIAL 0x1   /* the split-K partial kernel (writes out/lse itself with one split) */
#define MTV_STEP_COMBINE 0x2   /* the combine of the splits (nothing to do with one split)         */

/*
 * mla_tree_verify_run_steps -- mla_tree_verify_run split into its launches,
 * so that a caller (a profiler, a benchmark) can enqueue work such as CUDA
 * events between them.  `steps` is MTV_STEP_PARTIAL, MTV_STEP_COMBINE or both
 * (both is exactly mla_tree_verify_run).  MTV_STEP_PARTIAL followed by
 * MTV_STEP_COMBINE on the same stream with the same arguments gives the same
 * result as one mla_tree_verify_run, bit for bit; the combine launched alone
 * is an ordinary stream successor instead of a programmatic dependent of the
 * partial kernel.  Same arguments, checks and errors as mla_tree_verify_run;
 * MTV_E_BAD_ARGUMENT for an empty or unknown step mask.
 */
int mla_tree_verify_run_steps(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                              int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                              const int32_t* kv_indptr, const int64_t* out_cache_loc,
                              int64_t out_cache_loc_len, const int64_t* qo_indptr,
                              const uint8_t* custom_mask, int64_t custom_mask_len,
                              const int64_t* mask_indptr, float scale, void* out, float* lse,
                              void* workspace, uint64_t workspace_bytes, int steps, void* stream);

/* Text for a return code (static storage; never NULL). */
const char* mla_tree_verify_strerror(int code);

/* Enqueue a clear of the device error word at the head of `workspace`
 * (cudaMemsetAsync of 4 bytes on `stream`; capture-safe). */
int mla_tree_verify_clear_device_error(void* workspace, void* stream);

/* Copy the device error word to *flags_out.  Synchronises `stream`: a test and
 * diagnostics helper, not for use inside capture. */
int mla_tree_verify_read_device_error(const void* workspace, uint32_t* flags_out, void* stream);

/*
 * mla_tree_verify_run_static -- the same pass as mla_tree_verify_run, for
 * callers that cannot allocate device memory where they call attention: a
 * step being recorded into a CUDA graph (allocation calls are not allowed
 * while a stream captures), a host framework that owns every device
 * allocation through its own pool, or a latency-critical path that must not
 * touch an allocator.  The caller still owns and passes every input and
 * output; only the workspace is replaced by a fixed device array inside this
 * library.  (No counterpart on the pages: it is a packaging variant.)
 *
 * Limits and behaviour:
 *   - the array holds 64 MiB on every GPU that loads the library, until the
 *     process exits; a plan whose ws_bytes exceeds it is rejected with
 *     MTV_E_WORKSPACE_SMALL (plan with nsplit_override = 1 to need only the
 *     256-byte header);
 *   - the first call on each device looks up the array's device address with
 *     that device current: make that first call before any stream capture;
 *   - every call shares the one array and it keeps the last call's contents;
 *     calls whose kernels overlap on the GPU (other streams, other threads)
 *     race on it, so serialise them;
 *   - the device error word is cleared (an asynchronous 4-byte memset on
 *     `stream`) at the start of each call; read it back with
 *     mla_tree_verify_read_static_device_error;
 *   - no cudaMalloc, cudaFree or other allocating call is made.
 * Arguments are those of mla_tree_verify_run without the workspace.
 */
int mla_tree_verify_run_static(const mtv_plan_t* plan, const void* q, const void* kv_pool,
                               int64_t num_slots, const int64_t* kv_indices, int64_t kv_indices_len,
                               const int32_t* kv_indptr, const int64_t* out_cache_loc,
                               int64_t out_cache_loc_len, const int64_t* qo_indptr,
                               const uint8_t* custom_mask, int64_t custom_mask_len,
                               const int64_t* mask_indptr, float scale, void* out, float* lse,
                               void* stream);

/* Copy the device error word of the fixed scratch used by
 * mla_tree_verify_run_static on the current device (the bits the kernels of
 * the static calls since the last one's clear have set; 0 before any static
 * call) to *flags_out.  Synchronises `stream`; allocates nothing.  Like the
 * first static call, its first call on a device looks up the scratch address:
 * make it outside stream capture. */
int mla_tree_verify_read_static_device_error(uint32_t* flags_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TREE_VERIFY_H_ */
