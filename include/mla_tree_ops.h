/*
 * mla_tree_ops.h -- C ABI of the steps around MLA tree-verify attention on
 * GB300 (sm_103a): building the visibility mask from the draft tree,
 * accepting the verified tree, defragmenting a request's paged KV, and
 * merging requests that share a prefix.
 *
 * Where the pages define them (page title -- section):
 *   - the mask is rebuilt from the tree structure rather than reverse-
 *     engineered from a packed format: "The Glue That Binds" -- "The
 *     Thinking Process";
 *   - tree building and tree acceptance are entry points of the same C-ABI
 *     library as verify attention: "The Glue That Connects" -- "What the
 *     Edit Actually Does".
 *
 * Conventions (as in mla_tree_verify.h): every pointer named "device" is a
 * CUDA device pointer; buffers are caller-owned; nothing allocates or
 * synchronises, so every call may be captured in a CUDA graph; the return
 * value is MTV_OK (0) or a negative MTV_E* code (nothing is launched then).
 * `err` (device, may be NULL) is a sticky 32-bit word the kernels OR
 * MTV_DEVERR_* bits into; data-dependent problems never trap.
 */
#ifndef MLA_TREE_OPS_H_
#define MLA_TREE_OPS_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_tree_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* A parent index outside [-1, i-1] for node i (the node is then treated as
 * hanging off the prefix root). */
#define MTV_DEVERR_PARENT 0x8

/*
 * mla_tree_mask_build -- custom_mask + mask_indptr from per-request parent
 * arrays, in the layout mla_tree_verify_run reads.
 *
 * parents        device, int32 [qo_indptr[bs]]: parents[qo_indptr[r] + i] is
 *                the tree index of node i's parent, or -1 when node i hangs
 *                off the prefix (its last token).
 * qo_indptr      device, int64 [bs + 1]: CSR offsets of the tree nodes.
 * kv_indptr      device, int32 [bs + 1]: prefix lengths p_r (FULL_ROW only;
 *                may be NULL for TREE_ONLY).
 * bs, max_q_per_req  host: request count and the largest tree size n_r.
 * mask_layout    MTV_MASK_FULL_ROW: request r is row-major [n_r, p_r + n_r]
 *                with the p_r prefix columns set to 1; MTV_MASK_TREE_ONLY:
 *                [n_r, n_r].  Row i, tree column t is 1 iff t == i or t is an
 *                ancestor of i.
 * custom_mask    device, uint8 output of mask_capacity bytes.
 * mask_indptr    device, int64 [bs + 1] output: start of each request's block.
 * err            device uint32 or NULL: MTV_DEVERR_PARENT for a bad parent,
 *                MTV_DEVERR_INDPTR for a decreasing indptr, a tree larger than
 *                max_q_per_req or a mask that does not fit mask_capacity (the
 *                request's rows are then not written).
 */
int mla_tree_mask_build(const int32_t* parents, const int64_t* qo_indptr, const int32_t* kv_indptr, int bs,
                        int max_q_per_req, int mask_layout, uint8_t* custom_mask, uint64_t mask_capacity,
                        int64_t* mask_indptr, uint32_t* err, void* stream);

/*
 * mla_tree_accept -- greedy acceptance of each request's verified tree.
 *
 * Starting at the prefix root, move to the child whose draft token equals the
 * target model's token predicted at the current node (the lowest-index child
 * when several match), until no child matches.
 *
 * parents            device, int32 [qo_indptr[bs]] (as above).
 * draft_tokens       device, int32 [qo_indptr[bs]]: the token drafted at node i.
 * target_tokens      device, int32 [qo_indptr[bs]]: the target model's token
 *                    predicted after node i (e.g. the argmax of its logits).
 * target_root_tokens device, int32 [bs]: the target's token predicted after
 *                    the prefix.
 * out_cache_loc      device, int64 [qo_indptr[bs]]: KV slot of every node.
 * qo_indptr          device, int64 [bs + 1].
 * accept_len         device, int32 [bs] output: accepted node count.
 * accept_nodes       device, int32 [bs, max_q_per_req] output: accepted tree
 *                    indices in path order, -1 after the last.
 * accept_slots       device, int64 [bs, max_q_per_req] output: their KV slots
 *                    (the compaction list), -1 after the last.
 * bonus_tokens       device, int32 [bs] output: the target's prediction after
 *                    the last accepted node (after the prefix if none).
 * err                device uint32 or NULL: MTV_DEVERR_PARENT /
 *                    MTV_DEVERR_INDPTR as above (an oversized tree accepts
 *                    nothing).
 */
int mla_tree_accept(const int32_t* parents, const int32_t* draft_tokens, const int32_t* target_tokens,
                    const int32_t* target_root_tokens, const int64_t* out_cache_loc, const int64_t* qo_indptr,
                    int bs, int max_q_per_req, int32_t* accept_len, int32_t* accept_nodes,
                    int64_t* accept_slots, int32_t* bonus_tokens, uint32_t* err, void* stream);

/*
 * mla_kv_defrag -- copy each request's prefix rows into one contiguous run of
 * slots and rewrite its prefix indices to that run (the pages' plan to
 * defragment the paged KV for contiguous reads: "The Glue That Connects" --
 * "The Context" and "The Final Solder Joint" -- "The Mandate: Three
 * Priorities").
 *
 * For request r and prefix key j < p_r (p_r = kv_indptr[r+1] - kv_indptr[r]):
 *   kv_dst[dst_base[r] + j, :] = kv_src[kv_indices[kv_indptr[r] + j], :]
 *   kv_indices_out[kv_indptr[r] + j] = dst_base[r] + j
 *
 * kv_src, kv_dst  device, bf16 [num_slots, 576] each, 16-byte aligned; they
 *                 may be the same pool only if no destination slot of this
 *                 call is also a source slot of it (not checked).
 * num_slots       rows in both pools (slots are checked against it).
 * kv_indices      device, int64 [kv_indptr[bs]]; kv_indptr device, int32 [bs+1].
 * dst_base        device, int64 [bs]: first destination slot of each request.
 * kv_indices_out  device, int64 [kv_indptr[bs]] (may alias kv_indices).
 * max_prefix      host: largest p_r (sizes the grid); longer prefixes are
 *                 flagged MTV_DEVERR_INDPTR and not copied.
 * err             device uint32 or NULL: MTV_DEVERR_SLOT_RANGE for a source
 *                 or destination slot outside [0, num_slots) (that row is not
 *                 copied and its kv_indices_out entry is not written).
 */
int mla_kv_defrag(const void* kv_src, void* kv_dst, int64_t num_slots, const int64_t* kv_indices,
                  const int32_t* kv_indptr, int bs, int64_t max_prefix, const int64_t* dst_base,
                  int64_t* kv_indices_out, uint32_t* err, void* stream);

/* A follower request whose prefix differs from its group leader's (its own
 * prefix is then ignored: the group attends to the leader's). */
#define MTV_DEVERR_PREFIX 0x10

/*
 * mla_tree_group_prefix -- merge runs of consecutive requests that share one
 * prefix into single requests, so that verify attention gathers the shared
 * prefix once per row block and packs their tree rows into full row blocks.
 * (Not on the pages: the plainest extension of their per-request layout.)
 *
 * Group g holds requests [group_indptr[g], group_indptr[g+1]).  Its merged
 * request has the first request's prefix, and as its tree the group's trees
 * side by side: node i of request r becomes node i + (qo_indptr[r] -
 * qo_indptr[first]) with its parent shifted the same way (-1 stays -1), so no
 * tree token sees another request's tokens.  Token order is unchanged: q, out,
 * lse and out_cache_loc are used as they are.  Build the merged mask with
 * mla_tree_mask_build(parents_out, qo_indptr_out, kv_indptr_out, ...).
 *
 * group_indptr     device, int32 [num_groups + 1], non-decreasing from 0.
 * num_groups       host.
 * max_group_prefix host: largest leader prefix (sizes the grid); a longer one
 *                  is flagged MTV_DEVERR_INDPTR and copied as empty.
 * kv_indices, kv_indptr, qo_indptr, parents   device, the per-request inputs.
 * kv_indptr_out    device, int32 [num_groups + 1].
 * kv_indices_out   device, int64 [sum of the leaders' prefix lengths].
 * qo_indptr_out    device, int64 [num_groups + 1] (qo_indptr at group starts).
 * parents_out      device, int32 [qo_indptr[last request + 1]].
 * err              device uint32 or NULL: MTV_DEVERR_PREFIX for a follower
 *                  whose prefix is not the leader's (length or slots).
 */
int mla_tree_group_prefix(const int32_t* group_indptr, int num_groups, int64_t max_group_prefix,
                          const int64_t* kv_indices, const int32_t* kv_indptr, const int64_t* qo_indptr,
                          const int32_t* parents, int32_t* kv_indptr_out, int64_t* kv_indices_out,
                          int64_t* qo_indptr_out, int32_t* parents_out, uint32_t* err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TREE_OPS_H_ */
