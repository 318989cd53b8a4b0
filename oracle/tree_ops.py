"""CPU oracle for the two tree steps around verify attention -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module.  Plain Python loops over small trees; it shares no code
with the CUDA library.

* ``tree_mask``: the draft tree's visibility mask rebuilt from its parent
  array ("The Glue That Binds" -- "The Thinking Process": the mask is rebuilt
  from the tree structure instead of reverse-engineering a packed format;
  "The Glue That Connects" -- "What the Edit Actually Does": tree building is
  one of the library's entry points).  Tree token i sees token t iff t is i or
  an ancestor of i; in the full-row layout every prefix column is set.
* ``tree_accept``: greedy acceptance of the verified tree ("The Glue That
  Connects" -- "What the Edit Actually Does": tree acceptance is one of the
  library's entry points).  Starting at the prefix root, the walk moves to the
  child whose draft token equals the target model's token predicted at the
  current node (the lowest-index child when several match) until no child
  matches; the target's prediction at the last accepted node is the bonus
  token, and the accepted nodes' KV slots, in path order, are the compaction
  list.
* ``kv_defrag``: each request's prefix rows copied into one contiguous run of
  slots and its prefix indices rewritten to that run ("The Final Solder Joint"
  -- "The Mandate: Three Priorities": defragmentation is the next priority
  after graph capture; "The Glue That Connects" -- "The Context": the plan
  that introduces it).  A numpy gather (library primitive) does the copy.
* ``group_prefix``: runs of requests that share one prefix merged into single
  requests whose tree is the group's trees side by side (not on the pages:
  the plainest extension of their per-request layout).
"""
from __future__ import annotations

import numpy as np

ROOT = -1
MASK_FULL_ROW = 0
MASK_TREE_ONLY = 1


def ancestors_or_self(parents, i):
    """Tree indices on the path from node i up to (not including) the root."""
    out = []
    j = i
    while j != ROOT:
        out.append(j)
        j = parents[j]
    return out


def tree_mask(parents_per_req, prefix_lens, layout=MASK_FULL_ROW):
    """Packed uint8 mask and int64 mask_indptr for all requests.

    FULL_ROW: request r is row-major [n_r, p_r + n_r]; columns [0, p_r) are 1,
    column p_r + t is 1 iff t is i or an ancestor of i.
    TREE_ONLY: request r is row-major [n_r, n_r] with the tree columns only.
    """
    chunks, indptr = [], [0]
    for par, p in zip(parents_per_req, prefix_lens):
        n = len(par)
        width = (p + n) if layout == MASK_FULL_ROW else n
        off = p if layout == MASK_FULL_ROW else 0
        m = np.zeros((n, width), dtype=np.uint8)
        if layout == MASK_FULL_ROW:
            m[:, :p] = 1
        for i in range(n):
            for t in ancestors_or_self(par, i):
                m[i, off + t] = 1
        chunks.append(m.reshape(-1))
        indptr.append(indptr[-1] + m.size)
    mask = np.concatenate(chunks) if chunks else np.zeros(0, dtype=np.uint8)
    return mask, np.array(indptr, dtype=np.int64)


def tree_accept(parents, draft_tokens, target_tokens, target_root_token, slots):
    """Greedy walk of one request's verified tree.

    parents[i]: parent tree index of node i (ROOT for nodes under the prefix);
    draft_tokens[i]: the drafted token at node i; target_tokens[i]: the target
    model's token predicted after node i; target_root_token: its prediction
    after the prefix; slots[i]: KV slot of node i.
    Returns (accepted node indices in path order, bonus token, their slots).
    """
    n = len(parents)
    cur, want = ROOT, int(target_root_token)
    path = []
    while True:
        nxt = None
        for c in range(n):  # lowest-index child of `cur` that carries the predicted token
            if parents[c] == cur and int(draft_tokens[c]) == want:
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        cur, want = nxt, int(target_tokens[nxt])
    return path, want, [int(slots[c]) for c in path]


def kv_defrag(src_pool, dst_pool, kv_indices, kv_indptr, dst_base):
    """Returns (new destination pool, new kv_indices): for request r and prefix
    key j, row dst_base[r] + j of the destination takes source row
    kv_indices[kv_indptr[r] + j], and that index becomes dst_base[r] + j."""
    out = np.array(dst_pool, copy=True)
    idx = np.array(kv_indices, dtype=np.int64, copy=True)
    src = np.asarray(src_pool)
    for r in range(len(dst_base)):
        k0, k1 = int(kv_indptr[r]), int(kv_indptr[r + 1])
        run = np.arange(int(dst_base[r]), int(dst_base[r]) + (k1 - k0), dtype=np.int64)
        out[run] = src[idx[k0:k1]]
        idx[k0:k1] = run
    return out, idx


def group_prefix(group_indptr, kv_indices, kv_indptr, qo_indptr, parents_flat):
    """Merged (kv_indptr, kv_indices, qo_indptr, parents, prefix_mismatch) for
    groups [group_indptr[g], group_indptr[g+1]) of consecutive requests: the
    group keeps its first request's prefix; node i of request r becomes node
    i + qo_indptr[r] - qo_indptr[first] with its parent shifted alike."""
    kv_out, idx_out, qo_out = [0], [], [int(qo_indptr[int(group_indptr[0])])]
    par_out = list(int(p) for p in parents_flat)
    mismatch = False
    for g in range(len(group_indptr) - 1):
        a, b = int(group_indptr[g]), int(group_indptr[g + 1])
        if b > a:
            lead = list(kv_indices[int(kv_indptr[a]):int(kv_indptr[a + 1])])
            for r in range(a + 1, b):
                if list(kv_indices[int(kv_indptr[r]):int(kv_indptr[r + 1])]) != lead:
                    mismatch = True
            idx_out += [int(x) for x in lead]
            q0 = int(qo_indptr[a])
            for r in range(a, b):
                for t in range(int(qo_indptr[r]), int(qo_indptr[r + 1])):
                    p = int(parents_flat[t])
                    par_out[t] = -1 if p < 0 else p + int(qo_indptr[r]) - q0
        kv_out.append(len(idx_out))
        qo_out.append(int(qo_indptr[b if b > a else a]))
    return (np.array(kv_out, dtype=np.int32), np.array(idx_out, dtype=np.int64),
            np.array(qo_out, dtype=np.int64), np.array(par_out, dtype=np.int32), mismatch)
