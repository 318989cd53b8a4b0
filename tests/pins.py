"""Independent formulations used to pin the CPU oracle (test helpers only).

None of this is shared with the oracle or with the CUDA path:

* ``dense_reference`` materialises a visibility matrix over *every* pool slot,
  derived from the tree's parent array by a transitive closure (not from the
  packed mask), and runs a dense fp64 softmax with library matmul/logsumexp.
* ``sdpa_chain`` calls torch's scaled_dot_product_attention (fp64, CPU) with an
  explicit boolean mask over the concatenated [prefix; tree] sequence.
"""
from __future__ import annotations

import os

import numpy as np
import torch

D_LAT = 512


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def closure_visibility(parents) -> np.ndarray:
    """[n, n] bool: (i, t) true iff t == i or t is an ancestor of i, by repeated
    squaring of the parent adjacency matrix (a different route from walking)."""
    n = len(parents)
    A = np.zeros((n, n), dtype=np.int64)
    for i, p in enumerate(parents):
        if p >= 0:
            A[i, p] = 1
    R = np.eye(n, dtype=np.int64) + A
    for _ in range(max(1, int(np.ceil(np.log2(max(n, 2)))) + 1)):
        R = ((R @ R) > 0).astype(np.int64)
    return R > 0


def dense_reference(wl, tree_vis=None):
    """Returns (out [total_q*H, 512], lse [total_q*H]) in fp64 by a dense
    softmax over all pool slots with a visibility matrix V[row, slot]."""
    pool = bf16_to_f64(wl.kv_pool)
    q = bf16_to_f64(wl.q).reshape(-1, pool.shape[1])
    H = wl.num_heads
    S = wl.scale * (q @ pool.T)  # [rows, slots]
    V = np.zeros_like(S, dtype=bool)
    kvp = wl.kv_indptr.numpy().astype(np.int64)
    qop = wl.qo_indptr.numpy()
    kvi = wl.kv_indices.numpy()
    ocl = wl.out_cache_loc.numpy()
    for r in range(wl.bs):
        pre = kvi[kvp[r]:kvp[r + 1]]
        tree = ocl[qop[r]:qop[r + 1]]
        vis = closure_visibility(wl.parents[r]) if tree_vis is None else tree_vis[r]
        for i in range(qop[r + 1] - qop[r]):
            rows = slice((qop[r] + i) * H, (qop[r] + i + 1) * H)
            V[rows, pre] = True
            V[rows, tree[vis[i]]] = True
    Sm = np.where(V, S, -np.inf)
    lse = torch.logsumexp(torch.from_numpy(Sm), dim=1).numpy()
    W = np.exp(Sm - np.where(np.isfinite(lse), lse, 0.0)[:, None])
    W[~V] = 0.0
    out = W @ pool[:, :D_LAT]
    out[~np.isfinite(lse)] = 0.0
    return out, lse


def sdpa_chain(wl, r: int):
    """torch SDPA (fp64) for request r whose tree is a chain: visibility over
    [prefix; tree] is causal on the tree part."""
    pool = torch.from_numpy(bf16_to_f64(wl.kv_pool))
    kvp = wl.kv_indptr.long()
    qop = wl.qo_indptr
    pre = wl.kv_indices[kvp[r]:kvp[r + 1]]
    tree = wl.out_cache_loc[qop[r]:qop[r + 1]]
    keys = pool[torch.cat([pre, tree])]  # [p+n, 576]
    p, n = pre.numel(), tree.numel()
    q = torch.from_numpy(bf16_to_f64(wl.q[qop[r]:qop[r + 1]]))  # [n, H, 576]
    mask = torch.zeros((n, p + n), dtype=torch.bool)
    mask[:, :p] = True
    mask[:, p:] = torch.tril(torch.ones((n, n), dtype=torch.bool))
    qh = q.permute(1, 0, 2)  # [H, n, 576]
    k = keys.unsqueeze(0).expand(qh.shape[0], -1, -1)
    v = keys[:, :D_LAT].unsqueeze(0).expand(qh.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qh, k, v, attn_mask=mask, scale=wl.scale)
    return o.permute(1, 0, 2).reshape(-1, D_LAT).numpy()


# ------------------------------------------------------ hand-derived worked example

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_example.json")


def worked_example(mask_layout: int = 0):
    """The worked example of ``tests/golden/worked_example.json`` as a
    Workload, plus its expected (out, lse) from the closed forms derived there
    (rows token-major then head; out dims other than 0 and 1 are zero)."""
    import json
    import math

    from paged_mla_speculative_tree_gb300 import workloads as W
    ex = json.load(open(GOLDEN))
    H, D = 64, 576
    pool = torch.zeros((ex["num_slots"], D), dtype=torch.float32)
    for slot, dims in ex["kv_rows"].items():
        for d, v in dims.items():
            pool[int(slot), int(d)] = float(v)
    q = torch.zeros((2, H, D), dtype=torch.float32)
    q[:, :, 0] = float(ex["q_dim0"])
    q[:, :, 512] = torch.tensor([h % 2 for h in range(H)], dtype=torch.float32)
    rows = ex["mask_full_row"] if mask_layout == W.MASK_FULL_ROW else ex["mask_tree_only"]
    mask = torch.tensor([b for row in rows for b in row], dtype=torch.uint8)
    wl = W.Workload(name="worked_example", bs=1, prefix_lens=[2], tree_sizes=[2], parents=[[W.ROOT, 0]],
                    q=q.to(torch.bfloat16), kv_pool=pool.to(torch.bfloat16),
                    kv_indices=torch.tensor(ex["kv_indices"], dtype=torch.int64),
                    kv_indptr=torch.tensor(ex["kv_indptr"], dtype=torch.int32),
                    out_cache_loc=torch.tensor(ex["out_cache_loc"], dtype=torch.int64),
                    qo_indptr=torch.tensor(ex["qo_indptr"], dtype=torch.int64),
                    custom_mask=mask, mask_indptr=torch.tensor([0, mask.numel()], dtype=torch.int64),
                    mask_layout=mask_layout, scale=ex["scale"])
    e = math.e
    z0, z1 = e + 1 + e ** 2, e + 1 + e ** 2 + 1 / e
    even = [((e / 2 + e ** 2) / z0, (e / 8 + 1 / 4 + 3 * e ** 2 / 8) / z0, math.log(z0)),
            ((e / 2 + e ** 2 - 1 / (2 * e)) / z1, (e / 8 + 1 / 4 + 3 * e ** 2 / 8 + 1 / (2 * e)) / z1, math.log(z1))]
    odd = [(0.5, 0.25, 1 + math.log(3)), (0.25, 0.3125, 1 + math.log(4))]
    out = np.zeros((2 * H, D_LAT))
    lse = np.zeros(2 * H)
    for t in range(2):
        for h in range(H):
            o0, o1, l = (odd if h % 2 else even)[t]
            out[t * H + h, 0], out[t * H + h, 1], lse[t * H + h] = o0, o1, l
    return wl, out, lse
