"""Seeded synthetic workloads for MLA tree-verify attention.

This module only *draws inputs*: draft trees, slot maps, the packed visibility
mask and bf16 tensors.  It holds none of the attention arithmetic, so both the
CUDA path and the CPU oracle can consume the same inputs without sharing any
code of the method.

Input recipe (the pages fix the tensor layouts, not the values):

* absorbed query ``q``: ``[total_q, H=64, 576]`` bf16 (512 latent + 64 rope dims),
  "The Broader Engineering Effort" section of *The Glue That Binds*;
* paged latent pool ``kv_pool``: ``[num_slots, 576]`` bf16, one row per token;
* ``kv_indices`` int64 / ``kv_indptr`` int32 (prefix slots per request, CSR),
  ``out_cache_loc`` int64 (slots of the tree tokens), ``qo_indptr`` int64,
  ``custom_mask`` uint8 and ``mask_indptr`` int64 -- the buffer types listed in
  "The Investigation" section of *The Final Solder Joint*.

Values are drawn ~N(0,1) in fp32 and rounded to bf16 (round-to-nearest-even).
Trees: node 0 hangs off the prefix root; node i>=1 picks its parent uniformly
from {root, 0..i-1}.  Visibility is ancestors + self.  Slots come from a random
permutation of the pool, carved into consecutive runs (prefix first, then the
tree tokens) -- or the identity map for the contiguous variant.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NUM_HEADS = 64
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
SCALE = 192.0 ** -0.5  # qk_nope 128 + rope 64 head dim of the target model

MASK_FULL_ROW = 0  # per request [n, p+n]; prefix columns are ignored
MASK_TREE_ONLY = 1  # per request [n, n]

ROOT = -1


@dataclass
class Workload:
    name: str
    bs: int
    prefix_lens: list
    tree_sizes: list
    parents: list  # per request: list[int] with ROOT for nodes hanging off the prefix
    q: torch.Tensor  # [total_q, H, 576] bf16
    kv_pool: torch.Tensor  # [num_slots, 576] bf16
    kv_indices: torch.Tensor  # int64 [sum p]
    kv_indptr: torch.Tensor  # int32 [bs+1]
    out_cache_loc: torch.Tensor  # int64 [total_q]
    qo_indptr: torch.Tensor  # int64 [bs+1]
    custom_mask: torch.Tensor  # uint8
    mask_indptr: torch.Tensor  # int64 [bs+1]
    mask_layout: int = MASK_FULL_ROW
    scale: float = SCALE
    num_heads: int = NUM_HEADS
    meta: dict = field(default_factory=dict)

    @property
    def total_q(self) -> int:
        return int(sum(self.tree_sizes))

    @property
    def num_slots(self) -> int:
        return int(self.kv_pool.shape[0])

    @property
    def max_prefix(self) -> int:
        return int(max(self.prefix_lens)) if self.prefix_lens else 0

    @property
    def max_q_per_req(self) -> int:
        return int(max(self.tree_sizes)) if self.tree_sizes else 0

    def algorithmic_flops(self) -> float:
        """2 * rows * keys * (576 + 512) summed over requests (dense keys)."""
        return float(sum(2.0 * self.num_heads * n * (p + n) * (D_QK + D_LATENT)
                         for p, n in zip(self.prefix_lens, self.tree_sizes)))

    def algorithmic_bytes(self) -> float:
        """Each latent row read once, q/out/lse once, 8 B per index, n^2 mask bytes."""
        b = 0.0
        for p, n in zip(self.prefix_lens, self.tree_sizes):
            b += (p + n) * D_QK * 2          # latent rows (K and V share them)
            b += n * self.num_heads * D_QK * 2   # q
            b += n * self.num_heads * D_LATENT * 2  # out (bf16)
            b += n * self.num_heads * 4       # lse
            b += (p + n) * 8                  # kv_indices + out_cache_loc
            b += n * n                        # tree part of the mask
        return b


# ----------------------------------------------------------------------------
# tree / mask drawing
# ----------------------------------------------------------------------------

def random_parents(n: int, g: torch.Generator) -> list:
    """parent(0)=root; parent(i) uniform over {root, 0..i-1}."""
    par = [ROOT]
    for i in range(1, n):
        par.append(int(torch.randint(0, i + 1, (1,), generator=g).item()) - 1)
    return par[:n]


def chain_parents(n: int) -> list:
    return [ROOT] + list(range(0, n - 1)) if n > 0 else []


def star_parents(n: int) -> list:
    return [ROOT] + [0] * (n - 1) if n > 0 else []


def ancestors_and_self(parents: list) -> torch.Tensor:
    """Boolean [n, n] visibility among tree tokens: column t visible from row i
    iff t is i or an ancestor of i.  Input construction only."""
    n = len(parents)
    vis = torch.zeros((n, n), dtype=torch.uint8)
    for i in range(n):
        j = i
        while j != ROOT:
            vis[i, j] = 1
            j = parents[j]
    return vis


def pack_mask(prefix_lens, tree_vis, layout=MASK_FULL_ROW, prefix_fill=1):
    """Concatenate per-request masks.  FULL_ROW: row i of request r is
    ``[prefix_fill]*p_r + tree_vis[r][i]``.  TREE_ONLY: ``tree_vis[r][i]``."""
    chunks, indptr = [], [0]
    for p, vis in zip(prefix_lens, tree_vis):
        n = vis.shape[0]
        if layout == MASK_FULL_ROW:
            m = torch.empty((n, p + n), dtype=torch.uint8)
            m[:, :p] = prefix_fill
            m[:, p:] = vis
        else:
            m = vis.clone()
        chunks.append(m.reshape(-1))
        indptr.append(indptr[-1] + m.numel())
    mask = torch.cat(chunks) if chunks else torch.zeros(0, dtype=torch.uint8)
    return mask, torch.tensor(indptr, dtype=torch.int64)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------

def randn_bf16(shape, g: torch.Generator, chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0,1) fp32 rounded to bf16, drawn in fixed row chunks (bounded memory)."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        flat[s:e] = torch.randn((e - s, flat.shape[1]), generator=g).to(torch.bfloat16)
    return out


def build_workload(name, prefix_lens, parents, num_slots, g, *, contiguous=False,
                   mask_layout=MASK_FULL_ROW, pool=None, perm=None,
                   num_heads=NUM_HEADS, scale=SCALE) -> Workload:
    bs = len(prefix_lens)
    tree_sizes = [len(p) for p in parents]
    need = sum(prefix_lens) + sum(tree_sizes)
    if need > num_slots:
        raise ValueError(f"pool of {num_slots} slots cannot hold {need} tokens")
    if pool is None:
        pool = randn_bf16((num_slots, D_QK), g)
    if perm is None:
        perm = torch.arange(num_slots, dtype=torch.int64) if contiguous else \
            torch.randperm(num_slots, generator=g, dtype=torch.int64)
    kv_idx, ocl, off = [], [], 0
    for p, n in zip(prefix_lens, tree_sizes):
        kv_idx.append(perm[off:off + p]); off += p
        ocl.append(perm[off:off + n]); off += n
    kv_indices = torch.cat(kv_idx) if kv_idx else torch.zeros(0, dtype=torch.int64)
    out_cache_loc = torch.cat(ocl) if ocl else torch.zeros(0, dtype=torch.int64)
    kv_indptr = torch.tensor([0] + list(_cumsum(prefix_lens)), dtype=torch.int32)
    qo_indptr = torch.tensor([0] + list(_cumsum(tree_sizes)), dtype=torch.int64)
    vis = [ancestors_and_self(par) for par in parents]
    custom_mask, mask_indptr = pack_mask(prefix_lens, vis, mask_layout)
    q = randn_bf16((sum(tree_sizes), num_heads, D_QK), g)
    return Workload(name=name, bs=bs, prefix_lens=list(prefix_lens), tree_sizes=tree_sizes,
                    parents=[list(p) for p in parents], q=q, kv_pool=pool,
                    kv_indices=kv_indices.contiguous(), kv_indptr=kv_indptr,
                    out_cache_loc=out_cache_loc.contiguous(), qo_indptr=qo_indptr,
                    custom_mask=custom_mask, mask_indptr=mask_indptr,
                    mask_layout=mask_layout, scale=scale, num_heads=num_heads)


def _cumsum(xs):
    s = 0
    for x in xs:
        s += int(x)
        yield s


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

def tiny(seed: int = 1001, mask_layout=MASK_FULL_ROW) -> Workload:
    """1 request, prefix 256 on permuted slots of a 4096-slot pool, 8-node tree."""
    g = torch.Generator().manual_seed(seed)
    pool = randn_bf16((4096, D_QK), g)
    parents = [random_parents(8, g)]
    return build_workload("tiny_bs1_p256_n8", [256], parents, 4096, g, pool=pool,
                          mask_layout=mask_layout)


def batch4_short(seed: int = 1002) -> Workload:
    """4 requests x (5,760-token prefix, 16-node tree), 65,536-slot pool, random slots."""
    g = torch.Generator().manual_seed(seed)
    pool = randn_bf16((65536, D_QK), g)
    parents = [random_parents(16, g) for _ in range(4)]
    return build_workload("batch4_p5760_n16", [5760] * 4, parents, 65536, g, pool=pool)


def long_context(contiguous: bool, seed: int = 1003) -> Workload:
    """1 request, 32,768-token prefix, 32-node tree, 65,536-slot pool.  The two
    variants hold the same logical tokens; only the slot map differs."""
    g = torch.Generator().manual_seed(seed)
    logical = randn_bf16((65536, D_QK), g)
    parents = [random_parents(32, g)]
    perm = torch.randperm(65536, generator=g, dtype=torch.int64)
    q = randn_bf16((32, NUM_HEADS, D_QK), g)
    if contiguous:
        pool, slot_of = logical, torch.arange(65536, dtype=torch.int64)
    else:
        pool = torch.empty_like(logical)
        pool[perm] = logical
        slot_of = perm
    wl = build_workload("long_p32768_n32_" + ("contig" if contiguous else "random"),
                        [32768], parents, 65536, g, pool=pool, perm=slot_of)
    wl.q = q
    return wl


def mixed(seed: int = 1004) -> Workload:
    """8 requests, prefix log-uniform in [1k, 64k], 8..64-node trees of random
    shape (chain, star, random parents), 600,000-slot pool, random slots."""
    g = torch.Generator().manual_seed(seed)
    pool = randn_bf16((600_000, D_QK), g)
    prefix_lens, parents, shapes = [], [], []
    for _ in range(8):
        u = float(torch.rand((), generator=g))
        prefix_lens.append(int(round(math.exp(math.log(1024) + u * (math.log(65536) - math.log(1024))))))
        n = int(torch.randint(8, 65, (1,), generator=g).item())
        shape = ["chain", "star", "random"][int(torch.randint(0, 3, (1,), generator=g).item())]
        shapes.append(shape)
        parents.append(chain_parents(n) if shape == "chain" else
                       star_parents(n) if shape == "star" else random_parents(n, g))
    wl = build_workload("mixed_bs8", prefix_lens, parents, 600_000, g, pool=pool)
    wl.meta["shapes"] = shapes
    return wl


STRESS_SLOTS = 2_200_000


def stress_pool(seed: int = 1005) -> torch.Tensor:
    return randn_bf16((STRESS_SLOTS, D_QK), torch.Generator().manual_seed(seed))


def stress(replay: int = 0, pool: torch.Tensor | None = None, seed: int = 1005,
           bs: int = 16, prefix: int = 131072, tree: int = 64) -> Workload:
    """16 requests x (131,072-token prefix, 64-node tree) on a 2.2M-slot pool.
    Replay k redraws indices, masks, q and out_cache_loc from seed 5000+k; the
    pool itself is drawn once from ``seed``."""
    if pool is None:
        pool = stress_pool(seed)
    g = torch.Generator().manual_seed(5000 + replay)
    parents = [random_parents(tree, g) for _ in range(bs)]
    return build_workload(f"stress_bs{bs}_p{prefix}_n{tree}", [prefix] * bs, parents,
                          pool.shape[0], g, pool=pool)


def shared_prefix(bs: int = 16, prefix: int = 32768, tree: int = 1, num_slots: int = 65536,
                  seed: int = 1006) -> Workload:
    """bs requests whose prefixes are the same slots (one shared context), each
    with its own tree of ``tree`` nodes (random parents), random slot map."""
    g = torch.Generator().manual_seed(seed)
    pool = randn_bf16((num_slots, D_QK), g)
    perm = torch.randperm(num_slots, generator=g, dtype=torch.int64)
    parents = [random_parents(tree, g) for _ in range(bs)]
    shared = perm[:prefix]
    ocl = perm[prefix:prefix + bs * tree]
    kv_indices = shared.repeat(bs)
    kv_indptr = torch.tensor([0] + list(_cumsum([prefix] * bs)), dtype=torch.int32)
    qo_indptr = torch.tensor([0] + list(_cumsum([tree] * bs)), dtype=torch.int64)
    vis = [ancestors_and_self(par) for par in parents]
    custom_mask, mask_indptr = pack_mask([prefix] * bs, vis, MASK_FULL_ROW)
    q = randn_bf16((bs * tree, NUM_HEADS, D_QK), g)
    return Workload(name=f"shared_bs{bs}_p{prefix}_n{tree}", bs=bs, prefix_lens=[prefix] * bs,
                    tree_sizes=[tree] * bs, parents=parents, q=q, kv_pool=pool,
                    kv_indices=kv_indices.contiguous(), kv_indptr=kv_indptr, out_cache_loc=ocl.contiguous(),
                    qo_indptr=qo_indptr, custom_mask=custom_mask, mask_indptr=mask_indptr,
                    meta={"shared_prefix": True})


# ----------------------------------------------------------------------------
# large-logit variants (input transforms; the values stay exact bf16)
# ----------------------------------------------------------------------------

def scaled_q(wl: Workload, alpha: float) -> Workload:
    """q multiplied by ``alpha`` and rounded to bf16 again: scaled logits grow
    by alpha (alpha ~4.5 puts the largest logits of the N(0,1) workloads near
    30, where attention in trained models routinely sits)."""
    wl.q = (wl.q.float() * alpha).to(torch.bfloat16)
    wl.name += f"_qx{alpha:g}"
    wl.meta["q_scale"] = alpha
    return wl


def common_component(wl: Workload, a: float = 1.7, b: float = 2.0, seed: int = 7) -> Workload:
    """Every latent row of the pool gets ``a * u`` and every query ``b * u``
    added in the 512 latent dims, u a seeded +-1 vector: all scores share an
    offset of a*b*512 raw units (a*b*256 ~ 870 in each half of the latent
    dims) on top of their N(0,1)-driven spread -- keys that share a large
    common direction, as the latent rows of trained models do."""
    g = torch.Generator().manual_seed(seed)
    u = torch.where(torch.rand(D_LATENT, generator=g) < 0.5, -1.0, 1.0)
    pool = wl.kv_pool.float()
    pool[:, :D_LATENT] += a * u
    wl.kv_pool = pool.to(torch.bfloat16)
    q = wl.q.float()
    q[:, :, :D_LATENT] += b * u
    wl.q = q.to(torch.bfloat16)
    wl.name += "_common"
    wl.meta["common_component"] = (a, b)
    return wl


def sub_workload(wl: Workload, reqs) -> Workload:
    """The requests ``reqs`` of ``wl`` as a batch of their own (same pool; CSR
    offsets re-based, q / out_cache_loc / mask blocks gathered in order)."""
    kvp, qop, mip = wl.kv_indptr.tolist(), wl.qo_indptr.tolist(), wl.mask_indptr.tolist()
    kv_idx, ocl, qs, masks = [], [], [], []
    for r in reqs:
        kv_idx.append(wl.kv_indices[kvp[r]:kvp[r + 1]])
        ocl.append(wl.out_cache_loc[qop[r]:qop[r + 1]])
        qs.append(wl.q[qop[r]:qop[r + 1]])
        masks.append(wl.custom_mask[mip[r]:mip[r + 1]])
    prefix = [wl.prefix_lens[r] for r in reqs]
    sizes = [wl.tree_sizes[r] for r in reqs]
    cat = lambda xs, dt: torch.cat(xs) if xs else torch.empty(0, dtype=dt)
    q = torch.cat(qs) if qs else torch.empty((0, NUM_HEADS, D_QK), dtype=torch.bfloat16)
    return Workload(name=f"{wl.name}_part{len(reqs)}", bs=len(reqs), prefix_lens=prefix, tree_sizes=sizes,
                    parents=[wl.parents[r] for r in reqs], q=q, kv_pool=wl.kv_pool,
                    kv_indices=cat(kv_idx, torch.int64), kv_indptr=torch.tensor([0] + list(_cumsum(prefix)), dtype=torch.int32),
                    out_cache_loc=cat(ocl, torch.int64),
                    qo_indptr=torch.tensor([0] + list(_cumsum(sizes)), dtype=torch.int64),
                    custom_mask=cat(masks, torch.uint8),
                    mask_indptr=torch.tensor([0] + list(_cumsum([m.numel() for m in masks])), dtype=torch.int64),
                    mask_layout=wl.mask_layout, scale=wl.scale, meta=dict(wl.meta, parent=wl.name, reqs=list(reqs)))


def custom(prefix_lens, parents, num_slots, seed, contiguous=False,
           mask_layout=MASK_FULL_ROW, name="custom") -> Workload:
    """Any shape: used by the tests for ragged and degenerate cases."""
    g = torch.Generator().manual_seed(seed)
    return build_workload(name, list(prefix_lens), [list(p) for p in parents], num_slots, g,
                          contiguous=contiguous, mask_layout=mask_layout)


WORKLOADS = {
    "tiny": lambda: tiny(),
    "batch4": lambda: batch4_short(),
    "long_contig": lambda: long_context(True),
    "long_random": lambda: long_context(False),
    "mixed": lambda: mixed(),
    "mixed_s2": lambda: mixed(seed=2004),
    "mixed_s3": lambda: mixed(seed=3004),
    "stress": lambda: stress(0),
    # the stress request shape at 1/8 of the batch on a 300,000-slot pool: a
    # case small enough (~0.4 GB on the device) for full profiler captures of
    # the same kernel; per-request traffic scales to the full batch
    "stress_bs2": lambda: stress(0, pool=randn_bf16((300_000, D_QK), torch.Generator().manual_seed(1015)), bs=2),
    # not one of the five configurations: requests that share one prefix
    "shared_decode": lambda: shared_prefix(16, 32768, 1),
    "shared_tree3": lambda: shared_prefix(16, 32768, 3),
}
