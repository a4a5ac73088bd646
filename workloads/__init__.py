"""Seeded synthetic inputs for batched tree attention.

This module is the one piece shared by the CPU oracle (``oracle/``) and the
CUDA path (``tree_attention_gb300``): it builds token trees, their DFS
``[enter, exit)`` interval tables, positions and random q/k/v tensors.  It holds
none of the attention arithmetic -- no mask evaluation, no RoPE, no softmax.

Layouts follow the buffer list of ``batch_tree_attn`` on the page
"tree_attn.py" (python/tvm/relax/frontend/nn/llm/tree_attn.py, the prim_func
signature of ``tree_attn``):

* ``q``  ``[total_q, h_q, d]``, ``k``/``v`` ``[total_kv, h_kv, d]`` (fp16/bf16)
* ``q_indptr``/``kv_indptr``/``mn_indptr`` ``[B+1]`` int32 CSR offsets
* ``tree_order`` ``[total_tree, 2]`` int32, row ``mn_indptr[b] + i`` holds node
  ``i``'s ``(enter, exit)`` DFS interval (exit exclusive)
* ``rope_position`` ``[total_kv]`` int32, the position of every kv token

Sequence ``b`` holds ``kv_len = prefix + n`` kv tokens: a causal prefix that
every query sees, then the ``n`` tree nodes in node-index order.  Its q rows
are the last ``qo_len`` tree nodes (every built-in workload uses
``qo_len == n``).  Parent arrays satisfy ``parent[0] == -1`` and
``parent[i] < i``.

Random draws use ``numpy.random.default_rng`` (PCG64), which is stable across
platforms, so x86 and Arm hosts build identical inputs from the same seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

__all__ = [
    "Workload", "chain_tree", "star_tree", "binary_tree", "random_tree",
    "spec_decode_tree", "main_chain_tree", "tree_intervals", "tree_depths",
    "ancestors", "build_workload", "config", "CONFIG_NAMES", "visible_pairs",
    "algorithmic_bytes", "algorithmic_flops", "long_prefix",
]

# --------------------------------------------------------------------------
# tree shapes (parent arrays)
# --------------------------------------------------------------------------

def chain_tree(n: int) -> np.ndarray:
    """Pure chain: node i's parent is i-1 (a chain tree is causal attention)."""
    p = np.arange(-1, n - 1, dtype=np.int64)
    return p


def star_tree(n: int) -> np.ndarray:
    """Star: every non-root node hangs off the root."""
    p = np.zeros(n, dtype=np.int64)
    p[0] = -1
    return p


def binary_tree(n: int) -> np.ndarray:
    """Balanced binary tree in heap numbering: parent(i) = (i-1)//2."""
    p = (np.arange(n, dtype=np.int64) - 1) // 2
    p[0] = -1
    return p


def random_tree(n: int, rng: np.random.Generator) -> np.ndarray:
    """Random recursive tree: parent[i] ~ U[0, i)."""
    p = np.empty(n, dtype=np.int64)
    p[0] = -1
    for i in range(1, n):
        p[i] = rng.integers(0, i)
    return p


def spec_decode_tree(n: int, rng: np.random.Generator, max_depth: int = 8,
                     max_children: int = 4) -> np.ndarray:
    """Speculative-decoding draft tree with depth <= max_depth and at most
    max_children children per node: node i picks its parent uniformly among
    the existing nodes whose depth is < max_depth and which have fewer than
    max_children children (root depth 0)."""
    p = np.empty(n, dtype=np.int64)
    depth = np.zeros(n, dtype=np.int64)
    nchild = np.zeros(n, dtype=np.int64)
    p[0] = -1
    for i in range(1, n):
        ok = np.nonzero((depth[:i] < max_depth) & (nchild[:i] < max_children))[0]
        if ok.size == 0:
            raise ValueError("tree capacity exhausted")
        par = int(ok[rng.integers(0, ok.size)])
        p[i] = par
        depth[i] = depth[par] + 1
        nchild[par] += 1
    return p


def main_chain_tree(n: int, rng: np.random.Generator, p_branch: float = 0.3) -> np.ndarray:
    """A main chain with side branches: node i (i >= 1) attaches to a
    uniformly random earlier node with probability p_branch, otherwise it
    extends the tail of the main chain."""
    p = np.empty(n, dtype=np.int64)
    p[0] = -1
    tail = 0
    for i in range(1, n):
        if rng.random() < p_branch:
            p[i] = rng.integers(0, i)
        else:
            p[i] = tail
            tail = i
    return p


# --------------------------------------------------------------------------
# tree tables
# --------------------------------------------------------------------------

def _children(parent: np.ndarray) -> List[List[int]]:
    ch: List[List[int]] = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        ch[int(parent[i])].append(i)
    return ch


def tree_intervals(parent: np.ndarray) -> np.ndarray:
    """DFS ``[enter, exit)`` intervals, ``[n, 2]`` int32, row i = node i.

    ``enter`` is the DFS preorder index (children visited in increasing node
    index), ``exit = enter + subtree_size``.  Node a is an ancestor-or-self of
    node c iff ``enter[a] <= enter[c] < exit[a]``.
    """
    n = len(parent)
    if n == 0:
        return np.zeros((0, 2), dtype=np.int32)
    ch = _children(parent)
    out = np.zeros((n, 2), dtype=np.int64)
    counter = 0
    # iterative preorder; the stack holds (node, next child position)
    stack = [(0, 0)]
    out[0, 0] = counter
    counter += 1
    while stack:
        node, pos = stack[-1]
        if pos < len(ch[node]):
            stack[-1] = (node, pos + 1)
            c = ch[node][pos]
            out[c, 0] = counter
            counter += 1
            stack.append((c, 0))
        else:
            out[node, 1] = counter
            stack.pop()
    if counter != n:
        raise ValueError("parent array is not a single rooted tree")
    return out.astype(np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[int(parent[i])] + 1
    return d


def ancestors(parent: np.ndarray, i: int) -> List[int]:
    """Ancestor-or-self set of node i by walking parent links."""
    out = []
    while i >= 0:
        out.append(i)
        i = int(parent[i])
    return out


# --------------------------------------------------------------------------
# workload container
# --------------------------------------------------------------------------

_TORCH_DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                       # "fp16" | "bf16"
    h_q: int
    h_kv: int
    head_dim: int
    parents: List[np.ndarray]        # per sequence tree parent arrays
    prefix_lens: List[int]           # per sequence causal prefix length
    qo_lens: List[int]               # per sequence number of q rows
    q: torch.Tensor                  # [total_q, h_q, d]   CPU
    k: torch.Tensor                  # [total_kv, h_kv, d] CPU
    v: torch.Tensor                  # [total_kv, h_kv, d] CPU
    q_indptr: np.ndarray             # [B+1] int32
    kv_indptr: np.ndarray            # [B+1] int32
    mn_indptr: np.ndarray            # [B+1] int32
    tree_order: np.ndarray           # [total_tree, 2] int32
    rope_position: Optional[np.ndarray]  # [total_kv] int32 or None
    rotary_mode: int
    rope_scale: float
    rope_theta: float
    sm_scale: float

    @property
    def batch_size(self) -> int:
        return len(self.parents)

    @property
    def total_q(self) -> int:
        return int(self.q_indptr[-1])

    @property
    def total_kv(self) -> int:
        return int(self.kv_indptr[-1])

    @property
    def total_tree(self) -> int:
        return int(self.mn_indptr[-1])

    @property
    def group_size(self) -> int:
        return self.h_q // self.h_kv

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]


def _normal(rng: np.random.Generator, shape, dtype: str) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(_TORCH_DTYPE[dtype])


def build_workload(name: str, parents: Sequence[np.ndarray], *, h_q: int, h_kv: int,
                   head_dim: int, dtype: str, tensor_seed: int,
                   prefix_lens: Optional[Sequence[int]] = None,
                   qo_lens: Optional[Sequence[int]] = None,
                   positions: Optional[Sequence[np.ndarray]] = None,
                   rotary_mode: int = 0, rope_scale: float = 1.0,
                   rope_theta: float = 1e4, sm_scale: Optional[float] = None) -> Workload:
    """Assemble the ragged buffers for a batch of trees.

    ``positions[b]`` (length ``prefix + n``) gives the rope position of every
    kv token of sequence b; required when ``rotary_mode == 1``.
    """
    B = len(parents)
    prefix_lens = list(prefix_lens) if prefix_lens is not None else [0] * B
    qo_lens = list(qo_lens) if qo_lens is not None else [len(p) for p in parents]
    q_indptr = np.zeros(B + 1, dtype=np.int32)
    kv_indptr = np.zeros(B + 1, dtype=np.int32)
    mn_indptr = np.zeros(B + 1, dtype=np.int32)
    orders = []
    for b, par in enumerate(parents):
        n = len(par)
        if not 0 <= qo_lens[b] <= n:
            raise ValueError("qo_len must lie in [0, tree size]")
        q_indptr[b + 1] = q_indptr[b] + qo_lens[b]
        kv_indptr[b + 1] = kv_indptr[b] + prefix_lens[b] + n
        mn_indptr[b + 1] = mn_indptr[b] + n
        orders.append(tree_intervals(np.asarray(par)))
    tree_order = (np.concatenate(orders, axis=0) if orders else np.zeros((0, 2), np.int32))
    tree_order = np.ascontiguousarray(tree_order, dtype=np.int32)
    rng = np.random.default_rng(tensor_seed)
    tq, tkv = int(q_indptr[-1]), int(kv_indptr[-1])
    q = _normal(rng, (tq, h_q, head_dim), dtype)
    k = _normal(rng, (tkv, h_kv, head_dim), dtype)
    v = _normal(rng, (tkv, h_kv, head_dim), dtype)
    pos = None
    if positions is not None:
        pos = np.concatenate([np.asarray(p, dtype=np.int64) for p in positions]).astype(np.int32)
        if pos.shape[0] != tkv:
            raise ValueError("positions must cover every kv token")
    if rotary_mode == 1 and pos is None:
        raise ValueError("rotary_mode 1 needs positions")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    return Workload(name=name, dtype=dtype, h_q=h_q, h_kv=h_kv, head_dim=head_dim,
                    parents=[np.asarray(p, dtype=np.int64) for p in parents],
                    prefix_lens=list(prefix_lens), qo_lens=list(qo_lens), q=q, k=k, v=v,
                    q_indptr=q_indptr, kv_indptr=kv_indptr, mn_indptr=mn_indptr,
                    tree_order=tree_order, rope_position=pos, rotary_mode=rotary_mode,
                    rope_scale=float(rope_scale), rope_theta=float(rope_theta),
                    sm_scale=float(sm_scale))


# --------------------------------------------------------------------------
# the five workloads of the tree-attention benchmark
# --------------------------------------------------------------------------

CONFIG_NAMES = ["tiny", "spec-decode", "prefix+tree", "ragged-large", "degenerate"]


def config(idx: int, *, batch_scale: float = 1.0) -> Workload:
    """Workload ``idx`` (1-based, 1..5).  Tree seeds are 1000+idx, tensor
    seeds 2000+idx.  ``batch_scale`` < 1 keeps the first sequences only (for
    quick oracle samples); it never changes a sequence's shape."""
    if idx not in range(1, 6):
        raise ValueError("config index is 1..5")
    trng = np.random.default_rng(1000 + idx)
    tseed = 2000 + idx

    def keep(n_seq: int) -> int:
        return max(1, int(round(n_seq * batch_scale)))

    if idx == 1:
        parents = [random_tree(7, trng), random_tree(12, trng)]
        parents = parents[:keep(2)]
        return build_workload("tiny", parents, h_q=4, h_kv=2, head_dim=64, dtype="fp16",
                              tensor_seed=tseed, sm_scale=1.0 / 8.0, rotary_mode=0)
    if idx == 2:
        parents = [spec_decode_tree(64, trng) for _ in range(32)][:keep(32)]
        positions = [1000 + tree_depths(p) for p in parents]
        return build_workload("spec-decode", parents, h_q=32, h_kv=8, head_dim=128,
                              dtype="bf16", tensor_seed=tseed, positions=positions,
                              rotary_mode=1, rope_scale=1.0, rope_theta=1e4)
    if idx == 3:
        parents = [random_tree(128, trng) for _ in range(16)][:keep(16)]
        prefix = 2048
        positions = [np.concatenate([np.arange(prefix), prefix + tree_depths(p)])
                     for p in parents]
        return build_workload("prefix+tree", parents, h_q=32, h_kv=8, head_dim=128,
                              dtype="bf16", tensor_seed=tseed,
                              prefix_lens=[prefix] * len(parents), positions=positions,
                              rotary_mode=1, rope_scale=1.0, rope_theta=5e5)
    if idx == 4:
        sizes = trng.integers(16, 513, size=64)
        parents = [main_chain_tree(int(n), trng, 0.3) for n in sizes][:keep(64)]
        positions = [tree_depths(p) for p in parents]
        return build_workload("ragged-large", parents, h_q=64, h_kv=8, head_dim=128,
                              dtype="bf16", tensor_seed=tseed, positions=positions,
                              rotary_mode=1, rope_scale=1.0, rope_theta=1e4)
    # idx == 5
    n = 4096
    parents = [chain_tree(n), star_tree(n), binary_tree(n), random_tree(n, trng)][:keep(4)]
    return build_workload("degenerate", parents, h_q=16, h_kv=16, head_dim=128,
                          dtype="fp16", tensor_seed=tseed, rotary_mode=0)


def long_prefix(batch: int = 4, prefix: int = 32768, nodes: int = 64, seed: int = 6) -> Workload:
    """Few sequences with a long shared-history prefix: ``batch`` draft trees
    of ``nodes`` nodes shaped as in the spec-decode workload (depth <= 8,
    branching <= 4) after a causal prefix of ``prefix`` tokens, h_q=32 h_kv=8
    d=128 bf16 N(0,1), inline RoPE theta=1e4 at positions ``0..prefix-1`` then
    ``prefix + depth``.  With few (sequence, q tile) pairs each reading tens of
    thousands of kv columns, it is the case split-KV exists for.  Tree seed
    ``1000 + seed``, tensor seed ``2000 + seed``."""
    trng = np.random.default_rng(1000 + seed)
    parents = [spec_decode_tree(nodes, trng) for _ in range(batch)]
    positions = [np.concatenate([np.arange(prefix), prefix + tree_depths(p)]) for p in parents]
    return build_workload(f"long-prefix-{prefix}", parents, h_q=32, h_kv=8, head_dim=128,
                          dtype="bf16", tensor_seed=2000 + seed,
                          prefix_lens=[prefix] * batch, positions=positions, rotary_mode=1,
                          rope_scale=1.0, rope_theta=1e4)


# --------------------------------------------------------------------------
# work accounting for the benchmark metric (ancestor counts, not the mask)
# --------------------------------------------------------------------------

def visible_pairs(w: Workload) -> int:
    """Visible (q row, kv column) pairs per head: each q row sees the whole
    prefix plus its ancestor-or-self nodes (depth + 1 of them)."""
    total = 0
    for b, par in enumerate(w.parents):
        n = len(par)
        dep = tree_depths(par)
        rows = np.arange(n - w.qo_lens[b], n)
        total += int(np.sum(dep[rows] + 1)) + w.prefix_lens[b] * len(rows)
    return total


def algorithmic_flops(w: Workload) -> float:
    """2*d flops for q.k plus 2*d for p.v per visible pair and q head."""
    return 4.0 * w.head_dim * w.h_q * visible_pairs(w)


def algorithmic_bytes(w: Workload) -> float:
    """Every buffer touched once: q and out, k and v, lse, the index tables
    and (with RoPE) the position table."""
    es = 2
    b = 2 * w.total_q * w.h_q * w.head_dim * es           # q + out
    b += 2 * w.total_kv * w.h_kv * w.head_dim * es        # k + v
    b += 4 * w.total_q * w.h_q                            # lse
    b += 4 * (2 * w.total_tree + 3 * (w.batch_size + 1))  # tree_order + 3 indptr
    if w.rotary_mode == 1:
        b += 4 * w.total_kv
    return float(b)


def device_inputs(w: Workload, device="cuda") -> dict:
    """The workload's buffers as contiguous tensors on ``device`` (int32
    index arrays, q/k/v in the storage dtype)."""
    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return {
        "q": w.q.contiguous().to(device), "k": w.k.contiguous().to(device),
        "v": w.v.contiguous().to(device),
        "q_indptr": i32(w.q_indptr), "kv_indptr": i32(w.kv_indptr),
        "mn_indptr": i32(w.mn_indptr), "tree_order": i32(w.tree_order.reshape(-1, 2)),
        "q_rope_position": None if w.rope_position is None else i32(w.rope_position),
    }


# --------------------------------------------------------------------------
# paged KV cache layout of a workload (no arithmetic: a data layout only)
# --------------------------------------------------------------------------

PAGE_SIZE = 16


@dataclasses.dataclass
class PagedKV:
    """A workload's K/V moved into a paged cache ``pages [n_pages, 2, h_kv,
    16, d]`` (index 0 = K, 1 = V) with the page table of the paged tree
    attention: sequence b owns pages ``page_values[page_indptr[b]:
    page_indptr[b+1]]`` in order, its last page holding ``last_page_len[b]``
    rows."""
    pages: torch.Tensor          # [n_pages, 2, h_kv, 16, d]  CPU
    page_indptr: np.ndarray      # [B+1] int32
    page_values: np.ndarray      # [nnz_pages] int32 physical page ids
    last_page_len: np.ndarray    # [B] int32 (the pages' ``length_info``)


def paged_from(w: Workload, seed: int = 7, spare_pages: int = 3,
               fill: float = float("nan")) -> PagedKV:
    """Copies ``w.k``/``w.v`` into a paged cache: each sequence's kv rows fill
    ceil(kv / 16) logical pages, mapped to physical pages in a seeded random
    order within a pool that also has ``spare_pages`` unused pages.  Slots
    that hold no row (the tail of a last page, the spare pages) are set to
    ``fill`` -- NaN by default, so that any read of them shows."""
    rng = np.random.default_rng(seed)
    kv_lens = np.diff(w.kv_indptr.astype(np.int64))
    n_log = (kv_lens + PAGE_SIZE - 1) // PAGE_SIZE
    nnz = int(n_log.sum())
    n_pages = nnz + spare_pages
    perm = rng.permutation(n_pages)[:nnz]
    page_indptr = np.concatenate([[0], np.cumsum(n_log)]).astype(np.int32)
    last = np.where(n_log > 0, kv_lens - (n_log - 1) * PAGE_SIZE, 0).astype(np.int32)
    pages = torch.full((n_pages, 2, w.h_kv, PAGE_SIZE, w.head_dim), fill, dtype=w.k.dtype)
    for b in range(len(kv_lens)):
        k0 = int(w.kv_indptr[b])
        for lp in range(int(n_log[b])):
            phys = int(perm[page_indptr[b] + lp])
            r0 = lp * PAGE_SIZE
            r1 = min(int(kv_lens[b]), r0 + PAGE_SIZE)
            pages[phys, 0, :, : r1 - r0, :] = w.k[k0 + r0:k0 + r1].transpose(0, 1)
            pages[phys, 1, :, : r1 - r0, :] = w.v[k0 + r0:k0 + r1].transpose(0, 1)
    return PagedKV(pages=pages, page_indptr=page_indptr, page_values=perm.astype(np.int32),
                   last_page_len=last)
