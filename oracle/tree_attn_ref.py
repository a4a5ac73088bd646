"""Plain, slow, obviously-correct CPU oracle for batched tree attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg, never by the product path.

Precision.  The attention itself (scores, softmax, weighted sum of v) is
evaluated in float64.  The rotary embedding follows the precision the pages
fix for it: ``_rope`` on the page "_kernel_common.py" asks the frequency
function for float32 cos/sin of ``offset * scale``, multiplies them with the
float32-cast element and its rotate-half partner, adds, and casts the sum to
the q/k storage dtype.  The oracle performs exactly those float32 steps (each
product and the sum rounded to float32, no fused multiply-add), with the
frequency step read as ``angle = fl32(fl32(pos * scale) / fl32(theta **
(2 i / d)))`` and ``cos``/``sin`` taken correctly rounded from float64.

Functions and the passages they restate:

* ``visibility``      -- ``_check_tree_order`` (page "tree_attn.py").
* ``rope_cos_sin``,
  ``apply_rope``      -- ``_rope`` (page "_kernel_common.py"); rotary_dim = d,
                         as ``batch_tree_attn`` passes ``d``.
* ``tree_attention``  -- ``tree_attn_cpu`` / ``batch_tree_attn`` (page
                         "tree_attn.py"): per sequence, per q row, per head,
                         masked softmax over kv columns of sm_scale * q.k,
                         output the softmax-weighted sum of v and the
                         log-sum-exp in base 2 (``m + log2(d)`` with scores
                         pre-multiplied by log2(e)).
* ``merge_states``    -- combining attention states over disjoint kv sets
                         through their base-2 log-sum-exps (the ``lse_store``
                         epilogue of page "tree_attn.py" defines the lse).
* ``paged_kv_lengths``,
  ``tree_attention_paged`` -- ``_get_kv_chunk_len`` (page "_kernel_common.py")
                         and ``tree_attn_with_paged_kv_cache_cpu`` (page
                         "tree_attn.py"): the same attention with K/V rows
                         fetched through a page table of 16-slot pages.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np
import torch

LN2 = math.log(2.0)

_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16,
           torch.float16: torch.float16, torch.bfloat16: torch.bfloat16}


# --------------------------------------------------------------------------
# tree mask: _check_tree_order
# --------------------------------------------------------------------------

def visibility(q_indptr, kv_indptr, mn_indptr, tree_order, b: int) -> np.ndarray:
    """Boolean ``[qo_len, kv_len]`` visibility of sequence ``b``.

    Restates ``_check_tree_order`` (page "tree_attn.py"): with
    ``tree_len = mn_indptr[b+1] - mn_indptr[b]`` and
    ``tree_start = kv_len - tree_len``, q row ``r`` is tree node
    ``child = r + tree_len - qo_len`` and kv column ``c`` (if
    ``c >= tree_start``) is tree node ``parent = c - tree_start``.  Column c
    is visible iff ``c < kv_len`` and (``c < tree_start`` or
    ``enter[child] >= enter[parent]`` and ``enter[child] < exit[parent]``).
    Prefix columns never index the tree table.
    """
    qo = int(q_indptr[b + 1] - q_indptr[b])
    kv = int(kv_indptr[b + 1] - kv_indptr[b])
    tl = int(mn_indptr[b + 1] - mn_indptr[b])
    ts = kv - tl
    base = int(mn_indptr[b])
    order = np.asarray(tree_order, dtype=np.int64)
    vis = np.zeros((qo, kv), dtype=bool)
    if qo == 0 or kv == 0:
        return vis
    vis[:, :ts] = True
    child = np.arange(qo) + tl - qo                  # tree node of every q row
    e_child = order[base + child, 0][:, None]        # [qo, 1]
    par = np.arange(tl)
    e_par = order[base + par, 0][None, :]             # [1, tl]
    x_par = order[base + par, 1][None, :]
    vis[:, ts:] = (e_child >= e_par) & (e_child < x_par)
    return vis


# --------------------------------------------------------------------------
# rotary embedding: _rope, in the float32 steps the pages fix
# --------------------------------------------------------------------------

def rope_inv_freq_denominators(d: int, theta: float) -> np.ndarray:
    """``fl32(theta ** (2 i / d))`` for pair index ``i in [0, d/2)``: the
    element index ``j`` uses exponent ``(2 j mod d) / d``, so elements j and
    j + d/2 share frequency i = j mod d/2."""
    th = float(np.float32(theta))
    return np.array([th ** (2.0 * i / d) for i in range(d // 2)], dtype=np.float64).astype(np.float32)


def rope_cos_sin(pos: np.ndarray, d: int, theta: float, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """float32 cos/sin tables ``[len(pos), d/2]``.

    ``offset * scale`` is a float32 product (int position promoted to
    float32); the angle is that value divided in float32 by the frequency
    denominator; cos and sin are correctly rounded to float32.
    """
    pos32 = np.asarray(pos).astype(np.float32)
    s = pos32 * np.float32(scale)                                   # float32 product
    den = rope_inv_freq_denominators(d, theta)
    ang = (s[:, None] / den[None, :]).astype(np.float32)            # float32 division
    a64 = ang.astype(np.float64)
    return np.cos(a64).astype(np.float32), np.sin(a64).astype(np.float32)


def apply_rope(x: torch.Tensor, pos: np.ndarray, theta: float, scale: float) -> torch.Tensor:
    """Rotate-half RoPE of ``x`` ``[rows, heads, d]`` (fp16/bf16) at per-row
    positions ``pos``; returns the rotated tensor in x's dtype.

    For element j < d/2: ``cos*x[j] + sin*(-x[j+d/2])``; for j >= d/2:
    ``cos*x[j] + sin*x[j-d/2]``; each product and the sum are float32, the
    result is cast (round-to-nearest-even) to the storage dtype.
    """
    rows, heads, d = x.shape
    half = d // 2
    c, s = rope_cos_sin(pos, d, theta, scale)                      # [rows, half]
    c = np.concatenate([c, c], axis=1)[:, None, :]                 # [rows, 1, d]
    s = np.concatenate([s, s], axis=1)[:, None, :]
    xf = x.to(torch.float32).numpy()
    partner = np.concatenate([-xf[..., half:], xf[..., :half]], axis=-1)
    first = (c * xf).astype(np.float32)
    second = (s * partner).astype(np.float32)
    summed = (first + second).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(summed)).to(x.dtype)


# --------------------------------------------------------------------------
# tree attention: tree_attn_cpu / batch_tree_attn
# --------------------------------------------------------------------------

def _as_np(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        return a.detach().cpu().numpy()
    return np.asarray(a)


def tree_attention(q: torch.Tensor, q_indptr, k: torch.Tensor, v: torch.Tensor, kv_indptr,
                   q_rope_position, mn_indptr, tree_order, rotary_mode: int,
                   rope_scale: float, rope_theta: float, sm_scale: float,
                   seqs: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Batched tree attention; returns ``(out, lse)`` as float64 arrays
    ``[total_q, h_q, d]`` and ``[total_q, h_q]`` (lse in base 2).

    ``q_rope_position`` holds the position of every kv token (length
    ``total_kv``).  Key column c of sequence b takes position
    ``pos[kv_indptr[b] + c]`` (as the pages index it); q row r takes the
    position of its own tree node's kv slot,
    ``pos[kv_indptr[b] + tree_start + (tree_len - qo_len) + r]``, which is the
    pages' ``pos[q_indptr[b] + r]`` whenever q_indptr equals kv_indptr.

    A q row with no visible column gets ``out = 0`` and ``lse = -inf``.
    Rows of sequences outside ``seqs`` stay NaN.
    """
    q_indptr = _as_np(q_indptr).astype(np.int64)
    kv_indptr = _as_np(kv_indptr).astype(np.int64)
    mn_indptr = _as_np(mn_indptr).astype(np.int64)
    order = _as_np(tree_order).astype(np.int64).reshape(-1, 2)
    pos = None if q_rope_position is None else _as_np(q_rope_position).astype(np.int64)
    tq, h_q, d = q.shape
    h_kv = k.shape[1]
    if h_q % h_kv != 0:
        raise ValueError("h_q must be a multiple of h_kv")
    g = h_q // h_kv
    out = np.full((tq, h_q, d), np.nan, dtype=np.float64)
    lse = np.full((tq, h_q), np.nan, dtype=np.float64)
    B = len(q_indptr) - 1
    for b in (range(B) if seqs is None else seqs):
        q0, q1 = int(q_indptr[b]), int(q_indptr[b + 1])
        k0, k1 = int(kv_indptr[b]), int(kv_indptr[b + 1])
        qo, kv = q1 - q0, k1 - k0
        if qo == 0:
            continue
        tl = int(mn_indptr[b + 1] - mn_indptr[b])
        ts = kv - tl
        vis = visibility(q_indptr, kv_indptr, mn_indptr, order, b)
        qb, kb, vb = q[q0:q1], k[k0:k1], v[k0:k1]
        if rotary_mode == 1:
            qpos = pos[k0 + ts + (tl - qo) + np.arange(qo)]
            kpos = pos[k0:k1]
            qb = apply_rope(qb, qpos, rope_theta, rope_scale)
            kb = apply_rope(kb, kpos, rope_theta, rope_scale)
        _attend_sequence(qb, kb, vb, vis, sm_scale, g, out[q0:q1], lse[q0:q1])
    return out, lse


def _attend_sequence(qb: torch.Tensor, kb: torch.Tensor, vb: torch.Tensor, vis: np.ndarray,
                     sm_scale: float, g: int, out: np.ndarray, lse: np.ndarray) -> None:
    """One sequence of ``tree_attn_cpu`` (page "tree_attn.py") after the
    q/k/v rows are fetched (and rotated): per kv head and q head, the masked
    softmax over the visible columns of ``sm_scale * q.k`` in float64, the
    softmax-weighted sum of v into ``out [qo, h_q, d]`` and the base-2
    log-sum-exp into ``lse [qo, h_q]``.  A row with no visible column gets
    ``out = 0`` and ``lse = -inf``."""
    qo, kv = vis.shape
    h_kv = kb.shape[1]
    q64 = qb.to(torch.float64).numpy()
    k64 = kb.to(torch.float64).numpy()
    v64 = vb.to(torch.float64).numpy()
    any_vis = vis.any(axis=1)                                   # [qo]
    for kh in range(h_kv):
        heads = slice(kh * g, (kh + 1) * g)
        qh = np.transpose(q64[:, heads, :], (1, 0, 2))          # [g, qo, d]
        s = sm_scale * np.matmul(qh, k64[:, kh, :].T)            # [g, qo, kv]
        s = np.where(vis[None], s, -np.inf)
        m = np.max(s, axis=2, keepdims=True) if kv else np.full((g, qo, 1), -np.inf)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)                                        # masked -> 0
        z = np.sum(e, axis=2, keepdims=True)
        with np.errstate(divide="ignore", invalid="ignore"):
            L = m + np.log(z)                                    # natural log-sum-exp
            w = np.where(z > 0, e / z, 0.0)
        o = np.matmul(w, v64[:, kh, :]) if kv else np.zeros((g, qo, v64.shape[2]))
        o[:, ~any_vis, :] = 0.0
        Lr = L[..., 0]
        Lr[:, ~any_vis] = -np.inf
        out[:, heads, :] = np.transpose(o, (1, 0, 2))
        lse[:, heads] = (Lr / LN2).T


# --------------------------------------------------------------------------
# paged KV cache: tree_attn_with_paged_kv_cache_cpu
# --------------------------------------------------------------------------

PAGE_SIZE = 16


def paged_kv_lengths(page_indptr, last_page_len) -> np.ndarray:
    """kv length of every sequence of a paged cache, ``_get_kv_chunk_len``
    (page "_kernel_common.py") without a sliding window:
    ``(num_pages - 1) * page_size + last_page_len``, and 0 for a sequence that
    owns no page (the guard of ``tree_attn_with_paged_kv_cache_cpu``)."""
    page_indptr = _as_np(page_indptr).astype(np.int64)
    last = _as_np(last_page_len).astype(np.int64)
    n = page_indptr[1:] - page_indptr[:-1]
    return np.where(n > 0, (n - 1) * PAGE_SIZE + last, 0)


def tree_attention_paged(q: torch.Tensor, q_indptr, pages: torch.Tensor, page_indptr,
                         page_values, last_page_len, mn_indptr, tree_order, rotary_mode: int,
                         sm_scale: float,
                         seqs: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Tree attention over a paged KV cache; ``(out, lse)`` as in
    ``tree_attention``.

    Restates ``tree_attn_with_paged_kv_cache_cpu`` (page "tree_attn.py"):
    ``pages [max_num_pages, 2, h_kv, 16, d]`` holds K (index 0) and V (1);
    kv row r of sequence b lives in page
    ``page_values[page_indptr[b] + r // 16]`` at slot ``r % 16``; the kv length
    comes from ``paged_kv_lengths``; the tree mask is ``_check_tree_order``
    with that length.  The pages assert ``rotary_mode == 0`` for this kernel
    (no RoPE), and so does this function.  Slots past a sequence's length are
    never read.
    """
    if rotary_mode != 0:
        raise ValueError("paged tree attention supports rotary_mode 0 only")
    q_indptr = _as_np(q_indptr).astype(np.int64)
    page_indptr = _as_np(page_indptr).astype(np.int64)
    page_values = _as_np(page_values).astype(np.int64)
    mn_indptr = _as_np(mn_indptr).astype(np.int64)
    order = _as_np(tree_order).astype(np.int64).reshape(-1, 2)
    kv_len = paged_kv_lengths(page_indptr, last_page_len)
    kv_indptr = np.concatenate([[0], np.cumsum(kv_len)])
    tq, h_q, d = q.shape
    h_kv = pages.shape[2]
    if h_q % h_kv != 0:
        raise ValueError("h_q must be a multiple of h_kv")
    g = h_q // h_kv
    out = np.full((tq, h_q, d), np.nan, dtype=np.float64)
    lse = np.full((tq, h_q), np.nan, dtype=np.float64)
    B = len(q_indptr) - 1
    for b in (range(B) if seqs is None else seqs):
        q0, q1 = int(q_indptr[b]), int(q_indptr[b + 1])
        if q1 == q0:
            continue
        rows = np.arange(int(kv_len[b]))
        phys = page_values[page_indptr[b] + rows // PAGE_SIZE]
        slot = rows % PAGE_SIZE
        kb = pages[phys, 0, :, slot, :]                          # [kv, h_kv, d]
        vb = pages[phys, 1, :, slot, :]
        vis = visibility(q_indptr, kv_indptr, mn_indptr, order, b)
        _attend_sequence(q[q0:q1], kb, vb, vis, sm_scale, g, out[q0:q1], lse[q0:q1])
    return out, lse


def tree_attention_workload(w, seqs: Optional[Iterable[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """``tree_attention`` on a ``workloads.Workload``."""
    return tree_attention(w.q, w.q_indptr, w.k, w.v, w.kv_indptr, w.rope_position,
                          w.mn_indptr, w.tree_order, w.rotary_mode, w.rope_scale,
                          w.rope_theta, w.sm_scale, seqs=seqs)


# --------------------------------------------------------------------------
# merging partial attention states (split-KV)
# --------------------------------------------------------------------------

def merge_states(outs, lses) -> Tuple[np.ndarray, np.ndarray]:
    """Combines attention states over disjoint sets of kv columns into the
    state over their union.  ``outs [n, ..., d]`` are the normalised partial
    outputs, ``lses [n, ...]`` their base-2 log-sum-exps (the ``m + log2(d)``
    of ``lse_store``, page "tree_attn.py", which is what makes partial
    attentions mergeable): ``lse = log2(sum_i 2^lse_i)`` and ``out = sum_i
    2^(lse_i - lse) * out_i``.  Parts with ``lse = -inf`` (nothing visible)
    contribute nothing; if every part has ``-inf``, ``out = 0`` and
    ``lse = -inf``.  float64."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = np.max(lses, axis=0)
    any_fin = np.isfinite(m)
    m0 = np.where(any_fin, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp2(lses - m0[None]), 0.0)        # [n, ...]
    z = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(any_fin, m0 + np.log2(z), -np.inf)
        out = np.where(any_fin[..., None], np.sum(w[..., None] * outs, axis=0) / z[..., None], 0.0)
    return out, lse
