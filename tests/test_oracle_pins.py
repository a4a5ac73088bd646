"""Pins for the CPU oracle: each test checks it against something that does
not come from the oracle itself -- ancestor walks over parent arrays, the
pages' causal mask, torch's scaled_dot_product_attention, closed forms,
complex-number rotation and pure-Python brute force on tiny trees.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers written from the definitions, independent of the oracle
# --------------------------------------------------------------------------

def ancestor_mask(parent, prefix, qo):
    """Visibility by walking parent links: row r (tree node n = r + T - qo)
    sees every prefix column and the kv column of each ancestor-or-self."""
    n_nodes = len(parent)
    m = np.zeros((qo, prefix + n_nodes), dtype=bool)
    m[:, :prefix] = True
    for r in range(qo):
        node = r + n_nodes - qo
        for a in wl.ancestors(parent, node):
            m[r, prefix + a] = True
    return m


def _mk(parents, prefix_lens=None, qo_lens=None, h_q=4, h_kv=2, d=16, dtype="fp16",
        seed=7, sm_scale=None, rotary_mode=0, positions=None, theta=1e4):
    return wl.build_workload("t", parents, h_q=h_q, h_kv=h_kv, head_dim=d, dtype=dtype,
                             tensor_seed=seed, prefix_lens=prefix_lens, qo_lens=qo_lens,
                             sm_scale=sm_scale, rotary_mode=rotary_mode,
                             positions=positions, rope_theta=theta)


def _tree_families(rng, n):
    return [wl.chain_tree(n), wl.star_tree(n), wl.binary_tree(n), wl.random_tree(n, rng),
            wl.main_chain_tree(n, rng), wl.spec_decode_tree(n, rng)]


# --------------------------------------------------------------------------
# mask
# --------------------------------------------------------------------------

def test_mask_golden_hand_worked():
    rows, kv = [], {}
    with open(os.path.join(GOLDEN, "mask_small.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, vals = line.split(":", 1)
            if key == "row":
                rows.append([int(x) for x in vals.split()])
            else:
                kv[key] = [int(x) for x in vals.split()]
    parent = np.array(kv["parent"])
    iv = wl.tree_intervals(parent)
    assert iv[:, 0].tolist() == kv["enter"]
    assert iv[:, 1].tolist() == kv["exit"]
    w = _mk([parent], prefix_lens=kv["prefix"], qo_lens=kv["qo"])
    vis = oracle.visibility(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, 0)
    assert vis.astype(int).tolist() == rows


@pytest.mark.parametrize("seed", range(6))
def test_mask_equals_ancestor_walk(seed):
    rng = np.random.default_rng(seed)
    parents, prefixes, qos = [], [], []
    for n in (1, 2, 5, 17, 40):
        for p in _tree_families(rng, n):
            parents.append(p)
            prefixes.append(int(rng.integers(0, 9)))
            qos.append(int(rng.integers(0, n + 1)))
    w = _mk(parents, prefix_lens=prefixes, qo_lens=qos, d=8)
    for b, p in enumerate(parents):
        vis = oracle.visibility(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, b)
        assert np.array_equal(vis, ancestor_mask(p, prefixes[b], qos[b])), b


def test_chain_mask_is_causal_mask():
    """A chain tree reproduces _causal_mask (page "_kernel_common.py"):
    col < kv_len - qo_len + row + 1."""
    n, prefix, qo = 23, 6, 9
    w = _mk([wl.chain_tree(n)], prefix_lens=[prefix], qo_lens=[qo], d=8)
    vis = oracle.visibility(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, 0)
    kv = prefix + n
    causal = np.array([[c < kv - qo + r + 1 for c in range(kv)] for r in range(qo)])
    assert np.array_equal(vis, causal)


# --------------------------------------------------------------------------
# attention vs library / closed forms
# --------------------------------------------------------------------------

def _sdpa(q, k, v, mask, scale):
    """fp64 reference via torch's scaled_dot_product_attention; q [qo,hq,d]."""
    g = q.shape[1] // k.shape[1]
    qt = q.to(torch.float64).permute(1, 0, 2)
    kt = k.to(torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = v.to(torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n,prefix", [(1, 0), (9, 0), (64, 0), (33, 17)])
def test_chain_equals_causal_attention(n, prefix):
    w = _mk([wl.chain_tree(n)], prefix_lens=[prefix], h_q=6, h_kv=3, d=32, dtype="bf16",
            sm_scale=0.21)
    out, lse = oracle.tree_attention_workload(w)
    kv = prefix + n
    mask = torch.tensor([[c < kv - n + r + 1 for c in range(kv)] for r in range(n)])
    ref = _sdpa(w.q, w.k, w.v, mask, w.sm_scale)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    if prefix == 0 and n > 1:
        qt = w.q.to(torch.float64).permute(1, 0, 2)
        kt = w.k.to(torch.float64).repeat_interleave(2, 1).permute(1, 0, 2)
        vt = w.v.to(torch.float64).repeat_interleave(2, 1).permute(1, 0, 2)
        ref2 = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=w.sm_scale)
        np.testing.assert_allclose(out, ref2.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


def test_star_closed_form():
    """Each leaf attends exactly root and itself: a two-way softmax."""
    n = 11
    w = _mk([wl.star_tree(n)], h_q=2, h_kv=1, d=16, sm_scale=0.3)
    out, lse = oracle.tree_attention_workload(w)
    q = w.q.double().numpy()
    k = w.k.double().numpy()
    v = w.v.double().numpy()
    for i in range(1, n):
        for h in range(2):
            s_root = 0.3 * float(q[i, h] @ k[0, 0])
            s_self = 0.3 * float(q[i, h] @ k[i, 0])
            w_root = 1.0 / (1.0 + math.exp(s_self - s_root))
            exp_out = w_root * v[0, 0] + (1.0 - w_root) * v[i, 0]
            np.testing.assert_allclose(out[i, h], exp_out, atol=1e-12)
            exp_lse = (max(s_root, s_self) + math.log1p(math.exp(-abs(s_root - s_self)))) / math.log(2)
            assert abs(lse[i, h] - exp_lse) < 1e-12
    # the root attends only itself
    np.testing.assert_allclose(out[0], v[0].repeat(2, 0), atol=0)


def test_single_node_returns_v_and_lse():
    w = _mk([np.array([-1])] * 3, h_q=4, h_kv=4, d=64, sm_scale=0.125)
    out, lse = oracle.tree_attention_workload(w)
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    np.testing.assert_array_equal(out, v)
    exp = 0.125 * np.einsum("thd,thd->th", q, k) / math.log(2)
    np.testing.assert_allclose(lse, exp, atol=1e-12, rtol=0)


def test_prefix_plus_single_node_is_full_attention():
    prefix = 37
    w = _mk([np.array([-1])] * 2, prefix_lens=[prefix] * 2, h_q=4, h_kv=1, d=32, dtype="bf16")
    out, lse = oracle.tree_attention_workload(w)
    for b in range(2):
        q = w.q[b:b + 1]
        k = w.k[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        v = w.v[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        ref = _sdpa(q, k, v, None, w.sm_scale)
        np.testing.assert_allclose(out[b:b + 1], ref, atol=1e-12)


def test_lse_is_base2_logsumexp_and_weights_sum_to_one():
    from scipy.special import logsumexp
    rng = np.random.default_rng(3)
    parents = [wl.random_tree(15, rng), wl.binary_tree(9)]
    w = _mk(parents, prefix_lens=[4, 0], h_q=2, h_kv=1, d=16, sm_scale=0.4)
    out, lse = oracle.tree_attention_workload(w)
    q, k = w.q.double().numpy(), w.k.double().numpy()
    for b, p in enumerate(parents):
        m = ancestor_mask(p, w.prefix_lens[b], len(p))
        kb = k[w.kv_indptr[b]:w.kv_indptr[b + 1], 0]
        for r in range(len(p)):
            for h in range(2):
                s = 0.4 * kb[m[r]] @ q[w.q_indptr[b] + r, h]
                L = float(logsumexp(s))
                assert abs(lse[w.q_indptr[b] + r, h] * math.log(2) - L) < 1e-12
                # sum_c 2^(s*log2(e) - lse) == 1
                tot = np.sum(np.exp2(s / math.log(2) - lse[w.q_indptr[b] + r, h]))
                assert abs(tot - 1.0) < 1e-12
    # v == 1 everywhere -> out == 1
    w.v = torch.ones_like(w.v)
    out1, _ = oracle.tree_attention_workload(w)
    np.testing.assert_allclose(out1, 1.0, atol=1e-14)


def test_gqa_equals_replicated_heads():
    rng = np.random.default_rng(11)
    parents = [wl.random_tree(13, rng), wl.chain_tree(6)]
    pos = [np.arange(len(p)) + 3 for p in parents]
    wg = _mk(parents, h_q=6, h_kv=2, d=32, dtype="bf16", rotary_mode=1, positions=pos)
    wm = _mk(parents, h_q=6, h_kv=6, d=32, dtype="bf16", rotary_mode=1, positions=pos)
    wm.q = wg.q.clone()
    wm.k = wg.k.repeat_interleave(3, dim=1).contiguous()
    wm.v = wg.v.repeat_interleave(3, dim=1).contiguous()
    o1, l1 = oracle.tree_attention_workload(wg)
    o2, l2 = oracle.tree_attention_workload(wm)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_relabelling_permutes_outputs():
    """Renumbering the tree nodes (rows, kv tree columns and intervals
    together) permutes the outputs the same way."""
    rng = np.random.default_rng(5)
    parent = wl.random_tree(14, rng)
    n, prefix = len(parent), 3
    w = _mk([parent], prefix_lens=[prefix], h_q=2, h_kv=1, d=16)
    perm = rng.permutation(n)                  # new label j holds old node perm[j]
    w2 = _mk([parent], prefix_lens=[prefix], h_q=2, h_kv=1, d=16)
    w2.q = w.q[torch.from_numpy(perm)].contiguous()
    kv_perm = np.concatenate([np.arange(prefix), prefix + perm])
    w2.k = w.k[torch.from_numpy(kv_perm)].contiguous()
    w2.v = w.v[torch.from_numpy(kv_perm)].contiguous()
    w2.tree_order = np.ascontiguousarray(w.tree_order[perm])
    o1, l1 = oracle.tree_attention_workload(w)
    o2, l2 = oracle.tree_attention_workload(w2)
    np.testing.assert_allclose(o2, o1[perm], atol=1e-13)
    np.testing.assert_allclose(l2, l1[perm], atol=1e-13)


def test_dense_bruteforce_tiny_trees():
    """Pure-Python loops: ancestor walk for the mask, math.exp softmax."""
    rng = np.random.default_rng(21)
    for trial in range(4):
        parents = [wl.random_tree(int(rng.integers(1, 13)), rng) for _ in range(3)]
        prefixes = [int(rng.integers(0, 4)) for _ in parents]
        qos = [int(rng.integers(0, len(p) + 1)) for p in parents]
        w = _mk(parents, prefix_lens=prefixes, qo_lens=qos, h_q=4, h_kv=2, d=8,
                seed=100 + trial, sm_scale=0.37)
        out, lse = oracle.tree_attention_workload(w)
        q, k, v = (t.double().tolist() for t in (w.q, w.k, w.v))
        for b, p in enumerate(parents):
            n = len(p)
            for r in range(qos[b]):
                node = r + n - qos[b]
                cols = list(range(prefixes[b])) + [prefixes[b] + a for a in wl.ancestors(p, node)]
                for h in range(4):
                    kh = h // 2
                    row = w.q_indptr[b] + r
                    sc = []
                    for c in cols:
                        kvr = w.kv_indptr[b] + c
                        sc.append(0.37 * sum(q[row][h][i] * k[kvr][kh][i] for i in range(8)))
                    mx = max(sc)
                    z = sum(math.exp(s - mx) for s in sc)
                    for i in range(8):
                        o = sum(math.exp(s - mx) / z * v[w.kv_indptr[b] + c][kh][i]
                                for s, c in zip(sc, cols))
                        assert abs(out[row, h, i] - o) < 1e-12
                    assert abs(lse[row, h] - (mx + math.log(z)) / math.log(2)) < 1e-12


def test_row_without_visible_column():
    """An invalid interval (exit == enter) leaves a row nothing to attend:
    the oracle returns out = 0 and lse = -inf for it."""
    w = _mk([wl.chain_tree(3)], h_q=2, h_kv=1, d=8)
    w.tree_order = w.tree_order.copy()
    w.tree_order[2, 1] = w.tree_order[2, 0]        # node 2 now contains nothing
    out, lse = oracle.tree_attention_workload(w)
    # node 2's row still sees its ancestors 0 and 1 (their intervals hold it),
    # but nothing sees node 2 itself now; row 2 still has columns 0 and 1
    assert np.isfinite(lse[2]).all()
    w.tree_order[:, 1] = w.tree_order[:, 0]         # every interval empty
    out, lse = oracle.tree_attention_workload(w)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_empty_sequences_in_batch():
    rng = np.random.default_rng(2)
    parents = [wl.random_tree(5, rng), wl.random_tree(4, rng), wl.random_tree(6, rng)]
    w = _mk(parents, prefix_lens=[2, 3, 0], qo_lens=[5, 0, 6], d=16)
    out, lse = oracle.tree_attention_workload(w)
    assert out.shape[0] == 11 and not np.isnan(out).any() and not np.isnan(lse).any()


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_identity_at_position_zero():
    x = torch.randn(7, 3, 64).to(torch.bfloat16)
    y = oracle.apply_rope(x, np.zeros(7, dtype=np.int64), 1e4, 1.0)
    assert torch.equal(x, y)


@pytest.mark.parametrize("d,theta,scale", [(64, 1e4, 1.0), (128, 5e5, 1.0), (128, 1e4, 0.5)])
def test_rope_is_rotate_half_complex_rotation(d, theta, scale):
    """Rotate-half RoPE equals multiplying z = x[:d/2] + i x[d/2:] by
    exp(i * pos * scale * theta^(-2i/d)) (complex128 reference)."""
    rng = np.random.default_rng(1)
    rows = 40
    x = torch.from_numpy(rng.standard_normal((rows, 2, d)).astype(np.float32))
    pos = rng.integers(0, 3000, size=rows)
    y = oracle.apply_rope(x, pos, theta, scale).numpy().astype(np.float64)
    half = d // 2
    xd = x.numpy().astype(np.float64)
    z = xd[..., :half] + 1j * xd[..., half:]
    ang = (pos * scale)[:, None] * theta ** (-2.0 * np.arange(half) / d)[None, :]
    zr = z * np.exp(1j * ang)[:, None, :]
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    # float32 angle (|angle| <= 3000) carries ~3000 * 2^-24 of error
    np.testing.assert_allclose(y, ref, atol=2e-3 * np.abs(xd).max(), rtol=0)
    # and each (j, j + d/2) pair keeps its norm
    np.testing.assert_allclose(np.abs(y[..., :half] + 1j * y[..., half:]), np.abs(z), rtol=1e-5)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(4)
    d = 64
    q = torch.from_numpy(rng.standard_normal((1, 1, d)).astype(np.float32))
    k = torch.from_numpy(rng.standard_normal((1, 1, d)).astype(np.float32))
    s = []
    for shift in (0, 7, 100):
        qr = oracle.apply_rope(q, np.array([20 + shift]), 1e4, 1.0)
        kr = oracle.apply_rope(k, np.array([5 + shift]), 1e4, 1.0)
        s.append(float((qr.double() * kr.double()).sum()))
    assert max(s) - min(s) < 1e-4


def test_rope_rounds_to_storage_dtype_once():
    """_rope casts the float32 sum to the storage dtype: the result must be
    exactly the RNE rounding of the float32 rotation."""
    rng = np.random.default_rng(9)
    d = 128
    x = torch.from_numpy(rng.standard_normal((16, 4, d)).astype(np.float32))
    pos = rng.integers(0, 5000, size=16)
    y32 = oracle.apply_rope(x.to(torch.bfloat16).float(), pos, 1e4, 1.0)
    y16 = oracle.apply_rope(x.to(torch.bfloat16), pos, 1e4, 1.0)
    assert y16.dtype == torch.bfloat16
    assert torch.equal(y32.to(torch.bfloat16), y16)


def test_rope_frequency_denominators():
    den = oracle.rope_inv_freq_denominators(128, 1e4)
    assert den[0] == 1.0 and den.dtype == np.float32
    np.testing.assert_allclose(den.astype(np.float64), 1e4 ** (np.arange(64) / 64.0), rtol=1e-7)


def test_q_position_is_its_own_kv_slot():
    """With prefixes, q row r uses the position of its own tree node's kv
    token: if q equals that token's k, the self score is |rope(q)|^2."""
    prefix = 5
    parents = [np.array([-1]), np.array([-1])]
    pos = [np.array([0, 1, 2, 3, 4, 900]), np.array([10, 11, 12, 13, 14, 2500])]
    w = _mk(parents, prefix_lens=[prefix] * 2, h_q=1, h_kv=1, d=64, dtype="bf16",
            rotary_mode=1, positions=pos, sm_scale=1.0)
    w.k[:] = 0
    for b in range(2):
        w.k[w.kv_indptr[b] + prefix] = w.q[b]
    out, lse = oracle.tree_attention_workload(w)
    for b in range(2):
        qr = oracle.apply_rope(w.q[b:b + 1], np.array([pos[b][-1]]), 1e4, 1.0).double()
        s_self = float((qr * qr).sum())
        # prefix keys are zero: 5 scores of 0 plus the self score
        exp_lse = math.log(5 * math.exp(0.0) + math.exp(s_self)) / math.log(2)
        assert abs(lse[b, 0] - exp_lse) < 1e-9


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------

def test_workload_shapes_match_their_definitions():
    w2 = wl.config(2)
    for p in w2.parents:
        dep = wl.tree_depths(p)
        assert len(p) == 64 and dep.max() <= 8
        assert np.bincount(p[1:], minlength=64).max() <= 4
    assert (w2.h_q, w2.h_kv, w2.head_dim, w2.dtype, w2.rotary_mode) == (32, 8, 128, "bf16", 1)
    assert np.array_equal(w2.rope_position[:64], 1000 + wl.tree_depths(w2.parents[0]))
    w3 = wl.config(3)
    assert w3.total_kv == 16 * (2048 + 128) and w3.total_q == 16 * 128
    assert np.array_equal(w3.rope_position[:2048], np.arange(2048))
    assert w3.rope_theta == 5e5
    w5 = wl.config(5)
    assert np.array_equal(w5.parents[0], wl.chain_tree(4096))
    assert np.all(w5.parents[1][1:] == 0)
    assert np.array_equal(w5.parents[2][1:], (np.arange(1, 4096) - 1) // 2)
    assert (w5.h_q, w5.h_kv, w5.rotary_mode, w5.dtype) == (16, 16, 0, "fp16")
    w1 = wl.config(1)
    assert [len(p) for p in w1.parents] == [7, 12] and w1.sm_scale == 0.125


def test_visible_pairs_counts_ancestors():
    w = wl.config(5)
    n = 4096
    per = [n * (n + 1) // 2, 1 + 2 * (n - 1), None, None]
    assert wl.visible_pairs(wl.build_workload("c", [w.parents[0]], h_q=1, h_kv=1, head_dim=8,
                                              dtype="fp16", tensor_seed=0)) == per[0]
    assert wl.visible_pairs(wl.build_workload("s", [w.parents[1]], h_q=1, h_kv=1, head_dim=8,
                                              dtype="fp16", tensor_seed=0)) == per[1]
    # the count equals the number of True entries in the ancestor mask
    rng = np.random.default_rng(0)
    ps = [wl.random_tree(30, rng)]
    ww = wl.build_workload("r", ps, h_q=1, h_kv=1, head_dim=8, dtype="fp16", tensor_seed=0,
                           prefix_lens=[4])
    assert wl.visible_pairs(ww) == int(ancestor_mask(ps[0], 4, 30).sum())


# --------------------------------------------------------------------------
# paged KV cache (tree_attn_with_paged_kv_cache_cpu, page "tree_attn.py")
# --------------------------------------------------------------------------

def _paged_workloads():
    rng = np.random.default_rng(11)
    ws = [wl.config(1)]
    # prefix + tree, several pages per sequence, partial last pages, GQA
    ws.append(wl.build_workload("pp", [wl.random_tree(23, rng), wl.random_tree(40, rng),
                                       wl.random_tree(5, rng)],
                                h_q=4, h_kv=2, head_dim=64, dtype="bf16", tensor_seed=5,
                                prefix_lens=[37, 0, 16], qo_lens=[9, 40, 5]))
    # chain, star and binary trees whose lengths are exact multiples of 16
    ws.append(wl.build_workload("pd", [wl.chain_tree(32), wl.star_tree(48), wl.binary_tree(16)],
                                h_q=2, h_kv=2, head_dim=64, dtype="fp16", tensor_seed=6))
    return ws


@pytest.mark.parametrize("i", range(3))
def test_paged_equals_contiguous(i):
    """Fetching K/V rows through the page table (scattered physical pages,
    partial last pages, NaN in every slot no sequence owns) gives exactly the
    contiguous-cache attention, which is pinned on its own above."""
    w = _paged_workloads()[i]
    pk = wl.paged_from(w, seed=100 + i)
    assert not np.array_equal(pk.page_values, np.arange(len(pk.page_values)))
    o1, l1 = oracle.tree_attention_workload(w)
    o2, l2 = oracle.tree_attention_paged(w.q, w.q_indptr, pk.pages, pk.page_indptr,
                                         pk.page_values, pk.last_page_len, w.mn_indptr,
                                         w.tree_order, 0, w.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_kv_lengths_follow_the_page_count():
    # 3 pages with 5 rows in the last: 2*16 + 5; one full page: 16; no page: 0
    lens = oracle.paged_kv_lengths(np.array([0, 3, 4, 4]), np.array([5, 16, 7]))
    assert lens.tolist() == [37, 16, 0]
    w = _paged_workloads()[1]
    pk = wl.paged_from(w)
    assert np.array_equal(oracle.paged_kv_lengths(pk.page_indptr, pk.last_page_len),
                          np.diff(w.kv_indptr))


def test_paged_never_reads_unowned_slots():
    w = _paged_workloads()[1]
    outs = []
    for fill in (float("nan"), float("inf"), 0.0, 3.0):
        pk = wl.paged_from(w, seed=3, fill=fill)
        outs.append(oracle.tree_attention_paged(w.q, w.q_indptr, pk.pages, pk.page_indptr,
                                                pk.page_values, pk.last_page_len, w.mn_indptr,
                                                w.tree_order, 0, w.sm_scale))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    assert np.isfinite(outs[0][0]).all()


def test_paged_rejects_rope():
    w = _paged_workloads()[0]
    pk = wl.paged_from(w)
    with pytest.raises(ValueError):
        oracle.tree_attention_paged(w.q, w.q_indptr, pk.pages, pk.page_indptr, pk.page_values,
                                    pk.last_page_len, w.mn_indptr, w.tree_order, 1, w.sm_scale)


# --------------------------------------------------------------------------
# merging partial attention states (split-KV)
# --------------------------------------------------------------------------

def _masked_oracle(w, keep):
    """The oracle restricted to the kv columns where ``keep(b, c)`` holds:
    the same computation with the other columns' v and scores removed, done
    here by replacing the tree visibility (a plain boolean restriction)."""
    real = oracle.tree_attn_ref.visibility

    def restricted(q_indptr, kv_indptr, mn_indptr, order, b):
        vis = real(q_indptr, kv_indptr, mn_indptr, order, b)
        cols = np.arange(vis.shape[1])
        return vis & keep(b, cols)[None, :]

    oracle.tree_attn_ref.visibility = restricted
    try:
        return oracle.tree_attention_workload(w)
    finally:
        oracle.tree_attn_ref.visibility = real


@pytest.mark.parametrize("parts", [2, 3, 5])
def test_merge_of_disjoint_column_sets_equals_the_whole(parts):
    rng = np.random.default_rng(parts)
    w = wl.build_workload("m", [wl.random_tree(30, rng), wl.chain_tree(12)], h_q=4, h_kv=2,
                          head_dim=16, dtype="fp16", tensor_seed=parts, prefix_lens=[50, 7])
    o_all, l_all = oracle.tree_attention_workload(w)
    # columns dealt to parts in a scrambled pattern (not contiguous ranges)
    lab = [rng.integers(0, parts, size=int(w.kv_indptr[b + 1] - w.kv_indptr[b]))
           for b in range(w.batch_size)]
    outs, lses = [], []
    for i in range(parts):
        o, l = _masked_oracle(w, lambda b, c, i=i: lab[b][c] == i)
        outs.append(o)
        lses.append(l)
    o_m, l_m = oracle.merge_states(outs, lses)
    assert np.allclose(o_m, o_all, rtol=0, atol=1e-12)
    fin = np.isfinite(l_all)
    assert np.array_equal(fin, np.isfinite(l_m))
    assert np.allclose(l_m[fin], l_all[fin], rtol=0, atol=1e-12)


def test_merge_closed_forms():
    o1 = np.array([[1.0, 2.0]]); o2 = np.array([[3.0, 6.0]])
    # equal lse: the average; lse grows by one (base 2)
    o, l = oracle.merge_states([o1, o2], [np.array([0.5]), np.array([0.5])])
    assert np.allclose(o, [[2.0, 4.0]]) and np.allclose(l, [1.5])
    # a part with nothing visible contributes nothing
    o, l = oracle.merge_states([o1, o2], [np.array([3.0]), np.array([-np.inf])])
    assert np.allclose(o, o1) and np.allclose(l, [3.0])
    # nothing visible anywhere
    o, l = oracle.merge_states([o1, o2], [np.array([-np.inf]), np.array([-np.inf])])
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # weights 2^lse: lse 1 and 0 -> weights 2/3 and 1/3
    o, l = oracle.merge_states([o1, o2], [np.array([1.0]), np.array([0.0])])
    assert np.allclose(o, (2 * o1 + o2) / 3) and np.allclose(l, [np.log2(3.0)])
