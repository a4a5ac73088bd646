"""GPU parity of the paged-KV tree attention (``tree_attn_with_paged_kv_cache``
of the page "tree_attn.py"), called through the C ABI, against the CPU oracle
on seeded inputs, and against the library's contiguous-cache path.

Every cache slot that no sequence owns -- the tail of a partly filled last
page and the pool's spare pages -- holds NaN, so a kernel that let any of them
reach the output fails.  Bars as in test_gpu_parity: output max-abs error
<= 1e-2 (fp16) / 2e-2 (bf16), base-2 LSE error <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_attention_gb300 as ta
import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = {"fp16": 1e-2, "bf16": 2e-2}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tree_attention_gb300 import build
    build.build()
    ta.lib()


def _workloads():
    rng = np.random.default_rng(21)
    return {
        "tiny": wl.config(1),
        # prefix + random trees, several pages per sequence, partial last pages, GQA g = 2
        "prefix_gqa_d64": wl.build_workload(
            "pp", [wl.random_tree(23, rng), wl.random_tree(40, rng), wl.random_tree(5, rng)],
            h_q=4, h_kv=2, head_dim=64, dtype="bf16", tensor_seed=5,
            prefix_lens=[37, 0, 16], qo_lens=[9, 40, 5]),
        # draft trees after a 300-token prefix, g = 4, d = 128 (spec-decode shape)
        "spec_like_d128": wl.build_workload(
            "sd", [wl.spec_decode_tree(64, rng) for _ in range(6)], h_q=32, h_kv=8,
            head_dim=128, dtype="bf16", tensor_seed=9, prefix_lens=[300, 17, 0, 64, 129, 5]),
        # chain / star / binary trees, MHA fp16, lengths around page multiples
        "degenerate_fp16": wl.build_workload(
            "dg", [wl.chain_tree(200), wl.star_tree(161), wl.binary_tree(96)], h_q=4, h_kv=4,
            head_dim=128, dtype="fp16", tensor_seed=7),
        # g = 8 with long prefixes (several 64-row tiles of pages)
        "g8_long_prefix": wl.build_workload(
            "lp", [wl.random_tree(33, rng), wl.random_tree(70, rng)], h_q=64, h_kv=8,
            head_dim=128, dtype="bf16", tensor_seed=11, prefix_lens=[517, 250]),
    }


def _paged_gpu(w, pk):
    dev = "cuda"
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    q = w.q.contiguous().to(dev)
    pages = pk.pages.contiguous().to(dev)
    tree_order = i32(w.tree_order.reshape(-1, 2))
    page_values = i32(pk.page_values)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    dims = ta.make_paged_dims(q, pages, i32(w.q_indptr), page_values, tree_order)
    ws = torch.zeros(ta.paged_workspace_size(dims), dtype=torch.uint8, device=dev)
    ta.tree_attn_paged(q, i32(w.q_indptr), pages, i32(pk.page_indptr), page_values,
                       i32(pk.last_page_len), i32(w.mn_indptr), tree_order, out, lse, 0,
                       w.sm_scale, ws)
    st = ta.device_status(ws)
    assert st == ta.TA_OK, ta.status_string(st)
    return out, lse


@pytest.mark.parametrize("name", list(_workloads()))
def test_paged_matches_oracle(name):
    w = _workloads()[name]
    pk = wl.paged_from(w, seed=31)
    out, lse = _paged_gpu(w, pk)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    ro, rl = oracle.tree_attention_paged(w.q, w.q_indptr, pk.pages, pk.page_indptr,
                                         pk.page_values, pk.last_page_len, w.mn_indptr,
                                         w.tree_order, 0, w.sm_scale)
    assert np.isfinite(out).all(), "a slot no sequence owns reached the output"
    err_o = float(np.max(np.abs(out - ro)))
    assert err_o <= TOL_OUT[w.dtype], f"out max|err| {err_o}"
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    err_l = float(np.max(np.abs(lse[fin] - rl[fin])))
    assert err_l <= TOL_LSE, f"lse max|err| {err_l}"


@pytest.mark.parametrize("name", ["prefix_gqa_d64", "spec_like_d128", "degenerate_fp16"])
def test_paged_equals_contiguous_path(name):
    """The same K/V through the page table or contiguous: identical bits (the
    tiles hold the same values and go through the same arithmetic)."""
    w = _workloads()[name]
    out_p, lse_p = _paged_gpu(w, wl.paged_from(w, seed=5))
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], 0, 1.0, 1e4,
                            w.sm_scale)
    out_c, lse_c = attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    assert torch.equal(out_p, out_c)
    assert torch.equal(lse_p, lse_c)


def test_paged_bad_page_table_is_reported():
    w = _workloads()["prefix_gqa_d64"]
    pk = wl.paged_from(w)
    bad = pk.last_page_len.copy()
    bad[0] = 17                              # more than a page holds
    pk2 = wl.PagedKV(pages=pk.pages, page_indptr=pk.page_indptr, page_values=pk.page_values,
                     last_page_len=bad)
    dev = "cuda"
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    q = w.q.to(dev)
    pages = pk2.pages.to(dev)
    tree_order = i32(w.tree_order.reshape(-1, 2))
    page_values = i32(pk2.page_values)
    out = torch.full_like(q, 7.0)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    dims = ta.make_paged_dims(q, pages, i32(w.q_indptr), page_values, tree_order)
    ws = torch.zeros(ta.paged_workspace_size(dims), dtype=torch.uint8, device=dev)
    ta.tree_attn_paged(q, i32(w.q_indptr), pages, i32(pk2.page_indptr), page_values,
                       i32(bad), i32(w.mn_indptr), tree_order, out, lse, 0, w.sm_scale, ws)
    st = ta.device_status(ws)
    assert st == ta.TA_ERR_INVALID_ARGUMENT or st != ta.TA_OK
    assert torch.all(out == 7.0)             # nothing computed


@pytest.mark.parametrize("name,seqs", [("degenerate", [1, 3]), ("ragged-large", [0, 1, 2, 63])])
def test_paged_full_size_benchmark_shape(name, seqs):
    """The paged path at a benchmarked full-size shape (the workload ``bench.py
    --paged`` times: every sequence's K/V scattered over 16-slot pages, RoPE
    off as the pages' paged kernel has none), checked against the paged oracle
    on a subset of its sequences (the oracle is too slow for all of them)."""
    import dataclasses
    idx = {"degenerate": 5, "ragged-large": 4}[name]
    w = dataclasses.replace(wl.config(idx), rotary_mode=0)
    pk = wl.paged_from(w, seed=17)
    out, lse = _paged_gpu(w, pk)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(out).all(), "a slot no sequence owns reached the output"
    ro, rl = oracle.tree_attention_paged(w.q, w.q_indptr, pk.pages, pk.page_indptr,
                                         pk.page_values, pk.last_page_len, w.mn_indptr,
                                         w.tree_order, 0, w.sm_scale, seqs=seqs)
    rows = np.concatenate([np.arange(w.q_indptr[b], w.q_indptr[b + 1]) for b in seqs])
    err_o = float(np.max(np.abs(out[rows] - ro[rows])))
    assert err_o <= TOL_OUT[w.dtype], f"out max|err| {err_o}"
    fin = np.isfinite(rl[rows])
    assert np.array_equal(fin, np.isfinite(lse[rows]))
    err_l = float(np.max(np.abs(lse[rows][fin] - rl[rows][fin])))
    assert err_l <= TOL_LSE, f"lse max|err| {err_l}"
