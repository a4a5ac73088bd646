"""GPU parity of split-KV tree attention and of the attention-state merge,
called through the C ABI, against the CPU oracle on seeded inputs.

Split-KV cuts the kv tiles of a (sequence, q tile) pair into chunks that run
as separate work items; a merge kernel combines the chunks' float32 partial
states with the base-2 log-sum-exp rule (``merge_states`` of the oracle,
resting on the ``lse_store`` epilogue of the page "tree_attn.py").  The bars
are those of the unsplit path: output max-abs error <= 1e-2 (fp16) /
2e-2 (bf16), base-2 LSE error <= 1e-3.  The chunk parameters are swept down to
one kv tile per chunk, which leaves chunks with no visible column at all
(lse = -inf parts) in the sparse trees.
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
    rng = np.random.default_rng(41)
    return {
        "tiny": wl.config(1),
        "spec-decode/4": wl.config(2, batch_scale=0.125),
        "prefix+tree/4": wl.config(3, batch_scale=0.25),
        # ragged prefix (not a tile multiple), g = 4, RoPE
        "long-prefix-4000": wl.long_prefix(batch=2, prefix=4000, nodes=64, seed=8),
        # sparse trees (many empty tiles), MHA fp16, no RoPE
        "star_chain_fp16": wl.build_workload(
            "sc", [wl.star_tree(700), wl.chain_tree(300), wl.binary_tree(255)], h_q=4, h_kv=4,
            head_dim=128, dtype="fp16", tensor_seed=3, prefix_lens=[0, 150, 64]),
        # g = 8, d = 64, uneven prefixes
        "g8_d64": wl.build_workload(
            "g8", [wl.random_tree(33, rng), wl.random_tree(90, rng)], h_q=64, h_kv=8,
            head_dim=64, dtype="bf16", tensor_seed=11, prefix_lens=[1517, 250]),
    }


def run_split(w, max_chunks, chunk_tiles, ws=None):
    d = wl.device_inputs(w)
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
    if ws is None:
        n = ta.split_workspace_size(dims, max_chunks)
        assert n > 0
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    ta.tree_attn_split(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"],
                       d["q_rope_position"], d["mn_indptr"], d["tree_order"], out, lse,
                       w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale, max_chunks,
                       chunk_tiles, ws)
    st = ta.device_status(ws)
    assert st == ta.TA_OK, ta.status_string(st)
    return out, lse, ws


def run_plain(w):
    """The unsplit kernel: the plan / run entry points, which never split (the
    one-call tree_attn may split long sequences by itself)."""
    d = wl.device_inputs(w)
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
    ws = torch.zeros(ta.workspace_size(dims), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    ta.plan(d["q"], d["q_indptr"], d["k"], d["kv_indptr"], d["q_rope_position"],
            d["mn_indptr"], d["tree_order"], w.rotary_mode, w.rope_scale, w.rope_theta, ws)
    ta.run(d["q"], d["k"], d["v"], d["q_indptr"], d["kv_indptr"], d["q_rope_position"],
           d["mn_indptr"], d["tree_order"], out, lse, w.rotary_mode, w.rope_scale,
           w.rope_theta, w.sm_scale, ws)
    assert ta.device_status(ws) == ta.TA_OK
    return out, lse


def assert_parity(w, out, lse, ref, rows=None):
    ro, rl = ref
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    if rows is not None:
        out, lse, ro, rl = out[rows], lse[rows], ro[rows], rl[rows]
    err_o = float(np.max(np.abs(out - ro))) if out.size else 0.0
    assert err_o <= TOL_OUT[w.dtype], f"out max|err| {err_o}"
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), "finite-ness of lse differs"
    err_l = float(np.max(np.abs(lse[fin] - rl[fin]))) if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"lse max|err| {err_l}"


_REF = {}


def _ref(name):
    if name not in _REF:
        _REF[name] = oracle.tree_attention_workload(_workloads()[name])
    return _REF[name]


@pytest.mark.parametrize("name", list(_workloads()))
@pytest.mark.parametrize("max_chunks,chunk_tiles", [(16, 0), (4, 1), (16, 3), (2, 5), (16, 1)])
def test_split_matches_oracle(name, max_chunks, chunk_tiles):
    w = _workloads()[name]
    out, lse, _ = run_split(w, max_chunks, chunk_tiles)
    assert_parity(w, out, lse, _ref(name))


@pytest.mark.parametrize("name", ["spec-decode/4", "long-prefix-4000", "star_chain_fp16"])
def test_one_chunk_is_the_unsplit_kernel_bit_for_bit(name):
    w = _workloads()[name]
    out_s, lse_s, _ = run_split(w, 1, 0)
    out_p, lse_p = run_plain(w)
    assert torch.equal(out_s, out_p)
    assert torch.equal(lse_s, lse_p)


@pytest.mark.parametrize("name", ["long-prefix-4000", "g8_d64"])
def test_split_agrees_with_unsplit(name):
    """Split and unsplit differ only in float32 rounding order: the lse to
    float32 accuracy, the output to one rounding of the storage dtype."""
    w = _workloads()[name]
    out_s, lse_s, _ = run_split(w, 16, 2)
    out_p, lse_p = run_plain(w)
    assert float((lse_s - lse_p).abs().max()) <= 1e-4
    ulp = 2.0 ** -7 if w.dtype == "bf16" else 2.0 ** -10
    tol = ulp * max(1.0, float(out_p.float().abs().max()))
    assert float((out_s.float() - out_p.float()).abs().max()) <= tol


def test_split_repeated_calls_bitwise_identical():
    """One workspace serves many calls (the work queue re-arms itself) and the
    merge order is fixed, so results repeat bit for bit."""
    w = _workloads()["long-prefix-4000"]
    out1, lse1, ws = run_split(w, 16, 0)
    for _ in range(3):
        out2, lse2, _ = run_split(w, 16, 0, ws=ws)
        assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_split_long_prefix_full_size():
    """The 32768-token-prefix workload of the split benchmark, in its
    benchmark launch (automatic chunk length), against the oracle on two of
    its four sequences."""
    w = wl.long_prefix()
    out, lse, _ = run_split(w, 16, 0)
    seqs = [0, 3]
    ref = oracle.tree_attention(w.q, w.q_indptr, w.k, w.v, w.kv_indptr, w.rope_position,
                                w.mn_indptr, w.tree_order, w.rotary_mode, w.rope_scale,
                                w.rope_theta, w.sm_scale, seqs=seqs)
    rows = np.concatenate([np.arange(w.q_indptr[b], w.q_indptr[b + 1]) for b in seqs])
    assert_parity(w, out, lse, ref, rows=rows)


def test_one_call_splits_long_prefix_by_itself():
    """tree_attn on the long-prefix workload (4 sequences, 32768-token
    prefixes: 32 units for 8 kv heads, far fewer than the SMs) chooses
    split-KV itself, matches the oracle on two of its four sequences, and
    agrees with tree_attn_split at the same cap bit for bit."""
    w = wl.long_prefix()
    d = wl.device_inputs(w)
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
    cap = ta.auto_split_chunks(dims)
    assert cap > 1
    assert ta.workspace_size(dims) == ta.split_workspace_size(dims, cap)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    out, lse = attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    seqs = [1, 2]
    ref = oracle.tree_attention(w.q, w.q_indptr, w.k, w.v, w.kv_indptr, w.rope_position,
                                w.mn_indptr, w.tree_order, w.rotary_mode, w.rope_scale,
                                w.rope_theta, w.sm_scale, seqs=seqs)
    rows = np.concatenate([np.arange(w.q_indptr[b], w.q_indptr[b + 1]) for b in seqs])
    assert_parity(w, out, lse, ref, rows=rows)
    out_s, lse_s, _ = run_split(w, cap, 0)
    assert torch.equal(out, out_s) and torch.equal(lse, lse_s)


def test_one_call_does_not_split_the_benchmark_workloads():
    """Configs 2-5 give every SM work without a split: tree_attn keeps them
    in one pass."""
    for idx in (2, 3, 4, 5):
        w = wl.config(idx)
        d = wl.device_inputs(w)
        dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
        assert ta.auto_split_chunks(dims) == 1, w.name


def test_split_bad_index_arrays_are_reported():
    w = _workloads()["tiny"]
    d = wl.device_inputs(w)
    d["kv_indptr"][-1] += 1                  # no longer ends at total_kv
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], 0)
    ws = torch.zeros(ta.split_workspace_size(dims, 4), dtype=torch.uint8, device="cuda")
    out = torch.full_like(d["q"], 7.0)
    lse = torch.full(d["q"].shape[:2], 7.0, dtype=torch.float32, device="cuda")
    ta.tree_attn_split(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"], None,
                       d["mn_indptr"], d["tree_order"], out, lse, 0, 1.0, 1e4, w.sm_scale, 4, 1,
                       ws)
    assert ta.device_status(ws) == ta.TA_ERR_INVALID_ARGUMENT
    # nothing was computed: the outputs keep their fill
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())


# --------------------------------------------------------------------------
# stand-alone merge of attention states
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,d,n", [("bf16", 128, 3), ("fp16", 64, 7), ("bf16", 64, 1),
                                       ("fp16", 128, 40)])
def test_merge_states_matches_oracle(dtype, d, n):
    rng = np.random.default_rng(100 + n)
    rows, heads = 97, 8
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    parts = torch.from_numpy(rng.standard_normal((n, rows, heads, d))).to(tdt)
    lses = rng.normal(0.0, 4.0, size=(n, rows, heads)).astype(np.float32)
    lses[rng.random((n, rows, heads)) < 0.2] = -np.inf     # parts with nothing visible
    lses[:, 5, :] = -np.inf                                # rows with nothing visible at all
    lses[:, 6, 0] = 300.0                                  # large but equal lses
    ro, rl = oracle.merge_states(parts.double().numpy(), lses.astype(np.float64))
    out, lse = ta.merge_states(parts.cuda(), torch.from_numpy(lses).cuda())
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert float(np.max(np.abs(out - ro))) <= TOL_OUT[dtype]
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.all(lse[~fin] == -np.inf) and np.all(out[~fin] == 0.0)
    assert float(np.max(np.abs(lse[fin] - rl[fin]))) <= 1e-4


def test_merge_of_disjoint_tree_attentions_is_the_whole():
    """The oracle's attention states over three disjoint column sets of one
    workload (columns by index mod 3, the others masked out), rounded to bf16
    and merged by the library, give the oracle's state over all columns."""
    w = wl.long_prefix(batch=2, prefix=1000, nodes=64, seed=9)
    ref_o, ref_l = oracle.tree_attention_workload(w)
    # three disjoint column sets by column index mod 3, each attended in the
    # oracle with the other columns masked out
    parts_o, parts_l = [], []
    orig = oracle.tree_attn_ref.visibility
    for r in range(3):
        def vis_r(q_indptr, kv_indptr, mn_indptr, tree_order, b, _r=r):
            v = orig(q_indptr, kv_indptr, mn_indptr, tree_order, b).copy()
            v[:, np.arange(v.shape[1]) % 3 != _r] = False
            return v
        oracle.tree_attn_ref.visibility = vis_r
        try:
            o, l = oracle.tree_attention_workload(w)
        finally:
            oracle.tree_attn_ref.visibility = orig
        parts_o.append(o)
        parts_l.append(l)
    pt = torch.from_numpy(np.stack(parts_o)).to(torch.bfloat16).cuda()
    pl = torch.from_numpy(np.stack(parts_l).astype(np.float32)).cuda()
    out, lse = ta.merge_states(pt, pl)
    torch.cuda.synchronize()
    assert float(np.max(np.abs(out.float().cpu().numpy() - ref_o))) <= TOL_OUT["bf16"]
    assert float(np.max(np.abs(lse.cpu().numpy() - ref_l))) <= TOL_LSE
