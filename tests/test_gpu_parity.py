"""GPU parity: the sm_103a library, called through its C ABI, against the CPU
oracle on the same seeded inputs.

Bars: the tree mask bit-exact; output max-abs error <= 1e-2 (fp16) and
<= 2e-2 (bf16); LSE (base 2) abs error <= 1e-3; rows with nothing visible give
out = 0 and lse = -inf on both sides.
"""
import zlib

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


def run_gpu(w):
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    out, lse = attn(**d)
    st = ta.device_status(attn.workspace)
    assert st == ta.TA_OK, ta.status_string(st)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def assert_parity(w, out, lse, ref=None):
    ro, rl = ref if ref is not None else oracle.tree_attention_workload(w)
    assert out.shape == ro.shape and lse.shape == rl.shape
    err_o = float(np.max(np.abs(out - ro))) if out.size else 0.0
    assert err_o <= TOL_OUT[w.dtype], f"out max|err| {err_o}"
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), "finite-ness of lse differs"
    assert np.all(lse[~fin] == rl[~fin])
    err_l = float(np.max(np.abs(lse[fin] - rl[fin]))) if fin.any() else 0.0
    assert err_l <= TOL_LSE, f"lse max|err| {err_l}"
    return err_o, err_l


# --------------------------------------------------------------------------
# mask
# --------------------------------------------------------------------------

def _mask_workloads():
    rng = np.random.default_rng(77)
    fams = [wl.chain_tree(150), wl.star_tree(40), wl.binary_tree(63), wl.random_tree(90, rng),
            wl.main_chain_tree(70, rng), wl.spec_decode_tree(64, rng), np.array([-1])]
    prefixes = [0, 5, 130, 0, 17, 0, 3]
    qos = [150, 40, 20, 90, 1, 64, 1]
    return [wl.build_workload("mask", fams, h_q=2, h_kv=1, head_dim=64, dtype="fp16",
                              tensor_seed=1, prefix_lens=prefixes, qo_lens=qos),
            wl.config(1), wl.config(2, batch_scale=0.25), wl.config(3, batch_scale=0.125)]


@pytest.mark.parametrize("idx", range(4))
def test_mask_bit_exact(idx):
    w = _mask_workloads()[idx]
    d = wl.device_inputs(w)
    max_kv = int(np.max(np.diff(w.kv_indptr)))
    vis = ta.mask_dense(d["q_indptr"], d["kv_indptr"], d["mn_indptr"], d["tree_order"],
                        w.total_q, max_kv).cpu().numpy().astype(bool)
    torch.cuda.synchronize()
    for b in range(w.batch_size):
        ref = oracle.visibility(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, b)
        q0, q1 = w.q_indptr[b], w.q_indptr[b + 1]
        kv = w.kv_indptr[b + 1] - w.kv_indptr[b]
        assert np.array_equal(vis[q0:q1, :kv], ref), b
        assert not vis[q0:q1, kv:].any()


# --------------------------------------------------------------------------
# the five benchmark workloads at full size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_config_full_size(idx):
    w = wl.config(idx)
    out, lse = run_gpu(w)
    assert_parity(w, out, lse)


def test_degenerate_chain_equals_causal():
    """The chain sequence of the degenerate workload is causal attention."""
    w = wl.config(5)
    out, lse = run_gpu(w)
    n = len(w.parents[0])
    q = w.q[:n].to(torch.float64).permute(1, 0, 2)
    k = w.k[:n].to(torch.float64).permute(1, 0, 2)
    v = w.v[:n].to(torch.float64).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=w.sm_scale)
    err = np.max(np.abs(out[:n] - ref.permute(1, 0, 2).numpy()))
    assert err <= TOL_OUT["fp16"]


# --------------------------------------------------------------------------
# edge cases: ragged tiles, group sizes, prefixes, partial q sets, empty rows
# --------------------------------------------------------------------------

def _pos(parents, prefixes, base=0):
    return [np.concatenate([np.arange(pf), base + pf + wl.tree_depths(p)])
            for p, pf in zip(parents, prefixes)]


def _edge(name):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    if name == "mha_fp16_multi_tiles":
        ps = [wl.chain_tree(300), wl.random_tree(50, rng)]
        return wl.build_workload(name, ps, h_q=4, h_kv=4, head_dim=128, dtype="fp16",
                                 tensor_seed=1, prefix_lens=[0, 70])
    if name == "g2_d64_rope":
        ps = [wl.random_tree(1, rng), wl.random_tree(7, rng), wl.random_tree(130, rng)]
        pf = [5, 0, 200]
        return wl.build_workload(name, ps, h_q=4, h_kv=2, head_dim=64, dtype="fp16",
                                 tensor_seed=2, prefix_lens=pf, positions=_pos(ps, pf),
                                 rotary_mode=1, rope_theta=1e4)
    if name == "g4_bf16_rope":
        ps = [wl.main_chain_tree(200, rng), wl.star_tree(33)]
        pf = [150, 1]
        return wl.build_workload(name, ps, h_q=8, h_kv=2, head_dim=128, dtype="bf16",
                                 tensor_seed=3, prefix_lens=pf, positions=_pos(ps, pf, 7),
                                 rotary_mode=1, rope_theta=5e5)
    if name == "g8_bf16_rope":
        ps = [wl.random_tree(90, rng), wl.spec_decode_tree(64, rng), wl.binary_tree(31)]
        pf = [0, 0, 64]
        return wl.build_workload(name, ps, h_q=16, h_kv=2, head_dim=128, dtype="bf16",
                                 tensor_seed=4, prefix_lens=pf, positions=_pos(ps, pf),
                                 rotary_mode=1)
    if name == "g16_bf16":
        ps = [wl.random_tree(45, rng), wl.chain_tree(17)]
        return wl.build_workload(name, ps, h_q=32, h_kv=2, head_dim=128, dtype="bf16",
                                 tensor_seed=5, prefix_lens=[9, 0])
    if name == "g3_nonpow2":
        ps = [wl.random_tree(100, rng), wl.random_tree(61, rng)]
        pf = [11, 0]
        return wl.build_workload(name, ps, h_q=6, h_kv=2, head_dim=128, dtype="bf16",
                                 tensor_seed=6, prefix_lens=pf, positions=_pos(ps, pf),
                                 rotary_mode=1)
    if name == "g6_d64":
        ps = [wl.random_tree(70, rng), wl.star_tree(25)]
        return wl.build_workload(name, ps, h_q=12, h_kv=2, head_dim=64, dtype="fp16",
                                 tensor_seed=7, prefix_lens=[0, 40])
    if name == "g128_d64":
        ps = [wl.random_tree(5, rng), wl.chain_tree(3)]
        return wl.build_workload(name, ps, h_q=128, h_kv=1, head_dim=64, dtype="bf16",
                                 tensor_seed=8, prefix_lens=[130, 2])
    if name == "qo_less_than_tree":
        ps = [wl.random_tree(10, rng), wl.random_tree(4, rng), wl.random_tree(150, rng)]
        return wl.build_workload(name, ps, h_q=4, h_kv=1, head_dim=128, dtype="fp16",
                                 tensor_seed=9, prefix_lens=[3, 6, 0], qo_lens=[3, 0, 140])
    if name == "negative_scale":
        ps = [wl.random_tree(40, rng)]
        return wl.build_workload(name, ps, h_q=2, h_kv=1, head_dim=128, dtype="fp16",
                                 tensor_seed=10, prefix_lens=[20], sm_scale=-0.05)
    if name == "single_nodes":
        ps = [np.array([-1])] * 5
        pf = [0, 1, 63, 64, 129]
        return wl.build_workload(name, ps, h_q=8, h_kv=2, head_dim=128, dtype="bf16",
                                 tensor_seed=11, prefix_lens=pf, positions=_pos(ps, pf, 3),
                                 rotary_mode=1)
    if name == "large_positions":
        ps = [wl.random_tree(64, rng)]
        pf = [100]
        return wl.build_workload(name, ps, h_q=4, h_kv=1, head_dim=128, dtype="bf16",
                                 tensor_seed=12, prefix_lens=pf,
                                 positions=_pos(ps, pf, 90000), rotary_mode=1,
                                 rope_scale=0.75, rope_theta=5e5)
    if name == "empty_rows":
        ps = [wl.random_tree(12, rng), wl.random_tree(9, rng)]
        w = wl.build_workload(name, ps, h_q=4, h_kv=2, head_dim=64, dtype="fp16",
                              tensor_seed=13)
        # every interval of the second sequence is empty: its rows see nothing
        w.tree_order = w.tree_order.copy()
        w.tree_order[12:, 1] = w.tree_order[12:, 0]
        return w
    raise KeyError(name)


EDGE = ["mha_fp16_multi_tiles", "g2_d64_rope", "g4_bf16_rope", "g8_bf16_rope", "g16_bf16",
        "g3_nonpow2", "g6_d64", "g128_d64", "qo_less_than_tree", "negative_scale",
        "single_nodes", "large_positions", "empty_rows"]


@pytest.mark.parametrize("name", EDGE)
def test_edge_case(name):
    w = _edge(name)
    out, lse = run_gpu(w)
    assert_parity(w, out, lse)


@pytest.mark.parametrize("g,tree", [(1, "chain"), (1, "random"), (8, "chain"), (8, "random")])
def test_reference_moves_across_chunks(g, tree):
    """Scores that grow along the kv columns: every row's running reference
    (the lazy max of the online softmax) has to move several times within and
    across kv tiles, so the rare path that moves it -- re-forming the chunk's
    P and rescaling the tile's P chunks already written -- runs, and the
    result still matches the oracle."""
    rng = np.random.default_rng(91 + g)
    n = 700
    parents = [wl.chain_tree(n) if tree == "chain" else wl.random_tree(n, rng)]
    w = wl.build_workload(f"ref_moves_{tree}_g{g}", parents, h_q=g, h_kv=1, head_dim=64,
                          dtype="fp16", tensor_seed=5 + g, sm_scale=1.0)
    d = w.head_dim
    # q . k_j = 0.06 j (+ noise): log2-scaled scores rise ~11 per 128 columns
    q = torch.full((w.total_q, w.h_q, d), 1.0 / d ** 0.5)
    ramp = torch.arange(w.total_kv, dtype=torch.float32) * (0.06 / d ** 0.5)
    k = ramp[:, None, None].expand(w.total_kv, 1, d).clone()
    k += 0.05 * torch.randn(w.total_kv, 1, d, generator=torch.Generator().manual_seed(3))
    w.q = q.to(torch.float16)
    w.k = k.to(torch.float16)
    out, lse = run_gpu(w)
    assert_parity(w, out, lse)


def test_repeated_calls_are_bitwise_identical():
    w = wl.config(2, batch_scale=0.5)
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    o1, l1 = attn(**d)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("idx", [5, 2])
def test_many_runs_bitwise_identical(idx):
    """Each output row is computed by one CTA in a fixed order, so results
    must not depend on scheduling: any race between the warps of a CTA shows
    up as a difference (or a bounded-wait timeout) across repeated runs."""
    w = wl.config(idx)
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    o0, l0 = attn(**d)
    o0, l0 = o0.clone(), l0.clone()
    for _ in range(12):
        o, l = attn(**d)
        assert ta.device_status(attn.workspace) == ta.TA_OK
        assert torch.equal(o, o0) and torch.equal(l, l0)


def test_bad_index_arrays_are_reported_not_computed():
    w = wl.config(1)
    d = wl.device_inputs(w)
    d["q_indptr"][-1] += 1                         # no longer ends at total_q
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], 0, 1.0, 1e4,
                            w.sm_scale)
    out = torch.full_like(d["q"], 7.0)
    lse = torch.full(d["q"].shape[:2], 7.0, device="cuda")
    attn(**d, out=out, lse=lse)
    assert ta.device_status(attn.workspace) == ta.TA_ERR_INVALID_ARGUMENT
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    # the status word was cleared by the read
    assert ta.device_status(attn.workspace) == ta.TA_OK


# --------------------------------------------------------------------------
# RoPE table: float32 cos/sin rounded correctly (as the oracle takes them)
# --------------------------------------------------------------------------

def _rope_regions(w, attn):
    """The kv tokens' cos/sin table and the rotated keys: the last two
    regions of a tree_attn workspace with RoPE."""
    def r256(x):
        return (x + 255) // 256 * 256
    half = w.head_dim // 2
    tab_b = w.total_kv * half * 8
    krot_b = w.total_kv * w.h_kv * w.head_dim * 2
    off_krot = attn.workspace.numel() - r256(krot_b)
    off_tab = off_krot - r256(tab_b)
    tab = attn.workspace[off_tab:off_tab + tab_b].cpu().numpy().view(np.float32)
    krot = attn.workspace[off_krot:off_krot + krot_b].cpu().view(w.k.dtype)
    return tab.reshape(-1, half, 2), krot.reshape(w.total_kv, w.h_kv, w.head_dim)


def _run_rope(idx):
    w = wl.config(idx)
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    return w, attn


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_rope_table_matches_correctly_rounded_cos_sin(idx):
    """The per-kv-token cos/sin table (written by the key-rotation kernel,
    read by the attention kernel for its q rows) equals float32-rounded
    cos/sin of the pages' float32 angle; only rare near-ties (true value
    within ~1e-4 ulp of a rounding midpoint) may differ by one ulp."""
    w, attn = _run_rope(idx)
    tab, _ = _rope_regions(w, attn)
    c, s = oracle.rope_cos_sin(w.rope_position, w.head_dim, w.rope_theta, w.rope_scale)
    bad = int(np.sum(tab[..., 0] != c) + np.sum(tab[..., 1] != s))
    assert bad <= max(2, c.size * 2 // 100000), f"{bad} of {2 * c.size} entries differ"
    ulps = np.abs(tab[..., 0].view(np.int32).astype(np.int64) - c.view(np.int32))
    assert ulps.max() <= 1


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_rotated_keys_match_oracle_rope(idx):
    """The key-rotation kernel gives the oracle's ``apply_rope`` of k (the pages' float32 steps, one rounding
    to the storage dtype); a near-tie cos/sin may move an element by one
    storage ulp, rarely."""
    w, attn = _run_rope(idx)
    _, krot = _rope_regions(w, attn)
    ref = oracle.apply_rope(w.k, w.rope_position, w.rope_theta, w.rope_scale)
    diff = krot != ref
    n_bad = int(diff.sum())
    assert n_bad <= max(4, ref.numel() // 100000), f"{n_bad} of {ref.numel()} elements differ"
    if n_bad:
        a = krot[diff].float()
        b = ref[diff].float()
        ulp = 2.0 ** -7 if w.dtype == "bf16" else 2.0 ** -10
        assert bool(((a - b).abs() <= ulp * b.abs().clamp_min(2.0 ** -14) * 1.01).all())


@pytest.mark.parametrize("idx", [2, 3])
def test_plan_once_run_per_layer(idx):
    """tree_attn_plan once, tree_attn_run for two layers with different q/k/v
    on the same plan (the key rotation runs in the run half): each layer
    matches the oracle, and the first equals the one-call tree_attn bit for
    bit (same kernels and arithmetic; the one-call path folds the rotation of
    small problems into its plan kernel)."""
    import dataclasses
    w1 = wl.config(idx, batch_scale=0.25)
    gen = torch.Generator().manual_seed(4321 + idx)
    tdt = w1.q.dtype
    w2 = dataclasses.replace(
        w1, q=torch.randn(w1.q.shape, generator=gen, dtype=torch.float32).to(tdt),
        k=torch.randn(w1.k.shape, generator=gen, dtype=torch.float32).to(tdt),
        v=torch.randn(w1.v.shape, generator=gen, dtype=torch.float32).to(tdt))
    d1, d2 = wl.device_inputs(w1), wl.device_inputs(w2)
    dims = ta.make_dims(d1["q"], d1["k"], d1["q_indptr"], d1["tree_order"], w1.rotary_mode)
    ws = torch.zeros(ta.workspace_size(dims), dtype=torch.uint8, device="cuda")
    ta.plan(d1["q"], d1["q_indptr"], d1["k"], d1["kv_indptr"], d1["q_rope_position"],
            d1["mn_indptr"], d1["tree_order"], w1.rotary_mode, w1.rope_scale, w1.rope_theta, ws)
    outs = []
    for w, d in ((w1, d1), (w2, d2)):
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
        ta.run(d["q"], d["k"], d["v"], d["q_indptr"], d["kv_indptr"], d["q_rope_position"],
               d["mn_indptr"], d["tree_order"], out, lse, w.rotary_mode, w.rope_scale,
               w.rope_theta, w.sm_scale, ws)
        assert ta.device_status(ws) == ta.TA_OK
        assert_parity(w, out.float().cpu().numpy(), lse.cpu().numpy())
        outs.append((out, lse))
    attn = ta.TreeAttention(d1["q"], d1["k"], d1["q_indptr"], d1["tree_order"], w1.rotary_mode,
                            w1.rope_scale, w1.rope_theta, w1.sm_scale)
    out1, lse1 = attn(**d1)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    if ta.auto_split_chunks(dims) == 1:
        assert torch.equal(out1, outs[0][0]) and torch.equal(lse1, outs[0][1])
    else:
        # the one-call path split this batch of few long sequences: the same
        # states merged, equal up to float32 rounding order
        assert torch.allclose(lse1, outs[0][1], rtol=0, atol=1e-4)
        assert torch.allclose(out1.float(), outs[0][0].float(), rtol=0, atol=1e-2)
