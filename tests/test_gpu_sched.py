"""The two work schedulers of the attention kernel (page "tile_scheduler.py":
the persistent schedulers and ``ClusterLaunchControlScheduler``): the atomic
work queue over one CTA per SM, and cluster launch control (the default)
over one CTA per work unit, where a running CTA takes the units of CTAs whose
launches it cancels.  Every unit is computed by the same code either way, so the results
are equal bit for bit; the cluster-launch-control results are also checked
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import tree_attention_gb300 as ta
import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = {"fp16": 1e-2, "bf16": 2e-2}
DEFAULT = 1   # the library's default scheduler (cluster launch control)
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tree_attention_gb300 import build
    build.build()
    ta.lib()
    yield
    ta.set_scheduler(DEFAULT)


def _one_call(w, d, mode):
    ta.set_scheduler(mode)
    try:
        attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                                w.rope_scale, w.rope_theta, w.sm_scale)
        out, lse = attn(**d)
        st = ta.device_status(attn.workspace)
    finally:
        ta.set_scheduler(DEFAULT)
    assert st == ta.TA_OK, ta.status_string(st)
    return out, lse


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_clc_equals_queue_full_size(idx):
    w = wl.config(idx)
    d = wl.device_inputs(w)
    o0, l0 = _one_call(w, d, 0)
    o1, l1 = _one_call(w, d, 1)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_clc_matches_oracle():
    w = wl.config(3, batch_scale=0.25)
    d = wl.device_inputs(w)
    out, lse = _one_call(w, d, 1)
    ro, rl = oracle.tree_attention_workload(w)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert float(np.max(np.abs(out - ro))) <= TOL_OUT[w.dtype]
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert float(np.max(np.abs(lse[fin] - rl[fin]))) <= TOL_LSE


def test_clc_split_and_paged_paths():
    """tree_attn splitting by itself (few long sequences), and the paged call,
    under cluster launch control: equal to the queue's results."""
    w = wl.long_prefix(batch=2, prefix=6000, nodes=64, seed=12)
    d = wl.device_inputs(w)
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
    assert ta.auto_split_chunks(dims) > 1
    o0, l0 = _one_call(w, d, 0)
    o1, l1 = _one_call(w, d, 1)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)

    import dataclasses
    wp = dataclasses.replace(wl.config(4, batch_scale=0.25), rotary_mode=0)
    pk = wl.paged_from(wp, seed=3)
    dev = "cuda"
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    q = wp.q.contiguous().to(dev)
    pages = pk.pages.contiguous().to(dev)
    tree_order = i32(wp.tree_order.reshape(-1, 2))
    page_values = i32(pk.page_values)
    res = []
    for mode in (0, 1):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        pdims = ta.make_paged_dims(q, pages, i32(wp.q_indptr), page_values, tree_order)
        ws = torch.zeros(ta.paged_workspace_size(pdims), dtype=torch.uint8, device=dev)
        ta.set_scheduler(mode)
        try:
            ta.tree_attn_paged(q, i32(wp.q_indptr), pages, i32(pk.page_indptr), page_values,
                               i32(pk.last_page_len), i32(wp.mn_indptr), tree_order, out, lse, 0,
                               wp.sm_scale, ws)
            st = ta.device_status(ws)
        finally:
            ta.set_scheduler(DEFAULT)
        assert st == ta.TA_OK, ta.status_string(st)
        res.append((out, lse))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_clc_plan_reused_across_runs():
    """tree_attn_plan once, tree_attn_run under the queue, then under cluster
    launch control, then under the queue again: the queue re-arms itself and
    cluster launch control leaves it alone, so all three runs agree."""
    w = wl.config(2, batch_scale=0.5)
    d = wl.device_inputs(w)
    dims = ta.make_dims(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode)
    ws = torch.zeros(ta.workspace_size(dims), dtype=torch.uint8, device="cuda")
    ta.plan(d["q"], d["q_indptr"], d["k"], d["kv_indptr"], d["q_rope_position"],
            d["mn_indptr"], d["tree_order"], w.rotary_mode, w.rope_scale, w.rope_theta, ws)
    res = []
    for mode in (0, 1, 0):
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
        ta.set_scheduler(mode)
        try:
            ta.run(d["q"], d["k"], d["v"], d["q_indptr"], d["kv_indptr"], d["q_rope_position"],
                   d["mn_indptr"], d["tree_order"], out, lse, w.rotary_mode, w.rope_scale,
                   w.rope_theta, w.sm_scale, ws)
            st = ta.device_status(ws)
        finally:
            ta.set_scheduler(DEFAULT)
        assert st == ta.TA_OK, ta.status_string(st)
        res.append((out, lse))
    for o, l in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(l, res[0][1])
