"""tree_attn_noalloc: the entry point for callers that may not allocate device
memory (an engine that gave all free HBM to its own pool, or a framework
whose plugins may not call allocators).  It runs the same kernels as
tree_attn on a static device scratch array, which every call shares and
which keeps the previous call's contents; it must still give tree_attn's
results call after call.
"""
import ctypes

import numpy as np
import pytest
import torch

import tree_attention_gb300 as ta
import workloads as wl

TOL_OUT = {"fp16": 1e-2, "bf16": 2e-2}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from tree_attention_gb300 import build
    build.build()
    ta.lib()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    """Checked on the host before anything is enqueued (no GPU needed)."""
    big = ta.Dims(batch_size=1, total_q=64, total_kv=200_000, total_tree=64, h_q=8, h_kv=8,
                  head_dim=128, dtype=ta.TA_BF16, rotary_mode=1)
    assert ta.workspace_size(big) > 32 << 20
    fake = ctypes.c_void_p(0x10000)
    st = ta.lib().tree_attn_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                    1, 1.0, 1e4, 0.1, ctypes.byref(big), None)
    assert st == ta.TA_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("idx", [2, 1])
def test_noalloc_matches_tree_attn_on_two_calls_in_a_row(idx):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = wl.config(idx)
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    ref_out, ref_lse = attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        ta.tree_attn_noalloc(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"],
                             d["q_rope_position"], d["mn_indptr"], d["tree_order"], out, lse,
                             w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(l).all()
        assert np.max(np.abs(o - ref_out)) <= TOL_OUT[w.dtype]
        assert np.max(np.abs(l - ref_lse)) <= TOL_LSE
        assert ta.noalloc_device_status() == ta.TA_OK


@pytest.mark.gpu
def test_noalloc_reports_bad_index_arrays_then_recovers():
    """The status word lives in the static array, which the caller cannot
    address: tree_attn_noalloc_device_status reads and clears it.  Index
    arrays that break the layout rules are reported and nothing is computed;
    the next valid call reports TA_OK."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = wl.config(1)
    d = wl.device_inputs(w)
    assert ta.noalloc_device_status() == ta.TA_OK
    bad = dict(d)
    bad["q_indptr"] = d["q_indptr"].clone()
    bad["q_indptr"][-1] += 1                       # no longer ends at total_q
    out = torch.full_like(d["q"], 7.0)
    lse = torch.full(d["q"].shape[:2], 7.0, dtype=torch.float32, device="cuda")
    ta.tree_attn_noalloc(bad["q"], bad["q_indptr"], bad["k"], bad["v"], bad["kv_indptr"],
                         bad["q_rope_position"], bad["mn_indptr"], bad["tree_order"], out, lse,
                         w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale)
    assert ta.noalloc_device_status() == ta.TA_ERR_INVALID_ARGUMENT
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    ta.tree_attn_noalloc(d["q"], d["q_indptr"], d["k"], d["v"], d["kv_indptr"],
                         d["q_rope_position"], d["mn_indptr"], d["tree_order"], out, lse,
                         w.rotary_mode, w.rope_scale, w.rope_theta, w.sm_scale)
    assert ta.noalloc_device_status() == ta.TA_OK
    assert np.isfinite(out.float().cpu().numpy()).all()
