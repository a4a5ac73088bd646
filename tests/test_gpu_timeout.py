"""The failure detection of the attention kernel: every hand-off between its
warps is an mbarrier wait bounded by a wall-clock limit; when one runs out the
kernel records a timeout in the workspace status word, lets its in-flight
copies and tensor-core operations land, frees its tensor memory and returns.

The test makes a wait run out on purpose through the library's test hooks (a
short limit, and an MMA thread that first waits on a barrier nothing arrives
on), checks that the call returns with TA_ERR_DEVICE_TIMEOUT reported, and that
the next call on the same workspace, with the normal limit, is correct.  The
pages' own checks are compile-time asserts (``check_thread_limits``, page
"_kernel_common.py"); this detection is the library's own.
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


def _check(w, out, lse):
    ro, rl = oracle.tree_attention_workload(w)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.max(np.abs(o - ro)) <= TOL_OUT[w.dtype]
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.max(np.abs(l[fin] - rl[fin])) <= TOL_LSE


@pytest.mark.parametrize("idx,scale", [(1, 1.0), (2, 0.25), (5, 0.01)])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(idx, scale):
    w = wl.config(idx, batch_scale=scale) if scale != 1.0 else wl.config(idx)
    d = wl.device_inputs(w)
    attn = ta.TreeAttention(d["q"], d["k"], d["q_indptr"], d["tree_order"], w.rotary_mode,
                            w.rope_scale, w.rope_theta, w.sm_scale)
    out = torch.full_like(d["q"], 7.0)
    lse = torch.full(d["q"].shape[:2], 7.0, dtype=torch.float32, device="cuda")
    ta.set_wait_hooks(50_000, stall=True)          # 50 us, MMA threads stall
    try:
        attn(**d, out=out, lse=lse)
        st = ta.device_status(attn.workspace)
    finally:
        ta.set_wait_hooks(0, stall=False)
    assert st == ta.TA_ERR_DEVICE_TIMEOUT, ta.status_string(st)
    # nothing reached the outputs: no PV ran, so no output row was written
    assert torch.all(out == 7.0)
    # the read cleared the status word
    assert ta.device_status(attn.workspace) == ta.TA_OK
    # the same workspace serves the next call with the normal limit
    out2, lse2 = attn(**d)
    assert ta.device_status(attn.workspace) == ta.TA_OK
    _check(w, out2, lse2)
