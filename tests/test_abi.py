"""CPU tests of the C-ABI library: it builds for sm_103a, loads without a
GPU, exports every symbol include/tree_attn.h declares, and rejects bad
arguments on the host before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

import tree_attention_gb300 as ta
import workloads as wl
from tree_attention_gb300 import build as ta_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "tree_attn.h")


@pytest.fixture(scope="module")
def lib():
    ta_build.build()
    return ta.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tree_attn\w*)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tree_attn", "tree_attn_workspace_size", "tree_attn_device_status",
              "tree_attn_status_string", "tree_attn_mask_dense", "tree_attn_check_inputs"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert ta.status_string(ta.TA_OK) == "TA_OK"
    assert ta.status_string(ta.TA_ERR_DEVICE_TIMEOUT) == "TA_ERR_DEVICE_TIMEOUT"


def _dims(**kw):
    d = dict(batch_size=2, total_q=19, total_kv=19, total_tree=19, h_q=4, h_kv=2, head_dim=64,
             dtype=ta.TA_FP16)
    d.update(kw)
    return ta.Dims(**d)


def test_workspace_size(lib):
    n = ta.workspace_size(_dims())
    assert n > 0 and n % 256 == 0
    # grows with the problem, rejects what is not supported
    assert ta.workspace_size(_dims(total_q=4096, total_kv=4096, total_tree=4096)) > n
    assert ta.workspace_size(_dims(head_dim=96)) == 0
    assert ta.workspace_size(_dims(h_q=5)) == 0
    assert ta.workspace_size(_dims(h_q=256, h_kv=1)) == 0      # group size > 128
    assert ta.workspace_size(_dims(batch_size=0)) == 0


def _call(lib, dims, ptrs=None, **kw):
    """tree_attn with fake (never dereferenced) device pointers."""
    fake = ctypes.c_void_p(0x10000)
    args = dict(q=fake, q_indptr=fake, k=fake, v=fake, kv_indptr=fake, pos=fake, mn=fake,
                order=fake, out=fake, lse=fake, rotary=0, rs=1.0, rt=1e4, sm=0.125,
                ws=ctypes.c_void_p(0x20000), wsb=1 << 30)
    args.update(kw)
    return lib.tree_attn(args["q"], args["q_indptr"], args["k"], args["v"], args["kv_indptr"],
                         args["pos"], args["mn"], args["order"], args["out"], args["lse"],
                         args["rotary"], args["rs"], args["rt"], args["sm"], ctypes.byref(dims),
                         args["ws"], args["wsb"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(q_indptr=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(ws=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rotary=2), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rotary=1, pos=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rotary=1, rt=0.0), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(sm=float("nan")), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(sm=float("inf")), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(wsb=16), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(ws=ctypes.c_void_p(0x20010)), ta.TA_ERR_INVALID_ARGUMENT),   # not 256-aligned
    (dict(q=ctypes.c_void_p(0x10008)), ta.TA_ERR_INVALID_ARGUMENT),    # not 16-aligned
])
def test_host_validation_rejects_before_launch(lib, kw, expect):
    assert _call(lib, _dims(), **kw) == expect


def test_unsupported_shapes(lib):
    assert _call(lib, _dims(head_dim=96)) == ta.TA_ERR_UNSUPPORTED
    assert _call(lib, _dims(h_q=256, h_kv=1)) == ta.TA_ERR_UNSUPPORTED
    assert _call(lib, _dims(h_q=5)) == ta.TA_ERR_INVALID_ARGUMENT
    assert _call(lib, _dims(dtype=7)) == ta.TA_ERR_INVALID_ARGUMENT


def test_empty_problem_is_a_no_op(lib):
    assert _call(lib, _dims(total_q=0)) == ta.TA_OK


def test_check_inputs_accepts_generated_workloads(lib):
    for idx in (1, 2, 3):
        w = wl.config(idx, batch_scale=0.25)
        dims = ta.Dims(batch_size=w.batch_size, total_q=w.total_q, total_kv=w.total_kv,
                       total_tree=w.total_tree, h_q=w.h_q, h_kv=w.h_kv, head_dim=w.head_dim,
                       dtype=ta.TA_BF16)
        assert ta.check_inputs(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, dims) == ta.TA_OK


def test_check_inputs_rejects_bad_tables(lib):
    rng = np.random.default_rng(0)
    w = wl.build_workload("t", [wl.random_tree(9, rng), wl.binary_tree(6)], h_q=2, h_kv=1,
                          head_dim=64, dtype="fp16", tensor_seed=0, prefix_lens=[3, 0])
    dims = ta.Dims(batch_size=2, total_q=w.total_q, total_kv=w.total_kv, total_tree=w.total_tree,
                   h_q=2, h_kv=1, head_dim=64, dtype=ta.TA_FP16)
    ok = ta.check_inputs(w.q_indptr, w.kv_indptr, w.mn_indptr, w.tree_order, dims)
    assert ok == ta.TA_OK
    bad = w.q_indptr.copy(); bad[-1] += 1
    assert ta.check_inputs(bad, w.kv_indptr, w.mn_indptr, w.tree_order, dims) != ta.TA_OK
    bad = w.kv_indptr.copy(); bad[1] -= 4          # kv < T in sequence 0
    assert ta.check_inputs(w.q_indptr, bad, w.mn_indptr, w.tree_order, dims) != ta.TA_OK
    order = w.tree_order.copy(); order[1, 1] = order[1, 0]   # empty interval
    assert ta.check_inputs(w.q_indptr, w.kv_indptr, w.mn_indptr, order, dims) != ta.TA_OK
    order = w.tree_order.copy(); order[1] = (1, 9); order[2] = (2, 11)  # crossing intervals
    assert ta.check_inputs(w.q_indptr, w.kv_indptr, w.mn_indptr, order, dims) != ta.TA_OK


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The binding never imports the oracle and has no CPU path."""
    pkg = os.path.dirname(ta.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(root, f)).read()
                assert "oracle" not in src.replace("oracle/", ""), f


# --------------------------------------------------------------------------
# paged KV cache entry point: host-side validation (no launch)
# --------------------------------------------------------------------------

def _pdims(**kw):
    d = dict(batch_size=2, total_q=40, total_tree=40, h_q=8, h_kv=2, head_dim=128,
             dtype=ta.TA_BF16, num_pages=12, nnz_pages=6)
    d.update(kw)
    return ta.PagedDims(**d)


def _call_paged(lib, dims, **kw):
    """tree_attn_paged with fake (never dereferenced) device pointers."""
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, q_indptr=fake, pages=fake, page_indptr=fake, page_values=fake,
             length_info=fake, mn=fake, order=fake, out=fake, lse=fake, rotary=0, sm=0.125,
             ws=ctypes.c_void_p(0x20000), wsb=1 << 30)
    a.update(kw)
    return lib.tree_attn_paged(a["q"], a["q_indptr"], a["pages"], a["page_indptr"],
                               a["page_values"], a["length_info"], a["mn"], a["order"], a["out"],
                               a["lse"], a["rotary"], a["sm"], ctypes.byref(dims), a["ws"],
                               a["wsb"], None)


def test_paged_workspace_size(lib):
    n = ta.paged_workspace_size(_pdims())
    assert n > 0 and n % 256 == 0
    # the same layout as the contiguous call with nnz_pages * 16 kv rows
    assert n == ta.workspace_size(_dims(total_q=40, total_kv=6 * 16, total_tree=40, h_q=8,
                                        h_kv=2, head_dim=128, dtype=ta.TA_BF16))
    assert ta.paged_workspace_size(_pdims(num_pages=0)) == 0
    assert ta.paged_workspace_size(_pdims(head_dim=96)) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(rotary=1), ta.TA_ERR_UNSUPPORTED),            # the pages assert: no RoPE here
    (dict(page_indptr=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(length_info=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(page_values=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(pages=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(pages=ctypes.c_void_p(0x10008)), ta.TA_ERR_INVALID_ARGUMENT),   # not 16-aligned
    (dict(sm=float("nan")), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(wsb=16), ta.TA_ERR_INVALID_ARGUMENT),
])
def test_paged_host_validation_rejects_before_launch(lib, kw, expect):
    assert _call_paged(lib, _pdims(), **kw) == expect


def test_paged_bad_dims(lib):
    assert _call_paged(lib, _pdims(num_pages=0)) == ta.TA_ERR_INVALID_ARGUMENT
    assert _call_paged(lib, _pdims(head_dim=96)) == ta.TA_ERR_UNSUPPORTED
    assert _call_paged(lib, _pdims(total_q=0)) == ta.TA_OK


# --------------------------------------------------------------------------
# split-KV and the stand-alone state merge: host-side validation (no launch)
# --------------------------------------------------------------------------

def _round256(x):
    return (x + 255) // 256 * 256


def test_split_workspace_size(lib):
    d = _dims()
    plain = ta.workspace_size(d)
    # one chunk per pair is the unsplit layout
    assert ta.split_workspace_size(d, 1) == plain
    # g = 2 -> 64 q rows per Q tile, 128 per work unit of two tiles: 1 + 2
    # pairs at most; per record an h_kv x (2 x 128) x d float32 partial output
    # and its lse, plus the merge table
    max_pairs = (19 + 127) // 128 + 2
    for mc in (2, 7, 16):
        recs = max_pairs * mc
        extra = (_round256(recs * 64) - _round256(max_pairs * 64) + _round256(max_pairs * 16)
                 + _round256(recs * 2 * 256 * 64 * 4) + _round256(recs * 2 * 256 * 4))
        assert ta.split_workspace_size(d, mc) == plain + extra
    assert ta.split_workspace_size(d, 0) == 0
    assert ta.split_workspace_size(d, ta.MAX_CHUNKS + 1) == 0
    assert ta.split_workspace_size(_dims(head_dim=96), 4) == 0


def _call_split(lib, dims, max_chunks=4, chunk_tiles=0, **kw):
    fake = ctypes.c_void_p(0x10000)
    a = dict(q=fake, q_indptr=fake, k=fake, v=fake, kv_indptr=fake, pos=fake, mn=fake,
             order=fake, out=fake, lse=fake, rotary=0, rs=1.0, rt=1e4, sm=0.125,
             ws=ctypes.c_void_p(0x20000), wsb=1 << 30)
    a.update(kw)
    return lib.tree_attn_split(a["q"], a["q_indptr"], a["k"], a["v"], a["kv_indptr"], a["pos"],
                               a["mn"], a["order"], a["out"], a["lse"], a["rotary"], a["rs"],
                               a["rt"], a["sm"], max_chunks, chunk_tiles, ctypes.byref(dims),
                               a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(max_chunks=0), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(max_chunks=17), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(chunk_tiles=-1), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(q=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(ws=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rotary=1, pos=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(sm=float("nan")), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(ws=ctypes.c_void_p(0x20010)), ta.TA_ERR_INVALID_ARGUMENT),
])
def test_split_host_validation_rejects_before_launch(lib, kw, expect):
    assert _call_split(lib, _dims(), **kw) == expect


def test_split_workspace_must_hold_the_partial_states(lib):
    d = _dims()
    need = ta.split_workspace_size(d, 8)
    assert _call_split(lib, d, max_chunks=8, wsb=need - 256) == ta.TA_ERR_INVALID_ARGUMENT
    assert _call_split(lib, _dims(total_q=0), max_chunks=8, wsb=need) == ta.TA_OK
    assert _call_split(lib, _dims(head_dim=96)) == ta.TA_ERR_UNSUPPORTED


def _call_merge(lib, n=2, rows=10, d=128, dtype=ta.TA_BF16, **kw):
    fake = ctypes.c_void_p(0x10000)
    a = dict(parts=fake, lses=fake, out=fake, lse=fake)
    a.update(kw)
    return lib.tree_attn_merge_states(a["parts"], a["lses"], n, rows, d, dtype, a["out"],
                                      a["lse"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(n=0), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rows=-1), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(dtype=5), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(d=96), ta.TA_ERR_UNSUPPORTED),
    (dict(parts=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(lse=None), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(out=ctypes.c_void_p(0x10004)), ta.TA_ERR_INVALID_ARGUMENT),
    (dict(rows=0, parts=None), ta.TA_OK),
])
def test_merge_states_host_validation(lib, kw, expect):
    assert _call_merge(lib, **kw) == expect


def test_last_cuda_error_names_the_failure(lib):
    """A launching call that fails in CUDA returns TA_ERR_CUDA and leaves the
    CUDA error's text for tree_attn_last_cuda_error (here: no device).  The
    binding's exception carries it."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (the call would launch)")
    fake = ctypes.c_void_p(0x10000)
    st = lib.tree_attn_merge_states(fake, fake, 2, 10, 128, ta.TA_BF16, fake, fake, None)
    assert st == ta.TA_ERR_CUDA
    msg = ta.last_cuda_error()
    assert msg and msg != "no error"
    err = ta.TreeAttnError(st, "tree_attn_merge_states")
    assert msg in str(err)


def test_wait_hooks_validate_and_reset(lib):
    """The test hooks of the failure detection are host-only settings."""
    assert lib.tree_attn_set_wait_hooks(0, 2) == ta.TA_ERR_INVALID_ARGUMENT
    assert lib.tree_attn_set_wait_hooks(1000, 1) == ta.TA_OK
    assert lib.tree_attn_set_wait_hooks(0, 0) == ta.TA_OK


def test_auto_split_chunks(lib):
    """The one-call entry point's split-KV choice is a host function of the
    dims (and the device's SM count): invalid dims give 0, a batch with many
    short work units never splits, and the workspace it asks for is the split
    workspace at that cap."""
    assert ta.auto_split_chunks(_dims(h_kv=3)) == 0          # h_q % h_kv != 0
    small = _dims()
    assert ta.auto_split_chunks(small) == 1
    assert ta.workspace_size(small) == ta.split_workspace_size(small, 1)
    # 4096 sequences of 64 q rows: at least 4096 x h_kv units, never split
    many = _dims(batch_size=4096, total_q=4096 * 64, total_kv=4096 * 4096,
                 total_tree=4096 * 64)
    assert ta.auto_split_chunks(many) == 1
    # a few long sequences: split on a GPU, unsplit (no device) otherwise
    few = _dims(batch_size=4, total_q=256, total_kv=4 * 32832, total_tree=256)
    cap = ta.auto_split_chunks(few)
    assert 1 <= cap <= ta.MAX_CHUNKS
    assert ta.workspace_size(few) == ta.split_workspace_size(few, cap)


def test_scheduler_setting_validates(lib):
    """The scheduler choice is a host setting of the calling thread."""
    assert lib.tree_attn_set_scheduler(2) == ta.TA_ERR_INVALID_ARGUMENT
    assert lib.tree_attn_set_scheduler(-1) == ta.TA_ERR_INVALID_ARGUMENT
    assert lib.tree_attn_set_scheduler(0) == ta.TA_OK
    assert lib.tree_attn_set_scheduler(1) == ta.TA_OK   # the default again
