"""CPU oracle for batched tree attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``tree_attention_gb300``) never imports it and shares no code
with it; the two meet only in the seeded input generators of ``workloads``.

The oracle restates, in plain numpy, what the page "tree_attn.py"
(python/tvm/relax/frontend/nn/llm/tree_attn.py) computes in its sequential
``tree_attn_cpu`` kernel, with the tree mask of ``_check_tree_order`` and the
rotary embedding of ``_rope`` from the page "_kernel_common.py"
(python/tvm/relax/frontend/nn/llm/_kernel_common.py).
"""
from .tree_attn_ref import (  # noqa: F401
    rope_inv_freq_denominators, rope_cos_sin, apply_rope, visibility, tree_attention,
    tree_attention_workload, paged_kv_lengths, tree_attention_paged, PAGE_SIZE, merge_states,
)
