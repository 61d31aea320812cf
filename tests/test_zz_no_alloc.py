"""The allocation-free entry point, tree_attn_run_static().

Some callers may not allocate device memory (an engine plug-in whose host
owns all GPU memory, a serving loop with a fixed memory budget).  For them the
library runs a plan out of one fixed scratch array and can be driven by a
host-only plan, so nothing on the GPU is allocated by planning or running.
These tests call it through the C ABI and compare with the fp64 oracle under
the parity tolerances: two calls in a row with different plans (the shared
scratch must be refilled correctly each time), with the separate and the
fused merge (whose arrival counters each call must clear), and after a call
whose kernel gave up on a wait (the next call must start clean).  A plan too
large for the scratch must be refused.  The file is collected last so a
failure here never hides the other tests.
"""
import pytest
import torch

import workloads as W
from parity_utils import compare, make_inputs, oracle_on_tokens

pytestmark = pytest.mark.gpu


def _static(plan, spec, q, k, v):
    import tree_structured_decode_gb300 as ta

    out = torch.full((spec.n_queries, spec.n_q_heads, spec.head_dim), float("nan"),
                     dtype=torch.float32, device="cuda")
    lse = torch.full((spec.n_queries, spec.n_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    st = plan.run_static(q, k, v, out, lse)
    assert st == 0, ta.load_library().tree_attn_last_error()
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_static_entry_point_matches_the_oracle_on_two_calls_in_a_row(merge_mode):
    import tree_structured_decode_gb300 as ta

    specs = [W.config_tiny(), W.random_tree(77, n_nodes=30, max_len=300, hq=8, hkv=2, d=128,
                                            max_queries_per_node=3),
             # leaves of 4 tokens x GQA 16: 64-row tiles held by kv-head pairs
             W.two_level(300, 6, 90, 64, 4, 128, seed=21, tokens_per_leaf=4)]
    data = [make_inputs(s, tail_fill=float("nan")) for s in specs]
    refs = [oracle_on_tokens(s, *d, list(range(s.n_queries))) for s, d in zip(specs, data)]
    plans = [ta.Plan.from_spec(s, host_only=1, split_tokens=128, merge_mode=merge_mode)
             for s in specs]
    try:
        assert any(p.stats()["n_merge_tokens"] > 0 for p in plans)
        for _ in range(2):  # second round: the scratch holds the other plan's tables
            for spec, (q, k, v), (ro, rl), plan in zip(specs, data, refs, plans):
                out, lse = _static(plan, spec, q, k, v)
                compare(out, lse, ro, rl)
    finally:
        for p in plans:
            p.close()


def test_static_entry_point_recovers_after_a_wait_ran_out():
    import tree_structured_decode_gb300 as ta

    spec = W.two_level(2048, 8, 100, 16, 4, 128, seed=9)
    q, k, v = make_inputs(spec)
    # every CTA first waits on a barrier nothing signals (1 ms limit): the
    # kernel records the timeout, drains and returns; results undefined
    with ta.Plan.from_spec(spec, host_only=1, wait_timeout_us=1000, debug_stuck_wait=1,
                           merge_mode=1, split_tokens=256) as p:
        _static(p, spec, q, k, v)
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    with ta.Plan.from_spec(spec, host_only=1, merge_mode=1, split_tokens=256) as p:
        for _ in range(2):
            out, lse = _static(p, spec, q, k, v)
            compare(out, lse, ref, ref_lse)


def test_static_entry_point_refuses_a_plan_larger_than_its_scratch():
    import tree_structured_decode_gb300 as ta
    from tree_structured_decode_gb300 import _abi

    spec = W.config_irregular()  # ~0.14 GB of partial results: far above the scratch
    q = torch.zeros((spec.n_queries, spec.n_q_heads, spec.head_dim), dtype=torch.bfloat16,
                    device="cuda")
    kv = torch.zeros((1,), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((spec.n_queries, spec.n_q_heads, spec.head_dim), device="cuda")
    with ta.Plan.from_spec(spec, host_only=1) as p:
        st = p.run_static(q, kv, kv, out, None)
    assert _abi.STATUS_NAMES[st] == "TA_ERR_UNSUPPORTED"
    msg = ta.load_library().tree_attn_last_error().decode()
    assert "static scratch" in msg and str(_abi.STATIC_SCRATCH_BYTES) in msg
