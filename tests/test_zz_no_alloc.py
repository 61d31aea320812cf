"""The allocation-free entry point, tree_attn_run_static().

Some callers may not allocate device memory (an engine plug-in whose host
owns all GPU memory, a serving loop with a fixed memory budget).  For them the
library runs a plan out of one fixed scratch array and can be driven by a
host-only plan, so nothing on the GPU is allocated by planning or running.
These tests call it through the C ABI, twice in a row with different plans
(the shared scratch must be refilled correctly each time), and compare with
tree_attn_run() on the same inputs under the parity tolerance; they also check
that a plan too large for the scratch is refused.  The file is collected last
so a failure here never hides the other tests.
"""
import pytest
import torch

import workloads as W
from parity_utils import LSE_ABS, MAX_ABS, MEAN_ABS, make_inputs

pytestmark = pytest.mark.gpu


def _close(a, b, la, lb):
    err = (a.double() - b.double()).abs()
    assert float(err.max()) <= MAX_ABS and float(err.mean()) <= MEAN_ABS
    fin = torch.isfinite(lb)
    assert torch.equal(fin, torch.isfinite(la))
    if fin.any():
        assert float((la[fin].double() - lb[fin].double()).abs().max()) <= LSE_ABS


def _reference_run(spec, q, k, v):
    import tree_structured_decode_gb300 as ta

    with ta.Plan.from_spec(spec) as p:
        out, lse = p.run(q, k, v)
        torch.cuda.synchronize()
        assert p.device_status() == 0
    return out, lse


def test_static_entry_point_matches_run_on_two_calls_in_a_row():
    import tree_structured_decode_gb300 as ta

    specs = [W.config_tiny(), W.random_tree(77, n_nodes=30, max_len=300, hq=8, hkv=2, d=128,
                                            max_queries_per_node=3)]
    data = [make_inputs(s, tail_fill=float("nan")) for s in specs]
    refs = [_reference_run(s, *d) for s, d in zip(specs, data)]
    plans = [ta.Plan.from_spec(s, host_only=1, split_tokens=128) for s in specs]
    try:
        for rnd in range(2):  # second round: the scratch holds the other plan's tables
            for spec, (q, k, v), (ro, rl), plan in zip(specs, data, refs, plans):
                out = torch.full((spec.n_queries, spec.n_q_heads, spec.head_dim), float("nan"),
                                 dtype=torch.float32, device="cuda")
                lse = torch.full((spec.n_queries, spec.n_q_heads), float("nan"),
                                 dtype=torch.float32, device="cuda")
                st = plan.run_static(q, k, v, out, lse)
                assert st == 0, ta.load_library().tree_attn_last_error()
                torch.cuda.synchronize()
                _close(out, ro, lse, rl)
    finally:
        for p in plans:
            p.close()


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
