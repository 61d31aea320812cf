"""Back-to-back runs on one stream, as the layers of a decode step.

Each run's partial-attention kernel is a programmatic dependent of the
stream's previous kernel (often the previous run's merge): it may be
scheduled, and set itself up, while that kernel finishes, and it reads its
inputs and writes its outputs and partials only once that kernel has
completed.  These runs share one plan (so one partial workspace and, for the
fused merge, one set of arrival counters) or alternate two plans, take no
host synchronisation between them, and each layer is compared with the fp64
oracle.  A layer whose queries come from the previous layer's output (a
torch kernel between the runs) checks the read-after-write order too.
"""
import numpy as np
import pytest
import torch

import workloads as W
from parity_utils import compare, make_inputs, oracle_on_tokens

pytestmark = pytest.mark.gpu


def _buffers(spec, n):
    nq, hq, d = spec.n_queries, spec.n_q_heads, spec.head_dim
    outs = [torch.full((nq, hq, d), float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(n)]
    lses = [torch.full((nq, hq), float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(n)]
    return outs, lses


@pytest.mark.parametrize("options", [
    {"split_tokens": 128},                      # partials and a separate merge
    {"split_tokens": 128, "merge_mode": 1},     # fused merge: shared counters
    {"split_tokens": -1, "force_edges": "ones"},  # one partial per token: no merge
])
def test_layers_back_to_back_share_one_plan(options):
    import tree_structured_decode_gb300 as ta

    spec = W.random_tree(47, n_nodes=30, max_len=400, hq=16, hkv=4, d=128,
                         max_queries_per_node=3)
    options = dict(options)
    if options.get("force_edges") == "ones":
        options["force_edges"] = np.ones(spec.n_nodes, dtype=np.int8)
    layers = [make_inputs(spec, seed=300 + i) for i in range(4)]
    tokens = list(range(spec.n_queries))
    refs = [oracle_on_tokens(spec, q, k, v, tokens) for q, k, v in layers]
    outs, lses = _buffers(spec, len(layers))
    with ta.Plan.from_spec(spec, **options) as plan:
        if options.get("split_tokens", 0) > 0:
            assert plan.stats()["n_merge_tokens"] > 0
        else:
            assert plan.stats()["n_merge_tokens"] == 0
        for (q, k, v), o, l in zip(layers, outs, lses):
            plan.run(q, k, v, out=o, lse=l)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
    for o, l, (ref, ref_lse) in zip(outs, lses, refs):
        compare(o, l, ref, ref_lse)


def test_two_plans_alternate_on_one_stream():
    import tree_structured_decode_gb300 as ta

    spec_a = W.random_tree(48, n_nodes=25, max_len=300, hq=8, hkv=2, d=128,
                           max_queries_per_node=2)
    spec_b = W.two_level(700, 6, 90, 32, 8, 128, seed=49)
    data = [make_inputs(s, seed=400 + i) for i, s in enumerate([spec_a, spec_b, spec_a, spec_b])]
    specs = [spec_a, spec_b, spec_a, spec_b]
    refs = [oracle_on_tokens(s, *d, list(range(s.n_queries))) for s, d in zip(specs, data)]
    bufs = [_buffers(s, 1) for s in specs]
    with ta.Plan.from_spec(spec_a, split_tokens=64) as pa, \
            ta.Plan.from_spec(spec_b, split_tokens=128) as pb:
        for s, (q, k, v), (o, l) in zip(specs, data, bufs):
            (pa if s is spec_a else pb).run(q, k, v, out=o[0], lse=l[0])
        torch.cuda.synchronize()
        assert pa.device_status() == 0 and pb.device_status() == 0
    for (o, l), (ref, ref_lse) in zip(bufs, refs):
        compare(o[0], l[0], ref, ref_lse)


def test_queries_from_the_previous_layer_output():
    import tree_structured_decode_gb300 as ta

    spec = W.random_tree(50, n_nodes=20, max_len=300, hq=8, hkv=2, d=128,
                         max_queries_per_node=2)
    q0, k0, v0 = make_inputs(spec, seed=500)
    _, k1, v1 = make_inputs(spec, seed=501)
    outs, lses = _buffers(spec, 2)
    with ta.Plan.from_spec(spec, split_tokens=64) as plan:
        plan.run(q0, k0, v0, out=outs[0], lse=lses[0])
        q1 = (outs[0] * 4.0).to(torch.bfloat16)  # a torch kernel reads layer 0's output
        plan.run(q1, k1, v1, out=outs[1], lse=lses[1])
        torch.cuda.synchronize()
        assert plan.device_status() == 0
    tokens = list(range(spec.n_queries))
    ref0, ref_lse0 = oracle_on_tokens(spec, q0, k0, v0, tokens)
    compare(outs[0], lses[0], ref0, ref_lse0)
    # layer 1's oracle takes the queries the GPU saw (bf16 of layer 0's fp32
    # output), so only layer 1's attention is compared
    ref1, ref_lse1 = oracle_on_tokens(spec, q1, k1, v1, tokens)
    compare(outs[1], lses[1], ref1, ref_lse1)
