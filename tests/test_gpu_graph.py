"""Runs captured in a CUDA graph, one per layer.

A decode step calls run() once per layer with the same tree and plan.  The
calls take no host synchronisation and allocate nothing, so a whole step
can be captured once and replayed (FastTree review page, 高效树结构注意力内核设计:
the per-step launch cost matters most for the small trees).  Three layers
with their own q/K/V and outputs are captured, the outputs are poisoned,
the graph is replayed, and each layer is compared with the fp64 oracle;
the same for the fused merge.
"""
import pytest
import torch

import workloads as W
from parity_utils import compare, make_inputs, oracle_on_tokens

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("merge_mode", [0, 1])
def test_layers_replayed_from_a_cuda_graph_match_the_oracle(merge_mode):
    import tree_structured_decode_gb300 as ta

    spec = W.random_tree(31, n_nodes=40, max_len=300, hq=8, hkv=2, d=128, max_queries_per_node=3)
    layers = [make_inputs(spec, seed=100 + i) for i in range(3)]
    tokens = list(range(spec.n_queries))
    refs = [oracle_on_tokens(spec, q, k, v, tokens) for q, k, v in layers]
    nq, hq, d = spec.n_queries, spec.n_q_heads, spec.head_dim
    outs = [torch.empty((nq, hq, d), dtype=torch.float32, device="cuda") for _ in layers]
    lses = [torch.empty((nq, hq), dtype=torch.float32, device="cuda") for _ in layers]
    with ta.Plan.from_spec(spec, split_tokens=128, merge_mode=merge_mode) as plan:
        assert plan.stats()["n_merge_tokens"] > 0
        plan.run(*layers[0], out=outs[0], lse=lses[0])  # first launch outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        with torch.cuda.graph(graph, stream=stream):
            for (q, k, v), o, l in zip(layers, outs, lses):
                plan.run(q, k, v, out=o, lse=l)
        for _ in range(2):
            for o, l in zip(outs, lses):
                o.fill_(float("nan"))
                l.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            for o, l, (ro, rl) in zip(outs, lses, refs):
                compare(o, l, ro, rl)
