"""The append step on the GPU (tree_attn_append_kv): each query token's new
K/V lands at its own position of the paged cache, bit for bit as the oracle
places it, and attention over the appended cache matches the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.attention import append_kv as oracle_append
from parity_utils import compare, make_inputs, oracle_on_tokens

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("seed,hq,hkv,d", [(3, 8, 2, 128), (8, 4, 4, 64), (12, 64, 4, 128)])
def test_append_then_attend(seed, hq, hkv, d):
    import tree_structured_decode_gb300 as ta

    spec = W.random_tree(seed, n_nodes=25, max_len=300, hq=hq, hkv=hkv, d=d, zero_len_prob=0.1,
                         max_queries_per_node=4)
    q, k, v = make_inputs(spec, tail_fill=float("nan"))
    g = torch.Generator(device="cpu").manual_seed(seed)
    k_new = torch.randn((spec.n_queries, hkv, d), generator=g).to(torch.bfloat16)
    v_new = torch.randn((spec.n_queries, hkv, d), generator=g).to(torch.bfloat16)
    # tokens sharing a position carry the same values (the call leaves either's)
    first = {}
    for t in range(spec.n_queries):
        key = (int(spec.query_node[t]), int(spec.query_kv_end[t]))
        first.setdefault(key, t)
        k_new[t], v_new[t] = k_new[first[key]], v_new[first[key]]
    kk, vv = k.clone(), v.clone()
    with ta.Plan.from_spec(spec) as p:
        p.append_kv(k_new.cuda(), v_new.cuda(), kk, vv)
        torch.cuda.synchronize()
        ko, vo = oracle_append(spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                               spec.query_node, spec.query_kv_end, _bits(k), _bits(v),
                               _bits(k_new), _bits(v_new))
        assert np.array_equal(_bits(kk), ko) and np.array_equal(_bits(vv), vo)
        out, lse = p.run(q, kk, vv)
        torch.cuda.synchronize()
        assert p.device_status() == 0
    ref, ref_lse = oracle_on_tokens(spec, q, kk, vv, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)
