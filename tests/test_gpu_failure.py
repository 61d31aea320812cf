"""Failure detection on the GPU without a fault: every in-kernel wait has a
time limit.  With debug_stuck_wait each CTA first waits on a barrier that
nothing signals; the wait runs out (1 ms limit), the kernel records
TA_DEVERR_TIMEOUT, stops issuing work, drains what is in flight, frees TMEM and
returns.  The host reads the status and the context stays usable."""
import pytest
import torch

import workloads as W
from parity_utils import compare, make_inputs, oracle_on_tokens

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    import tree_structured_decode_gb300 as ta
    from tree_structured_decode_gb300 import _abi

    spec = W.two_level(2048, 8, 100, 16, 4, 128, seed=9)
    q, k, v = make_inputs(spec)
    with ta.Plan.from_spec(spec, wait_timeout_us=1000, debug_stuck_wait=1) as p:
        p.run(q, k, v)
        code = p.device_status()
    assert code == _abi.DEVERR_TIMEOUT
    # the same inputs through a normal plan: correct results
    with ta.Plan.from_spec(spec) as p:
        out, lse = p.run(q, k, v)
        torch.cuda.synchronize()
        assert p.device_status() == 0
    ref, ref_lse = oracle_on_tokens(spec, q, k, v, list(range(spec.n_queries)))
    compare(out, lse, ref, ref_lse)
