"""Oracle for tree-structured decode attention: TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU code (numpy, float64) that states what the
GPU path must compute.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it; the product path
(``tree_structured_decode_gb300``) never does, and shares no code with it.

Modules
  attention  the tree-attention definition (fp64), the log-sum-exp merge and
             the append of the query tokens' own K/V before attention.
  planner    the greedy binary edge assignment and grouping plan, written
             from the FastTree review page (Algorithm 1 and its cost model),
             and the chunks of the long-context split for a given chunk
             length: the decisions the pages define, used to check the native
             planner decision by decision.  How groups become GPU work units
             (tiles, packing, the automatic chunk length, the CTA schedule)
             is not the pages' and is not restated here; the tests check it
             by invariants on the device tables.

Parity status: every function here is pinned by tests that do not call it to
check itself (closed forms, brute force, an independent tree-mask
formulation, a library routine on special cases, the worked cases on the
pages, the cost of a plan worked out by hand); none is "parity unpinned".
"""
from .attention import (  # noqa: F401
    node_path,
    gather_node_kv,
    query_kv,
    tree_attention,
    tree_attention_spec,
    merge_partials,
    attention_rows,
    append_kv,
)
from .planner import (  # noqa: F401
    PlannerOptions,
    subtree_rows,
    greedy_edges,
    plan_groups,
    split_chunks,
    build_plan,
    plan_cost,
)
