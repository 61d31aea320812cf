"""Tree-structured decode attention on GB300 (sm_103a).

Thin Python binding over the C ABI of ``libtreeattn.so`` (declared in
``include/tree_attn.h``): argument marshalling only.  Every step of the
attention runs in the library's CUDA kernels; PyTorch supplies device memory
and streams.  There is no CPU fallback: if the library is missing, importing
the binding's entry points raises.

    plan = Plan(parent, node_kv_len, node_page_offsets, node_pages, num_pages,
                query_node, query_kv_end, n_q_heads, n_kv_heads, head_dim)
    out, lse = plan.run(q, k_pages, v_pages)
"""
from ._abi import (  # noqa: F401
    LIB_PATH,
    Options,
    PlanStats,
    TreeAttnError,
    load_library,
    status_string,
)
from .api import Plan, plan, run  # noqa: F401

__all__ = ["Plan", "plan", "run", "Options", "PlanStats", "TreeAttnError",
           "load_library", "status_string", "LIB_PATH"]
