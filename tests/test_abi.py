"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects bad input with the documented status (no GPU calls)."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W

ta = pytest.importorskip("tree_structured_decode_gb300")
from tree_structured_decode_gb300 import _abi  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "tree_attn.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tree_attn_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = _abi.load_library()
    declared = _declared_functions()
    assert declared == sorted(_abi.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    for code, name in _abi.STATUS_NAMES.items():
        assert _abi.status_string(code) == name


def test_options_init_defaults():
    o = ta.Options()
    _abi.load_library().tree_attn_options_init(ctypes.byref(o))
    assert o.gamma == 64 and list(o.ts_q_set) == [16, 64, 128, 0] and o.ts_c == 64
    assert o.wait_timeout_us == 2_000_000 and o.force_path == 0


def _plan(spec, **kw):
    return ta.Plan.from_spec(spec, host_only=1, num_sms=152, **kw)


def _expect(status_name, fn):
    with pytest.raises(ta.TreeAttnError) as e:
        fn()
    assert _abi.STATUS_NAMES[e.value.status] == status_name, str(e.value)
    return e.value


def test_rejects_two_roots_and_cycles():
    spec = W.random_tree(1, n_nodes=6)
    spec.parent = spec.parent.copy()
    spec.parent[3] = -1
    _expect("TA_ERR_NOT_A_TREE", lambda: _plan(spec))
    spec = W.random_tree(1, n_nodes=6)
    spec.parent = spec.parent.copy()
    spec.parent[1], spec.parent[2] = 2, 1  # cycle 1 <-> 2
    _expect("TA_ERR_NOT_A_TREE", lambda: _plan(spec))
    spec.parent[1] = 99
    _expect("TA_ERR_NOT_A_TREE", lambda: _plan(spec))


def test_rejects_bad_block_tables():
    spec = W.random_tree(2, n_nodes=5, max_len=40)
    spec.node_pages = spec.node_pages.copy()
    spec.node_pages[0] = spec.num_pages
    err = _expect("TA_ERR_PAGE_RANGE", lambda: _plan(spec))
    assert "page id" in str(err)
    spec = W.random_tree(2, n_nodes=5, max_len=40)
    spec.node_kv_len = spec.node_kv_len.copy()
    spec.node_kv_len[0] += 16  # one page short
    _expect("TA_ERR_PAGE_RANGE", lambda: _plan(spec))


def test_rejects_bad_queries_and_shapes():
    spec = W.random_tree(3, n_nodes=5, max_len=40)
    spec.query_kv_end = spec.query_kv_end.copy()
    spec.query_kv_end[0] = int(spec.node_kv_len[spec.query_node[0]]) + 1
    _expect("TA_ERR_INVALID_ARG", lambda: _plan(spec))
    spec = W.random_tree(3, n_nodes=5, max_len=40)
    spec.query_node = spec.query_node.copy()
    spec.query_node[0] = spec.n_nodes
    _expect("TA_ERR_INVALID_ARG", lambda: _plan(spec))
    spec = W.random_tree(3, n_nodes=5, max_len=40, d=96)
    _expect("TA_ERR_UNSUPPORTED", lambda: _plan(spec))
    spec = W.random_tree(3, n_nodes=5, max_len=40, hq=6, hkv=4)
    _expect("TA_ERR_UNSUPPORTED", lambda: _plan(spec))


def test_unknown_option_is_rejected():
    spec = W.random_tree(4, n_nodes=3)
    with pytest.raises(TypeError):
        _plan(spec, not_an_option=1)


def test_run_on_host_only_plan_fails_without_touching_the_gpu():
    spec = W.random_tree(4, n_nodes=3)
    p = _plan(spec)
    st = p.run_ptrs(16, 16, 16, 16, 0, 0)
    assert _abi.STATUS_NAMES[st] == "TA_ERR_HOST_ONLY_PLAN"


def test_append_on_host_only_plan_fails_without_touching_the_gpu():
    spec = W.random_tree(4, n_nodes=3)
    p = _plan(spec)
    f = [ctypes.c_void_p(16)] * 4
    st = ta.load_library().tree_attn_append_kv(p._handle, *f, ctypes.c_void_p(0))
    assert _abi.STATUS_NAMES[st] == "TA_ERR_HOST_ONLY_PLAN"
    st = ta.load_library().tree_attn_append_kv(None, *f, ctypes.c_void_p(0))
    assert _abi.STATUS_NAMES[st] == "TA_ERR_INVALID_ARG"


def test_empty_query_set_and_zero_length_nodes_plan():
    spec = W._finish("empty", [-1, 0], [0, 0], [], [], 4, 2, 64, seed=0)
    with _plan(spec) as p:
        d = p.describe()
        assert d["groups"] == [] and d["units"] == 0 and d["partials"] == []
    spec = W._finish("zero", [-1, 0], [0, 0], [1], [0], 4, 2, 64, seed=0)
    with _plan(spec) as p:
        d = p.describe()
        assert len(d["groups"]) >= 1 and all(g["span"] == 0 for g in d["groups"])


def test_query_kv_end_null_means_whole_node():
    spec = W.config_tiny()
    with ta.Plan(spec.parent, spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                 spec.num_pages, spec.query_node, None, 4, 4, 64, host_only=1) as p:
        a = p.describe()
    with _plan(spec) as p:
        b = p.describe()
    assert a == b
