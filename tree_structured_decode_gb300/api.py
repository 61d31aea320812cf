"""Python entry points: ``Plan`` / ``plan`` / ``run`` over the C ABI.

Argument marshalling only (array conversion, pointer and stream handles);
planning happens in the library's host planner and attention in its CUDA
kernels.
"""
from __future__ import annotations

import ctypes
import json

import numpy as np

from . import _abi
from ._abi import Options, PlanStats, check, load_library

_OPTION_KEYS = {
    "gamma", "beta", "ts_q_set", "ts_c", "mma_min_rows", "split_tokens",
    "min_split_tokens", "split_waves", "num_sms", "force_path", "host_only",
    "wait_timeout_us", "force_edges", "debug_stuck_wait", "merge_mode", "no_pack", "cost_model",
}


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def make_options(**kw) -> tuple[Options, object]:
    """An ``Options`` struct from keyword arguments (unknown keys raise).

    Returns the struct and an object that must stay alive while it is used
    (the forced edge array)."""
    bad = set(kw) - _OPTION_KEYS
    if bad:
        raise TypeError(f"unknown planner options: {sorted(bad)}")
    o = Options()
    load_library().tree_attn_options_init(ctypes.byref(o))
    keep = None
    for k, v in kw.items():
        if v is None:
            continue
        if k == "ts_q_set":
            vals = list(v)[:4] + [0] * (4 - min(4, len(v)))
            o.ts_q_set = (ctypes.c_int32 * 4)(*vals)
        elif k == "force_edges":
            keep = np.ascontiguousarray(np.asarray(v, dtype=np.int8))
            o.force_edges = keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
        else:
            setattr(o, k, int(v))
    return o, keep


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Plan:
    """A planned tree: groups, units and device tables (tree_attn_plan)."""

    def __init__(self, parent, node_kv_len, node_page_offsets, node_pages, num_pages,
                 query_node, query_kv_end=None, n_q_heads=1, n_kv_heads=1, head_dim=128,
                 softmax_scale: float = 0.0, page_size: int = 16, **options):
        lib = load_library()
        self._lib = lib
        self._handle = ctypes.c_void_p()
        parent = _i32(parent)
        lens = _i32(node_kv_len)
        offs = _i32(node_page_offsets)
        pages = _i32(node_pages)
        qn = _i32(query_node)
        qe = None if query_kv_end is None else _i32(query_kv_end)
        opts, keep = make_options(**options)
        st = lib.tree_attn_plan(
            _ptr(parent), int(parent.shape[0]), _ptr(lens), _ptr(offs), _ptr(pages),
            int(page_size), int(num_pages), _ptr(qn), None if qe is None else _ptr(qe),
            int(qn.shape[0]), int(n_q_heads), int(n_kv_heads), int(head_dim),
            float(softmax_scale), ctypes.byref(opts), ctypes.byref(self._handle))
        del keep
        check(st, "tree_attn_plan")
        self.n_query_tokens = int(qn.shape[0])
        self.n_q_heads = int(n_q_heads)
        self.n_kv_heads = int(n_kv_heads)
        self.head_dim = int(head_dim)
        self.num_pages = int(num_pages)
        self.page_size = int(page_size)
        self.host_only = bool(options.get("host_only", 0))

    @classmethod
    def from_spec(cls, spec, **options):
        """Plan a workload description (``workloads.TreeSpec``-like object)."""
        return cls(spec.parent, spec.node_kv_len, spec.node_page_offsets, spec.node_pages,
                   spec.num_pages, spec.query_node, spec.query_kv_end, spec.n_q_heads,
                   spec.n_kv_heads, spec.head_dim, page_size=spec.page_size, **options)

    # -------------------------------------------------------------- run
    def run(self, q, k_pages, v_pages, out=None, lse=None, stream=None, want_lse=True):
        """Attention of every query token; returns (out, lse) (fp32 tensors)."""
        import torch

        nq, hq, d = self.n_query_tokens, self.n_q_heads, self.head_dim
        for name, t, shape in (("q", q, (nq, hq, d)),
                               ("k_pages", k_pages, (self.num_pages, self.n_kv_heads,
                                                     self.page_size, d)),
                               ("v_pages", v_pages, (self.num_pages, self.n_kv_heads,
                                                     self.page_size, d))):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} shape {tuple(t.shape)} != {shape}")
        if out is None:
            out = torch.empty((nq, hq, d), dtype=torch.float32, device=q.device)
        if lse is None and want_lse:
            lse = torch.empty((nq, hq), dtype=torch.float32, device=q.device)
        st = self._lib.tree_attn_run(
            self._handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pages.data_ptr()),
            ctypes.c_void_p(v_pages.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr() if lse is not None else 0), _stream_handle(stream))
        check(st, "tree_attn_run")
        return out, lse

    def append_kv(self, k_new, v_new, k_pages, v_pages, stream=None):
        """``tree_attn_append_kv``: write every query token's key and value
        (bf16 ``[n_query_tokens, n_kv_heads, head_dim]``) into its own
        position of the page pools (its visible end - 1), in place."""
        import torch

        for name, t in (("k_new", k_new), ("v_new", v_new), ("k_pages", k_pages),
                        ("v_pages", v_pages)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
        st = self._lib.tree_attn_append_kv(
            self._handle, ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
            ctypes.c_void_p(k_pages.data_ptr()), ctypes.c_void_p(v_pages.data_ptr()),
            _stream_handle(stream))
        check(st, "tree_attn_append_kv")

    def run_static(self, q, k_pages, v_pages, out, lse, stream=None) -> int:
        """tree_attn_run_static(): run without any device allocation (the
        library's fixed scratch holds the tables and partial results).  For
        callers that may not allocate device memory; ``out`` and ``lse`` must
        be given.  Returns the status (0 = TA_OK); see include/tree_attn.h for
        the size limit and the rule that calls must not overlap."""
        return self._lib.tree_attn_run_static(
            self._handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_pages.data_ptr()),
            ctypes.c_void_p(v_pages.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr() if lse is not None else 0), _stream_handle(stream))

    def run_ptrs(self, q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, lse_ptr: int,
                 stream_handle: int) -> int:
        """Raw-pointer run (no checks beyond the library's); returns the status."""
        return self._lib.tree_attn_run(self._handle, ctypes.c_void_p(q_ptr),
                                       ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                       ctypes.c_void_p(out_ptr), ctypes.c_void_p(lse_ptr),
                                       ctypes.c_void_p(stream_handle))

    def device_status(self, stream=None) -> int:
        """Synchronise and read (and clear) the device error word."""
        code = ctypes.c_int32(0)
        st = self._lib.tree_attn_device_status(self._handle, _stream_handle(stream),
                                               ctypes.byref(code))
        if st not in (_abi.TA_OK, 8):
            check(st, "tree_attn_device_status")
        return int(code.value)

    def profile(self, enable: bool = True):
        """Record CUDA events around each kernel of later runs."""
        check(self._lib.tree_attn_profile_enable(self._handle, int(bool(enable))),
              "tree_attn_profile_enable")

    def kernel_times(self) -> tuple[float, float]:
        """(partial pass ms, merge pass ms) of the last profiled run."""
        a, b = ctypes.c_float(0), ctypes.c_float(0)
        check(self._lib.tree_attn_profile_read(self._handle, ctypes.byref(a), ctypes.byref(b)),
              "tree_attn_profile_read")
        return float(a.value), float(b.value)

    # -------------------------------------------------------------- info
    def describe(self) -> dict:
        need = ctypes.c_size_t(0)
        self._lib.tree_attn_plan_describe(self._handle, None, 0, ctypes.byref(need))
        buf = ctypes.create_string_buffer(need.value)
        check(self._lib.tree_attn_plan_describe(self._handle, buf, need.value, None),
              "tree_attn_plan_describe")
        return json.loads(buf.value.decode())

    def schedule(self) -> dict:
        """``tree_attn_plan_describe_schedule``: the device tables of a run
        (units in schedule order, CTA ranges, blocks, row records, merge
        items), as flat int lists."""
        need = ctypes.c_size_t(0)
        self._lib.tree_attn_plan_describe_schedule(self._handle, None, 0, ctypes.byref(need))
        buf = ctypes.create_string_buffer(need.value)
        check(self._lib.tree_attn_plan_describe_schedule(self._handle, buf, need.value, None),
              "tree_attn_plan_describe_schedule")
        return json.loads(buf.value.decode())

    def stats(self) -> dict:
        s = PlanStats()
        check(self._lib.tree_attn_plan_get_stats(self._handle, ctypes.byref(s)),
              "tree_attn_plan_get_stats")
        return s.as_dict()

    def close(self):
        if getattr(self, "_handle", None) and self._handle.value:
            self._lib.tree_attn_plan_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def plan(*args, **kw) -> Plan:
    """``tree_attn_plan``: see ``Plan``."""
    return Plan(*args, **kw)


def run(p: Plan, q, k_pages, v_pages, out=None, lse=None, stream=None):
    """``tree_attn_run``: attention of every query token of plan ``p``."""
    return p.run(q, k_pages, v_pages, out=out, lse=lse, stream=stream)
