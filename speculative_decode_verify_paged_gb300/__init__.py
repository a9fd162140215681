"""Block attention for speculative-decoding verify and draft over a paged KV cache, on GB300.

A thin ctypes binding over ``libspec_attn.so`` (C ABI in ``include/spec_attn.h``).
Every step of the computation runs in the library's CUDA kernels; this module
only marshals arguments: torch tensors are passed as device pointers and the
current torch CUDA stream is used unless another is given.  There is no CPU
path: if the library is missing, every call raises.

Names follow the C ABI::

    plan = spec_attn_plan_create(num_reqs=..., total_q_rows=..., max_w=..., ...,
                                 seq_lens=host_seq_lens, q_indptr=host_q_indptr)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    spec_attn_run(plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, ws)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libspec_attn.so")

SPEC_ATTN_OK = 0
SPEC_ATTN_E_INVALID_ARG = -1
SPEC_ATTN_E_UNSUPPORTED = -2
SPEC_ATTN_E_WORKSPACE_TOO_SMALL = -3
SPEC_ATTN_E_CUDA = -4
SPEC_ATTN_E_DEVICE_CHECK = -5

SPEC_ATTN_MASK_CAUSAL_IN_BLOCK = 0
SPEC_ATTN_MASK_NON_CAUSAL = 1
SPEC_ATTN_KV_BF16 = 0
SPEC_ATTN_KV_NVFP4 = 1
SPEC_ATTN_VARIANT_AUTO = 0
SPEC_ATTN_VARIANT_CUDA_CORE = 1
SPEC_ATTN_VARIANT_TCGEN05 = 2

SPEC_ATTN_DEV_BAD_PAGE = 0x1
SPEC_ATTN_DEV_BAD_SEQ_LEN = 0x2
SPEC_ATTN_DEV_BAD_WINDOW = 0x4
SPEC_ATTN_DEV_WAIT_TIMEOUT = 0x8

# every symbol include/spec_attn.h declares
EXPORTED_SYMBOLS = (
    "spec_attn_plan_create", "spec_attn_plan_destroy", "spec_attn_plan_get_info",
    "spec_attn_run", "spec_attn_run_traced", "spec_attn_plan_set_timing_events",
    "spec_attn_reset_device_status", "spec_attn_check_device_status",
    "spec_attn_status_string", "spec_attn_last_cuda_error", "spec_attn_version",
    "spec_attn_run_noalloc", "spec_attn_noalloc_check_device_status", "spec_attn_append_kv",
    "spec_attn_run_append", "spec_attn_run_dense_block",
)


class SpecAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class spec_attn_problem(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("total_q_rows", ctypes.c_int32), ("max_w", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("block_table_stride", ctypes.c_int32), ("mask_mode", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("sm_scale", ctypes.c_float), ("max_seq_len", ctypes.c_int64),
        ("force_splits", ctypes.c_int32), ("kernel_variant", ctypes.c_int32),
        ("w_invariant", ctypes.c_int32), ("fixed_keys_per_split", ctypes.c_int32),
        ("window_left", ctypes.c_int32), ("kv_page_stride", ctypes.c_int64),
        ("scale_page_stride", ctypes.c_int64), ("dense_block_kv", ctypes.c_int32),
        ("early_metadata", ctypes.c_int32), ("test_stall", ctypes.c_int32),
        ("early_context_kv", ctypes.c_int32),
    ]


class spec_attn_plan_info(ctypes.Structure):
    _fields_ = [
        ("kernel_variant", ctypes.c_int32), ("keys_per_split", ctypes.c_int32),
        ("max_splits", ctypes.c_int32), ("row_groups", ctypes.c_int32),
        ("grid_x", ctypes.c_int32), ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
        ("block_threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
        ("uses_merge", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None):
    """Load libspec_attn.so (built by ``build.build()``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libspec_attn.so not found at {p}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.spec_attn_plan_create.restype = i32
        lib.spec_attn_plan_create.argtypes = [ctypes.POINTER(spec_attn_problem), vp, vp,
                                              ctypes.POINTER(vp), ctypes.POINTER(sz)]
        lib.spec_attn_plan_destroy.restype = i32
        lib.spec_attn_plan_destroy.argtypes = [vp]
        lib.spec_attn_plan_get_info.restype = i32
        lib.spec_attn_plan_get_info.argtypes = [vp, ctypes.POINTER(spec_attn_plan_info)]
        run_args = [vp, vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp, vp, vp, vp]
        lib.spec_attn_run.restype = i32
        lib.spec_attn_run.argtypes = run_args + [vp, sz, vp]
        lib.spec_attn_run_traced.restype = i32
        lib.spec_attn_run_traced.argtypes = run_args + [vp, vp, sz, vp]
        lib.spec_attn_plan_set_timing_events.restype = i32
        lib.spec_attn_plan_set_timing_events.argtypes = [vp, vp, vp]
        lib.spec_attn_reset_device_status.restype = i32
        lib.spec_attn_reset_device_status.argtypes = [vp, vp]
        lib.spec_attn_check_device_status.restype = i32
        lib.spec_attn_check_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.spec_attn_status_string.restype = ctypes.c_char_p
        lib.spec_attn_status_string.argtypes = [i32]
        lib.spec_attn_last_cuda_error.restype = i32
        lib.spec_attn_last_cuda_error.argtypes = []
        lib.spec_attn_version.restype = i32
        lib.spec_attn_version.argtypes = []
        lib.spec_attn_run_noalloc.restype = i32
        lib.spec_attn_run_noalloc.argtypes = run_args + [vp]
        lib.spec_attn_noalloc_check_device_status.restype = i32
        lib.spec_attn_noalloc_check_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        cache_args = [vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp, vp]
        lib.spec_attn_append_kv.restype = i32
        lib.spec_attn_append_kv.argtypes = [vp, vp, vp] + cache_args + [vp, sz, vp]
        lib.spec_attn_run_append.restype = i32
        lib.spec_attn_run_append.argtypes = [vp, vp, vp, vp] + cache_args + [vp, vp, vp, sz, vp]
        lib.spec_attn_run_dense_block.restype = i32
        lib.spec_attn_run_dense_block.argtypes = [vp] * 13 + [sz, vp]
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().spec_attn_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != SPEC_ATTN_OK:
        raise SpecAttnError(status, what)


def _host_i32(t):
    """Host int32 array (torch tensor / sequence) -> (ctypes pointer, keepalive)."""
    if t is None:
        return None, None
    import numpy as np
    if hasattr(t, "detach"):
        t = t.detach().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(t, dtype=np.int32))
    return a.ctypes.data_as(ctypes.c_void_p), a


def _dptr(t, what, dtype=None, contiguous=True):
    """Device pointer of a CUDA tensor.  contiguous=False admits a view whose
    layout the plan describes (a pool with a page stride)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Owns a spec_attn_plan* (destroyed with this object)."""

    def __init__(self, handle, workspace_bytes, problem):
        self._lib = load_library()
        self.handle = handle
        self.workspace_bytes = int(workspace_bytes)
        self.problem = problem
        info = spec_attn_plan_info()
        _check(self._lib.spec_attn_plan_get_info(handle, ctypes.byref(info)), "spec_attn_plan_get_info")
        self.info = {name: getattr(info, name) for name, _ in spec_attn_plan_info._fields_}

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h is not None:
            try:
                self._lib.spec_attn_plan_destroy(h)
            except Exception:
                pass

    def set_timing_events(self, begin, end):
        b = None if begin is None else ctypes.c_void_p(begin.cuda_event)
        e = None if end is None else ctypes.c_void_p(end.cuda_event)
        _check(self._lib.spec_attn_plan_set_timing_events(self.handle, b, e),
               "spec_attn_plan_set_timing_events")


def spec_attn_plan_create(*, num_reqs, total_q_rows, max_w, num_q_heads, num_kv_heads, head_dim,
                          num_pages, block_table_stride, max_seq_len, mask_mode=0, kv_dtype=0,
                          page_size=16, sm_scale=0.0, force_splits=0, kernel_variant=0,
                          seq_lens=None, q_indptr=None, w_invariant=0, fixed_keys_per_split=0,
                          window_left=0, kv_page_stride=0, scale_page_stride=0, dense_block_kv=0,
                          early_metadata=0, test_stall=0, early_context_kv=0) -> Plan:
    lib = load_library()
    prob = spec_attn_problem(num_reqs, total_q_rows, max_w, num_q_heads, num_kv_heads, head_dim,
                             page_size, num_pages, block_table_stride, mask_mode, kv_dtype,
                             float(sm_scale), int(max_seq_len), force_splits, kernel_variant,
                             int(w_invariant), int(fixed_keys_per_split), int(window_left),
                             int(kv_page_stride), int(scale_page_stride), int(dense_block_kv),
                             int(early_metadata), int(test_stall), int(early_context_kv))
    sl, _k1 = _host_i32(seq_lens)
    qi, _k2 = _host_i32(q_indptr)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib.spec_attn_plan_create(ctypes.byref(prob), sl, qi, ctypes.byref(handle), ctypes.byref(ws)),
           "spec_attn_plan_create")
    return Plan(handle, ws.value, prob)


def _pool_ptrs(plan, k_pool, v_pool, k_scales, v_scales):
    """Pool pointers; a plan with a page stride takes strided views."""
    import torch
    fp4 = plan.problem.kv_dtype == SPEC_ATTN_KV_NVFP4
    dense = plan.problem.kv_page_stride == 0
    dense_sc = plan.problem.scale_page_stride == 0
    return [_dptr(k_pool, "k_pool", torch.uint8 if fp4 else torch.bfloat16, dense),
            _dptr(v_pool, "v_pool", torch.uint8 if fp4 else torch.bfloat16, dense),
            _dptr(k_scales, "k_scales", torch.uint8, dense_sc), _dptr(v_scales, "v_scales", torch.uint8, dense_sc)]


def _run_args(plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, k_scales, v_scales,
              k_gscale, v_gscale):
    import torch
    return [plan.handle,
            _dptr(q, "q", torch.bfloat16),
            *_pool_ptrs(plan, k_pool, v_pool, k_scales, v_scales),
            ctypes.c_float(k_gscale), ctypes.c_float(v_gscale),
            _dptr(block_table, "block_table", torch.int32), _dptr(seq_lens, "seq_lens", torch.int32),
            _dptr(q_indptr, "q_indptr", torch.int32), _dptr(o, "o", torch.bfloat16),
            _dptr(lse, "lse", torch.float32)]


def spec_attn_run(plan: Plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, workspace,
                  k_scales=None, v_scales=None, k_gscale=1.0, v_gscale=1.0, stream=None):
    """Launch one attention call (asynchronous).  Raises SpecAttnError on a bad status."""
    lib = load_library()
    args = _run_args(plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, k_scales,
                     v_scales, k_gscale, v_gscale)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.spec_attn_run(*args, _dptr(workspace, "workspace"), ctypes.c_size_t(ws_bytes),
                             _stream_handle(stream)), "spec_attn_run")


def spec_attn_run_traced(plan: Plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, trace,
                         workspace, k_scales=None, v_scales=None, k_gscale=1.0, v_gscale=1.0,
                         stream=None):
    import torch
    lib = load_library()
    args = _run_args(plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, k_scales,
                     v_scales, k_gscale, v_gscale)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.spec_attn_run_traced(*args, _dptr(trace, "trace", torch.int64), _dptr(workspace, "workspace"),
                                    ctypes.c_size_t(ws_bytes), _stream_handle(stream)),
           "spec_attn_run_traced")


def spec_attn_run_noalloc(plan: Plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse,
                          k_scales=None, v_scales=None, k_gscale=1.0, v_gscale=1.0, stream=None):
    """spec_attn_run for callers that cannot allocate device memory: the
    library's built-in scratch array stands in for the workspace (calls that
    may overlap on the GPU must be serialised by the caller)."""
    lib = load_library()
    args = _run_args(plan, q, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse, k_scales,
                     v_scales, k_gscale, v_gscale)
    _check(lib.spec_attn_run_noalloc(*args, _stream_handle(stream)), "spec_attn_run_noalloc")


def spec_attn_noalloc_check_device_status(stream=None) -> int:
    """Device-status bits the last spec_attn_run_noalloc call on the current
    device left (and clear them); 0 means no device check tripped."""
    bits = ctypes.c_uint32()
    st = load_library().spec_attn_noalloc_check_device_status(_stream_handle(stream), ctypes.byref(bits))
    if st not in (SPEC_ATTN_OK, SPEC_ATTN_E_DEVICE_CHECK):
        _check(st, "spec_attn_noalloc_check_device_status")
    return int(bits.value)


def _cache_args(plan, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale, block_table, seq_lens,
                q_indptr):
    import torch
    return [*_pool_ptrs(plan, k_pool, v_pool, k_scales, v_scales),
            ctypes.c_float(k_gscale), ctypes.c_float(v_gscale),
            _dptr(block_table, "block_table", torch.int32), _dptr(seq_lens, "seq_lens", torch.int32),
            _dptr(q_indptr, "q_indptr", torch.int32)]


def spec_attn_append_kv(plan: Plan, k_new, v_new, k_pool, v_pool, block_table, seq_lens, q_indptr, workspace,
                        k_scales=None, v_scales=None, k_gscale=1.0, v_gscale=1.0, stream=None):
    """Write the windows' new K/V rows ([total_rows, Hkv, d] bf16) into their
    cache slots, quantising for NVFP4 caches (asynchronous)."""
    import torch
    lib = load_library()
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.spec_attn_append_kv(plan.handle, _dptr(k_new, "k_new", torch.bfloat16),
                                   _dptr(v_new, "v_new", torch.bfloat16),
                                   *_cache_args(plan, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                                block_table, seq_lens, q_indptr),
                                   _dptr(workspace, "workspace"), ctypes.c_size_t(ws_bytes),
                                   _stream_handle(stream)), "spec_attn_append_kv")


def spec_attn_run_append(plan: Plan, q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, q_indptr, o, lse,
                         workspace, k_scales=None, v_scales=None, k_gscale=1.0, v_gscale=1.0, stream=None):
    """KV append, then the attention call, on one stream (asynchronous)."""
    import torch
    lib = load_library()
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.spec_attn_run_append(plan.handle, _dptr(q, "q", torch.bfloat16),
                                    _dptr(k_new, "k_new", torch.bfloat16), _dptr(v_new, "v_new", torch.bfloat16),
                                    *_cache_args(plan, k_pool, v_pool, k_scales, v_scales, k_gscale, v_gscale,
                                                 block_table, seq_lens, q_indptr),
                                    _dptr(o, "o", torch.bfloat16), _dptr(lse, "lse", torch.float32),
                                    _dptr(workspace, "workspace"), ctypes.c_size_t(ws_bytes),
                                    _stream_handle(stream)), "spec_attn_run_append")


def spec_attn_run_dense_block(plan: Plan, q, block_k, block_v, k_pool, v_pool, block_table, seq_lens, q_indptr,
                              o, lse, workspace, trace=None, stream=None):
    """Attention with the window's own keys from dense block tensors
    ([total_rows, Hkv, d] bf16) and the context from the cache (asynchronous)."""
    import torch
    lib = load_library()
    ws_bytes = workspace.numel() * workspace.element_size()
    dense = plan.problem.kv_page_stride == 0
    _check(lib.spec_attn_run_dense_block(
        plan.handle, _dptr(q, "q", torch.bfloat16), _dptr(block_k, "block_k", torch.bfloat16),
        _dptr(block_v, "block_v", torch.bfloat16), _dptr(k_pool, "k_pool", torch.bfloat16, dense),
        _dptr(v_pool, "v_pool", torch.bfloat16, dense), _dptr(block_table, "block_table", torch.int32),
        _dptr(seq_lens, "seq_lens", torch.int32), _dptr(q_indptr, "q_indptr", torch.int32),
        _dptr(o, "o", torch.bfloat16), _dptr(lse, "lse", torch.float32), _dptr(trace, "trace", torch.int64),
        _dptr(workspace, "workspace"), ctypes.c_size_t(ws_bytes), _stream_handle(stream)),
        "spec_attn_run_dense_block")


def spec_attn_reset_device_status(workspace, stream=None):
    _check(load_library().spec_attn_reset_device_status(_dptr(workspace, "workspace"),
                                                        _stream_handle(stream)),
           "spec_attn_reset_device_status")


def spec_attn_check_device_status(workspace, stream=None) -> int:
    """Return the device-status bits (and clear them); 0 means no device check tripped."""
    bits = ctypes.c_uint32()
    st = load_library().spec_attn_check_device_status(_dptr(workspace, "workspace"),
                                                      _stream_handle(stream), ctypes.byref(bits))
    if st not in (SPEC_ATTN_OK, SPEC_ATTN_E_DEVICE_CHECK):
        _check(st, "spec_attn_check_device_status")
    return int(bits.value)


def spec_attn_version() -> int:
    return load_library().spec_attn_version()


def spec_attn_last_cuda_error() -> int:
    return load_library().spec_attn_last_cuda_error()


# --------------------------------------------------------------------------- #
# Convenience: run a workload (from .workloads) that lives on the GPU
# --------------------------------------------------------------------------- #
class DeviceWorkload:
    """A workload's tensors moved to a CUDA device, plus output and workspace buffers."""

    def __init__(self, wl, device="cuda", force_splits=0, kernel_variant=0, host_lens=True, w_invariant=0,
                 fixed_keys_per_split=0, append_rows=None, mode="run", interleave=False, early_metadata=0,
                 early_context_kv=0):
        """``append_rows``: (k_new, v_new) [total_rows, Hkv, d] bf16 for the KV
        append.  ``mode``: what :meth:`run` launches -- "run" (attention),
        "run_append" (append, then attention) or "append" (the append alone).
        ``interleave``: K and V pages (and NVFP4 scale pages) share one
        allocation [num_pages, 2, Hkv, page_size, row], so the pools are views
        with a page stride of twice their dense page."""
        import torch
        assert mode in ("run", "run_append", "append")
        assert mode == "run" or append_rows is not None
        self.wl = wl
        self.mode = mode
        dev = torch.device(device)
        self.q = wl.q.to(dev)
        kv_stride = sc_stride = 0
        if interleave:
            both = torch.stack([wl.k_pool, wl.v_pool], 1).to(dev)          # [pages, 2, Hkv, ps, row]
            self.kv_storage = both
            self.k_pool, self.v_pool = both[:, 0], both[:, 1]
            kv_stride = both[0].numel() * both.element_size()
            self.k_scales = self.v_scales = None
            if wl.k_scales is not None:
                sboth = torch.stack([wl.k_scales, wl.v_scales], 1).to(dev)
                self.scale_storage = sboth
                self.k_scales, self.v_scales = sboth[:, 0], sboth[:, 1]
                sc_stride = sboth[0].numel()
        else:
            self.k_pool = wl.k_pool.to(dev)
            self.v_pool = wl.v_pool.to(dev)
            self.k_scales = None if wl.k_scales is None else wl.k_scales.to(dev)
            self.v_scales = None if wl.v_scales is None else wl.v_scales.to(dev)
        self.block_table = wl.block_table.to(dev)
        self.seq_lens = wl.seq_lens.to(dev)
        self.q_indptr = wl.q_indptr.to(dev)
        self.o = torch.zeros(wl.total_rows, wl.num_q_heads, wl.head_dim, dtype=torch.bfloat16, device=dev)
        self.lse = torch.zeros(wl.total_rows, wl.num_q_heads, dtype=torch.float32, device=dev)
        self.plan = spec_attn_plan_create(
            num_reqs=wl.num_reqs, total_q_rows=wl.total_rows, max_w=max(1, wl.max_w),
            num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
            num_pages=wl.num_pages, block_table_stride=int(wl.block_table.shape[1]),
            max_seq_len=max(1, wl.max_seq_len), mask_mode=wl.mask_mode, kv_dtype=wl.kv_dtype,
            page_size=wl.page_size, sm_scale=wl.sm_scale, force_splits=force_splits,
            kernel_variant=kernel_variant, seq_lens=wl.seq_lens if host_lens else None,
            q_indptr=wl.q_indptr if host_lens else None, w_invariant=w_invariant,
            fixed_keys_per_split=fixed_keys_per_split, window_left=wl.window_left, kv_page_stride=kv_stride,
            scale_page_stride=sc_stride, dense_block_kv=int(wl.block_k is not None),
            early_metadata=early_metadata, early_context_kv=early_context_kv)
        self.workspace = torch.zeros(max(256, self.plan.workspace_bytes), dtype=torch.uint8, device=dev)
        self.block_k = None if wl.block_k is None else wl.block_k.to(dev)
        self.block_v = None if wl.block_v is None else wl.block_v.to(dev)
        self.k_new = self.v_new = None
        if append_rows is not None:
            self.k_new = append_rows[0].to(dev).contiguous()
            self.v_new = append_rows[1].to(dev).contiguous()

    def run(self, stream=None):
        if self.mode == "append":
            spec_attn_append_kv(self.plan, self.k_new, self.v_new, self.k_pool, self.v_pool, self.block_table,
                                self.seq_lens, self.q_indptr, self.workspace, self.k_scales, self.v_scales,
                                self.wl.k_gscale, self.wl.v_gscale, stream)
        elif self.mode == "run_append":
            spec_attn_run_append(self.plan, self.q, self.k_new, self.v_new, self.k_pool, self.v_pool,
                                 self.block_table, self.seq_lens, self.q_indptr, self.o, self.lse, self.workspace,
                                 self.k_scales, self.v_scales, self.wl.k_gscale, self.wl.v_gscale, stream)
        elif self.block_k is not None:
            spec_attn_run_dense_block(self.plan, self.q, self.block_k, self.block_v, self.k_pool, self.v_pool,
                                      self.block_table, self.seq_lens, self.q_indptr, self.o, self.lse,
                                      self.workspace, stream=stream)
        else:
            spec_attn_run(self.plan, self.q, self.k_pool, self.v_pool, self.block_table, self.seq_lens,
                          self.q_indptr, self.o, self.lse, self.workspace, self.k_scales, self.v_scales,
                          self.wl.k_gscale, self.wl.v_gscale, stream)

    def run_traced(self, trace, stream=None):
        if self.block_k is not None:
            spec_attn_run_dense_block(self.plan, self.q, self.block_k, self.block_v, self.k_pool, self.v_pool,
                                      self.block_table, self.seq_lens, self.q_indptr, self.o, self.lse,
                                      self.workspace, trace=trace, stream=stream)
            return
        spec_attn_run_traced(self.plan, self.q, self.k_pool, self.v_pool, self.block_table,
                             self.seq_lens, self.q_indptr, self.o, self.lse, trace, self.workspace,
                             self.k_scales, self.v_scales, self.wl.k_gscale, self.wl.v_gscale, stream)

    def device_status(self) -> int:
        return spec_attn_check_device_status(self.workspace)
