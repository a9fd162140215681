"""CPU fp64 oracle for speculative-decoding block attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  The oracle is the slow, plainly-written definition
of what the CUDA library computes; only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may load it.  It shares no code with
the CUDA library and never serves as a fallback for it.

The arithmetic lives in ``spec_attn_oracle.c`` (plain C, fp64, OpenMP over
independent output rows only) and ``kv_append_oracle.c`` (the KV append that
precedes a verify call, with its NVFP4 quantiser); this module compiles both
with gcc into ``oracle/_build/libspec_attn_oracle.so`` and wraps them with
ctypes.

Parity pins (tests/test_oracle_pins.py) hold every function here to values
fixed independently of this code: torch's fp64 scaled-dot-product attention on
CPU for W=1 decode, a pure-Python brute force on tiny shapes, closed forms
(zero queries, one visible key, constant power-of-two values), invariances
(page permutation, row-wise reduction to decode, last-row agreement of the two
masks) and the OCP e2m1 / e4m3 format definitions.  The append and its
quantiser are pinned in tests/test_oracle_append_pins.py: exact round trips of
representable blocks, midpoint and saturation cases of both encoders, a
rational-arithmetic brute force of every code, torch's own e4m3 rounding, and
the placement of every row checked slot by slot.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = (os.path.join(_HERE, "spec_attn_oracle.c"), os.path.join(_HERE, "kv_append_oracle.c"))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libspec_attn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, f64, vp = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.spec_attn_oracle_run.restype = i32
            lib.spec_attn_oracle_run.argtypes = [
                i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, f64,
                vp, vp, vp, vp, vp, f64, f64, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_e2m1.restype = f64
            lib.oracle_e2m1.argtypes = [ctypes.c_uint]
            lib.oracle_e4m3.restype = f64
            lib.oracle_e4m3.argtypes = [ctypes.c_uint]
            lib.oracle_bf16_value.restype = f64
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint]
            lib.oracle_round_bf16.restype = ctypes.c_uint
            lib.oracle_round_bf16.argtypes = [f64]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            lib.oracle_nvfp4_quantise_block.restype = None
            lib.oracle_nvfp4_quantise_block.argtypes = [vp, ctypes.c_float, vp, vp]
            lib.spec_attn_oracle_append_kv.restype = i32
            lib.spec_attn_oracle_append_kv.argtypes = [
                i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                ctypes.c_float, vp, i32, vp, vp]
            lib.spec_attn_oracle_num_threads.restype = i32
            lib.spec_attn_oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """torch tensor or numpy array -> contiguous numpy array of ``dtype`` bits."""
    if t is None:
        return None
    if hasattr(t, "detach"):  # torch tensor
        import torch
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        t = t.numpy()
    a = np.ascontiguousarray(t)
    return a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)


def e2m1(code: int) -> float:
    return _load().oracle_e2m1(code)


def e4m3(byte: int) -> float:
    return _load().oracle_e4m3(byte)


def round_bf16_bits(x: float) -> int:
    return _load().oracle_round_bf16(float(x))


def e4m3_encode(x: float) -> int:
    """binary32 value -> E4M3 byte (nearest even, saturating at 448)."""
    return _load().oracle_e4m3_encode(float(x))


def e2m1_encode(x: float) -> int:
    """binary32 value -> E2M1 code (nearest even, saturating at 6)."""
    return _load().oracle_e2m1_encode(float(x))


def nvfp4_quantise_block(x_bf16_bits, g: float):
    """16 bf16 bit patterns -> (8 code bytes, scale byte) against decode scale g."""
    x = np.ascontiguousarray(np.asarray(x_bf16_bits, dtype=np.uint16).reshape(16))
    codes = np.zeros(8, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.uint8)
    _load().oracle_nvfp4_quantise_block(_ptr(x), float(g), _ptr(codes), _ptr(sc))
    return codes, int(sc[0])


def append_kv(*, num_kv_heads, head_dim, page_size, kv_dtype, k_new, v_new, k_pool, v_pool,
              block_table, seq_lens, q_indptr, k_scales=None, v_scales=None, k_gscale=1.0,
              v_gscale=1.0):
    """Write every request's window rows of ``k_new`` / ``v_new`` ([total_rows,
    Hkv, d] bf16) into copies of the pools.  Returns numpy arrays
    ``(k_pool, v_pool, k_scales, v_scales)`` (scales None for bf16)."""
    lib = _load()
    kn = _np(k_new, np.uint16).copy()
    vn = _np(v_new, np.uint16).copy()
    pool_t = np.uint16 if kv_dtype == 0 else np.uint8
    kp = _np(k_pool, pool_t).copy()
    vp_ = _np(v_pool, pool_t).copy()
    ks = None if k_scales is None else _np(k_scales, np.uint8).copy()
    vs = None if v_scales is None else _np(v_scales, np.uint8).copy()
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    qin = _np(q_indptr, np.int32)
    num_pages = kp.shape[0]
    bt_stride = btn.shape[1] if btn.ndim == 2 else btn.shape[0]
    rc = lib.spec_attn_oracle_append_kv(
        sln.shape[0], kn.shape[0], num_kv_heads, head_dim, page_size, num_pages, kv_dtype,
        _ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp_), _ptr(ks), _ptr(vs), float(k_gscale),
        float(v_gscale), _ptr(btn), bt_stride, _ptr(sln), _ptr(qin))
    if rc != 0:
        raise ValueError(f"spec_attn_oracle_append_kv failed with code {rc}")
    return kp, vp_, ks, vs


def num_threads() -> int:
    return _load().spec_attn_oracle_num_threads()


def run(*, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, mask_mode, kv_dtype,
        sm_scale, q, k_pool, v_pool, block_table, seq_lens, q_indptr, k_scales=None,
        v_scales=None, k_gscale=1.0, v_gscale=1.0, row_select=None, want_o=True,
        want_lse=True, want_trace=False, window_left=0, block_k=None, block_v=None):
    """Run the oracle.  Arrays may be torch tensors (bf16 is taken bit-wise) or
    numpy arrays.  Returns ``(o, lse, trace)`` as numpy arrays (fp64, fp64,
    int64) or ``None`` for outputs not requested.  ``o`` and ``lse`` rows that
    ``row_select`` skips hold NaN."""
    lib = _load()
    qn = _np(q, np.uint16)
    total_rows = qn.shape[0]
    kn = _np(k_pool, np.uint16 if kv_dtype == 0 else np.uint8)
    vn = _np(v_pool, np.uint16 if kv_dtype == 0 else np.uint8)
    ksn = _np(k_scales, np.uint8)
    vsn = _np(v_scales, np.uint8)
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    qin = _np(q_indptr, np.int32)
    bkn = _np(block_k, np.uint16)
    bvn = _np(block_v, np.uint16)
    num_reqs = sln.shape[0]
    bt_stride = btn.shape[1] if btn.ndim == 2 else btn.shape[0]
    sel = None if row_select is None else np.ascontiguousarray(
        np.asarray(row_select, dtype=np.uint8).reshape(total_rows * num_q_heads))
    o = np.full((total_rows, num_q_heads, head_dim), np.nan) if want_o else None
    lse = np.full((total_rows, num_q_heads), np.nan) if want_lse else None
    trace = np.zeros((total_rows, num_q_heads, 2), dtype=np.int64) if want_trace else None
    rc = lib.spec_attn_oracle_run(
        num_reqs, total_rows, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
        mask_mode, int(window_left), kv_dtype, float(sm_scale), _ptr(qn), _ptr(kn), _ptr(vn), _ptr(ksn),
        _ptr(vsn), float(k_gscale), float(v_gscale), _ptr(bkn), _ptr(bvn), _ptr(btn), bt_stride, _ptr(sln),
        _ptr(qin), _ptr(sel), _ptr(o), _ptr(lse), _ptr(trace))
    if rc != 0:
        raise ValueError(f"spec_attn_oracle_run failed with code {rc}")
    return o, lse, trace


def run_workload(wl, **kw):
    """Run the oracle on a :class:`Workload` from the seeded input generators."""
    return run(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
               page_size=wl.page_size, num_pages=wl.num_pages, mask_mode=wl.mask_mode,
               kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale, q=wl.q, k_pool=wl.k_pool,
               v_pool=wl.v_pool, block_table=wl.block_table, seq_lens=wl.seq_lens,
               q_indptr=wl.q_indptr, k_scales=wl.k_scales, v_scales=wl.v_scales,
               k_gscale=wl.k_gscale, v_gscale=wl.v_gscale, window_left=wl.window_left, block_k=wl.block_k,
               block_v=wl.block_v, **kw)
