"""The allocation-free entry point, spec_attn_run_noalloc.

Some callers cannot allocate device memory at the point where they run
attention (inside an allocator hook or host callback, or a plugin that is
handed only its input and output buffers), so they cannot supply the
workspace spec_attn_run needs.  spec_attn_run_noalloc takes its scratch from a
fixed array inside the library instead.  These tests call it through the C ABI
(and once through the Python wrapper) two calls in a row, and check:

- each result has the same bits as spec_attn_run with a normal workspace (same
  plan, same kernels, same split count), and lies within the parity
  tolerances of the other GPU tests;
- the free device memory does not change across the calls: nothing is
  allocated;
- a plan needing more scratch than the array holds is rejected, and a call
  rejected by a host check writes nothing;
- a device-side failure (the stall hook makes every bounded wait run out) is
  reported by spec_attn_noalloc_check_device_status.

The file is collected last, and passes alone or after the other tests.
"""
import ctypes

import pytest
import torch

import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 1e-2, 1e-3, 1e-4


@pytest.fixture(scope="module")
def lib():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    torch.cuda.set_device(0)
    return sa.load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(o, lse, o_ref, lse_ref):
    err = (o.float() - o_ref.float()).abs()
    assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN
    rel = (lse - lse_ref).abs() / lse_ref.abs().clamp(min=1.0)
    assert rel.max().item() <= LSE_REL


def _noalloc_c(lib, dw, o, lse, stream):
    return lib.spec_attn_run_noalloc(
        dw.plan.handle, _ptr(dw.q), _ptr(dw.k_pool), _ptr(dw.v_pool), _ptr(dw.k_scales), _ptr(dw.v_scales),
        ctypes.c_float(dw.wl.k_gscale), ctypes.c_float(dw.wl.v_gscale), _ptr(dw.block_table), _ptr(dw.seq_lens),
        _ptr(dw.q_indptr), _ptr(o), _ptr(lse), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("variant,kv", [(sa.SPEC_ATTN_VARIANT_CUDA_CORE, W.KV_BF16),
                                        (sa.SPEC_ATTN_VARIANT_TCGEN05, W.KV_BF16),
                                        (sa.SPEC_ATTN_VARIANT_TCGEN05, W.KV_NVFP4)])
def test_noalloc_matches_run_on_two_calls(lib, variant, kv):
    wl = W.make_workload("noalloc", [3000, 700, 45], [16, 9, 4], 24, 4, 256,
                         W.MASK_CAUSAL_IN_BLOCK, kv_dtype=kv, seed=31, pool_slack=0.1)
    dw = sa.DeviceWorkload(wl, "cuda", force_splits=5, kernel_variant=variant)
    assert dw.plan.info["uses_merge"] == 1            # the split partials need scratch
    assert dw.plan.workspace_bytes <= (32 << 20)
    dw.run()
    torch.cuda.synchronize()
    o_ref, lse_ref = dw.o.clone(), dw.lse.clone()

    stream = torch.cuda.current_stream()
    outs = [(torch.full_like(o_ref, float("nan")), torch.full_like(lse_ref, float("nan"))) for _ in range(3)]
    # first call: looks up the array's address; then measure around two more
    assert _noalloc_c(lib, dw, *outs[0], stream) == sa.SPEC_ATTN_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    st = _noalloc_c(lib, dw, *outs[1], stream)
    assert st == sa.SPEC_ATTN_OK, sa.status_string(st)
    sa.spec_attn_run_noalloc(dw.plan, dw.q, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens, dw.q_indptr,
                             *outs[2], dw.k_scales, dw.v_scales, dw.wl.k_gscale, dw.wl.v_gscale)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "spec_attn_run_noalloc changed the free device memory"
    assert sa.spec_attn_noalloc_check_device_status() == 0
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
        _close(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_plans_larger_than_its_scratch(lib):
    # 513 splits x 16 rows x 32 heads x (256 fp16 values + lse + scale) = 68 MB of partials > 32 MiB
    wl = W.make_workload("big", [32768], [16], 32, 2, 256, W.MASK_NON_CAUSAL, seed=32)
    dw = sa.DeviceWorkload(wl, "cuda", force_splits=512)
    assert dw.plan.workspace_bytes > (32 << 20)
    st = lib.spec_attn_run_noalloc(
        dw.plan.handle, _ptr(dw.q), _ptr(dw.k_pool), _ptr(dw.v_pool), None, None,
        ctypes.c_float(1.0), ctypes.c_float(1.0), _ptr(dw.block_table), _ptr(dw.seq_lens),
        _ptr(dw.q_indptr), _ptr(dw.o), _ptr(dw.lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == sa.SPEC_ATTN_E_WORKSPACE_TOO_SMALL


def test_noalloc_reports_a_device_failure_and_rejected_calls_write_nothing(lib):
    wl = W.make_workload("stall", [300, 40], [8, 3], 8, 2, 128, W.MASK_CAUSAL_IN_BLOCK, seed=95)
    dev = "cuda"
    plan = sa.spec_attn_plan_create(
        num_reqs=wl.num_reqs, total_q_rows=wl.total_rows, max_w=wl.max_w, num_q_heads=8, num_kv_heads=2,
        head_dim=128, num_pages=wl.num_pages, block_table_stride=int(wl.block_table.shape[1]),
        max_seq_len=wl.max_seq_len, mask_mode=wl.mask_mode, kernel_variant=sa.SPEC_ATTN_VARIANT_TCGEN05,
        seq_lens=wl.seq_lens, q_indptr=wl.q_indptr, test_stall=1)
    t = {n: getattr(wl, n).to(dev) for n in ("q", "k_pool", "v_pool", "block_table", "seq_lens", "q_indptr")}
    o = torch.zeros(wl.total_rows, 8, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(wl.total_rows, 8, dtype=torch.float32, device=dev)
    # every bounded wait of the stalled call runs out (about a second): the bit comes back
    sa.spec_attn_run_noalloc(plan, t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                             t["q_indptr"], o, lse)
    torch.cuda.synchronize()
    assert sa.spec_attn_noalloc_check_device_status() == sa.SPEC_ATTN_DEV_WAIT_TIMEOUT
    assert sa.spec_attn_noalloc_check_device_status() == 0          # read and cleared
    # a call that a host check rejects (misaligned output) launches nothing and
    # leaves the status word alone
    sa.spec_attn_run_noalloc(plan, t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                             t["q_indptr"], o, lse)
    torch.cuda.synchronize()
    o_before = o.clone()
    bad_o = ctypes.c_void_p(o.data_ptr() + 2)
    st = lib.spec_attn_run_noalloc(
        plan.handle, _ptr(t["q"]), _ptr(t["k_pool"]), _ptr(t["v_pool"]), None, None, ctypes.c_float(1.0),
        ctypes.c_float(1.0), _ptr(t["block_table"]), _ptr(t["seq_lens"]), _ptr(t["q_indptr"]), bad_o, _ptr(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == sa.SPEC_ATTN_E_INVALID_ARG
    torch.cuda.synchronize()
    # bitwise (the stalled call leaves NaN, which equal() would call different)
    assert torch.equal(o.view(torch.int16), o_before.view(torch.int16))
    assert sa.spec_attn_noalloc_check_device_status() == sa.SPEC_ATTN_DEV_WAIT_TIMEOUT
