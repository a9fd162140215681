"""The allocation-free entry point, spec_attn_run_noalloc.

Some callers cannot allocate device memory at the point where they run
attention (inside an allocator hook or host callback, or a plugin that is
handed only its input and output buffers), so they cannot supply the
workspace spec_attn_run needs.  spec_attn_run_noalloc takes its scratch from a
fixed array inside the library instead.  This test calls it through the C ABI
twice in a row and checks each result against spec_attn_run with a normal
workspace, within the parity tolerances the other GPU tests use.  It lives in
its own file, collected last, and passes alone or after the other tests.
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


@pytest.mark.parametrize("variant", [sa.SPEC_ATTN_VARIANT_CUDA_CORE, sa.SPEC_ATTN_VARIANT_TCGEN05])
def test_noalloc_matches_run_on_two_calls(lib, variant):
    wl = W.make_workload("noalloc", [3000, 700, 45], [16, 9, 4], 24, 4, 256,
                         W.MASK_CAUSAL_IN_BLOCK, seed=31, pool_slack=0.1)
    dw = sa.DeviceWorkload(wl, "cuda", force_splits=5, kernel_variant=variant)
    assert dw.plan.info["uses_merge"] == 1            # the split partials need scratch
    assert dw.plan.workspace_bytes <= (32 << 20)
    dw.run()
    torch.cuda.synchronize()
    o_ref, lse_ref = dw.o.clone(), dw.lse.clone()

    stream = torch.cuda.current_stream()
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = lib.spec_attn_run_noalloc(
            dw.plan.handle, _ptr(dw.q), _ptr(dw.k_pool), _ptr(dw.v_pool), None, None,
            ctypes.c_float(1.0), ctypes.c_float(1.0), _ptr(dw.block_table), _ptr(dw.seq_lens),
            _ptr(dw.q_indptr), _ptr(o), _ptr(lse), ctypes.c_void_p(stream.cuda_stream))
        assert st == sa.SPEC_ATTN_OK, sa.status_string(st)
        torch.cuda.synchronize()
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
