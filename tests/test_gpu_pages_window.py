"""GPU parity for 32- and 64-key pages, pools with a page stride (K and V, and
their NVFP4 scales, interleaved in one allocation) and the causal sliding
window, through the C ABI against the oracle.  Same tolerances and exact
index/mask trace as tests/test_gpu_parity.py; the KV append into such caches
is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W
from test_gpu_parity import VARIANTS, _row_alone, check_close, run_and_check

pytestmark = pytest.mark.gpu

KVS = [W.KV_BF16, W.KV_NVFP4]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


SHAPES = [
    # ctx list, W list, Hq, Hkv, d, mask
    ([517, 16, 0], [16, 3, 5], 24, 4, 256, 0),
    ([1234, 45], [9, 9], 32, 8, 128, 1),
    ([150, 63, 1000], [12, 16, 1], 16, 2, 64, 0),
]


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("kv", KVS)
@pytest.mark.parametrize("page_size", [32, 64])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_larger_pages(shape, page_size, kv, variant):
    ctx, win, hq, hkv, d, mask = SHAPES[shape]
    wl = W.make_workload("pages", ctx, win, hq, hkv, d, mask, kv_dtype=kv, page_size=page_size,
                         seed=60 + shape, pool_slack=0.3)
    run_and_check(wl, variant)
    run_and_check(wl, variant, force_splits=5, trace=False)


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("kv", KVS)
@pytest.mark.parametrize("page_size", [16, 64])
def test_interleaved_pools_with_a_page_stride(page_size, kv, variant):
    wl = W.make_workload("inter", [700, 33, 2000], [16, 4, 9], 24, 4, 128, 0, kv_dtype=kv, page_size=page_size,
                         seed=63, pool_slack=0.2)
    dw = run_and_check(wl, variant, interleave=True)
    assert dw.plan.problem.kv_page_stride == 2 * dw.k_pool[0].numel() * dw.k_pool.element_size()


WINDOWS = [1, 17, 64, 300, 5000]


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("kv", KVS)
@pytest.mark.parametrize("window", WINDOWS)
def test_sliding_window(window, kv, variant):
    wl = W.make_workload("win", [2000, 45, 0, 700], [16, 9, 4, 1], 24, 4, 256, 0, kv_dtype=kv, seed=64,
                         pool_slack=0.2, window_left=window)
    run_and_check(wl, variant)
    run_and_check(wl, variant, force_splits=7, trace=False)
    run_and_check(wl, variant, host_lens=False, trace=False)


def test_window_narrows_the_grid():
    """With a 256-key window at ctx 16000 the plan splits only the window's
    keys (plus alignment), not the whole cache."""
    wl = W.make_workload("wgrid", [16000], [16], 24, 4, 256, 0, seed=65, window_left=256)
    dw = sa.DeviceWorkload(wl, "cuda")
    span = 16 + 256 - 1 + 63
    assert dw.plan.info["max_splits"] * dw.plan.info["keys_per_split"] < span + dw.plan.info["keys_per_split"]
    o_ref, lse_ref, _ = oracle.run_workload(wl)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    check_close(dw.o, dw.lse, o_ref, lse_ref)


@pytest.mark.parametrize("kv,page_size,window,fixed",
                         [(W.KV_BF16, 32, 100, 64), (W.KV_BF16, 64, 700, 256), (W.KV_NVFP4, 32, 300, 128)])
def test_w_invariant_with_window_and_larger_pages(kv, page_size, window, fixed):
    """Exactness rule with a sliding window and 32/64-key pages: every row of
    the window equals its own W = 1 call bit for bit."""
    wl = W.make_workload("winvw", [2300, 700], [16, 9], 24, 4, 256, 0, kv_dtype=kv, seed=66, pool_slack=0.2,
                         page_size=page_size, window_left=window)
    dw = sa.DeviceWorkload(wl, "cuda", w_invariant=1, fixed_keys_per_split=fixed)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    o_ref, lse_ref, _ = oracle.run_workload(wl)
    check_close(dw.o, dw.lse, o_ref, lse_ref)
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        for i in range(ind[r + 1] - ind[r]):
            o1, l1 = _row_alone(wl, dw, r, i, fixed)
            assert torch.equal(dw.o[ind[r] + i], o1) and torch.equal(dw.lse[ind[r] + i], l1), (r, i)


def _bytes(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


@pytest.mark.parametrize("kv", KVS)
@pytest.mark.parametrize("page_size,interleave", [(32, False), (64, True), (16, True)])
def test_append_into_larger_and_strided_pages(kv, page_size, interleave):
    wl = W.make_workload("appps", [100, 31, 0], [16, 9, 3], 24, 4, 128, 0, kv_dtype=kv, seed=67, pool_slack=0.3,
                         page_size=page_size, nvfp4_gscale=2.0 ** -3)
    # N(0, 1) rows: the attention check below uses absolute tolerances
    kn, vn = W.window_kv_rows(wl.total_rows, 4, 128, seed=68, mix=False)
    ref = oracle.append_kv(num_kv_heads=4, head_dim=128, page_size=page_size, kv_dtype=kv, k_new=kn, v_new=vn,
                           k_pool=wl.k_pool, v_pool=wl.v_pool, k_scales=wl.k_scales, v_scales=wl.v_scales,
                           k_gscale=wl.k_gscale, v_gscale=wl.v_gscale, block_table=wl.block_table,
                           seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    dw = sa.DeviceWorkload(wl, "cuda", append_rows=(kn, vn), mode="run_append", interleave=interleave)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    for got, want in zip((dw.k_pool, dw.v_pool, dw.k_scales, dw.v_scales), ref):
        if want is not None:
            assert np.array_equal(_bytes(got), want.view(np.uint8))
    if interleave:
        # the other half of each page is the other tensor, untouched by position
        assert torch.equal(dw.kv_storage[:, 0], dw.k_pool) and torch.equal(dw.kv_storage[:, 1], dw.v_pool)
    kp, vp, ks, vs = ref
    o_ref, lse_ref, _ = oracle.run(num_q_heads=24, num_kv_heads=4, head_dim=128, page_size=page_size,
                                   num_pages=wl.num_pages, mask_mode=0, kv_dtype=kv, sm_scale=wl.sm_scale, q=wl.q,
                                   k_pool=kp, v_pool=vp, k_scales=ks, v_scales=vs, k_gscale=wl.k_gscale,
                                   v_gscale=wl.v_gscale, block_table=wl.block_table, seq_lens=wl.seq_lens,
                                   q_indptr=wl.q_indptr)
    check_close(dw.o, dw.lse, o_ref, lse_ref)


def test_full_size_window_and_64_key_pages_sampled():
    """The 16K verify shape with 64-key pages and a 4096-key window: the whole
    call on the GPU, sampled (row, head) pairs and the trace against the oracle."""
    wl = W.make_workload("verify_ctx16384_w16_ps64", [16384], 16, 24, 4, 256, W.MASK_CAUSAL_IN_BLOCK, seed=0,
                         page_size=64, pool_pages=320, window_left=4096)
    dw = sa.DeviceWorkload(wl, "cuda")
    rng = np.random.default_rng(69)
    sel = np.zeros((16, 24), dtype=np.uint8)
    sel[rng.integers(0, 16, 24), rng.integers(0, 24, 24)] = 1
    sel[0, :] = 1
    o_ref, lse_ref, tr_ref = oracle.run_workload(wl, row_select=sel, want_trace=True)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    check_close(dw.o, dw.lse, o_ref, lse_ref, sel)
    tr = torch.zeros(16, 24, 2, dtype=torch.int64, device="cuda")
    dw.run_traced(tr)
    torch.cuda.synchronize()
    m = sel.astype(bool)
    assert np.array_equal(tr.cpu().numpy()[m], tr_ref[m])
