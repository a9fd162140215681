"""GPU parity of the dense block operand (the window's own keys from dense
block_k / block_v tensors, the cache holding the context only) through the C
ABI against the oracle: the attention tolerances of tests/test_gpu_parity.py,
the index/mask trace exactly (a block key counts slot id -(1 + its row)), the
cache slots past each context poisoned with NaN."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W
from test_gpu_parity import VARIANTS, check_close, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


SHAPES = [
    # ctx list, W list, Hq, Hkv, d, mask, page_size, window
    ([1300, 1100, 1601], [9, 9, 9], 32, 8, 128, 1, 16, 0),     # the batched draft's shape (non-causal)
    ([0, 7, 16, 200], [16, 1, 5, 3], 24, 4, 256, 0, 16, 0),   # no cached key at all; a window one key long
    ([517, 33], [12, 16], 16, 2, 64, 0, 32, 0),
    ([2000, 90], [16, 9], 24, 4, 128, 0, 64, 100),             # with a sliding window
]


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_dense_block_parity(shape, variant):
    ctx, win, hq, hkv, d, mask, ps, window = SHAPES[shape]
    wl = W.make_workload("blk", ctx, win, hq, hkv, d, mask, seed=80 + shape, pool_slack=0.2, page_size=ps,
                         window_left=window, dense_block=True, poison_unread=True)
    dw = run_and_check(wl, variant)
    assert dw.plan.problem.dense_block_kv == 1
    run_and_check(wl, variant, force_splits=4, trace=False)
    run_and_check(wl, variant, host_lens=False, trace=False)


def test_dense_block_equals_the_cache_holding_the_same_rows():
    """The same keys through the cache (window rows written into their slots)
    and through the block operand agree to the tolerance (the tiles group the
    keys differently, so not bit for bit)."""
    wl = W.make_workload("blkeq", [700, 41, 0], [9, 16, 4], 24, 4, 256, W.MASK_NON_CAUSAL, seed=84, pool_slack=0.2)
    ind = wl.q_indptr.tolist()
    bk = torch.zeros(wl.total_rows, 4, 256, dtype=torch.bfloat16)
    bv = torch.zeros_like(bk)
    for r in range(wl.num_reqs):
        w = ind[r + 1] - ind[r]
        L = int(wl.seq_lens[r])
        for i in range(w):
            j = L - w + i
            pg = int(wl.block_table[r, j // 16])
            bk[ind[r] + i] = wl.k_pool[pg, :, j % 16]
            bv[ind[r] + i] = wl.v_pool[pg, :, j % 16]
    blk = W.Workload(**{**wl.__dict__, "block_k": bk, "block_v": bv})
    a = sa.DeviceWorkload(wl, "cuda")
    b = sa.DeviceWorkload(blk, "cuda")
    a.run()
    b.run()
    torch.cuda.synchronize()
    o_ref, lse_ref, _ = oracle.run_workload(wl)
    check_close(a.o, a.lse, o_ref, lse_ref)
    check_close(b.o, b.lse, o_ref, lse_ref)


def test_dense_block_plans_and_entry_points_do_not_mix():
    wl = W.make_workload("blkmix", [300], [8], 24, 4, 128, 1, seed=85, dense_block=True)
    dw = sa.DeviceWorkload(wl, "cuda")
    with pytest.raises(sa.SpecAttnError) as e:   # the plain entry point carries no block operand
        sa.spec_attn_run(dw.plan, dw.q, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens, dw.q_indptr, dw.o,
                         dw.lse, dw.workspace)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG
    kn = torch.zeros(wl.total_rows, 4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.SpecAttnError) as e:   # nothing of the window goes into the cache
        sa.spec_attn_append_kv(dw.plan, kn, kn, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens, dw.q_indptr,
                               dw.workspace)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG
    plain = sa.DeviceWorkload(W.make_workload("plain", [300], [8], 24, 4, 128, 1, seed=86), "cuda")
    with pytest.raises(sa.SpecAttnError) as e:   # a plain plan takes no block operand
        sa.spec_attn_run_dense_block(plain.plan, plain.q, dw.block_k, dw.block_v, plain.k_pool, plain.v_pool,
                                     plain.block_table, plain.seq_lens, plain.q_indptr, plain.o, plain.lse,
                                     plain.workspace)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG


def test_dense_block_full_size_draft_sampled():
    """The batched draft workload with its block K/V kept apart: the whole call,
    sampled rows and the trace against the oracle."""
    wl = W.batched_draft(dense_block=True)
    dw = sa.DeviceWorkload(wl, "cuda")
    rng = np.random.default_rng(87)
    sel = np.zeros((wl.total_rows, wl.num_q_heads), dtype=np.uint8)
    sel[rng.integers(0, wl.total_rows, 64), rng.integers(0, wl.num_q_heads, 64)] = 1
    o_ref, lse_ref, tr_ref = oracle.run_workload(wl, row_select=sel, want_trace=True)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    check_close(dw.o, dw.lse, o_ref, lse_ref, sel)
    tr = torch.zeros(wl.total_rows, wl.num_q_heads, 2, dtype=torch.int64, device="cuda")
    dw.run_traced(tr)
    torch.cuda.synchronize()
    m = sel.astype(bool)
    assert np.array_equal(tr.cpu().numpy()[m], tr_ref[m])
