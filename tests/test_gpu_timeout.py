"""The time-out path of the tensor-core kernel's bounded waits, made to run
out without any fault: with the test_stall hook the K producer issues
nothing, every consumer's wait gives up after about a second, the CTA frees
its tensor memory and the call raises SPEC_ATTN_DEV_WAIT_TIMEOUT in the
device-status word.  A full-grid call afterwards (tensor memory allocated on
every SM) must still be correct: the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W
from test_gpu_parity import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_NVFP4])
def test_a_wait_that_runs_out_sets_the_status_and_leaves_the_context_usable(kv):
    wl = W.make_workload("stall", [300, 40], [8, 3], 8, 2, 128, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=kv, seed=95)
    dev = "cuda"
    plan = sa.spec_attn_plan_create(
        num_reqs=wl.num_reqs, total_q_rows=wl.total_rows, max_w=wl.max_w, num_q_heads=8, num_kv_heads=2,
        head_dim=128, num_pages=wl.num_pages, block_table_stride=int(wl.block_table.shape[1]),
        max_seq_len=wl.max_seq_len, mask_mode=wl.mask_mode, kv_dtype=kv,
        kernel_variant=sa.SPEC_ATTN_VARIANT_TCGEN05, seq_lens=wl.seq_lens, q_indptr=wl.q_indptr, test_stall=1)
    t = {n: getattr(wl, n).to(dev) if getattr(wl, n) is not None else None
         for n in ("q", "k_pool", "v_pool", "k_scales", "v_scales", "block_table", "seq_lens", "q_indptr")}
    o = torch.zeros(wl.total_rows, 8, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(wl.total_rows, 8, dtype=torch.float32, device=dev)
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    sa.spec_attn_run(plan, t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], t["q_indptr"], o, lse,
                     ws, t["k_scales"], t["v_scales"], wl.k_gscale, wl.v_gscale)
    torch.cuda.synchronize()
    assert sa.spec_attn_check_device_status(ws) == sa.SPEC_ATTN_DEV_WAIT_TIMEOUT
    # every SM runs a CTA that allocates tensor memory: none was left held
    full = W.verify_sweep(16)
    dw = sa.DeviceWorkload(full, dev)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    sel = np.zeros((16, 24), dtype=np.uint8)
    sel[15, :] = 1
    sel[0, :3] = 1
    o_ref, lse_ref, _ = oracle.run_workload(full, row_select=sel)
    check_close(dw.o, dw.lse, o_ref, lse_ref, sel)


def test_the_stall_hook_is_tensor_core_only():
    wl = W.make_workload("stall2", [100], [4], 8, 2, 128, 0, seed=96)
    with pytest.raises(sa.SpecAttnError) as e:
        sa.spec_attn_plan_create(num_reqs=1, total_q_rows=4, max_w=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 num_pages=wl.num_pages, block_table_stride=int(wl.block_table.shape[1]),
                                 max_seq_len=104, test_stall=1)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG
