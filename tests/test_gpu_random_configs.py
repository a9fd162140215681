"""Seeded random configurations across every option at once -- KV dtype, head
dim, group size, ragged windows (with empty ones), both masks, page sizes,
page strides, sliding windows, the dense block operand, forced splits and both
kernels -- each through the C ABI against the oracle (the attention
tolerances of tests/test_gpu_parity.py and the index/mask trace exactly).
Options that do not combine (NVFP4 with the dense block operand, a window
with the non-causal mask) are drawn out, not skipped."""
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


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    kv = int(rng.integers(0, 2))
    d = int(rng.choice([64, 128, 256]))
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 6, 8, 12, 16]))
    P = int(rng.integers(1, 5))
    win = [int(rng.integers(0, 17)) for _ in range(P)]
    if max(win) == 0:
        win[0] = 1
    ctx = [int(rng.choice([0, int(rng.integers(1, 64)), int(rng.integers(64, 3000))])) for _ in range(P)]
    mask = int(rng.integers(0, 2))
    page = int(rng.choice([16, 32, 64]))
    window = int(rng.choice([0, 0, int(rng.integers(1, 40)), int(rng.integers(40, 2000))])) if mask == 0 else 0
    dense = kv == 0 and bool(rng.integers(0, 4) == 0)
    interleave = bool(rng.integers(0, 3) == 0)
    variant = int(rng.choice([sa.SPEC_ATTN_VARIANT_CUDA_CORE, sa.SPEC_ATTN_VARIANT_TCGEN05]))
    splits = int(rng.choice([0, 0, int(rng.integers(1, 9))]))
    return dict(kv=kv, d=d, hkv=hkv, g=g, ctx=ctx, win=win, mask=mask, page=page, window=window, dense=dense,
                interleave=interleave, variant=variant, splits=splits)


@pytest.mark.parametrize("seed", range(64))
def test_random_configuration(seed):
    c = _draw(seed)
    wl = W.make_workload(f"rand{seed}", c["ctx"], c["win"], c["hkv"] * c["g"], c["hkv"], c["d"], c["mask"],
                         kv_dtype=c["kv"], page_size=c["page"], seed=2000 + seed, pool_slack=0.25,
                         window_left=c["window"], dense_block=c["dense"], poison_unread=True)
    dw = sa.DeviceWorkload(wl, "cuda", force_splits=c["splits"], kernel_variant=c["variant"],
                           interleave=c["interleave"])
    o_ref, lse_ref, tr_ref = oracle.run_workload(wl, want_trace=True)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0, c
    check_close(dw.o, dw.lse, o_ref, lse_ref)
    tr = torch.zeros(wl.total_rows, wl.num_q_heads, 2, dtype=torch.int64, device="cuda")
    dw.run_traced(tr)
    torch.cuda.synchronize()
    assert np.array_equal(tr.cpu().numpy(), tr_ref), c
