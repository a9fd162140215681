"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Tolerances (bf16 output, fp32 accumulation): |dO| <= 1e-2 max and <= 1e-3
mean over the compared elements; |dLSE| <= 1e-4 * max(1, |LSE|).  Index and
mask decisions are compared bit-exactly through the traced run (count of
keys let into each row's softmax and the sum of their physical slot ids).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 1e-2, 1e-3, 1e-4
VARIANTS = [sa.SPEC_ATTN_VARIANT_AUTO, sa.SPEC_ATTN_VARIANT_CUDA_CORE, sa.SPEC_ATTN_VARIANT_TCGEN05]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


def check_close(o_gpu, lse_gpu, o_ref, lse_ref, sel=None):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    if sel is not None:
        m = sel.astype(bool)
        o, o_ref, lse, lse_ref = o[m], o_ref[m], lse[m], lse_ref[m]
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"max |dO| {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"mean |dO| {err.mean():.3e}"
    rel = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert rel.max() <= LSE_REL, f"max rel dLSE {rel.max():.3e}"
    return err.max(), rel.max()


def make_dw(wl, variant=0, **kw):
    try:
        return sa.DeviceWorkload(wl, "cuda", kernel_variant=variant, **kw)
    except sa.SpecAttnError as e:
        if e.status == sa.SPEC_ATTN_E_UNSUPPORTED and variant != sa.SPEC_ATTN_VARIANT_AUTO:
            pytest.skip("variant does not support this shape")
        raise


def run_and_check(wl, variant=0, force_splits=0, trace=True, sel=None, host_lens=True, **kw):
    """Untraced run vs the oracle, then (if trace) the traced run: outputs vs the
    oracle again and the index/mask trace bit-exactly."""
    dw = make_dw(wl, variant, force_splits=force_splits, host_lens=host_lens, **kw)
    o_ref, lse_ref, tr_ref = oracle.run_workload(wl, row_select=sel, want_trace=trace)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    check_close(dw.o, dw.lse, o_ref, lse_ref, sel)
    if trace:
        dw.o.zero_()
        dw.lse.zero_()
        tr = torch.zeros(wl.total_rows, wl.num_q_heads, 2, dtype=torch.int64, device="cuda")
        dw.run_traced(tr)
        torch.cuda.synchronize()
        assert dw.device_status() == 0
        check_close(dw.o, dw.lse, o_ref, lse_ref, sel)
        t = tr.cpu().numpy()
        if sel is not None:
            assert np.array_equal(t[sel.astype(bool)], tr_ref[sel.astype(bool)])
        else:
            assert np.array_equal(t, tr_ref)
    return dw


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_repeated_runs_are_bitwise_stable_across_interleaved_workloads(variant):
    """Runs of one plan give identical bits however the previous launches (other
    shapes, other head_dims) left shared memory and TMEM."""
    shapes = [([1800, 900, 60], [9, 9, 9], 32, 8, 128, 1), ([300], [16], 64, 8, 128, 0),
              ([100], [9], 32, 8, 64, 0), ([700], [16], 24, 4, 256, 0), ([40], [3], 8, 8, 128, 0)]
    dws = []
    for k, (ctx, win, hq, hkv, d, mask) in enumerate(shapes):
        wl = W.make_workload(f"i{k}", ctx, win, hq, hkv, d, mask, seed=40 + k, pool_slack=0.1)
        dws.append((wl, make_dw(wl, variant)))
    first = []
    for wl, dw in dws:
        dw.run()
        torch.cuda.synchronize()
        first.append((dw.o.clone(), dw.lse.clone()))
        o_ref, lse_ref, _ = oracle.run_workload(wl)
        check_close(dw.o, dw.lse, o_ref, lse_ref)
    for rep in range(3):
        for (wl, dw), (o0, l0) in zip(reversed(dws), reversed(first)):
            dw.o.zero_()
            dw.run()
            torch.cuda.synchronize()
            assert torch.equal(dw.o, o0) and torch.equal(dw.lse, l0)


# --------------------------------------------------------------------------- #
# Small shapes that the oracle finishes in seconds (several splits, ragged tails)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny(variant):
    run_and_check(W.tiny(0), variant)


SHAPES = [
    # ctx list, W list, Hq, Hkv, d, mask
    ([300], [1], 8, 8, 64, 0),
    ([517, 16], [16, 3], 24, 4, 256, 0),
    ([77, 1000, 0], [8, 9, 5], 24, 4, 256, 0),
    ([1234, 45, 700], [9, 9, 9], 32, 8, 128, 1),
    ([150, 63], [12, 16], 16, 1, 64, 1),
    ([801], [16], 64, 4, 128, 0),          # G = 16, W = 16: 256 rows per KV head
    ([129, 64, 255], [2, 1, 7], 8, 1, 256, 1),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=[f"s{i}" for i in range(len(SHAPES))])
def test_random_shapes_bf16(shape, variant):
    ctx, win, hq, hkv, d, mask = shape
    wl = W.make_workload("shape", ctx, win, hq, hkv, d, mask, seed=len(ctx) + d, pool_slack=0.2)
    run_and_check(wl, variant)


NVFP4_SHAPES = SHAPES[1:5] + [([150, 63, 1000], [12, 16, 1], 16, 2, 64, 0)]   # d 64 on the tensor cores


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", NVFP4_SHAPES, ids=[f"s{i}" for i in range(len(NVFP4_SHAPES))])
def test_random_shapes_nvfp4(shape, variant):
    ctx, win, hq, hkv, d, mask = shape
    wl = W.make_workload("fp4", ctx, win, hq, hkv, d, mask, kv_dtype=W.KV_NVFP4, seed=3,
                         pool_slack=0.2)
    run_and_check(wl, variant)


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_count_invariance(splits, variant):
    wl = W.make_workload("splits", [2000, 333], [8, 16], 24, 4, 256, 0, seed=5, pool_slack=0.1)
    dw = run_and_check(wl, variant, force_splits=splits, trace=True)
    if splits:
        assert dw.plan.info["max_splits"] <= splits


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_empty_windows_and_zero_context(variant):
    wl = W.make_workload("edge", [0, 40, 0, 5], [1, 0, 16, 0], 8, 2, 64, 0, seed=6)
    run_and_check(wl, variant)


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_plan_without_host_lengths(variant):
    wl = W.make_workload("nohost", [900, 31], [4, 11], 12, 2, 128, 1, seed=7, pool_slack=0.2)
    run_and_check(wl, variant, host_lens=False)


# --------------------------------------------------------------------------- #
# Invariants on the GPU
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_page_permutation_is_bitwise_invariant(variant):
    wl = W.make_workload("perm", [1500, 200], [16, 8], 24, 4, 256, 0, seed=8, pool_slack=0.3)
    a = make_dw(wl, variant)
    a.run()
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(wl.num_pages, generator=g)
    inv = torch.argsort(perm)
    bt2 = torch.where(wl.block_table >= 0, perm[wl.block_table.clamp(min=0).long()].to(torch.int32),
                      wl.block_table)
    wl2 = W.Workload(**{**wl.__dict__, "k_pool": wl.k_pool[inv], "v_pool": wl.v_pool[inv],
                        "block_table": bt2})
    b = make_dw(wl2, variant)
    assert a.plan.info == b.plan.info
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_NVFP4])
def test_poisoned_unread_slots_change_nothing(kv, variant):
    kw = dict(ctx_lens=[700, 41], windows=[9, 4], num_q_heads=24, num_kv_heads=4, head_dim=256,
              mask_mode=1, kv_dtype=kv, seed=9, pool_slack=0.4)
    a = make_dw(W.make_workload("clean", **kw), variant)
    b = make_dw(W.make_workload("poison", poison_unread=True, **kw), variant)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)
    assert torch.isfinite(b.o.float()).all()


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_causal_row_i_matches_decode_at_ctx_plus_i_plus_1(variant):
    ctx, Wn = 1000, 12
    wl = W.make_workload("rowwise", [ctx], Wn, 24, 4, 256, 0, seed=10)
    full = make_dw(wl, variant)
    full.run()
    for i in (0, 5, 11):
        one = W.Workload(**{**wl.__dict__, "q": wl.q[i:i + 1].clone(),
                            "seq_lens": torch.tensor([ctx + i + 1], dtype=torch.int32),
                            "q_indptr": torch.tensor([0, 1], dtype=torch.int32)})
        d1 = make_dw(one, variant)
        d1.run()
        torch.cuda.synchronize()
        diff = (d1.o[0].float() - full.o[i].float()).abs().max().item()
        assert diff <= O_MAX
        assert torch.allclose(d1.lse[0], full.lse[i], rtol=LSE_REL, atol=LSE_REL)


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_non_causal_and_causal_agree_on_last_row(variant):
    kw = dict(ctx_lens=[333, 1200], windows=[7, 16], num_q_heads=8, num_kv_heads=2, head_dim=128,
              seed=11)
    c = make_dw(W.make_workload("c", mask_mode=0, **kw), variant)
    n = make_dw(W.make_workload("n", mask_mode=1, **kw), variant)
    c.run()
    n.run()
    torch.cuda.synchronize()
    for last in (6, 22):
        assert torch.equal(c.o[last], n.o[last]) and torch.equal(c.lse[last], n.lse[last])


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_zero_queries_count_visible_keys_exactly(variant):
    wl = W.make_workload("q0", [1000, 77], [16, 5], 24, 4, 256, 0, seed=12, q_mode="zero")
    dw = run_and_check(wl, variant, trace=False)
    lse = dw.lse.cpu().numpy().astype(np.float64)
    for r, (c, w) in enumerate(zip([1000, 77], [16, 5])):
        row0 = int(wl.q_indptr[r])
        for i in range(w):
            assert np.all(np.round(np.exp(lse[row0 + i])) == c + i + 1)


@pytest.mark.parametrize("kv", [W.KV_BF16])
@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_constant_values_come_back_bit_exactly(kv, variant):
    wl = W.make_workload("vconst", [2100, 9], [16, 3], 24, 4, 256, 0, seed=13, v_mode="const")
    dw = make_dw(wl, variant)
    dw.run()
    torch.cuda.synchronize()
    v = wl.v_pool[int(wl.block_table[0, 0]), :, 0, :]  # [Hkv, d], same for every key
    want = v.repeat_interleave(6, dim=0)                 # query head h -> KV head h // 6
    got = dw.o.cpu()
    for row in range(wl.total_rows):
        assert torch.equal(got[row], want)


# --------------------------------------------------------------------------- #
# Compact block order (tensor-core kernel, 2..64 requests of uneven lengths)
# --------------------------------------------------------------------------- #
def _ragged(name, num_reqs, seed, **kw):
    g = np.random.default_rng(seed)
    ctx = g.integers(0, 900, size=num_reqs).tolist()
    ws = g.integers(1, 17, size=num_reqs).tolist()
    return W.make_workload(name, ctx, ws, 24, 4, 128, W.MASK_CAUSAL_IN_BLOCK, seed=seed, pool_slack=0.1, **kw)


def test_compact_order_over_two_request_chunks_reports_a_bad_request():
    """40 requests (two 32-request chunks of the block-order scan): the grid is
    one-dimensional, every row matches the oracle, and a request made invalid
    on the device (length below its window) sets the status bit -- reported by
    block 0 from the second chunk -- while the other requests' rows stay right."""
    wl = _ragged("compact40", 40, 81)
    dw = make_dw(wl, sa.SPEC_ATTN_VARIANT_TCGEN05, force_splits=3)
    assert dw.plan.info["grid_y"] == 1 and dw.plan.info["grid_z"] == 1
    o_ref, lse_ref, _ = oracle.run_workload(wl, want_trace=False)
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    check_close(dw.o, dw.lse, o_ref, lse_ref)
    bad = 37
    a, b = int(wl.q_indptr[bad]), int(wl.q_indptr[bad + 1])
    dw.seq_lens[bad] = b - a - 1            # shorter than its own window
    dw.o.zero_()
    dw.lse.zero_()
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() & sa.SPEC_ATTN_DEV_BAD_SEQ_LEN
    keep = np.ones((wl.total_rows, wl.num_q_heads), dtype=np.uint8)
    keep[a:b] = 0
    check_close(dw.o, dw.lse, o_ref, lse_ref, sel=keep)


def test_more_than_64_requests_keep_the_three_dimensional_grid():
    wl = _ragged("grid70", 70, 82)
    dw = run_and_check(wl, sa.SPEC_ATTN_VARIANT_TCGEN05, trace=True)
    assert dw.plan.info["grid_z"] == 70


def test_even_batches_keep_the_three_dimensional_grid():
    wl = W.make_workload("even", [700] * 4, 8, 24, 4, 128, W.MASK_CAUSAL_IN_BLOCK, seed=83)
    dw = run_and_check(wl, sa.SPEC_ATTN_VARIANT_TCGEN05, trace=False)
    assert dw.plan.info["grid_z"] == 4


# --------------------------------------------------------------------------- #
# Device-side checks: bad inputs become a status bit, never a fault
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_bad_page_id_sets_status_and_keeps_going(variant):
    wl = W.make_workload("badpage", [200], [4], 8, 2, 128, 0, seed=14)
    dw = make_dw(wl, variant)
    dw.block_table[0, 3] = wl.num_pages + 1000
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() & sa.SPEC_ATTN_DEV_BAD_PAGE
    dw.block_table.copy_(wl.block_table.cuda())
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_seq_len_above_plan_sets_status(variant):
    wl = W.make_workload("badlen", [200, 50], [4, 4], 8, 2, 128, 0, seed=15, pool_slack=1.0,
                         bt_stride=40)
    dw = make_dw(wl, variant)
    dw.seq_lens[1] = wl.max_seq_len + 100     # above the plan's max_seq_len
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() & sa.SPEC_ATTN_DEV_BAD_SEQ_LEN
    dw.seq_lens[1] = 2                         # below its window
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() & sa.SPEC_ATTN_DEV_BAD_SEQ_LEN


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_window_wider_than_plan_sets_status(variant):
    wl = W.make_workload("badw", [100, 100], [4, 4], 8, 2, 128, 0, seed=16)
    dw = make_dw(wl, variant)
    dw.q_indptr.copy_(torch.tensor([0, 1, 8], dtype=torch.int32))  # W = 1 and 7 > max_w 4
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() & sa.SPEC_ATTN_DEV_BAD_WINDOW


def test_run_rejects_small_workspace_and_misalignment():
    wl = W.make_workload("ws", [3000], [8], 24, 4, 256, 0, seed=17)
    dw = make_dw(wl, 0)
    assert dw.plan.workspace_bytes > 256
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(sa.SpecAttnError) as ei:
        sa.spec_attn_run(dw.plan, dw.q, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens,
                         dw.q_indptr, dw.o, dw.lse, small)
    assert ei.value.status == sa.SPEC_ATTN_E_WORKSPACE_TOO_SMALL
    qv = torch.zeros(dw.q.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + dw.q.numel()].view_as(dw.q)
    with pytest.raises(sa.SpecAttnError) as ei:
        sa.spec_attn_run(dw.plan, qv, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens,
                         dw.q_indptr, dw.o, dw.lse, dw.workspace)
    assert ei.value.status == sa.SPEC_ATTN_E_INVALID_ARG


# --------------------------------------------------------------------------- #
# CUDA graph capture and replay
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_graph_capture_replay_matches_eager(variant):
    wl = W.make_workload("graph", [1800, 900, 60], [9, 9, 9], 32, 8, 128, 1, seed=18, pool_slack=0.1)
    dw = make_dw(wl, variant)
    dw.run()
    torch.cuda.synchronize()
    o_eager = dw.o.clone()
    dw.o.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.run(stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dw.o, o_eager)
    # new lengths (<= the plan's max) and replay again
    dw.seq_lens.copy_(torch.tensor([1000, 900, 60], dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    wl2 = W.Workload(**{**wl.__dict__, "seq_lens": torch.tensor([1000, 900, 60], dtype=torch.int32)})
    o_ref, lse_ref, _ = oracle.run_workload(wl2)
    check_close(dw.o, dw.lse, o_ref, lse_ref)


# --------------------------------------------------------------------------- #
# Full-size workloads in the bench's launch configuration, sampled rows
# --------------------------------------------------------------------------- #
def _sample(wl, n_rows=6, seed=0):
    g = np.random.default_rng(seed)
    sel = np.zeros((wl.total_rows, wl.num_q_heads), dtype=np.uint8)
    rows = set()
    for r in range(wl.num_reqs):  # first and last row of every window
        a, b = int(wl.q_indptr[r]), int(wl.q_indptr[r + 1])
        if b > a:
            rows.update([a, b - 1])
    rows.update(g.integers(0, wl.total_rows, size=n_rows).tolist())
    for row in rows:
        sel[row, g.integers(0, wl.num_q_heads, size=3)] = 1
        sel[row, 0] = 1
        sel[row, wl.num_q_heads - 1] = 1
    return sel


FULL = [
    ("verify_sweep_w1", lambda: W.verify_sweep(1)),
    ("verify_sweep_w8", lambda: W.verify_sweep(8)),
    ("verify_sweep_w16", lambda: W.verify_sweep(16)),
    ("long_verify_w8", lambda: W.long_verify(8)),
    ("long_verify_w9", lambda: W.long_verify(9)),
    ("long_verify_w12", lambda: W.long_verify(12)),
    ("long_verify_w16", lambda: W.long_verify(16)),
    ("batched_draft", lambda: W.batched_draft()),
    ("nvfp4", lambda: W.nvfp4()),
]


@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("name,make", FULL, ids=[n for n, _ in FULL])
def test_full_size_sampled(name, make, variant):
    wl = make()
    run_and_check(wl, variant, trace=True, sel=_sample(wl))


# Every row and head of the full-size single-GPU workloads (the 64K ones stay
# sampled above: the oracle takes minutes there), in the bench's launch
# configuration (tensor-core kernel, heuristic split count).
EVERY_ROW = [
    ("verify_sweep_w1", lambda: W.verify_sweep(1)),
    ("verify_sweep_w8", lambda: W.verify_sweep(8)),
    ("verify_sweep_w16", lambda: W.verify_sweep(16)),
    ("batched_draft", lambda: W.batched_draft()),
    ("nvfp4", lambda: W.nvfp4()),
    # 64 query heads over 4 KV heads (G 16): 256 rows per KV head, two row groups
    ("verify_w16_ctx16k_hq64_g16", lambda: W.make_workload("verify_ctx16384_w16_hq64", [16384], 16, 64, 4, 256,
                                                          W.MASK_CAUSAL_IN_BLOCK, pool_pages=2048)),
    # NVFP4 with block-scale bytes over the whole finite e4m3 range (0, the
    # subnormals, up to 448); the V decode scale keeps |v| <= 6 x 448 / 800 =
    # 3.36, as in the standard NVFP4 workload (6 x 1.875 x 0.3 = 3.375): the bf16
    # output alone rounds by up to |O| x 2^-9, which stays under the 1e-2 bound
    # only while |O| < 4
    ("nvfp4_full_scale_range", lambda: W.nvfp4(nvfp4_scale_bytes=W.NVFP4_SCALE_BYTES_FULL,
                                                nvfp4_gscale=0.3, nvfp4_v_gscale=1 / 800)),
]


@pytest.mark.parametrize("name,make", EVERY_ROW, ids=[n for n, _ in EVERY_ROW])
def test_full_size_every_row(name, make):
    wl = make()
    run_and_check(wl, sa.SPEC_ATTN_VARIANT_TCGEN05, trace=True)


# NVFP4 caches whose block scales span every non-negative finite e4m3 byte, at
# several per-tensor decode scales (K's sets the score range, V's the output
# size: max |v| = 6 x 448 x v_gscale stays below 4, where the bf16 output's own
# rounding is within the 1e-2 bound), every head_dim, both kernels, split and
# unsplit.
@pytest.mark.parametrize("variant", VARIANTS[1:])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("kg,vg", [(0.3, 1 / 800), (1 / 448, 1 / 800), (0.02, 0.00125), (4.0, 0.0005)])
def test_nvfp4_full_scale_range(variant, d, kg, vg):
    wl = W.make_workload(f"fp4wide_d{d}", [2500, 700, 33], [8, 5, 1], 24, 4, d, W.MASK_CAUSAL_IN_BLOCK,
                         kv_dtype=W.KV_NVFP4, seed=41 + d, pool_slack=0.1,
                         nvfp4_scale_bytes=W.NVFP4_SCALE_BYTES_FULL, nvfp4_gscale=kg, nvfp4_v_gscale=vg)
    for splits in (0, 3):
        run_and_check(wl, variant, force_splits=splits, trace=False)


def test_bench_main_step_as_timed():
    """The timed step of bench.py exactly as it runs there: its three calls
    (ctx 16384, W 1, 8, 16) with early_metadata, captured in one CUDA graph and
    replayed with the L2 flush in between; sampled (row, head) pairs of every
    call against the oracle, and the replayed bits equal to each call run
    alone and eagerly."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    wls = bench.main_workloads()
    dws = [sa.DeviceWorkload(wl, "cuda", early_metadata=1) for wl in wls]
    cap = bench.Captured(dws, torch.cuda.current_stream())
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = (torch.empty(2 * l2, dtype=torch.uint8, device="cuda"),
             torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda"))
    for dw in dws:
        dw.o.zero_()
        dw.lse.zero_()
    for _ in range(3):
        bench.flush_l2(flush)
        cap.replay()
    torch.cuda.synchronize()
    for dw, wl in zip(dws, wls):
        assert dw.device_status() == 0
        alone = sa.DeviceWorkload(wl, "cuda")
        alone.run()
        torch.cuda.synchronize()
        assert torch.equal(dw.o, alone.o) and torch.equal(dw.lse, alone.lse), wl.name
        sel = _sample(wl)
        o_ref, lse_ref, _ = oracle.run_workload(wl, row_select=sel)
        check_close(dw.o, dw.lse, o_ref, lse_ref, sel)


# --------------------------------------------------------------------------- #
# W-invariant mode: a window row equals the same row computed alone
# --------------------------------------------------------------------------- #
def _row_alone(wl, dw_full, r, i, fixed):
    """Window row i of request r as its own W = 1 call on the same cache: seq_len
    ctx_r + i + 1, the row's own queries, the same pools and block table."""
    lens = wl.seq_lens.tolist()
    ind = wl.q_indptr.tolist()
    w_r = ind[r + 1] - ind[r]
    ctx = lens[r] - w_r
    row = ind[r] + i
    plan = sa.spec_attn_plan_create(
        num_reqs=1, total_q_rows=1, max_w=1, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
        head_dim=wl.head_dim, num_pages=wl.num_pages, block_table_stride=int(wl.block_table.shape[1]),
        max_seq_len=ctx + i + 1, mask_mode=wl.mask_mode, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale,
        page_size=wl.page_size, w_invariant=1, fixed_keys_per_split=fixed, window_left=wl.window_left,
        kv_page_stride=dw_full.plan.problem.kv_page_stride, scale_page_stride=dw_full.plan.problem.scale_page_stride)
    q = dw_full.q[row:row + 1].contiguous()
    bt = dw_full.block_table[r:r + 1].contiguous()
    sl = torch.tensor([ctx + i + 1], dtype=torch.int32, device="cuda")
    qi = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    o = torch.zeros(1, wl.num_q_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, wl.num_q_heads, dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    sa.spec_attn_run(plan, q, dw_full.k_pool, dw_full.v_pool, bt, sl, qi, o, lse, ws, dw_full.k_scales,
                     dw_full.v_scales, wl.k_gscale, wl.v_gscale)
    torch.cuda.synchronize()
    assert sa.spec_attn_check_device_status(ws) == 0
    return o[0], lse[0]


# 64-key splits give 37 splits at ctx 2300, more than the merge's split groups
# (8 at d 256, 32 at d 64), so each group folds several, and a split boundary
# (key 2304) falls inside the 16-row window.
@pytest.mark.parametrize("kv,d,fixed", [(W.KV_BF16, 256, 0), (W.KV_BF16, 128, 192), (W.KV_NVFP4, 256, 512),
                                        (W.KV_BF16, 256, 64), (W.KV_BF16, 64, 64)])
def test_w_invariant_rows_match_the_row_alone_bitwise(kv, d, fixed):
    """Exactness rule: in W-invariant mode every row of a batched causal
    verify call is bit-identical to its own W = 1 decode at seq_len ctx + i + 1,
    and the call still matches the oracle."""
    wl = W.make_workload("winv", [2300, 700, 90], [16, 9, 5], 24, 4, d, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=kv,
                         seed=71, pool_slack=0.2)
    dw = sa.DeviceWorkload(wl, "cuda", w_invariant=1, fixed_keys_per_split=fixed)
    assert dw.plan.info["uses_merge"] == 1
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    o_ref, lse_ref, _ = oracle.run_workload(wl)
    check_close(dw.o, dw.lse, o_ref, lse_ref)
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        for i in range(ind[r + 1] - ind[r]):
            o1, l1 = _row_alone(wl, dw, r, i, fixed)
            row = ind[r] + i
            assert torch.equal(dw.o[row], o1), (r, i)
            assert torch.equal(dw.lse[row], l1), (r, i)


def test_w_invariant_is_independent_of_the_batch():
    """The same request alone and inside a batch of others gives identical bits."""
    kw = dict(num_q_heads=24, num_kv_heads=4, head_dim=256, mask_mode=W.MASK_CAUSAL_IN_BLOCK, seed=72,
              pool_slack=0.2)
    batch = W.make_workload("winvb", [1500, 3100, 400], [8, 12, 3], **kw)
    a = sa.DeviceWorkload(batch, "cuda", w_invariant=1)
    a.run()
    torch.cuda.synchronize()
    ind = batch.q_indptr.tolist()
    r = 1
    alone = W.Workload(**{**batch.__dict__, "seq_lens": batch.seq_lens[r:r + 1],
                          "q_indptr": torch.tensor([0, ind[r + 1] - ind[r]], dtype=torch.int32),
                          "block_table": batch.block_table[r:r + 1],
                          "q": batch.q[ind[r]:ind[r + 1]]})
    b = sa.DeviceWorkload(alone, "cuda", w_invariant=1)
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.o[ind[r]:ind[r + 1]], b.o) and torch.equal(a.lse[ind[r]:ind[r + 1]], b.lse)


def test_w_invariant_needs_the_tensor_core_kernel():
    wl = W.make_workload("winvu", [300], [16], 64, 4, 128, 0, seed=73)    # 256 rows per KV head
    with pytest.raises(sa.SpecAttnError) as ei:
        sa.DeviceWorkload(wl, "cuda", w_invariant=1, kernel_variant=sa.SPEC_ATTN_VARIANT_CUDA_CORE)
    assert ei.value.status == sa.SPEC_ATTN_E_UNSUPPORTED


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_NVFP4])
def test_w_invariant_across_row_groups(kv):
    """256 query rows per KV head (G 16, W 16) take two row groups on the
    tensor cores; every row still equals its own W = 1 call bit for bit."""
    wl = W.make_workload("winvrg", [900, 40], [16, 11], 64, 4, 128, 0, kv_dtype=kv, seed=74, pool_slack=0.2)
    dw = sa.DeviceWorkload(wl, "cuda", w_invariant=1, fixed_keys_per_split=128)
    assert dw.plan.info["row_groups"] == 2 and dw.plan.info["kernel_variant"] == sa.SPEC_ATTN_VARIANT_TCGEN05
    dw.run()
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    o_ref, lse_ref, _ = oracle.run_workload(wl)
    check_close(dw.o, dw.lse, o_ref, lse_ref)
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        for i in range(ind[r + 1] - ind[r]):
            o1, l1 = _row_alone(wl, dw, r, i, 128)
            assert torch.equal(dw.o[ind[r] + i], o1) and torch.equal(dw.lse[ind[r] + i], l1), (r, i)


@pytest.mark.parametrize("variant", VARIANTS[1:])
def test_early_metadata_changes_no_bit(variant):
    """Reading the lengths, windows and block table before the programmatic
    wait (early_metadata) gives the same bits as waiting first, also for calls
    back to back in one captured graph (each a dependent of the previous)."""
    shapes = [([16000], [16], 24, 4, 256, 0), ([700, 3, 1900], [9, 16, 1], 24, 4, 128, 1),
              ([100, 2000], [4, 12], 32, 8, 64, 0)]
    wls = [W.make_workload(f"em{k}", *sh, seed=90 + k, pool_slack=0.1) for k, sh in enumerate(shapes)]
    late = [make_dw(wl, variant) for wl in wls]
    early = [make_dw(wl, variant, early_metadata=1) for wl in wls]
    # and the first context K/V tile read before the wait too
    early_kv = [make_dw(wl, variant, early_metadata=1, early_context_kv=1) for wl in wls]
    s = torch.cuda.Stream()
    outs = []
    for dws in (late, early, early_kv):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for dw in dws:
                dw.run(s)
        g.replay()
        torch.cuda.synchronize()
        outs.append([(dw.o.clone(), dw.lse.clone()) for dw in dws])
    for other in outs[1:]:
        for (o0, l0), (o1, l1) in zip(outs[0], other):
            assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for dw, wl in zip(early_kv, wls):
        o_ref, lse_ref, _ = oracle.run_workload(wl)
        check_close(dw.o, dw.lse, o_ref, lse_ref)


def test_early_context_kv_after_the_append_changes_no_bit():
    """The KV append writes the window's slots just before the attention call,
    which with early_context_kv starts copying its first context tiles while
    the append runs: bits equal to waiting first, for splits whose first tile
    holds context keys only and for splits that start at the window."""
    wl = W.make_workload("ekv_app", [3000, 40, 0, 700], [16, 9, 4, 1], 24, 4, 256, 0, seed=97, pool_slack=0.2)
    rows = W.window_kv_rows(wl.total_rows, wl.num_kv_heads, wl.head_dim, seed=3, mix=False)
    outs = []
    for kw in (dict(), dict(early_metadata=1, early_context_kv=1)):
        dw = sa.DeviceWorkload(wl, "cuda", kernel_variant=sa.SPEC_ATTN_VARIANT_TCGEN05, force_splits=5,
                               mode="run_append", append_rows=rows, **kw)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dw.run(s)
        g.replay()
        torch.cuda.synchronize()
        assert dw.device_status() == 0
        outs.append((dw.o.clone(), dw.lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
