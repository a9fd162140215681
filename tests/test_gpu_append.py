"""GPU parity of the KV append (through the C ABI) against the CPU oracle.

The append writes bytes, so the bar is bit-exact: after the call, every byte
of both pools (and, for NVFP4, both scale pools) equals the oracle's append
on the same inputs -- the window slots hold the copied or quantised rows and
no other byte changed.  The append-then-attend entry point is checked
against the separate calls (bitwise) and against the oracle's attention over
the oracle-appended cache (the attention tolerances).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_paged_gb300 as sa
from speculative_decode_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 1e-2, 1e-3, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_verify_paged_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


def _oracle_append(wl, kn, vn):
    return oracle.append_kv(num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, page_size=wl.page_size,
                            kv_dtype=wl.kv_dtype, k_new=kn, v_new=vn, k_pool=wl.k_pool, v_pool=wl.v_pool,
                            k_scales=wl.k_scales, v_scales=wl.v_scales, k_gscale=wl.k_gscale,
                            v_gscale=wl.v_gscale, block_table=wl.block_table, seq_lens=wl.seq_lens,
                            q_indptr=wl.q_indptr)


def _bytes(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


def _first_mismatch(dw, ref):
    """(pool, index, got, want) of the first differing byte, for a readable failure."""
    names = ("k_pool", "v_pool", "k_scales", "v_scales")
    for name, want in zip(names, ref):
        if want is None:
            continue
        got = _bytes(getattr(dw, name)).reshape(-1)
        w = want.view(np.uint8).reshape(-1)
        bad = np.nonzero(got != w)[0]
        if bad.size:
            return name, int(bad[0]), int(got[bad[0]]), int(w[bad[0]]), int(bad.size)
    return None


def _append(dw, kn, vn, ws=None):
    sa.spec_attn_append_kv(dw.plan, kn, vn, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens, dw.q_indptr,
                           dw.workspace if ws is None else ws, dw.k_scales, dw.v_scales, dw.wl.k_gscale,
                           dw.wl.v_gscale)


CASES = [
    # ctx per request, windows, Hq, Hkv, d: ragged windows, a zero-length one,
    # windows that cross a page boundary, contexts of 0
    ([0, 13, 40, 1000], [3, 16, 0, 9], 8, 2, 64),
    ([250, 17, 5], [16, 7, 1], 24, 4, 128),
    ([2000, 31], [12, 16], 24, 4, 256),
]


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_NVFP4])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_matches_oracle_bitwise(kv, case):
    ctx, win, hq, hkv, d = CASES[case]
    # a power-of-two decode scale puts the dyadic rows' quotients on rounding midpoints
    wl = W.make_workload("append", ctx, win, hq, hkv, d, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=kv, seed=40 + case,
                         pool_slack=0.3, nvfp4_gscale=2.0 ** -4)
    kn, vn = W.window_kv_rows(wl.total_rows, hkv, d, seed=50 + case)
    ref = _oracle_append(wl, kn, vn)
    dw = sa.DeviceWorkload(wl, "cuda")
    _append(dw, kn.cuda(), vn.cuda())
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    assert _first_mismatch(dw, ref) is None, _first_mismatch(dw, ref)


@pytest.mark.parametrize("gscale", [0.3, 1.0 / 2688, 7.5e-6])
def test_append_nvfp4_other_decode_scales(gscale):
    wl = W.make_workload("append_g", [77, 300], [16, 5], 24, 4, 256, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=W.KV_NVFP4,
                         seed=45, pool_slack=0.2, nvfp4_gscale=gscale)
    kn, vn = W.window_kv_rows(wl.total_rows, 4, 256, seed=46)
    ref = _oracle_append(wl, kn, vn)
    dw = sa.DeviceWorkload(wl, "cuda")
    _append(dw, kn.cuda(), vn.cuda())
    torch.cuda.synchronize()
    assert _first_mismatch(dw, ref) is None, _first_mismatch(dw, ref)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_NVFP4])
def test_run_append_equals_the_two_calls_and_the_oracle(kv):
    wl = W.make_workload("runapp", [900, 33, 4100], [16, 5, 9], 24, 4, 256, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=kv,
                         seed=47, pool_slack=0.2)
    kn, vn = W.window_kv_rows(wl.total_rows, 4, 256, seed=48, mix=False)
    kn_d, vn_d = kn.cuda(), vn.cuda()
    a = sa.DeviceWorkload(wl, "cuda")
    sa.spec_attn_run_append(a.plan, a.q, kn_d, vn_d, a.k_pool, a.v_pool, a.block_table, a.seq_lens, a.q_indptr,
                            a.o, a.lse, a.workspace, a.k_scales, a.v_scales, wl.k_gscale, wl.v_gscale)
    b = sa.DeviceWorkload(wl, "cuda")
    _append(b, kn_d, vn_d)
    b.run()
    torch.cuda.synchronize()
    assert a.device_status() == 0 and b.device_status() == 0
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)
    kp, vp, ks, vs = _oracle_append(wl, kn, vn)
    o_ref, lse_ref, _ = oracle.run(num_q_heads=24, num_kv_heads=4, head_dim=256, page_size=16,
                                   num_pages=wl.num_pages, mask_mode=wl.mask_mode, kv_dtype=kv,
                                   sm_scale=wl.sm_scale, q=wl.q, k_pool=kp, v_pool=vp, k_scales=ks, v_scales=vs,
                                   k_gscale=wl.k_gscale, v_gscale=wl.v_gscale, block_table=wl.block_table,
                                   seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    o = a.o.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lse = a.lse.cpu().numpy().astype(np.float64)
    assert (np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))).max() <= LSE_REL


def test_run_append_in_a_graph_replays_like_eager():
    wl = W.make_workload("appgraph", [500, 70], [8, 16], 24, 4, 128, W.MASK_CAUSAL_IN_BLOCK,
                         kv_dtype=W.KV_NVFP4, seed=49, pool_slack=0.2)
    kn, vn = W.window_kv_rows(wl.total_rows, 4, 128, seed=50)
    kn_d, vn_d = kn.cuda(), vn.cuda()
    eager = sa.DeviceWorkload(wl, "cuda")
    sa.spec_attn_run_append(eager.plan, eager.q, kn_d, vn_d, eager.k_pool, eager.v_pool, eager.block_table,
                            eager.seq_lens, eager.q_indptr, eager.o, eager.lse, eager.workspace, eager.k_scales,
                            eager.v_scales, wl.k_gscale, wl.v_gscale)
    g_dw = sa.DeviceWorkload(wl, "cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sa.spec_attn_run_append(g_dw.plan, g_dw.q, kn_d, vn_d, g_dw.k_pool, g_dw.v_pool, g_dw.block_table,
                                g_dw.seq_lens, g_dw.q_indptr, g_dw.o, g_dw.lse, g_dw.workspace, g_dw.k_scales,
                                g_dw.v_scales, wl.k_gscale, wl.v_gscale, stream=s)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.o, g_dw.o) and torch.equal(eager.lse, g_dw.lse)
    assert torch.equal(eager.k_pool, g_dw.k_pool) and torch.equal(eager.v_scales, g_dw.v_scales)


def test_append_bad_page_sets_status_and_skips_only_that_row():
    wl = W.make_workload("appbad", [30, 60], [4, 6], 8, 2, 64, W.MASK_CAUSAL_IN_BLOCK, seed=51, pool_slack=0.5)
    bt = wl.block_table.clone()
    bt[1, (60 + 6 - 1) // 16] = wl.num_pages + 3       # the page of request 1's last window row
    kn, vn = W.window_kv_rows(wl.total_rows, 2, 64, seed=52)
    good = W.Workload(**{**wl.__dict__, "block_table": bt})
    dw = sa.DeviceWorkload(good, "cuda")
    _append(dw, kn.cuda(), vn.cuda())
    torch.cuda.synchronize()
    assert dw.device_status() == sa.SPEC_ATTN_DEV_BAD_PAGE
    # the oracle, told to skip the rows on the bad page, must match byte for byte
    ok_rows = [i for i in range(4)] + [4 + i for i in range(6) if (60 + i) // 16 != (60 + 6 - 1) // 16]
    sel_q = torch.tensor([0, 4, 4 + len(ok_rows) - 4], dtype=torch.int32)
    part = W.Workload(**{**wl.__dict__, "q_indptr": sel_q,
                         "seq_lens": torch.tensor([34, 60 + len(ok_rows) - 4], dtype=torch.int32)})
    kp, vp, _, _ = _oracle_append(part, kn[ok_rows], vn[ok_rows])
    assert np.array_equal(_bytes(dw.k_pool), kp.view(np.uint8))
    assert np.array_equal(_bytes(dw.v_pool), vp.view(np.uint8))


def test_append_rejections_write_nothing():
    wl = W.make_workload("apprej", [3000], [8], 8, 2, 64, W.MASK_CAUSAL_IN_BLOCK, kv_dtype=W.KV_NVFP4, seed=53)
    kn, vn = W.window_kv_rows(wl.total_rows, 2, 64, seed=54)
    dw = sa.DeviceWorkload(wl, "cuda")
    before = [_bytes(t).copy() for t in (dw.k_pool, dw.v_pool, dw.k_scales, dw.v_scales)]
    kn_d, vn_d = kn.cuda(), vn.cuda()
    with pytest.raises(sa.SpecAttnError) as e:       # zero decode scale
        sa.spec_attn_append_kv(dw.plan, kn_d, vn_d, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens,
                               dw.q_indptr, dw.workspace, dw.k_scales, dw.v_scales, 0.0, wl.v_gscale)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG
    raw = torch.empty(kn_d.numel() * 2 + 16, dtype=torch.uint8, device="cuda")
    odd = raw[2:2 + kn_d.numel() * 2].view(torch.bfloat16)      # 2-byte aligned only
    with pytest.raises(sa.SpecAttnError) as e:
        sa.spec_attn_append_kv(dw.plan, odd, vn_d, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens,
                               dw.q_indptr, dw.workspace, dw.k_scales, dw.v_scales, wl.k_gscale, wl.v_gscale)
    assert e.value.status == sa.SPEC_ATTN_E_INVALID_ARG
    assert dw.plan.workspace_bytes > 256
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")   # enough for the append, not the attention
    with pytest.raises(sa.SpecAttnError) as e:
        sa.spec_attn_run_append(dw.plan, dw.q, kn_d, vn_d, dw.k_pool, dw.v_pool, dw.block_table, dw.seq_lens,
                                dw.q_indptr, dw.o, dw.lse, small, dw.k_scales, dw.v_scales, wl.k_gscale,
                                wl.v_gscale)
    assert e.value.status == sa.SPEC_ATTN_E_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    after = [_bytes(t) for t in (dw.k_pool, dw.v_pool, dw.k_scales, dw.v_scales)]
    assert all(np.array_equal(x, y) for x, y in zip(before, after))


def test_run_append_full_size_sampled():
    """The bench shape (one request, ctx 16384, W 16): the whole call on the
    GPU, the appended cache bitwise and sampled (row, head) pairs against the
    oracle's attention over the oracle-appended cache."""
    wl = W.verify_sweep(16)
    kn, vn = W.window_kv_rows(wl.total_rows, 4, 256, seed=55, mix=False)
    dw = sa.DeviceWorkload(wl, "cuda")
    sa.spec_attn_run_append(dw.plan, dw.q, kn.cuda(), vn.cuda(), dw.k_pool, dw.v_pool, dw.block_table,
                            dw.seq_lens, dw.q_indptr, dw.o, dw.lse, dw.workspace)
    torch.cuda.synchronize()
    assert dw.device_status() == 0
    kp, vp, _, _ = _oracle_append(wl, kn, vn)
    assert np.array_equal(_bytes(dw.k_pool), kp.view(np.uint8))
    assert np.array_equal(_bytes(dw.v_pool), vp.view(np.uint8))
    rng = np.random.default_rng(56)
    sel = np.zeros((16, 24), dtype=np.uint8)
    sel[rng.integers(0, 16, 24), rng.integers(0, 24, 24)] = 1
    sel[15, :] = 1
    o_ref, lse_ref, _ = oracle.run(num_q_heads=24, num_kv_heads=4, head_dim=256, page_size=16,
                                   num_pages=wl.num_pages, mask_mode=wl.mask_mode, kv_dtype=0, sm_scale=wl.sm_scale,
                                   q=wl.q, k_pool=kp, v_pool=vp, block_table=wl.block_table, seq_lens=wl.seq_lens,
                                   q_indptr=wl.q_indptr, row_select=sel)
    m = sel.astype(bool)
    o = dw.o.float().cpu().numpy().astype(np.float64)[m]
    err = np.abs(o - o_ref[m])
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lse = dw.lse.cpu().numpy().astype(np.float64)[m]
    assert (np.abs(lse - lse_ref[m]) / np.maximum(1.0, np.abs(lse_ref[m]))).max() <= LSE_REL
