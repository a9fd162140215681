"""Pins that hold the CPU oracle to facts fixed outside it.

Each check compares the oracle with something it does not share code with:
torch's fp64 scaled-dot-product attention, a pure-Python brute force, closed
forms, invariances of the definition, published format tables, or the pages'
own printed numbers (tests/golden/).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decode_verify_paged_gb300 import workloads as wlmod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gather(wl, r, kvh):
    """Dense fp64 K and V of request r, KV head kvh, by torch indexing (bf16 pools)."""
    L = int(wl.seq_lens[r])
    j = torch.arange(L)
    pages = wl.block_table[r, (j // wl.page_size)].long()
    slots = (j % wl.page_size).long()
    k = wl.k_pool[pages, kvh, slots, :].to(torch.float64)
    v = wl.v_pool[pages, kvh, slots, :].to(torch.float64)
    return k, v


# --------------------------------------------------------------------------- #
# Formats
# --------------------------------------------------------------------------- #
def test_e2m1_decoder_matches_ocp_table():
    tab = json.load(open(os.path.join(GOLDEN, "ocp_fp4_fp8_values.json")))
    mags = tab["e2m1_magnitudes"]
    for code in range(16):
        want = mags[code & 7] * (-1.0 if code & 8 else 1.0)
        got = oracle.e2m1(code)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e4m3_decoder_matches_ocp_points_and_torch():
    tab = json.load(open(os.path.join(GOLDEN, "ocp_fp4_fp8_values.json")))
    for pt in tab["e4m3_points"]:
        got = oracle.e4m3(pt["byte"])
        if pt["value"] == "nan":
            assert math.isnan(got)
        else:
            assert got == pt["value"], pt
    # every byte against torch's independent float8_e4m3fn decoder
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for i in range(256):
        got = oracle.e4m3(i)
        if math.isnan(ref[i]):
            assert math.isnan(got), i
        else:
            assert got == ref[i], (i, got, ref[i])


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(4000, generator=g, dtype=torch.float64) *
         torch.exp2(torch.randint(-20, 20, (4000,), generator=g).to(torch.float64)))
    want = x.to(torch.float32).to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    for xi, wi in zip(x.tolist(), want.tolist()):
        assert oracle.round_bf16_bits(xi) == wi


# --------------------------------------------------------------------------- #
# W = 1 is ordinary decode attention: torch SDPA in fp64 on CPU
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("mask", [wlmod.MASK_CAUSAL_IN_BLOCK, wlmod.MASK_NON_CAUSAL])
def test_w1_equals_torch_sdpa(mask):
    wl = wlmod.make_workload("w1", [37, 100, 5], 1, 8, 2, 32, mask, page_size=16, seed=3,
                             pool_slack=0.5)
    o, lse, _ = oracle.run_workload(wl)
    G = wl.num_q_heads // wl.num_kv_heads
    for r in range(wl.num_reqs):
        row = int(wl.q_indptr[r])
        for h in range(wl.num_q_heads):
            k, v = _gather(wl, r, h // G)
            q = wl.q[row, h].to(torch.float64)[None, None, None, :]
            ref = torch.nn.functional.scaled_dot_product_attention(
                q, k[None, None], v[None, None], scale=wl.sm_scale)[0, 0, 0]
            ref_lse = torch.logsumexp((k @ wl.q[row, h].to(torch.float64)) * wl.sm_scale, 0)
            np.testing.assert_allclose(o[row, h], ref.numpy(), rtol=1e-12, atol=1e-13)
            assert abs(lse[row, h] - ref_lse.item()) <= 1e-12 * max(1.0, abs(ref_lse.item()))


@pytest.mark.parametrize("mask", [wlmod.MASK_CAUSAL_IN_BLOCK, wlmod.MASK_NON_CAUSAL])
def test_window_equals_sdpa_with_explicit_mask(mask):
    """W > 1 against SDPA with a boolean mask built from the definition."""
    wl = wlmod.make_workload("wmask", [20, 3], [6, 2], 4, 2, 16, mask, seed=11, pool_slack=0.3)
    o, lse, _ = oracle.run_workload(wl)
    G = wl.num_q_heads // wl.num_kv_heads
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r])
        W = int(wl.q_indptr[r + 1]) - row0
        L = int(wl.seq_lens[r])
        ctx = L - W
        keep = torch.ones(W, L, dtype=torch.bool)
        if mask == wlmod.MASK_CAUSAL_IN_BLOCK:
            keep = torch.arange(L)[None, :] <= (ctx + torch.arange(W))[:, None]
        for h in range(wl.num_q_heads):
            k, v = _gather(wl, r, h // G)
            q = wl.q[row0:row0 + W, h].to(torch.float64)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[None, None], k[None, None], v[None, None], attn_mask=keep[None, None],
                scale=wl.sm_scale)[0, 0]
            s = (q @ k.T) * wl.sm_scale
            ref_lse = torch.logsumexp(s.masked_fill(~keep, float("-inf")), 1)
            np.testing.assert_allclose(o[row0:row0 + W, h], ref.numpy(), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[row0:row0 + W, h], ref_lse.numpy(), rtol=1e-12)


# --------------------------------------------------------------------------- #
# Pure-Python brute force on tiny shapes (no numpy/torch arithmetic)
# --------------------------------------------------------------------------- #
def _brute(wl):
    q = wl.q.to(torch.float64).tolist()
    kp = wl.k_pool.to(torch.float64).tolist()
    vp = wl.v_pool.to(torch.float64).tolist()
    bt = wl.block_table.tolist()
    out, lses = {}, {}
    G = wl.num_q_heads // wl.num_kv_heads
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r]); W = int(wl.q_indptr[r + 1]) - row0; L = int(wl.seq_lens[r])
        for i in range(W):
            for h in range(wl.num_q_heads):
                kvh = h // G
                top = (L - W + i) if wl.mask_mode == 0 else (L - 1)
                bottom = max(0, top - wl.window_left + 1) if wl.window_left > 0 else 0
                scores = []
                for j in range(bottom, top + 1):
                    page, slot = bt[r][j // wl.page_size], j % wl.page_size
                    dot = 0.0
                    for e in range(wl.head_dim):
                        dot += q[row0 + i][h][e] * kp[page][kvh][slot][e]
                    scores.append((wl.sm_scale * dot, page, slot))
                mx = max(s for s, _, _ in scores)
                den = sum(math.exp(s - mx) for s, _, _ in scores)
                vec = [0.0] * wl.head_dim
                for s, page, slot in scores:
                    w = math.exp(s - mx)
                    for e in range(wl.head_dim):
                        vec[e] += w * vp[page][kvh][slot][e]
                out[(row0 + i, h)] = [x / den for x in vec]
                lses[(row0 + i, h)] = mx + math.log(den)
    return out, lses


@pytest.mark.parametrize("mask", [wlmod.MASK_CAUSAL_IN_BLOCK, wlmod.MASK_NON_CAUSAL])
@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_tiny(mask, seed):
    g = torch.Generator().manual_seed(100 + seed)
    P = int(torch.randint(1, 4, (1,), generator=g))
    ctx = torch.randint(0, 41, (P,), generator=g).tolist()
    W = torch.randint(1, 5, (P,), generator=g).tolist()
    d = [8, 16][seed]
    wl = wlmod.make_workload("brute", ctx, W, 4, 2, d, mask, seed=seed, pool_slack=0.5)
    o, lse, _ = oracle.run_workload(wl)
    ref_o, ref_lse = _brute(wl)
    for (row, h), vec in ref_o.items():
        np.testing.assert_allclose(o[row, h], vec, rtol=1e-12, atol=1e-13)
        assert abs(lse[row, h] - ref_lse[(row, h)]) <= 1e-12 * max(1.0, abs(ref_lse[(row, h)]))


@pytest.mark.parametrize("page_size,window", [(32, 0), (64, 0), (32, 9), (16, 3)])
def test_brute_force_larger_pages_and_window(page_size, window):
    wl = wlmod.make_workload("brutepw", [70, 5, 130], [4, 3, 2], 4, 2, 8, wlmod.MASK_CAUSAL_IN_BLOCK,
                             page_size=page_size, seed=7, pool_slack=0.5, window_left=window)
    o, lse, _ = oracle.run_workload(wl)
    ref_o, ref_lse = _brute(wl)
    for (row, h), vec in ref_o.items():
        np.testing.assert_allclose(o[row, h], vec, rtol=1e-12, atol=1e-13)
        assert abs(lse[row, h] - ref_lse[(row, h)]) <= 1e-12 * max(1.0, abs(ref_lse[(row, h)]))


@pytest.mark.parametrize("window", [1, 5, 37])
def test_sliding_window_equals_sdpa_with_banded_mask(window):
    """Causal rows with a sliding window against SDPA with a banded boolean
    mask built from the definition (keys hi - window + 1 .. hi)."""
    wl = wlmod.make_workload("band", [60, 3], [6, 2], 4, 2, 16, wlmod.MASK_CAUSAL_IN_BLOCK, seed=12,
                             pool_slack=0.3, window_left=window)
    o, lse, _ = oracle.run_workload(wl)
    G = wl.num_q_heads // wl.num_kv_heads
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r])
        W = int(wl.q_indptr[r + 1]) - row0
        L = int(wl.seq_lens[r])
        hi = (L - W + torch.arange(W))[:, None]
        j = torch.arange(L)[None, :]
        keep = (j <= hi) & (j > hi - window)
        for h in range(wl.num_q_heads):
            k, v = _gather(wl, r, h // G)
            q = wl.q[row0:row0 + W, h].to(torch.float64)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[None, None], k[None, None], v[None, None], attn_mask=keep[None, None],
                scale=wl.sm_scale)[0, 0]
            s = (q @ k.T) * wl.sm_scale
            ref_lse = torch.logsumexp(s.masked_fill(~keep, float("-inf")), 1)
            np.testing.assert_allclose(o[row0:row0 + W, h], ref.numpy(), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[row0:row0 + W, h], ref_lse.numpy(), rtol=1e-12)


def test_window_covering_every_key_changes_nothing_and_window_one_is_own_key():
    base = wlmod.make_workload("wall", [50, 0], [5, 3], 4, 2, 16, wlmod.MASK_CAUSAL_IN_BLOCK, seed=13)
    o0, l0, t0 = oracle.run_workload(base, want_trace=True)
    wide = wlmod.Workload(**{**base.__dict__, "window_left": 55})
    o1, l1, t1 = oracle.run_workload(wide, want_trace=True)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1) and np.array_equal(t0, t1)
    one = wlmod.Workload(**{**base.__dict__, "window_left": 1})
    o2, l2, t2 = oracle.run_workload(one, want_trace=True)
    assert (t2[..., 0] == 1).all()
    G = 2
    for r in range(2):
        row0 = int(base.q_indptr[r]); W = int(base.q_indptr[r + 1]) - row0; L = int(base.seq_lens[r])
        for i in range(W):
            for h in range(4):
                k, v = _gather(base, r, h // G)
                key = L - W + i
                np.testing.assert_array_equal(o2[row0 + i, h], v[key].numpy())
                s = float((base.q[row0 + i, h].to(torch.float64) @ k[key]) * base.sm_scale)
                assert abs(l2[row0 + i, h] - s) <= 1e-12 * max(1.0, abs(s))


def test_window_needs_the_causal_mask():
    wl = wlmod.make_workload("wnc", [20], [3], 4, 2, 16, wlmod.MASK_NON_CAUSAL, seed=14, window_left=4)
    with pytest.raises(ValueError):
        oracle.run_workload(wl)


# --------------------------------------------------------------------------- #
# Invariants of the definition
# --------------------------------------------------------------------------- #
def test_causal_row_i_equals_decode_at_ctx_plus_i_plus_1():
    W, ctx = 5, 70
    wl = wlmod.make_workload("rowwise", [ctx], W, 6, 2, 32, wlmod.MASK_CAUSAL_IN_BLOCK, seed=7)
    o, lse, _ = oracle.run_workload(wl)
    for i in range(W):
        # same cache, one-row window whose cache ends at key ctx + i
        one = dict(num_q_heads=6, num_kv_heads=2, head_dim=32, page_size=16,
                   num_pages=wl.num_pages, mask_mode=wlmod.MASK_CAUSAL_IN_BLOCK, kv_dtype=0,
                   sm_scale=wl.sm_scale, q=wl.q[i:i + 1], k_pool=wl.k_pool, v_pool=wl.v_pool,
                   block_table=wl.block_table, seq_lens=torch.tensor([ctx + i + 1], dtype=torch.int32),
                   q_indptr=torch.tensor([0, 1], dtype=torch.int32))
        o1, lse1, _ = oracle.run(**one)
        assert np.array_equal(o1[0], o[i]) and np.array_equal(lse1[0], lse[i])


def test_last_row_agrees_between_masks():
    kw = dict(ctx_lens=[50, 9, 33], windows=[4, 7, 1], num_q_heads=4, num_kv_heads=1,
              head_dim=16, seed=21, pool_slack=0.2)
    wc = wlmod.make_workload("c", mask_mode=wlmod.MASK_CAUSAL_IN_BLOCK, **kw)
    wn = wlmod.make_workload("n", mask_mode=wlmod.MASK_NON_CAUSAL, **kw)
    oc, lc, _ = oracle.run_workload(wc)
    on, ln, _ = oracle.run_workload(wn)
    for r in range(wc.num_reqs):
        last = int(wc.q_indptr[r + 1]) - 1
        assert np.array_equal(oc[last], on[last]) and np.array_equal(lc[last], ln[last])
        first = int(wc.q_indptr[r])
        if last > first:  # earlier causal rows see strictly fewer keys
            assert not np.array_equal(lc[first], ln[first])


def test_page_permutation_invariance():
    wl = wlmod.make_workload("perm", [90, 40], [3, 5], 4, 2, 16, wlmod.MASK_CAUSAL_IN_BLOCK,
                             seed=4, pool_slack=0.6)
    o, lse, tr = oracle.run_workload(wl, want_trace=True)
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(wl.num_pages, generator=g)      # new page id of old page p
    inv = torch.argsort(perm)
    bt2 = torch.where(wl.block_table >= 0, perm[wl.block_table.clamp(min=0).long()].to(torch.int32),
                      wl.block_table)
    kw = dict(num_q_heads=4, num_kv_heads=2, head_dim=16, page_size=16, num_pages=wl.num_pages,
              mask_mode=0, kv_dtype=0, sm_scale=wl.sm_scale, q=wl.q,
              k_pool=wl.k_pool[inv], v_pool=wl.v_pool[inv], block_table=bt2,
              seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    o2, lse2, tr2 = oracle.run(**kw, want_trace=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    assert np.array_equal(tr[..., 0], tr2[..., 0])


def test_unread_slots_poisoned_do_not_change_output():
    base = dict(ctx_lens=[21, 70], windows=[3, 2], num_q_heads=2, num_kv_heads=1, head_dim=16,
                mask_mode=wlmod.MASK_NON_CAUSAL, seed=8, pool_slack=0.5)
    o, lse, _ = oracle.run_workload(wlmod.make_workload("clean", **base))
    wp = wlmod.make_workload("poison", poison_unread=True, **base)
    assert torch.isnan(wp.k_pool.float()).any()
    o2, lse2, _ = oracle.run_workload(wp)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


# --------------------------------------------------------------------------- #
# Closed forms
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("mask", [wlmod.MASK_CAUSAL_IN_BLOCK, wlmod.MASK_NON_CAUSAL])
def test_zero_queries_give_mean_of_visible_values(mask):
    wl = wlmod.make_workload("q0", [30, 64], [4, 3], 4, 2, 16, mask, seed=12, q_mode="zero")
    o, lse, _ = oracle.run_workload(wl)
    G = 2
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r]); W = int(wl.q_indptr[r + 1]) - row0; L = int(wl.seq_lens[r])
        for i in range(W):
            n = (L - W + i + 1) if mask == 0 else L
            for h in range(4):
                _, v = _gather(wl, r, h // G)
                np.testing.assert_allclose(o[row0 + i, h], v[:n].mean(0).numpy(), rtol=1e-12, atol=1e-14)
                assert lse[row0 + i, h] == math.log(n)
                assert round(math.exp(lse[row0 + i, h])) == n


def test_one_visible_key_returns_its_value_and_score():
    wl = wlmod.make_workload("one", [0], 1, 3, 1, 32, wlmod.MASK_CAUSAL_IN_BLOCK, seed=13)
    o, lse, _ = oracle.run_workload(wl)
    k, v = _gather(wl, 0, 0)
    for h in range(3):
        assert np.array_equal(o[0, h], v[0].numpy())
        s = float(np.dot(wl.q[0, h].to(torch.float64).numpy(), k[0].numpy())) * wl.sm_scale
        assert abs(lse[0, h] - s) <= 1e-13 * max(1.0, abs(s))


def test_constant_power_of_two_values_come_back_exactly():
    wl = wlmod.make_workload("vconst", [45, 17], [5, 2], 4, 2, 16, wlmod.MASK_CAUSAL_IN_BLOCK,
                             seed=14, v_mode="const")
    o, _, _ = oracle.run_workload(wl)
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r])
        for h in range(4):
            _, v = _gather(wl, r, h // 2)
            for row in range(row0, int(wl.q_indptr[r + 1])):
                assert np.array_equal(o[row, h], v[0].numpy())


@pytest.mark.parametrize("page_size,window", [(16, 0), (32, 0), (64, 11)])
def test_trace_counts_and_slot_sums(page_size, window):
    wl = wlmod.make_workload("trace", [33, 7, 100], [4, 2, 3], 2, 1, 8, wlmod.MASK_CAUSAL_IN_BLOCK,
                             seed=15, pool_slack=1.0, page_size=page_size, window_left=window)
    _, _, tr = oracle.run_workload(wl, want_o=False, want_lse=False, want_trace=True)
    bt = wl.block_table.tolist()
    ps = page_size
    for r in range(wl.num_reqs):
        row0 = int(wl.q_indptr[r]); W = int(wl.q_indptr[r + 1]) - row0; L = int(wl.seq_lens[r])
        for i in range(W):
            hi = L - W + i
            lo = max(0, hi - window + 1) if window else 0
            s = sum(bt[r][j // ps] * ps + j % ps for j in range(lo, hi + 1))
            assert tr[row0 + i, 0, 0] == hi - lo + 1 and tr[row0 + i, 0, 1] == s


# --------------------------------------------------------------------------- #
# NVFP4: the quantised cache decoded in the test == bf16 oracle on those values
# --------------------------------------------------------------------------- #
def test_nvfp4_equals_bf16_oracle_on_decoded_values():
    wl = wlmod.make_workload("fp4", [40, 18], [3, 4], 4, 2, 32, wlmod.MASK_CAUSAL_IN_BLOCK,
                             kv_dtype=wlmod.KV_NVFP4, seed=16, pool_slack=0.3)
    tab = json.load(open(os.path.join(GOLDEN, "ocp_fp4_fp8_values.json")))
    grid = torch.tensor(tab["e2m1_magnitudes"], dtype=torch.float64)

    def decode(codes, scales):
        lo = (codes & 0xF).long(); hi = (codes >> 4).long()
        c = torch.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
        val = grid[c & 7] * torch.where((c & 8) > 0, -1.0, 1.0).to(torch.float64)
        sc = scales.view(torch.float8_e4m3fn).to(torch.float64)
        return val * sc.repeat_interleave(16, dim=-1)

    kd = decode(wl.k_pool, wl.k_scales)
    vd = decode(wl.v_pool, wl.v_scales)
    # e2m1 x e4m3 has at most 6 significant bits: exact in bf16
    assert torch.equal(kd.to(torch.bfloat16).to(torch.float64), kd)
    assert torch.equal(vd.to(torch.bfloat16).to(torch.float64), vd)
    o4, l4, _ = oracle.run_workload(wl)
    kw = dict(num_q_heads=4, num_kv_heads=2, head_dim=32, page_size=16, num_pages=wl.num_pages,
              mask_mode=0, kv_dtype=0, sm_scale=wl.sm_scale * wl.k_gscale, q=wl.q,
              k_pool=kd.to(torch.bfloat16), v_pool=vd.to(torch.bfloat16),
              block_table=wl.block_table, seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    ob, lb, _ = oracle.run(**kw)
    np.testing.assert_allclose(o4, ob * wl.v_gscale, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(l4, lb, rtol=1e-12)


# --------------------------------------------------------------------------- #
# The pages' own numbers
# --------------------------------------------------------------------------- #
def test_p1_gbs_is_one_sweep_kv_bytes_over_time():
    """time x GB/s printed on the page equals one sweep of K and V for
    q24 with Hkv=4, d=256, bf16 -- the byte count this library reports."""
    fx = json.load(open(os.path.join(GOLDEN, "p1_measurement.json")))
    for row in fx["rows"]:
        seq = row["context"] + row["w"]
        wl_bytes = seq * fx["inferred_num_kv_heads"] * 2 * (2 * fx["inferred_head_dim"])
        page_bytes = row["us"] * 1e-6 * row["gbs"] * 1e9
        assert abs(page_bytes / wl_bytes - 1) < 0.02, row
    # and the workload object's own byte count follows the same definition
    wl = wlmod.make_workload("b", [100], 16, 24, 4, 256, 0, seed=0)
    assert wl.kv_bytes == 116 * 4 * 2 * 512
    # with a sliding window only the keys some row can see count: the last W + window - 1
    wl = wlmod.make_workload("bw", [100, 3], [16, 2], 24, 4, 256, 0, seed=0, window_left=10)
    assert wl.kv_bytes == (25 + 5) * 4 * 2 * 512


def test_p2_non_causal_pair_count_and_blowup():
    fx = json.load(open(os.path.join(GOLDEN, "p2_attention_pairs.json")))
    k, ctx = fx["k"], fx["ctx"]
    W = 1 + k
    wl = wlmod.make_workload("pairs", [ctx], W, 1, 1, 8, wlmod.MASK_NON_CAUSAL, seed=1)
    _, _, tr = oracle.run_workload(wl, want_o=False, want_lse=False, want_trace=True)
    pairs = int(tr[..., 0].sum())
    assert pairs == W * (ctx + W)                  # block rows only, whole span each
    fallback_pairs = (ctx + W) ** 2                # every context row attends as well
    blowup = fallback_pairs / pairs
    assert abs(blowup / fx["claimed_blowup"] - 1) < 0.05


# --------------------------------------------------------------------------- #
# Dense block operand: the window's own keys outside the cache
# --------------------------------------------------------------------------- #
def _as_block_workload(wl):
    """The same keys, the window's own rows moved out of the cache into dense
    block tensors (gathered from the cache by torch indexing), and the cache
    slots they came from poisoned with NaN."""
    ind = wl.q_indptr.tolist()
    bk = torch.zeros(wl.total_rows, wl.num_kv_heads, wl.head_dim, dtype=torch.bfloat16)
    bv = torch.zeros_like(bk)
    kp, vp = wl.k_pool.clone(), wl.v_pool.clone()
    for r in range(wl.num_reqs):
        W = ind[r + 1] - ind[r]
        L = int(wl.seq_lens[r])
        for i in range(W):
            j = L - W + i
            page, slot = int(wl.block_table[r, j // wl.page_size]), j % wl.page_size
            bk[ind[r] + i] = kp[page, :, slot]
            bv[ind[r] + i] = vp[page, :, slot]
            kp[page, :, slot] = float("nan")
            vp[page, :, slot] = float("nan")
    return wlmod.Workload(**{**wl.__dict__, "k_pool": kp, "v_pool": vp, "block_k": bk, "block_v": bv})


@pytest.mark.parametrize("mask", [wlmod.MASK_CAUSAL_IN_BLOCK, wlmod.MASK_NON_CAUSAL])
def test_block_operand_equals_the_cache_holding_the_same_rows(mask):
    """Moving the window's keys out of the cache into the block operand changes
    nothing but the trace's slot ids: outputs bit for bit, key counts exactly,
    and the NaN left in the vacated slots is never read."""
    wl = wlmod.make_workload("blk", [40, 0, 17], [5, 3, 16], 4, 2, 16, mask, seed=31, pool_slack=0.3)
    blk = _as_block_workload(wl)
    o0, l0, t0 = oracle.run_workload(wl, want_trace=True)
    o1, l1, t1 = oracle.run_workload(blk, want_trace=True)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    assert np.array_equal(t0[..., 0], t1[..., 0])
    # slot sums: the window's keys now count -(1 + row) instead of their slot id
    ind = wl.q_indptr.tolist()
    bt = wl.block_table.tolist()
    for r in range(wl.num_reqs):
        W = ind[r + 1] - ind[r]
        L = int(wl.seq_lens[r])
        for i in range(W):
            hi = (L - W + i) if mask == wlmod.MASK_CAUSAL_IN_BLOCK else L - 1
            want = sum(bt[r][j // 16] * 16 + j % 16 if j < L - W else -1 - (ind[r] + j - (L - W))
                       for j in range(hi + 1))
            assert (t1[ind[r] + i, :, 1] == want).all()


def test_block_operand_equals_sdpa_on_concatenated_keys():
    wl = wlmod.make_workload("blks", [33, 70], [4, 9], 4, 2, 16, wlmod.MASK_NON_CAUSAL, seed=32,
                             pool_slack=0.3, dense_block=True, poison_unread=True)
    o, lse, _ = oracle.run_workload(wl)
    G = 2
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        W = ind[r + 1] - ind[r]
        ctx = int(wl.seq_lens[r]) - W
        j = torch.arange(ctx)
        pages = wl.block_table[r, (j // 16)].long()
        for h in range(4):
            kvh = h // G
            k = torch.cat([wl.k_pool[pages, kvh, (j % 16).long()], wl.block_k[ind[r]:ind[r + 1], kvh]]).double()
            v = torch.cat([wl.v_pool[pages, kvh, (j % 16).long()], wl.block_v[ind[r]:ind[r + 1], kvh]]).double()
            q = wl.q[ind[r]:ind[r + 1], h].double()
            ref = torch.nn.functional.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None],
                                                                   scale=wl.sm_scale)[0, 0]
            ref_lse = torch.logsumexp((q @ k.T) * wl.sm_scale, 1)
            np.testing.assert_allclose(o[ind[r]:ind[r + 1], h], ref.numpy(), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[ind[r]:ind[r + 1], h], ref_lse.numpy(), rtol=1e-12)


@pytest.mark.parametrize("make", [lambda: wlmod.verify_sweep(16), lambda: wlmod.long_verify(16)],
                         ids=["verify_ctx16384_w16", "long_verify_ctx65536_w16_peaky"])
def test_full_size_rows_equal_sdpa(make):
    """The oracle at the measured sizes (the peaky 64K workload included), on
    sampled (row, head) pairs, against SDPA in fp64 with the causal-in-block
    mask of each row (keys 0 .. ctx + i) on the gathered K/V."""
    wl = make()
    G = wl.num_q_heads // wl.num_kv_heads
    pairs = [(0, 0), (7, 13), (15, wl.num_q_heads - 1), (15, 5)]
    sel = np.zeros((wl.total_rows, wl.num_q_heads), dtype=np.uint8)
    for i, h in pairs:
        sel[i, h] = 1
    o, lse, _ = oracle.run_workload(wl, row_select=sel)
    L = int(wl.seq_lens[0])
    ctx = L - wl.total_rows
    for kvh in sorted({h // G for _, h in pairs}):
        k, v = _gather(wl, 0, kvh)
        for i, h in pairs:
            if h // G != kvh:
                continue
            q = wl.q[i, h].to(torch.float64)
            vis = ctx + i + 1
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, None, :], k[None, None, :vis], v[None, None, :vis], scale=wl.sm_scale)[0, 0, 0]
            ref_lse = torch.logsumexp((k[:vis] @ q) * wl.sm_scale, 0).item()
            np.testing.assert_allclose(o[i, h], ref.numpy(), rtol=1e-10, atol=1e-12)
            assert abs(lse[i, h] - ref_lse) <= 1e-11 * max(1.0, abs(ref_lse)), (i, h)


def test_full_size_nvfp4_and_noncausal_draft_rows_equal_sdpa():
    """The other two measured workloads at full size, on sampled pairs: the
    NVFP4 cache (4 requests x ctx 16384, W 8) decoded here from the OCP tables
    and torch's e4m3, then SDPA with the global scales applied as the format
    defines them; and the non-causal batched draft (8 requests, W 9, d 128),
    where every row sees the whole context and block."""
    tab = json.load(open(os.path.join(GOLDEN, "ocp_fp4_fp8_values.json")))
    grid = torch.tensor(tab["e2m1_magnitudes"], dtype=torch.float64)

    def gathered(wl, r, kvh, pool, scales):
        L = int(wl.seq_lens[r])
        j = torch.arange(L)
        pages = wl.block_table[r, (j // wl.page_size)].long()
        slots = (j % wl.page_size).long()
        if scales is None:
            return pool[pages, kvh, slots, :].to(torch.float64)
        codes = pool[pages, kvh, slots, :]
        c = torch.stack([(codes & 0xF).long(), (codes >> 4).long()], -1).reshape(L, -1)
        val = grid[c & 7] * torch.where((c & 8) > 0, -1.0, 1.0).to(torch.float64)
        sc = scales[pages, kvh, slots, :].view(torch.float8_e4m3fn).to(torch.float64)
        return val * sc.repeat_interleave(16, dim=-1)

    for wl, pairs in ((wlmod.nvfp4(), [(0, 0), (8, 23), (17, 6), (31, 12)]),
                      (wlmod.batched_draft(), [(0, 0), (13, 31), (40, 9), (71, 17)])):
        G = wl.num_q_heads // wl.num_kv_heads
        sel = np.zeros((wl.total_rows, wl.num_q_heads), dtype=np.uint8)
        for row, h in pairs:
            sel[row, h] = 1
        o, lse, _ = oracle.run_workload(wl, row_select=sel)
        ind = wl.q_indptr.tolist()
        fp4 = wl.kv_dtype == wlmod.KV_NVFP4
        kscale = wl.sm_scale * (wl.k_gscale if fp4 else 1.0)
        vscale = wl.v_gscale if fp4 else 1.0
        for row, h in pairs:
            r = max(i for i in range(wl.num_reqs) if ind[i] <= row)
            i = row - ind[r]
            L = int(wl.seq_lens[r])
            w_r = ind[r + 1] - ind[r]
            vis = (L - w_r + i + 1) if wl.mask_mode == wlmod.MASK_CAUSAL_IN_BLOCK else L
            k = gathered(wl, r, h // G, wl.k_pool, wl.k_scales if fp4 else None)[:vis]
            v = gathered(wl, r, h // G, wl.v_pool, wl.v_scales if fp4 else None)[:vis]
            q = wl.q[row, h].to(torch.float64)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, None, :], k[None, None], v[None, None], scale=kscale)[0, 0, 0] * vscale
            ref_lse = torch.logsumexp((k @ q) * kscale, 0).item()
            np.testing.assert_allclose(o[row, h], ref.numpy(), rtol=1e-10, atol=1e-12)
            assert abs(lse[row, h] - ref_lse) <= 1e-11 * max(1.0, abs(ref_lse)), (wl.name, row, h)
