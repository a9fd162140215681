"""CPU checks of the seeded input recipe: the named workloads have the shapes
and structure they are documented with, and the same seed draws the same
bytes (every parity test and the bench depend on both)."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from speculative_decode_verify_paged_gb300 import workloads as W  # noqa: E402


def _tensors(wl):
    out = [wl.q, wl.k_pool, wl.v_pool, wl.block_table, wl.seq_lens, wl.q_indptr]
    if wl.k_scales is not None:
        out += [wl.k_scales, wl.v_scales]
    if wl.block_k is not None:
        out += [wl.block_k, wl.block_v]
    return out


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("make", [lambda s: W.verify_sweep(8, seed=s), lambda s: W.batched_draft(seed=s),
                                  lambda s: W.make_workload("d", [300, 5], [16, 3], 24, 4, 128, 0, seed=s,
                                                            kv_dtype=W.KV_NVFP4, pool_slack=0.3),
                                  lambda s: W.make_workload("b", [300, 5], [16, 3], 24, 4, 128, 1, seed=s,
                                                            dense_block=True, page_size=32)])
def test_same_seed_same_bytes_other_seed_other_bytes(make):
    a, b, c = make(3), make(3), make(4)
    for x, y in zip(_tensors(a), _tensors(b)):
        assert torch.equal(_bits(x), _bits(y))
    assert not torch.equal(_bits(a.q), _bits(c.q))


def _check_structure(wl, ctx, windows, pool_pages=None):
    P = len(ctx)
    assert wl.num_reqs == P
    assert wl.seq_lens.tolist() == [c + w for c, w in zip(ctx, windows)]
    assert wl.q_indptr.tolist() == [sum(windows[:r]) for r in range(P + 1)]
    assert wl.q.shape == (sum(windows), wl.num_q_heads, wl.head_dim)
    pages = wl.k_pool.shape[0]
    if pool_pages is not None:
        assert pages == pool_pages
    seen = set()
    for r in range(P):
        cached = ctx[r] if wl.block_k is not None else ctx[r] + windows[r]
        n = -(-cached // wl.page_size)
        row = wl.block_table[r].tolist()
        used = row[:n]
        assert all(0 <= p < pages for p in used)
        assert all(p == -1 for p in row[n:])            # padding past the request's pages
        assert not (set(used) & seen), "a page owned by two requests"
        seen |= set(used)
    return seen


def test_verify_sweep_matches_its_description():
    for w in (1, 8, 16):
        wl = W.verify_sweep(w)
        assert (wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size) == (24, 4, 256, 16)
        assert wl.mask_mode == W.MASK_CAUSAL_IN_BLOCK and wl.kv_dtype == W.KV_BF16
        used = _check_structure(wl, [16384], [w], pool_pages=2048)
        table = wl.block_table[0, :len(used)].tolist()
        assert table != sorted(table)                  # a shuffled (fragmented) table
        assert wl.kv_bytes == (16384 + w) * 4 * 2 * 512


def test_long_verify_is_peaky_on_one_percent_of_keys():
    wl = W.long_verify(16)
    _check_structure(wl, [65536], [16], pool_pages=4608)
    L = 65536 + 16
    j = torch.arange(L)
    pages = wl.block_table[0, (j // 16)].long()
    k = wl.k_pool[pages, 0, (j % 16).long(), :].float()
    rms = k.pow(2).mean(1).sqrt()
    big = (rms > 2.0).float().mean().item()           # N(0, 1) rows have RMS ~1; the scaled ones ~3
    assert 0.008 <= big <= 0.012, big


def test_batched_draft_matches_its_description():
    wl = W.batched_draft()
    assert (wl.num_q_heads, wl.num_kv_heads, wl.head_dim) == (32, 8, 128)
    assert wl.mask_mode == W.MASK_NON_CAUSAL
    ctx = wl.meta["ctx_lens"]
    assert len(ctx) == 8 and all(1024 <= c <= 1600 for c in ctx)
    used = _check_structure(wl, ctx, [9] * 8)
    assert wl.k_pool.shape[0] == len(used) + -(-len(used) * 10 // 100)   # 10 % slack


def test_nvfp4_pools_hold_codes_and_scales_in_their_documented_ranges():
    wl = W.nvfp4()
    _check_structure(wl, [16384] * 4, [8] * 4)
    assert wl.k_pool.dtype == torch.uint8 and wl.k_pool.shape[-1] == 128
    assert wl.k_scales.shape[-1] == 16
    for s in (wl.k_scales, wl.v_scales):
        assert int(s.min()) >= 0x30 and int(s.max()) <= 0x3F
    assert wl.k_gscale == wl.v_gscale == W.NVFP4_GSCALE
    assert wl.kv_bytes == 4 * (16384 + 8) * 4 * 2 * (128 + 16)


def test_nvfp4_full_scale_range_draws_zero_subnormal_and_large_scale_bytes():
    wl = W.make_workload("wide", [3000], [8], 24, 4, 256, 0, kv_dtype=W.KV_NVFP4, seed=5,
                         nvfp4_scale_bytes=W.NVFP4_SCALE_BYTES_FULL, nvfp4_gscale=0.3, nvfp4_v_gscale=1 / 448)
    for s in (wl.k_scales, wl.v_scales):
        vals = set(torch.unique(s).tolist())
        assert max(vals) <= 0x7E and 0x00 in vals           # finite, non-negative, zero included
        assert any(1 <= v <= 7 for v in vals)               # e4m3 subnormals
        assert 0x7E in vals and len(vals) == 0x7F           # up to 448: every byte appears
    assert wl.k_gscale == 0.3 and wl.v_gscale == 1 / 448
    with pytest.raises(AssertionError):
        W.make_workload("nan", [100], [4], 4, 1, 64, 0, kv_dtype=W.KV_NVFP4, nvfp4_scale_bytes=(0, 0x80))


def test_dense_block_keeps_the_window_out_of_the_cache():
    wl = W.make_workload("db", [100, 0, 33], [16, 4, 9], 24, 4, 128, 0, seed=1, dense_block=True)
    _check_structure(wl, [100, 0, 33], [16, 4, 9])
    assert wl.block_k.shape == wl.block_v.shape == (29, 4, 128)


def test_poisoned_slots_are_exactly_the_unowned_ones():
    wl = W.make_workload("pz", [20, 7], [3, 2], 4, 2, 16, 0, seed=2, pool_slack=0.5, poison_unread=True)
    nan = torch.isnan(wl.k_pool.float())[:, 0, :, 0]      # [pages, slots]
    owned = torch.zeros_like(nan)
    for r, L in enumerate(wl.seq_lens.tolist()):
        for j in range(L):
            owned[int(wl.block_table[r, j // 16]), j % 16] = True
    assert torch.equal(nan, ~owned)


def test_window_rows_without_mix_are_standard_normal():
    k, v = W.window_kv_rows(64, 4, 256, seed=5, mix=False)
    for t in (k, v):
        assert t.shape == (64, 4, 256) and t.dtype == torch.bfloat16
        x = t.float()
        assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02
