"""Pins for the oracle's KV append and its NVFP4 quantiser.

Each check compares the oracle with something it shares no code with: the
OCP format tables in tests/golden/, torch's float8_e4m3fn rounding, exact
rational arithmetic (fractions) over numpy's binary32 operations, blocks built
from representable values (whose quantisation must give them back exactly),
the grid's own error bound, and a slot-by-slot walk of the block table.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from speculative_decode_verify_paged_gb300 import workloads as wlmod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_TAB = json.load(open(os.path.join(GOLDEN, "ocp_fp4_fp8_values.json")))
E2M1 = [float(m) for m in _TAB["e2m1_magnitudes"]]                       # codes 0..7
E4M3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).tolist()


def f32(x):
    return np.float32(x)


def f32_next(x, direction):
    return np.nextafter(np.float32(x), np.float32(direction), dtype=np.float32)


# --------------------------------------------------------------------------- #
# E4M3 encoder
# --------------------------------------------------------------------------- #
def test_e4m3_encode_round_trips_every_finite_byte():
    for b in range(256):
        if b & 0x7F == 0x7F:
            continue                                        # NaN encodings
        v = (-1.0 if b & 0x80 else 1.0) * E4M3[b & 0x7F]
        x = f32(v) if v != 0 else (f32(-0.0) if b & 0x80 else f32(0.0))
        assert oracle.e4m3_encode(x) == b, (b, v)


def test_e4m3_encode_midpoints_tie_to_even_and_saturate():
    for b in range(126):
        lo, hi = E4M3[b], E4M3[b + 1]
        mid = (lo + hi) / 2                                  # exact: five significant bits
        assert float(f32(mid)) == mid
        even = b if b % 2 == 0 else b + 1
        assert oracle.e4m3_encode(f32(mid)) == even, b
        assert oracle.e4m3_encode(f32_next(mid, math.inf)) == b + 1, b
        assert oracle.e4m3_encode(f32_next(mid, -math.inf)) == b, b
        assert oracle.e4m3_encode(f32(-mid)) == 0x80 | even, b
    for big in (448.0 * (1 + 2 ** -10), 464.0, 480.0, 1e6, 3.0e38):
        assert oracle.e4m3_encode(f32(big)) == 0x7E
        assert oracle.e4m3_encode(f32(-big)) == 0xFE


def test_e4m3_encode_matches_torch_rounding_in_range():
    g = torch.Generator().manual_seed(5)
    mag = torch.exp2(torch.empty(20000).uniform_(-12.0, 8.8, generator=g))
    x = (mag * torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0)).to(torch.float32)
    x = x[x.abs() <= 448.0]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    for xi, r in zip(x.tolist(), ref):
        assert oracle.e4m3_encode(f32(xi)) == r, xi


# --------------------------------------------------------------------------- #
# E2M1 encoder
# --------------------------------------------------------------------------- #
def test_e2m1_encode_round_trips_and_ties_to_even():
    for c in range(16):
        v = (-1.0 if c & 8 else 1.0) * E2M1[c & 7]
        x = f32(v) if v != 0 else (f32(-0.0) if c & 8 else f32(0.0))
        assert oracle.e2m1_encode(x) == c, c
    for c in range(7):
        mid = (E2M1[c] + E2M1[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e2m1_encode(f32(mid)) == even, c
        assert oracle.e2m1_encode(f32_next(mid, math.inf)) == c + 1, c
        assert oracle.e2m1_encode(f32_next(mid, -math.inf)) == c, c
        assert oracle.e2m1_encode(f32(-mid)) == 8 | even, c
    for big in (6.0001, 7.0, 100.0, 3.0e38):
        assert oracle.e2m1_encode(f32(big)) == 7
        assert oracle.e2m1_encode(f32(-big)) == 15
    assert oracle.e2m1_encode(f32(-1e-30)) == 8             # sign kept when rounding to zero


# --------------------------------------------------------------------------- #
# Block quantiser
# --------------------------------------------------------------------------- #
def _bf16_bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _unpack(codes):
    out = []
    for byte in codes.tolist():
        out += [byte & 0xF, byte >> 4]
    return out


def test_representable_blocks_come_back_exactly():
    """x = e2m1(c) * e4m3(s) * g with g a power of two and one |c| at 6:
    every step of the quantiser is exact, so it must return c and s."""
    rng = np.random.default_rng(7)
    for it in range(400):
        s = int(rng.integers(1, 127))                       # nonzero finite scale byte
        g = 2.0 ** int(rng.integers(-12, 3))
        c = rng.integers(0, 16, 16)
        c[int(rng.integers(0, 16))] = 7 | (8 * int(rng.integers(0, 2)))
        x = [(-1.0 if ci & 8 else 1.0) * E2M1[ci & 7] * E4M3[s] * g for ci in c]
        bits = _bf16_bits(x)
        assert np.array_equal(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy(),
                              np.array(x)), it
        # -0.0 must keep its sign through the bf16 input
        bits = np.array([b | 0x8000 if (ci & 8 and ci & 7 == 0) else b for b, ci in zip(bits, c)],
                        dtype=np.uint16)
        codes, sc = oracle.nvfp4_quantise_block(bits, g)
        assert sc == s, (it, sc, s)
        assert _unpack(codes) == [int(ci) for ci in c], it


def _nearest_even_exact(a, mags):
    """Index of the magnitude nearest to the Fraction a, ties to the even index,
    by exact distances to every candidate (saturating at the last one)."""
    best, bd = None, None
    for i, m in enumerate(mags):
        d = abs(a - Fraction(m))
        if bd is None or d < bd or (d == bd and i % 2 == 0):
            best, bd = i, d
    return best


def _brute_block(x, g):
    """The quantiser's definition with numpy binary32 operations and exact
    nearest-value searches."""
    xs = [np.float32(v) for v in x]
    amax = max(abs(v) for v in xs)
    s = np.float32(amax) / (np.float32(6.0) * np.float32(g))
    sb = _nearest_even_exact(Fraction(float(s)), E4M3)
    den = np.float32(E4M3[sb]) * np.float32(g)
    codes = []
    for v in xs:
        if den == 0:
            codes.append(0)
            continue
        t = np.float32(v) / den
        c = _nearest_even_exact(Fraction(abs(float(t))), E2M1)
        codes.append(c | (8 if math.copysign(1.0, float(t)) < 0 else 0))
    return codes, sb


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_quantiser_matches_exact_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    for it in range(300):
        spread = float(rng.choice([0.01, 1.0, 30.0]))
        x = (rng.standard_normal(16) * spread).astype(np.float32)
        if it % 7 == 0:
            x[rng.integers(0, 16, 3)] = 0.0
        bits = _bf16_bits(x)
        xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
        g = float(np.float32(rng.choice([1.0 / 2688, 0.37, 3.1e-3, 1.7e-5]) * rng.uniform(0.5, 2.0)))
        codes, sc = oracle.nvfp4_quantise_block(bits, g)
        want_c, want_s = _brute_block(xb, g)
        assert sc == want_s, (seed, it)
        assert _unpack(codes) == want_c, (seed, it)


def test_dequantised_error_within_half_grid_step():
    """Unsaturated elements decode to within half an e2m1 step (times the
    block's decode scale) of their input."""
    rng = np.random.default_rng(11)
    for it in range(300):
        x = (rng.standard_normal(16) * rng.uniform(0.1, 10)).astype(np.float32)
        bits = _bf16_bits(x)
        xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
        g = float(np.float32(np.abs(xb).max() / (6 * 448) * rng.uniform(0.5, 4)))
        codes, sc = oracle.nvfp4_quantise_block(bits, g)
        den = E4M3[sc] * g
        for xe, c in zip(xb, _unpack(codes)):
            t = abs(xe) / den
            if t > 6:
                assert c & 7 == 7
                continue
            step = 0.5 if t < 2 else (1.0 if t < 4 else 2.0)
            dec = (-1.0 if c & 8 else 1.0) * E2M1[c & 7] * den
            assert abs(dec - xe) <= 0.5 * step * den * (1 + 1e-6), (it, xe, dec)


# --------------------------------------------------------------------------- #
# Placement
# --------------------------------------------------------------------------- #
def _new_rows(total_rows, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(total_rows, hkv, d, generator=g).to(torch.bfloat16),
            torch.randn(total_rows, hkv, d, generator=g).to(torch.bfloat16))


def test_append_writes_each_row_to_its_slot_and_nothing_else_bf16():
    wl = wlmod.make_workload("app", [0, 13, 40], [3, 16, 5], 4, 2, 32, 0, seed=21, pool_slack=0.5)
    kn, vn = _new_rows(wl.total_rows, 2, 32, 22)
    kp, vp, _, _ = oracle.append_kv(num_kv_heads=2, head_dim=32, page_size=16, kv_dtype=0, k_new=kn,
                                    v_new=vn, k_pool=wl.k_pool, v_pool=wl.v_pool,
                                    block_table=wl.block_table, seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    k0 = wl.k_pool.view(torch.int16).numpy()
    v0 = wl.v_pool.view(torch.int16).numpy()
    touched = np.zeros(k0.shape[:3], dtype=bool)
    knb = kn.view(torch.int16).numpy().view(np.uint16)
    vnb = vn.view(torch.int16).numpy().view(np.uint16)
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        w = ind[r + 1] - ind[r]
        L = int(wl.seq_lens[r])
        for i in range(w):
            pos = L - w + i
            page = int(wl.block_table[r, pos // 16])
            for h in range(2):
                assert np.array_equal(kp[page, h, pos % 16], knb[ind[r] + i, h])
                assert np.array_equal(vp[page, h, pos % 16], vnb[ind[r] + i, h])
                touched[page, h, pos % 16] = True
    assert np.array_equal(kp[~touched], k0.view(np.uint16)[~touched])
    assert np.array_equal(vp[~touched], v0.view(np.uint16)[~touched])


def test_append_nvfp4_quantises_each_block_in_place():
    wl = wlmod.make_workload("app4", [7, 30], [9, 4], 4, 2, 64, 0, kv_dtype=wlmod.KV_NVFP4, seed=23,
                             pool_slack=0.5)
    kn, vn = _new_rows(wl.total_rows, 2, 64, 24)
    kp, vp, ks, vs = oracle.append_kv(num_kv_heads=2, head_dim=64, page_size=16, kv_dtype=1, k_new=kn,
                                      v_new=vn, k_pool=wl.k_pool, v_pool=wl.v_pool, k_scales=wl.k_scales,
                                      v_scales=wl.v_scales, k_gscale=wl.k_gscale, v_gscale=wl.v_gscale,
                                      block_table=wl.block_table, seq_lens=wl.seq_lens, q_indptr=wl.q_indptr)
    touched = np.zeros(kp.shape[:3], dtype=bool)
    knb = kn.view(torch.int16).numpy().view(np.uint16)
    vnb = vn.view(torch.int16).numpy().view(np.uint16)
    ind = wl.q_indptr.tolist()
    for r in range(wl.num_reqs):
        w = ind[r + 1] - ind[r]
        L = int(wl.seq_lens[r])
        for i in range(w):
            pos = L - w + i
            page = int(wl.block_table[r, pos // 16])
            for h in range(2):
                for b in range(4):
                    c, s = oracle.nvfp4_quantise_block(knb[ind[r] + i, h, 16 * b:16 * b + 16], wl.k_gscale)
                    assert np.array_equal(kp[page, h, pos % 16, 8 * b:8 * b + 8], c) and ks[page, h, pos % 16, b] == s
                    c, s = oracle.nvfp4_quantise_block(vnb[ind[r] + i, h, 16 * b:16 * b + 16], wl.v_gscale)
                    assert np.array_equal(vp[page, h, pos % 16, 8 * b:8 * b + 8], c) and vs[page, h, pos % 16, b] == s
                touched[page, h, pos % 16] = True
    assert np.array_equal(kp[~touched], wl.k_pool.numpy()[~touched])
    assert np.array_equal(ks[~touched], wl.k_scales.numpy()[~touched])
    assert np.array_equal(vs[~touched], wl.v_scales.numpy()[~touched])


def test_append_rejects_a_bad_page_before_writing():
    wl = wlmod.make_workload("appbad", [20], [4], 4, 2, 32, 0, seed=25)
    bt = wl.block_table.clone()
    bt[0, 1] = wl.num_pages                                 # the window's page
    kn, vn = _new_rows(wl.total_rows, 2, 32, 26)
    with pytest.raises(ValueError):
        oracle.append_kv(num_kv_heads=2, head_dim=32, page_size=16, kv_dtype=0, k_new=kn, v_new=vn,
                         k_pool=wl.k_pool, v_pool=wl.v_pool, block_table=bt, seq_lens=wl.seq_lens,
                         q_indptr=wl.q_indptr)
