"""Seeded synthetic inputs for speculative-decoding block attention.

This module only draws inputs: query rows, paged K/V pools, block tables,
sequence lengths and window offsets.  It holds none of the attention
arithmetic; the CUDA library and the CPU oracle both consume exactly the
tensors it returns.  Everything is generated on the CPU from
``torch.Generator().manual_seed(seed)``; values are fp32 N(0, 1) cast to bf16
(round to nearest even).

The named workloads mirror the shapes the pages measure or describe:

* ``tiny``           1 request, ctx 256, W 4, Hq 4, Hkv 1, d 64, causal,
                     17-page pool with a contiguous block table.
* ``verify_sweep``   1 request, ctx 16384, W in {1, 8, 16}, Hq 24, Hkv 4,
                     d 256, causal, block table = the first ceil(seq_len/16)
                     entries of a seeded permutation of a 2048-page pool
                     (page "ChunkedSmallT re-streams full KV per query chunk",
                     section "Measurement": q24, batch 1, 16K bf16 and 16K
                     fragmented rows).
* ``long_verify``    1 request, ctx 65536, W in {8, 9, 12, 16}, same heads,
                     K multiplied by 3 (before the bf16 cast) on a seeded 1%
                     of key positions, 4608-page shuffled pool (same page and
                     section, 64K bf16 row).
* ``batched_draft``  8 requests, ctx_r uniform in [1024, 1600], W 9 (k = 8),
                     Hq 32, Hkv 8, d 128, non-causal, one shared shuffled pool
                     with 10% slack, block-table rows padded with -1 (page
                     "DFlash2 leaves the paged graph fast path at every c>1",
                     sections "The cost" and "Scope": k = 8, ctx ~ 1300,
                     non-causal draft layers, shared paged pool).
* ``nvfp4``          4 requests, ctx 16384, W 8, Hq 24, Hkv 4, d 256, causal,
                     K/V as e2m1 codes + one e4m3 scale per 16 head_dim
                     elements + one fp32 scale per tensor, codes and scales
                     drawn directly (``_draw_nvfp4``), shuffled pool (page
                     "ChunkedSmallT ...", section "Measurement", 16K nvfp4
                     row; the format is this library's reading).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

MASK_CAUSAL_IN_BLOCK = 0
MASK_NON_CAUSAL = 1
KV_BF16 = 0
KV_NVFP4 = 1


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    mask_mode: int
    kv_dtype: int
    sm_scale: float
    q: torch.Tensor               # [sum W, Hq, d] bf16
    k_pool: torch.Tensor          # [pages, Hkv, ps, d] bf16 | [pages, Hkv, ps, d/2] uint8
    v_pool: torch.Tensor
    block_table: torch.Tensor     # [P, max_pages_per_req] int32, -1 past a request's pages
    seq_lens: torch.Tensor        # [P] int32, keys in cache incl. the window's own
    q_indptr: torch.Tensor        # [P + 1] int32 window offsets into Q rows
    k_scales: Optional[torch.Tensor] = None   # [pages, Hkv, ps, d/16] uint8 (e4m3)
    v_scales: Optional[torch.Tensor] = None
    k_gscale: float = 1.0
    v_gscale: float = 1.0
    window_left: int = 0          # causal sliding window (keys); 0 = none
    block_k: Optional[torch.Tensor] = None   # dense block operand [sum W, Hkv, d] bf16: the
    block_v: Optional[torch.Tensor] = None   # windows' own keys, kept out of the cache
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_w(self) -> int:
        w = self.q_indptr[1:] - self.q_indptr[:-1]
        return int(w.max().item()) if w.numel() else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    @property
    def bytes_per_token_head(self) -> int:
        """Bytes of one key (or one value) for one KV head in the pool."""
        if self.kv_dtype == KV_BF16:
            return 2 * self.head_dim
        return self.head_dim // 2 + self.head_dim // 16

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one call reads: every key some window row of
        the request may see (all cached keys, or with a sliding window the last
        W + window_left - 1), every KV head, K and V once (a single sweep)."""
        keys = 0
        for r in range(self.num_reqs):
            L = int(self.seq_lens[r])
            w = int(self.q_indptr[r + 1] - self.q_indptr[r])
            keys += min(L, w + self.window_left - 1) if self.window_left > 0 and w > 0 else L
        return keys * self.num_kv_heads * 2 * self.bytes_per_token_head

    @property
    def append_bytes(self) -> int:
        """Algorithmic bytes of the KV append: the windows' new K and V rows
        read as bf16, written in the pool's format."""
        rows = int(self.q_indptr[-1].item()) * self.num_kv_heads * 2
        return rows * (2 * self.head_dim + self.bytes_per_token_head)

    def window_lengths(self):
        return (self.q_indptr[1:] - self.q_indptr[:-1]).tolist()


# --------------------------------------------------------------------------- #
# NVFP4 pools, drawn directly
# --------------------------------------------------------------------------- #
NVFP4_GSCALE = 0.3          # decode scale of both drawn tensors: element RMS ~ 1


NVFP4_SCALE_BYTES = (0x30, 0x40)     # default block-scale bytes: e4m3 0.5 .. 1.875
NVFP4_SCALE_BYTES_FULL = (0x00, 0x7F)  # every non-negative finite e4m3 byte: 0, the
                                       # subnormals 2^-9 .. 7 x 2^-9, normals up to 448


def _draw_nvfp4(lead_shape, d: int, gen: torch.Generator, scale_bytes=NVFP4_SCALE_BYTES):
    """Random NVFP4 cache contents: codes uint8 [*lead_shape, d/2] (two
    independent uniform 4-bit codes per byte) and e4m3 block-scale bytes
    [*lead_shape, d/16] drawn uniformly from [scale_bytes[0], scale_bytes[1])
    (by default 0x30..0x3F, values 0.5 .. 1.875).  Drawn rather than
    quantised, so this module holds no quantiser; with the default bytes and
    the decode scale NVFP4_GSCALE the elements have an RMS near 1, like the
    bf16 pools' N(0, 1)."""
    lo, hi = int(scale_bytes[0]), int(scale_bytes[1])
    assert 0 <= lo < hi <= 0x7F, "non-negative finite e4m3 bytes (0x7F is NaN)"
    codes = torch.randint(0, 256, (*lead_shape, d // 2), generator=gen, dtype=torch.int32).to(torch.uint8)
    scales = torch.randint(lo, hi, (*lead_shape, d // 16), generator=gen, dtype=torch.int32).to(torch.uint8)
    return codes, scales


# --------------------------------------------------------------------------- #
# Generic generator
# --------------------------------------------------------------------------- #
def window_kv_rows(total_rows: int, num_kv_heads: int, head_dim: int, seed: int = 0, mix: bool = True):
    """New key and value rows of the windows, [total_rows, Hkv, d] bf16 each,
    for the KV append.  With ``mix`` every 16-element run draws one of:
    N(0, 1) scaled by 2^U(-8, 6) (wide dynamic range); integers in [-48, 48]
    times 2^U(-10, 2) (dyadic values, so quotients land exactly on rounding
    midpoints); all zeros, half of them negative zeros; N(0, 1) * 2^-30 (far
    below any scale); N(0, 1) * 2^12 (far above).  Without ``mix``: N(0, 1)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (2, total_rows, num_kv_heads, head_dim // 16, 16)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if mix:
        kind = torch.randint(0, 10, shape[:-1], generator=g)
        wide = torch.exp2(torch.randint(-8, 7, shape[:-1], generator=g).float())
        ints = torch.randint(-48, 49, shape, generator=g).float()
        dy = ints * torch.exp2(torch.randint(-10, 3, shape[:-1], generator=g).float())[..., None]
        negz = torch.where(torch.rand(shape, generator=g) < 0.5, -0.0, 0.0)
        out = x * wide[..., None]
        out = torch.where((kind >= 4)[..., None] & (kind < 7)[..., None], dy, out)
        out = torch.where((kind == 7)[..., None], negz, out)
        out = torch.where((kind == 8)[..., None], x * 2.0 ** -30, out)
        out = torch.where((kind == 9)[..., None], x * 2.0 ** 12, out)
        x = out
    x = x.reshape(2, total_rows, num_kv_heads, head_dim).to(torch.bfloat16)
    return x[0].contiguous(), x[1].contiguous()


def make_workload(name: str, ctx_lens: Sequence[int], windows, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, mask_mode: int, kv_dtype: int = KV_BF16,
                  page_size: int = 16, seed: int = 0, pool_pages: Optional[int] = None,
                  pool_slack: float = 0.0, fragmented: bool = True, peaky_frac: float = 0.0,
                  peaky_mult: float = 3.0, poison_unread: bool = False,
                  sm_scale: Optional[float] = None, bt_stride: Optional[int] = None,
                  q_mode: str = "randn", v_mode: str = "randn",
                  nvfp4_gscale: float = NVFP4_GSCALE, window_left: int = 0,
                  dense_block: bool = False, nvfp4_v_gscale: Optional[float] = None,
                  nvfp4_scale_bytes=NVFP4_SCALE_BYTES) -> Workload:
    """Draw one seeded workload.

    ``windows`` is one int (same W for every request) or a per-request list.
    ``poison_unread`` fills every pool slot no request may read (slots past a
    request's seq_len in its last page, and pages no request owns) with NaN
    (bf16) or NaN block scales (NVFP4).  ``q_mode``/``v_mode`` 'zero' and
    'const' (V only: a per-(kv head, dim) power of two) produce the closed-form
    cases.  NVFP4: ``nvfp4_gscale`` is the K (and, unless ``nvfp4_v_gscale``
    is given, the V) per-tensor decode scale; ``nvfp4_scale_bytes`` the
    half-open range the block-scale bytes are drawn from.
    ``dense_block``: the windows' own keys are drawn as dense
    ``block_k`` / ``block_v`` [sum W, Hkv, d] bf16 tensors and kept out of the
    cache, whose pages then cover each request's context only (bf16 pools).
    """
    assert not (dense_block and kv_dtype != KV_BF16), "the dense block operand is bf16"
    P = len(ctx_lens)
    if isinstance(windows, int):
        windows = [windows] * P
    assert len(windows) == P
    g = torch.Generator(device="cpu").manual_seed(seed)
    seq = [int(c) + int(w) for c, w in zip(ctx_lens, windows)]
    cached = [int(c) for c in ctx_lens] if dense_block else seq   # keys the cache holds
    pages_needed = [math.ceil(s / page_size) for s in cached]
    need = sum(pages_needed)
    if pool_pages is None:
        # at least one page: the library takes a pool even when no key is cached
        pool_pages = max(1, need + int(math.ceil(need * pool_slack)))
    assert pool_pages >= need, "pool too small"
    perm = torch.randperm(pool_pages, generator=g) if fragmented else torch.arange(pool_pages)
    stride = bt_stride if bt_stride is not None else max(max(pages_needed, default=1), 1)
    block_table = torch.full((P, stride), -1, dtype=torch.int32)
    off = 0
    for r in range(P):
        block_table[r, : pages_needed[r]] = perm[off: off + pages_needed[r]].to(torch.int32)
        off += pages_needed[r]
    seq_lens = torch.tensor(seq, dtype=torch.int32)
    q_indptr = torch.zeros(P + 1, dtype=torch.int32)
    q_indptr[1:] = torch.cumsum(torch.tensor(windows, dtype=torch.int32), 0)
    total_rows = int(q_indptr[-1].item())

    Hq, Hkv, d, ps = num_q_heads, num_kv_heads, head_dim, page_size
    qf = torch.randn(total_rows, Hq, d, generator=g, dtype=torch.float32)
    if q_mode == "zero":
        qf.zero_()
    fp4 = kv_dtype != KV_BF16
    assert not (fp4 and (v_mode != "randn" or peaky_frac > 0)), "value shaping is bf16-only"
    # NVFP4 pools are drawn as codes below: no bf16 values to draw for them
    kf = torch.randn(0 if fp4 else pool_pages, Hkv, ps, d, generator=g, dtype=torch.float32)
    vf = torch.randn(0 if fp4 else pool_pages, Hkv, ps, d, generator=g, dtype=torch.float32)
    if v_mode == "const":
        # per (kv head, dim) a power of two in [2^-3, 2^3], sign alternating
        expo = torch.randint(-3, 4, (Hkv, d), generator=g).to(torch.float32)
        sign = torch.where(torch.arange(d) % 2 == 0, 1.0, -1.0)
        vf[:] = (torch.pow(2.0, expo) * sign)[None, :, None, :]
    if peaky_frac > 0:
        for r in range(P):
            n = max(1, int(round(peaky_frac * cached[r])))
            pos = torch.randperm(cached[r], generator=g)[:n]
            pg = block_table[r, (pos // ps).long()].long()
            sl = (pos % ps).long()
            kf[pg, :, sl, :] *= peaky_mult

    owned = torch.zeros(pool_pages, ps, dtype=torch.bool)
    for r in range(P):
        for p_i in range(pages_needed[r]):
            first = p_i * ps
            n_valid = min(ps, cached[r] - first)
            owned[int(block_table[r, p_i]), :n_valid] = True

    q = qf.to(torch.bfloat16)
    wl_kw = {}
    if dense_block:
        wl_kw = dict(block_k=torch.randn(total_rows, Hkv, d, generator=g).to(torch.bfloat16),
                     block_v=torch.randn(total_rows, Hkv, d, generator=g).to(torch.bfloat16))
    if kv_dtype == KV_BF16:
        k_pool = kf.to(torch.bfloat16)
        v_pool = vf.to(torch.bfloat16)
        if poison_unread:
            bad = (~owned)[:, None, :, None].expand_as(k_pool)
            k_pool[bad] = float("nan")
            v_pool[bad] = float("nan")
    else:
        kc, ks = _draw_nvfp4((pool_pages, Hkv, ps), d, g, nvfp4_scale_bytes)
        vc, vs = _draw_nvfp4((pool_pages, Hkv, ps), d, g, nvfp4_scale_bytes)
        kg = float(nvfp4_gscale)
        vg = float(nvfp4_gscale if nvfp4_v_gscale is None else nvfp4_v_gscale)
        if poison_unread:
            bad = (~owned)[:, None, :, None]
            ks[bad.expand_as(ks)] = 0xFF  # e4m3 NaN
            vs[bad.expand_as(vs)] = 0xFF
        k_pool, v_pool = kc, vc
        wl_kw = dict(k_scales=ks, v_scales=vs, k_gscale=kg, v_gscale=vg)
    return Workload(name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=ps,
                    mask_mode=mask_mode, kv_dtype=kv_dtype,
                    sm_scale=(1.0 / math.sqrt(d)) if sm_scale is None else float(sm_scale),
                    window_left=int(window_left),
                    q=q, k_pool=k_pool, v_pool=v_pool, block_table=block_table,
                    seq_lens=seq_lens, q_indptr=q_indptr,
                    meta=dict(seed=seed, ctx_lens=list(map(int, ctx_lens)),
                              windows=list(map(int, windows)), fragmented=fragmented,
                              peaky_frac=peaky_frac, poison_unread=poison_unread), **wl_kw)


# --------------------------------------------------------------------------- #
# Named workloads
# --------------------------------------------------------------------------- #
def tiny(seed: int = 0, **kw) -> Workload:
    return make_workload("tiny", [256], 4, 4, 1, 64, MASK_CAUSAL_IN_BLOCK, seed=seed,
                         pool_pages=17, fragmented=False, **kw)


def verify_sweep(w: int, seed: int = 0, ctx: int = 16384, pool_pages: int = 2048, **kw) -> Workload:
    return make_workload(f"verify_sweep_ctx{ctx}_w{w}", [ctx], w, 24, 4, 256,
                         MASK_CAUSAL_IN_BLOCK, seed=seed, pool_pages=pool_pages, **kw)


def long_verify(w: int, seed: int = 0, ctx: int = 65536, **kw) -> Workload:
    return make_workload(f"long_verify_ctx{ctx}_w{w}", [ctx], w, 24, 4, 256,
                         MASK_CAUSAL_IN_BLOCK, seed=seed, pool_pages=4608, peaky_frac=0.01, **kw)


def batched_draft(seed: int = 0, num_reqs: int = 8, w: int = 9, **kw) -> Workload:
    g = torch.Generator(device="cpu").manual_seed(seed + 1_000_003)
    ctx = torch.randint(1024, 1601, (num_reqs,), generator=g).tolist()
    return make_workload("batched_draft", ctx, w, 32, 8, 128, MASK_NON_CAUSAL, seed=seed,
                         pool_slack=0.10, **kw)


def nvfp4(seed: int = 0, num_reqs: int = 4, ctx: int = 16384, w: int = 8, **kw) -> Workload:
    return make_workload(f"nvfp4_ctx{ctx}", [ctx] * num_reqs, w, 24, 4, 256,
                         MASK_CAUSAL_IN_BLOCK, kv_dtype=KV_NVFP4, seed=seed, **kw)


NAMED = {
    "tiny": lambda seed=0: tiny(seed),
    "verify_sweep_w1": lambda seed=0: verify_sweep(1, seed),
    "verify_sweep_w8": lambda seed=0: verify_sweep(8, seed),
    "verify_sweep_w16": lambda seed=0: verify_sweep(16, seed),
    "long_verify_w8": lambda seed=0: long_verify(8, seed),
    "long_verify_w9": lambda seed=0: long_verify(9, seed),
    "long_verify_w12": lambda seed=0: long_verify(12, seed),
    "long_verify_w16": lambda seed=0: long_verify(16, seed),
    "batched_draft": lambda seed=0: batched_draft(seed),
    "nvfp4": lambda seed=0: nvfp4(seed),
}
