"""Seeded synthetic inputs for the lightning indexer.

This module only draws random numbers and packs them into the byte layouts
the indexer reads.  It holds none of the indexer's arithmetic (no score, no
mask, no selection), so both the CUDA path and the CPU oracle can be fed from
it without sharing any of the computation under test.

Workload recipes (one per benchmark configuration), all from fixed seeds:

* contiguous FP8 (``config1``, ``config2``): q, k ~ N(0, 1) clipped to +-448
  and rounded to e4m3 (round-to-nearest-even), k_scale ~ U(0.5, 2) / 448 per
  key, weights ~ N(0, 1) / sqrt(H), causal row ranges ks = 0, ke = pos + 1.
* paged FP8 (``config3``, ``config4``): the same value distributions stored in
  block-flat pages (``page_size * D`` e4m3 bytes, then ``page_size`` fp32
  scales), pages taken in order from one random permutation of the pool.
* paged MXFP4 (``config5``): q, k ~ N(0, 1) quantised per 32 elements to e2m1
  with an e8m0 scale.  The scale exponent follows the MXFP8 rule of the vLLM
  page rocm_aiter_mla_sparse (_mxfp8_scale_bits) with the e2m1 maximum 6 in
  place of 448: e = clamp(ceil(log2(max(amax, 2^-126) / 6)) + 127, 0, 254);
  elements are divided by 2^(e-127) and rounded to the nearest e2m1 value,
  ties to the even code.  Element 2i is the low nibble of byte i.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

FMT_FP8 = 0
FMT_MXFP4 = 1

# --------------------------------------------------------------------------
# byte packing helpers (data preparation only)
# --------------------------------------------------------------------------

_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
_E2M1_MID = ((_E2M1_GRID[1:] + _E2M1_GRID[:-1]) / 2).astype(np.float32)


def e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Round float32 values to OCP e4m3 (RNE) and return the raw bytes."""
    t = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32, copy=False))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def mx_quantize(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4-quantise the last axis of ``x`` (a multiple of 32).

    Returns (packed e2m1 bytes [..., D/2], e8m0 scale bytes [..., D/32]).
    Runs on torch CPU ops (multi-threaded); fp64 where a rounding could bite."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    D = t.shape[-1]
    assert D % 32 == 0
    blocks = t.reshape(*t.shape[:-1], D // 32, 32)
    amax = blocks.abs().amax(dim=-1).clamp_min(2.0 ** -126).double()
    e = (torch.ceil(torch.log2(amax / 6.0)) + 127.0).clamp(0, 254)
    scaled = blocks.double() * torch.exp2(127.0 - e).unsqueeze(-1)
    a = scaled.abs()
    mids = torch.from_numpy(_E2M1_MID.astype(np.float64))
    code = torch.bucketize(a, mids, right=False).clamp_max(7)
    hit = (code < 7) & (a == mids[code.clamp_max(6)]) & (code % 2 == 1)
    code = code + hit.to(code.dtype)
    neg = (scaled < 0) & (code > 0)
    nib = (code | (neg.to(code.dtype) << 3)).to(torch.uint8).reshape(t.shape)
    packed = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return packed.contiguous().numpy(), e.to(torch.uint8).numpy()


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


# --------------------------------------------------------------------------
# problem containers
# --------------------------------------------------------------------------


@dataclass
class ContiguousCase:
    """Inputs of one non-paged logits + top-k problem."""

    fmt: int
    M: int
    N: int
    H: int
    D: int
    q: np.ndarray            # uint8 [M,H,D] (fp8) or [M,H,D/2] (mxfp4)
    q_scale: np.ndarray | None  # fp32 [M,H] or None (fp8); uint8 [M,H,D/32] (mxfp4)
    weights: np.ndarray      # fp32 [M,H]
    k: np.ndarray            # uint8 [N,D] or [N,D/2]
    k_scale: np.ndarray      # fp32 [N] (fp8) or uint8 [N,D/32] (mxfp4)
    ks: np.ndarray           # int32 [M]
    ke: np.ndarray           # int32 [M]
    topk: int
    name: str = ""

    @property
    def keys_scored(self) -> int:
        return int(np.maximum(self.ke - self.ks, 0).sum())


@dataclass
class PagedCase:
    """Inputs of one paged logits (+ mask) + top-k + slot-map problem."""

    fmt: int
    B: int
    next_n: int
    H: int
    D: int
    page_size: int
    num_pages: int
    page_stride: int
    width: int               # logits row width (max_model_len)
    q: np.ndarray            # uint8 [B*next_n,H,D] or [B*next_n,H,D/2]
    q_scale: np.ndarray | None
    weights: np.ndarray      # fp32 [B*next_n,H]
    pages: np.ndarray        # uint8 [num_pages, page_stride]
    block_table: np.ndarray  # int32 [B, max_blocks], -1 where unused
    context_lens: np.ndarray  # int32 [B] (or [B*next_n] when ctx_per_row)
    ctx_per_row: bool
    topk: int
    row_ks: np.ndarray | None = None
    cand: np.ndarray | None = None   # int32 [rows, C], -1 padded
    cand_block: int = 0
    name: str = ""
    extra: dict = field(default_factory=dict)
    # candidate source: block maxima of source_block keys and the
    # source_cands best blocks of each row (0: not a source)
    source_block: int = 0
    source_cands: int = 0

    @property
    def rows(self) -> int:
        return self.B * self.next_n

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def row_ends(self) -> np.ndarray:
        """ke of every row: the last of a sequence's next_n query tokens sees
        the whole context, earlier ones stop at their own position."""
        r = np.arange(self.rows)
        if self.ctx_per_row:
            return self.context_lens.astype(np.int64)
        b, j = r // self.next_n, r % self.next_n
        return (self.context_lens[b].astype(np.int64) - self.next_n + j + 1)

    @property
    def keys_scored(self) -> int:
        ke = np.clip(self.row_ends(), 0, self.width)
        ks = np.zeros_like(ke) if self.row_ks is None else np.minimum(self.row_ks, ke)
        return int((ke - ks).sum())


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------


def contiguous_case(seed: int, M: int, N: int, H: int, D: int, ke, ks=None,
                    fmt: int = FMT_FP8, topk: int = 256, with_q_scale: bool = False,
                    name: str = "") -> ContiguousCase:
    rng = np.random.default_rng(seed)
    qf = _normal(rng, (M, H, D))
    kf = _normal(rng, (N, D))
    w = (_normal(rng, (M, H)) / np.float32(math.sqrt(H))).astype(np.float32)
    if fmt == FMT_FP8:
        q, k = e4m3_bytes(qf), e4m3_bytes(kf)
        k_scale = (rng.uniform(0.5, 2.0, size=N) / 448.0).astype(np.float32)
        q_scale = rng.uniform(0.5, 2.0, size=(M, H)).astype(np.float32) if with_q_scale else None
    else:
        q, q_scale = mx_quantize(qf)
        k, k_scale = mx_quantize(kf)
    ke = np.asarray(ke, dtype=np.int32).reshape(M)
    ks = np.zeros(M, np.int32) if ks is None else np.asarray(ks, dtype=np.int32).reshape(M)
    return ContiguousCase(fmt, M, N, H, D, q, q_scale, w, k, k_scale, ks, ke, topk, name)


def _fill_pool(rng, fmt, num_pages, P, D, chunk_pages=4096):
    """Random pages: block-flat [P*D e4m3][P fp32 scales] for fp8,
    [P*D/2 packed e2m1][P*D/32 e8m0] for mxfp4."""
    if fmt == FMT_FP8:
        stride = P * (D + 4)
    else:
        stride = P * (D // 2 + D // 32)
    pool = np.empty((num_pages, stride), dtype=np.uint8)
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        kf = _normal(rng, (n, P, D))
        if fmt == FMT_FP8:
            pool[p0:p0 + n, :P * D] = e4m3_bytes(kf).reshape(n, P * D)
            sc = (rng.uniform(0.5, 2.0, size=(n, P)) / 448.0).astype(np.float32)
            pool[p0:p0 + n, P * D:] = sc.view(np.uint8).reshape(n, P * 4)
        else:
            packed, sc = mx_quantize(kf)
            pool[p0:p0 + n, :P * D // 2] = packed.reshape(n, P * D // 2)
            pool[p0:p0 + n, P * D // 2:] = sc.reshape(n, P * D // 32)
    return pool, stride


def paged_case(seed: int, context_lens, next_n: int, H: int, D: int, page_size: int,
               width: int, fmt: int = FMT_FP8, pool_pages: int | None = None,
               pool_factor: float = 1.0, topk: int = 2048, cand_num: int = 0,
               cand_block: int = 128, row_ks=None, ctx_per_row: bool = False,
               name: str = "") -> PagedCase:
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32).reshape(-1)
    B = ctx.size // next_n if ctx_per_row else ctx.size
    rows = B * next_n
    P = page_size
    seq_len = ctx.reshape(B, next_n).max(axis=1) if ctx_per_row else ctx
    npages = (seq_len.astype(np.int64) + P - 1) // P
    need = int(npages.sum())
    if pool_pages is None:
        pool_pages = max(1, int(math.ceil(need * pool_factor)))
    assert pool_pages >= need, "pool too small for the contexts"
    max_blocks = (width + P - 1) // P
    perm = rng.permutation(pool_pages).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(npages[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    qf = _normal(rng, (rows, H, D))
    w = (_normal(rng, (rows, H)) / np.float32(math.sqrt(H))).astype(np.float32)
    if fmt == FMT_FP8:
        q, q_scale = e4m3_bytes(qf), None
    else:
        q, q_scale = mx_quantize(qf)
    pool, stride = _fill_pool(rng, fmt, pool_pages, P, D)
    case = PagedCase(fmt, B, next_n, H, D, P, pool_pages, stride, width, q, q_scale, w,
                     pool, bt, ctx, ctx_per_row, topk,
                     None if row_ks is None else np.asarray(row_ks, np.int32), None, 0, name)
    if cand_num > 0:
        ke = np.clip(case.row_ends(), 0, width)
        ks = np.zeros(rows, np.int64) if case.row_ks is None else case.row_ks.astype(np.int64)
        cand = np.full((rows, cand_num), -1, dtype=np.int32)
        for r in range(rows):
            live = int((max(ke[r] - ks[r], 0) + cand_block - 1) // cand_block)
            if live <= cand_num:
                cand[r, :live] = rng.permutation(live)
            else:
                cand[r] = rng.choice(live, size=cand_num, replace=False)
        case.cand, case.cand_block = cand, cand_block
    return case


# --------------------------------------------------------------------------
# the five benchmark workloads
# --------------------------------------------------------------------------


def shard_seed(base: int, shard: int) -> int:
    """Data seed of one shard of a workload: shard 0 is the workload itself,
    every other shard (one per data-parallel rank) draws its own values with
    the same shapes and lengths."""
    return base + 7919 * shard


def config1(shard: int = 0) -> ContiguousCase:
    """Non-paged FP8: 16 rows x 1024 keys, H=64, D=128, ke_i = 1009 + i, top-256."""
    M = 16
    return contiguous_case(shard_seed(0, shard), M, 1024, 64, 128, ke=1009 + np.arange(M),
                           topk=256, name="contig_fp8_M16_N1024")


def config2(shard: int = 0) -> ContiguousCase:
    """Prefill chunk: rows 6144..8191 of an 8192-token sequence, causal, top-2048."""
    pos = np.arange(6144, 8192)
    return contiguous_case(shard_seed(1, shard), pos.size, 8192, 64, 128, ke=pos + 1,
                           topk=2048, name="prefill_fp8_2048x8192")


def config3(shard: int = 0) -> PagedCase:
    """Paged FP8 decode: B=64, next_n=1, ctx ~ U[4096, 32768], 40,000-page pool."""
    rng = np.random.default_rng(1003)
    ctx = rng.integers(4096, 32768, size=64, endpoint=True).astype(np.int32)
    return paged_case(shard_seed(3, shard), ctx, 1, 64, 128, 64, 65536, pool_pages=40000,
                      topk=2048, name="paged_fp8_decode_B64")


def config4_context_lens() -> np.ndarray:
    rng = np.random.default_rng(1004)
    ctx = np.rint(rng.lognormal(mean=math.log(16384.0), sigma=1.0, size=128))
    return np.clip(ctx, 2, 131072).astype(np.int32)


def config4(shard: int = 0) -> PagedCase:
    """Paged FP8 MTP decode: B=128, next_n=2, lognormal ctx (median 16384),
    64 candidate blocks of 128 per row, top-2048 mapped to ragged slots."""
    return paged_case(shard_seed(4, shard), config4_context_lens(), 2, 64, 128, 64, 131072,
                      pool_factor=1.1, topk=2048, cand_num=64, cand_block=128,
                      name="paged_fp8_mtp_cand_B128")


def config5(shard: int = 0) -> PagedCase:
    """Paged MXFP4: B=32, ctx 131072 each, 65,536-page pool, top-2048."""
    ctx = np.full(32, 131072, dtype=np.int32)
    return paged_case(shard_seed(5, shard), ctx, 1, 64, 128, 64, 131072, fmt=FMT_MXFP4,
                      pool_pages=65536, topk=2048, name="paged_mxfp4_decode_B32")


def config6(shard: int = 0) -> PagedCase:
    """Candidate source at the config-4 shapes: paged FP8 MTP decode, B=128,
    next_n=2, lognormal ctx (median 16384), every live key scored, block
    maxima of 128 keys, the 64 best blocks per row as the candidate pool, the
    row's top-2048 mapped to ragged slots."""
    c = paged_case(shard_seed(6, shard), config4_context_lens(), 2, 64, 128, 64, 131072,
                   pool_factor=1.1, topk=2048, name="paged_fp8_mtp_source_B128")
    c.source_block, c.source_cands = 128, 64
    return c


@dataclass
class ProducerCase:
    """Inputs of one K/Q producer step: T new tokens whose keys are
    normalised, rotated, quantised and stored into cache slots, and whose
    query heads are rotated and quantised with their weights scaled."""

    fmt: int
    T: int
    H: int
    D: int
    rope_dim: int
    page_size: int
    num_pages: int
    page_stride: int
    k_pre: np.ndarray        # float32 [T, D] holding bf16-exact values
    q: np.ndarray            # float32 [T, H, D] holding bf16-exact values
    weights: np.ndarray      # float32 [T, H]
    weight_scale: float
    positions: np.ndarray    # int32 [T]
    cos_sin: np.ndarray      # float32 [num_positions, rope_dim]: cos | sin
    norm_weight: np.ndarray  # float32 [D]
    eps: float
    slots: np.ndarray        # int64 [T] cache slots
    name: str = ""

    @property
    def rows(self) -> int:
        return self.T


def _bf16_exact(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even) and return
    them as float32."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def rope_table(num_positions: int, rope_dim: int, base: float = 10000.0) -> np.ndarray:
    """Rotary table, row p = cos(p f_i) for i < rope_dim/2, then sin(p f_i),
    f_i = base^(-i / (rope_dim/2))."""
    half = rope_dim // 2
    f = base ** (-np.arange(half, dtype=np.float64) / half)
    ang = np.arange(num_positions, dtype=np.float64)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def producer_case(seed: int, T: int, H: int, D: int, rope_dim: int, page_size: int,
                  fmt: int = FMT_MXFP4, start_pos: int = 0, pool_factor: float = 1.0,
                  name: str = "") -> ProducerCase:
    rng = np.random.default_rng(seed)
    npages = max(1, int(math.ceil(T / page_size * pool_factor)))
    rowb = D if fmt == FMT_FP8 else D // 2
    sbytes = 4 if fmt == FMT_FP8 else D // 32
    stride = page_size * (rowb + sbytes)
    stride = (stride + 15) // 16 * 16
    scale = rng.uniform(0.1, 10.0, (T, 1))
    k_pre = _bf16_exact((rng.standard_normal((T, D)) * scale).astype(np.float32))
    q = _bf16_exact(rng.standard_normal((T, H, D)).astype(np.float32))
    w = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    pos = (start_pos + np.arange(T)).astype(np.int32)
    slots = rng.permutation(npages * page_size)[:T].astype(np.int64)
    return ProducerCase(fmt, T, H, D, rope_dim, page_size, npages, stride, k_pre, q, w,
                        float(np.float32(1.0 / math.sqrt(D) * H ** -0.5)), pos,
                        rope_table(start_pos + T, rope_dim),
                        rng.uniform(0.5, 1.5, D).astype(np.float32), 1e-6, slots, name)


def config7(shard: int = 0) -> ProducerCase:
    """K/Q producers of a prefill chunk: 8192 new tokens at positions
    0..8191, H=64, D=128, rope_dim=64, MXFP4 keys into 64-token pages and
    MXFP4 query heads."""
    return producer_case(shard_seed(7, shard), 8192, 64, 128, 64, 64,
                         name="producers_prefill_T8192_mxfp4")


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5, 6: config6, 7: config7}
