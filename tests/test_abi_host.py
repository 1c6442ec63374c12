"""CPU-side checks of the C ABI: the library builds, loads and exports every
entry point include/idx.h declares, and host-side argument checks reject bad
calls before anything reaches a GPU (only arguments that fail those checks
are passed here, so no device memory is touched)."""
import ctypes
import os
import re

import pytest

from sparse_attention_indexer_mxfp4_gb300 import _binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "idx.h")
INVALID, UNSUPPORTED = 1, 2
FAKE = 0x10000  # never dereferenced: every call below fails its host checks first


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:idx_status|const char \*|size_t)\s*(idx_\w+)\(", text, re.M)))


def test_header_declares_the_five_operations():
    names = _declared()
    for n in ["idx_mqa_logits", "idx_paged_mqa_logits", "idx_apply_candidate_mask", "idx_topk",
              "idx_topk_to_ragged_slots", "idx_topk_ragged_slots", "idx_get_device_status",
              "idx_version",
              "idx_topk_workspace_size"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = B.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert B.version().startswith("idx")


def test_mqa_logits_argument_checks():
    L = B.lib()
    f = L.idx_mqa_logits
    ok = dict(q=FAKE, qs=None, w=FAKE, k=FAKE, ks=FAKE, rks=FAKE, rke=FAKE, M=4, N=8, H=64,
              D=128, fmt=0, lg=FAKE, ld=8)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["qs"], a["w"], a["k"], a["ks"], a["rks"], a["rke"], a["M"], a["N"],
                 a["H"], a["D"], a["fmt"], a["lg"], a["ld"], None, 0, None)
    assert call(M=-1) == INVALID
    assert call(fmt=7) == INVALID
    assert call(q=None) == INVALID
    assert call(ld=7) == INVALID
    assert call(fmt=1) == INVALID          # MXFP4 needs q_scale
    assert call(D=96) == UNSUPPORTED
    assert call(H=48) == UNSUPPORTED
    assert call(k=FAKE + 4) == UNSUPPORTED  # TMA base must be 16-byte aligned
    assert call(M=0) == 0 and call(N=0) == 0


def test_paged_argument_checks():
    f = B.lib().idx_paged_mqa_logits
    base = [FAKE, None, FAKE, FAKE, 8448, 10, FAKE, 1024, FAKE, 0, None, 2, 1, 64, 128, 64, 0,
            None, 0, 0, 0, FAKE, 65536, 65536, 0, None, 0, None]

    def call(**kw):
        a = list(base)
        idx = dict(stride=4, npages=5, bt_stride=7, B=11, next_n=12, H=13, D=14, P=15, fmt=16,
                   cand=17, cand_stride=18, num_cand=19, cand_block=20, ld=22, mml=23)
        for k, v in kw.items():
            a[idx[k]] = v
        return f(*a)
    assert call(next_n=0) == INVALID
    assert call(bt_stride=10) == INVALID        # fewer columns than max_model_len / P
    assert call(stride=8000) == INVALID         # page smaller than P * (D + 4)
    assert call(ld=100) == INVALID
    assert call(cand=FAKE, num_cand=4, cand_stride=4, cand_block=0) == INVALID
    assert call(P=96, bt_stride=700, stride=96 * 132) == UNSUPPORTED
    assert call(next_n=5) == UNSUPPORTED        # next_n * H > 256
    assert call(stride=8456) == UNSUPPORTED     # page stride not a multiple of 16
    assert call(B=0) == 0


def test_block_max_argument_checks():
    f = B.lib().idx_paged_mqa_logits_block_max
    # q, q_scale, w, pages, stride, npages, bt, bt_stride, ctx, ctx_per_row, row_ks, B,
    # next_n, H, D, P, fmt, logits, ld, mml, block_max, ld_bmax, block, num_ctas, stream
    base = [FAKE, None, FAKE, FAKE, 8448, 10, FAKE, 1024, FAKE, 0, None, 2, 1, 64, 128, 64, 0,
            FAKE, 65536, 65536, FAKE, 512, 128, 0, None]

    def call(**kw):
        a = list(base)
        idx = dict(B=11, next_n=12, bmax=20, ld_bmax=21, block=22)
        for k, v in kw.items():
            a[idx[k]] = v
        return f(*a)
    assert call(bmax=None) == INVALID
    assert call(block=0) == INVALID
    assert call(ld_bmax=511) == INVALID          # fewer columns than 65536 / 128
    assert call(block=16, ld_bmax=4096) == UNSUPPORTED
    assert call(next_n=4) == UNSUPPORTED
    assert call(B=0) == 0


def test_logits_topk_argument_checks():
    f = B.lib().idx_paged_mqa_logits_topk
    # q, q_scale, w, pages, stride, npages, bt, bt_stride, ctx, ctx_per_row, row_ks, B,
    # next_n, H, D, P, fmt, logits, ld, mml, block_max, ld_bmax, block, lengths, k,
    # out_idx, ld_out, num_ctas, ws, ws_bytes, stream
    base = [FAKE, None, FAKE, FAKE, 8448, 10, FAKE, 1024, FAKE, 0, None, 2, 1, 64, 128, 64, 0,
            FAKE, 65536, 65536, None, 0, 0, FAKE, 2048, FAKE, 2048, 0, FAKE, 1 << 20, None]

    def call(**kw):
        a = list(base)
        idx = dict(B=11, next_n=12, ld=18, lengths=23, k=24, out=25, ld_out=26)
        for k, v in kw.items():
            a[idx[k]] = v
        return f(*a)
    assert call(k=-1) == INVALID
    assert call(ld_out=2047) == INVALID          # fewer columns than k
    assert call(lengths=None) == INVALID
    assert call(out=None) == INVALID
    assert call(next_n=0) == INVALID
    assert call(ld=0) == INVALID
    assert call(B=0) == 0


def test_producer_argument_checks():
    L = B.lib()
    k = L.idx_k_norm_rope_store
    # k_pre, ld_k, pos, cos_sin, ld_cs, npos, rope_dim, norm_w, eps, T, D, fmt, pages, stride,
    # npages, P, slots, stream
    kb = [FAKE, 128, FAKE, FAKE, 64, 100, 64, FAKE, 1e-6, 8, 128, 0, FAKE, 8448, 4, 64, FAKE,
          None]

    def kc(**kw):
        a = list(kb)
        idx = dict(ld=1, rd=6, eps=8, T=9, D=10, fmt=11, stride=13, slots=16)
        for n, v in kw.items():
            a[idx[n]] = v
        return k(*a)
    assert kc(rd=63) == INVALID            # odd rope_dim
    assert kc(rd=130) == INVALID           # rope_dim > D
    assert kc(eps=-1.0) == INVALID
    assert kc(stride=8000) == INVALID      # page smaller than P * (D + 4)
    assert kc(slots=None) == INVALID
    assert kc(fmt=5) == INVALID
    assert kc(D=64, stride=64 * 68) == UNSUPPORTED
    assert kc(ld=130) == UNSUPPORTED       # rows of k_pre not 8-byte aligned
    assert kc(T=0) == 0
    q = L.idx_q_rope_quant
    # q, pos, cos_sin, ld_cs, npos, rope_dim, w, w_scale, T, H, D, fmt, q_out, q_sf, w_out, stream
    qb = [FAKE, FAKE, FAKE, 64, 100, 64, FAKE, 0.5, 4, 64, 128, 1, FAKE, FAKE, FAKE, None]

    def qc(**kw):
        a = list(qb)
        idx = dict(rd=5, T=8, H=9, D=10, fmt=11, qsf=13)
        for n, v in kw.items():
            a[idx[n]] = v
        return q(*a)
    assert qc(qsf=None) == INVALID          # MXFP4 needs the scale output
    assert qc(H=0) == INVALID
    assert qc(rd=3) == INVALID
    assert qc(D=256) == UNSUPPORTED
    assert qc(T=0) == 0


def test_select_argument_checks():
    L = B.lib()
    assert L.idx_topk(FAKE, 100, 2, FAKE, 10, FAKE, 5, None, 0, None) == INVALID  # ld_out < k
    assert L.idx_topk(FAKE, 100, -1, FAKE, 10, FAKE, 10, None, 0, None) == INVALID
    assert L.idx_topk(None, 100, 2, FAKE, 10, FAKE, 10, None, 0, None) == INVALID
    assert L.idx_topk(FAKE, 100, 0, FAKE, 10, FAKE, 10, None, 0, None) == 0
    f = L.idx_apply_candidate_mask
    assert f(FAKE, 10, 2, 20, None, FAKE, FAKE, 4, 4, 8, 1, None) == INVALID  # ld < width
    assert f(FAKE, 20, 2, 20, None, FAKE, FAKE, 4, 4, 0, 1, None) == INVALID
    assert f(FAKE, 20, 2, 20, None, FAKE, FAKE, 4, 4, 8, 0, None) == INVALID
    g = L.idx_topk_to_ragged_slots
    assert g(FAKE, 4, 2, 8, None, 1, FAKE, 10, 10, 64, 100, FAKE, FAKE, FAKE, None) == INVALID
    assert g(FAKE, 8, 2, 8, None, 0, FAKE, 10, 10, 64, 100, FAKE, FAKE, FAKE, None) == INVALID
    assert g(FAKE, 8, 2, 8, None, 1, FAKE, 10, 10, 0, 100, FAKE, FAKE, FAKE, None) == INVALID
    h = L.idx_topk_ragged_slots  # top-k checks, then the slot map's
    assert h(FAKE, 100, 2, FAKE, 10, FAKE, 5, None, 0, None, 1, FAKE, 10, 10, 64, 100, FAKE,
             FAKE, FAKE, None) == INVALID  # ld_out < k
    assert h(None, 100, 2, FAKE, 10, FAKE, 10, None, 0, None, 1, FAKE, 10, 10, 64, 100, FAKE,
             FAKE, FAKE, None) == INVALID
    assert h(FAKE, 100, 2, FAKE, 10, FAKE, 10, None, 0, None, 0, FAKE, 10, 10, 64, 100, FAKE,
             FAKE, FAKE, None) == INVALID  # next_n 0 without row_to_seq
    assert h(FAKE, 100, 2, FAKE, 10, FAKE, 10, None, 0, None, 1, FAKE, 10, 10, 0, 100, FAKE,
             FAKE, FAKE, None) == INVALID  # page_size 0
    assert h(FAKE, 100, 2, FAKE, 10, FAKE, 10, None, 0, None, 1, FAKE, 10, 10, 64, 100, FAKE,
             None, FAKE, None) == INVALID  # no indptr
    assert L.idx_get_device_status(None, None) == INVALID


def test_row_helper_argument_checks():
    L = B.lib()
    r = L.idx_row_ends
    assert r(FAKE, 0, -1, 1, 10, FAKE, None) == INVALID     # negative batch
    assert r(FAKE, 0, 2, 0, 10, FAKE, None) == INVALID      # next_n <= 0
    assert r(None, 0, 2, 1, 10, FAKE, None) == INVALID
    assert r(FAKE, 0, 0, 2, 10, FAKE, None) == 0            # no rows
    f = L.idx_fill_logits_tail
    assert f(FAKE, 5, 2, FAKE, 10, None) == INVALID          # ld < width
    assert f(FAKE, 10, -1, FAKE, 10, None) == INVALID
    assert f(FAKE, 10, 2, None, 10, None) == INVALID
    assert f(FAKE, 10, 0, FAKE, 10, None) == 0               # nothing to fill


def test_topk_workspace_size_query():
    f = B.topk_workspace_size
    assert f(0, 1000, 10) == 0 and f(4, 0, 10) == 0
    assert f(2, 8192 * 1024 + 1, 10) == 0          # more chunks than the path supports
    one, two = f(3, 8192, 64), f(3, 8193, 64)       # 1 vs 2 chunks per row
    assert 0 < one < two and two - one == 3 * 8 * 4  # eight per-chunk words per row
    assert f(6, 100000, 64) > f(3, 100000, 64)
