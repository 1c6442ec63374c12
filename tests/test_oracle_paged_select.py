"""Oracle pins for paging, masking, top-k and the slot map: layout
equivalences, brute-force enumeration and round trips.  CPU only."""
import itertools

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_mxfp4_gb300 import synth


def _scatter_to_pages(k_vals, k_scales, fmt, P, D, num_pages, rng):
    """Lay a contiguous K (values + scales) out in block-flat pages through a
    random block table; returns (pages, page_stride, block_table row)."""
    N = k_vals.shape[0]
    npg = -(-N // P)
    table = rng.permutation(num_pages)[:npg].astype(np.int32)
    if fmt == synth.FMT_FP8:
        stride = P * (D + 4)
        vb, sb = D, 4
        sc_bytes = k_scales.astype(np.float32).view(np.uint8).reshape(N, 4)
    else:
        stride = P * (D // 2 + D // 32)
        vb, sb = D // 2, D // 32
        sc_bytes = k_scales.reshape(N, D // 32)
    pages = rng.integers(0, 256, size=(num_pages, stride), dtype=np.uint8)
    for t in range(N):
        pg, s = table[t // P], t % P
        pages[pg, s * vb:(s + 1) * vb] = k_vals[t]
        pages[pg, P * vb + s * sb:P * vb + (s + 1) * sb] = sc_bytes[t]
    return pages, stride, table


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4])
@pytest.mark.parametrize("P", [64, 128])
def test_paged_equals_contiguous(fmt, P):
    rng = np.random.default_rng(31)
    N, H, D, next_n = 333, 4, 128, 2
    c = synth.contiguous_case(8, next_n, N, H, D, ke=[N - 1, N], fmt=fmt)
    pages, stride, table = _scatter_to_pages(c.k, c.k_scale, fmt, P, D, 20, rng)
    bt = np.full((1, 8), -1, np.int32)
    bt[0, :table.size] = table
    contig = oracle.mqa_logits(fmt, c.q, c.q_scale, c.weights, c.k, c.k_scale, c.ks, c.ke,
                               next_n, N, H, D)
    paged, bad = oracle.paged_mqa_logits(fmt, c.q, c.q_scale, c.weights, pages, stride, 20,
                                         bt, np.array([N], np.int32), False, None, 1, next_n,
                                         H, D, P, 512)
    assert bad == 0
    # rows of one sequence: row j of next_n ends at N - next_n + j + 1
    for j in range(next_n):
        ke = N - next_n + j + 1
        np.testing.assert_array_equal(paged[j, :ke], contig[j, :ke])
        assert np.isnan(paged[j, ke:]).all()  # untouched tail


def test_ctx_per_row_and_row_ks():
    rng = np.random.default_rng(32)
    N, H, D, P = 200, 2, 32, 64
    c = synth.contiguous_case(9, 3, N, H, D, ke=[50, 200, 130], ks=[0, 17, 64])
    pages, stride, table = _scatter_to_pages(c.k, c.k_scale, c.fmt, P, D, 8, rng)
    # three rows of one sequence, each with its own length
    bt = table[None, :]
    ctx = np.array([50, 200, 130], np.int32)
    paged, bad = oracle.paged_mqa_logits(c.fmt, c.q, None, c.weights, pages, stride, 8, bt,
                                         ctx, True, c.ks, 1, 3, H, D, P, 256)
    contig = oracle.mqa_logits(c.fmt, c.q, None, c.weights, c.k, c.k_scale, c.ks, c.ke, 3,
                               N, H, D)
    for r in range(3):
        np.testing.assert_array_equal(paged[r, :ctx[r]], contig[r, :ctx[r]])
    assert bad == 0


def test_bad_page_ids_are_counted_and_masked():
    rng = np.random.default_rng(33)
    N, H, D, P = 128, 1, 16, 64
    c = synth.contiguous_case(10, 1, N, H, D, ke=[N])
    pages, stride, table = _scatter_to_pages(c.k, c.k_scale, c.fmt, P, D, 4, rng)
    bt = table[None, :].copy()
    bt[0, 1] = 99
    paged, bad = oracle.paged_mqa_logits(c.fmt, c.q, None, c.weights, pages, stride, 4, bt,
                                         np.array([N], np.int32), False, None, 1, 1, H, D, P,
                                         N)
    assert bad == 64
    assert np.isneginf(paged[0, 64:]).all() and np.isfinite(paged[0, :64]).all()


# ------------------------------------------------------------ candidate mask


def _mask_by_sets(width, ks, ke, cand_row, blk):
    keep = set()
    for c in cand_row:
        if c < 0:
            continue
        for t in range(ks + c * blk, ks + (c + 1) * blk):
            if ks <= t < ke:
                keep.add(t)
    return keep


def test_candidate_mask_brute_force():
    rng = np.random.default_rng(40)
    for trial in range(200):
        width = int(rng.integers(1, 13))
        blk = int(rng.integers(1, 5))
        rows, repeat = int(rng.integers(1, 5)), int(rng.integers(1, 3))
        crow = -(-rows // repeat)
        C = int(rng.integers(0, 4))
        cand = rng.integers(-2, width // blk + 3, size=(crow, max(C, 1))).astype(np.int32)
        if C == 0:
            cand[:] = -1
        ke = rng.integers(0, width + 1, size=rows).astype(np.int32)
        ks = np.minimum(rng.integers(0, width + 1, size=rows), ke).astype(np.int32)
        base = rng.standard_normal((rows, width)).astype(np.float32)
        got = oracle.apply_candidate_mask(base.copy(), ks, ke, cand, blk, repeat)
        for r in range(rows):
            keep = _mask_by_sets(width, int(ks[r]), int(ke[r]), cand[r // repeat], blk)
            for t in range(width):
                if t >= ke[r]:
                    assert got[r, t] == base[r, t]
                elif t in keep:
                    assert got[r, t] == base[r, t]
                else:
                    assert np.isneginf(got[r, t])


def test_all_candidates_listed_is_range_mask_only():
    rows, width, blk = 3, 40, 8
    ks = np.array([0, 3, 9], np.int32)
    ke = np.array([40, 33, 20], np.int32)
    cand = np.tile(np.arange(width // blk + 1, dtype=np.int32), (rows, 1))
    base = np.arange(rows * width, dtype=np.float32).reshape(rows, width)
    got = oracle.apply_candidate_mask(base.copy(), ks, ke, cand, blk)
    cols = np.arange(width)
    for r in range(rows):
        np.testing.assert_array_equal(np.isneginf(got[r]), (cols < ks[r]))
        np.testing.assert_array_equal(got[r, ks[r]:], base[r, ks[r]:])


# -------------------------------------------------------------------- top-k


def _topk_by_rank(row, length, k):
    """Select i iff fewer than k finite entries beat it (value, then lower index)."""
    sel = []
    for i in range(length):
        if not np.isfinite(row[i]):
            continue
        rank = sum(1 for j in range(length) if np.isfinite(row[j]) and
                   (row[j] > row[i] or (row[j] == row[i] and j < i)))
        if rank < k:
            sel.append((rank, i))
    return [i for _, i in sorted(sel)]


def test_topk_brute_force_with_ties_and_masks():
    rng = np.random.default_rng(41)
    for trial in range(300):
        width = int(rng.integers(1, 13))
        rows, k = int(rng.integers(1, 4)), int(rng.integers(1, 15))
        vals = rng.integers(-3, 4, size=(rows, width)).astype(np.float32)
        vals[rng.random((rows, width)) < 0.2] = -np.inf
        vals[rng.random((rows, width)) < 0.05] = np.nan
        lengths = rng.integers(0, width + 1, size=rows).astype(np.int32)
        got = oracle.topk(vals, lengths, k)
        for r in range(rows):
            want = _topk_by_rank(vals[r], int(lengths[r]), k)
            assert list(got[r, :len(want)]) == want
            assert (got[r, len(want):] == -1).all()


def test_topk_exhaustive_permutations():
    vals = np.array([0.5, -1.0, 0.5, 2.0, -np.inf, 1.0], np.float32)
    for perm in itertools.permutations(range(6)):
        row = vals[list(perm)][None, :]
        got = oracle.topk(row, np.array([6]), 3)
        assert list(got[0]) == _topk_by_rank(row[0], 6, 3)


# ---------------------------------------------------------------- slot map


def test_slot_map_round_trip_and_ragged_layout():
    rng = np.random.default_rng(42)
    P, num_pages, B, next_n, k = 16, 50, 3, 2, 7
    bt = np.stack([rng.permutation(num_pages)[:10] for _ in range(B)]).astype(np.int32)
    topk_idx = rng.integers(-1, 10 * P, size=(B * next_n, k)).astype(np.int32)
    topk_idx[1, :] = -1
    slots, indptr, lens, bad = oracle.topk_to_ragged_slots(topk_idx, bt, P, num_pages,
                                                           next_n=next_n)
    assert bad == 0
    assert indptr[0] == 0 and np.array_equal(np.diff(indptr), lens)
    assert lens[1] == 0
    for r in range(B * next_n):
        b = r // next_n
        kept = [p for p in topk_idx[r] if p >= 0]
        seg = slots[indptr[r]:indptr[r + 1]]
        assert len(seg) == len(kept)
        inv = {int(pg): lg for lg, pg in enumerate(bt[b])}
        for p, s in zip(kept, seg):
            assert inv[int(s) // P] * P + int(s) % P == p


def test_slot_map_row_to_seq_and_invalid_pages():
    P = 4
    bt = np.array([[3, 1, -1], [0, 2, 9]], np.int32)
    topk_idx = np.array([[0, 5, 9, -1], [11, 4, -1, 8]], np.int32)
    slots, indptr, lens, bad = oracle.topk_to_ragged_slots(topk_idx, bt, P, 4,
                                                           row_to_seq=np.array([1, 0]))
    # row 0 -> seq 1: 0 -> 0*4+0, 5 -> 2*4+1, 9 -> page 9 invalid (dropped)
    # row 1 -> seq 0: 11 -> logical 2 -> -1 invalid, 4 -> 1*4+0, 8 -> invalid
    assert list(slots) == [0, 9, 4]
    assert list(indptr) == [0, 2, 3] and list(lens) == [2, 1] and bad == 3
