"""GPU parity of top-k, the standalone candidate mask and the slot map
against the oracle, bit-exact, on identical inputs."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from parity import assert_topk_exact

pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_topk(logits, lengths, k, ld_out=None, workspace=True):
    rows = logits.shape[0]
    out = torch.full((rows, ld_out or k), -7, dtype=torch.int32, device="cuda")
    B.idx_topk(_t(logits), _t(lengths.astype(np.int32)), k, out, workspace=workspace)
    torch.cuda.synchronize()
    return out.cpu().numpy()[:, :k]


def _random_logits(rng, rows, width, tie_levels=None, neg_inf_frac=0.1):
    if tie_levels:
        x = rng.integers(0, tie_levels, size=(rows, width)).astype(np.float32) - tie_levels / 2
    else:
        x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < neg_inf_frac] = -np.inf
    return x


@pytest.mark.parametrize("rows,width,k", [
    (1, 1, 1), (3, 100, 7), (16, 1024, 256), (5, 1000, 2048), (64, 8192, 2048),
    (7, 65536, 2048), (2, 131072, 2048), (300, 4096, 256), (33, 20000, 1), (4, 24577, 300),
    (3, 262144, 2048), (2, 300001, 2048), (40, 32769, 2048), (160, 40000, 512)])
@pytest.mark.parametrize("workspace", [True, False])
def test_topk_random(rows, width, k, workspace):
    rng = np.random.default_rng(rows * 7 + width + k)
    x = _random_logits(rng, rows, width)
    lengths = rng.integers(0, width + 1, size=rows)
    lengths[0] = width
    got = gpu_topk(x, lengths, k, workspace=workspace)
    assert_topk_exact(got, oracle.topk(x, lengths, k))


@pytest.mark.parametrize("levels", [1, 2, 5, 300])
@pytest.mark.parametrize("workspace", [True, False])
def test_topk_ties_lowest_index_wins(levels, workspace):
    rng = np.random.default_rng(levels)
    rows, width, k = 6, 50000, 2048
    x = _random_logits(rng, rows, width, tie_levels=levels, neg_inf_frac=0.05)
    lengths = np.full(rows, width)
    lengths[3] = 1000
    got = gpu_topk(x, lengths, k, workspace=workspace)
    assert_topk_exact(got, oracle.topk(x, lengths, k))


@pytest.mark.parametrize("workspace", [True, False])
def test_topk_candidate_overflow(workspace):
    """Values packed into a narrow range put far more keys in the threshold
    bin than either candidate list holds, forcing the streaming fallback."""
    rng = np.random.default_rng(77)
    rows, width, k = 3, 100000, 2048
    x = (1.0 + rng.random((rows, width)) * 1e-3).astype(np.float32)
    lengths = np.array([100000, 70000, 30000])
    got = gpu_topk(x, lengths, k, workspace=workspace)
    assert_topk_exact(got, oracle.topk(x, lengths, k))


@pytest.mark.parametrize("width", [5000, 40000, 150000])
@pytest.mark.parametrize("case", ["digit1_bin_taken", "digit2_bin_taken", "digit3_splits_bin"])
def test_topk_threshold_bin(width, case):
    """Where the radix select stops: the threshold bin of digit 1 wholly
    taken (k equals the keys of the top bin), of digit 2 (distinct random
    values), or split by digit 3 (consecutive floats fill whole 22-bit bins,
    k ends inside one).  Register (5000) and cluster (40000, 150000) forms."""
    rng = np.random.default_rng(width + len(case))
    rows, k = 4, 2048
    if case == "digit1_bin_taken":
        # k keys in [64, 80) -- one digit-1 bin (sign, exponent, two mantissa
        # bits) -- and the rest in [1, 2)
        x = (1.0 + rng.random((rows, width))).astype(np.float32)
        for r in range(rows):
            top = rng.choice(width, size=k, replace=False)
            x[r, top] = (64.0 + 16.0 * rng.random(k) * 0.999).astype(np.float32)
    elif case == "digit2_bin_taken":
        x = rng.standard_normal((rows, width)).astype(np.float32)
    else:
        base = np.float32(1.0).view(np.int32)
        x = np.empty((rows, width), np.float32)
        for r in range(rows):
            # 4096 consecutive floats from 1.0, shuffled, the rest below 0.5;
            # the 2048th largest falls inside the second 1024-key bin
            v = (base + 700 + np.arange(4096, dtype=np.int32)).view(np.float32)
            x[r] = (0.25 * rng.random(width)).astype(np.float32)
            x[r, rng.choice(width, size=4096, replace=False)] = v
    lengths = np.full(rows, width)
    got = gpu_topk(x, lengths, k)
    assert_topk_exact(got, oracle.topk(x, lengths, k))


@pytest.mark.parametrize("width", [8192, 8191, 4099, 130])
@pytest.mark.parametrize("kind", ["ties1", "ties3", "narrow", "normal"])
def test_topk_short_rows(width, kind):
    """Rows of at most 8192 keys (held in registers by the short-row
    kernel): exact ties, three tie levels, values packed into one digit-1
    bin, k above the row's finite count, empty rows, lengths past the row."""
    rng = np.random.default_rng(width + len(kind))
    rows = 37
    if kind == "ties1":
        x = _random_logits(rng, rows, width, tie_levels=1, neg_inf_frac=0.02)
    elif kind == "ties3":
        x = _random_logits(rng, rows, width, tie_levels=3, neg_inf_frac=0.02)
    elif kind == "narrow":
        x = (1.0 + rng.random((rows, width)) * 1e-4).astype(np.float32)
    else:
        x = _random_logits(rng, rows, width)
    lengths = rng.integers(0, width + 1, size=rows)
    lengths[0], lengths[1], lengths[2], lengths[3] = width, 0, 5, width + 100
    for k in (2048, 1, width):
        got = gpu_topk(x, lengths, k)
        assert_topk_exact(got, oracle.topk(x, np.minimum(lengths, width), k))


def test_topk_nonfinite_never_selected():
    rows, width, k = 4, 3000, 2048
    x = np.full((rows, width), -np.inf, np.float32)
    x[0, ::2] = 1.0
    x[1, 5] = np.nan
    x[1, 7] = np.inf
    x[1, 9] = 0.25
    x[2, :] = np.nan
    x[3, :] = -0.0
    x[3, 10] = 0.0
    lengths = np.full(rows, width)
    got = gpu_topk(x, lengths, k)
    assert_topk_exact(got, oracle.topk(x, lengths, k))
    assert list(got[1, :2]) == [9, -1]


def test_topk_extreme_values():
    rng = np.random.default_rng(5)
    rows, width, k = 3, 5000, 100
    x = rng.standard_normal((rows, width)).astype(np.float32) * 1e-38
    x[1] = np.float32(3.4e38) * np.sign(rng.standard_normal(width)).astype(np.float32)
    x[2, :] = np.float32(1e-45)
    lengths = np.full(rows, width)
    got = gpu_topk(x, lengths, k)
    assert_topk_exact(got, oracle.topk(x, lengths, k))


def test_topk_wide_out_stride():
    rng = np.random.default_rng(9)
    x = _random_logits(rng, 5, 777)
    lengths = np.array([777, 0, 5, 600, 700])
    got = gpu_topk(x, lengths, 64, ld_out=100)
    assert_topk_exact(got, oracle.topk(x, lengths, 64))


# ------------------------------------------------------------ candidate mask


@pytest.mark.parametrize("width,blk,C,repeat", [(1, 1, 1, 1), (1000, 16, 9, 1), (131072, 128, 64, 2),
                                                (5000, 1, 300, 3), (70000, 64, 40, 1)])
def test_candidate_mask(width, blk, C, repeat):
    rng = np.random.default_rng(width + blk)
    rows = 7
    crow = -(-rows // repeat)
    nblk = -(-width // blk)
    cand = rng.integers(-3, nblk + 4, size=(crow, C)).astype(np.int32)
    ke = rng.integers(0, width + 1, size=rows).astype(np.int32)
    ks = np.minimum(rng.integers(0, width + 1, size=rows), ke).astype(np.int32)
    x = rng.standard_normal((rows, width)).astype(np.float32)
    ref = oracle.apply_candidate_mask(x.copy(), ks, ke, cand, blk, repeat)
    g = _t(x)
    B.idx_apply_candidate_mask(g, _t(ks), _t(ke), _t(cand), blk, row_repeat=repeat)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g.cpu().numpy(), ref)
    g = _t(x)
    B.idx_apply_candidate_mask(g, None, _t(ke), _t(cand), blk, row_repeat=repeat)
    ref0 = oracle.apply_candidate_mask(x.copy(), None, ke, cand, blk, repeat)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g.cpu().numpy(), ref0)


# ------------------------------------------------------------------ slot map


# The one-launch cluster kernel takes calls with at most 4 (row, 1024-entry
# step) pairs and 32768 block-table words per CTA of a 16-CTA cluster:
# (1, 1), (6, 50), (12, 3000) with a partial third step, (16, 4096) with
# four, (32, 2048) at two rows a CTA, (64, 1024) at four, (4, 100) with
# 20000-entry block-table rows.  The count and write kernels take the rest:
# (20, 3000) and (64, 2048) at six and eight pairs a CTA, (65, 1024),
# (256, 2048), (64, 4096), (16, 4097), (40, 100) with 20000 entries (60000
# words a CTA), (1500, 300); 4096 rows is the largest batch whose write
# kernel sums its own offsets; 4097 and up run the scan kernel first.  (On a
# device that holds no 16-CTA cluster the 8-CTA one takes the calls of up
# to half the rows.)
@pytest.mark.parametrize("rows,k,P,next_n,max_blocks", [
    (1, 1, 64, 1, 40), (6, 50, 16, 2, 40), (12, 3000, 64, 2, 60), (16, 4096, 64, 1, 70),
    (32, 2048, 64, 1, 40), (64, 1024, 16, 1, 70), (4, 100, 16, 2, 20000),
    (20, 3000, 64, 2, 60), (64, 2048, 64, 1, 40), (65, 1024, 16, 1, 70),
    (256, 2048, 64, 2, 40), (64, 4096, 64, 1, 70), (16, 4097, 64, 1, 70),
    (40, 100, 16, 1, 20000), (1500, 300, 128, 1, 40),
    (4096, 40, 16, 2, 40), (4097, 40, 16, 1, 40), (9000, 17, 64, 3, 40)])
def test_slots(rows, k, P, next_n, max_blocks):
    rng = np.random.default_rng(rows + k)
    nseq = -(-rows // next_n)
    num_pages = max(5000, max_blocks)
    bt = np.stack([rng.permutation(num_pages)[:max_blocks] for _ in range(nseq)]).astype(np.int32)
    topk = rng.integers(-1, max_blocks * P, size=(rows, k)).astype(np.int32)
    topk[rng.random((rows, k)) < 0.3] = -1
    slots = torch.empty(rows * k, dtype=torch.int32, device="cuda")
    indptr = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    lens = torch.empty(rows, dtype=torch.int32, device="cuda")
    B.idx_get_device_status()
    B.idx_topk_to_ragged_slots(_t(topk), _t(bt), P, num_pages, slots, indptr, lens,
                               next_n=next_n)
    torch.cuda.synchronize()
    s, ip, ln, bad = oracle.topk_to_ragged_slots(topk, bt, P, num_pages, next_n=next_n)
    assert bad == 0 and B.idx_get_device_status() == 0
    np.testing.assert_array_equal(indptr.cpu().numpy(), ip)
    np.testing.assert_array_equal(lens.cpu().numpy(), ln)
    np.testing.assert_array_equal(slots.cpu().numpy()[:ip[-1]], s)


def test_slots_row_to_seq_and_invalid_pages():
    P, num_pages = 4, 4
    bt = np.array([[3, 1, -1], [0, 2, 9]], np.int32)
    topk = np.array([[0, 5, 9, -1], [11, 4, -1, 8]], np.int32)
    r2s = np.array([1, 0], np.int32)
    slots = torch.empty(8, dtype=torch.int32, device="cuda")
    indptr = torch.empty(3, dtype=torch.int32, device="cuda")
    lens = torch.empty(2, dtype=torch.int32, device="cuda")
    B.idx_get_device_status()
    B.idx_topk_to_ragged_slots(_t(topk), _t(bt), P, num_pages, slots, indptr, lens,
                               row_to_seq=_t(r2s))
    torch.cuda.synchronize()
    s, ip, ln, bad = oracle.topk_to_ragged_slots(topk, bt, P, num_pages, row_to_seq=r2s)
    assert bad == 3 and B.idx_get_device_status() & B.DEV_BAD_PAGE
    np.testing.assert_array_equal(indptr.cpu().numpy(), ip)
    np.testing.assert_array_equal(slots.cpu().numpy()[:ip[-1]], s)


@pytest.mark.parametrize("rows,k", [(40, 1024), (48, 1000), (700, 300)])
def test_slots_row_to_seq_invalid_pages_many_rows(rows, k):
    """Invalid block-table entries and an explicit row-to-sequence map with
    several rows per CTA: (40, 1024) and (48, 1000) take the one-launch
    cluster kernel (three rows a CTA), (700, 300) the count and write
    kernels."""
    rng = np.random.default_rng(rows * 3 + k)
    P, num_pages, max_blocks, nseq = 16, 3000, 64, 29
    bt = np.stack([rng.permutation(num_pages)[:max_blocks] for _ in range(nseq)]).astype(np.int32)
    bad = rng.random(bt.shape) < 0.02
    bt[bad] = rng.choice([-1, num_pages, num_pages + 7], size=int(bad.sum()))
    r2s = rng.integers(0, nseq, size=rows).astype(np.int32)
    topk = rng.integers(-1, max_blocks * P + 40, size=(rows, k)).astype(np.int32)
    topk[rng.random((rows, k)) < 0.2] = -1
    slots = torch.empty(rows * k, dtype=torch.int32, device="cuda")
    indptr = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    lens = torch.empty(rows, dtype=torch.int32, device="cuda")
    B.idx_get_device_status()
    B.idx_topk_to_ragged_slots(_t(topk), _t(bt), P, num_pages, slots, indptr, lens,
                               row_to_seq=_t(r2s))
    torch.cuda.synchronize()
    s_, ip, ln, nbad = oracle.topk_to_ragged_slots(topk, bt, P, num_pages, row_to_seq=r2s)
    assert nbad > 0 and B.idx_get_device_status() & B.DEV_BAD_PAGE
    np.testing.assert_array_equal(indptr.cpu().numpy(), ip)
    np.testing.assert_array_equal(lens.cpu().numpy(), ln)
    np.testing.assert_array_equal(slots.cpu().numpy()[:ip[-1]], s_)


def _ascending(ora_idx):
    """The oracle's top-k rows in the library's layout: ascending indices,
    then -1 padding (the slot map keeps the order of its top-k rows)."""
    out = np.full_like(ora_idx, -1)
    for r, row in enumerate(ora_idx):
        v = np.sort(row[row >= 0])
        out[r, :len(v)] = v
    return out


# idx_topk_ragged_slots.  The cluster top-k counting slots as it writes, where
# the one-launch slot map does not take the call: (64, 65536, 2048) and
# (40, 40000, 2048) at more than four (row, 1024-entry step) pairs a CTA of
# its 16-CTA cluster, (2, 150000, 5000) at five steps a row, 4-token pages
# of 150000 and 262144-key rows (over 32768 block-table words a CTA).  The
# two-call forms: (12, 40000, 2048) (the one-launch slot map), 5000-key rows
# (one CTA a row), 160 rows of 40000 (320 cluster CTAs: the chunked top-k),
# 300001-key rows (past the cluster).  Beside each: an explicit
# row-to-sequence map or next_n rows a sequence, block-table entries outside
# the pool, positions past the table.
@pytest.mark.parametrize("rows,width,k,P,next_n,r2s,ties", [
    (64, 65536, 2048, 64, 1, False, None), (40, 40000, 2048, 64, 2, False, None),
    (2, 150000, 5000, 64, 1, True, None), (6, 150000, 512, 4, 3, True, 4),
    (3, 262144, 2048, 4, 1, False, None), (12, 40000, 2048, 64, 2, False, None),
    (9, 5000, 2048, 64, 1, True, None), (160, 40000, 512, 64, 2, False, None),
    (2, 300001, 2048, 64, 1, True, None)])
def test_topk_ragged_slots_fused(rows, width, k, P, next_n, r2s, ties):
    rng = np.random.default_rng(rows * 11 + width + k)
    x = _random_logits(rng, rows, width, tie_levels=ties, neg_inf_frac=0.05)
    lengths = rng.integers(0, width + 1, size=rows).astype(np.int32)
    lengths[0] = width
    nseq = -(-rows // next_n) if not r2s else max(2, rows // 3)
    max_blocks = -(-width // P) - 3                 # the last pages' keys map past the row
    num_pages = nseq * max_blocks + 100
    bt = np.stack([rng.permutation(num_pages)[:max_blocks] for _ in range(nseq)]).astype(np.int32)
    bad = rng.random(bt.shape) < 0.01
    bt[bad] = rng.choice([-1, num_pages, num_pages + 5], size=int(bad.sum()))
    bt[::2, 0] = -1                                  # first pages of every other sequence
    row_to_seq = rng.integers(0, nseq, size=rows).astype(np.int32) if r2s else None
    out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    slots = torch.empty(rows * k, dtype=torch.int32, device="cuda")
    indptr = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    lens = torch.full((rows,), -9, dtype=torch.int32, device="cuda")
    B.idx_get_device_status()
    B.idx_topk_ragged_slots(_t(x), _t(lengths), k, out, _t(bt), P, num_pages, slots, indptr,
                            lens, next_n=next_n,
                            row_to_seq=None if row_to_seq is None else _t(row_to_seq))
    torch.cuda.synchronize()
    ora = oracle.topk(x, lengths, k)
    assert_topk_exact(out.cpu().numpy(), ora)
    s, ip, ln, nbad = oracle.topk_to_ragged_slots(_ascending(ora), bt, P, num_pages,
                                                  next_n=next_n, row_to_seq=row_to_seq)
    assert bool(B.idx_get_device_status() & B.DEV_BAD_PAGE) == (nbad > 0)
    np.testing.assert_array_equal(lens.cpu().numpy(), ln)
    np.testing.assert_array_equal(indptr.cpu().numpy(), ip)
    np.testing.assert_array_equal(slots.cpu().numpy()[:ip[-1]], s)


def test_topk_ragged_slots_fused_all_valid():
    """No invalid slot: the device status stays clear (40 rows of 2048:
    the cluster top-k counts the slots)."""
    rng = np.random.default_rng(5)
    rows, width, k, P = 40, 65536, 2048, 64
    x = _random_logits(rng, rows, width)
    lengths = rng.integers(width // 2, width + 1, size=rows).astype(np.int32)
    max_blocks = width // P
    bt = np.stack([rng.permutation(rows * max_blocks)[:max_blocks]
                   for _ in range(rows)]).astype(np.int32)
    out = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    slots = torch.empty(rows * k, dtype=torch.int32, device="cuda")
    indptr = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    lens = torch.empty(rows, dtype=torch.int32, device="cuda")
    B.idx_get_device_status()
    B.idx_topk_ragged_slots(_t(x), _t(lengths), k, out, _t(bt), P, rows * max_blocks, slots,
                            indptr, lens)
    torch.cuda.synchronize()
    ora = oracle.topk(x, lengths, k)
    s, ip, ln, nbad = oracle.topk_to_ragged_slots(_ascending(ora), bt, P, rows * max_blocks)
    assert nbad == 0 and B.idx_get_device_status() == 0
    assert (ln == k).all()
    np.testing.assert_array_equal(indptr.cpu().numpy(), ip)
    np.testing.assert_array_equal(slots.cpu().numpy()[:ip[-1]], s)


def _cand_case(rng, rows, width, num_cand, blk, row_repeat=1, ties=None):
    if ties == "narrow":
        # distinct values inside one bin of the first radix digit
        x = rng.uniform(1.0, 1.2, size=(rows, width)).astype(np.float32)
    elif ties:
        x = rng.integers(0, ties, size=(rows, width)).astype(np.float32)
    else:
        x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < 0.05] = -np.inf
    ke = rng.integers(0, width + 1, size=rows).astype(np.int32)
    ke[0] = width
    ks = np.minimum(rng.integers(0, 300, size=rows), ke).astype(np.int32)
    crow = -(-rows // row_repeat)
    nblk = width // blk + 2
    cand = rng.integers(-2, nblk + 3, size=(crow, num_cand)).astype(np.int32)
    cand[:, 1] = cand[:, 0]          # a repeated id per row
    return x, ks, ke, cand


# The last three: candidate ids over a wide range (blocks of one key), and a
# threshold bin holding most keys, with ties left out and with distinct values.
@pytest.mark.parametrize("rows,width,num_cand,blk,k,rr,ties", [
    (3, 1000, 4, 64, 50, 1, None), (17, 20000, 64, 128, 2048, 1, None),
    (8, 9000, 64, 128, 300, 2, None), (5, 40000, 128, 128, 2048, 1, 3),
    (4, 5000, 16, 100, 4000, 1, None), (6, 70000, 64, 256, 2048, 1, 7),
    (4, 80000, 256, 1, 100, 1, None), (3, 20000, 128, 128, 2048, 1, 2),
    (3, 20000, 128, 128, 2048, 1, "narrow")])
def test_topk_candidates_equals_mask_then_topk(rows, width, num_cand, blk, k, rr, ties):
    rng = np.random.default_rng(rows * 31 + num_cand + blk)
    x, ks, ke, cand = _cand_case(rng, rows, width, num_cand, blk, rr, ties)
    masked = oracle.apply_candidate_mask(x.copy(), ks, ke, cand, blk, rr)
    ref = oracle.topk(masked, ke, k)
    out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    B.idx_topk_candidates(_t(x), _t(ke), k, out, _t(cand), blk, row_ks=_t(ks), row_repeat=rr)
    torch.cuda.synchronize()
    assert_topk_exact(out.cpu().numpy(), ref)
