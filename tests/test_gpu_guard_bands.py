"""Guard bands: every kernel writes its outputs and nothing around them.

Each output is a view into a larger buffer filled with a canary (a NaN with a
payload for floats, 0x5A5A5A5A for integers): guard rows before and after,
columns past the row stride's end, and the parts of an output the contract
leaves untouched (paged logits past each row's end, the standalone mask past
each row's end, the slot list past its last entry).  After the call every
canary must be intact and every element the contract writes must be
written."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth

pytestmark = pytest.mark.gpu

CANARY_F = np.array([0x7FC0CAFE], np.uint32).view(np.float32)[0]
CANARY_I = 0x5A5A5A5A
PR, PC = 3, 40  # guard rows above and below, guard columns after each row


def _guarded(rows, cols, dtype):
    fill = float(CANARY_F) if dtype == torch.float32 else CANARY_I
    full = torch.full((rows + 2 * PR, cols + PC), fill, dtype=dtype, device="cuda")
    if dtype == torch.float32:
        full.view(torch.int32).fill_(0x7FC0CAFE)
    return full, full[PR:PR + rows, :cols]


def _canary(a):
    a = np.asarray(a)
    if a.dtype == np.float32:
        return a.view(np.uint32) == np.uint32(0x7FC0CAFE)
    return a == CANARY_I


def _check(full, rows, cols, untouched=None, written=None):
    f = full.cpu().numpy()
    assert _canary(f[:PR]).all() and _canary(f[PR + rows:]).all(), "guard rows written"
    assert _canary(f[:, cols:]).all(), "columns past the row written"
    inner = f[PR:PR + rows, :cols]
    if untouched is not None:
        assert _canary(inner[untouched]).all(), "an element left to the caller was written"
    if written is not None:
        assert not _canary(inner[written]).any(), "an element of the output was not written"


def test_paged_logits_and_block_max_stay_in_bounds():
    ctx = np.array([5, 130, 700, 64, 1000, 3], np.int32)
    row_ks = np.array([0, 3, 100, 0, 512, 0], np.int32)
    c = synth.paged_case(201, ctx, 2, 64, 128, 64, 1100, pool_factor=1.3, ctx_per_row=True,
                         row_ks=row_ks)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    full, view = _guarded(c.rows, c.width, torch.float32)
    B.idx_paged_mqa_logits(d(c.q), None, d(c.weights), d(c.pages), d(c.block_table),
                           d(c.context_lens), c.next_n, c.page_size, c.fmt, view, c.width,
                           row_ks=d(c.row_ks), ctx_per_row=True)
    torch.cuda.synchronize()
    ke = np.clip(c.row_ends(), 0, c.width)
    col = np.arange(c.width)[None, :]
    _check(full, c.rows, c.width, untouched=col >= ke[:, None], written=col < ke[:, None])
    # block maxima: [rows, nb] inside a guarded buffer, every column written
    bs = 128
    nb = -(-c.width // bs)
    lfull, lview = _guarded(c.rows, c.width, torch.float32)
    bfull, bview = _guarded(c.rows, nb, torch.float32)
    B.idx_paged_mqa_logits_block_max(d(c.q), None, d(c.weights), d(c.pages), d(c.block_table),
                                     d(c.context_lens), c.next_n, c.page_size, c.fmt, lview,
                                     c.width, bview, bs, row_ks=d(c.row_ks), ctx_per_row=True)
    torch.cuda.synchronize()
    _check(lfull, c.rows, c.width, untouched=col >= ke[:, None], written=col < ke[:, None])
    _check(bfull, c.rows, nb, written=np.ones((c.rows, nb), bool))
    assert B.idx_get_device_status() == 0


def test_contiguous_logits_stay_in_bounds():
    M, N = 37, 333
    c = synth.contiguous_case(202, M, N, 64, 128, ke=np.arange(M) * 9 + 1)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    full, view = _guarded(M, N, torch.float32)
    B.idx_mqa_logits(d(c.q), None, d(c.weights), d(c.k), d(c.k_scale), d(c.ks), d(c.ke), c.fmt,
                     view)
    torch.cuda.synchronize()
    _check(full, M, N, written=np.ones((M, N), bool))


@pytest.mark.parametrize("width", [1000, 20000, 150000, 300000])
def test_topk_and_slots_stay_in_bounds(width):
    rng = np.random.default_rng(width)
    rows, k = 6, 512
    x = rng.standard_normal((rows, width)).astype(np.float32)
    lengths = np.array([0, 1, 100, width // 2, width, width - 3], np.int32)
    out_full, out = _guarded(rows, k, torch.int32)
    B.idx_topk(torch.from_numpy(x).cuda(), torch.from_numpy(lengths).cuda(), k, out)
    torch.cuda.synchronize()
    _check(out_full, rows, k, written=np.ones((rows, k), bool))
    # the slot map of those indices: rows of one sequence each, 64-token pages
    P = 64
    mb = -(-width // P)
    bt = torch.from_numpy(rng.permutation(mb).astype(np.int32).reshape(1, mb).repeat(rows, 0)).cuda()
    cap = rows * k
    slots_full = torch.full((cap + 64,), CANARY_I, dtype=torch.int32, device="cuda")
    indptr_full = torch.full((rows + 1 + 8,), CANARY_I, dtype=torch.int32, device="cuda")
    lens_full = torch.full((rows + 8,), CANARY_I, dtype=torch.int32, device="cuda")
    B.idx_topk_to_ragged_slots(out, bt, P, mb, slots_full[:cap], indptr_full[:rows + 1],
                               lens_full[:rows], next_n=1)
    torch.cuda.synchronize()
    ip = indptr_full.cpu().numpy()
    sl = slots_full.cpu().numpy()
    assert (ip[rows + 1:] == CANARY_I).all() and (lens_full.cpu().numpy()[rows:] == CANARY_I).all()
    total = int(ip[rows])
    assert not (sl[:total] == CANARY_I).any()
    assert (sl[total:] == CANARY_I).all(), "slot list written past its last entry"


def test_candidate_mask_stays_in_bounds():
    rows, width = 5, 2000
    rng = np.random.default_rng(9)
    x = rng.standard_normal((rows, width)).astype(np.float32)
    full, view = _guarded(rows, width, torch.float32)
    view.copy_(torch.from_numpy(x))
    ke = np.array([0, 1, 700, 1999, 2000], np.int32)
    cand = np.array([[0, 3], [1, -1], [2, 5], [0, 15], [7, 3]], np.int32)
    B.idx_apply_candidate_mask(view, None, torch.from_numpy(ke).cuda(),
                               torch.from_numpy(cand).cuda(), 128)
    torch.cuda.synchronize()
    f = full.cpu().numpy()
    assert _canary(f[:PR]).all() and _canary(f[PR + rows:]).all()
    assert _canary(f[:, width:]).all()
    inner = f[PR:PR + rows, :width]
    col = np.arange(width)[None, :]
    beyond = col >= ke[:, None]
    np.testing.assert_array_equal(inner[beyond], x[beyond])  # past each row's end untouched
