"""The seeded input generators follow the stated recipe: value ranges and
scales, context-length laws, pools and block tables, candidate draws.  CPU
only, on small cases (the full workloads hold hundreds of MB of K pages)."""
import math

import numpy as np

import oracle
from sparse_attention_indexer_mxfp4_gb300 import synth


def test_contiguous_values_scales_and_weights():
    c = synth.contiguous_case(11, 64, 512, 64, 128, ke=np.full(64, 512))
    codes = np.unique(np.concatenate([c.q.reshape(-1), c.k.reshape(-1)]))
    vals = np.array([oracle.e4m3_to_double(int(b)) for b in codes])
    assert np.isfinite(vals).all() and np.abs(vals).max() <= 448.0   # clipped, no NaN codes
    ks = c.k_scale.astype(np.float64) * 448.0
    assert ks.min() >= 0.5 and ks.max() <= 2.0                        # U(0.5, 2) / 448
    assert abs(float(c.weights.std()) * math.sqrt(64) - 1.0) < 0.05   # N(0,1) / sqrt(H)
    # q ~ N(0, 1) before rounding to e4m3: the decoded values keep unit spread
    q = np.array([oracle.e4m3_to_double(int(b)) for b in c.q.reshape(-1)[:20000]])
    assert abs(q.std() - 1.0) < 0.05 and abs(q.mean()) < 0.05


def test_lognormal_context_lengths():
    ctx = synth.config4_context_lens()
    assert ctx.shape == (128,) and ctx.dtype == np.int32
    assert ctx.min() >= 2 and ctx.max() <= 131072
    # median 16384 and sigma 1 in log space, within sampling error of 128 draws
    assert 11000 <= np.median(ctx) <= 24000
    assert 0.7 <= float(np.log(ctx).std()) <= 1.3


def test_paged_pool_block_table_and_candidates():
    ctx = np.array([700, 64, 1500, 3000], np.int32)
    c = synth.paged_case(5, ctx, 2, 64, 128, 64, 4096, pool_factor=1.3, cand_num=8,
                         cand_block=128)
    npages = (ctx + 63) // 64
    assert c.num_pages == math.ceil(int(npages.sum()) * 1.3)
    used = []
    for b in range(c.B):
        row = c.block_table[b]
        assert (row[:npages[b]] >= 0).all() and (row[:npages[b]] < c.num_pages).all()
        assert (row[npages[b]:] == -1).all()
        used.extend(row[:npages[b]].tolist())
    assert len(used) == len(set(used))          # one permutation of the pool
    ke = np.clip(c.row_ends(), 0, c.width)
    for r in range(c.rows):
        live = (int(ke[r]) + 127) // 128
        ids = c.cand[r][c.cand[r] >= 0]
        assert len(ids) == min(live, 8) and len(set(ids.tolist())) == len(ids)
        assert (ids < live).all()
        assert (c.cand[r][len(ids):] == -1).all()


def test_mtp_row_ranges_end_at_each_rows_own_token():
    ctx = np.array([100, 2000], np.int32)
    c = synth.paged_case(7, ctx, 3, 64, 128, 64, 4096)
    # row j of a 3-token verify ends at context_len - 3 + j + 1
    np.testing.assert_array_equal(c.row_ends(), [98, 99, 100, 1998, 1999, 2000])
