"""Host-side accounting without a GPU: which slot-map form the binding counts
for a call (its kernel count feeds the bench's gpu_launches), and the top-k
stage's algorithmic bytes with and without the slot map."""
import numpy as np
import pytest

import bench
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth


# (rows, k, max_blocks) -> kernels of one idx_topk_to_ragged_slots call on a
# device that holds a 16-CTA cluster: one cluster launch up to four (row,
# 1024-entry step) pairs and 32768 block-table words a CTA, else the count
# and write kernels, with the scan kernel between them above 4096 rows.
@pytest.mark.parametrize("rows,k,max_blocks,kernels", [
    (1, 1, 40, 1), (32, 2048, 2048, 1), (64, 1024, 70, 1), (4, 100, 20000, 1),
    (64, 2048, 512, 2), (16, 4097, 70, 2), (40, 100, 20000, 2), (20, 3000, 60, 2),
    (4096, 40, 40, 2), (4097, 40, 40, 3), (9000, 17, 40, 3), (8, 0, 40, 2)])
def test_slot_map_kernel_count(rows, k, max_blocks, kernels):
    assert B._slot_kernels(rows, k, max_blocks) == kernels


def test_topk_bytes_with_the_slot_map():
    """The stage that also runs the slot map writes k slots, a row length and
    an indptr entry per row, and the leading indptr entry."""
    c = synth.paged_case(3, [700, 64, 1300], 1, 64, 128, 64, 2048, pool_factor=1.2)
    base = bench.topk_bytes(c)
    assert base == 4.0 * bench.scored_keys(c) + 4.0 * c.rows * c.topk
    assert bench.topk_bytes(c, True) - base == 4.0 * c.rows * (c.topk + 2) + 4.0


def test_topk_bytes_count_only_live_keys():
    c = synth.paged_case(4, [5, 4096], 2, 64, 128, 64, 4096, pool_factor=1.1)
    ke = np.clip(c.row_ends(), 0, c.width)
    assert bench.scored_keys(c) == int(ke.sum())
