"""GPU parity of the candidate source (idx_paged_mqa_logits_block_max): its
logits against the oracle, its block maxima bit-exact against the oracle's
block maxima of the GPU's own logits and within the logits tolerance against
the oracle's block maxima of the oracle's logits; columns past the blocks
are not written."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth
from parity import assert_logits_close

pytestmark = pytest.mark.gpu


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(c, block, num_ctas=0):
    nb = -(-c.width // block)
    ld = nb + 3
    logits = torch.full((c.rows, c.width), float("nan"), dtype=torch.float32, device="cuda")
    bmax = torch.full((c.rows, ld), float("nan"), dtype=torch.float32, device="cuda")
    pages = _t(c.pages)
    B.idx_paged_mqa_logits_block_max(_t(c.q), _t(c.q_scale), _t(c.weights), pages,
                                     _t(c.block_table), _t(c.context_lens), c.next_n,
                                     c.page_size, c.fmt, logits, c.width, bmax, block,
                                     row_ks=_t(c.row_ks), ctx_per_row=c.ctx_per_row,
                                     num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    return logits.cpu().numpy(), bmax.cpu().numpy(), nb


def _check(c, block, num_ctas=0):
    gl, gb, nb = _run(c, block, num_ctas)
    ref, bad = oracle.paged_mqa_logits(c.fmt, c.q, c.q_scale, c.weights, c.pages, c.page_stride,
                                       c.num_pages, c.block_table, c.context_lens,
                                       c.ctx_per_row, c.row_ks, c.B, c.next_n, c.H, c.D,
                                       c.page_size, c.width)
    assert bad == 0
    ke = np.clip(c.row_ends(), 0, c.width).astype(np.int32)
    ks = np.zeros_like(ke) if c.row_ks is None else np.minimum(c.row_ks, ke).astype(np.int32)
    for r in range(c.rows):
        assert_logits_close(gl[r, :ke[r]], ref[r, :ke[r]], f"logits row {r}")
    # bit-exact against the block maxima of the GPU's own logits
    own = oracle.block_max(np.where(np.isnan(gl), -np.inf, gl), ks, ke, block)
    np.testing.assert_array_equal(gb[:, :nb], own)
    # within the logits tolerance of the oracle's whole step
    assert_logits_close(gb[:, :nb], oracle.block_max(ref, ks, ke, block), "block maxima")
    assert np.isnan(gb[:, nb:]).all(), "columns past the blocks were written"


@pytest.mark.parametrize("block", [32, 64, 100, 128, 300])
def test_block_max_fp8_mtp(block):
    ctx = [2, 63, 64, 129, 700, 2049, 4000]
    c = synth.paged_case(70 + block, ctx, 2, 64, 128, 64, 4096, pool_factor=1.3)
    _check(c, block)


def test_block_max_fp8_row_ks_relative_blocks():
    ctx = np.array([10, 200, 130, 131, 700, 699], np.int32)
    row_ks = np.array([0, 17, 64, 130, 5, 600], np.int32)
    c = synth.paged_case(77, ctx, 2, 64, 128, 64, 768, pool_factor=1.3, ctx_per_row=True,
                         row_ks=row_ks)
    for block in (32, 48, 128):
        _check(c, block)


@pytest.mark.parametrize("next_n", [1, 2])
def test_block_max_mxfp4(next_n):
    ctx = [5, 300, 1000, 3000]
    c = synth.paged_case(80 + next_n, ctx, next_n, 64, 128, 64, 3072, fmt=synth.FMT_MXFP4,
                         pool_factor=1.2)
    _check(c, 128)


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 1000])
def test_block_max_grid_sizes(num_ctas):
    """The block-maxima kernel takes its tiles from descriptors: CTA ranges
    that end inside a group, groups with fewer tiles than accumulators and
    CTAs without units (1000) all end on the same outputs."""
    ctx = [2, 63, 700, 2049, 130, 4000]
    c = synth.paged_case(91, ctx, 2, 64, 128, 64, 4096, pool_factor=1.3)
    _check(c, 128, num_ctas)
