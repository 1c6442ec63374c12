"""GPU parity of idx_paged_mqa_logits_topk, the logits -> top-k prefilter:
the fused call's logits are within the logits tolerance of the oracle's,
element by element over every row's [0, ke); its top-k indices and block
maxima equal the oracle's top-k and block maxima of the fused call's own
logits exactly, and its block maxima are within the logits tolerance of the
oracle's block maxima of the oracle's logits."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth
from sparse_attention_indexer_mxfp4_gb300.pipeline import IndexerStep
from parity import assert_logits_close, assert_topk_exact

pytestmark = pytest.mark.gpu


def _run(c, fused):
    st = IndexerStep(c, fused_topk=fused)
    st.logits.fill_(float("nan"))
    st.topk.fill_(-7)
    B.idx_get_device_status()
    st.logits_stage()
    st.topk_stage()
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    bm = st.block_max.cpu().numpy() if st.source else None
    return st, st.logits.cpu().numpy(), st.topk.cpu().numpy(), bm


def _compare(c):
    st_f, lf, tf, bf = _run(c, True)
    assert st_f.fused_topk
    ref, bad = oracle.paged_mqa_logits(c.fmt, c.q, c.q_scale, c.weights, c.pages, c.page_stride,
                                       c.num_pages, c.block_table, c.context_lens, c.ctx_per_row,
                                       c.row_ks, c.B, c.next_n, c.H, c.D, c.page_size, c.width)
    assert bad == 0
    ke = np.clip(c.row_ends(), 0, c.width).astype(np.int32)
    for r in range(c.rows):
        assert_logits_close(lf[r, :ke[r]], ref[r, :ke[r]], f"fused logits row {r}")
    own = np.where(np.isnan(lf), -np.inf, lf)
    ora = oracle.topk(own, ke, c.topk)
    assert_topk_exact(tf, ora, "fused top-k on its own logits")
    if bf is not None:
        ks = np.zeros_like(ke) if c.row_ks is None else np.minimum(c.row_ks, ke).astype(np.int32)
        np.testing.assert_array_equal(bf, oracle.block_max(own, ks, ke, c.source_block))
        ref_bm = oracle.block_max(np.where(np.isnan(ref), -np.inf, ref), ks, ke, c.source_block)
        assert_logits_close(bf, ref_bm, "fused block maxima")


@pytest.mark.parametrize("next_n", [1, 2])
@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4])
def test_fused_topk_matches_separate_calls(next_n, fmt):
    # rows from empty to several 8192-key chunks, some shorter than k
    ctx = [0, 5, 700, 8192, 8193, 20000, 33000]
    ctx = [max(v, next_n) for v in ctx]
    c = synth.paged_case(110 + 4 * next_n + fmt, ctx, next_n, 64, 128, 64, 33024, fmt=fmt,
                         pool_factor=1.2, topk=1000)
    _compare(c)


def test_fused_topk_with_block_maxima_and_row_ks():
    ctx = np.array([100, 9000, 20000, 20001, 16384, 30000], np.int32)
    row_ks = np.array([0, 17, 4096, 0, 9000, 5], np.int32)
    c = synth.paged_case(120, ctx, 2, 64, 128, 64, 30720, pool_factor=1.2, ctx_per_row=True,
                         row_ks=row_ks, topk=2048)
    c.source_block, c.source_cands = 128, 16
    _compare(c)


def test_fused_topk_heavy_ties():
    # equal logits everywhere in a row: zero weights give logits of 0 on every
    # live key, so the threshold bin holds the whole row
    ctx = [9000, 25000, 17000]
    c = synth.paged_case(130, ctx, 1, 64, 128, 64, 25088, pool_factor=1.2, topk=3000)
    c.weights[1] = 0.0
    _compare(c)
