"""GPU parity of the logits kernels (through the C ABI) against the oracle,
element by element, on sizes that span several tiles and a ragged tail."""
import functools

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth
from sparse_attention_indexer_mxfp4_gb300.pipeline import IndexerStep
from parity import assert_logits_close

pytestmark = pytest.mark.gpu


def _t(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_contig(c: synth.ContiguousCase, ld=None):
    ld = c.N if ld is None else ld
    out = torch.full((c.M, ld), float("nan"), dtype=torch.float32, device="cuda")
    B.idx_mqa_logits(_t(c.q), _t(c.q_scale), _t(c.weights), _t(c.k), _t(c.k_scale), _t(c.ks),
                     _t(c.ke), c.fmt, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def ora_contig(c: synth.ContiguousCase):
    return oracle.mqa_logits(c.fmt, c.q, c.q_scale, c.weights, c.k, c.k_scale, c.ks, c.ke,
                             c.M, c.N, c.H, c.D)


def gpu_paged(c: synth.PagedCase, fused=True, num_ctas=0, gather=True, cand_topk=False):
    st = IndexerStep(c, fused_mask=fused, num_ctas=num_ctas, gather=gather, cand_topk=cand_topk)
    st.logits.fill_(float("nan"))
    st.logits_stage()
    torch.cuda.synchronize()
    return st.logits.cpu().numpy()


def ora_paged(c: synth.PagedCase, rows=None):
    out, bad = oracle.paged_mqa_logits(c.fmt, c.q, c.q_scale, c.weights, c.pages, c.page_stride,
                                       c.num_pages, c.block_table, c.context_lens, c.ctx_per_row,
                                       c.row_ks, c.B, c.next_n, c.H, c.D, c.page_size, c.width)
    if c.cand is not None:
        ke = np.clip(c.row_ends(), 0, c.width).astype(np.int32)
        oracle.apply_candidate_mask(out, c.row_ks, ke, c.cand, c.cand_block)
    return out, bad


def compare_paged(c, gpu, ref):
    ke = np.clip(c.row_ends(), 0, c.width)
    for r in range(c.rows):
        assert_logits_close(gpu[r, :ke[r]], ref[r, :ke[r]], f"row {r}")
        # columns past the row end are not written
        assert np.isnan(gpu[r, ke[r]:]).all(), f"row {r}: tail was written"


# ----------------------------------------------------------------- contiguous


@pytest.mark.parametrize("M", [1, 3, 10])
def test_contig_fp8_ragged(M):
    N = 333  # two full 128-key tiles and a ragged tail of 77
    ke = np.array([333, 1, 0, 200, 128, 129, 333, 64, 300, 77][:M])
    ks = np.array([0, 0, 0, 50, 127, 0, 300, 0, 299, 77][:M])
    c = synth.contiguous_case(100 + M, M, N, 64, 128, ke=ke, ks=ks)
    assert_logits_close(gpu_contig(c), ora_contig(c))


def test_contig_fp8_q_scale_and_negative_k_scale():
    c = synth.contiguous_case(7, 6, 260, 64, 128, ke=[260] * 6, with_q_scale=True)
    c.k_scale[::3] *= -1.0
    c.q_scale[1, ::5] *= -1.0
    assert_logits_close(gpu_contig(c), ora_contig(c))


def test_contig_fp8_negative_k_scale_no_q_scale():
    c = synth.contiguous_case(8, 5, 256, 64, 128, ke=[256] * 5)
    c.k_scale[1::2] *= -1.0
    assert_logits_close(gpu_contig(c), ora_contig(c))


def test_contig_fp8_wide_ld():
    c = synth.contiguous_case(9, 9, 200, 64, 128, ke=np.arange(9) * 20 + 40)
    g = gpu_contig(c, ld=512)
    assert_logits_close(g[:, :200], ora_contig(c))
    assert np.isnan(g[:, 200:]).all()


def test_contig_fp8_config1_full():
    c = synth.config1()
    assert_logits_close(gpu_contig(c), ora_contig(c))


def test_contig_fp8_many_groups():
    # enough rows that the launch groups four rows per MMA (N = 256)
    M, N = 1200, 1100
    pos = np.arange(M) + (N - M) % N
    c = synth.contiguous_case(11, M, N, 64, 128, ke=np.minimum(pos + 1, N))
    g = gpu_contig(c)
    rows = np.r_[0:6, 597:603, M - 6:M]
    sub = synth.ContiguousCase(c.fmt, len(rows), N, 64, 128, c.q[rows], None, c.weights[rows],
                               c.k, c.k_scale, c.ks[rows], c.ke[rows], c.topk)
    assert_logits_close(g[rows], ora_contig(sub))


@pytest.mark.parametrize("rare", [False, True], ids=["common", "q_scale+negative_k_scale"])
def test_contig_fp8_four_row_groups_ragged(rare):
    # four-row groups (each group's rows reduced by two epilogue warpgroups),
    # a last group of three rows, and a ragged key tail; with per-head q
    # scales and negative key scales the epilogue takes its other path
    M, N = 1203, 777
    pos = np.arange(M) % N
    c = synth.contiguous_case(12 + rare, M, N, 64, 128, ke=pos + 1,
                              ks=np.maximum(pos - 500, 0), with_q_scale=rare)
    if rare:
        c.k_scale[::7] *= -1.0
        c.q_scale[:, ::5] *= -1.0
    assert_logits_close(gpu_contig(c), ora_contig(c))


@pytest.mark.parametrize("M", [1, 5])
def test_contig_mxfp4(M):
    N = 332
    c = synth.contiguous_case(20 + M, M, N, 64, 128, ke=[332, 100, 1, 331, 200][:M],
                              ks=[0, 3, 0, 129, 64][:M], fmt=synth.FMT_MXFP4)
    assert_logits_close(gpu_contig(c), ora_contig(c))


# ---------------------------------------------------------------------- paged


CTX = [0, 1, 63, 64, 65, 129, 300, 777]


@pytest.mark.parametrize("next_n", [1, 2, 4])
@pytest.mark.parametrize("P", [64, 128])
def test_paged_fp8(next_n, P):
    ctx = [max(v, next_n) for v in CTX]
    c = synth.paged_case(30 + next_n + P, ctx, next_n, 64, 128, P, 1024, pool_factor=1.5)
    gpu = gpu_paged(c)
    ref, bad = ora_paged(c)
    assert bad == 0
    compare_paged(c, gpu, ref)


def test_paged_fp8_ctx_per_row_and_row_ks():
    ctx = np.array([10, 200, 130, 131, 700, 699], np.int32)
    row_ks = np.array([0, 17, 64, 130, 5, 600], np.int32)
    c = synth.paged_case(41, ctx, 2, 64, 128, 64, 768, pool_factor=1.3, ctx_per_row=True,
                         row_ks=row_ks)
    compare_paged(c, gpu_paged(c), ora_paged(c)[0])


@pytest.mark.parametrize("next_n", [1, 2])
def test_paged_fused_candidate_mask(next_n):
    ctx = [1, 130, 500, 1000, 2049]
    c = synth.paged_case(50 + next_n, ctx, next_n, 64, 128, 64, 4096, pool_factor=1.2,
                         cand_num=5, cand_block=128)
    c.cand[0, 1] = 999   # out-of-range ids are ignored
    c.cand[1, 2] = -7
    ref, _ = ora_paged(c)
    compare_paged(c, gpu_paged(c, fused=True), ref)
    compare_paged(c, gpu_paged(c, fused=True, gather=False), ref)
    compare_paged(c, gpu_paged(c, fused=False), ref)


@functools.lru_cache(maxsize=None)
def _sparse_candidate_case(fmt):
    ctx = [40000, 3, 700, 16385, 9000, 257]
    c = synth.paged_case(90 + fmt, ctx, 2, 64, 128, 64, 40960, fmt=fmt, pool_factor=1.2,
                         cand_num=6, cand_block=128)
    c.cand[2, 0] = 10**6  # far out of range
    c.cand[3, :] = -1     # a row without candidates
    return c, ora_paged(c)[0]


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4])
@pytest.mark.parametrize("num_ctas", [0, 1, 5, 1000])
def test_paged_candidate_gather_plan(fmt, num_ctas):
    """Sparse candidates over long rows: most tiles hold no candidate and are
    only written -inf, and the work split follows the candidate tiles."""
    c, ref = _sparse_candidate_case(fmt)
    compare_paged(c, gpu_paged(c, num_ctas=num_ctas), ref)


@pytest.mark.parametrize("num_ctas", [0, 7])
def test_paged_candidate_gather_plan_four_rows(num_ctas):
    """Four rows a sequence (next_n = 4) with candidates: the gather plan on
    four-row groups, whose accumulators are split into two column halves."""
    ctx = [40000, 9, 700, 16385, 260]
    c = synth.paged_case(95, ctx, 4, 64, 128, 64, 40960, pool_factor=1.2, cand_num=6,
                         cand_block=128)
    c.cand[1, :] = -1     # a row without candidates
    ref = ora_paged(c)[0]
    compare_paged(c, gpu_paged(c, num_ctas=num_ctas), ref)
    compare_paged(c, gpu_paged(c, num_ctas=num_ctas, gather=False), ref)


@pytest.mark.parametrize("fmt", [synth.FMT_FP8, synth.FMT_MXFP4])
def test_paged_candidates_only_writes_candidate_tiles(fmt):
    """idx_paged_mqa_logits_candidates: every candidate key is written and
    matches; columns outside the plan's tiles stay untouched (NaN here)."""
    c, ref = _sparse_candidate_case(fmt)
    gpu = gpu_paged(c, cand_topk=True)
    ke = np.clip(c.row_ends(), 0, c.width)
    for r in range(c.rows):
        live = np.isfinite(ref[r, :ke[r]])
        assert_logits_close(gpu[r, :ke[r]][live], ref[r, :ke[r]][live], f"row {r}")
        wrote = ~np.isnan(gpu[r, :ke[r]])
        assert wrote[live].all()
        # whatever was written is either a candidate logit or -inf
        assert np.isneginf(gpu[r, :ke[r]][wrote & ~live]).all()
        assert np.isnan(gpu[r, ke[r]:]).all()


@pytest.mark.parametrize("next_n", [1, 2])
def test_paged_mxfp4(next_n):
    ctx = [max(v, next_n) for v in CTX]
    c = synth.paged_case(60 + next_n, ctx, next_n, 64, 128, 64, 1024, fmt=synth.FMT_MXFP4,
                         pool_factor=1.5)
    compare_paged(c, gpu_paged(c), ora_paged(c)[0])


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 1000])
def test_paged_grid_sizes_agree(num_ctas):
    c = synth.paged_case(70, [900, 5, 333, 1200], 2, 64, 128, 64, 2048, pool_factor=1.1)
    compare_paged(c, gpu_paged(c, num_ctas=num_ctas), ora_paged(c)[0])


@pytest.mark.parametrize("next_n", [1, 2])
@pytest.mark.parametrize("num_ctas", [1, 3, 7, 1000])
def test_paged_mxfp4_grid_sizes_agree(next_n, num_ctas):
    """MXFP4 kernels take their tiles from descriptors (one-row groups on two
    accumulators, two-row groups on three): every split of the units over
    the CTAs, empty CTAs included, gives the oracle's logits."""
    c = synth.paged_case(72 + next_n, [900, 5, 333, 1200, 64], next_n, 64, 128, 64, 2048,
                         fmt=synth.FMT_MXFP4, pool_factor=1.1)
    compare_paged(c, gpu_paged(c, num_ctas=num_ctas), ora_paged(c)[0])


def test_paged_bad_page_sets_status_and_masks():
    c = synth.paged_case(80, [300, 300], 1, 64, 128, 64, 512, pool_factor=1.0)
    c.block_table[1, 2] = c.num_pages + 5  # keys 128..191 of sequence 1
    B.idx_get_device_status()  # clear
    gpu = gpu_paged(c)
    assert B.idx_get_device_status() & B.DEV_BAD_PAGE
    ref, bad = ora_paged(c)
    assert bad == 64
    compare_paged(c, gpu, ref)
    assert B.idx_get_device_status() == 0  # read-and-clear
