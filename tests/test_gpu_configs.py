"""The benchmark workloads at full size, in the launch configuration the
benchmark times (IndexerStep).

* Logits: the oracle computes 16 sampled sequences per paged workload (the
  longest and the shortest among them, the rest evenly spaced) and sampled
  rows of the contiguous ones; each is compared element by element.  With
  152 persistent CTAs sharing 32 to 128 sequences, every sequence is split
  between CTAs, so each sample also crosses the split's boundaries.
* Top-k: every row of the workload is compared exactly with the oracle's
  top-k of the GPU's own logits (the candidate mask applied for the
  candidate pipeline); the sampled rows also end to end against the
  oracle's logits with the near-tie rule, and exactly on the oracle's own
  logits.
* Slots: the ragged rows of the sampled rows are the oracle's slot map of
  the same top-k sets."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth
from sparse_attention_indexer_mxfp4_gb300.pipeline import IndexerStep
from parity import assert_logits_close, assert_topk_exact, assert_topk_near_tie

pytestmark = pytest.mark.gpu


def _sub_paged(c: synth.PagedCase, seqs):
    """The same problem restricted to some sequences (rows are independent)."""
    seqs = np.asarray(seqs)
    rows = (seqs[:, None] * c.next_n + np.arange(c.next_n)[None, :]).reshape(-1)
    ctx = c.context_lens[rows] if c.ctx_per_row else c.context_lens[seqs]
    sub = synth.PagedCase(c.fmt, len(seqs), c.next_n, c.H, c.D, c.page_size, c.num_pages,
                          c.page_stride, c.width, c.q[rows],
                          None if c.q_scale is None else c.q_scale[rows], c.weights[rows],
                          c.pages, c.block_table[seqs], ctx, c.ctx_per_row, c.topk,
                          None if c.row_ks is None else c.row_ks[rows],
                          None if c.cand is None else c.cand[rows], c.cand_block)
    return sub, rows


def _sample_seqs(c: synth.PagedCase, n: int = 16):
    """n sequences: the longest, the shortest, the rest evenly spaced."""
    lens = np.clip(c.row_ends(), 0, c.width).reshape(c.B, c.next_n).max(axis=1)
    pick = set(np.linspace(0, c.B - 1, max(n - 2, 1)).round().astype(int).tolist())
    pick |= {int(np.argmax(lens)), int(np.argmin(lens))}
    return sorted(pick)


def _assert_all_rows_topk_on_own_logits(st, c, what):
    """Every row: the GPU's top-k equals the oracle's top-k of the GPU's own
    logits over [0, ke) (candidate-masked when the step selects among
    candidates, whose other columns the step leaves unwritten)."""
    ke = (np.clip(c.row_ends(), 0, c.width) if st.paged else c.ke).astype(np.int32)
    own = st.logits.cpu().numpy()
    if st.paged and c.cand is not None:
        ks = None if c.row_ks is None else c.row_ks.astype(np.int32)
        oracle.apply_candidate_mask(own, ks, ke, c.cand, c.cand_block)
    own = np.where(np.isnan(own), -np.inf, own)
    for r in range(own.shape[0]):
        own[r, ke[r]:] = -np.inf
    assert_topk_exact(st.topk.cpu().numpy(), oracle.topk(own, ke, c.topk),
                      f"{what}: top-k of every row on the GPU's logits")


def _oracle_paged_rows(sub):
    out, bad = oracle.paged_mqa_logits(sub.fmt, sub.q, sub.q_scale, sub.weights, sub.pages,
                                       sub.page_stride, sub.num_pages, sub.block_table,
                                       sub.context_lens, sub.ctx_per_row, sub.row_ks, sub.B,
                                       sub.next_n, sub.H, sub.D, sub.page_size, sub.width)
    ke = np.clip(sub.row_ends(), 0, sub.width).astype(np.int32)
    if sub.cand is not None:
        oracle.apply_candidate_mask(out, sub.row_ks, ke, sub.cand, sub.cand_block)
    return out, ke, bad


@pytest.fixture(scope="module", params=[3, 4, 5, 6])
def paged_cfg(request):
    return request.param, synth.CONFIGS[request.param]()


@pytest.mark.parametrize("cand_topk", [True, False])
def test_paged_config(paged_cfg, cand_topk):
    cfg, c = paged_cfg
    if c.cand is None and not cand_topk:
        pytest.skip("no candidates: one pipeline")
    st = IndexerStep(c, cand_topk=cand_topk)
    st.run()
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    _assert_all_rows_topk_on_own_logits(st, c, f"config {cfg}")
    seqs = _sample_seqs(c)
    sub, rows = _sub_paged(c, seqs)
    ref, ke, bad = _oracle_paged_rows(sub)
    assert bad == 0
    gl = st.logits[torch.from_numpy(rows).cuda()].cpu().numpy()
    for i in range(len(rows)):
        # the candidate pipeline writes only tiles holding candidate keys
        cols = np.isfinite(ref[i, :ke[i]]) if st.cand_topk else slice(None)
        assert_logits_close(gl[i, :ke[i]][cols], ref[i, :ke[i]][cols],
                            f"config {cfg} row {rows[i]}")
    # top-k: end to end (near-tie rule), then exact on the oracle's logits
    ora_idx = oracle.topk(np.where(np.isnan(ref), -np.inf, ref), ke, c.topk)
    gpu_idx = st.topk[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_topk_near_tie(gpu_idx, ora_idx, ref, ke, c.topk, f"config {cfg}")
    ref_dev = torch.from_numpy(np.where(np.isnan(ref), -np.inf, ref).astype(np.float32)).cuda()
    out = torch.empty((len(rows), c.topk), dtype=torch.int32, device="cuda")
    B.idx_topk(ref_dev, torch.from_numpy(ke).cuda(), c.topk, out)
    assert_topk_exact(out.cpu().numpy(), ora_idx, f"config {cfg} top-k on oracle logits")
    # slots: the ragged rows of the sampled rows are the oracle's slot map of
    # the same top-k sets
    indptr = st.indptr.cpu().numpy()
    slots = st.slots.cpu().numpy()
    s, ip, ln, _ = oracle.topk_to_ragged_slots(ora_idx, sub.block_table, c.page_size,
                                               c.num_pages, next_n=c.next_n)
    for i, r in enumerate(rows):
        g = np.sort(slots[indptr[r]:indptr[r + 1]])
        o = np.sort(s[ip[i]:ip[i + 1]])
        if len(np.setxor1d(gpu_idx[i][gpu_idx[i] >= 0], ora_idx[i][ora_idx[i] >= 0])) == 0:
            np.testing.assert_array_equal(g, o)
    assert indptr[0] == 0 and (np.diff(indptr) == st.lens.cpu().numpy()).all()
    if st.source:
        # candidate source: block maxima bit-exact on the GPU's own logits and
        # within tolerance of the oracle's; the pool (best blocks) with the
        # near-tie rule, and exactly on the GPU's own block maxima
        bs = c.source_block
        gb = st.block_max[torch.from_numpy(rows).cuda()].cpu().numpy()
        bl = ((ke + bs - 1) // bs).astype(np.int32)
        own = oracle.block_max(np.where(np.isnan(gl), -np.inf, gl), None, ke, bs)
        np.testing.assert_array_equal(gb, own)
        ref_bm = oracle.block_max(np.where(np.isnan(ref), -np.inf, ref), None, ke, bs)
        assert_logits_close(gb, ref_bm, f"config {cfg} block maxima")
        gpu_pool = st.pool[torch.from_numpy(rows).cuda()].cpu().numpy()
        ora_pool = oracle.topk(ref_bm, bl, c.source_cands)
        assert_topk_near_tie(gpu_pool, ora_pool, ref_bm, bl, c.source_cands,
                             f"config {cfg} candidate pool")
        assert_topk_exact(gpu_pool, oracle.topk(own, bl, c.source_cands),
                          f"config {cfg} pool on the GPU block maxima")


@pytest.mark.parametrize("cfg", [1, 2])
def test_contiguous_config(cfg):
    c = synth.CONFIGS[cfg]()
    st = IndexerStep(c)
    st.run()
    torch.cuda.synchronize()
    _assert_all_rows_topk_on_own_logits(st, c, f"config {cfg}")
    rows = np.unique(np.r_[0:3, np.linspace(0, c.M - 1, 13).round().astype(int), c.M - 3:c.M])
    sub = synth.ContiguousCase(c.fmt, len(rows), c.N, c.H, c.D, c.q[rows], None, c.weights[rows],
                               c.k, c.k_scale, c.ks[rows], c.ke[rows], c.topk)
    ref = oracle.mqa_logits(sub.fmt, sub.q, None, sub.weights, sub.k, sub.k_scale, sub.ks,
                            sub.ke, sub.M, sub.N, sub.H, sub.D)
    gl = st.logits[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_logits_close(gl, ref, f"config {cfg}")
    ora_idx = oracle.topk(ref, sub.ke, c.topk)
    gpu_idx = st.topk[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_topk_near_tie(gpu_idx, ora_idx, ref, sub.ke, c.topk, f"config {cfg}")


def test_producer_config():
    """Config 7 (K/Q producers of an 8192-token prefill chunk) through
    ProducerStep: sampled tokens against the oracle, with the same rounding
    rule as the producer tests."""
    from sparse_attention_indexer_mxfp4_gb300.pipeline import ProducerStep
    from test_gpu_producers import _bits_ok, _check_block, _decode
    c = synth.CONFIGS[7]()
    st = ProducerStep(c)
    st.run()
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    toks = np.array([0, 1, c.T // 2, c.T - 1])
    kbits = torch.from_numpy(c.k_pre[toks]).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    pages = np.zeros((c.num_pages, c.page_stride), np.uint8)
    bad, pre, obits = oracle.k_norm_rope_store(c.fmt, kbits, c.positions[toks], c.cos_sin,
                                               c.rope_dim, c.norm_weight, c.eps, pages,
                                               c.page_size, c.slots[toks])
    assert bad == 0
    g = st.pages.cpu().numpy()
    rowb, sbytes, span = c.D // 2, c.D // 32, 32
    for i, t in enumerate(toks):
        pg, off = divmod(int(c.slots[t]), c.page_size)
        dec = _decode(c.fmt, g[pg, off * rowb:(off + 1) * rowb])
        sb = g[pg, c.page_size * rowb + off * sbytes:c.page_size * rowb + (off + 1) * sbytes]
        for j in range(c.D // span):
            seg = pre[i, j * span:(j + 1) * span]
            assert _bits_ok(c.fmt, np.abs(seg).max(), int(sb[j]), int(obits[i, j]))
            if int(sb[j]) == int(obits[i, j]):
                _check_block(c.fmt, seg * 2.0 ** (127 - int(obits[i, j])),
                             dec[j * span:(j + 1) * span])
    qbits = torch.from_numpy(c.q[toks]).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    bad, o_q, o_sf, o_w, qpre, qob = oracle.q_rope_quant(c.fmt, qbits, c.positions[toks],
                                                         c.cos_sin, c.rope_dim, c.weights[toks],
                                                         c.weight_scale)
    assert bad == 0
    gq = st.q_out.cpu().numpy()[toks].reshape(len(toks) * c.H, rowb)
    gsf = st.q_sf.cpu().numpy()[toks].reshape(-1).view(np.uint8).reshape(-1, 4)
    np.testing.assert_array_equal(st.weights_out.cpu().numpy()[toks], o_w)
    for th in range(len(toks) * c.H):
        dec = _decode(c.fmt, gq[th])
        for j in range(c.D // span):
            seg = qpre[th, j * span:(j + 1) * span]
            assert _bits_ok(c.fmt, np.abs(seg).max(), int(gsf[th, j]), int(qob[th, j]))
            if int(gsf[th, j]) == int(qob[th, j]):
                _check_block(c.fmt, seg * 2.0 ** (127 - int(qob[th, j])),
                             dec[j * span:(j + 1) * span])
