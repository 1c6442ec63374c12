"""One indexer step over resident device buffers: logits (with the range and,
when given, the candidate mask fused in), per-row top-k, and for paged
caches the top-k -> ragged slot map.  Every stage is a libidx.so call."""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B
from .synth import ContiguousCase, PagedCase


def _dev(a, device, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class IndexerStep:
    """Device-resident inputs and outputs of one workload and the calls of one
    step.  ``fused_mask=False`` applies the candidate mask with the standalone
    kernel after the logits instead of inside them; ``gather=False`` keeps the
    fused mask but scores every key (no candidate gather plan).
    ``cand_topk`` (with a fused mask and the gather plan) writes only the
    tiles holding candidate keys and selects with idx_topk_candidates, which
    reads only the candidate blocks; the top-k and slots are the same, the
    logits outside those tiles are left unwritten.  ``kv_from`` (another
    IndexerStep of the same case) shares its device K cache instead of
    uploading a second copy; with ``kv_copy`` it takes a device copy of it
    instead (the same keys at other addresses).  ``fused_topk`` (paged, no candidate list) runs
    the logits and the row top-k as one idx_paged_mqa_logits_topk call, the
    logits kernel counting the top-k's first digit; its logits stage then
    holds the top-k too.  ``fused_slots`` (paged, the row top-k as its own
    call) runs the top-k and the slot map as one idx_topk_ragged_slots call,
    the top-k counting each row's valid slots; its top-k stage then holds
    the slot map too."""

    def __init__(self, case, device="cuda", fused_mask: bool = True, num_ctas: int = 0,
                 gather: bool = True, cand_topk: bool = True, kv_from=None,
                 fused_topk: bool = False, kv_copy: bool = False, fused_slots: bool = True):
        self.case = case
        self.device = torch.device(device)
        self.fused_mask = fused_mask
        self.gather = gather
        self.cand_topk = bool(cand_topk and gather and fused_mask)
        self.fused_topk = bool(fused_topk and isinstance(case, PagedCase) and case.cand is None)
        self.num_ctas = num_ctas
        self.fused_slots = fused_slots
        d = self.device
        self.paged = isinstance(case, PagedCase)
        self.q = _dev(case.q, d)
        self.weights = _dev(case.weights, d)
        self.q_scale = _dev(case.q_scale, d)
        if self.paged:
            if kv_from is not None:
                self.pages = kv_from.pages.clone() if kv_copy else kv_from.pages
            else:
                self.pages = _dev(case.pages, d)
            self.block_table = _dev(case.block_table, d)
            self.context_lens = _dev(case.context_lens, d)
            self.row_ks = _dev(case.row_ks, d)
            self.cand = _dev(case.cand, d)
            ke = np.clip(case.row_ends(), 0, case.width).astype(np.int32)
            # each row's end, derived on the device from the context lengths
            # by the library (idx_row_ends) at the head of every step
            self.lengths = torch.empty(case.rows, dtype=torch.int32, device=d)
            self.rows, self.width = case.rows, case.width
            self.max_blocks = case.max_blocks
        else:
            if kv_from is not None:
                self.k = kv_from.k.clone() if kv_copy else kv_from.k
                self.k_scale = kv_from.k_scale.clone() if kv_copy else kv_from.k_scale
            else:
                self.k, self.k_scale = _dev(case.k, d), _dev(case.k_scale, d)
            self.ks = _dev(case.ks, d)
            self.ke = _dev(case.ke, d)
            self.lengths = self.ke
            self.rows, self.width = case.M, case.N
        self.k_top = case.topk
        self.logits = torch.empty((self.rows, self.width), dtype=torch.float32, device=d)
        self.topk = torch.empty((self.rows, self.k_top), dtype=torch.int32, device=d)
        if self.paged:
            self.slots = torch.empty(max(1, self.rows * self.k_top), dtype=torch.int32, device=d)
            self.indptr = torch.empty(self.rows + 1, dtype=torch.int32, device=d)
            self.lens = torch.empty(self.rows, dtype=torch.int32, device=d)
        self.source = self.paged and getattr(case, "source_block", 0) > 0
        if self.source:
            # candidate source: block maxima, and the best blocks of each row
            bs = case.source_block
            self.nblocks = -(-case.width // bs)
            self.block_max = torch.empty((self.rows, self.nblocks), dtype=torch.float32, device=d)
            ks = np.zeros(self.rows, np.int64) if case.row_ks is None else case.row_ks
            span = np.maximum(ke - np.minimum(ks, ke), 0)
            self.block_lens = _dev(((span + bs - 1) // bs).astype(np.int32), d)
            self.pool = torch.empty((self.rows, case.source_cands), dtype=torch.int32, device=d)

        self._prepare()

    def _prepare(self):
        """Marshal every call of the step once; run() only launches."""
        c = self.case
        self._logits_calls = []
        # the rows' ends: the logits kernel derives its own from the context
        # lengths, so they are needed first by the top-k -- or already in the
        # logits stage, when it holds the top-k or the standalone candidate mask
        self._ends_call = (B.prepare_row_ends(self.context_lens, c.next_n, c.width, self.lengths,
                                              ctx_per_row=c.ctx_per_row)
                           if self.paged else None)
        self._ends_first = self.paged and (
            self.fused_topk or (self.cand is not None and not self.fused_mask))
        if self._ends_call is not None and self._ends_first:
            self._logits_calls.append(self._ends_call)
        fused = None
        if self.fused_topk:
            fused = B.prepare_paged_mqa_logits_topk(
                self.q, self.q_scale, self.weights, self.pages, self.block_table,
                self.context_lens, c.next_n, c.page_size, c.fmt, self.logits, c.width,
                self.lengths, self.k_top, self.topk,
                block_max=self.block_max if self.source else None,
                block_size=c.source_block if self.source else 0, row_ks=self.row_ks,
                ctx_per_row=c.ctx_per_row, num_ctas=self.num_ctas)
            self._logits_calls.append(fused)
            self._slots_call = B.prepare_topk_to_ragged_slots(
                self.topk, self.block_table, c.page_size, c.num_pages, self.slots, self.indptr,
                self.lens, next_n=c.next_n, max_blocks=self.max_blocks)
        elif self.source:
            self._logits_calls.append(B.prepare_paged_mqa_logits_block_max(
                self.q, self.q_scale, self.weights, self.pages, self.block_table,
                self.context_lens, c.next_n, c.page_size, c.fmt, self.logits, c.width,
                self.block_max, c.source_block, row_ks=self.row_ks, ctx_per_row=c.ctx_per_row,
                num_ctas=self.num_ctas))
            self._slots_call = B.prepare_topk_to_ragged_slots(
                self.topk, self.block_table, c.page_size, c.num_pages, self.slots, self.indptr,
                self.lens, next_n=c.next_n, max_blocks=self.max_blocks)
        elif self.paged:
            cand = self.cand if (self.cand is not None and self.fused_mask) else None
            self._logits_calls.append(B.prepare_paged_mqa_logits(
                self.q, self.q_scale, self.weights, self.pages, self.block_table,
                self.context_lens, c.next_n, c.page_size, c.fmt, self.logits, c.width,
                row_ks=self.row_ks, ctx_per_row=c.ctx_per_row, candidate_blocks=cand,
                cand_block=c.cand_block, num_ctas=self.num_ctas, workspace=self.gather,
                candidates_only=self.cand_topk and cand is not None))
            if self.cand is not None and not self.fused_mask:
                self._logits_calls.append(B.prepare_apply_candidate_mask(
                    self.logits, self.row_ks, self.lengths, self.cand, c.cand_block))
            self._slots_call = B.prepare_topk_to_ragged_slots(
                self.topk, self.block_table, c.page_size, c.num_pages, self.slots, self.indptr,
                self.lens, next_n=c.next_n, max_blocks=self.max_blocks)
        else:
            self._logits_calls.append(B.prepare_mqa_logits(
                self.q, self.q_scale, self.weights, self.k, self.k_scale, self.ks, self.ke,
                c.fmt, self.logits))
            self._slots_call = None
        if self.paged and self.cand is not None and self.cand_topk:
            self._topk_call = B.prepare_topk_candidates(
                self.logits, self.lengths, self.k_top, self.topk, self.cand, c.cand_block,
                row_ks=self.row_ks)
        elif fused is not None:
            self._topk_call = None  # inside the fused logits call
        elif self.paged and self.fused_slots:
            self._topk_call = B.prepare_topk_ragged_slots(
                self.logits, self.lengths, self.k_top, self.topk, self.block_table, c.page_size,
                c.num_pages, self.slots, self.indptr, self.lens, next_n=c.next_n,
                max_blocks=self.max_blocks)
            self._slots_call = None  # inside the top-k call
        else:
            self._topk_call = B.prepare_topk(self.logits, self.lengths, self.k_top, self.topk)
        # the candidate pool: the best blocks of each row, from the block maxima
        self._pool_call = (B.prepare_topk(self.block_max, self.block_lens, c.source_cands,
                                          self.pool) if self.source else None)

    # -------------------------------------------------------------- stages
    def logits_stage(self, stream=None):
        for call in self._logits_calls:
            call(stream)

    def topk_stage(self, stream=None):
        if self._ends_call is not None and not self._ends_first:
            self._ends_call(stream)
        if self._topk_call is not None:
            self._topk_call(stream)
        if self._pool_call is not None:
            self._pool_call(stream)

    def slots_stage(self, stream=None):
        if self._slots_call is not None:
            self._slots_call(stream)

    def run(self, stream=None):
        self.logits_stage(stream)
        self.topk_stage(stream)
        self.slots_stage(stream)

    # ---------------------------------------------------- host round trip
    def twin(self, kv_copy: bool = False):
        """A second buffer set for the same case, sharing the K cache (or,
        with kv_copy, holding its own device copy of it)."""
        return IndexerStep(self.case, device=self.device, fused_mask=self.fused_mask,
                           num_ctas=self.num_ctas, gather=self.gather,
                           cand_topk=self.cand_topk, kv_from=self, fused_topk=self.fused_topk,
                           kv_copy=kv_copy, fused_slots=self.fused_slots)

    def input_names(self):
        """The per-step inputs a caller copies in (the K cache is state; paged
        row ends are derived on the device from the context lengths)."""
        names = ["q", "weights"]
        if self.paged:
            return names + ["block_table", "context_lens"] + (
                ["row_ks"] if self.row_ks is not None else []) + (
                ["cand"] if self.cand is not None else [])
        return names + ["ks", "ke"]

    def results(self):
        """The per-step outputs a caller reads back."""
        return [self.topk] + ([self.slots, self.indptr] if self.paged else [])

    @property
    def launches_per_step(self) -> int:
        calls = self._logits_calls + ([self._topk_call] if self._topk_call is not None else [])
        if self._ends_call is not None and not self._ends_first:
            calls.append(self._ends_call)
        if self._pool_call is not None:
            calls.append(self._pool_call)
        if self._slots_call is not None:
            calls.append(self._slots_call)
        return sum(c.kernels for c in calls)


class ProducerStep:
    """Device-resident inputs and outputs of one K/Q producer step
    (synth.ProducerCase) and its two calls: the K producer writes the new
    keys into the cache pages, the Q producer quantises the query heads and
    scales their weights.  ``logits_stage``/``topk_stage`` name the K and Q
    calls so the benchmark's stage timing applies unchanged."""

    def __init__(self, case, device="cuda", consts_from=None):
        self.case = case
        self.device = torch.device(device)
        d = self.device
        c = case
        self.k_pre = torch.from_numpy(c.k_pre).to(d).to(torch.bfloat16)
        self.q = torch.from_numpy(c.q).to(d).to(torch.bfloat16)
        self.weights = _dev(c.weights, d)
        self.positions = _dev(c.positions, d)
        self.slots = _dev(c.slots, d)
        if consts_from is not None:  # model constants: the rotary table and the norm weight
            self.cos_sin, self.norm_weight = consts_from.cos_sin, consts_from.norm_weight
        else:
            self.cos_sin, self.norm_weight = _dev(c.cos_sin, d), _dev(c.norm_weight, d)
        self.pages = torch.zeros((c.num_pages, c.page_stride), dtype=torch.uint8, device=d)
        rowb = c.D if c.fmt == 0 else c.D // 2
        self.q_out = torch.empty((c.T, c.H, rowb), dtype=torch.uint8, device=d)
        self.q_sf = (torch.empty((c.T, c.H), dtype=torch.int32, device=d) if c.fmt == 1
                     else None)
        self.weights_out = torch.empty((c.T, c.H), dtype=torch.float32, device=d)
        self._k_call = B.prepare_k_norm_rope_store(
            self.k_pre, self.positions, self.cos_sin, c.rope_dim, self.norm_weight, c.eps,
            self.pages, c.page_size, self.slots, c.fmt)
        self._q_call = B.prepare_q_rope_quant(
            self.q, self.positions, self.cos_sin, c.rope_dim, self.weights, c.weight_scale,
            c.fmt, self.q_out, self.weights_out, self.q_sf)

    def logits_stage(self, stream=None):
        self._k_call(stream)

    def topk_stage(self, stream=None):
        self._q_call(stream)

    def slots_stage(self, stream=None):
        pass

    def run(self, stream=None):
        self._k_call(stream)
        self._q_call(stream)

    def twin(self, kv_copy: bool = False):
        return ProducerStep(self.case, device=self.device, consts_from=self)

    def input_names(self):
        return ["k_pre", "q", "weights", "positions", "slots"]

    def results(self):
        return [self.q_out] + ([self.q_sf] if self.q_sf is not None else []) + [self.weights_out]

    @property
    def launches_per_step(self) -> int:
        return 2
