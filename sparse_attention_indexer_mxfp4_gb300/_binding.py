"""Thin ctypes binding of libidx.so (include/idx.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtype / shape / device, and passes raw device pointers, sizes and the current
CUDA stream to the C entry point of the same name.  All computation happens in
the library's CUDA kernels; there is no fallback path.  A missing or unloadable
library raises at import of this module's first call.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

FMT_FP8 = 0
FMT_MXFP4 = 1

IDX_OK = 0
_ERRORS = {1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED", 3: "IDX_ERR_WORKSPACE",
           4: "IDX_ERR_CUDA"}
DEV_BAD_PAGE = 1
DEV_TIMEOUT = 4
DEV_BAD_POSITION = 8
SLOT_DIRECT_ROWS = 4096  # above it the slot map runs a third (scan) kernel
TOPK_CLUSTER_MAX_LEN = 262144  # rows the one-cluster-per-row top-k holds (8 x 32768 keys)

_lib = None
_lock = threading.Lock()

_P, _I, _L, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t

_SIGNATURES = {
    "idx_mqa_logits": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _L, _P, _S, _P],
    "idx_paged_mqa_logits": [_P, _P, _P, _P, _L, _I, _P, _L, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                             _P, _L, _I, _I, _P, _L, _I, _I, _P, _S, _P],
    "idx_apply_candidate_mask": [_P, _L, _I, _I, _P, _P, _P, _L, _I, _I, _I, _P],
    "idx_topk": [_P, _L, _I, _P, _I, _P, _L, _P, _S, _P],
    "idx_paged_mqa_logits_candidates": None,  # same as idx_paged_mqa_logits
    "idx_paged_mqa_logits_block_max": [_P, _P, _P, _P, _L, _I, _P, _L, _P, _I, _P, _I, _I, _I,
                                       _I, _I, _I, _P, _L, _I, _P, _L, _I, _I, _P],
    "idx_topk_noalloc": [_P, _L, _I, _P, _I, _P, _L, _P],
    "idx_topk_candidates": [_P, _L, _I, _P, _P, _P, _L, _I, _I, _I, _I, _P, _L, _P],
    "idx_topk_to_ragged_slots": [_P, _L, _I, _I, _P, _I, _P, _L, _I, _I, _I, _P, _P, _P, _P],
    "idx_topk_ragged_slots": [_P, _L, _I, _P, _I, _P, _L, _P, _S, _P, _I, _P, _L, _I, _I, _I, _P,
                              _P, _P, _P],
    "idx_paged_mqa_logits_topk": [_P, _P, _P, _P, _L, _I, _P, _L, _P, _I, _P, _I, _I, _I, _I,
                                  _I, _I, _P, _L, _I, _P, _L, _I, _P, _I, _P, _L, _I, _P, _S,
                                  _P],
    "idx_k_norm_rope_store": [_P, _L, _P, _P, _L, _I, _I, _P, ctypes.c_float, _I, _I, _I, _P,
                              _L, _I, _I, _P, _P],
    "idx_q_rope_quant": [_P, _P, _P, _L, _I, _I, _P, ctypes.c_float, _I, _I, _I, _I, _P, _P, _P,
                         _P],
    "idx_get_device_status": [_P, ctypes.POINTER(ctypes.c_uint32)],
    "idx_debug_wait_expiry": [_I, ctypes.c_uint64, _P],
    "idx_row_ends": [_P, _I, _I, _I, _I, _P, _P],
    "idx_fill_logits_tail": [_P, _L, _I, _P, _I, _P],
}


class IndexerError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libidx.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if not os.environ.get("IDX_NO_BUILD") else _build.LIB
            if not os.path.exists(path):
                raise IndexerError(f"indexer library missing: {path}")
            L = ctypes.CDLL(path)
            for name, args in _SIGNATURES.items():
                fn = getattr(L, name)
                if args is None:
                    args = _SIGNATURES["idx_paged_mqa_logits"]
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.idx_version.restype = ctypes.c_char_p
            L.idx_topk_workspace_size.argtypes = [_I, _L, _I]
            L.idx_topk_workspace_size.restype = _S
            L.idx_paged_mqa_logits_workspace_size.argtypes = [_I, _I, _I, _I]
            L.idx_paged_mqa_logits_workspace_size.restype = _S
            _lib = L
    return _lib


def _check(rc: int, name: str):
    if rc != IDX_OK:
        raise IndexerError(f"{name} returned {_ERRORS.get(rc, rc)}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("indexer tensors must live on a CUDA device")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _u8(t):
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def version() -> str:
    return lib().idx_version().decode()


class Prepared:
    """One validated library call with its arguments already marshalled;
    calling it launches on the given (or current) stream."""

    __slots__ = ("fn", "args", "name", "keep", "kernels")

    def __init__(self, name, args, keep, kernels=1):
        self.fn = getattr(lib(), name)
        self.name = name
        self.args = tuple(args)
        self.keep = keep  # tensors that must outlive the call
        self.kernels = kernels  # kernel launches per call

    def __call__(self, stream=None):
        _check(self.fn(*self.args, _stream(stream)), self.name)


def prepare_mqa_logits(q, q_scale, weights, k, k_scale, row_ks, row_ke, fmt, logits):
    q, k = _u8(q), _u8(k)
    M, H = q.shape[0], q.shape[1]
    D = q.shape[2] if fmt == FMT_FP8 else 2 * q.shape[2]
    N = k.shape[0]
    _need(weights, torch.float32, "weights")
    _need(row_ks, torch.int32, "row_ks")
    _need(row_ke, torch.int32, "row_ke")
    if logits.dtype != torch.float32 or logits.stride(1) != 1:
        raise ValueError("logits must be float32 with unit column stride")
    args = (_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(k), _ptr(k_scale), _ptr(row_ks),
            _ptr(row_ke), M, N, H, D, fmt, _ptr(logits), logits.stride(0), None, 0)
    return Prepared("idx_mqa_logits", args, (q, q_scale, weights, k, k_scale, row_ks, row_ke,
                                             logits))


def idx_mqa_logits(q, q_scale, weights, k, k_scale, row_ks, row_ke, fmt, logits,
                   stream=None):
    """Non-paged logits.  q [M,H,D] (fp8) or [M,H,D/2] (mxfp4) bytes; k [N,D] or
    [N,D/2]; logits fp32 [M, >= N] (row stride used as ld)."""
    prepare_mqa_logits(q, q_scale, weights, k, k_scale, row_ks, row_ke, fmt, logits)(stream)


def prepare_paged_mqa_logits(q, q_scale, weights, kv_pages, block_table, context_lens, next_n,
                             page_size, fmt, logits, max_model_len, row_ks=None,
                             ctx_per_row=False, candidate_blocks=None, cand_block=0,
                             num_ctas=0, workspace=True, candidates_only=False):
    """workspace (used with candidate_blocks): True allocates the gather plan
    scratch here (held by the returned call), a uint8 CUDA tensor supplies it,
    False or None scores every key of the context.  candidates_only calls
    idx_paged_mqa_logits_candidates: only tiles holding a candidate key are
    written (for idx_topk_candidates)."""
    q = _u8(q)
    rows, H = q.shape[0], q.shape[1]
    D = q.shape[2] if fmt == FMT_FP8 else 2 * q.shape[2]
    B = rows // next_n
    _need(weights, torch.float32, "weights")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    if kv_pages.dtype != torch.uint8 or kv_pages.dim() != 2 or kv_pages.stride(1) != 1:
        raise ValueError("kv_pages must be uint8 [num_pages, page_stride] with unit byte stride")
    cand_stride, num_cand = 0, 0
    if candidate_blocks is not None:
        _need(candidate_blocks, torch.int32, "candidate_blocks")
        cand_stride, num_cand = candidate_blocks.stride(0), candidate_blocks.shape[1]
    ws = None
    need = paged_workspace_size(B, next_n, max_model_len, num_cand)
    if need and workspace is True:
        ws = torch.empty(need, dtype=torch.uint8, device=logits.device)
    elif need and workspace is not None and workspace is not False:
        ws = workspace
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    args = (_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(kv_pages), kv_pages.stride(0),
            kv_pages.shape[0], _ptr(block_table), block_table.stride(0), _ptr(context_lens),
            int(ctx_per_row), _ptr(row_ks), B, next_n, H, D, page_size, fmt,
            _ptr(candidate_blocks), cand_stride, num_cand, cand_block, _ptr(logits),
            logits.stride(0), max_model_len, num_ctas, _ptr(ws), nbytes)
    # with a plan the library launches the plan kernel before the logits kernel
    planned = ws is not None and need > 0 and nbytes >= need
    name = "idx_paged_mqa_logits_candidates" if candidates_only else "idx_paged_mqa_logits"
    return Prepared(name, args, (q, q_scale, weights, kv_pages, block_table,
                                                   context_lens, row_ks, candidate_blocks,
                                                   logits, ws), 2 if planned else 1)


def prepare_paged_mqa_logits_block_max(q, q_scale, weights, kv_pages, block_table,
                                       context_lens, next_n, page_size, fmt, logits,
                                       max_model_len, block_max, block_size, row_ks=None,
                                       ctx_per_row=False, num_ctas=0):
    """The candidate source: dense paged logits plus block maxima
    block_max fp32 [B*next_n, >= ceil(max_model_len / block_size)]."""
    q = _u8(q)
    rows, H = q.shape[0], q.shape[1]
    D = q.shape[2] if fmt == FMT_FP8 else 2 * q.shape[2]
    B = rows // next_n
    _need(weights, torch.float32, "weights")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    if block_max.dtype != torch.float32 or block_max.stride(1) != 1:
        raise ValueError("block_max must be float32 with unit column stride")
    if kv_pages.dtype != torch.uint8 or kv_pages.dim() != 2 or kv_pages.stride(1) != 1:
        raise ValueError("kv_pages must be uint8 [num_pages, page_stride] with unit byte stride")
    args = (_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(kv_pages), kv_pages.stride(0),
            kv_pages.shape[0], _ptr(block_table), block_table.stride(0), _ptr(context_lens),
            int(ctx_per_row), _ptr(row_ks), B, next_n, H, D, page_size, fmt, _ptr(logits),
            logits.stride(0), max_model_len, _ptr(block_max), block_max.stride(0), block_size,
            num_ctas)
    # the -inf fill of the block maxima, then the logits kernel
    return Prepared("idx_paged_mqa_logits_block_max", args,
                    (q, q_scale, weights, kv_pages, block_table, context_lens, row_ks, logits,
                     block_max), 2)


def idx_paged_mqa_logits_block_max(q, q_scale, weights, kv_pages, block_table, context_lens,
                                   next_n, page_size, fmt, logits, max_model_len, block_max,
                                   block_size, row_ks=None, ctx_per_row=False, num_ctas=0,
                                   stream=None):
    prepare_paged_mqa_logits_block_max(q, q_scale, weights, kv_pages, block_table,
                                       context_lens, next_n, page_size, fmt, logits,
                                       max_model_len, block_max, block_size, row_ks,
                                       ctx_per_row, num_ctas)(stream)


def prepare_paged_mqa_logits_topk(q, q_scale, weights, kv_pages, block_table, context_lens,
                                  next_n, page_size, fmt, logits, max_model_len, lengths, k, out,
                                  block_max=None, block_size=0, row_ks=None, ctx_per_row=False,
                                  num_ctas=0, workspace=True):
    """Paged logits (+ block maxima) and their top-k in one call; with the
    top-k scratch (workspace=True allocates it) the logits kernel counts the
    top-k's first digit and the top-k skips a pass.  lengths: each row's ke."""
    q = _u8(q)
    rows, H = q.shape[0], q.shape[1]
    D = q.shape[2] if fmt == FMT_FP8 else 2 * q.shape[2]
    B = rows // next_n
    _need(weights, torch.float32, "weights")
    _need(block_table, torch.int32, "block_table")
    _need(context_lens, torch.int32, "context_lens")
    _need(lengths, torch.int32, "lengths")
    if out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError("out must be int32 with unit column stride")
    if block_max is not None:
        _need(block_max, torch.float32, "block_max")
    if kv_pages.dtype != torch.uint8 or kv_pages.dim() != 2 or kv_pages.stride(1) != 1:
        raise ValueError("kv_pages must be uint8 [num_pages, page_stride] with unit byte stride")
    ld = logits.stride(0)
    ws = None
    if workspace is True:
        nbytes = topk_workspace_size(rows, ld, k)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=logits.device)
    elif workspace is not None and workspace is not False:
        ws = workspace
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    args = (_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(kv_pages), kv_pages.stride(0),
            kv_pages.shape[0], _ptr(block_table), block_table.stride(0), _ptr(context_lens),
            int(ctx_per_row), _ptr(row_ks), B, next_n, H, D, page_size, fmt, _ptr(logits), ld,
            max_model_len, _ptr(block_max), 0 if block_max is None else block_max.stride(0),
            block_size, _ptr(lengths), k, _ptr(out), out.stride(0), num_ctas, _ptr(ws), nbytes)
    need = topk_workspace_size(rows, ld, k)
    chunked = ws is not None and need > 0 and nbytes >= need and ld > 8192
    # launches: top-k plan, (block-maxima fill), logits, top-k phases
    kernels = (1 if block_max is not None else 0) + (3 if chunked else 2)
    return Prepared("idx_paged_mqa_logits_topk", args,
                    (q, q_scale, weights, kv_pages, block_table, context_lens, row_ks, logits,
                     block_max, lengths, out, ws), kernels)


def paged_workspace_size(B, next_n, max_model_len, num_cand) -> int:
    """Bytes of the gather-plan scratch of idx_paged_mqa_logits (0: not used)."""
    return int(lib().idx_paged_mqa_logits_workspace_size(B, next_n, max_model_len, num_cand))


def idx_paged_mqa_logits(q, q_scale, weights, kv_pages, block_table, context_lens, next_n,
                         page_size, fmt, logits, max_model_len, row_ks=None, ctx_per_row=False,
                         candidate_blocks=None, cand_block=0, num_ctas=0, stream=None,
                         workspace=True):
    """Paged logits.  q [B*next_n,H,D|D/2] bytes; kv_pages uint8 [num_pages, page_stride];
    block_table int32 [B, >= ceil(max_model_len/page_size)]; logits fp32
    [B*next_n, >= max_model_len]."""
    prepare_paged_mqa_logits(q, q_scale, weights, kv_pages, block_table, context_lens, next_n,
                             page_size, fmt, logits, max_model_len, row_ks, ctx_per_row,
                             candidate_blocks, cand_block, num_ctas, workspace)(stream)


def prepare_apply_candidate_mask(logits, row_ks, row_ke, candidate_blocks, block_size,
                                 row_repeat=1, width=None):
    rows = logits.shape[0]
    width = logits.shape[1] if width is None else width
    _need(row_ke, torch.int32, "row_ke")
    _need(candidate_blocks, torch.int32, "candidate_blocks")
    args = (_ptr(logits), logits.stride(0), rows, width, _ptr(row_ks), _ptr(row_ke),
            _ptr(candidate_blocks), candidate_blocks.stride(0), candidate_blocks.shape[1],
            block_size, row_repeat)
    return Prepared("idx_apply_candidate_mask", args, (logits, row_ks, row_ke, candidate_blocks))


def idx_apply_candidate_mask(logits, row_ks, row_ke, candidate_blocks, block_size,
                             row_repeat=1, width=None, stream=None):
    prepare_apply_candidate_mask(logits, row_ks, row_ke, candidate_blocks, block_size,
                                 row_repeat, width)(stream)


def topk_workspace_size(rows, ld, k) -> int:
    """Bytes of device scratch idx_topk's chunked path needs (0: not used)."""
    return int(lib().idx_topk_workspace_size(rows, ld, k))


def _sm_count(device) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


def prepare_topk(logits, lengths, k, out, workspace=True):
    """workspace: True allocates the scratch for the chunked path once here
    (held by the returned call), a uint8 CUDA tensor supplies it, False or
    None passes none (calls that would take the chunked path then stream
    each row in one CTA; the register and cluster paths need no scratch)."""
    if logits.dtype != torch.float32 or logits.stride(1) != 1:
        raise ValueError("logits must be float32 with unit column stride")
    _need(lengths, torch.int32, "lengths")
    if out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError("out must be int32 with unit column stride")
    rows, ld = logits.shape[0], logits.stride(0)
    ws = None
    if workspace is True:
        nbytes = topk_workspace_size(rows, ld, k)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=logits.device)
    elif workspace is not None and workspace is not False:
        ws = workspace
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    args = (_ptr(logits), ld, rows, _ptr(lengths), k, _ptr(out), out.stride(0), _ptr(ws), nbytes)
    # one kernel for rows of up to 8192 keys (a CTA per row) and for rows of
    # up to TOPK_CLUSTER_MAX_LEN keys whose clusters fit the GPU in one wave;
    # otherwise, with scratch, the chunked path (two kernels)
    need = topk_workspace_size(rows, ld, k)
    clusters = -(-ld // 32768) if ld <= TOPK_CLUSTER_MAX_LEN else 0
    one_wave = ld <= 8192 or (clusters and rows * clusters <= _sm_count(logits.device))
    chunked = ws is not None and need > 0 and nbytes >= need and not one_wave
    return Prepared("idx_topk", args, (logits, lengths, out, ws), 2 if chunked else 1)


def idx_topk(logits, lengths, k, out, stream=None, workspace=True):
    """out int32 [rows, >= k]: ascending indices of the k largest finite logits
    of each row within [0, lengths[r]), -1 padded."""
    prepare_topk(logits, lengths, k, out, workspace)(stream)


def idx_topk_noalloc(logits, lengths, k, out, stream=None):
    """idx_topk over the library's fixed per-device scratch array: no
    allocation, no workspace argument; calls on one device must not overlap."""
    if logits.dtype != torch.float32 or logits.stride(1) != 1:
        raise ValueError("logits must be float32 with unit column stride")
    _need(lengths, torch.int32, "lengths")
    if out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError("out must be int32 with unit column stride")
    rc = lib().idx_topk_noalloc(_ptr(logits), logits.stride(0), logits.shape[0], _ptr(lengths),
                                k, _ptr(out), out.stride(0), _stream(stream))
    _check(rc, "idx_topk_noalloc")


def prepare_topk_candidates(logits, lengths, k, out, candidate_blocks, block_size, row_ks=None,
                            row_repeat=1):
    """out int32 [rows, >= k]: ascending indices of the k largest finite logits
    of each row among the keys of its candidate blocks within [ks, lengths)."""
    if logits.dtype != torch.float32 or logits.stride(1) != 1:
        raise ValueError("logits must be float32 with unit column stride")
    _need(lengths, torch.int32, "lengths")
    _need(candidate_blocks, torch.int32, "candidate_blocks")
    if out.dtype != torch.int32 or out.stride(1) != 1:
        raise ValueError("out must be int32 with unit column stride")
    args = (_ptr(logits), logits.stride(0), logits.shape[0], _ptr(lengths), _ptr(row_ks),
            _ptr(candidate_blocks), candidate_blocks.stride(0), candidate_blocks.shape[1],
            block_size, row_repeat, k, _ptr(out), out.stride(0))
    return Prepared("idx_topk_candidates", args,
                    (logits, lengths, out, candidate_blocks, row_ks))


def idx_topk_candidates(logits, lengths, k, out, candidate_blocks, block_size, row_ks=None,
                        row_repeat=1, stream=None):
    prepare_topk_candidates(logits, lengths, k, out, candidate_blocks, block_size, row_ks,
                            row_repeat)(stream)


def prepare_topk_to_ragged_slots(topk, block_table, page_size, num_pages, slots, indptr, lens,
                                 next_n=1, row_to_seq=None, max_blocks=None):
    if topk.dtype != torch.int32 or topk.stride(1) != 1:
        raise ValueError("topk must be int32 with unit column stride")
    _need(block_table, torch.int32, "block_table")
    rows, k = topk.shape
    mb = block_table.shape[1] if max_blocks is None else max_blocks
    args = (_ptr(topk), topk.stride(0), rows, k, _ptr(row_to_seq), next_n, _ptr(block_table),
            block_table.stride(0), mb, page_size, num_pages, _ptr(slots), _ptr(indptr),
            _ptr(lens))
    return Prepared("idx_topk_to_ragged_slots", args,
                    (topk, block_table, slots, indptr, lens, row_to_seq),
                    _slot_kernels(rows, k, mb))


def _slot_kernels(rows, k, max_blocks):
    """Kernels of one slot-map call: one 16-CTA cluster when each CTA holds
    at most four (row, 1024-entry step) pairs and 32768 block-table words,
    else a count and a write kernel (and a scan above SLOT_DIRECT_ROWS rows)."""
    r = -(-rows // 16)
    if k >= 1 and r * -(-k // 1024) <= 4 and r * max_blocks <= 32768:
        return 1
    return 2 + (rows > SLOT_DIRECT_ROWS)


def idx_topk_to_ragged_slots(topk, block_table, page_size, num_pages, slots, indptr, lens,
                             next_n=1, row_to_seq=None, max_blocks=None, stream=None):
    prepare_topk_to_ragged_slots(topk, block_table, page_size, num_pages, slots, indptr, lens,
                                 next_n, row_to_seq, max_blocks)(stream)


def prepare_topk_ragged_slots(logits, lengths, k, out, block_table, page_size, num_pages, slots,
                              indptr, lens, next_n=1, row_to_seq=None, max_blocks=None,
                              workspace=True):
    """idx_topk into out, then idx_topk_to_ragged_slots of out, as one call
    (the cluster top-k counts each row's valid slots as it writes the row
    where the one-launch slot map does not take the call)."""
    top = prepare_topk(logits, lengths, k, out, workspace)
    _need(block_table, torch.int32, "block_table")
    rows, ld = logits.shape[0], logits.stride(0)
    mb = block_table.shape[1] if max_blocks is None else max_blocks
    ws = top.keep[3]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    args = (_ptr(logits), ld, rows, _ptr(lengths), k, _ptr(out), out.stride(0), _ptr(ws), nbytes,
            _ptr(row_to_seq), next_n, _ptr(block_table), block_table.stride(0), mb, page_size,
            num_pages, _ptr(slots), _ptr(indptr), _ptr(lens))
    clusters = -(-ld // 32768)
    fused = (rows > 0 and k > 0 and 8192 < ld <= TOPK_CLUSTER_MAX_LEN
             and rows * clusters <= _sm_count(logits.device) and _slot_kernels(rows, k, mb) != 1)
    kernels = 2 + (rows > SLOT_DIRECT_ROWS) if fused else (
        top.kernels + _slot_kernels(rows, k, mb))
    return Prepared("idx_topk_ragged_slots", args,
                    (logits, lengths, out, ws, block_table, slots, indptr, lens, row_to_seq),
                    kernels)


def idx_topk_ragged_slots(logits, lengths, k, out, block_table, page_size, num_pages, slots,
                          indptr, lens, next_n=1, row_to_seq=None, max_blocks=None, stream=None,
                          workspace=True):
    prepare_topk_ragged_slots(logits, lengths, k, out, block_table, page_size, num_pages, slots,
                              indptr, lens, next_n, row_to_seq, max_blocks, workspace)(stream)


def _bf16_bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype in (torch.int16, torch.uint16):
        return t
    raise ValueError("expected bfloat16 (or its 16-bit pattern)")


def prepare_k_norm_rope_store(k_pre, positions, cos_sin, rope_dim, norm_weight, eps, kv_pages,
                              page_size, slot_mapping, fmt):
    """K producer into kv_pages (uint8 [num_pages, page_stride]).  k_pre
    bf16 [T, >= D]; positions int32 [T]; cos_sin fp32 [P, >= rope_dim];
    norm_weight fp32 [D]; slot_mapping int64 [T] (-1 skips)."""
    k = _bf16_bits(k_pre)
    T = k.shape[0]
    _need(positions, torch.int32, "positions")
    _need(norm_weight, torch.float32, "norm_weight")
    _need(slot_mapping, torch.int64, "slot_mapping")
    if cos_sin is not None:
        _need(cos_sin, torch.float32, "cos_sin")
    if kv_pages.dtype != torch.uint8 or kv_pages.dim() != 2 or kv_pages.stride(1) != 1:
        raise ValueError("kv_pages must be uint8 [num_pages, page_stride] with unit byte stride")
    # no table (rope_dim 0): positions are not bounded by one
    ncs, ldcs = (2 ** 31 - 1, rope_dim) if cos_sin is None else (cos_sin.shape[0],
                                                                cos_sin.stride(0))
    args = (_ptr(k), k.stride(0), _ptr(positions), _ptr(cos_sin), ldcs, ncs, rope_dim,
            _ptr(norm_weight), float(eps), T, norm_weight.shape[0], fmt, _ptr(kv_pages),
            kv_pages.stride(0), kv_pages.shape[0], page_size, _ptr(slot_mapping))
    return Prepared("idx_k_norm_rope_store", args,
                    (k, positions, cos_sin, norm_weight, kv_pages, slot_mapping))


def idx_k_norm_rope_store(k_pre, positions, cos_sin, rope_dim, norm_weight, eps, kv_pages,
                          page_size, slot_mapping, fmt, stream=None):
    prepare_k_norm_rope_store(k_pre, positions, cos_sin, rope_dim, norm_weight, eps, kv_pages,
                              page_size, slot_mapping, fmt)(stream)


def prepare_q_rope_quant(q, positions, cos_sin, rope_dim, weights, weight_scale, fmt, q_out,
                         weights_out, q_scale_out=None):
    """Q producer.  q bf16 [T, H, D]; weights fp32 [T, H]; q_out uint8
    [T, H, D] (FP8) or [T, H, D/2] (MXFP4); q_scale_out int32 [T, H] (MXFP4);
    weights_out fp32 [T, H]."""
    qb = _bf16_bits(q)
    if not qb.is_contiguous():
        raise ValueError("q must be contiguous [T, H, D]")
    T, H, D = qb.shape
    _need(positions, torch.int32, "positions")
    _need(weights, torch.float32, "weights")
    _need(weights_out, torch.float32, "weights_out")
    if cos_sin is not None:
        _need(cos_sin, torch.float32, "cos_sin")
    ncs, ldcs = (2 ** 31 - 1, rope_dim) if cos_sin is None else (cos_sin.shape[0],
                                                                cos_sin.stride(0))
    args = (_ptr(qb), _ptr(positions), _ptr(cos_sin), ldcs, ncs, rope_dim, _ptr(weights),
            float(weight_scale), T, H, D, fmt, _ptr(q_out), _ptr(q_scale_out), _ptr(weights_out))
    return Prepared("idx_q_rope_quant", args,
                    (qb, positions, cos_sin, weights, q_out, q_scale_out, weights_out))


def idx_q_rope_quant(q, positions, cos_sin, rope_dim, weights, weight_scale, fmt, q_out,
                     weights_out, q_scale_out=None, stream=None):
    prepare_q_rope_quant(q, positions, cos_sin, rope_dim, weights, weight_scale, fmt, q_out,
                         weights_out, q_scale_out)(stream)


def prepare_row_ends(context_lens, next_n, max_model_len, row_ends, ctx_per_row=False):
    """row_ends int32 [B * next_n]: each paged row's end ke from the context
    lengths (the rule of the paged logits), computed on the device."""
    _need(context_lens, torch.int32, "context_lens")
    _need(row_ends, torch.int32, "row_ends")
    rows = row_ends.numel()
    if rows % next_n:
        raise ValueError("row_ends must hold B * next_n entries")
    B_ = rows // next_n
    want = rows if ctx_per_row else B_
    if context_lens.numel() != want:
        raise ValueError(f"context_lens must hold {want} entries")
    return Prepared("idx_row_ends", [_ptr(context_lens), 1 if ctx_per_row else 0, B_, next_n,
                                     max_model_len, _ptr(row_ends)],
                    (context_lens, row_ends))


def idx_row_ends(context_lens, next_n, max_model_len, row_ends, ctx_per_row=False, stream=None):
    prepare_row_ends(context_lens, next_n, max_model_len, row_ends, ctx_per_row)(stream)


def idx_fill_logits_tail(logits, row_ends, width=None, stream=None):
    """-inf over [row_ends[r], width) of every row of logits (fp32 [rows, ld])."""
    if logits.dtype != torch.float32 or logits.stride(1) != 1:
        raise ValueError("logits must be float32 with unit column stride")
    _need(row_ends, torch.int32, "row_ends")
    width = logits.shape[1] if width is None else width
    _check(lib().idx_fill_logits_tail(_ptr(logits), logits.stride(0), logits.shape[0],
                                      _ptr(row_ends), width, _stream(stream)),
           "idx_fill_logits_tail")


def idx_debug_wait_expiry(which: int, limit_ns: int, stream=None):
    """Diagnostic: one of the library's bounded device waits (0: the logits
    pipeline's mbarrier wait, 1: the chunked top-k's grid barrier) on a
    condition that never holds; it gives up after limit_ns and sets
    DEV_TIMEOUT in the device status."""
    _check(lib().idx_debug_wait_expiry(int(which), int(limit_ns), _stream(stream)),
           "idx_debug_wait_expiry")


def idx_get_device_status(stream=None) -> int:
    v = ctypes.c_uint32(0)
    rc = lib().idx_get_device_status(_stream(stream), ctypes.byref(v))
    _check(rc, "idx_get_device_status")
    return int(v.value)
