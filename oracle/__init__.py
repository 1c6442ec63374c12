"""CPU oracle for the lightning indexer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or calls it.

The arithmetic lives in ``idx_oracle.c`` (scalar C, fp64); this module only
compiles it with gcc and passes numpy arrays to it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "idx_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libidx_oracle.so")
_lib = None
_lock = threading.Lock()

FMT_FP8 = 0
FMT_MXFP4 = 1


def build(force: bool = False) -> str:
    """Compile the oracle to a shared object (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64


def _declare(L):
    L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_to_double.restype = ctypes.c_double
    L.orc_e2m1_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e2m1_to_double.restype = ctypes.c_double
    L.orc_e8m0_to_double.argtypes = [ctypes.c_uint8]
    L.orc_e8m0_to_double.restype = ctypes.c_double
    L.orc_default_threads.restype = _I
    L.orc_row_end.argtypes = [_P, _I, _I, _I]
    L.orc_row_end.restype = _I
    L.orc_mqa_logits.argtypes = [_I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _L, _I]
    L.orc_mqa_logits.restype = _I
    L.orc_paged_mqa_logits.argtypes = [_I, _P, _P, _P, _P, _L, _I, _P, _L, _I, _P, _I, _P,
                                       _I, _I, _I, _I, _I, _P, _L, _I, _I]
    L.orc_paged_mqa_logits.restype = _I
    L.orc_apply_candidate_mask.argtypes = [_P, _L, _I, _I, _P, _P, _P, _L, _I, _I, _I, _I]
    L.orc_apply_candidate_mask.restype = _I
    L.orc_block_max.argtypes = [_P, _L, _I, _I, _P, _P, _I, _P, _L, _I, _I]
    L.orc_block_max.restype = _I
    _D = ctypes.c_double
    L.orc_e4m3_encode.argtypes = [_D]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e2m1_encode.argtypes = [_D]
    L.orc_e2m1_encode.restype = ctypes.c_uint8
    L.orc_scale_bits.argtypes = [_D, _D]
    L.orc_scale_bits.restype = _I
    L.orc_k_norm_rope_store.argtypes = [_P, _L, _P, _P, _L, _I, _I, _P, _D, _P, _L, _I, _I, _P,
                                        _I, _I, _I, _P, _P]
    L.orc_k_norm_rope_store.restype = _I
    L.orc_q_rope_quant.argtypes = [_P, _P, _P, _L, _I, _I, _P, _D, _I, _I, _I, _I, _P, _P, _P,
                                   _P, _P]
    L.orc_q_rope_quant.restype = _I
    L.orc_topk.argtypes = [_P, _L, _I, _I, _P, _I, _P, _L, _I]
    L.orc_topk.restype = _I
    L.orc_topk_to_ragged_slots.argtypes = [_P, _L, _I, _I, _P, _I, _P, _L, _I, _I, _I,
                                           _P, _P, _P]
    L.orc_topk_to_ragged_slots.restype = _I


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return lib().orc_default_threads()


def e4m3_to_double(code: int) -> float:
    return lib().orc_e4m3_to_double(code)


def e2m1_to_double(code: int) -> float:
    return lib().orc_e2m1_to_double(code)


def e8m0_to_double(code: int) -> float:
    return lib().orc_e8m0_to_double(code)


def mqa_logits(fmt, q, q_scale, weights, k, k_scale, ks, ke, M, N, H, D,
               ld=None, nthreads=0) -> np.ndarray:
    """Non-paged logits [M, ld] (columns [0, N) defined)."""
    ld = N if ld is None else ld
    out = np.full((M, max(ld, 1)), np.nan, dtype=np.float32)
    q, k = _c(q, np.uint8), _c(k, np.uint8)
    if fmt == FMT_FP8:
        q_scale, k_scale = _c(q_scale, np.float32), _c(k_scale, np.float32)
    else:
        q_scale, k_scale = _c(q_scale, np.uint8), _c(k_scale, np.uint8)
    w, ks, ke = _c(weights, np.float32), _c(ks, np.int32), _c(ke, np.int32)
    rc = lib().orc_mqa_logits(fmt, _ptr(q), _ptr(q_scale), _ptr(w), _ptr(k), _ptr(k_scale),
                              _ptr(ks), _ptr(ke), M, N, H, D, _ptr(out), ld, nthreads)
    if rc != 0:
        raise ValueError("oracle mqa_logits rejected its arguments")
    return out[:, :ld]


def paged_mqa_logits(fmt, q, q_scale, weights, pages, page_stride, num_pages, block_table,
                     context_lens, ctx_per_row, row_ks, B, next_n, H, D, page_size, width,
                     out=None, nthreads=0):
    """Paged logits [B*next_n, width]; columns [ke_r, width) keep ``out``'s
    contents (NaN when ``out`` is None).  Returns (logits, bad_key_count)."""
    rows = B * next_n
    if out is None:
        out = np.full((rows, width), np.nan, dtype=np.float32)
    q = _c(q, np.uint8)
    q_scale = _c(q_scale, np.float32 if fmt == FMT_FP8 else np.uint8)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    rks = _c(row_ks, np.int32)
    w = _c(weights, np.float32)
    pages = _c(pages, np.uint8)
    bad = lib().orc_paged_mqa_logits(fmt, _ptr(q), _ptr(q_scale), _ptr(w), _ptr(pages),
                                     page_stride, num_pages, _ptr(bt), bt.shape[1],
                                     bt.shape[1], _ptr(ctx), int(ctx_per_row), _ptr(rks),
                                     B, next_n, H, D, page_size, _ptr(out), out.shape[1],
                                     width, nthreads)
    if bad < 0:
        raise ValueError("oracle paged_mqa_logits rejected its arguments")
    return out, bad


def row_end(context_lens, ctx_per_row, next_n, r) -> int:
    ctx = _c(context_lens, np.int32)
    return lib().orc_row_end(_ptr(ctx), int(ctx_per_row), next_n, r)


def apply_candidate_mask(logits, row_ks, row_ke, cand, block_size, row_repeat=1,
                         nthreads=0):
    """In place on a C-contiguous float32 [rows, width] array."""
    assert logits.dtype == np.float32 and logits.flags["C_CONTIGUOUS"]
    rows, width = logits.shape
    rks, rke, cand = _c(row_ks, np.int32), _c(row_ke, np.int32), _c(cand, np.int32)
    rc = lib().orc_apply_candidate_mask(_ptr(logits), width, rows, width, _ptr(rks),
                                        _ptr(rke), _ptr(cand), cand.shape[1], cand.shape[1],
                                        block_size, row_repeat, nthreads)
    if rc != 0:
        raise ValueError("oracle apply_candidate_mask rejected its arguments")
    return logits


def block_max(logits, row_ks, row_ke, block_size, nthreads=0) -> np.ndarray:
    """Block maxima [rows, cdiv(width, block_size)] float32 of the candidate
    source: block j of row r is [ks + j*bs, ks + (j+1)*bs) clipped to
    [ks, ke); -inf when empty."""
    lg = _c(logits, np.float32)
    rows, width = lg.shape
    nb = -(-width // block_size)
    out = np.empty((rows, max(nb, 1)), dtype=np.float32)
    rks, rke = _c(row_ks, np.int32), _c(row_ke, np.int32)
    rc = lib().orc_block_max(_ptr(lg), width, rows, width, _ptr(rks), _ptr(rke), block_size,
                             _ptr(out), out.shape[1], nb, nthreads)
    if rc != 0:
        raise ValueError("oracle block_max rejected its arguments")
    return out[:, :nb]


def e4m3_encode(y: float) -> int:
    """Nearest e4m3 code (ties to the even code) of |y| <= 448."""
    return int(lib().orc_e4m3_encode(float(y)))


def e2m1_encode(y: float) -> int:
    """Nearest e2m1 code (ties to the even code) of |y| <= 6."""
    return int(lib().orc_e2m1_encode(float(y)))


def scale_bits(amax: float, top: float) -> int:
    """Biased E8M0 exponent putting amax at the top of the element range."""
    return int(lib().orc_scale_bits(float(amax), float(top)))


def k_norm_rope_store(fmt, k_pre_bits, positions, cos_sin, rope_dim, norm_w, eps, pages,
                      page_size, slots):
    """K producer into ``pages`` (uint8 [num_pages, stride], in place).
    k_pre_bits: uint16 bf16 bits [T, D].  Returns (bad, pre [T, D] float64,
    bits [T, D/32] int32)."""
    k = _c(k_pre_bits, np.uint16)
    T, D = k.shape
    pos, cs = _c(positions, np.int32), _c(cos_sin, np.float32)
    w, sl = _c(norm_w, np.float32), _c(slots, np.int64)
    assert pages.dtype == np.uint8 and pages.flags["C_CONTIGUOUS"]
    pre = np.zeros((T, D), np.float64)
    bits = np.zeros((T, max(D // 32, 1)), np.int32)
    ldcs, ncs = (0, 2 ** 31 - 1) if cs is None else (cs.shape[1], cs.shape[0])
    bad = lib().orc_k_norm_rope_store(_ptr(k), D, _ptr(pos), _ptr(cs), ldcs, ncs,
                                      rope_dim, _ptr(w), float(eps), _ptr(pages), pages.shape[1],
                                      pages.shape[0], page_size, _ptr(sl), T, D, fmt, _ptr(pre),
                                      _ptr(bits))
    return bad, pre, bits


def q_rope_quant(fmt, q_bits, positions, cos_sin, rope_dim, w_in, w_scale):
    """Q producer.  q_bits: uint16 bf16 bits [T, H, D].  Returns (bad, q_out
    uint8 [T, H, D or D/2], q_sf uint8 [T, H, D/32] (MXFP4), w_out float32
    [T, H], pre [T*H, D] float64, bits [T*H, D/32] int32)."""
    q = _c(q_bits, np.uint16)
    T, H, D = q.shape
    pos, cs, w = _c(positions, np.int32), _c(cos_sin, np.float32), _c(w_in, np.float32)
    rowb = D if fmt == 0 else D // 2
    q_out = np.zeros((T, H, rowb), np.uint8)
    q_sf = np.zeros((T, H, max(D // 32, 1)), np.uint8)
    w_out = np.zeros((T, H), np.float32)
    pre = np.zeros((T * H, D), np.float64)
    bits = np.zeros((T * H, max(D // 32, 1)), np.int32)
    ldcs, ncs = (0, 2 ** 31 - 1) if cs is None else (cs.shape[1], cs.shape[0])
    bad = lib().orc_q_rope_quant(_ptr(q), _ptr(pos), _ptr(cs), ldcs, ncs,
                                 rope_dim, _ptr(w), float(w_scale), T, H, D, fmt, _ptr(q_out),
                                 _ptr(q_sf), _ptr(w_out), _ptr(pre), _ptr(bits))
    return bad, q_out, q_sf, w_out, pre, bits


def topk(logits, lengths, k, nthreads=0) -> np.ndarray:
    """[rows, k] int32, largest first (ties: lower index first), -1 padded."""
    logits = _c(logits, np.float32)
    rows, width = logits.shape
    lengths = _c(lengths, np.int32)
    out = np.empty((rows, k), dtype=np.int32)
    rc = lib().orc_topk(_ptr(logits), width, rows, width, _ptr(lengths), k, _ptr(out), k,
                        nthreads)
    if rc != 0:
        raise ValueError("oracle topk rejected its arguments")
    return out


def topk_to_ragged_slots(topk_idx, block_table, page_size, num_pages, next_n=1,
                         row_to_seq=None):
    """Returns (slots [nnz], indptr [rows+1], lens [rows], invalid_count)."""
    t = _c(topk_idx, np.int32)
    rows, k = t.shape
    bt = _c(block_table, np.int32)
    r2s = _c(row_to_seq, np.int32)
    slots = np.empty(max(rows * k, 1), dtype=np.int32)
    indptr = np.empty(rows + 1, dtype=np.int32)
    lens = np.empty(max(rows, 1), dtype=np.int32)
    bad = lib().orc_topk_to_ragged_slots(_ptr(t), k, rows, k, _ptr(r2s), next_n, _ptr(bt),
                                         bt.shape[1], bt.shape[1], page_size, num_pages,
                                         _ptr(slots), _ptr(indptr), _ptr(lens))
    return slots[:indptr[rows]], indptr, lens[:rows], bad
