"""GB300-native sparse-attention lightning indexer.

The compute path is the C ABI library libidx.so (include/idx.h), built from
hand-written sm_103a CUDA kernels in ``csrc/``; this package only builds it,
loads it and marshals torch tensors into its calls.
"""
from ._binding import (  # noqa: F401
    DEV_BAD_PAGE,
    DEV_TIMEOUT,
    FMT_FP8,
    FMT_MXFP4,
    IndexerError,
    idx_apply_candidate_mask,
    idx_fill_logits_tail,
    idx_get_device_status,
    idx_mqa_logits,
    idx_paged_mqa_logits,
    idx_row_ends,
    idx_topk,
    idx_topk_ragged_slots,
    idx_topk_to_ragged_slots,
    lib,
    library_path,
    version,
)
from .pipeline import IndexerStep, ProducerStep  # noqa: F401
