"""idx_topk_noalloc, the top-k entry point for callers that cannot allocate
device scratch (an engine that hands almost all free memory to its KV cache
at start-up, a loop where cudaMalloc / cudaFree could synchronise the device):
it runs from the library's fixed per-device array instead of caller memory.

Its indices must equal the oracle's top-k of the same logits exactly, on
several calls in a row that take different paths and grids through the one
shared array: a long-row batch on the chunked path, then a heavy-tie batch
on the chunked path with another grid (nothing the first call left in the
array may leak into the second), rows wider than the cluster path, and a
call with more rows than the array holds (the scratch-free per-row kernel).
Kept in its own file, collected after the others, so it runs both alone in a
fresh process and after every other GPU test in one process."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_topk_exact
from sparse_attention_indexer_mxfp4_gb300 import _binding as B

INVALID = 1
FAKE = 0x10000  # never dereferenced: these calls fail their host checks first
ARRAY_BYTES = 32 << 20


def test_noalloc_host_checks():
    f = B.lib().idx_topk_noalloc
    ld, k = B.TOPK_CLUSTER_MAX_LEN + 4, 2048
    assert f(FAKE, ld, 4, FAKE, k, FAKE, k - 1, None) == INVALID  # ld_out < k
    assert f(FAKE, ld, -1, FAKE, k, FAKE, k, None) == INVALID
    assert f(FAKE, ld, 0, FAKE, k, FAKE, k, None) == 0   # nothing to do
    assert f(FAKE, ld, 4, FAKE, 0, FAKE, k, None) == 0   # k = 0 writes nothing


def _case(rng, rows, width, tie_levels=None, long_frac=1.0):
    if tie_levels:
        x = rng.integers(0, tie_levels, size=(rows, width)).astype(np.float32)
    else:
        x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < 0.3] = -np.inf
    lengths = rng.integers(0, width + 1, size=rows).astype(np.int32)
    short = rng.random(rows) >= long_frac
    lengths[short] = rng.integers(0, 3000, size=int(short.sum()))
    lengths[0] = width
    return x, lengths


@pytest.mark.gpu
def test_noalloc_equals_oracle_over_calls_in_a_row():
    rng = np.random.default_rng(2024)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k = 2048
    # rows beyond what the fixed array holds at this width: the fallback
    wide = B.TOPK_CLUSTER_MAX_LEN + 4
    over = next(r for r in range(1, 4096) if B.topk_workspace_size(r, wide, k) > ARRAY_BYTES)
    tie_rows = sms // 4 + 8  # 4 cluster CTAs per row would not fit one wave: chunked
    cases = [
        (_case(rng, 96, 131072), k),                        # chunked, 96 x 16 chunks
        (_case(rng, tie_rows, 100000, tie_levels=3), 300),  # chunked, ties, another grid
        (_case(rng, 5, 300000), k),                         # wider than a cluster holds
        (_case(rng, over, wide, long_frac=0.05), k),        # more rows than the array holds
    ]
    assert tie_rows * 4 > sms
    assert B.topk_workspace_size(96, 131072, k) <= ARRAY_BYTES
    got = []
    for (x, lengths), kk in cases:
        xd, ld = torch.from_numpy(x).cuda(), torch.from_numpy(lengths).cuda()
        out = torch.full((x.shape[0], kk), -7, dtype=torch.int32, device="cuda")
        B.idx_topk_noalloc(xd, ld, kk, out)
        got.append(out)
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    for i, (((x, lengths), kk), out) in enumerate(zip(cases, got)):
        ref = oracle.topk(x, lengths, kk)
        assert_topk_exact(out.cpu().numpy(), ref, f"noalloc call {i}")
