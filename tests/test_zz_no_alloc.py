"""idx_topk_noalloc, the top-k entry point that runs from the library's fixed
per-device scratch array instead of caller memory: the same indices as
idx_topk on two calls in a row, and host-side rejection of calls that do
not fit the array.  Kept in its own file, collected after the others, so it
runs both alone and after every other GPU test in one process."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_mxfp4_gb300 import _binding as B

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3
FAKE = 0x10000  # never dereferenced: these calls fail their host checks first


def test_noalloc_rejects_calls_beyond_the_array():
    f = B.lib().idx_topk_noalloc
    ld, k = B.TOPK_CLUSTER_MAX_LEN + 4, 2048  # rows past the cluster path use the array
    too_many = next(r for r in range(1, 4096) if B.topk_workspace_size(r, ld, k) > (32 << 20))
    assert B.topk_workspace_size(too_many - 1, ld, k) <= (32 << 20)
    assert f(FAKE, ld, too_many, FAKE, k, FAKE, k, None) == WORKSPACE
    assert f(FAKE, 8192 * 1024 + 4, 2, FAKE, k, FAKE, k, None) == UNSUPPORTED
    assert f(FAKE, ld, 4, FAKE, k, FAKE, k - 1, None) == INVALID
    assert f(FAKE, ld, 0, FAKE, k, FAKE, k, None) == 0


def _case(rng, rows, width, tie_levels=None):
    if tie_levels:
        x = rng.integers(0, tie_levels, size=(rows, width)).astype(np.float32)
    else:
        x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < 0.3] = -np.inf
    lengths = rng.integers(0, width + 1, size=rows).astype(np.int32)
    lengths[0] = width
    return torch.from_numpy(x).cuda(), torch.from_numpy(lengths).cuda()


@pytest.mark.gpu
def test_noalloc_matches_idx_topk_on_two_calls_in_a_row():
    rng = np.random.default_rng(2024)
    # a long-row decode batch, then a smaller one with heavy ties: the second
    # call must not see anything the first left in the shared array
    cases = [(_case(rng, 96, 131072), 2048), (_case(rng, 7, 20000, tie_levels=3), 300),
             (_case(rng, 5, 300000), 2048)]
    got = []
    for (x, lengths), k in cases:
        out = torch.full((x.shape[0], k), -7, dtype=torch.int32, device="cuda")
        B.idx_topk_noalloc(x, lengths, k, out)
        got.append(out)
    for ((x, lengths), k), out in zip(cases, got):
        ref = torch.full_like(out, -9)
        B.idx_topk(x, lengths, k, ref, workspace=True)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert (out >= -1).all()
    assert B.idx_get_device_status() == 0
