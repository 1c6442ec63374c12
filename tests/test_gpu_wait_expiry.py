"""The timeout path of the library's bounded device waits, made to run out
on purpose without breaking a kernel: idx_debug_wait_expiry waits, with the
same wait functions the kernels use, on a condition that never holds (an
mbarrier no thread arrives on; a grid barrier one CTA never reaches).  The
wait must give up after its limit, set IDX_DEV_TIMEOUT, end the kernel, and
leave the context usable: the next call, a chunked top-k whose phases meet
at real grid barriers, runs clean and matches the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
from parity import assert_topk_exact
from sparse_attention_indexer_mxfp4_gb300 import _binding as B

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000  # 50 ms


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "grid-barrier"])
def test_wait_runs_out_then_next_call_is_clean(which):
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    t0 = time.perf_counter()
    B.idx_debug_wait_expiry(which, LIMIT_NS)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    status = B.idx_get_device_status()
    assert status & B.DEV_TIMEOUT, f"status {status}: the wait did not report its timeout"
    assert waited >= 0.9 * LIMIT_NS * 1e-9, f"returned after {waited * 1e3:.1f} ms"
    assert B.idx_get_device_status() == 0, "reading the status clears it"

    # the next call: 200 rows of 131072 keys take the chunked top-k (its
    # clusters would not fit one wave), with grid barriers between phases
    rng = np.random.default_rng(7 + which)
    rows, width, k = 200, 131072, 2048
    x = rng.standard_normal((rows, width)).astype(np.float32)
    lengths = rng.integers(1, width + 1, size=rows).astype(np.int32)
    out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    B.idx_topk(torch.from_numpy(x).cuda(), torch.from_numpy(lengths).cuda(), k, out,
               workspace=True)
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    assert_topk_exact(out.cpu().numpy(), oracle.topk(x, lengths, k), "top-k after a timeout")


def test_wait_expiry_rejects_bad_arguments():
    with pytest.raises(B.IndexerError):
        B.idx_debug_wait_expiry(2, LIMIT_NS)
    with pytest.raises(B.IndexerError):
        B.idx_debug_wait_expiry(0, 0)
