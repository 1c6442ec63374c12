"""idx_row_ends and idx_fill_logits_tail on the GPU.

Row ends follow the rule the paged logits apply to their rows (one length
per sequence: row j of an n-row step ends at L - n + j + 1; one length per
row: that length), clamped to [0, width]; the tail fill writes -inf over
[ke, width) of every row and nothing else.  Both are compared with numpy
statements of the same rules, and the row ends also with the paged case's
own row_ends()."""
import numpy as np
import pytest
import torch

from sparse_attention_indexer_mxfp4_gb300 import _binding as B
from sparse_attention_indexer_mxfp4_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("next_n", [1, 2, 4])
@pytest.mark.parametrize("ctx_per_row", [False, True])
def test_row_ends_rule(next_n, ctx_per_row):
    rng = np.random.default_rng(3 + next_n)
    Bq, width = 37, 5000
    n = Bq * next_n if ctx_per_row else Bq
    ctx = rng.integers(-3, width + 300, size=n).astype(np.int32)
    ctx[:3] = [0, 1, next_n]
    out = torch.full((Bq * next_n,), -7, dtype=torch.int32, device="cuda")
    B.idx_row_ends(torch.from_numpy(ctx).cuda(), next_n, width, out, ctx_per_row=ctx_per_row)
    r = np.arange(Bq * next_n)
    raw = ctx if ctx_per_row else ctx[r // next_n] - next_n + r % next_n + 1
    np.testing.assert_array_equal(out.cpu().numpy(), np.clip(raw, 0, width))


def test_row_ends_match_the_paged_case():
    c = synth.CONFIGS[4]()
    out = torch.empty(c.rows, dtype=torch.int32, device="cuda")
    B.idx_row_ends(torch.from_numpy(c.context_lens).cuda(), c.next_n, c.width, out)
    np.testing.assert_array_equal(out.cpu().numpy(), np.clip(c.row_ends(), 0, c.width))


@pytest.mark.parametrize("ld,width", [(1031, 1031), (1032, 1030), (4096, 4096)])
def test_fill_logits_tail(ld, width):
    rng = np.random.default_rng(ld)
    rows = 9
    x = rng.standard_normal((rows, ld)).astype(np.float32)
    ends = np.array([0, 1, 3, 4, 5, width - 1, width, width + 50, -2], np.int32)
    xd = torch.from_numpy(x).cuda()
    B.idx_fill_logits_tail(xd, torch.from_numpy(ends).cuda(), width)
    want = x.copy()
    for i, e in enumerate(np.clip(ends, 0, width)):
        want[i, e:width] = -np.inf
    np.testing.assert_array_equal(xd.cpu().numpy(), want)
