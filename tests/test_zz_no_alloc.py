"""dfl2_topk_noalloc: the top-16 for callers that cannot allocate device memory
(engines that pre-reserve the GPU's memory for their own pool and forbid later
cudaMalloc, or plug-ins handed only input and output pointers).  It must give
exactly what dfl2_topk gives with a caller workspace, call after call, using
only the library's fixed scratch array.

This file is collected last on purpose, so that a failure here comes after
every other test has run.  It also runs on its own in a fresh process."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
WORKSPACE = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def with_workspace(lg):
    B, L, V = lg.shape
    idx = torch.empty(B, L, 16, dtype=torch.int32, device="cuda")
    val = torch.empty(B, L, 16, dtype=torch.float32, device="cuda")
    dfl2.dfl2_topk(lg, idx, val, dfl2.workspace(dfl2.dfl2_topk_workspace_size(B, L, V)))
    return idx, val


def without_workspace(lg):
    B, L, V = lg.shape
    idx = torch.full((B, L, 16), -7, dtype=torch.int32, device="cuda")
    val = torch.full((B, L, 16), -7.0, dtype=torch.float32, device="cuda")
    dfl2.dfl2_topk_noalloc(lg, idx, val)
    return idx, val


def test_matches_dfl2_topk_on_two_calls_in_a_row():
    # Call 1: the batch-1 4B-drafter block (16 rows, each split across many CTAs,
    # so the scratch tickets and partial lists are used).  Call 2: a different
    # shape and dtype right after, on the same stream, reusing the same scratch.
    first = wl.make_logits(wl.WORKLOADS["drafter4b_l16"], "cpu").cuda()
    second = wl.make_logits(wl.WORKLOADS["tiny_l8_v32k"].with_(B=3, L=5), "cpu").cuda()
    a1 = without_workspace(first)
    a2 = without_workspace(second)
    b1 = with_workspace(first)
    b2 = with_workspace(second)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    for (ia, va), (ib, vb) in ((a1, b1), (a2, b2)):
        np.testing.assert_array_equal(ia.cpu().numpy(), ib.cpu().numpy())
        np.testing.assert_array_equal(va.cpu().numpy(), vb.cpu().numpy())


def test_rejects_problems_larger_than_the_scratch():
    B, L, V = 2048, 16, 1024  # 32768 rows: about 8 MB of partial lists, over the 4 MiB limit
    assert dfl2.dfl2_topk_workspace_size(B, L, V) > 4 << 20
    lg = torch.empty(8, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    out = torch.empty(8, dtype=torch.int32, device="cuda")
    with pytest.raises(dfl2.Dfl2Error) as e:
        dfl2.dfl2_topk_noalloc(lg, out, out, dims=(B, L, V), dtype=dfl2.DFL2_BF16)
    assert e.value.status == WORKSPACE and "4194304" in e.value.message
