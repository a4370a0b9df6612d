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


def _persistent_split_path(B, L, V):
    """True when dfl2_topk runs its persistent kernel for this shape, where rows
    are split across CTAs and the partial lists and per-row tickets live in the
    scratch; the row kernels (one cluster, or one CTA, per row) use no scratch.
    The rule restates the library's dispatch: one cluster of C <= 8 CTAs per row
    while rows * C <= 2 * SMs and each CTA streams at most 16 tiles of 8 KB;
    otherwise one CTA per row once there are at least as many rows as SMs;
    otherwise the persistent kernel."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = B * L
    tiles = -(-V * 2 // 8192)  # bf16 rows
    C = min(8, tiles)
    while C > 1 and rows * C > 2 * sms:
        C //= 2
    clusters = rows * C <= 2 * sms and -(-tiles // C) <= 16
    return not clusters and rows < sms


def test_matches_dfl2_topk_on_calls_in_a_row():
    # Two calls in a row on a shape whose rows are split across CTAs (few rows of
    # a 524,288-entry vocabulary: the scratch's partial lists and tickets are
    # used; the second call reuses the tickets the first one left), then a shape
    # with twice the rows (a different ticket and partial-list layout in the
    # same array), then the batch-1 4B-drafter block, which takes the
    # scratch-free cluster kernel.
    base = wl.WORKLOADS["serving_b64"].with_(V=524288)
    split_a = base.with_(B=4)
    split_b = base.with_(B=8, seed=2003)
    for w in (split_a, split_b):
        assert _persistent_split_path(w.B, w.L, w.V), w
        assert dfl2.dfl2_topk_workspace_size(w.B, w.L, w.V) <= 4 << 20
    first = wl.make_logits(split_a, "cuda")
    second = wl.make_logits(split_b, "cuda")
    third = wl.make_logits(wl.WORKLOADS["drafter4b_l16"], "cpu").cuda()
    got = [without_workspace(first), without_workspace(first), without_workspace(second),
           without_workspace(third)]
    want = [with_workspace(first), with_workspace(first), with_workspace(second),
            with_workspace(third)]
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    for (ia, va), (ib, vb) in zip(got, want):
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
