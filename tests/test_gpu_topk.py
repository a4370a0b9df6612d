"""GPU parity of the top-16 step against the oracle's full sort, through the C ABI.

Bit-exact: indices and values, with ties broken by value descending then index
ascending.  Small workloads are compared on every row; the batched workloads
on sampled rows against the oracle and on every row through properties that
hold at any size."""
import json
import os

import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def gpu_topk(logits: torch.Tensor):
    B, L, V = logits.shape
    idx = torch.empty(B, L, 16, dtype=torch.int32, device="cuda")
    val = torch.empty(B, L, 16, dtype=torch.float32, device="cuda")
    ws = dfl2.workspace(dfl2.dfl2_topk_workspace_size(B, L, V))
    dfl2.dfl2_topk(logits, idx, val, ws)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    return idx.cpu().numpy(), val.cpu().numpy()


def check_rows(logits: torch.Tensor, idx, val, rows=None):
    host = wl.host(logits)
    V = host.shape[-1]
    flat = host.reshape(-1, V)
    gi, gv = idx.reshape(-1, 16), val.reshape(-1, 16)
    rows = range(flat.shape[0]) if rows is None else rows
    sel = np.array(list(rows))
    ri, rv = oracle.topk(flat[sel], 16)
    np.testing.assert_array_equal(gi[sel], ri)
    np.testing.assert_array_equal(gv[sel], rv)


def check_properties(logits: torch.Tensor, idx: np.ndarray, val: np.ndarray):
    """At any size: values are the 16 largest (torch.topk's multiset, sorted),
    each index holds its value, and the members tied with the 16th value are the
    lowest-index elements of that value."""
    R = idx.shape[0] * idx.shape[1]
    V = logits.shape[-1]
    lg = logits.reshape(R, V)
    gi = torch.from_numpy(idx.reshape(R, 16)).cuda().long()
    gv = torch.from_numpy(val.reshape(R, 16)).cuda()
    for r0 in range(0, R, 256):
        x = lg[r0:r0 + 256].float()
        i, v = gi[r0:r0 + 256], gv[r0:r0 + 256]
        tv = torch.topk(x, 16, dim=1, sorted=True).values
        assert torch.equal(tv, v), "values differ from the 16 largest"
        assert torch.equal(torch.gather(x, 1, i), v), "an index does not hold its value"
        v16 = v[:, 15:16]
        n_gt = (x > v16).sum(1)
        members_eq = (v == v16).sum(1)
        assert torch.all(n_gt + members_eq == 16)
        # the tied members must be the first `members_eq` positions holding v16
        eq = (x == v16)
        rank = torch.cumsum(eq.int(), dim=1)
        first_ok = torch.gather(rank, 1, i) <= members_eq[:, None]
        assert torch.all(first_ok | (v != v16)), "tie-break is not index ascending"
        assert torch.all(i[:, 1:] != i[:, :-1])


def test_golden_ties_case():
    g = json.load(open(os.path.join(GOLD, "topk_ties.json")))
    row = np.array([float(x) for x in g["logits"]], np.float32)
    for dt in (torch.float32, torch.bfloat16):
        lg = torch.tensor(row).to(dt).view(1, 1, -1).cuda()
        idx, val = gpu_topk(lg)
        assert idx[0, 0].tolist() == g["idx"]
        assert val[0, 0].tolist() == g["val"]


@pytest.mark.parametrize("name", ["tiny_l8_v32k", "drafter4b_l16", "drafter27b_l8"])
def test_small_workloads_all_rows(name):
    w = wl.WORKLOADS[name]
    lg = wl.make_logits(w, "cpu").cuda()
    idx, val = gpu_topk(lg)
    check_rows(lg, idx, val)


def test_serving_b64_sampled_rows_and_properties():
    w = wl.WORKLOADS["serving_b64"]
    lg = wl.make_logits(w, "cuda")
    idx, val = gpu_topk(lg)
    check_properties(lg, idx, val)
    rng = np.random.default_rng(0)
    rows = sorted(set(rng.choice(w.rows, 24, replace=False).tolist()) | {0, w.rows - 1})
    sub = lg.reshape(w.rows, w.V)[rows].reshape(1, len(rows), w.V)
    check_rows(sub, idx.reshape(-1, 16)[rows].reshape(1, -1, 16),
               val.reshape(-1, 16)[rows].reshape(1, -1, 16))


def test_stress_ties_sampled_rows_and_properties():
    w = wl.WORKLOADS["stress_b256_ties"]
    lg = wl.make_logits(w, "cuda")
    idx, val = gpu_topk(lg)
    check_properties(lg, idx, val)
    rng = np.random.default_rng(1)
    rows = sorted(set(rng.choice(w.rows, 12, replace=False).tolist()) | {0, w.rows - 1})
    sub = lg.reshape(w.rows, w.V)[rows].reshape(1, len(rows), w.V)
    check_rows(sub, idx.reshape(-1, 16)[rows].reshape(1, -1, 16),
               val.reshape(-1, 16)[rows].reshape(1, -1, 16))
    # the quantised logits must actually produce ties at the 16th place
    v = val.reshape(-1, 16)
    assert np.mean(v[:, 14] == v[:, 15]) > 0.5


@pytest.mark.parametrize("B,L,V,dt", [
    (1, 1, 16, torch.float32),       # minimum vocabulary, one row
    (1, 1, 16, torch.bfloat16),
    (1, 3, 24, torch.float32),       # less than one 16-byte vector past the minimum
    (2, 3, 8200, torch.bfloat16),    # two full 8 KB tiles plus a 16-byte ragged tile
    (1, 5, 12292, torch.float32),    # ragged last tile, float32
    (37, 3, 1000, torch.bfloat16),   # many short rows: several rows per CTA
    (3, 7, 65536 + 8, torch.bfloat16),
])
def test_edge_shapes(B, L, V, dt):
    g = torch.Generator().manual_seed(B * 1000 + L * 10 + V)
    lg = (torch.randn(B, L, V, generator=g) * 3).to(dt)
    idx, val = gpu_topk(lg.cuda())
    check_rows(lg, idx, val)


@pytest.mark.parametrize("B,L,V,dt", [
    (1, 7, 50257, torch.bfloat16),   # rows start anywhere in a 16-byte unit: cluster kernel
    (64, 16, 50257, torch.bfloat16),  # the same, one CTA per row
    (3, 5, 1021, torch.float32),     # float32 rows of an odd length
    (40, 16, 1023, torch.float32),   # many short odd rows
    (1, 3, 17, torch.bfloat16),      # one past the minimum: rows of 34 bytes
    (5, 3, 4099, torch.bfloat16),    # the buffer ends 10 bytes past its last whole 16
    (37, 9, 1023, torch.float32),    # the same, one CTA per row (float32)
    (63, 5, 50257, torch.bfloat16),  # and bf16
    (2, 8, 1000003, torch.bfloat16),  # few long rows split across CTAs: persistent kernel
    (1, 5, 500009, torch.float32),   # the same in float32
    (20, 8, 16, torch.bfloat16),     # many rows of the minimum length, one CTA per row
    (200, 1, 17, torch.float32),     # many 68-byte rows, several in each 16-byte-aligned window
])
def test_unaligned_rows(B, L, V, dt):
    """Rows whose start is not a multiple of 16 bytes: each is streamed as the
    aligned window around it, the neighbours' elements masked, and the bytes past
    the buffer's last whole 16 read with plain loads."""
    g = torch.Generator().manual_seed(B * 7 + L * 3 + V)
    lg = (torch.randn(B, L, V, generator=g) * 3).to(dt)
    idx, val = gpu_topk(lg.cuda())
    check_rows(lg, idx, val)
    # winners at the very first and last elements of every row, -inf everywhere else
    x = torch.full((B, L, V), float("-inf"))
    x[..., 0] = 2.0
    x[..., -1] = 3.0
    x = x.to(dt)
    idx, val = gpu_topk(x.cuda())
    check_rows(x, idx, val)
    assert (idx[..., 0] == V - 1).all() and (idx[..., 1] == 0).all()
    assert (idx >= 0).all() and (idx < V).all()


def test_degenerate_rows():
    V = 4096
    rows = []
    rows.append(torch.zeros(V))                                   # all equal: indices 0..15
    r = torch.full((V,), float("-inf")); r[100] = 1.0; rows.append(r)   # mostly -inf
    r = torch.zeros(V); r[::2] = -0.0; rows.append(r)             # signed zeros tie
    r = torch.arange(V, dtype=torch.float32); rows.append(r)      # best at the very end
    r = -torch.arange(V, dtype=torch.float32); rows.append(r)     # best at the start
    r = torch.full((V,), 5.0); r[-16:] = 6.0; rows.append(r)      # winners in the last vector
    lg = torch.stack(rows).view(1, len(rows), V)
    for dt in (torch.float32, torch.bfloat16):
        x = lg.to(dt)
        idx, val = gpu_topk(x.cuda())
        check_rows(x, idx, val)
    assert idx[0, 0].tolist() == list(range(16))


def test_adversarial_long_rows():
    """Full-vocabulary rows whose order defeats an early bound: rising values (every
    element beats everything before it, so the candidate buffer fills and the bound
    keeps rising), falling values, one constant (all tied), a sawtooth with a rising
    envelope, and rows with their winners spread one per tile."""
    V = 151936
    ar = torch.arange(V, dtype=torch.float32)
    rows = [ar / 64.0, -ar / 64.0, torch.full((V,), 0.25),
            (ar % 4096) / 4096.0 + ar / V,
            torch.where(ar % 4096 == 17, 3.0 + ar / V, torch.zeros(V))]
    for dt in (torch.float32, torch.bfloat16):
        lg = torch.stack(rows).view(1, len(rows), V).to(dt)
        idx, val = gpu_topk(lg.cuda())
        check_rows(lg, idx, val)
