"""GPU parity of the fused tail (top-16 -> pair scores -> walk in one call)
against the oracle run step by step, on every workload shape.

Candidates: bit-exact.  Scores: 1e-3 relative.  Walk: step-wise replay
against the oracle's own double-precision scores, given the GPU's previous
choice; steps inside the greedy margin / sampling boundary are counted."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import assert_scores_close, replay_walk, report
from test_gpu_select import oracle_select_subset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def run_tail(w, lg, inp, T, seeds, cycle=0):
    B, L, V, d = w.B, w.L, w.V, w.d
    out = dict(
        tokens=torch.empty(B, L, dtype=torch.int32, device="cuda"),
        slots=torch.empty(B, L, dtype=torch.int32, device="cuda"),
        q=torch.empty(B, L, 16, dtype=torch.float32, device="cuda"),
        cand_idx=torch.empty(B, L, 16, dtype=torch.int32, device="cuda"),
        cand_val=torch.empty(B, L, 16, dtype=torch.float32, device="cuda"),
        scores=torch.empty(B, L, 16, 16, dtype=torch.float32, device="cuda"),
    )
    ws = dfl2.workspace(dfl2.dfl2_tail_workspace_size(B, L, V, d))
    sd = torch.from_numpy(seeds.view(np.int64)).cuda()
    c = lambda t: t if t.is_cuda else t.cuda()
    dfl2.dfl2_tail(c(lg), c(inp["verified"]), c(inp["hidden"]), c(inp["E"]), c(inp["W_A"]),
                   c(inp["W_B"]), c(inp["W_H"]), T, sd, cycle, out["tokens"], ws,
                   slots=out["slots"], q=out["q"], cand_idx=out["cand_idx"],
                   cand_val=out["cand_val"], scores=out["scores"])
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def check_tail(w, lg, inp, T, seeds, cycle, seqs, runner=None):
    g = (runner or run_tail)(w, lg, inp, T, seeds, cycle)
    V = w.V
    flat = lg.reshape(w.rows, V)
    rows = [b * w.L + t for b in seqs for t in range(w.L)]
    ri, rv = oracle.topk(wl.host(flat[rows]), 16)
    np.testing.assert_array_equal(g["cand_idx"][seqs].reshape(-1, 16), ri)
    np.testing.assert_array_equal(g["cand_val"][seqs].reshape(-1, 16), rv)
    ci = torch.from_numpy(g["cand_idx"])
    cv = torch.from_numpy(g["cand_val"])
    ref = oracle_select_subset(ci, cv, inp["verified"].cpu(), inp, seqs)
    worst = assert_scores_close(g["scores"][seqs], ref, w.name)
    allowed = replay_walk(ref, g["slots"][seqs], T, seeds[seqs], cycle, what=f"{w.name} T={T}")
    # q: the draft distribution of each step's row, where the paths agree with the oracle's
    _, rs, rq = oracle.walk(ref, g["cand_idx"][seqs], T, seeds[seqs], cycle)
    same = np.all(g["slots"][seqs] == rs, axis=1)
    np.testing.assert_allclose(g["q"][seqs][same], rq[same], rtol=1e-3, atol=1e-6)
    np.testing.assert_array_equal(
        g["tokens"], np.take_along_axis(g["cand_idx"], g["slots"][..., None].astype(np.int64),
                                        2)[..., 0])
    report(kind="tail", what=f"{w.name} T={T}", seqs=len(seqs), worst_err_over_tol=worst,
           allowed_walk_mismatches=allowed)
    return g


@pytest.mark.parametrize("name,T,e_std", [
    ("tiny_l8_v32k", 0.0, 0.02), ("tiny_l8_v32k", 0.0, 1.0),
    ("drafter4b_l16", 0.0, 0.02), ("drafter4b_l16", 1.0, 0.02), ("drafter4b_l16", 1.0, 1.0),
    ("drafter27b_l8", 0.0, 0.02), ("drafter27b_l8", 0.0, 1.0),
])
def test_small_workloads(name, T, e_std):
    w = wl.WORKLOADS[name].with_(e_std=e_std)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    check_tail(w, lg, inp, T, inp["seeds"], 0, list(range(w.B)))


def batched_seqs(w, nseq):
    """Every sequence when nseq >= B; otherwise nseq sequences spread evenly over
    the batch (first and last included), so that the checked rows fall in every
    row tile and every wave of the projection GEMM."""
    if nseq >= w.B:
        return list(range(w.B))
    return sorted({int(round(i * (w.B - 1) / (nseq - 1))) for i in range(nseq)})


@pytest.mark.parametrize("name,T,nseq", [("serving_b64", 1.0, 64), ("stress_b256_ties", 0.0, 32),
                                         ("stress_b256_ties", 0.7, 32)])
def test_batched_workloads(name, T, nseq):
    w = wl.WORKLOADS[name]
    lg = wl.make_logits(w, "cuda")
    inp = wl.make_tail_inputs(w, "cuda")
    check_tail(w, lg, inp, T, inp["seeds"], 12345, batched_seqs(w, nseq))


def test_tail_equals_the_three_calls():
    """The fused call gives exactly what dfl2_topk, dfl2_select and dfl2_walk give."""
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=3, e_std=1.0)
    lg = wl.make_logits(w, "cpu").cuda()
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in wl.make_tail_inputs(w, "cpu").items()}
    g = run_tail(w, lg, inp, 1.0, inp["seeds"], 77)
    B, L, V, d = w.B, w.L, w.V, w.d
    idx = torch.empty(B, L, 16, dtype=torch.int32, device="cuda")
    val = torch.empty(B, L, 16, dtype=torch.float32, device="cuda")
    dfl2.dfl2_topk(lg, idx, val, dfl2.workspace(dfl2.dfl2_topk_workspace_size(B, L, V)))
    S = torch.empty(B, L, 16, 16, device="cuda")
    dfl2.dfl2_select(idx, val, inp["verified"], inp["hidden"], inp["E"], inp["W_A"], inp["W_B"],
                     inp["W_H"], S, dfl2.workspace(dfl2.dfl2_select_workspace_size(B, L, d)))
    tok = torch.empty(B, L, dtype=torch.int32, device="cuda")
    sd = torch.from_numpy(inp["seeds"].view(np.int64)).cuda()
    dfl2.dfl2_walk(S, idx, 1.0, sd, 77, tok)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), g["cand_idx"])
    np.testing.assert_array_equal(S.cpu().numpy(), g["scores"])
    np.testing.assert_array_equal(tok.cpu().numpy(), g["tokens"])


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_batched_projection_path(T):
    """Enough sequences for the batched projection (each E row gathered once,
    [W_A; W_B] as one N = 512 product); the last row tile is ragged."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=40, L=16, V=4096, d=256, e_std=1.0)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    check_tail(w, lg, inp, T, inp["seeds"], 3, list(range(w.B)))


@pytest.mark.parametrize("B,L,V,d,T", [
    (1, 5, 50257, 2576, 1.0),   # batch 1: split K over a cluster, a 16-wide last K block
    (3, 16, 50257, 2576, 0.0),  # a few sequences, odd vocabulary
    (40, 16, 4099, 2576, 1.0),  # the batched projection ([W_A; W_B] as N = 512)
    (2, 8, 1021, 1040, 0.0),    # float32 logits of an odd length, d = 1040
])
def test_any_vocabulary_and_hidden_size(B, L, V, d, T):
    """Every V >= 16 and every d that is a multiple of 16: logits rows that do not
    start on 16 bytes, and a last K block of the projections that is only partly
    inside d."""
    base = "tiny_l8_v32k" if d == 1040 else "drafter4b_l16"
    w = wl.WORKLOADS[base].with_(B=B, L=L, V=V, d=d, e_std=1.0)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    check_tail(w, lg, inp, T, inp["seeds"], 9, list(range(B)))


def test_minimal_block():
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(L=1, V=16, d=64, e_std=1.0)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    check_tail(w, lg, inp, 0.0, inp["seeds"], 0, [0])
