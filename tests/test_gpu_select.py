"""GPU parity of the pair scores S_t(a,b) = U_t(b) + <A(a) ⊙ H(h_t), B(b)>
against the oracle's literal double-precision evaluation, through the C ABI.

Tolerance: |gpu - oracle| <= 1e-3 * max(|oracle|, 1) (fp32 accumulation).
The candidates fed to both sides come from the oracle's own top-16, so this
test does not depend on the GPU top-16."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import assert_scores_close, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def gpu_select(cand_idx, cand_val, verified, inp):
    B, L, d = inp["hidden"].shape
    V = inp["E"].shape[0]
    dev = lambda t: t.cuda() if not t.is_cuda else t
    scores = torch.empty(B, L, 16, 16, dtype=torch.float32, device="cuda")
    ws = dfl2.workspace(dfl2.dfl2_select_workspace_size(B, L, d))
    dfl2.dfl2_select(dev(cand_idx), dev(cand_val), dev(verified), dev(inp["hidden"]),
                     dev(inp["E"]), dev(inp["W_A"]), dev(inp["W_B"]), dev(inp["W_H"]), scores, ws)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    return scores.cpu().numpy()


def oracle_select_subset(cand_idx, cand_val, verified, inp, seqs):
    """Oracle scores for the sequences `seqs`, gathering only the E rows they use."""
    ci = cand_idx[seqs].cpu().numpy()
    vt = verified[seqs].cpu().numpy()
    toks = np.unique(np.concatenate([ci.ravel(), vt.ravel()]))
    remap = {int(t): i for i, t in enumerate(toks)}
    E_sub = wl.host(inp["E"][torch.from_numpy(toks).to(inp["E"].device).long()])
    ci_r = np.vectorize(remap.get)(ci).astype(np.int32)
    vt_r = np.array([remap[int(t)] for t in vt], np.int32)
    return oracle.select(ci_r, cand_val[seqs].cpu().numpy(), vt_r, wl.host(inp["hidden"][seqs]),
                         E_sub, wl.host(inp["W_A"]), wl.host(inp["W_B"]), wl.host(inp["W_H"]))


def candidates_from_oracle(logits):
    idx, val = oracle.topk(wl.host(logits), 16)
    return torch.from_numpy(idx), torch.from_numpy(val)


@pytest.mark.parametrize("name,e_std", [
    ("tiny_l8_v32k", 0.02), ("tiny_l8_v32k", 1.0),
    ("drafter4b_l16", 0.02), ("drafter4b_l16", 1.0),
    ("drafter27b_l8", 0.02),
])
def test_small_workloads(name, e_std):
    w = wl.WORKLOADS[name].with_(e_std=e_std)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    S = gpu_select(idx, val, inp["verified"], inp)
    ref = oracle_select_subset(idx, val, inp["verified"], inp, list(range(w.B)))
    worst = assert_scores_close(S, ref, name)
    bil = np.abs(ref - val.numpy()[:, :, None, :].astype(np.float64))
    report(kind="scores", what=f"{name} e_std={e_std}", worst_err_over_tol=worst,
           bilinear_mean_abs=float(np.nanmean(np.where(np.isinf(ref), np.nan, bil))))


@pytest.mark.parametrize("name,nseq", [("serving_b64", 64), ("stress_b256_ties", 32)])
def test_batched_workloads(name, nseq):
    w = wl.WORKLOADS[name]
    inp = wl.make_tail_inputs(w, "cuda")
    lg = wl.make_logits(w, "cuda")
    # candidates by torch.topk (exact for values; ties resolved arbitrarily, which is
    # fine here: the selector must score whatever candidates it is given)
    val, idx = torch.topk(lg.float(), 16, dim=-1)
    idx = idx.int().contiguous()
    val = val.contiguous()
    S = gpu_select(idx, val, inp["verified"], inp)
    # every sequence, or nseq spread evenly over the batch (every row tile and wave)
    seqs = (list(range(w.B)) if nseq >= w.B else
            sorted({int(round(i * (w.B - 1) / (nseq - 1))) for i in range(nseq)}))
    ref = oracle_select_subset(idx.cpu(), val.cpu(), inp["verified"].cpu(), inp, seqs)
    worst = assert_scores_close(S[seqs], ref, name)
    report(kind="scores", what=f"{name} {len(seqs)} of {w.B} sequences", worst_err_over_tol=worst)


# (40, 16) and (19, 33) have enough row tiles for the batched projection (no K
# split, every E row gathered once for both maps), with a ragged last row tile
@pytest.mark.parametrize("B,L,d", [(1, 1, 128), (3, 2, 128), (5, 17, 128), (40, 16, 256),
                                   (19, 33, 128)])
def test_edge_shapes(B, L, d):
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=B, L=L, V=4096, d=d, e_std=1.0)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    S = gpu_select(idx, val, inp["verified"], inp)
    ref = oracle_select_subset(idx, val, inp["verified"], inp, list(range(B)))
    assert_scores_close(S, ref, f"B={B} L={L} d={d}")


def test_zero_W_A_gives_plain_logits():
    w = wl.WORKLOADS["tiny_l8_v32k"]
    inp = wl.make_tail_inputs(w, "cpu")
    inp["W_A"] = torch.zeros_like(inp["W_A"])
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    S = gpu_select(idx, val, inp["verified"], inp)
    for t in range(w.L):
        rows = 1 if t == 0 else 16
        np.testing.assert_array_equal(S[:, t, :rows, :],
                                      np.broadcast_to(val.numpy()[:, t, None, :], (1, rows, 16)))


def test_out_of_range_candidate_is_reported_not_read():
    """A token id outside [0, V) is caught by the gather's bounds check: the row is
    treated as zeros and the device error word says so; nothing is read out of E."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(V=1024, d=64)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    idx = idx.clone()
    idx[0, 3, 5] = w.V  # one past the end
    dfl2.dfl2_device_error(clear=True)
    B, L, d = inp["hidden"].shape
    scores = torch.empty(B, L, 16, 16, device="cuda")
    ws = dfl2.workspace(dfl2.dfl2_select_workspace_size(B, L, d))
    dfl2.dfl2_select(idx.cuda(), val.cuda(), inp["verified"].cuda(), inp["hidden"].cuda(),
                     inp["E"].cuda(), inp["W_A"].cuda(), inp["W_B"].cuda(), inp["W_H"].cuda(),
                     scores, ws)
    assert dfl2.dfl2_device_error(clear=True) == 5
