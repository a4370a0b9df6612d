"""GPU parity of the token-table variant (P_A = E W_A^T, P_B = E W_B^T built
once; the per-cycle path gathers their rows) against the oracle, through the
C ABI.  Tables: every sampled row against the oracle's double-precision
projection.  Scores and the tail: the same rules as the per-cycle path
(tests/_parity.py)."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import assert_scores_close, report
from test_gpu_select import candidates_from_oracle, oracle_select_subset
from test_gpu_tail import check_tail

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def build_tables(inp):
    E = inp["E"].cuda()
    V = E.shape[0]
    PA = torch.empty(V, 256, dtype=torch.float32, device="cuda")
    PB = torch.empty_like(PA)
    dfl2.dfl2_tables_build(E, inp["W_A"].cuda(), inp["W_B"].cuda(), PA, PB)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    return PA, PB


@pytest.mark.parametrize("name,e_std", [("tiny_l8_v32k", 1.0), ("drafter4b_l16", 0.02),
                                        ("drafter27b_l8", 1.0)])
def test_tables_match_the_projection(name, e_std):
    w = wl.WORKLOADS[name].with_(e_std=e_std)
    inp = wl.make_tail_inputs(w, "cpu")
    PA, PB = build_tables(inp)
    PA, PB = PA.cpu().numpy(), PB.cpu().numpy()
    rng = np.random.default_rng(3)
    toks = sorted(set(rng.choice(w.V, 48, replace=False).tolist()) | {0, w.V - 1})
    E, WA, WB = wl.host(inp["E"]), wl.host(inp["W_A"]), wl.host(inp["W_B"])
    wmax = {id(WA): inp["W_A"].float().abs().max().item(),
            id(WB): inp["W_B"].float().abs().max().item()}
    worst = 0.0
    for t in toks:
        for tab, W in ((PA, WA), (PB, WB)):
            ref = oracle.proj_token(E, W, t)
            # float32 accumulation of d exact products: bounded by a small
            # multiple of eps times the sum of their magnitudes
            scale = inp["E"][t].float().abs().sum().item() * wmax[id(W)]
            err = np.abs(tab[t] - ref).max() / max(scale * 1e-6, 1e-30)
            worst = max(worst, err)
            np.testing.assert_allclose(tab[t], ref, rtol=1e-5, atol=2e-5 * scale)
    report(kind="tables", what=name, rows=len(toks), worst_err_over_1e6_scale=worst)


@pytest.mark.parametrize("name,e_std", [("tiny_l8_v32k", 1.0), ("drafter4b_l16", 1.0),
                                        ("drafter27b_l8", 0.02)])
def test_select_tables(name, e_std):
    w = wl.WORKLOADS[name].with_(e_std=e_std)
    inp = wl.make_tail_inputs(w, "cpu")
    PA, PB = build_tables(inp)
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    B, L, d = w.B, w.L, w.d
    S = torch.empty(B, L, 16, 16, device="cuda")
    ws = dfl2.workspace(dfl2.dfl2_select_workspace_size(B, L, d))
    dfl2.dfl2_select_tables(idx.cuda(), val.cuda(), inp["verified"].cuda(), inp["hidden"].cuda(),
                            inp["W_H"].cuda(), PA, PB, S, ws)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    ref = oracle_select_subset(idx, val, inp["verified"], inp, list(range(B)))
    worst = assert_scores_close(S.cpu().numpy(), ref, name)
    report(kind="select_tables", what=f"{name} e_std={e_std}", worst_err_over_tol=worst)


def run_tail_tables_with(PA, PB):
    def run(w, lg, inp, T, seeds, cycle=0):
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
        dfl2.dfl2_tail_tables(c(lg), c(inp["verified"]), c(inp["hidden"]), c(inp["W_H"]), PA, PB,
                              T, sd, cycle, out["tokens"], ws, slots=out["slots"], q=out["q"],
                              cand_idx=out["cand_idx"], cand_val=out["cand_val"],
                              scores=out["scores"])
        torch.cuda.synchronize()
        assert dfl2.dfl2_device_error() == 0
        return {k: v.cpu().numpy() for k, v in out.items()}
    return run


@pytest.mark.parametrize("name,T,e_std", [("tiny_l8_v32k", 0.0, 1.0), ("drafter4b_l16", 1.0, 1.0),
                                          ("drafter4b_l16", 0.0, 0.02), ("drafter27b_l8", 0.0, 1.0)])
def test_tail_tables_small(name, T, e_std):
    w = wl.WORKLOADS[name].with_(e_std=e_std)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    PA, PB = build_tables(inp)
    check_tail(w, lg, inp, T, inp["seeds"], 3, list(range(w.B)), runner=run_tail_tables_with(PA, PB))


def test_tail_tables_serving_b64_sampled():
    w = wl.WORKLOADS["serving_b64"]
    lg = wl.make_logits(w, "cuda")
    inp = wl.make_tail_inputs(w, "cuda")
    PA, PB = build_tables(inp)
    seqs = sorted({0, w.B - 1} | set(np.random.default_rng(9).choice(w.B, 3, False).tolist()))
    check_tail(w, lg, inp, 1.0, inp["seeds"], 4321, seqs, runner=run_tail_tables_with(PA, PB))


def test_tail_tables_equals_the_per_cycle_tail():
    """Both variants pick the same candidates, and their scores agree to the
    score tolerance (the tables only reorder the float32 accumulation)."""
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=2, e_std=1.0)
    lg = wl.make_logits(w, "cpu").cuda()
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in wl.make_tail_inputs(w, "cpu").items()}
    PA, PB = build_tables(inp)
    from test_gpu_tail import run_tail
    a = run_tail(w, lg, inp, 0.0, inp["seeds"], 0)
    b = run_tail_tables_with(PA, PB)(w, lg, inp, 0.0, inp["seeds"], 0)
    np.testing.assert_array_equal(a["cand_idx"], b["cand_idx"])
    assert_scores_close(b["scores"], a["scores"].astype(np.float64), "tables vs per-cycle")
