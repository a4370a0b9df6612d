"""The warp-level projection engine (mma.sync, each warp owning 32 output
columns) against the oracle, and against the tcgen05 engine, on the shapes
whose split-K plan gives CTAs of 128 output columns (batch 1 and 2 of the
4B drafter shape).  Same tolerances as the selector and tail tests."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
from _parity import assert_scores_close, report
from test_gpu_select import candidates_from_oracle, gpu_select, oracle_select_subset
from test_gpu_tail import check_tail

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


class engine:
    def __init__(self, e):
        self.e = e

    def __enter__(self):
        self.prev = dfl2.dfl2_set_projection_engine(self.e)

    def __exit__(self, *exc):
        dfl2.dfl2_set_projection_engine(self.prev)


@pytest.mark.parametrize("B,e_std,d", [(1, 1.0, 2560), (1, 0.02, 2560), (2, 1.0, 2560),
                                       (1, 1.0, 2576)])
def test_select_warp_engine(B, e_std, d):
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=B, d=d, e_std=e_std)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    with engine(dfl2.PROJ_WARP):
        S = gpu_select(idx, val, inp["verified"], inp)
    ref = oracle_select_subset(idx, val, inp["verified"], inp, list(range(B)))
    worst = assert_scores_close(S, ref, f"warp engine B={B} d={d}")
    report(kind="scores", what=f"warp engine drafter4b_l16 B={B} d={d} e_std={e_std}",
           worst_err_over_tol=worst)


def test_engines_agree():
    """Both engines run 16-deep tensor-core steps into fp32 accumulators over the
    same K blocks and the same rank-order split-K sum, so they agree closely (they
    may even round identically); each is also checked against the oracle above."""
    w = wl.WORKLOADS["drafter4b_l16"].with_(e_std=1.0)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    with engine(dfl2.PROJ_TENSOR):
        St = gpu_select(idx, val, inp["verified"], inp)
    with engine(dfl2.PROJ_WARP):
        Sw = gpu_select(idx, val, inp["verified"], inp)
    fin = np.isfinite(St)
    assert np.array_equal(fin, np.isfinite(Sw))
    err = np.abs(St[fin] - Sw[fin]) / np.maximum(np.abs(St[fin]), 1.0)
    assert err.max() <= 1e-4, err.max()
    report(kind="scores", what="tensor vs warp engine drafter4b_l16",
           identical=bool(np.array_equal(St, Sw)), max_rel_diff=float(err.max()))


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tail_warp_engine(T):
    w = wl.WORKLOADS["drafter4b_l16"].with_(e_std=1.0)
    lg = wl.make_logits(w, "cpu")
    inp = wl.make_tail_inputs(w, "cpu")
    with engine(dfl2.PROJ_WARP):
        check_tail(w, lg, inp, T, inp["seeds"], 5, [0])


@pytest.mark.parametrize("name,B,L,V,d", [
    ("drafter4b_l16", 3, 16, 151936, 2560),   # CTAs of 256 columns: the tcgen05 engine runs
    ("tiny_l8_v32k", 1, 8, 32768, 1024),     # CTAs of 64 columns: the tcgen05 engine runs
    ("tiny_l8_v32k", 40, 16, 4096, 256),     # the batched projection (no split K)
])
def test_warp_engine_request_elsewhere(name, B, L, V, d):
    """Asking for the warp-level engine on a plan it does not apply to leaves
    the scores exact to the usual tolerance."""
    w = wl.WORKLOADS[name].with_(B=B, L=L, V=V, d=d, e_std=1.0)
    inp = wl.make_tail_inputs(w, "cpu")
    idx, val = candidates_from_oracle(wl.make_logits(w, "cpu"))
    with engine(dfl2.PROJ_WARP):
        S = gpu_select(idx, val, inp["verified"], inp)
    seqs = list(range(min(B, 8)))
    ref = oracle_select_subset(idx, val, inp["verified"], inp, seqs)
    assert_scores_close(S[seqs], ref, f"warp engine requested, {name} B={B}")
