"""GPU parity of block verification (dfl2_verify) against the oracle, through
the C ABI, on synthetic target distributions.

Greedy: n_accepted and out_tokens bit-exact.  Sampling: the acceptance
decisions are exact (double precision on both sides), so n_accepted must match
exactly; the replacement or appended token may differ only where u1 * Z lies
within 1e-5 * Z of a boundary of the oracle's exact running sum (the GPU sums in
single precision inside 512-element tiles); such cases are counted and reported."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def gpu_verify(inp, greedy, cycle=0):
    p = inp["p"].cuda()
    B, L1, V = p.shape
    L = L1 - 1
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, L1, dtype=torch.int32, device="cuda")
    ws = dfl2.workspace(dfl2.dfl2_verify_workspace_size(B, L, V))
    seeds = torch.from_numpy(inp["seeds"].view(np.int64)).cuda()
    dfl2.dfl2_verify(p, inp["tokens"].cuda(), n, out, greedy=greedy, slots=inp["slots"].cuda(),
                     q=inp["q"].cuda(), cand_idx=inp["cand_idx"].cuda(), seeds=seeds,
                     cycle_offset=cycle, ws=ws)
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    return n.cpu().numpy(), out.cpu().numpy()


def ref_verify(inp, greedy, cycle=0, seqs=None):
    sel = slice(None) if seqs is None else seqs
    h = lambda k: wl.host(inp[k])[sel]
    return oracle.verify(h("p"), h("tokens"), h("slots"), h("q"), h("cand_idx"), greedy=greedy,
                         seeds=inp["seeds"][sel], cycle=cycle)


def near_boundary(p_row, cand, qrow, use_res, u1, pick_gpu, pick_ref):
    """True when the oracle's draw and the GPU's straddle a boundary within 1e-5 Z."""
    r = p_row.astype(np.float64).copy()
    if use_res:
        for k, c in enumerate(cand):
            r[c] -= qrow[k]
        r = np.maximum(r, 0.0)
        if r.sum() <= 0:
            r = p_row.astype(np.float64)
    Z = r.sum()
    cum = np.cumsum(r)
    lo, hi = min(pick_gpu, pick_ref), max(pick_gpu, pick_ref)
    T = u1 * Z
    return abs(T - cum[lo]) <= 1e-5 * Z or abs(T - cum[hi - 1]) <= 1e-5 * Z


def check_sampling(inp, cycle, seqs=None):
    n, out = gpu_verify(inp, greedy=False, cycle=cycle)
    sel = np.arange(n.shape[0]) if seqs is None else np.asarray(seqs)
    rn, rout = ref_verify(inp, greedy=False, cycle=cycle, seqs=sel)
    n, out = n[sel], out[sel]
    np.testing.assert_array_equal(n, rn)
    L = out.shape[1] - 1
    allowed = 0
    p = wl.host(inp["p"])
    for i, b in enumerate(sel):
        j = rn[i]
        np.testing.assert_array_equal(out[i, :j], rout[i, :j])
        assert (out[i, j + 1:] == -1).all()
        if out[i, j] != rout[i, j]:
            u1 = oracle.verify_uniforms(int(inp["seeds"][b]), cycle, int(j))[1]
            use_res = j < L
            cand = wl.host(inp["cand_idx"])[b, j] if use_res else []
            qrow = wl.host(inp["q"])[b, j] if use_res else []
            assert near_boundary(p[b, j], cand, qrow, use_res, u1, out[i, j], rout[i, j]), (b, j)
            allowed += 1
    return n, allowed


def test_greedy_small():
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=6, L=5, V=1000)
    inp = wl.make_verify_inputs(w)
    # make some drafts the target's argmax so that prefixes of every length occur
    p = inp["p"]
    am = p[:, :w.L].argmax(-1).to(torch.int32)
    keep = torch.arange(w.L)[None, :] < torch.arange(w.B)[:, None]
    inp["tokens"] = torch.where(keep, am, inp["tokens"])
    n, out = gpu_verify(inp, greedy=True)
    rn, rout = ref_verify(inp, greedy=True)
    np.testing.assert_array_equal(n, rn)
    np.testing.assert_array_equal(out, rout)
    assert len(set(rn.tolist())) >= 2


@pytest.mark.parametrize("B,L,V", [(64, 4, 4096), (3, 7, 1000), (1, 1, 16), (2, 16, 65536 + 4)])
def test_sampling_shapes(B, L, V):
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=B, L=L, V=V)
    inp = wl.make_verify_inputs(w)
    for cycle in (0, 5):
        n, allowed = check_sampling(inp, cycle)
        report(kind="verify", what=f"B={B} L={L} V={V} cycle={cycle}",
               mean_accepted=float(n.mean()), boundary_cases=allowed)


def test_sampling_all_accepted_appends_from_the_last_row():
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=32, L=3, V=2048)
    inp = wl.make_verify_inputs(w)
    # p_t = q_t on the candidates: every draft is kept
    p = torch.zeros_like(inp["p"])
    p[:, :w.L].scatter_(2, inp["cand_idx"].long(), inp["q"])
    p[:, w.L] = inp["p"][:, w.L]
    inp["p"] = p
    n, _ = check_sampling(inp, 3)
    assert (n == w.L).mean() > 0.9


def test_serving_b64_shape():
    w = wl.WORKLOADS["serving_b64"]
    inp = {k: (v.cpu() if isinstance(v, torch.Tensor) else v)
           for k, v in wl.make_verify_inputs(w, device="cuda").items()}
    n, allowed = check_sampling(inp, 11)
    ng, outg = gpu_verify(inp, greedy=True)
    rn, rout = ref_verify(inp, greedy=True)
    np.testing.assert_array_equal(ng, rn)
    np.testing.assert_array_equal(outg, rout)
    report(kind="verify", what="serving_b64", mean_accepted=float(n.mean()),
           boundary_cases=allowed, greedy_mean_accepted=float(ng.mean()))
