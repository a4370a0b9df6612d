"""GPU parity of the two-tap dynamic conv against the oracle, through the C ABI.

Tolerance: |gpu - oracle_bf16| <= max(2e-2, 1 bf16 ulp of the oracle value):
both round once to bf16 and a value near a rounding boundary may land on
either neighbour."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import assert_conv_close, bf16_bits_to_f64, bf16_ulp, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def gpu_conv(c):
    x = c["x"].cuda()
    y = torch.empty_like(x)
    dfl2.dfl2_conv2(x, c["x_prev"].cuda(), c["base"].cuda(), c["W_c"].cuda(), y)
    torch.cuda.synchronize()
    return wl.host(y)


def ref_conv(c, seqs=None):
    x, xp = c["x"], c["x_prev"]
    if seqs is not None:
        x, xp = x[seqs], xp[seqs]
    return oracle.conv2(wl.host(x), wl.host(xp), wl.host(c["base"]), wl.host(c["W_c"]))


@pytest.mark.parametrize("name,calls", [("tiny_l8_v32k", [0]), ("drafter4b_l16", [0, 7, 19]),
                                        ("drafter27b_l8", [0, 13])])
def test_small_workloads(name, calls):
    w = wl.WORKLOADS[name]
    for k in calls:
        c = wl.make_conv_inputs(w, k, "cpu")
        y = gpu_conv(c)
        _, yr = ref_conv(c)
        exact = assert_conv_close(y, yr, f"{name} call {k}")
        report(kind="conv", what=f"{name} call {k}", bitwise_equal_fraction=exact)


@pytest.mark.parametrize("name,nseq", [("serving_b64", 64), ("stress_b256_ties", 3)])
def test_batched_workloads(name, nseq):
    w = wl.WORKLOADS[name]
    c = wl.make_conv_inputs(w, 5, "cuda")
    y = gpu_conv(c)
    seqs = list(range(w.B)) if nseq >= w.B else sorted(
        {0, w.B - 1} | set(np.random.default_rng(4).choice(w.B, nseq, False).tolist()))
    _, yr = ref_conv(c, seqs)
    exact = assert_conv_close(y[seqs], yr, name)
    report(kind="conv", what=f"{name} seqs={len(seqs)}", bitwise_equal_fraction=exact)


@pytest.mark.parametrize("B,L,d", [(1, 1, 16), (1, 17, 48), (3, 5, 1024), (2, 33, 6144),
                                   (4, 16, 2560), (1, 2, 10240), (2, 8, 2560), (1, 16, 48),
                                   (1, 3, 32), (1, 4, 20480), (16, 1, 2560), (5, 16, 2560),
                                   (3, 50, 512), (9, 17, 4096), (70, 16, 2560),
                                   (5, 13, 512), (4, 17, 2560), (20, 16, 6144)])
def test_edge_shapes(B, L, d):
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=B, L=L, d=d)
    c = wl.make_conv_inputs(w, 3, "cpu")
    y = gpu_conv(c)
    _, yr = ref_conv(c)
    assert_conv_close(y, yr, f"B={B} L={L} d={d}")


@pytest.mark.parametrize("B", [2, 9])
def test_identity_and_shift(B):
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=B)
    c = wl.make_conv_inputs(w, 0, "cpu")
    c["W_c"] = torch.zeros_like(c["W_c"])
    d = w.d
    c["base"] = torch.stack([torch.ones(d), torch.zeros(d)])
    np.testing.assert_array_equal(gpu_conv(c), wl.host(c["x"]))
    c["base"] = torch.stack([torch.zeros(d), torch.ones(d)])
    y = gpu_conv(c)
    np.testing.assert_array_equal(y[:, 0], wl.host(c["x_prev"]))
    np.testing.assert_array_equal(y[:, 1:], wl.host(c["x"])[:, :-1])


# ---- dfl2_conv2_ws: the split-K kernel for many positions ----------------------

def gpu_conv_ws(c):
    x = c["x"].cuda()
    B, L, d = x.shape
    n = dfl2.dfl2_conv2_workspace_size(B, L, d)
    ws = dfl2.workspace(n, "cuda") if n else None
    y = torch.empty_like(x)
    dfl2.dfl2_conv2_ws(x, c["x_prev"].cuda(), c["base"].cuda(), c["W_c"].cuda(), y, ws)
    torch.cuda.synchronize()
    return wl.host(y), n


@pytest.mark.parametrize("B,L,d", [(64, 16, 2560), (8, 16, 2560), (5, 16, 2560), (70, 16, 2560),
                                   (3, 50, 512), (9, 17, 4096), (2, 33, 6144), (5, 13, 512),
                                   (20, 16, 6144), (4, 17, 2560), (1, 16, 2560), (3, 5, 1024),
                                   (40, 13, 2560), (25, 21, 4096), (32, 16, 2560),
                                   (128, 16, 2560)])
def test_ws_edge_shapes(B, L, d):
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=B, L=L, d=d)
    c = wl.make_conv_inputs(w, 3, "cpu")
    y, n = gpu_conv_ws(c)
    if B * L <= 64:
        assert n == 0, (B, L, d, n)  # few positions: no split, no workspace
    _, yr = ref_conv(c)
    assert_conv_close(y, yr, f"ws B={B} L={L} d={d}")
    y2, _ = gpu_conv_ws(c)
    np.testing.assert_array_equal(y2, y)  # fixed summation order: same bits every call


def test_ws_serving_workload_against_oracle_and_plain_call():
    w = wl.WORKLOADS["serving_b64"]
    c = wl.make_conv_inputs(w, 11, "cuda")
    y, n = gpu_conv_ws(c)
    assert n > 0  # this shape takes the split kernel
    seqs = [0, 17, 40, w.B - 1]
    _, yr = ref_conv(c, seqs)
    exact = assert_conv_close(y[seqs], yr, "serving_b64 ws")
    report(kind="conv", what="serving_b64 ws seqs=4", bitwise_equal_fraction=exact)
    # against the workspace-free call on every sequence: both within the
    # oracle's tolerance, so at most one bf16 step apart
    yp = bf16_bits_to_f64(gpu_conv(c))
    diff = np.abs(bf16_bits_to_f64(y) - yp)
    assert np.all(diff <= np.maximum(2e-2, bf16_ulp(yp))), float(diff.max())


def test_ws_identity_and_shift():
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=64)
    c = wl.make_conv_inputs(w, 0, "cpu")
    c["W_c"] = torch.zeros_like(c["W_c"])
    d = w.d
    c["base"] = torch.stack([torch.ones(d), torch.zeros(d)])
    np.testing.assert_array_equal(gpu_conv_ws(c)[0], wl.host(c["x"]))
    c["base"] = torch.stack([torch.zeros(d), torch.ones(d)])
    y = gpu_conv_ws(c)[0]
    np.testing.assert_array_equal(y[:, 0], wl.host(c["x_prev"]))
    np.testing.assert_array_equal(y[:, 1:], wl.host(c["x"])[:, :-1])


def test_ws_too_small_is_rejected():
    x = torch.zeros(64, 16, 2560, dtype=torch.bfloat16, device="cuda")
    n = dfl2.dfl2_conv2_workspace_size(64, 16, 2560)
    assert n > 0
    ws = dfl2.workspace(n, "cuda")
    base = torch.zeros(2, 2560, device="cuda")
    W_c = torch.zeros(320, 2560, dtype=torch.bfloat16, device="cuda")
    xp = torch.zeros(64, 2560, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(RuntimeError, match="workspace"):
        dfl2.dfl2_conv2_ws(x, xp, base, W_c, y, ws, ws_bytes=n - 16)
    with pytest.raises(RuntimeError, match="workspace"):
        dfl2.dfl2_conv2_ws(x, xp, base, W_c, y, None)
