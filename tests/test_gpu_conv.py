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
from _parity import assert_conv_close, report

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
                                   (3, 50, 512), (9, 17, 4096), (70, 16, 2560)])
def test_edge_shapes(B, L, d):
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(B=B, L=L, d=d)
    c = wl.make_conv_inputs(w, 3, "cpu")
    y = gpu_conv(c)
    _, yr = ref_conv(c)
    assert_conv_close(y, yr, f"B={B} L={L} d={d}")


def test_identity_and_shift():
    w = wl.WORKLOADS["drafter4b_l16"].with_(B=2)
    c = wl.make_conv_inputs(w, 0, "cpu")
    c["W_c"] = torch.zeros_like(c["W_c"])
    d = w.d
    c["base"] = torch.stack([torch.ones(d), torch.zeros(d)])
    np.testing.assert_array_equal(gpu_conv(c), wl.host(c["x"]))
    c["base"] = torch.stack([torch.zeros(d), torch.ones(d)])
    y = gpu_conv(c)
    np.testing.assert_array_equal(y[:, 0], wl.host(c["x_prev"]))
    np.testing.assert_array_equal(y[:, 1:], wl.host(c["x"])[:, :-1])
