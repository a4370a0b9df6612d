"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what pins it: hand-computed golden cases (tests/golden, each
with its citation), published known-answer vectors, closed forms of special
cases, library routines, invariants stated on the pages, brute force on tiny
inputs, and exact sampling distributions.  None of these needs a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from draft_selection_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bf16(a) -> np.ndarray:
    """float values (exact in bf16) -> bf16 bit patterns."""
    t = torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f(x):
    return float(x) if not isinstance(x, str) else float(x.replace("inf", "inf"))


# ------------------------------------------------------------------ Philox


def test_philox_known_answer_vectors():
    """Pin: published Random123 known-answer vectors for Philox4x32-10."""
    kat = _load("philox4x32_10_kat.json")
    for v in kat["vectors"]:
        ctr = [int(x, 16) for x in v["counter"]]
        key = [int(x, 16) for x in v["key"]]
        want = [int(x, 16) for x in v["output"]]
        assert list(oracle.philox4x32_10(ctr, key)) == want


def test_walk_uniform_counter_layout():
    """Pin: the walk's uniform at (seed 0, cycle 0, step 0) is word 0 of the
    all-zero known-answer vector, top 24 bits, scaled by 2^-24."""
    kat = _load("philox4x32_10_kat.json")["vectors"][0]
    word0 = int(kat["output"][0], 16)
    assert oracle.walk_uniform(0, 0, 0) == (word0 >> 8) * 2.0**-24
    # counter word 0 is the step, words 1-2 the cycle, key the seed
    seed, cycle, t = 0x0123456789ABCDEF, 0xFEDCBA9876543210, 5
    out = oracle.philox4x32_10([t, cycle & 0xFFFFFFFF, cycle >> 32, 0],
                               [seed & 0xFFFFFFFF, seed >> 32])
    assert oracle.walk_uniform(seed, cycle, t) == (int(out[0]) >> 8) * 2.0**-24


# ------------------------------------------------------------------ bf16 rounding


def test_round_bf16_matches_torch_on_float32_values():
    """Pin: library routine. For values that are exact float32, rounding the
    double to bf16 must agree with torch's float32 -> bf16 (round to nearest even)."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(3.0),
        rng.standard_normal(500).astype(np.float32) * np.float32(1e-39),  # subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4e38, -3.4e38, 1.0078125, 1.01171875],
                 np.float32),
    ])
    # exact halfway cases: 1 + 2^-8 (ties to even -> 1), 1 + 3*2^-8 (-> 1 + 2^-6)
    vals = np.concatenate([vals, np.array([1 + 2**-8, 1 + 3 * 2**-8], np.float32)])
    want = torch.tensor(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------------ top-16


def test_topk_golden_ties():
    """Pin: hand-built case with equal logits, signed zeros and -inf."""
    g = _load("topk_ties.json")
    logits = np.array([_f(x) for x in g["logits"]], np.float32)
    for arr in (logits, _bf16(logits)):
        idx, val = oracle.topk(arr[None, :], g["k"])
        assert idx[0].tolist() == g["idx"]
        assert val[0].tolist() == g["val"]


def _brute_topk(row, k):
    """Repeated selection: the largest remaining value, lowest index on ties."""
    vals = [float(v) for v in row]
    taken = [False] * len(vals)
    out = []
    for _ in range(k):
        best = None
        for i, v in enumerate(vals):
            if taken[i]:
                continue
            if best is None or v > vals[best]:
                best = i
        taken[best] = True
        out.append(best)
    return out


@pytest.mark.parametrize("V", [16, 17, 40, 64])
def test_topk_brute_force_tiny(V):
    """Pin: brute-force selection on tiny vocabularies, with heavy ties."""
    rng = np.random.default_rng(V)
    rows = rng.integers(-4, 5, size=(12, V)).astype(np.float32) * np.float32(0.5)
    idx, val = oracle.topk(rows, 16)
    for r in range(rows.shape[0]):
        want = _brute_topk(rows[r], 16)
        assert idx[r].tolist() == want
        np.testing.assert_array_equal(val[r], rows[r][want])


def test_topk_matches_torch_topk_on_distinct_values():
    """Pin: library routine. With all-distinct values the result is torch.topk's."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(6, 5000, generator=g)
    idx, val = oracle.topk(x.numpy(), 16)
    tv, ti = torch.topk(x, 16, dim=1, sorted=True)
    np.testing.assert_array_equal(idx, ti.numpy())
    np.testing.assert_array_equal(val, tv.numpy())


# ------------------------------------------------------------------ pair scores


def _hand_setup():
    V, d, r = 20, 4, 2
    E = np.array([[t % 3, t % 2, t % 5 - 2, 1] for t in range(V)], np.float32)
    W_A = np.array([[1, 0, 0, 0], [0, 1, 0, 0]], np.float32)
    W_B = np.array([[0, 0, 1, 0], [0, 0, 0, 1]], np.float32)
    W_H = np.zeros((r, d), np.float32)
    cand = np.stack([np.arange(16), np.arange(4, 20)])[None].astype(np.int32)   # [1,2,16]
    cval = np.stack([10.0 - np.arange(16), 20.0 - np.arange(16)])[None].astype(np.float32)
    hidden = np.ones((1, 2, d), np.float32)
    verified = np.array([7], np.int32)
    return dict(E=E, W_A=W_A, W_B=W_B, W_H=W_H, cand=cand, cval=cval, hidden=hidden,
                verified=verified)


def _select(s, **over):
    s = dict(s, **over)
    return oracle.select(s["cand"], s["cval"], s["verified"], _bf16(s["hidden"]), _bf16(s["E"]),
                         _bf16(s["W_A"]), _bf16(s["W_B"]), _bf16(s["W_H"]))


def test_select_golden_hand_case():
    """Pin: hand-computed scores (tests/golden/select_hand.json)."""
    g = _load("select_hand.json")
    S = _select(_hand_setup())
    for t, i, j, want in g["expected"]:
        assert S[0, t, i, j] == want, (t, i, j)
    assert np.all(np.isneginf(S[0, 0, 1:, :]))


def test_select_gate_closed_form():
    """Pin: closed form. With W_H row 0 = e_0 and h[0] = 2 the gate is
    (sigmoid(2), 1/2), so S = U + sigmoid(2) A_0 B_0 + A_1 B_1 / 2."""
    s = _hand_setup()
    W_H = np.zeros((2, 4), np.float32)
    W_H[0, 0] = 1.0
    hidden = np.zeros((1, 2, 4), np.float32)
    hidden[0, :, 0] = 2.0
    S = _select(s, W_H=W_H, hidden=hidden)
    sig2 = 1.0 / (1.0 + math.exp(-2.0))
    E = s["E"].astype(np.float64)
    for t in range(2):
        preds = [7] if t == 0 else list(range(16))
        for i, a in enumerate(preds):
            for j in range(16):
                b = int(s["cand"][0, t, j])
                want = float(s["cval"][0, t, j]) + sig2 * E[a, 0] * E[b, 2] + 0.5 * E[a, 1] * E[b, 3]
                assert S[0, t, i, j] == pytest.approx(want, rel=1e-12, abs=1e-12)


def test_select_zero_W_A_is_plain_logits():
    """Pin (invariant on the pages): with the bilinear term off (W_A = 0) every
    score is the candidate's own logit, U_t(b)."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(V=500, d=64, L=3, B=2)
    inp = wl.make_tail_inputs(w)
    logits = wl.make_logits(w)
    idx, val = oracle.topk(logits.numpy(), 16)
    S = oracle.select(idx, val, inp["verified"].numpy(), wl.host(inp["hidden"]), wl.host(inp["E"]),
                      np.zeros((256, 64), np.uint16), wl.host(inp["W_B"]), wl.host(inp["W_H"]))
    for t in range(3):
        rows = 1 if t == 0 else 16
        for i in range(rows):
            np.testing.assert_array_equal(S[:, t, i, :], val[:, t, :].astype(np.float64))


def test_select_sign_and_transpose_sensitivity():
    """Pin: negating W_B negates the bilinear term exactly; swapping the roles of
    W_A and W_B changes the hand-case scores (the map is not symmetric)."""
    s = _hand_setup()
    S = _select(s)
    Sneg = _select(s, W_B=-s["W_B"])
    U = np.broadcast_to(s["cval"][0][:, None, :], (2, 16, 16)).astype(np.float64)
    ok = np.isfinite(S[0])
    np.testing.assert_allclose((Sneg[0] - U)[ok], -(S[0] - U)[ok], rtol=0, atol=1e-12)
    Sswap = _select(s, W_A=s["W_B"], W_B=s["W_A"])
    assert Sswap[0, 1, 2, 0] != S[0, 1, 2, 0]


# ------------------------------------------------------------------ walk


def test_walk_greedy_hand_case():
    """Pin: hand-built score tables with a known greedy path and ties."""
    S = np.full((1, 3, 16, 16), -1.0)
    S[0, 0, 0, :] = 0.0
    S[0, 0, 0, 5] = 3.0
    S[0, 0, 0, 9] = 3.0          # tie with slot 5: the lower slot wins
    S[0, 1, 5, :] = 1.0
    S[0, 1, 5, 2] = 4.0
    S[0, 1, 9, 7] = 100.0        # a row the walk never visits
    S[0, 2, 2, 15] = 2.0
    S[0, 0, 1:, :] = -np.inf
    cand = np.arange(48, dtype=np.int32).reshape(1, 3, 16) * 10
    tok, slots, q = oracle.walk(S, cand, 0.0)
    assert slots.tolist() == [[5, 2, 15]]
    assert tok.tolist() == [[50, 180, 470]]
    assert np.all(q.sum(-1) == 1.0) and q[0, 0, 5] == 1.0


def test_walk_zero_W_A_is_per_position_top1():
    """Pin (invariant on the pages): with W_A = 0 the greedy walk is plain
    per-position top-1, i.e. DFlash without the selector."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(V=3000, d=64, L=6, B=3)
    inp = wl.make_tail_inputs(w)
    idx, val = oracle.topk(wl.make_logits(w).numpy(), 16)
    S = oracle.select(idx, val, inp["verified"].numpy(), wl.host(inp["hidden"]), wl.host(inp["E"]),
                      np.zeros((256, 64), np.uint16), wl.host(inp["W_B"]), wl.host(inp["W_H"]))
    tok, slots, _ = oracle.walk(S, idx, 0.0)
    np.testing.assert_array_equal(slots, 0)
    np.testing.assert_array_equal(tok, idx[:, :, 0])


def test_walk_tiny_temperature_equals_greedy():
    """Pin: as T -> 0 the sampling walk follows the greedy path."""
    rng = np.random.default_rng(11)
    S = rng.standard_normal((40, 5, 16, 16)) * 3.0
    S[:, 0, 1:, :] = -np.inf
    cand = rng.integers(0, 1000, size=(40, 5, 16)).astype(np.int32)
    seeds = np.arange(40, dtype=np.uint64) * 7919 + 1
    g_tok, g_slots, _ = oracle.walk(S, cand, 0.0)
    s_tok, s_slots, _ = oracle.walk(S, cand, 1e-4, seeds, cycle=3)
    np.testing.assert_array_equal(s_slots, g_slots)


def test_walk_sampling_distribution_chi_square():
    """Pin: the exact path distribution.  Over many seeds, the frequencies of the
    first two steps match prod_t softmax(S_t(prev, .) / T) (chi-square test)."""
    rng = np.random.default_rng(5)
    T = 0.8
    base = rng.standard_normal((1, 2, 16, 16)) * 1.5
    base[:, 0, 1:, :] = -np.inf
    n = 40000
    S = np.broadcast_to(base, (n, 2, 16, 16)).copy()
    cand = np.broadcast_to(np.arange(32, dtype=np.int32).reshape(1, 2, 16), (n, 2, 16)).copy()
    seeds = np.array([wl.splitmix64(i) for i in range(n)], np.uint64)
    _, slots, q = oracle.walk(S, cand, T, seeds, cycle=12345)

    def softmax(v):
        e = np.exp((v - v.max()) / T)
        return e / e.sum()

    p0 = softmax(base[0, 0, 0])
    expect = np.array([[p0[a] * softmax(base[0, 1, a])[b] for b in range(16)] for a in range(16)])
    counts = np.zeros((16, 16))
    np.add.at(counts, (slots[:, 0], slots[:, 1]), 1)
    e = expect.ravel() * n
    keep = e >= 5
    chi2 = (((counts.ravel() - e) ** 2) / e)[keep].sum() + 0.0
    dof = keep.sum() - 1
    # 99.9% quantile of chi-square via the Wilson-Hilferty approximation
    z = 3.09
    crit = dof * (1 - 2 / (9 * dof) + z * math.sqrt(2 / (9 * dof))) ** 3
    assert chi2 < crit, (chi2, crit)
    # q is the step's draft distribution
    np.testing.assert_allclose(q[0, 0], p0, rtol=1e-12)


# ------------------------------------------------------------------ conv


def _conv_case(d, L, x_prev, xs, base0, base1, Wc):
    x = _bf16(np.array(xs, np.float32).reshape(1, L, d))
    xp = _bf16(np.array(x_prev, np.float32).reshape(1, d))
    base = np.stack([base0, base1]).astype(np.float32)
    return oracle.conv2(x, xp, base, _bf16(Wc))


def test_conv_golden_hand_cases():
    """Pin: hand-computed cases (tests/golden/conv_hand.json)."""
    d = 16
    y, _ = _conv_case(d, 2, np.ones(d), [np.full(d, 2.0), np.full(d, 3.0)],
                      np.full(d, 0.5), np.full(d, 0.25), np.zeros((2, d)))
    np.testing.assert_array_equal(y[0, 0], 1.25)
    np.testing.assert_array_equal(y[0, 1], 2.0)
    d = 32
    x0 = np.full(d, 0.5)
    x0[0] = 1.0
    z = np.zeros(d)
    for row, col, val, want in [
        (0, 0, 1.0, np.concatenate([x0[:16], np.zeros(16)])),
        (1, 0, 1.0, np.concatenate([np.zeros(16), np.full(16, 0.5)])),
        (3, 5, 2.0, np.concatenate([np.zeros(16), np.full(16, 2.0)])),
    ]:
        Wc = np.zeros((4, d))
        Wc[row, col] = val
        y, _ = _conv_case(d, 1, np.full(d, 2.0), [x0], z, z, Wc)
        np.testing.assert_array_equal(y[0, 0], want)


def test_conv_identity_and_shift():
    """Pin (invariants): base [1,0] with no correction is the identity; base [0,1]
    is a pure shift whose position 0 reads the verified token's representation."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(d=64, L=5, B=3)
    c = wl.make_conv_inputs(w, 0)
    x, xp = wl.host(c["x"]), wl.host(c["x_prev"])
    Wc = np.zeros((8, 64), np.uint16)
    ones, zeros = np.ones(64, np.float32), np.zeros(64, np.float32)
    _, yb = oracle.conv2(x, xp, np.stack([ones, zeros]), Wc)
    np.testing.assert_array_equal(yb, x)
    _, yb = oracle.conv2(x, xp, np.stack([zeros, ones]), Wc)
    np.testing.assert_array_equal(yb[:, 0], xp)
    np.testing.assert_array_equal(yb[:, 1:], x[:, :-1])


def test_conv_bf16_output_is_rounded_exact_value():
    """The bf16 output is the exact value rounded once (checked with torch's
    rounding on values whose double->float step is exact)."""
    w = wl.WORKLOADS["tiny_l8_v32k"].with_(d=32, L=4, B=2)
    c = wl.make_conv_inputs(w, 1)
    y, yb = oracle.conv2(wl.host(c["x"]), wl.host(c["x_prev"]), c["base"].numpy(), wl.host(c["W_c"]))
    exact32 = y.astype(np.float32)
    same = exact32.astype(np.float64) == y
    want = torch.tensor(exact32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(yb[same], want[same])


# ------------------------------------------------------------------ shapes


def test_parameter_counts_pin_the_shape_readings():
    """Pin: the pages' parameter counts.  Selector: three 256 x d maps at d = 2560
    is 1,966,080 ~ 2.0M (Table 2).  Conv: 5 layers x 4 insertion points, each with
    a base kernel [2, d] and a correction map [2 d/16, d], is 16,486,400 ~ 16.5M."""
    w = wl.WORKLOADS["drafter4b_l16"]
    d = w.d
    selector = 3 * wl.RANK * d
    assert selector == 1_966_080 and round(selector / 1e6, 1) == 2.0
    conv_call = 2 * d + (2 * d // wl.GROUP) * d
    assert w.conv_calls == 20
    assert conv_call * w.conv_calls == 16_486_400 and round(conv_call * 20 / 1e6, 1) == 16.5
