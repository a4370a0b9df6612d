"""GPU parity of the walk, fed the same float32 score tables as the oracle.

Greedy: bit-exact (the same fp32 inputs decide the same argmax).  Sampling:
the GPU's Philox4x32-10 draws and decisions must match the oracle's except at
steps where u*Z falls within 1e-4*Z of a cumulative boundary (the two sides sum
in different precisions); those are counted and reported."""
import numpy as np
import pytest
import torch

import draft_selection_gb300 as dfl2
from draft_selection_gb300 import workloads as wl
import oracle
from _parity import replay_walk, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from draft_selection_gb300 import build
    build.build()
    dfl2.load()


def gpu_walk(S: np.ndarray, cand: np.ndarray, T: float, seeds=None, cycle=0):
    B, L = S.shape[:2]
    Sd = torch.from_numpy(S.astype(np.float32)).cuda()
    cd = torch.from_numpy(cand.astype(np.int32)).cuda()
    tok = torch.empty(B, L, dtype=torch.int32, device="cuda")
    slots = torch.empty(B, L, dtype=torch.int32, device="cuda")
    q = torch.empty(B, L, 16, dtype=torch.float32, device="cuda")
    sd = None if seeds is None else torch.from_numpy(seeds.view(np.int64)).cuda()
    dfl2.dfl2_walk(Sd, cd, T, sd, cycle, tok, slots, q)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), slots.cpu().numpy(), q.cpu().numpy()


def random_tables(B, L, scale, seed, ties=False):
    rng = np.random.default_rng(seed)
    S = rng.standard_normal((B, L, 16, 16)) * scale
    if ties:
        S = np.round(S * 2) / 2
    S = S.astype(np.float32).astype(np.float64)
    S[:, 0, 1:, :] = -np.inf
    cand = rng.integers(0, 151936, size=(B, L, 16)).astype(np.int32)
    return S, cand


@pytest.mark.parametrize("B,L,ties", [(1, 16, False), (64, 16, False), (256, 16, True),
                                      (7, 1, True), (3, 40, False)])
def test_greedy_bit_exact(B, L, ties):
    S, cand = random_tables(B, L, 3.0, B * 100 + L, ties)
    tok, slots, q = gpu_walk(S, cand, 0.0)
    rt, rs, rq = oracle.walk(S, cand, 0.0)
    np.testing.assert_array_equal(slots, rs)
    np.testing.assert_array_equal(tok, rt)
    np.testing.assert_array_equal(q, rq.astype(np.float32))


@pytest.mark.parametrize("B,L,T,cycle", [(1, 16, 1.0, 0), (64, 16, 1.0, 7),
                                         (256, 16, 0.7, 2**40 + 3), (5, 33, 0.25, 99)])
def test_sampling_matches_oracle(B, L, T, cycle):
    S, cand = random_tables(B, L, 2.0, B + L, False)
    w = wl.WORKLOADS["serving_b64"].with_(B=B)
    seeds = wl.philox_seeds(w, salt=L)
    tok, slots, q = gpu_walk(S, cand, T, seeds, cycle)
    allowed = replay_walk(S, slots, T, seeds, cycle, what=f"walk B={B} L={L} T={T}")
    assert allowed <= max(1, B * L // 1000)
    # where the paths agree, the draft distributions agree
    rt, rs, rq = oracle.walk(S, cand, T, seeds, cycle)
    same = np.all(slots == rs, axis=1)
    np.testing.assert_allclose(q[same], rq[same], rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(tok, np.take_along_axis(cand, slots[..., None], 2)[..., 0])


def test_sampling_reveals_the_uniform_bits():
    """Two-way splits sweep the boundary: with p = (a, 1-a) the choice is slot 0
    exactly when u < a, so many steps pin the top bits of every Philox draw."""
    B, L = 512, 16
    rng = np.random.default_rng(9)
    a = rng.uniform(0.05, 0.95, size=(B, L))
    S = np.full((B, L, 16, 16), -np.inf)
    T = 1.0
    S[:, :, :, 0] = np.log(a)[:, :, None]
    S[:, :, :, 1] = np.log1p(-a)[:, :, None]
    S = S.astype(np.float32).astype(np.float64)
    S[:, 0, 1:, :] = -np.inf
    cand = np.arange(B * L * 16, dtype=np.int32).reshape(B, L, 16)
    seeds = np.array([wl.splitmix64(1 << 20 | b) for b in range(B)], np.uint64)
    _, slots, _ = gpu_walk(S, cand, T, seeds, cycle=31337)
    allowed = replay_walk(S, slots, T, seeds, 31337, what="two-way splits")
    assert allowed <= 2


def test_greedy_from_real_scores_zero_W_A():
    """With W_A = 0 the GPU walk is plain per-position top-1 (slot 0 everywhere)."""
    w = wl.WORKLOADS["tiny_l8_v32k"]
    idx, val = oracle.topk(wl.host(wl.make_logits(w, "cpu")), 16)
    S = np.broadcast_to(val[:, :, None, :].astype(np.float64), (w.B, w.L, 16, 16)).copy()
    S[:, 0, 1:, :] = -np.inf
    tok, slots, _ = gpu_walk(S, idx, 0.0)
    np.testing.assert_array_equal(slots, 0)
    np.testing.assert_array_equal(tok, idx[:, :, 0])
