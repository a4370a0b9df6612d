"""Pins for the oracle's block verification (lossless rejection sampling),
checked against what the mathematics fixes rather than against the oracle's own
formula:

* greedy: hand cases whose answer follows from the rule (keep the matching
  prefix, replace the first miss by the target's argmax, append the target's
  next token when everything matched);
* sampling, lossless: whatever the draft distribution q, the first emitted token
  is distributed exactly as the target's p_0 (chi-square over many seeds);
* sampling, acceptance: the first draft token is kept with probability
  sum_v min(p_0(v), q_0(v)) (binomial bound);
* sampling, bonus: with p_0 = q_0 every draft is kept and the appended token
  follows p_1.

Sources: "DFlash 2: Keep Drafting Parallel", 方法细节 > 轻量级路径选择器
("全并行打分与低延迟路径步进": lossless rejection sampling recovers the target's
distribution); "DFlash 2: The Drafter Stopped Guessing Alone", "One pass to
draft, one pass to verify"; the speculative-sampling step of Leviathan et al.
(ICML 2023) and Chen et al. (2023)."""
import numpy as np
import pytest
from scipy import stats

import oracle


def test_greedy_hand_cases():
    V, L = 12, 3
    tok = np.array([[3, 5, 7]], np.int32)
    p = np.zeros((1, L + 1, V), np.float32)
    for t in range(L):
        p[0, t, tok[0, t]] = 0.6
        p[0, t, 0] = 0.4
    p[0, L, 11] = 1.0
    n, out = oracle.verify(p, tok, greedy=True)
    assert n.tolist() == [3] and out.tolist() == [[3, 5, 7, 11]]
    # a miss at position 1: the target's argmax replaces it, the rest is dropped
    p[0, 1, 5] = 0.1
    p[0, 1, 9] = 0.5
    n, out = oracle.verify(p, tok, greedy=True)
    assert n.tolist() == [1] and out.tolist() == [[3, 9, -1, -1]]
    # ties at the maximum go to the lowest index: a draft of the higher one misses
    p[0, 1, :] = 0.0
    p[0, 1, 4] = p[0, 1, 5] = 0.5
    n, out = oracle.verify(p, tok, greedy=True)
    assert n.tolist() == [1] and out.tolist() == [[3, 4, -1, -1]]
    # a miss at position 0
    p[0, 0, 3] = 0.0
    n, out = oracle.verify(p, tok, greedy=True)
    assert n.tolist() == [0] and out.tolist() == [[0, -1, -1, -1]]


def _sampling_case(N, V, seed):
    """N sequences with one drafted position: the draft token is drawn from q_0 by
    an independent generator; candidates are 16 distinct tokens of V."""
    rng = np.random.default_rng(seed)
    p0 = rng.dirichlet(np.full(V, 0.7))
    p1 = rng.dirichlet(np.full(V, 0.7))
    cand = rng.permutation(V)[:16].astype(np.int32)
    q0 = rng.dirichlet(np.full(16, 0.7))
    slot = rng.choice(16, size=N, p=q0).astype(np.int32)
    p = np.broadcast_to(np.stack([p0, p1])[None], (N, 2, V)).astype(np.float32)
    q = np.broadcast_to(q0[None, None], (N, 1, 16)).astype(np.float32)
    ci = np.broadcast_to(cand[None, None], (N, 1, 16)).astype(np.int32)
    tokens = cand[slot][:, None].astype(np.int32)
    seeds = (np.arange(N, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15)) ^ np.uint64(seed)
    n, out = oracle.verify(p, tokens, slot[:, None], q, ci, greedy=False, seeds=seeds, cycle=7)
    return p.astype(np.float64)[0], q0.astype(np.float64), cand, n, out


@pytest.mark.parametrize("seed", [1, 2])
def test_sampling_first_token_is_distributed_as_the_target(seed):
    N, V = 200_000, 24
    p, q0, cand, n, out = _sampling_case(N, V, seed)
    counts = np.bincount(out[:, 0], minlength=V)
    expected = p[0] * N
    keep = expected > 5
    chi2 = (((counts - expected) ** 2) / np.maximum(expected, 1e-12))[keep].sum()
    dof = keep.sum() - 1
    assert chi2 < stats.chi2.ppf(1 - 1e-4, dof), (chi2, dof)


def test_sampling_acceptance_rate_is_the_overlap():
    N, V = 200_000, 24
    p, q0, cand, n, out = _sampling_case(N, V, 3)
    qv = np.zeros(V)
    qv[cand] = q0
    rate = np.minimum(p[0], qv).sum()
    acc = (n == 1).mean()
    sd = np.sqrt(rate * (1 - rate) / N)
    assert abs(acc - rate) < 5 * sd, (acc, rate)


def test_sampling_bonus_follows_the_next_row_when_all_accepted():
    N, V = 100_000, 20
    rng = np.random.default_rng(5)
    cand = rng.permutation(V)[:16].astype(np.int32)
    q0 = rng.dirichlet(np.full(16, 1.0))
    p0 = np.zeros(V)
    p0[cand] = q0                      # p_0 = q_0: every draft must be kept
    p1 = rng.dirichlet(np.full(V, 1.0))
    slot = rng.choice(16, size=N, p=q0).astype(np.int32)
    p = np.broadcast_to(np.stack([p0, p1])[None], (N, 2, V)).astype(np.float32)
    q = np.broadcast_to(q0[None, None], (N, 1, 16)).astype(np.float32)
    ci = np.broadcast_to(cand[None, None], (N, 1, 16)).astype(np.int32)
    tokens = cand[slot][:, None].astype(np.int32)
    seeds = np.arange(N, dtype=np.uint64) + np.uint64(12345)
    n, out = oracle.verify(p, tokens, slot[:, None], q, ci, greedy=False, seeds=seeds, cycle=0)
    # float32 rounding of p_0 vs q_0 may reject a handful; those are still valid draws
    assert (n == 1).mean() > 0.999
    counts = np.bincount(out[n == 1, 1], minlength=V)
    expected = p1 * (n == 1).sum()
    keep = expected > 5
    chi2 = (((counts - expected) ** 2) / expected)[keep].sum()
    assert chi2 < stats.chi2.ppf(1 - 1e-4, keep.sum() - 1)


def test_verify_uniforms_use_their_own_counter_word():
    # the acceptance draws are Philox4x32-10 with counter word 3 = 1: distinct
    # from the walk's draws (word 3 = 0) at the same (seed, cycle, t)
    u = oracle.verify_uniforms(42, 9, 3)
    w = oracle.walk_uniform(42, 9, 3)
    ctr = np.array([3, 9, 0, 1], np.uint32)
    key = np.array([42, 0], np.uint32)
    ref = oracle.philox4x32_10(ctr, key)
    assert u[0] == (int(ref[0]) >> 8) * 2.0 ** -24 and u[1] == (int(ref[1]) >> 8) * 2.0 ** -24
    assert u[0] != w
