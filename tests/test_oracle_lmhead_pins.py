"""Pins for the oracle's LM head + top-16 (the logits U_t(.) the selector's
"Top-16" step reads, "DFlash 2: Keep Drafting Parallel", 方法细节 > 轻量级路径选择器,
computed from the drafter's last hidden state instead of being given).

Each pin fixes the answer by something other than the oracle's own loop:

* brute force in pure Python on tiny integer-valued inputs (exact arithmetic,
  heavy ties, so the index-ascending tie rule is exercised);
* a one-hot hidden state reads one column of W_lm, whose order is known by
  construction;
* W_lm = 0: every logit ties at zero, so the answer is indices 0..15;
* relabelling the vocabulary (a row permutation of W_lm) relabels the indices,
  and scaling h by a power of two scales the values exactly.
"""
import numpy as np
import pytest

import oracle


def bf16_bits(a) -> np.ndarray:
    """Bit patterns of values that bf16 represents exactly (asserted)."""
    f = np.asarray(a, np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f), "value not exact in bf16"
    return bits


def brute_force(h_int, W_int, k=16):
    out_i, out_v = [], []
    for row in h_int.tolist():
        logits = [sum(a * b for a, b in zip(row, w)) for w in W_int.tolist()]
        order = sorted(range(len(logits)), key=lambda v: (-logits[v], v))[:k]
        out_i.append(order)
        out_v.append([logits[v] for v in order])
    return np.array(out_i), np.array(out_v, np.float64)


def test_brute_force_integer_ties():
    rng = np.random.default_rng(7)
    R, V, d = 3, 37, 8
    h = rng.integers(-3, 4, (R, d))
    W = rng.integers(-3, 4, (V, d))
    idx, val = oracle.lmhead_topk(bf16_bits(h), bf16_bits(W))
    ei, ev = brute_force(h, W)
    assert np.array_equal(idx, ei)
    assert np.array_equal(val, ev)
    # the inputs really tie: some logit value repeats inside the top 16
    assert any(len(set(r)) < 16 for r in ev.tolist())


def test_brute_force_fractional():
    # quarters and eighths are exact in bf16 and in double: the sum is exact
    rng = np.random.default_rng(11)
    R, V, d = 2, 29, 12
    h = rng.integers(-16, 17, (R, d)) / 8.0
    W = rng.integers(-16, 17, (V, d)) / 4.0
    idx, val = oracle.lmhead_topk(bf16_bits(h), bf16_bits(W))
    ei, ev = brute_force(h, W)
    assert np.array_equal(idx, ei)
    assert np.array_equal(val, ev)


def test_one_hot_reads_a_column():
    V, d, c = 100, 16, 5
    perm = np.random.default_rng(3).permutation(V)
    W = np.zeros((V, d))
    W[:, c] = perm / 4.0            # distinct, exact in bf16 (perm < 256)
    W[:, c + 1] = 1.0               # a column the one-hot state must ignore
    h = np.zeros((1, d))
    h[0, c] = 2.0
    idx, val = oracle.lmhead_topk(bf16_bits(h), bf16_bits(W))
    want = np.argsort(-perm)[:16]   # the 16 largest perm values, largest first
    assert idx[0].tolist() == want.tolist()
    assert val[0].tolist() == (2.0 * perm[want] / 4.0).tolist()


def test_all_ties_give_lowest_indices():
    V, d = 40, 8
    h = bf16_bits(np.ones((2, d)))
    W = bf16_bits(np.zeros((V, d)))
    idx, val = oracle.lmhead_topk(h, W)
    assert idx.tolist() == [list(range(16))] * 2
    assert np.all(val == 0.0)


def test_relabel_and_scale():
    rng = np.random.default_rng(5)
    R, V, d = 2, 64, 16
    h = rng.integers(-8, 9, (R, d)) / 4.0
    W = rng.integers(-8, 9, (V, d)) / 8.0
    idx, val = oracle.lmhead_topk(bf16_bits(h), bf16_bits(W))
    perm = rng.permutation(V)       # new row j holds old row perm[j]
    idx_p, val_p = oracle.lmhead_topk(bf16_bits(h), bf16_bits(W[perm]))
    inv = np.argsort(perm)
    # same values; the relabelled indices name the same old rows wherever the
    # values are distinct (ties may reorder under the new labels)
    assert np.array_equal(val_p, val)
    for r in range(R):
        distinct = [j for j in range(16) if list(val[r]).count(val[r, j]) == 1]
        assert [perm[idx_p[r, j]] for j in distinct] == [idx[r, j] for j in distinct]
    assert np.all(inv[perm] == np.arange(V))
    idx2, val2 = oracle.lmhead_topk(bf16_bits(4.0 * h), bf16_bits(W))
    assert np.array_equal(idx2, idx)
    assert np.array_equal(val2, 4.0 * val)


def test_rejects_bad_arguments():
    h = bf16_bits(np.ones((1, 8)))
    with pytest.raises(ValueError):
        oracle.lmhead_topk(h, bf16_bits(np.ones((8, 8))))   # V < 16
    with pytest.raises(ValueError):
        oracle.lmhead_topk(h, bf16_bits(np.ones((20, 4))))  # d mismatch
