"""Helpers shared by the GPU parity tests: tolerances, the step-wise walk replay
and a place to report the walk steps that were allowed to differ.

Tolerances (see the test files for where each applies):
  * top-16 indices and values: bit-exact (values compared numerically, so a
    zero logit of either sign matches).
  * pair scores: |gpu - oracle| <= 1e-3 * max(|oracle|, 1)  (fp32 accumulation).
  * greedy walk: the GPU's choice must equal the oracle's choice given the
    GPU's own previous choice, unless the GPU's slot scores within
    1e-3 * |S_max| of the row's maximum (a near tie); such steps are counted
    and reported.
  * sampling walk: likewise, unless every cumulative boundary between the two
    choices lies within 1e-4 * Z of u*Z.
  * conv: |gpu - oracle_bf16| <= max(2e-2, 1 bf16 ulp of the oracle value).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

SCORE_RTOL = 1e-3
GREEDY_MARGIN_REL = 1e-3
SAMPLE_BOUNDARY_REL = 1e-4
CONV_ATOL = 2e-2

REPORT = []


def report(**kw):
    REPORT.append(kw)


def dump_report(path):
    with open(path, "w") as f:
        for r in REPORT:
            f.write(json.dumps(r) + "\n")


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(gpu), inf) and np.all(np.sign(gpu[inf]) == np.sign(ref[inf])), \
        f"{what}: -inf pattern differs"
    fin = ~inf
    err = np.abs(gpu[fin] - ref[fin])
    tol = SCORE_RTOL * np.maximum(np.abs(ref[fin]), 1.0)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} scores outside 1e-3*max(|ref|,1); "
                           f"worst err {err.max():.3e}")
    return float((err / tol).max()) if err.size else 0.0


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    a = np.where(a < 2.0**-126, 2.0**-126, a)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 7)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def assert_conv_close(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, what=""):
    g = bf16_bits_to_f64(y_gpu_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    err = np.abs(g - r)
    tol = np.maximum(CONV_ATOL, bf16_ulp(r))
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {err.size} outside tolerance; worst {err.max()}"
    exact = float(np.mean(y_gpu_bits == y_ref_bits))
    return exact


def replay_walk(S_ref: np.ndarray, gpu_slots: np.ndarray, T: float, seeds=None, cycle: int = 0,
                what=""):
    """Checks each GPU walk step against the oracle's choice given the GPU's
    previous choice.  Returns the number of steps allowed to differ."""
    B, L = gpu_slots.shape
    allowed = 0
    for b in range(B):
        for t in range(L):
            prev = 0 if t == 0 else int(gpu_slots[b, t - 1])
            row = np.asarray(S_ref[b, t, prev], np.float64)
            got = int(gpu_slots[b, t])
            if T == 0.0:
                want = int(np.argmax(row))  # first maximum = lowest slot
                if got == want:
                    continue
                # only a slot within the near-tie margin of the maximum is excused
                ok = row[want] - row[got] <= GREEDY_MARGIN_REL * abs(row[want])
            else:
                m = row.max()
                p = np.exp((row - m) / T)
                Z = p.sum()
                cum = np.cumsum(p)
                uZ = oracle.walk_uniform(int(seeds[b]), cycle, t) * Z
                hits = np.nonzero(uZ < cum)[0]
                want = int(hits[0]) if hits.size else int(np.nonzero(p > 0)[0][-1])
                if got == want:
                    continue
                # every cumulative boundary between the two picks must lie within
                # the tolerance of u*Z (the boundaries rise, so the two extremes do)
                lo, hi = min(got, want), max(got, want)
                tol = SAMPLE_BOUNDARY_REL * Z
                ok = abs(uZ - cum[lo]) < tol and abs(uZ - cum[hi - 1]) < tol
            assert ok, f"{what}: walk step (b={b}, t={t}) chose slot {got}, oracle {want}"
            allowed += 1
    report(kind="walk", what=what, T=T, steps=B * L, allowed_mismatches=allowed)
    return allowed


def walk_tokens_from_slots(cand_idx: np.ndarray, slots: np.ndarray) -> np.ndarray:
    B, L = slots.shape
    return np.take_along_axis(cand_idx, slots[:, :, None].astype(np.int64), axis=2)[:, :, 0]


def cuda_available() -> bool:
    return torch.cuda.is_available()
