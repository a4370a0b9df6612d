"""dfl2 oracle: TEST INFRASTRUCTURE, not part of the product.

A plain double-precision CPU restatement of the DFlash 2 draft tail (top-16,
pair scores, walk, two-tap dynamic conv), written in C (``dfl2_oracle.c``) and
wrapped here with ctypes.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library in ``draft_selection_gb300``; the two meet only through
the seeded inputs of ``draft_selection_gb300.workloads``.

Every function cites the passage it restates in ``dfl2_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dfl2_oracle.c")
_HDR = os.path.join(_HERE, "dfl2_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11 + OpenMP) if it is missing or stale."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if fresh and not force:
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I, D, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_uint64
        L.oracle_set_threads.argtypes = [I]
        L.oracle_get_threads.restype = I
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_walk_uniform.argtypes = [U64, U64, I]
        L.oracle_walk_uniform.restype = D
        L.oracle_topk.argtypes = [P, I, I, I, I, I, P, P]
        L.oracle_topk.restype = I
        L.oracle_proj_token.argtypes = [P, P, I, I, ctypes.c_int32, P]
        L.oracle_gate.argtypes = [P, P, I, I, P]
        L.oracle_select.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P]
        L.oracle_select.restype = I
        L.oracle_walk.argtypes = [P, P, I, I, D, P, U64, P, P, P]
        L.oracle_walk.restype = I
        L.oracle_conv2.argtypes = [P, P, P, P, I, I, I, P, P]
        L.oracle_conv2.restype = I
        L.oracle_verify_uniforms.argtypes = [U64, U64, I, P]
        L.oracle_verify.argtypes = [P, P, P, P, P, I, I, I, I, P, U64, P, P]
        L.oracle_verify.restype = I
        L.oracle_lmhead_topk.argtypes = [P, P, I, I, I, I, P, P]
        L.oracle_lmhead_topk.restype = I
        L.oracle_round_bf16.argtypes = [D]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def walk_uniform(seed: int, cycle: int, t: int) -> float:
    return float(lib().oracle_walk_uniform(seed, cycle, t))


def round_bf16(v: float) -> int:
    return int(lib().oracle_round_bf16(float(v)))


def topk(logits: np.ndarray, k: int = 16):
    """logits [..., V] as float32 or as bf16 bit patterns (uint16). Returns (idx int32, val float32)."""
    if logits.dtype == np.uint16:
        dt = BF16
    elif logits.dtype == np.float32:
        dt = F32
    else:
        raise TypeError("oracle.topk takes float32 or bf16 bit patterns (uint16)")
    lg = _c(logits, logits.dtype)
    V = lg.shape[-1]
    rows = lg.size // V
    idx = np.zeros((rows, k), np.int32)
    val = np.zeros((rows, k), np.float32)
    rc = lib().oracle_topk(_ptr(lg), dt, 1, rows, V, k, _ptr(idx), _ptr(val))
    if rc != 0:
        raise ValueError("oracle_topk rejected its arguments")
    shape = lg.shape[:-1] + (k,)
    return idx.reshape(shape), val.reshape(shape)


def lmhead_topk(hidden: np.ndarray, W_lm: np.ndarray, k: int = 16):
    """hidden [..., d] and W_lm [V, d] as bf16 bit patterns (uint16).

    Returns (idx int32 [..., k], val float64 [..., k]): the k largest exact
    logits hidden . W_lm[v] per row, value descending then index ascending.
    """
    h = _c(hidden, np.uint16)
    W = _c(W_lm, np.uint16)
    V, d = W.shape
    if h.shape[-1] != d:
        raise ValueError("hidden and W_lm disagree on d")
    R = h.size // d
    idx = np.zeros((R, k), np.int32)
    val = np.zeros((R, k), np.float64)
    if lib().oracle_lmhead_topk(_ptr(h), _ptr(W), R, V, d, k, _ptr(idx), _ptr(val)) != 0:
        raise ValueError("oracle_lmhead_topk rejected its arguments")
    shape = h.shape[:-1] + (k,)
    return idx.reshape(shape), val.reshape(shape)


def proj_token(E: np.ndarray, W: np.ndarray, tok: int) -> np.ndarray:
    E = _c(E, np.uint16)
    W = _c(W, np.uint16)
    out = np.zeros(W.shape[0], np.float64)
    lib().oracle_proj_token(_ptr(E), _ptr(W), E.shape[1], W.shape[0], int(tok), _ptr(out))
    return out


def gate(W_H: np.ndarray, h: np.ndarray) -> np.ndarray:
    W_H = _c(W_H, np.uint16)
    h = _c(h, np.uint16)
    out = np.zeros(W_H.shape[0], np.float64)
    lib().oracle_gate(_ptr(W_H), _ptr(h), W_H.shape[1], W_H.shape[0], _ptr(out))
    return out


def select(cand_idx, cand_val, verified, hidden, E, W_A, W_B, W_H) -> np.ndarray:
    """Pair scores [B,L,16,16] in float64.  bf16 tensors are passed as uint16 bit patterns."""
    cand_idx = _c(cand_idx, np.int32)
    cand_val = _c(cand_val, np.float32)
    verified = _c(verified, np.int32)
    hidden = _c(hidden, np.uint16)
    E = _c(E, np.uint16)
    W_A, W_B, W_H = (_c(w, np.uint16) for w in (W_A, W_B, W_H))
    B, L, d = hidden.shape
    V = E.shape[0]
    r = W_A.shape[0]
    assert cand_idx.shape == (B, L, 16) and cand_val.shape == (B, L, 16)
    out = np.zeros((B, L, 16, 16), np.float64)
    rc = lib().oracle_select(_ptr(cand_idx), _ptr(cand_val), _ptr(verified), _ptr(hidden),
                             _ptr(E), _ptr(W_A), _ptr(W_B), _ptr(W_H), B, L, V, d, r, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_select rejected its arguments")
    return out


def walk(scores, cand_idx, T: float, seeds=None, cycle: int = 0):
    """Returns (tokens [B,L] int32, slots [B,L] int32, q [B,L,16] float64)."""
    scores = _c(scores, np.float64)
    cand_idx = _c(cand_idx, np.int32)
    B, L = scores.shape[:2]
    sd = None if seeds is None else _c(seeds, np.uint64)
    tokens = np.zeros((B, L), np.int32)
    slots = np.zeros((B, L), np.int32)
    q = np.zeros((B, L, 16), np.float64)
    rc = lib().oracle_walk(_ptr(scores), _ptr(cand_idx), B, L, float(T), _ptr(sd),
                           int(cycle), _ptr(tokens), _ptr(slots), _ptr(q))
    if rc != 0:
        raise ValueError("oracle_walk rejected its arguments")
    return tokens, slots, q


def conv2(x, x_prev, base, W_c):
    """Returns (y_exact float64 [B,L,d], y_bf16 uint16 bit patterns [B,L,d])."""
    x = _c(x, np.uint16)
    x_prev = _c(x_prev, np.uint16)
    base = _c(base, np.float32)
    W_c = _c(W_c, np.uint16)
    B, L, d = x.shape
    y = np.zeros((B, L, d), np.float64)
    yb = np.zeros((B, L, d), np.uint16)
    rc = lib().oracle_conv2(_ptr(x), _ptr(x_prev), _ptr(base), _ptr(W_c), B, L, d,
                            _ptr(y), _ptr(yb))
    if rc != 0:
        raise ValueError("oracle_conv2 rejected its arguments")
    return y, yb


def verify_uniforms(seed: int, cycle: int, t: int) -> tuple[float, float]:
    u = np.zeros(2, np.float64)
    lib().oracle_verify_uniforms(seed, cycle, t, _ptr(u))
    return float(u[0]), float(u[1])


def verify(p, tokens, slots=None, q=None, cand_idx=None, greedy: bool = True, seeds=None,
           cycle: int = 0):
    """p [B, L+1, V] float32 target distributions.  Returns (n_accepted [B] int32,
    out [B, L+1] int32)."""
    p = _c(p, np.float32)
    tokens = _c(tokens, np.int32)
    B, L = tokens.shape
    V = p.shape[-1]
    if p.shape != (B, L + 1, V):
        raise ValueError("p must be [B, L+1, V]")
    sl = None if slots is None else _c(slots, np.int32)
    qq = None if q is None else _c(q, np.float32)
    ci = None if cand_idx is None else _c(cand_idx, np.int32)
    sd = None if seeds is None else _c(seeds, np.uint64)
    n = np.zeros(B, np.int32)
    out = np.zeros((B, L + 1), np.int32)
    rc = lib().oracle_verify(_ptr(p), _ptr(tokens), _ptr(sl), _ptr(qq), _ptr(ci), B, L, V,
                             int(bool(greedy)), _ptr(sd), int(cycle), _ptr(n), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    return n, out
