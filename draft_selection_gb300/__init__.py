"""dfl2: the DFlash 2 draft tail on one GB300, through its C ABI (include/dfl2.h).

This module is argument marshalling only: every function has the name of the C
entry point it calls, takes torch tensors (or raw integer addresses), passes
their device pointers, sizes and the current CUDA stream to libdfl2.so, and
raises Dfl2Error on a non-zero status.  Every step of the path runs in the
library's CUDA kernels; there is no other implementation to fall back to, so a
missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

STATUS = {0: "DFL2_OK", 1: "DFL2_ERR_INVALID_ARG", 2: "DFL2_ERR_UNSUPPORTED",
          3: "DFL2_ERR_WORKSPACE", 4: "DFL2_ERR_CUDA", 5: "DFL2_ERR_TIMEOUT"}
DFL2_F32, DFL2_BF16 = 0, 1
NCAND, RANK = 16, 256

_lib = None


class Dfl2Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


def lib_path() -> str:
    return _build.LIB


def load():
    """Loads libdfl2.so (built in-tree by draft_selection_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with draft_selection_gb300.build.build() "
                           "(nvcc, sm_103a); dfl2 has no other implementation")
    L = ctypes.CDLL(path)
    P, I, F, U64, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64,
                        ctypes.c_size_t)
    L.dfl2_version.restype = ctypes.c_char_p
    L.dfl2_last_error.argtypes = [ctypes.c_char_p, SZ]
    L.dfl2_last_error.restype = SZ
    L.dfl2_launch_count.restype = U64
    L.dfl2_workspace_init.argtypes = [P, SZ, P]
    L.dfl2_set_projection_engine.argtypes = [I]
    L.dfl2_set_projection_engine.restype = I
    L.dfl2_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), I]
    L.dfl2_topk_workspace_size.argtypes = [I, I, I]
    L.dfl2_topk_workspace_size.restype = SZ
    L.dfl2_topk.argtypes = [P, I, I, I, I, I, P, P, P, SZ, P]
    L.dfl2_topk_noalloc.argtypes = [P, I, I, I, I, I, P, P, P]
    L.dfl2_topk_noalloc.restype = I
    L.dfl2_lmhead_topk_workspace_size.argtypes = [I, I, I, I]
    L.dfl2_lmhead_topk_workspace_size.restype = SZ
    L.dfl2_lmhead_topk.argtypes = [P, P, I, I, I, I, I, P, P, P, SZ, P]
    L.dfl2_select_workspace_size.argtypes = [I, I, I]
    L.dfl2_select_workspace_size.restype = SZ
    L.dfl2_select.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, SZ, P]
    L.dfl2_walk.argtypes = [P, P, I, I, F, P, U64, P, P, P, P]
    L.dfl2_conv2.argtypes = [P, P, P, P, I, I, I, P, P]
    L.dfl2_conv2_workspace_size.argtypes = [I, I, I]
    L.dfl2_conv2_workspace_size.restype = SZ
    L.dfl2_conv2_ws.argtypes = [P, P, P, P, I, I, I, P, P, SZ, P]
    L.dfl2_tail_workspace_size.argtypes = [I, I, I, I]
    L.dfl2_tail_workspace_size.restype = SZ
    L.dfl2_tail.argtypes = [P, I, P, P, P, P, P, P, I, I, I, I, F, P, U64, P, P, P, P, P, P,
                            P, SZ, P]
    L.dfl2_tables_bytes.argtypes = [I]
    L.dfl2_tables_bytes.restype = SZ
    L.dfl2_tables_build.argtypes = [P, P, P, I, I, P, P, P]
    L.dfl2_select_tables.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, SZ, P]
    L.dfl2_tail_tables.argtypes = [P, I, P, P, P, P, P, I, I, I, I, F, P, U64, P, P, P, P, P, P,
                                   P, SZ, P]
    L.dfl2_verify_workspace_size.argtypes = [I, I, I]
    L.dfl2_verify_workspace_size.restype = SZ
    L.dfl2_verify.argtypes = [P, P, P, P, P, I, I, I, I, P, U64, P, P, P, SZ, P]
    for name in ("dfl2_workspace_init", "dfl2_device_error", "dfl2_topk", "dfl2_select",
                 "dfl2_walk", "dfl2_conv2", "dfl2_conv2_ws", "dfl2_tail", "dfl2_verify", "dfl2_tables_build",
                 "dfl2_select_tables", "dfl2_tail_tables"):
        getattr(L, name).restype = I
    _lib = L
    return _lib


def dfl2_last_error() -> str:
    buf = ctypes.create_string_buffer(1024)
    load().dfl2_last_error(buf, len(buf))
    return buf.value.decode(errors="replace")


def _check(status: int) -> None:
    if status != 0:
        raise Dfl2Error(status, dfl2_last_error())


def _ptr(t):
    """A tensor's device address, an int address as is, None as NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DFL2_F32
    if t.dtype == torch.bfloat16:
        return DFL2_BF16
    raise TypeError(f"logits must be float32 or bfloat16, not {t.dtype}")


def dfl2_version() -> str:
    return load().dfl2_version().decode()


def dfl2_launch_count() -> int:
    return int(load().dfl2_launch_count())


PROJ_TENSOR, PROJ_WARP = 0, 1


def dfl2_set_projection_engine(engine: int) -> int:
    """Engine of the split-K projection GEMM (PROJ_TENSOR or PROJ_WARP); returns the previous one."""
    prev = int(load().dfl2_set_projection_engine(int(engine)))
    if prev < 0:
        raise ValueError(f"unknown projection engine {engine}")
    return prev


def dfl2_workspace_init(ws, nbytes: int | None = None, stream=None) -> None:
    n = ws.numel() * ws.element_size() if nbytes is None else nbytes
    _check(load().dfl2_workspace_init(_ptr(ws), n, _stream(stream)))


def dfl2_device_error(clear: bool = True) -> int:
    code = ctypes.c_uint32(0)
    _check(load().dfl2_device_error(ctypes.byref(code), int(clear)))
    return int(code.value)


def dfl2_topk_workspace_size(B: int, L: int, V: int) -> int:
    return int(load().dfl2_topk_workspace_size(B, L, V))


def dfl2_lmhead_topk_workspace_size(B: int, L: int, V: int, d: int) -> int:
    return int(load().dfl2_lmhead_topk_workspace_size(B, L, V, d))


def dfl2_select_workspace_size(B: int, L: int, d: int) -> int:
    return int(load().dfl2_select_workspace_size(B, L, d))


def dfl2_tail_workspace_size(B: int, L: int, V: int, d: int) -> int:
    return int(load().dfl2_tail_workspace_size(B, L, V, d))


def workspace(nbytes: int, device="cuda"):
    """A zero-filled device workspace of nbytes (torch allocation; plumbing only)."""
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def dfl2_topk(logits, cand_idx, cand_val, ws, k: int = NCAND, stream=None, *, dims=None,
              dtype=None, ws_bytes=None) -> None:
    """logits [B,L,V] float32/bf16 -> cand_idx int32 [B,L,16], cand_val float32 [B,L,16]."""
    B, L, V = dims if dims is not None else logits.shape
    dt = dtype if dtype is not None else _dtype_code(logits)
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_topk(_ptr(logits), dt, B, L, V, k, _ptr(cand_idx), _ptr(cand_val),
                            _ptr(ws), wb, _stream(stream)))


def dfl2_lmhead_topk(hidden, W_lm, cand_idx, cand_val, ws, k: int = NCAND, stream=None, *,
                     dims=None, ws_bytes=None) -> None:
    """hidden bf16 [B,L,d], W_lm bf16 [V,d] -> the top 16 of hidden . W_lm^T per row:
    cand_idx int32 [B,L,16], cand_val float32 [B,L,16]."""
    if dims is not None:
        B, L, V, d = dims
    else:
        B, L, d = hidden.shape
        V = W_lm.shape[0]
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_lmhead_topk(_ptr(hidden), _ptr(W_lm), B, L, V, d, k, _ptr(cand_idx),
                                   _ptr(cand_val), _ptr(ws), wb, _stream(stream)))


def dfl2_topk_noalloc(logits, cand_idx, cand_val, k: int = NCAND, stream=None, *, dims=None,
                      dtype=None) -> None:
    """dfl2_topk without a workspace, for callers that cannot allocate device
    memory: the library's own fixed scratch array is used instead."""
    B, L, V = dims if dims is not None else logits.shape
    dt = dtype if dtype is not None else _dtype_code(logits)
    _check(load().dfl2_topk_noalloc(_ptr(logits), dt, B, L, V, k, _ptr(cand_idx), _ptr(cand_val),
                                    _stream(stream)))


def dfl2_select(cand_idx, cand_val, verified_tok, hidden, E, W_A, W_B, W_H, scores, ws,
                r: int = RANK, stream=None, *, dims=None, ws_bytes=None) -> None:
    """Pair scores [B,L,16,16] float32 from the candidates, hidden [B,L,d] and E [V,d]."""
    if dims is not None:
        B, L, V, d = dims
    else:
        B, L, d = hidden.shape
        V = E.shape[0]
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_select(_ptr(cand_idx), _ptr(cand_val), _ptr(verified_tok), _ptr(hidden),
                              _ptr(E), _ptr(W_A), _ptr(W_B), _ptr(W_H), B, L, V, d, r,
                              _ptr(scores), _ptr(ws), wb, _stream(stream)))


def dfl2_walk(scores, cand_idx, temperature: float, seeds, cycle_offset: int, tokens,
              slots=None, q=None, stream=None, *, dims=None) -> None:
    """Greedy (T = 0) or Philox-sampled (T > 0) walk over scores [B,L,16,16]."""
    B, L = dims if dims is not None else scores.shape[:2]
    _check(load().dfl2_walk(_ptr(scores), _ptr(cand_idx), B, L, float(temperature), _ptr(seeds),
                            int(cycle_offset), _ptr(tokens), _ptr(slots), _ptr(q),
                            _stream(stream)))


def dfl2_verify_workspace_size(B: int, L: int, V: int) -> int:
    return int(load().dfl2_verify_workspace_size(B, L, V))


def dfl2_verify(p, tokens, n_accepted, out_tokens, *, greedy: bool, slots=None, q=None,
                cand_idx=None, seeds=None, cycle_offset: int = 0, ws=None, ws_bytes=None,
                stream=None, dims=None) -> None:
    """Verification of drafted tokens [B,L] against target probabilities p [B,L+1,V]:
    n_accepted [B] and out_tokens [B,L+1] (kept tokens, then the emitted token, then -1)."""
    B, L1, V = dims if dims is not None else p.shape
    L = L1 - 1
    wb = ws_bytes if ws_bytes is not None else (_nbytes(ws) if ws is not None else 0)
    _check(load().dfl2_verify(_ptr(p), _ptr(tokens), _ptr(slots), _ptr(q), _ptr(cand_idx), B, L,
                              V, int(bool(greedy)), _ptr(seeds), int(cycle_offset),
                              _ptr(n_accepted), _ptr(out_tokens), _ptr(ws), wb, _stream(stream)))


def dfl2_conv2(x, x_prev, base, W_c, y, stream=None, *, dims=None) -> None:
    """y [B,L,d] bf16 = two-tap dynamic conv of x with x_prev as position -1."""
    B, L, d = dims if dims is not None else x.shape
    _check(load().dfl2_conv2(_ptr(x), _ptr(x_prev), _ptr(base), _ptr(W_c), B, L, d, _ptr(y),
                             _stream(stream)))


def dfl2_conv2_workspace_size(B: int, L: int, d: int) -> int:
    return int(load().dfl2_conv2_workspace_size(B, L, d))


def dfl2_conv2_ws(x, x_prev, base, W_c, y, ws, stream=None, *, dims=None, ws_bytes=None) -> None:
    """dfl2_conv2 with a workspace of dfl2_conv2_workspace_size bytes (ws may be
    None when that is 0): the split-K kernel for many positions."""
    B, L, d = dims if dims is not None else x.shape
    wb = ws_bytes if ws_bytes is not None else (_nbytes(ws) if ws is not None else 0)
    _check(load().dfl2_conv2_ws(_ptr(x), _ptr(x_prev), _ptr(base), _ptr(W_c), B, L, d, _ptr(y),
                                _ptr(ws), wb, _stream(stream)))


def dfl2_tail(logits, verified_tok, hidden, E, W_A, W_B, W_H, temperature: float, seeds,
              cycle_offset: int, tokens, ws, slots=None, q=None, cand_idx=None, cand_val=None,
              scores=None, stream=None, *, dims=None, dtype=None, ws_bytes=None) -> None:
    """top-16 -> pair scores -> walk in one call; tokens [B,L] int32 out."""
    if dims is not None:
        B, L, V, d = dims
    else:
        B, L, V = logits.shape
        d = hidden.shape[-1]
    dt = dtype if dtype is not None else _dtype_code(logits)
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_tail(_ptr(logits), dt, _ptr(verified_tok), _ptr(hidden), _ptr(E),
                            _ptr(W_A), _ptr(W_B), _ptr(W_H), B, L, V, d, float(temperature),
                            _ptr(seeds), int(cycle_offset), _ptr(tokens), _ptr(slots), _ptr(q),
                            _ptr(cand_idx), _ptr(cand_val), _ptr(scores), _ptr(ws), wb,
                            _stream(stream)))


def dfl2_tables_bytes(V: int) -> int:
    return int(load().dfl2_tables_bytes(V))


def dfl2_tables_build(E, W_A, W_B, P_A, P_B, stream=None, *, dims=None) -> None:
    """P_A = E W_A^T, P_B = E W_B^T (float32 [V, 256]), once per set of weights."""
    V, d = dims if dims is not None else E.shape
    _check(load().dfl2_tables_build(_ptr(E), _ptr(W_A), _ptr(W_B), V, d, _ptr(P_A), _ptr(P_B),
                                    _stream(stream)))


def dfl2_select_tables(cand_idx, cand_val, verified_tok, hidden, W_H, P_A, P_B, scores, ws,
                       stream=None, *, dims=None, ws_bytes=None) -> None:
    """Pair scores [B,L,16,16] with A(.) and B(.) from the token tables."""
    if dims is not None:
        B, L, V, d = dims
    else:
        B, L, d = hidden.shape
        V = P_A.shape[0]
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_select_tables(_ptr(cand_idx), _ptr(cand_val), _ptr(verified_tok),
                                     _ptr(hidden), _ptr(W_H), _ptr(P_A), _ptr(P_B), B, L, V, d,
                                     256, _ptr(scores), _ptr(ws), wb, _stream(stream)))


def dfl2_tail_tables(logits, verified_tok, hidden, W_H, P_A, P_B, temperature: float, seeds,
                     cycle_offset: int, tokens, ws, slots=None, q=None, cand_idx=None,
                     cand_val=None, scores=None, stream=None, *, dims=None, dtype=None,
                     ws_bytes=None) -> None:
    """dfl2_tail with the token tables (the gate projection beside the top-16)."""
    if dims is not None:
        B, L, V, d = dims
    else:
        B, L, V = logits.shape
        d = hidden.shape[-1]
    dt = dtype if dtype is not None else _dtype_code(logits)
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check(load().dfl2_tail_tables(_ptr(logits), dt, _ptr(verified_tok), _ptr(hidden), _ptr(W_H),
                                   _ptr(P_A), _ptr(P_B), B, L, V, d, float(temperature),
                                   _ptr(seeds), int(cycle_offset), _ptr(tokens), _ptr(slots),
                                   _ptr(q), _ptr(cand_idx), _ptr(cand_val), _ptr(scores),
                                   _ptr(ws), wb, _stream(stream)))
