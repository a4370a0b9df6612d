"""Seeded synthetic inputs for the DFlash 2 draft tail.

This module only draws random tensors of the right shapes, dtypes and value
distributions; it holds none of the method's arithmetic.  The tests feed the
same tensors to the CUDA library and to the CPU oracle, and ``bench.py`` times
the library on them.

The pages measure on GSM8K-style suites with trained drafters
("DFlash 2: Keep Drafting Parallel", 实验环境).  Neither the suites nor the
weights are used here: these synthetic tensors stand in for the drafter's
logits, hidden states, token embeddings and selector / conv weights, with the
shapes of the 4B- and 27B-drafter settings the pages describe (block sizes 8
and 16, hidden sizes 2560 and 5120, a 151,936-token vocabulary).
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np
import torch

RANK = 256     # width of A(.), B(.) and H(.): "256 维" in the selector paragraph
NCAND = 16     # candidates kept per position: "Top-16"
GROUP = 16     # channels sharing one conv correction: "每 16 个通道"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int            # base seed; every tensor gets its own stream keyed by its name
    B: int               # independent sequences
    L: int               # drafted positions per block
    V: int               # vocabulary
    d: int               # drafter hidden size
    logits: str          # "peak6_f32" | "zipf_bf16" | "quant64_bf16"
    temperatures: tuple  # walks to run (0.0 = greedy)
    conv_calls: int      # conv invocations per block (5 layers x 4 insertion points = 20)
    e_std: float = 0.02  # token-embedding scale; 1.0 makes the bilinear term O(1)

    @property
    def rows(self) -> int:
        return self.B * self.L

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five draft-tail workloads, smallest first.
WORKLOADS = {
    "tiny_l8_v32k": Workload("tiny_l8_v32k", 1000, 1, 8, 32768, 1024, "peak6_f32", (0.0,), 1),
    "drafter4b_l16": Workload("drafter4b_l16", 1001, 1, 16, 151936, 2560, "zipf_bf16",
                              (0.0, 1.0), 20),
    "drafter27b_l8": Workload("drafter27b_l8", 1002, 1, 8, 151936, 5120, "zipf_bf16", (0.0,), 20),
    "serving_b64": Workload("serving_b64", 1003, 64, 16, 151936, 2560, "zipf_bf16", (1.0,), 20),
    "stress_b256_ties": Workload("stress_b256_ties", 1004, 256, 16, 262144, 6144,
                                 "quant64_bf16", (0.0, 0.7), 20),
}


def _generator(w: Workload, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((w.seed * 1_000_003 + zlib.crc32(name.encode())) % (2**63))
    return g


def splitmix64(x: int) -> int:
    """The splitmix64 output function (Steele, Lea, Flood 2014); used to derive Philox keys."""
    m = (1 << 64) - 1
    z = (x + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def philox_seeds(w: Workload, salt: int = 0) -> np.ndarray:
    """One 64-bit Philox key per sequence."""
    return np.array([splitmix64(w.seed * 65536 + salt * 4096 + b) for b in range(w.B)],
                    dtype=np.uint64)


def make_logits(w: Workload, device="cpu") -> torch.Tensor:
    """Drafter LM-head logits U [B, L, V]."""
    R, V = w.rows, w.V
    g = _generator(w, "logits", device)
    if w.logits == "peak6_f32":
        # N(0,1) with one +6 peak per position at a uniform index.
        u = torch.randn(R, V, generator=g, device=device, dtype=torch.float32)
        pos = torch.randint(0, V, (R,), generator=g, device=device)
        u[torch.arange(R, device=device), pos] += 6.0
        return u.view(w.B, w.L, V)
    if w.logits == "zipf_bf16":
        # N(0, std 2) plus a Zipf-ranked boost 8/r on 50 distinct uniform ids per position.
        u = 2.0 * torch.randn(R, V, generator=g, device=device, dtype=torch.float32)
        ids = torch.multinomial(torch.ones(R, V, device=device), 50, replacement=False,
                                generator=g)
        boost = 8.0 / torch.arange(1, 51, device=device, dtype=torch.float32)
        u.scatter_add_(1, ids, boost.expand(R, 50).contiguous())
        return u.to(torch.bfloat16).view(w.B, w.L, V)
    if w.logits == "quant64_bf16":
        # N(0, std 2), clipped and quantised to the 64 levels -8, -7.75, ..., 7.75
        # (all exact in bf16): heavy ties for the tie-break rule.
        u = 2.0 * torch.randn(R, V, generator=g, device=device, dtype=torch.float32)
        u = torch.clamp(torch.round(u * 4.0) * 0.25, -8.0, 7.75)
        return u.to(torch.bfloat16).view(w.B, w.L, V)
    raise ValueError(f"unknown logits recipe {w.logits!r}")


def make_tail_inputs(w: Workload, device="cpu", salt: int = 0) -> dict:
    """Everything the draft tail reads besides the logits."""
    d, V = w.d, w.V
    sfx = "" if salt == 0 else f"#{salt}"
    out = {}
    g = _generator(w, "verified" + sfx, device)
    out["verified"] = torch.randint(0, V, (w.B,), generator=g, device=device, dtype=torch.int32)
    g = _generator(w, "hidden" + sfx, device)
    out["hidden"] = torch.randn(w.B, w.L, d, generator=g, device=device).to(torch.bfloat16)
    g = _generator(w, "E", device)
    out["E"] = (w.e_std * torch.randn(V, d, generator=g, device=device)).to(torch.bfloat16)
    for name in ("W_A", "W_B", "W_H"):
        g = _generator(w, name, device)
        out[name] = (torch.randn(RANK, d, generator=g, device=device) / np.sqrt(d)).to(
            torch.bfloat16)
    out["seeds"] = philox_seeds(w, salt)
    return out


def make_conv_inputs(w: Workload, call: int, device="cpu") -> dict:
    """One conv invocation: x [B,L,d], x_prev [B,d] (the verified token's
    representation at this insertion point), base [2,d] fp32, W_c [2*d/16, d]."""
    d = w.d
    out = {}
    g = _generator(w, f"conv{call}.x", device)
    out["x"] = torch.randn(w.B, w.L, d, generator=g, device=device).to(torch.bfloat16)
    g = _generator(w, f"conv{call}.x_prev", device)
    out["x_prev"] = torch.randn(w.B, d, generator=g, device=device).to(torch.bfloat16)
    g = _generator(w, f"conv{call}.base", device)
    out["base"] = 0.5 * torch.randn(2, d, generator=g, device=device, dtype=torch.float32)
    g = _generator(w, f"conv{call}.W_c", device)
    out["W_c"] = (0.01 * torch.randn(2 * d // GROUP, d, generator=g, device=device)).to(
        torch.bfloat16)
    return out


def make_verify_inputs(w: Workload, device="cpu", temperature: float = 1.0,
                       sharp: float = 3.0) -> dict:
    """Synthetic inputs for block verification.  p [B, L+1, V] float32: the
    target's next-token distributions, softmax of `sharp` times a target logit
    field that agrees with the drafter's logits up to N(0, 1) noise (row L is a
    fresh field); `sharp` sets how much mass the top candidates hold, and so
    the spread of accepted lengths.  The draft side is drawn independently of any kernel: 16 distinct
    candidates per position sampled from p without replacement, a draft
    distribution q over them (the target's probabilities on the candidates,
    perturbed by N(0, 0.5) in log space, renormalised, at the temperature), and
    the slot (and so the token) drawn from q."""
    B, L, V = w.B, w.L, w.V
    g = _generator(w, "verify.noise", device)
    lg = make_logits(w, device).float()
    tgt = torch.empty(B, L + 1, V, device=device)
    tgt[:, :L] = lg + torch.randn(B, L, V, generator=g, device=device)
    tgt[:, L] = 2.0 * torch.randn(B, V, generator=g, device=device)
    p = torch.softmax(sharp * tgt, dim=-1)
    g = _generator(w, "verify.cand", device)
    cand = torch.multinomial(p[:, :L].reshape(B * L, V), 16, replacement=False, generator=g)
    g = _generator(w, "verify.q", device)
    pc = torch.gather(p[:, :L].reshape(B * L, V), 1, cand)
    noise = 0.5 * torch.randn(B * L, 16, generator=g, device=device)
    q = torch.softmax((torch.log(pc) + noise) / max(temperature, 1e-3), dim=-1)
    g = _generator(w, "verify.slot", device)
    slots = torch.multinomial(q, 1, generator=g).view(B, L)
    cand = cand.view(B, L, 16).to(torch.int32)
    tokens = torch.gather(cand, 2, slots.view(B, L, 1).long()).view(B, L).to(torch.int32)
    return {"p": p.contiguous(), "cand_idx": cand, "q": q.view(B, L, 16).contiguous(),
            "slots": slots.to(torch.int32), "tokens": tokens,
            "seeds": philox_seeds(w, salt=7)}


def make_lmhead_inputs(w: Workload, device="cpu", kind: str = "gauss") -> dict:
    """Synthetic inputs for the LM head + top-16: the drafter's last hidden
    state [B, L, d] and an LM-head weight W_lm [V, d], both bf16.

    kind "gauss": h ~ N(0, 1), W_lm ~ N(0, 1/sqrt(d)), so the logits are about
    N(0, 1).  kind "int": h and W_lm uniform integers in [-3, 3]; every partial
    sum is an integer below 2^24, so float32 accumulation is exact in any order
    and the result can be compared bit for bit.  kind "ties": W_lm as in "int",
    h one-hot on 4 random channels, so the logits take 25 values and the top 16
    is decided by the index tie rule.  W_lm is drawn in row chunks to bound the
    temporaries."""
    B, L, V, d = w.B, w.L, w.V, w.d
    g = _generator(w, f"lmhead.{kind}.hidden", device)
    if kind == "gauss":
        hidden = torch.randn(B, L, d, generator=g, device=device).to(torch.bfloat16)
    elif kind == "int":
        hidden = torch.randint(-3, 4, (B, L, d), generator=g, device=device,
                               dtype=torch.int8).to(torch.bfloat16)
    elif kind == "ties":
        hidden = torch.zeros(B * L, d, dtype=torch.bfloat16, device=device)
        ch = torch.stack([torch.randperm(d, generator=g, device=device)[:4]
                          for _ in range(B * L)])
        hidden.scatter_(1, ch, torch.ones(B * L, 4, dtype=torch.bfloat16, device=device))
        hidden = hidden.view(B, L, d)
    else:
        raise ValueError(f"unknown LM-head input kind {kind!r}")
    g = _generator(w, f"lmhead.{kind}.W", device)
    W = torch.empty(V, d, dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 26) // d)
    for r0 in range(0, V, chunk):
        n = min(chunk, V - r0)
        if kind == "gauss":
            W[r0:r0 + n] = (torch.randn(n, d, generator=g, device=device) / d ** 0.5).to(torch.bfloat16)
        else:
            W[r0:r0 + n] = torch.randint(-3, 4, (n, d), generator=g, device=device,
                                         dtype=torch.int8).to(torch.bfloat16)
    return {"hidden": hidden.contiguous(), "W_lm": W}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's bit patterns as a host uint16 array (what the oracle takes)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    """A tensor as a host numpy array; bf16 becomes its uint16 bit patterns."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().contiguous().cpu().numpy()
