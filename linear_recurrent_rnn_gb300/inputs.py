"""Seeded synthetic inputs for the RG-LRU layer.

This module only draws random numbers and arranges them into tensors; it holds none of the
layer's arithmetic.  The same generator feeds the CUDA library and the float64 oracle: values
are drawn with numpy's PCG64, cast to the storage dtype on the host, and the oracle widens the
*stored* values back to float64, so both sides see identical inputs.

The five workloads are the RG-LRU configurations named by the layer's specification (sizes,
value distributions and reset structure); none comes from a dataset.  Two readings are taken
where the specification leaves a step open:

* "Lambda set so that a^c is uniform in [lo, hi]": draw u ~ U[lo, hi] per channel and choose
  Lambda so that c * softplus(Lambda) = -ln(u), i.e. a_t = u ** r_t lies in (u, 1).
* Packed segments: segment lengths are drawn uniform in [lo, hi] until the row is full (the
  last one truncated).  In the packed configurations that also carry an initial state, the
  first segment is read as the continuation of an earlier one: its positions start at a
  seeded offset >= 1, so token 0 is not a reset and h0 matters.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

DECAY_C = 8.0  # the layer's decay constant, used only to place Lambda (see module docstring)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    W: int
    k: int
    io: str                      # "f32" or "bf16"
    mode: str                    # "canonical" or "restricted"
    u_range: tuple = (0.9, 0.999)
    reset_p: float = 0.0         # Bernoulli reset probability per token
    reset_t0: bool = False       # force a reset at token 0
    seg_len: Optional[tuple] = None   # packed segment lengths U[lo, hi]
    continuation: bool = False   # first packed segment continues an earlier one
    h0_std: float = 0.0          # 0 => no initial state

    @property
    def nblk(self) -> int:
        return self.W // self.k

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Tiny canonical, fp32 I/O: B1 T64 W128, 2 blocks of 64; resets p=0.05 plus token 0.
    1: Workload("tiny-canonical-f32", 1, 64, 128, 64, "f32", "canonical", (0.9, 0.999),
                reset_p=0.05, reset_t0=True, h0_std=1.0),
    # Restricted protocol, bf16 I/O: B4 T2048 W2048, 16 blocks of 128; no resets, h0 = 0.
    2: Workload("restricted-B4-T2048-W2048-bf16", 4, 2048, 2048, 128, "bf16", "restricted",
                (0.9, 0.999)),
    # Canonical packed, bf16: segment lengths U[1, 2048]; h0 ~ N(0, 0.5^2).
    3: Workload("packed-B4-T2048-W2048-bf16", 4, 2048, 2048, 128, "bf16", "canonical",
                (0.9, 0.999), seg_len=(1, 2048), continuation=True, h0_std=0.5),
    # Long sequence with partial chunks, bf16: B1 T32771 W2560, 20 blocks; resets p=1e-3.
    4: Workload("long-B1-T32771-W2560-bf16", 1, 32771, 2560, 128, "bf16", "canonical",
                (0.99, 0.9999), reset_p=1e-3),
    # Large training shape, bf16: B8 T4096 W4000, 25 blocks of 160; packed U[256, 4096]; h0.
    5: Workload("packed-B8-T4096-W4000-k160-bf16", 8, 4096, 4000, 160, "bf16", "canonical",
                (0.9, 0.999), seg_len=(256, 4096), continuation=True, h0_std=1.0),
}

IO_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def lambda_for_decay(u: np.ndarray) -> np.ndarray:
    """Lambda with DECAY_C * softplus(Lambda) = -ln(u) (so that a = u at r = 1)."""
    s = -np.log(u) / DECAY_C
    return np.log(np.expm1(s))


def segment_positions(rng: np.random.Generator, T: int, lo: int, hi: int,
                      continuation: bool) -> np.ndarray:
    """Per-token position inside its packed segment for one row of length T."""
    pos = np.empty(T, dtype=np.int32)
    t = 0
    first = True
    while t < T:
        L = int(rng.integers(lo, hi + 1))
        start = int(rng.integers(1, hi + 1)) if (first and continuation) else 0
        n = min(L, T - t)
        pos[t:t + n] = np.arange(start, start + n, dtype=np.int32)
        t += n
        first = False
    return pos


def packed_lengths(seed: int, T: int, lo: int, hi: int) -> list:
    """Sequence lengths drawn U[lo, hi] until they fill T tokens (the last one truncated), for
    packed variable-length sequences given by cu_seqlens."""
    rng = np.random.default_rng(seed)
    lengths, t = [], 0
    while t < T:
        n = min(int(rng.integers(lo, hi + 1)), T - t)
        lengths.append(n)
        t += n
    return lengths

def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


def generate(wl: Workload, seed: int, *, want_logits: bool = False,
             want_dlogits: bool = False) -> dict:
    """Draw every input of one RG-LRU call for workload `wl` (torch CPU tensors in their
    storage dtypes).  Keys: x, Wa, ba, Wx, bx, Lambda, reset_mask|segment_pos|None, h0, dy,
    dhT, and optionally lr, li (logits ~ N(0,1), the distribution of the projected logits)
    and dlr, dli (upstream logit gradients for the projection backward)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    io = IO_DTYPE[wl.io]
    B, T, W, k = wl.B, wl.T, wl.W, wl.k
    out = {}
    out["x"] = torch.from_numpy(_normal(rng, (B, T, W))).to(io)
    wstd = 1.0 / np.sqrt(k)
    out["Wa"] = torch.from_numpy(_normal(rng, (wl.nblk, k, k), wstd)).to(io)
    out["Wx"] = torch.from_numpy(_normal(rng, (wl.nblk, k, k), wstd)).to(io)
    out["ba"] = torch.zeros(W, dtype=torch.float32)
    out["bx"] = torch.zeros(W, dtype=torch.float32)
    u = rng.uniform(wl.u_range[0], wl.u_range[1], size=W)
    out["Lambda"] = torch.from_numpy(lambda_for_decay(u).astype(np.float32))
    out["reset_mask"] = None
    out["segment_pos"] = None
    if wl.mode == "canonical":
        if wl.seg_len is not None:
            sp = np.stack([segment_positions(rng, T, wl.seg_len[0], wl.seg_len[1],
                                             wl.continuation) for _ in range(B)])
            out["segment_pos"] = torch.from_numpy(sp)
        elif wl.reset_p > 0 or wl.reset_t0:
            rm = (rng.random((B, T)) < wl.reset_p).astype(np.uint8)
            if wl.reset_t0:
                rm[:, 0] = 1
            out["reset_mask"] = torch.from_numpy(rm)
    out["h0"] = (torch.from_numpy(_normal(rng, (B, W), wl.h0_std))
                 if (wl.mode == "canonical" and wl.h0_std > 0) else None)
    out["dy"] = torch.from_numpy(_normal(rng, (B, T, W))).to(io)
    out["dhT"] = (torch.from_numpy(_normal(rng, (B, W))) if wl.mode == "canonical" else None)
    if want_logits:
        out["lr"] = torch.from_numpy(_normal(rng, (B, T, W))).to(io)
        out["li"] = torch.from_numpy(_normal(rng, (B, T, W))).to(io)
    if want_dlogits:
        out["dlr"] = torch.from_numpy(_normal(rng, (B, T, W), 0.1)).to(io)
        out["dli"] = torch.from_numpy(_normal(rng, (B, T, W), 0.1)).to(io)
    return out


def as_f64(t) -> Optional[np.ndarray]:
    """The stored values widened to float64 (what the oracle consumes)."""
    if t is None:
        return None
    if t.dtype in (torch.uint8, torch.int32):
        return t.numpy()
    return t.to(torch.float64).numpy()
