"""Seeded synthetic inputs for the gated delta rule (GDN / KDA).

This module only draws random numbers and arranges them into tensors; it holds none of the
recurrence's arithmetic.  The same draws feed the CUDA library and the float64 oracle: values
come from numpy's PCG64, are cast to the storage dtype on the host, and the oracle widens the
stored values back to float64.

The reference page takes q, k, v and beta as already normalised / activated and the gates as
natural logarithms, and prints no workload sizes.  The recipe: q and k drawn N(0, 1) and
scaled to unit length per head vector (the usual normalisation of delta-rule keys); v N(0, 1);
beta U(0, 1) (a sigmoid-activated write strength); the decays exp(g) U[lo, hi] per token and
head (GDN) or per token, head and key channel (KDA), g their natural logarithm; initial states
N(0, h0_std^2).  The timed workload is B4 T2048 with 16 heads of 128 x 128 (model width 2048,
the RG-LRU headline width).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class DeltaWorkload:
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    io: str = "bf16"                 # storage dtype of q, k, v and o: "f32" or "bf16"
    kda: bool = False                # per-key decays
    decay: tuple = (0.8, 1.0)        # exp(g) ~ U[lo, hi]
    h0_std: float = 0.0              # 0: no initial state
    lengths: Optional[tuple] = None  # packed sequence lengths (B must be 1)

    def scaled(self, **kw):
        return dataclasses.replace(self, **kw)


DELTA_WORKLOADS = {
    "small": DeltaWorkload("gdn-small", 2, 100, 2, 4, 64, 64, "f32", h0_std=0.5),
    "headline": DeltaWorkload("gdn-B4-T2048-H16-D128", 4, 2048, 16, 16, 128, 128, "bf16"),
}


def _dt(io):
    return torch.float32 if io == "f32" else torch.bfloat16


def generate(wl: DeltaWorkload, seed: int) -> dict:
    """Tensors on the host: q, k, v, do in the storage dtype; g, beta, h0, dhT float32;
    cu_seqlens int32 (or None)."""
    rng = np.random.default_rng(seed)
    B, T = wl.B, wl.T
    q = rng.standard_normal((B, T, wl.Hk, wl.Dk))
    k = rng.standard_normal((B, T, wl.Hk, wl.Dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, wl.Hv, wl.Dv))
    beta = rng.uniform(0.0, 1.0, (B, T, wl.Hv))
    gshape = (B, T, wl.Hv, wl.Dk) if wl.kda else (B, T, wl.Hv)
    g = np.log(rng.uniform(wl.decay[0], wl.decay[1], gshape))
    do = rng.standard_normal((B, T, wl.Hv, wl.Dv))
    cu = None
    if wl.lengths is not None:
        assert B == 1 and sum(wl.lengths) == T
        cu = np.concatenate([[0], np.cumsum(wl.lengths)]).astype(np.int32)
    N = B if cu is None else len(cu) - 1
    h0 = dhT = None
    if wl.h0_std > 0:
        h0 = rng.standard_normal((N, wl.Hv, wl.Dk, wl.Dv)) * wl.h0_std
        dhT = rng.standard_normal((N, wl.Hv, wl.Dk, wl.Dv))
    dt = _dt(wl.io)
    out = {
        "q": torch.from_numpy(q).to(dt), "k": torch.from_numpy(k).to(dt),
        "v": torch.from_numpy(v).to(dt), "do": torch.from_numpy(do).to(dt),
        "g": torch.from_numpy(g).float(), "beta": torch.from_numpy(beta).float(),
        "h0": None if h0 is None else torch.from_numpy(h0).float(),
        "dhT": None if dhT is None else torch.from_numpy(dhT).float(),
        "cu_seqlens": None if cu is None else torch.from_numpy(cu),
    }
    return out


def as_f64(t):
    return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()
