"""Shared test utilities: tolerance rules, device transfer, and one-call drivers that run the
CUDA library and the float64 oracle on the same seeded inputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.inputs import Workload, as_f64, generate

# Tolerances (element-wise E = |gpu - ref| / max(1, |ref|)):
#  float32 I/O: E <= 1e-5 for every output.
#  bf16 I/O:    outputs (y, hT, logits) E <= 4e-3; gradients stored in float32 E <= 2e-3;
#               gradients stored in bf16 |gpu - ref| <= 2e-3 max(1,|ref|) + ulp_bf16(ref)/2.
TOL_F32 = 1e-5
TOL_BF16_OUT = 4e-3
TOL_BF16_GRAD = 2e-3


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, np.finfo(np.float64).tiny)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def err_E(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


def assert_close(name, got, ref, *, io: str, kind: str, stored: str = "f32"):
    """kind: "out" or "grad"; stored: dtype the GPU wrote ("f32" or "bf16")."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    d = np.abs(got - ref)
    s = np.maximum(1.0, np.abs(ref))
    if io == "f32":
        bound = TOL_F32 * s
    elif kind == "out":
        bound = TOL_BF16_OUT * s
    elif stored == "bf16":
        bound = TOL_BF16_GRAD * s + half_ulp_bf16(ref)
    else:
        bound = TOL_BF16_GRAD * s
    bad = d > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(d / bound), d.shape)
        raise AssertionError(f"{name}: {int(bad.sum())}/{d.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r} (E={err_E(got, ref):.3e})")


def dev(t, device="cuda"):
    return None if t is None else t.to(device).contiguous()


def host(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def mode_id(wl: Workload) -> int:
    return R.CANONICAL if wl.mode == "canonical" else R.RESTRICTED


def shape_for(wl: Workload, grad: str | None = None) -> R.Shape:
    io = R.F32 if wl.io == "f32" else R.BF16
    g = io if grad is None else (R.F32 if grad == "f32" else R.BF16)
    return R.make_shape(wl.B, wl.T, wl.W, wl.nblk, io, g, mode_id(wl))


def oracle_inputs(inp: dict) -> dict:
    return {k: (as_f64(v) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
