"""RG-LRU oracle: TEST INFRASTRUCTURE ONLY.

A float64 CPU statement of the RG-LRU forward and backward (the recurrence, its reset
semantics, the block-diagonal gate projections and their hand-derived gradients), used to
check the CUDA library element by element.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the CUDA library:
the arithmetic lives in ``rglru_oracle.c`` (compiled here with gcc, IEEE double, no FMA
contraction) and this module only marshals numpy arrays.

Passages followed (all on the Fattori comparison page unless noted): the list of what the
operator fuses (sigmoid gates, softplus(a_param) and dynamic decay, the stationary square-root
multiplier, the input-gated write, the sequential recurrence, and the reverse recurrence with
pointwise derivatives in the backward); the "semantic limits" list (segment_pos / arbitrary
reset / nonzero initial state; reset-token normalisation) for canonical mode; the benchmark
record's "protocol" and "correctness.contract" (zero initial state, no resets) for restricted
mode; and the first paragraph plus the record's "protocol.scope" for the block-diagonal gate
projections.  The decay constant c = 8 and its sign are fixed by the specification.

Every function here has a pin in ``tests/test_oracle_pins.py`` (closed forms, special
cases, invariants, finite differences, a library matmul); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

CANONICAL = 0
RESTRICTED = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rglru_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_rglru.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (IEEE double, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            i64 = ctypes.c_long
            lib.oracle_forward.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]
            lib.oracle_backward.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P,
                                            P, P, P, P]
            lib.oracle_gate_proj.argtypes = [i64, i32, i32, P, P, P, P, P, P, P]
            lib.oracle_gate_proj_backward.argtypes = [i64, i32, i32, P, P, P, P, P, P, P, P,
                                                      P, P]
            for f in (lib.oracle_forward, lib.oracle_backward, lib.oracle_gate_proj,
                      lib.oracle_gate_proj_backward):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _d(a):
    """Widen to a C-contiguous float64 array (None stays None)."""
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _masks(reset_mask, segment_pos):
    if reset_mask is not None and segment_pos is not None:
        raise ValueError("give at most one of reset_mask / segment_pos")
    rm = None if reset_mask is None else np.ascontiguousarray(np.asarray(reset_mask, dtype=np.uint8))
    sp = None if segment_pos is None else np.ascontiguousarray(np.asarray(segment_pos, dtype=np.int32))
    return rm, sp


def forward(mode, x, lr, li, Lambda, reset_mask=None, segment_pos=None, h0=None):
    """Recurrence forward.  x, lr, li: [B, T, W]; Lambda: [W]; reset_mask/segment_pos: [B, T];
    h0: [B, W] or None.  Returns (y [B,T,W], hT [B,W]) in float64."""
    x, lr, li, Lambda, h0 = _d(x), _d(lr), _d(li), _d(Lambda), _d(h0)
    B, T, W = x.shape
    rm, sp = _masks(reset_mask, segment_pos)
    y = np.empty_like(x)
    hT = np.empty((B, W))
    st = _load().oracle_forward(int(mode), B, T, W, _ptr(x), _ptr(lr), _ptr(li), _ptr(Lambda),
                                _ptr(rm), _ptr(sp), _ptr(h0), _ptr(y), _ptr(hT))
    if st:
        raise RuntimeError(f"oracle_forward failed ({st})")
    return y, hT


def backward(mode, x, lr, li, Lambda, dy, dhT=None, reset_mask=None, segment_pos=None, h0=None):
    """Recurrence backward.  Returns dict with dx, dlr, dli [B,T,W], dLambda [W], dh0 [B,W]."""
    x, lr, li, Lambda, h0, dy, dhT = map(_d, (x, lr, li, Lambda, h0, dy, dhT))
    B, T, W = x.shape
    rm, sp = _masks(reset_mask, segment_pos)
    out = {k: np.empty_like(x) for k in ("dx", "dlr", "dli")}
    out["dLambda"] = np.empty(W)
    out["dh0"] = np.empty((B, W))
    st = _load().oracle_backward(int(mode), B, T, W, _ptr(x), _ptr(lr), _ptr(li), _ptr(Lambda),
                                 _ptr(rm), _ptr(sp), _ptr(h0), _ptr(dy), _ptr(dhT),
                                 _ptr(out["dx"]), _ptr(out["dlr"]), _ptr(out["dli"]),
                                 _ptr(out["dLambda"]), _ptr(out["dh0"]))
    if st:
        raise RuntimeError(f"oracle_backward failed ({st})")
    return out


def gate_proj(x, Wa, ba, Wx, bx):
    """Block-diagonal projections.  x: [..., W]; Wa, Wx: [nblk, k, k] (in, out); ba, bx: [W]
    or None.  Returns (lr, li) shaped like x."""
    x, Wa, ba, Wx, bx = map(_d, (x, Wa, ba, Wx, bx))
    W = x.shape[-1]
    nblk = Wa.shape[0]
    BT = x.size // W
    lr = np.empty_like(x)
    li = np.empty_like(x)
    st = _load().oracle_gate_proj(BT, W, nblk, _ptr(x), _ptr(Wa), _ptr(ba), _ptr(Wx), _ptr(bx),
                                  _ptr(lr), _ptr(li))
    if st:
        raise RuntimeError(f"oracle_gate_proj failed ({st})")
    return lr, li


def gate_proj_backward(x, Wa, Wx, dlr, dli, dx_in=None):
    """Projection backward.  Returns dict with dx (= dx_in + dlr Wa^T + dli Wx^T), dWa, dba,
    dWx, dbx."""
    x, Wa, Wx, dlr, dli = map(_d, (x, Wa, Wx, dlr, dli))
    W = x.shape[-1]
    nblk = Wa.shape[0]
    BT = x.size // W
    dx = np.zeros_like(x) if dx_in is None else np.array(dx_in, dtype=np.float64, copy=True, order="C")
    out = {"dx": dx, "dWa": np.empty_like(Wa), "dWx": np.empty_like(Wx),
           "dba": np.empty(W), "dbx": np.empty(W)}
    st = _load().oracle_gate_proj_backward(BT, W, nblk, _ptr(x), _ptr(Wa), _ptr(Wx), _ptr(dlr),
                                           _ptr(dli), _ptr(dx), _ptr(out["dWa"]),
                                           _ptr(out["dba"]), _ptr(out["dWx"]), _ptr(out["dbx"]))
    if st:
        raise RuntimeError(f"oracle_gate_proj_backward failed ({st})")
    return out


def fused_forward(mode, x, Wa, ba, Wx, bx, Lambda, reset_mask=None, segment_pos=None, h0=None):
    """Projections then recurrence; the logits stay float64 (never rounded)."""
    lr, li = gate_proj(x, Wa, ba, Wx, bx)
    y, hT = forward(mode, x, lr, li, Lambda, reset_mask, segment_pos, h0)
    return y, hT


def fused_backward(mode, x, Wa, ba, Wx, bx, Lambda, dy, dhT=None, reset_mask=None,
                   segment_pos=None, h0=None):
    """Gradients of the fused layer: dx (direct + through both projections), dWa, dba, dWx,
    dbx, dLambda, dh0."""
    lr, li = gate_proj(x, Wa, ba, Wx, bx)
    g = backward(mode, x, lr, li, Lambda, dy, dhT, reset_mask, segment_pos, h0)
    p = gate_proj_backward(x, Wa, Wx, g["dlr"], g["dli"], dx_in=g["dx"])
    return {"dx": p["dx"], "dWa": p["dWa"], "dba": p["dba"], "dWx": p["dWx"], "dbx": p["dbx"],
            "dLambda": g["dLambda"], "dh0": g["dh0"]}
