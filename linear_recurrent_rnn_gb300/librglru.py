"""Thin ctypes binding of librglru (include/librglru.h and include/delta_rule.h).

Argument marshalling only: every function here checks that its tensors are contiguous CUDA
tensors, passes their device pointers and the current CUDA stream to the C ABI call of the
same name, and raises ``RglruError`` on a non-OK status.  No arithmetic runs in Python and
there is no fallback: if the shared library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

F32, BF16 = 0, 1
CANONICAL, RESTRICTED = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(5)

_DT = {torch.float32: F32, torch.bfloat16: BF16}
TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


class RglruError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("W", ctypes.c_int32),
                ("nblk", ctypes.c_int32), ("io", ctypes.c_int32), ("grad", ctypes.c_int32),
                ("mode", ctypes.c_int32)]

    def __repr__(self):
        return (f"Shape(B={self.B}, T={self.T}, W={self.W}, nblk={self.nblk}, io={self.io}, "
                f"grad={self.grad}, mode={self.mode})")


class DeltaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hk", ctypes.c_int32),
                ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
                ("io", ctypes.c_int32), ("kda", ctypes.c_int32),
                ("state_v_first", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None

EXPORTS = ("rglru_status_string", "rglru_saved_bytes", "rglru_workspace_bytes",
           "rglru_gate_proj", "rglru_forward", "rglru_backward", "rglru_gate_proj_backward",
           "rglru_fused_forward", "rglru_fused_backward", "rglru_sync_status",
           "rglru_debug_lookback", "rglru_kernel_launches", "rglru_forward_noalloc",
           "rglru_forward_noalloc_status", "rglru_fused_path",
           "rglru_debug_kernel_events", "rglru_step", "rglru_fused_forward_varlen",
           "rglru_fused_backward_varlen", "delta_rule_saved_bytes", "delta_rule_workspace_bytes",
           "delta_rule_forward", "delta_rule_backward", "delta_rule_state_fp8_qdq")

# Static look-back scratch of rglru_forward_noalloc, per GPU (RGLRU_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 16 << 20


def library_path() -> str:
    return os.environ.get("RGLRU_LIBRARY", _build.LIB)


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"librglru is not built ({path} missing); call "
                                   "linear_recurrent_rnn_gb300.build.build() first")
            L = ctypes.CDLL(path)
            P, S = ctypes.c_void_p, ctypes.POINTER(Shape)
            L.rglru_status_string.argtypes = [ctypes.c_int]
            L.rglru_status_string.restype = ctypes.c_char_p
            L.rglru_saved_bytes.argtypes = [S]
            L.rglru_saved_bytes.restype = ctypes.c_size_t
            L.rglru_workspace_bytes.argtypes = [S]
            L.rglru_workspace_bytes.restype = ctypes.c_size_t
            L.rglru_gate_proj.argtypes = [S] + [P] * 8
            L.rglru_forward.argtypes = [S] + [P] * 11
            L.rglru_backward.argtypes = [S] + [P] * 17
            L.rglru_gate_proj_backward.argtypes = [S] + [P] * 12
            L.rglru_fused_forward.argtypes = [S] + [P] * 13
            L.rglru_fused_backward.argtypes = [S] + [P] * 21
            L.rglru_sync_status.argtypes = [P, P]
            L.rglru_debug_lookback.argtypes = [ctypes.c_int32, ctypes.c_int32]
            L.rglru_debug_lookback.restype = None
            L.rglru_forward_noalloc.argtypes = [S] + [P] * 10
            L.rglru_forward_noalloc.restype = ctypes.c_int
            L.rglru_forward_noalloc_status.argtypes = [P]
            L.rglru_forward_noalloc_status.restype = ctypes.c_int
            L.rglru_fused_path.argtypes = [S]
            L.rglru_fused_path.restype = ctypes.c_char_p
            L.rglru_debug_kernel_events.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            L.rglru_debug_kernel_events.restype = None
            L.rglru_step.argtypes = [S] + [P] * 11
            L.rglru_fused_forward_varlen.argtypes = [S] + [P] * 7 + [ctypes.c_int32] + [P] * 5
            L.rglru_fused_backward_varlen.argtypes = ([S] + [P] * 9 + [ctypes.c_int32] +
                                                      [P] * 11)
            DS = ctypes.POINTER(DeltaShape)
            L.delta_rule_saved_bytes.argtypes = [DS, ctypes.c_int32]
            L.delta_rule_saved_bytes.restype = ctypes.c_size_t
            L.delta_rule_workspace_bytes.argtypes = [DS]
            L.delta_rule_workspace_bytes.restype = ctypes.c_size_t
            L.delta_rule_forward.argtypes = ([DS] + [P] * 5 + [ctypes.c_float, P, ctypes.c_int32] +
                                             [P] * 5)
            L.delta_rule_backward.argtypes = ([DS] + [P] * 5 + [ctypes.c_float, P, ctypes.c_int32] +
                                              [P] * 12)
            L.delta_rule_state_fp8_qdq.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, P]
            L.delta_rule_state_fp8_qdq.restype = ctypes.c_int
            L.delta_rule_forward.restype = ctypes.c_int
            L.delta_rule_backward.restype = ctypes.c_int
            L.rglru_kernel_launches.argtypes = []
            L.rglru_kernel_launches.restype = ctypes.c_uint64
            for n in ("rglru_gate_proj", "rglru_forward", "rglru_backward",
                      "rglru_gate_proj_backward", "rglru_fused_forward", "rglru_fused_backward",
                      "rglru_sync_status", "rglru_step", "rglru_fused_forward_varlen",
                      "rglru_fused_backward_varlen"):
                getattr(L, n).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().rglru_status_string(int(status)).decode()


def make_shape(B, T, W, nblk, io=BF16, grad=None, mode=CANONICAL) -> Shape:
    if isinstance(io, torch.dtype):
        io = _DT[io]
    if grad is None:
        grad = io
    elif isinstance(grad, torch.dtype):
        grad = _DT[grad]
    return Shape(int(B), int(T), int(W), int(nblk), int(io), int(grad), int(mode))


def fused_path(shape: Shape) -> str:
    """Which kernels the fused calls run for this shape (a description from the library)."""
    return lib().rglru_fused_path(ctypes.byref(shape)).decode()


def saved_bytes(shape: Shape) -> int:
    return int(lib().rglru_saved_bytes(ctypes.byref(shape)))


def workspace_bytes(shape: Shape) -> int:
    return int(lib().rglru_workspace_bytes(ctypes.byref(shape)))


def alloc_saved(shape: Shape, device="cuda") -> torch.Tensor:
    return torch.empty(max(1, saved_bytes(shape)), dtype=torch.uint8, device=device)


def alloc_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    return torch.empty(max(1, workspace_bytes(shape)), dtype=torch.uint8, device=device)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("librglru takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("librglru takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, st):
    if st != OK:
        raise RglruError(fn, st)


def rglru_gate_proj(shape, x, Wa, ba, Wx, bx, lr, li, stream=None):
    _check("rglru_gate_proj", lib().rglru_gate_proj(
        ctypes.byref(shape), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(lr), _p(li),
        _stream(stream)))


def rglru_forward(shape, x, lr, li, Lambda, reset_mask, segment_pos, h0, y, hT, saved,
                  stream=None):
    _check("rglru_forward", lib().rglru_forward(
        ctypes.byref(shape), _p(x), _p(lr), _p(li), _p(Lambda), _p(reset_mask), _p(segment_pos),
        _p(h0), _p(y), _p(hT), _p(saved), _stream(stream)))


def rglru_backward(shape, dy, dhT, x, lr, li, Lambda, reset_mask, segment_pos, h0, saved, dx,
                   dlr, dli, dLambda, dh0, workspace, stream=None):
    _check("rglru_backward", lib().rglru_backward(
        ctypes.byref(shape), _p(dy), _p(dhT), _p(x), _p(lr), _p(li), _p(Lambda),
        _p(reset_mask), _p(segment_pos), _p(h0), _p(saved), _p(dx), _p(dlr), _p(dli),
        _p(dLambda), _p(dh0), _p(workspace), _stream(stream)))


def rglru_forward_noalloc(shape, x, lr, li, Lambda, reset_mask, segment_pos, h0, y, hT,
                          stream=None):
    """rglru_forward for callers that may not allocate: no `saved` buffer, the look-back
    scratch is the library's static per-GPU array (first call per device outside capture)."""
    _check("rglru_forward_noalloc", lib().rglru_forward_noalloc(
        ctypes.byref(shape), _p(x), _p(lr), _p(li), _p(Lambda), _p(reset_mask), _p(segment_pos),
        _p(h0), _p(y), _p(hT), _stream(stream)))


def rglru_forward_noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns the status word of the last rglru_forward_noalloc
    call on the current device (the next call clears it)."""
    return int(lib().rglru_forward_noalloc_status(_stream(stream)))


def rglru_gate_proj_backward(shape, dlr, dli, x, Wa, Wx, dx, dWa, dba, dWx, dbx, workspace,
                             stream=None):
    _check("rglru_gate_proj_backward", lib().rglru_gate_proj_backward(
        ctypes.byref(shape), _p(dlr), _p(dli), _p(x), _p(Wa), _p(Wx), _p(dx), _p(dWa), _p(dba),
        _p(dWx), _p(dbx), _p(workspace), _stream(stream)))


def rglru_fused_forward(shape, x, Wa, ba, Wx, bx, Lambda, reset_mask, segment_pos, h0, y, hT,
                        saved, stream=None):
    _check("rglru_fused_forward", lib().rglru_fused_forward(
        ctypes.byref(shape), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(Lambda), _p(reset_mask),
        _p(segment_pos), _p(h0), _p(y), _p(hT), _p(saved), _stream(stream)))


def rglru_fused_backward(shape, dy, dhT, x, Wa, ba, Wx, bx, Lambda, reset_mask, segment_pos, h0,
                         saved, dx, dWa, dba, dWx, dbx, dLambda, dh0, workspace, stream=None):
    _check("rglru_fused_backward", lib().rglru_fused_backward(
        ctypes.byref(shape), _p(dy), _p(dhT), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(Lambda),
        _p(reset_mask), _p(segment_pos), _p(h0), _p(saved), _p(dx), _p(dWa), _p(dba), _p(dWx),
        _p(dbx), _p(dLambda), _p(dh0), _p(workspace), _stream(stream)))


def rglru_step(shape, x, Wa, ba, Wx, bx, Lambda, reset, h_in, y, h_out, stream=None):
    _check("rglru_step", lib().rglru_step(
        ctypes.byref(shape), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(Lambda), _p(reset),
        _p(h_in), _p(y), _p(h_out), _stream(stream)))


def rglru_fused_forward_varlen(shape, x, Wa, ba, Wx, bx, Lambda, cu_seqlens, num_seqs, h0, y,
                               hT, saved, stream=None):
    _check("rglru_fused_forward_varlen", lib().rglru_fused_forward_varlen(
        ctypes.byref(shape), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(Lambda), _p(cu_seqlens),
        int(num_seqs), _p(h0), _p(y), _p(hT), _p(saved), _stream(stream)))


def rglru_fused_backward_varlen(shape, dy, dhT, x, Wa, ba, Wx, bx, Lambda, cu_seqlens, num_seqs,
                                h0, saved, dx, dWa, dba, dWx, dbx, dLambda, dh0, workspace,
                                stream=None):
    _check("rglru_fused_backward_varlen", lib().rglru_fused_backward_varlen(
        ctypes.byref(shape), _p(dy), _p(dhT), _p(x), _p(Wa), _p(ba), _p(Wx), _p(bx), _p(Lambda),
        _p(cu_seqlens), int(num_seqs), _p(h0), _p(saved), _p(dx), _p(dWa), _p(dba), _p(dWx),
        _p(dbx), _p(dLambda), _p(dh0), _p(workspace), _stream(stream)))


def rglru_sync_status(buf: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the status word of a saved/workspace buffer."""
    return int(lib().rglru_sync_status(_p(buf), _stream(stream)))


def rglru_debug_lookback(spin_limit: int, drop_tile: int) -> None:
    lib().rglru_debug_lookback(int(spin_limit), int(drop_tile))


def rglru_debug_kernel_events(start, stop) -> None:
    """Records the torch.cuda.Event pair `start`/`stop` around the next fused call's
    tensor-core kernel (both already created, i.e. recorded once); None, None cancels."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    lib().rglru_debug_kernel_events(h(start), h(stop))


def rglru_kernel_launches() -> int:
    return int(lib().rglru_kernel_launches())


# ---------------------------------------------------------------- gated delta rule

def make_delta_shape(B, T, Hk, Hv, Dk, Dv, io=BF16, kda=False, state_v_first=False):
    if isinstance(io, torch.dtype):
        io = _DT[io]
    return DeltaShape(int(B), int(T), int(Hk), int(Hv), int(Dk), int(Dv), int(io), int(bool(kda)),
                      int(bool(state_v_first)))


def delta_rule_saved_bytes(shape: DeltaShape, num_seqs: int) -> int:
    return int(lib().delta_rule_saved_bytes(ctypes.byref(shape), int(num_seqs)))


def delta_rule_workspace_bytes(shape: DeltaShape) -> int:
    return int(lib().delta_rule_workspace_bytes(ctypes.byref(shape)))


def delta_rule_forward(shape, q, k, v, g, beta, scale, cu_seqlens, num_seqs, h0, o, hT, saved,
                       stream=None):
    _check("delta_rule_forward", lib().delta_rule_forward(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta), ctypes.c_float(scale),
        _p(cu_seqlens), int(num_seqs), _p(h0), _p(o), _p(hT), _p(saved), _stream(stream)))


def delta_rule_backward(shape, q, k, v, g, beta, scale, cu_seqlens, num_seqs, h0, saved, do,
                        dhT, dq, dk, dv, dg, dbeta, dh0, workspace, stream=None):
    _check("delta_rule_backward", lib().delta_rule_backward(
        ctypes.byref(shape), _p(q), _p(k), _p(v), _p(g), _p(beta), ctypes.c_float(scale),
        _p(cu_seqlens), int(num_seqs), _p(h0), _p(saved), _p(do), _p(dhT), _p(dq), _p(dk),
        _p(dv), _p(dg), _p(dbeta), _p(dh0), _p(workspace), _stream(stream)))


def delta_rule_state_fp8_qdq(state, out, block_v=64, stream=None):
    """E4M3 quantize-dequantize of float32 key-first states [..., Dk, Dv] (out may be state)."""
    Dk, Dv = state.shape[-2], state.shape[-1]
    n = state.numel() // (Dk * Dv)
    _check("delta_rule_state_fp8_qdq", lib().delta_rule_state_fp8_qdq(
        _p(state), _p(out), int(n), int(Dk), int(Dv), int(block_v), _stream(stream)))
