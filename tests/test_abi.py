"""CPU checks of the C ABI: the library builds and loads without a GPU, exports every symbol
that include/librglru.h declares, sizes its scratch buffers, and rejects invalid arguments on
the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

from linear_recurrent_rnn_gb300 import build as B_
from linear_recurrent_rnn_gb300 import librglru as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "librglru.h")
HEADERS = (HEADER, os.path.join(ROOT, "include", "delta_rule.h"))


@pytest.fixture(scope="module")
def lib():
    B_.build()
    return R.lib()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:rglru|delta_rule)_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("rglru_gate_proj", "rglru_forward", "rglru_backward", "rglru_gate_proj_backward",
              "rglru_fused_forward", "rglru_fused_backward", "rglru_saved_bytes",
              "rglru_workspace_bytes", "rglru_status_string", "rglru_sync_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B_.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT ((?:rglru|delta_rule)_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)
    assert set(R.EXPORTS) <= set(declared_functions())


def test_status_strings(lib):
    assert R.status_string(R.OK) == "ok"
    assert "timed out" in R.status_string(R.ERR_TIMEOUT)


def test_scratch_sizes(lib):
    sh = R.make_shape(4, 2048, 2048, 16, R.BF16, R.BF16, R.RESTRICTED)
    s, w = R.saved_bytes(sh), R.workspace_bytes(sh)
    # the saved chunk states alone are B*(ceil(T/16)+1)*W float32
    assert s >= 4 * (2048 // 16 + 1) * 2048 * 4
    assert w > 0
    assert R.saved_bytes(R.make_shape(1, 1, 8, 1)) > 0
    # invalid shapes size to zero
    assert R.saved_bytes(R.make_shape(0, 1, 8, 1)) == 0
    assert R.saved_bytes(R.make_shape(1, 1, 10, 3)) == 0          # W % nblk
    assert R.workspace_bytes(R.make_shape(1, 1, 12, 1)) == 0      # 12 bf16 = 24 bytes, not 16-aligned
    assert R.saved_bytes(R.make_shape(1, 4, 8, 1, R.F32, R.BF16)) == 0   # f32 io needs f32 grads


def _call_forward(lib, sh, x=16, lr=16, li=16, L=16, rm=None, sp=None, h0=None, y=16, saved=16):
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.rglru_forward(ctypes.byref(sh), P(x), P(lr), P(li), P(L), P(rm), P(sp), P(h0),
                             P(y), None, P(saved), None)


def test_host_validation_rejects_before_cuda(lib):
    """Fake (never dereferenced) addresses: every one of these fails validation on the host."""
    good = R.make_shape(1, 4, 16, 1, R.BF16, R.BF16, R.CANONICAL)
    res = R.make_shape(1, 4, 16, 1, R.BF16, R.BF16, R.RESTRICTED)
    A = 1 << 20
    assert _call_forward(lib, good, x=None) == R.ERR_INVALID_ARG
    assert _call_forward(lib, good, x=A + 8) == R.ERR_INVALID_ARG          # misaligned
    assert _call_forward(lib, good, rm=A, sp=A) == R.ERR_INVALID_ARG       # both reset forms
    assert _call_forward(lib, res, rm=A) == R.ERR_INVALID_ARG              # restricted + resets
    assert _call_forward(lib, res, h0=A) == R.ERR_INVALID_ARG              # restricted + h0
    bad = R.make_shape(1, 4, 12, 1, R.BF16, R.BF16, R.CANONICAL)
    assert _call_forward(lib, bad) == R.ERR_UNSUPPORTED
    bad = R.make_shape(1, 0, 16, 1, R.BF16, R.BF16, R.CANONICAL)
    assert _call_forward(lib, bad) == R.ERR_INVALID_ARG
    assert lib.rglru_sync_status(None, None) == R.ERR_INVALID_ARG


def test_step_host_validation(lib):
    """rglru_step checks its shape and pointers on the host (fake, never dereferenced
    addresses): T must be 1, restricted mode takes no resets, k is bounded."""
    A = 1 << 20
    P = lambda v: None if v is None else ctypes.c_void_p(v)

    def call(sh, reset=None, h_in=A, x=A):
        return lib.rglru_step(ctypes.byref(sh), P(x), P(A), None, P(A), None, P(A), P(reset),
                              P(h_in), P(A), P(A), None)
    assert call(R.make_shape(2, 2, 256, 2, R.BF16, R.BF16, R.CANONICAL)) == R.ERR_INVALID_ARG
    assert call(R.make_shape(2, 1, 256, 2, R.BF16, R.BF16, R.RESTRICTED),
                reset=A) == R.ERR_INVALID_ARG
    assert call(R.make_shape(2, 1, 256, 2, R.BF16, R.BF16, R.CANONICAL),
                x=A + 4) == R.ERR_INVALID_ARG
    assert call(R.make_shape(2, 1, 1024, 1, R.BF16, R.BF16, R.CANONICAL)) == R.ERR_UNSUPPORTED


def test_varlen_host_validation(lib):
    """The packed-sequence entry points check on the host (fake, never dereferenced
    addresses): one row, canonical mode, at least one sequence, the offsets array present,
    and a supported shape (bf16 with gate blocks a multiple of 16 up to 160, or float32 I/O)."""
    A = 1 << 20
    P = lambda v: None if v is None else ctypes.c_void_p(v)

    def fwd(sh, cu=A, S=3, saved=A):
        return lib.rglru_fused_forward_varlen(ctypes.byref(sh), P(A), P(A), None, P(A), None,
                                              P(A), P(cu), S, None, P(A), None, P(saved), None)

    def bwd(sh, cu=A, S=3, ws=A):
        return lib.rglru_fused_backward_varlen(ctypes.byref(sh), P(A), None, P(A), P(A), None,
                                               P(A), None, P(A), P(cu), S, None, P(A), P(A),
                                               P(A), None, P(A), None, P(A), None, P(ws), None)
    good = R.make_shape(1, 256, 256, 2, R.BF16, R.BF16, R.CANONICAL)
    for call in (fwd, bwd):
        assert call(R.make_shape(2, 256, 256, 2, R.BF16, R.BF16, R.CANONICAL)) == R.ERR_INVALID_ARG
        assert call(R.make_shape(1, 256, 256, 2, R.BF16, R.BF16, R.RESTRICTED)) == R.ERR_INVALID_ARG
        assert call(good, S=0) == R.ERR_INVALID_ARG
        assert call(good, cu=None) == R.ERR_INVALID_ARG
        # bf16 with gate blocks off the tensor-core routes (k = 24) has no packed path
        assert call(R.make_shape(1, 256, 192, 8, R.BF16, R.BF16, R.CANONICAL)) == R.ERR_UNSUPPORTED
    assert fwd(good, saved=None) == R.ERR_INVALID_ARG
    assert bwd(good, ws=None) == R.ERR_INVALID_ARG


def test_delta_rule_sizes_and_host_validation(lib):
    """Scratch queries and host-side checks of the delta-rule entry points (fake, never
    dereferenced addresses)."""
    A = 1 << 20
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    sh = R.make_delta_shape(2, 64, 2, 4, 64, 32, R.BF16)
    assert R.delta_rule_saved_bytes(sh, 2) == (2 * 64 // 16 + 2 * 2 + 1) * 4 * 64 * 32 * 4
    assert R.delta_rule_workspace_bytes(sh) == 2 * 2 * 64 * 4 * 64 * 4   # Hv > Hk
    assert R.delta_rule_workspace_bytes(R.make_delta_shape(2, 64, 4, 4, 64, 32)) == 0
    assert R.delta_rule_saved_bytes(R.make_delta_shape(2, 64, 2, 4, 48, 32), 2) == 0  # Dk 48
    assert R.delta_rule_saved_bytes(R.make_delta_shape(2, 64, 2, 4, 64, 256), 2) == 0  # Dv 256

    def fwd(shape, q=A, cu=None, N=2):
        return lib.delta_rule_forward(ctypes.byref(shape), P(q), P(A), P(A), P(A), P(A),
                                      ctypes.c_float(0.125), P(cu), N, None, P(A), None, P(A),
                                      None)
    assert fwd(sh, q=None) == R.ERR_INVALID_ARG
    assert fwd(sh, q=A + 4) == R.ERR_INVALID_ARG                     # misaligned
    assert fwd(sh, N=3) == R.ERR_INVALID_ARG                         # N must be B
    assert fwd(sh, cu=A) == R.ERR_INVALID_ARG                        # packed needs B = 1
    assert fwd(R.make_delta_shape(2, 64, 3, 4, 64, 32)) == R.ERR_INVALID_ARG   # Hv % Hk
    assert fwd(R.make_delta_shape(2, 64, 2, 4, 96, 32)) == R.ERR_UNSUPPORTED   # Dk 96
    assert fwd(R.make_delta_shape(2, 64, 2, 4, 64, 12)) == R.ERR_UNSUPPORTED   # 24-byte v rows


def test_state_qdq_host_validation(lib):
    A = 1 << 20
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    q = lambda st=A, out=A, n=2, dk=8, dv=8, bv=4: lib.delta_rule_state_fp8_qdq(P(st), P(out), n, dk, dv, bv, None)
    assert q(st=None) == R.ERR_INVALID_ARG
    assert q(out=A + 4) == R.ERR_INVALID_ARG
    assert q(n=0) == R.ERR_INVALID_ARG
    assert q(bv=0) == R.ERR_INVALID_ARG
