"""rglru_forward_noalloc: the forward for callers that may not allocate device memory (code
inside another owner's stream capture, under a fixed memory pool, in an allocation-free
real-time loop, or in a plugin handed only its inputs and outputs).  It keeps its look-back
scratch in the library's static per-GPU array instead of a caller `saved` buffer.

Checked through the C ABI on two calls in a row with different shapes and modes (so the
second call sees the first call's leftovers in the shared array): against rglru_forward, the
entry point that takes a caller buffer and runs the same kernel on the same inputs, bit for
bit; and against the float64 oracle within the tolerance of the other parity tests.  A
dropped look-back publish must show up in rglru_forward_noalloc_status.  This file is
collected last so that a failure here leaves every other test already run."""
import pytest
import torch

import oracle
from helpers import assert_close, dev, host, mode_id, oracle_inputs, shape_for
from linear_recurrent_rnn_gb300 import build as B_
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.inputs import Workload, generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B_.build()
    R.lib()


def _both(wl, seed):
    inp = generate(wl, seed, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    args = (d["x"], d["lr"], d["li"], d["Lambda"], d["reset_mask"], d["segment_pos"], d["h0"])
    y_ref = torch.empty_like(d["x"])
    h_ref = torch.empty(wl.B, wl.W, device="cuda")
    saved = R.alloc_saved(sh)
    R.rglru_forward(sh, *args, y_ref, h_ref, saved)
    assert R.rglru_sync_status(saved) == R.OK
    y = torch.full_like(d["x"], float("nan"))
    h = torch.full((wl.B, wl.W), float("nan"), device="cuda")
    R.rglru_forward_noalloc(sh, *args, y, h)
    assert R.rglru_forward_noalloc_status() == R.OK
    return inp, y, h, y_ref, h_ref


def test_noalloc_forward_matches_forward_twice():
    first = Workload("noalloc-1", 2, 300, 256, 128, "bf16", "canonical", reset_p=0.02,
                     h0_std=1.0)
    second = Workload("noalloc-2", 3, 1000, 128, 128, "bf16", "restricted")
    for wl, seed in ((first, 51), (second, 52)):
        inp, y, h, y_ref, h_ref = _both(wl, seed)
        # the same kernel on the same inputs: equal bit for bit
        assert torch.equal(y, y_ref)
        assert torch.equal(h, h_ref)
        o = oracle_inputs(inp)
        yo, ho = oracle.forward(mode_id(wl), o["x"], o["lr"], o["li"], o["Lambda"],
                                o["reset_mask"], o["segment_pos"], o["h0"])
        assert_close("y", host(y), yo, io=wl.io, kind="out")
        assert_close("hT", host(h), ho, io=wl.io, kind="out")


def test_noalloc_timeout_is_reported():
    """A tile that never publishes makes its successors' bounded waits run out; the call
    finishes, and the status query of the static scratch reports the timeout.  The next call
    clears the word."""
    # 12 chunks of one 128-channel slice: every tile has a CTA of its own, and the dropped
    # tile (chunk 5) lies inside its successors' look-back windows
    wl = Workload("noalloc-timeout", 1, 12 * 64, 128, 128, "bf16", "restricted")
    inp = generate(wl, 43, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    R.rglru_debug_lookback(2000, 5)
    try:
        R.rglru_forward_noalloc(sh, d["x"], d["lr"], d["li"], d["Lambda"], None, None, None, y,
                                None)
        assert R.rglru_forward_noalloc_status() == R.ERR_TIMEOUT
    finally:
        R.rglru_debug_lookback(0, -1)
    R.rglru_forward_noalloc(sh, d["x"], d["lr"], d["li"], d["Lambda"], None, None, None, y, None)
    assert R.rglru_forward_noalloc_status() == R.OK
    o = oracle_inputs(inp)
    yo, _ = oracle.forward(oracle.RESTRICTED, o["x"], o["lr"], o["li"], o["Lambda"])
    assert_close("y", host(y), yo, io="bf16", kind="out")


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    wl = Workload("too-big", 8, 4096, 4000, 160, "bf16", "restricted")
    sh = shape_for(wl)
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected first
    L = torch.empty(16, device="cuda")
    with pytest.raises(R.RglruError) as e:
        R.rglru_forward_noalloc(sh, x, x, x, L, None, None, None, x, None)
    assert e.value.status == R.ERR_UNSUPPORTED
