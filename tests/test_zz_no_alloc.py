"""rglru_forward_noalloc: the forward for callers that may not allocate device memory (code
inside another owner's stream capture, under a fixed memory pool, in an allocation-free
real-time loop, or in a plugin handed only its inputs and outputs).  It keeps its look-back
scratch in the library's static per-GPU array instead of a caller `saved` buffer.

Checked through the C ABI against rglru_forward, the entry point that takes a caller buffer,
on two calls in a row with different shapes and modes (so the second call sees the first
call's leftovers in the shared array), within the tolerance the other parity tests use.
This file is collected last so that a failure here leaves every other test already run."""
import pytest
import torch

from helpers import assert_close, dev, host, shape_for
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
    y = torch.full_like(d["x"], float("nan"))
    h = torch.full((wl.B, wl.W), float("nan"), device="cuda")
    R.rglru_forward_noalloc(sh, *args, y, h)
    torch.cuda.synchronize()
    return y, h, y_ref, h_ref


def test_noalloc_forward_matches_forward_twice():
    first = Workload("noalloc-1", 2, 300, 256, 128, "bf16", "canonical", reset_p=0.02,
                     h0_std=1.0)
    second = Workload("noalloc-2", 3, 1000, 128, 128, "bf16", "restricted")
    for wl, seed in ((first, 51), (second, 52)):
        y, h, y_ref, h_ref = _both(wl, seed)
        assert_close("y", host(y), host(y_ref), io=wl.io, kind="out")
        assert_close("hT", host(h), host(h_ref), io=wl.io, kind="out")


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    wl = Workload("too-big", 8, 4096, 4000, 160, "bf16", "restricted")
    sh = shape_for(wl)
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected first
    L = torch.empty(16, device="cuda")
    with pytest.raises(R.RglruError) as e:
        R.rglru_forward_noalloc(sh, x, x, x, L, None, None, None, x, None)
    assert e.value.status == R.ERR_UNSUPPORTED
