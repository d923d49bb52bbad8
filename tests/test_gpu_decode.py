"""The decode step (rglru_step) against the float64 oracle: one token from carried states
equals the layer's forward with T = 1 and h0 = the carried state; and a loop of steps that
feeds each step's state to the next reproduces the forward over the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.inputs import Workload, generate

from helpers import assert_close, dev, host, mode_id, oracle_inputs, shape_for

pytestmark = pytest.mark.gpu

# B spans one CTA row group (32 rows) and a ragged tail; k = 96 and 160 are not powers of two.
STEP_CASES = [
    (Workload("step-bf16-canonical", 37, 1, 256, 128, "bf16", "canonical", reset_p=0.3,
              h0_std=1.0), 3),
    (Workload("step-bf16-restricted", 5, 1, 192, 96, "bf16", "restricted"), 4),
    (Workload("step-f32-canonical", 70, 1, 128, 64, "f32", "canonical", reset_p=0.2,
              h0_std=0.5), 5),
    (Workload("step-bf16-k160", 1, 1, 320, 160, "bf16", "canonical", h0_std=1.0), 6),
    # batches of 64 and more take the tensor-core step (128-row tiles: one ragged, two)
    (Workload("step-tc-bf16-canonical", 200, 1, 256, 128, "bf16", "canonical", reset_p=0.3,
              h0_std=1.0), 7),
    (Workload("step-tc-bf16-k160", 70, 1, 320, 160, "bf16", "restricted"), 8),
    (Workload("step-tc-bf16-k64", 128, 1, 192, 64, "bf16", "canonical", h0_std=0.5), 9),
]


def _step(sh, d, x, reset, h_in, io_dtype):
    B, W = x.shape
    y = torch.empty(B, W, dtype=io_dtype, device="cuda")
    h_out = torch.empty(B, W, dtype=torch.float32, device="cuda")
    R.rglru_step(sh, x, d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], reset, h_in, y, h_out)
    return y, h_out


@pytest.mark.parametrize("wl,seed", STEP_CASES, ids=[c[0].name for c in STEP_CASES])
def test_step_matches_forward_of_one_token(wl, seed):
    inp = generate(wl, seed)
    d = {k: dev(v) if isinstance(v, torch.Tensor) else v for k, v in inp.items()}
    sh = shape_for(wl)
    x = d["x"].reshape(wl.B, wl.W).contiguous()
    reset = None if d.get("reset_mask") is None else d["reset_mask"].reshape(wl.B).contiguous()
    y, h_out = _step(sh, d, x, reset, d.get("h0"), d["x"].dtype)
    torch.cuda.synchronize()
    o = oracle_inputs(inp)
    yr, hr = oracle.fused_forward(mode_id(wl), o["x"], o["Wa"], o["ba"], o["Wx"], o["bx"],
                                  o["Lambda"], o["reset_mask"], None, o["h0"])
    assert_close("y", host(y), yr.reshape(wl.B, wl.W), io=wl.io, kind="out")
    assert_close("h_out", host(h_out), hr, io=wl.io, kind="out")


@pytest.mark.parametrize("B", [3, 96])
def test_decode_loop_reproduces_forward(B):
    """T steps with the state updated in place equal the forward over T tokens (B = 96: the
    tensor-core step)."""
    wl = Workload("decode-loop", B, 40, 256, 128, "bf16", "canonical", reset_p=0.05, h0_std=1.0)
    inp = generate(wl, 11)
    d = {k: dev(v) if isinstance(v, torch.Tensor) else v for k, v in inp.items()}
    sh = R.make_shape(wl.B, 1, wl.W, wl.nblk, R.BF16, R.BF16, R.CANONICAL)
    h = d["h0"].clone()
    ys = []
    for t in range(wl.T):
        x = d["x"][:, t, :].contiguous()
        reset = d["reset_mask"][:, t].contiguous()
        y = torch.empty(wl.B, wl.W, dtype=torch.bfloat16, device="cuda")
        R.rglru_step(sh, x, d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], reset, h, y, h)
        ys.append(y)
    torch.cuda.synchronize()
    o = oracle_inputs(inp)
    yr, hr = oracle.fused_forward(R.CANONICAL, o["x"], o["Wa"], o["ba"], o["Wx"], o["bx"],
                                  o["Lambda"], o["reset_mask"], None, o["h0"])
    assert_close("y", np.stack([host(y) for y in ys], axis=1), yr, io="bf16", kind="out")
    assert_close("hT", host(h), hr, io="bf16", kind="out")


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_decode_steps_back_to_back(graph):
    """The steps of a decode loop with nothing launched between them (every token's x, reset
    flags and y prepared beforehand, the state updated in place), issued directly or captured
    in a CUDA graph and replayed: each step reads the state the step before it wrote, so the
    loop equals the forward over the whole sequence."""
    wl = Workload("decode-back-to-back", 96, 24, 256, 128, "bf16", "canonical", reset_p=0.05,
                  h0_std=1.0)
    inp = generate(wl, 12)
    d = {k: dev(v) if isinstance(v, torch.Tensor) else v for k, v in inp.items()}
    sh = R.make_shape(wl.B, 1, wl.W, wl.nblk, R.BF16, R.BF16, R.CANONICAL)
    xs = [d["x"][:, t, :].contiguous() for t in range(wl.T)]
    rs = [d["reset_mask"][:, t].contiguous() for t in range(wl.T)]
    ys = [torch.empty(wl.B, wl.W, dtype=torch.bfloat16, device="cuda") for _ in range(wl.T)]
    h = d["h0"].clone()

    def loop(s=None):
        for t in range(wl.T):
            R.rglru_step(sh, xs[t], d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], rs[t], h,
                         ys[t], h, s)

    torch.cuda.synchronize()
    if graph:
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            loop(gs)
        torch.cuda.current_stream().wait_stream(gs)
        h.copy_(d["h0"])
        torch.cuda.synchronize()
        g.replay()
    else:
        loop()
    torch.cuda.synchronize()
    o = oracle_inputs(inp)
    yr, hr = oracle.fused_forward(R.CANONICAL, o["x"], o["Wa"], o["ba"], o["Wx"], o["bx"],
                                  o["Lambda"], o["reset_mask"], None, o["h0"])
    assert_close("y", np.stack([host(y) for y in ys], axis=1), yr, io="bf16", kind="out")
    assert_close("hT", host(h), hr, io="bf16", kind="out")
