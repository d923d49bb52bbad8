"""GPU parity: every librglru entry point against the float64 oracle on identical seeded
inputs, at sizes the oracle finishes in seconds that still span several scan chunks, warp
tiles and GEMM tiles, with ragged tails and the method's degenerate cases."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, dev, host, mode_id, oracle_inputs, shape_for
from linear_recurrent_rnn_gb300 import build as B_
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.inputs import WORKLOADS, Workload, generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B_.build()
    R.lib()


def W_(name, B, T, W, k, io, mode, *args, **kw):
    return Workload(name, B, T, W, k, io, mode, *args, **kw)


SCAN_CASES = [
    (WORKLOADS[1], 1, None),
    (W_("f32-res", 2, 37, 64, 64, "f32", "restricted"), 2, None),
    (W_("bf16-res-ragged", 2, 100, 256, 256, "bf16", "restricted"), 3, None),
    (W_("bf16-res-ragged-g32", 2, 100, 256, 256, "bf16", "restricted"), 3, "f32"),
    (W_("bf16-can-W72", 3, 129, 72, 72, "bf16", "canonical", reset_p=0.1, h0_std=1.0), 4, None),
    (W_("bf16-can-packed", 2, 200, 128, 128, "bf16", "canonical", seg_len=(1, 40),
        continuation=True, h0_std=0.5), 5, "f32"),
    (W_("bf16-T1", 3, 1, 64, 64, "bf16", "canonical", h0_std=1.0), 6, None),
    (W_("bf16-T1-res", 2, 1, 64, 64, "bf16", "restricted"), 7, None),
    (W_("bf16-W8-T33", 2, 33, 8, 8, "bf16", "canonical", reset_p=0.2, h0_std=1.0), 8, None),
    (W_("bf16-all-reset", 2, 40, 64, 64, "bf16", "canonical", reset_p=1.0, h0_std=1.0), 9, None),
    (W_("f32-T17-noreset-h0", 2, 17, 32, 32, "f32", "canonical", h0_std=1.0), 10, None),
    (W_("bf16-longmem", 1, 600, 96, 96, "bf16", "canonical", (0.99, 0.9999), reset_p=1e-3), 11,
     "f32"),
]


def _gdt(sh):
    return R.TORCH_DT[sh.grad]


def run_scan_gpu(wl, inp, sh):
    d = {k: dev(v) for k, v in inp.items()}
    io = d["x"].dtype
    y = torch.empty_like(d["x"])
    hT = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    saved = R.alloc_saved(sh)
    ws = R.alloc_workspace(sh)
    R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], d["reset_mask"], d["segment_pos"],
                    d["h0"], y, hT, saved)
    gd = _gdt(sh)
    out = {"y": y, "hT": hT}
    out["dx"] = torch.empty(d["x"].shape, dtype=gd, device="cuda")
    out["dlr"] = torch.empty_like(out["dx"])
    out["dli"] = torch.empty_like(out["dx"])
    out["dLambda"] = torch.empty(wl.W, dtype=torch.float32, device="cuda")
    out["dh0"] = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    R.rglru_backward(sh, d["dy"], d["dhT"], d["x"], d["lr"], d["li"], d["Lambda"],
                     d["reset_mask"], d["segment_pos"], d["h0"], saved, out["dx"], out["dlr"],
                     out["dli"], out["dLambda"], out["dh0"], ws)
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK
    return {k: host(v) for k, v in out.items()}


@pytest.mark.parametrize("wl,seed,grad", SCAN_CASES, ids=[c[0].name + ("-g" + c[2] if c[2] else "") for c in SCAN_CASES])
def test_scan_forward_backward(wl, seed, grad):
    inp = generate(wl, seed, want_logits=True)
    sh = shape_for(wl, grad)
    got = run_scan_gpu(wl, inp, sh)
    o = oracle_inputs(inp)
    mode = mode_id(wl)
    y, hT = oracle.forward(mode, o["x"], o["lr"], o["li"], o["Lambda"], o["reset_mask"],
                           o["segment_pos"], o["h0"])
    g = oracle.backward(mode, o["x"], o["lr"], o["li"], o["Lambda"], o["dy"], o["dhT"],
                        o["reset_mask"], o["segment_pos"], o["h0"])
    gst = "f32" if sh.grad == R.F32 else "bf16"
    assert_close("y", got["y"], y, io=wl.io, kind="out")
    assert_close("hT", got["hT"], hT, io=wl.io, kind="out")
    for k in ("dx", "dlr", "dli"):
        assert_close(k, got[k], g[k], io=wl.io, kind="grad", stored=gst)
    assert_close("dLambda", got["dLambda"], g["dLambda"], io=wl.io, kind="grad")
    assert_close("dh0", got["dh0"], g["dh0"], io=wl.io, kind="grad")


GEMM_CASES = [
    (WORKLOADS[1], 21, None),
    (W_("bf16-k128", 2, 70, 256, 128, "bf16", "restricted"), 22, None),
    (W_("bf16-k160", 1, 150, 320, 160, "bf16", "restricted"), 23, "f32"),
    (W_("bf16-k64", 1, 33, 192, 64, "bf16", "restricted"), 24, None),
    (W_("bf16-k16-T1", 1, 1, 32, 16, "bf16", "restricted"), 25, None),
    # tensor-core projections: k = 160 (dW of one matrix per CTA, two 128-channel row blocks),
    # k = 48 (accumulators padded to 64 columns), and more row tiles than CTAs per gate block
    # so that the operand rings and TMEM buffers turn over
    (W_("bf16-k160-g16", 1, 150, 320, 160, "bf16", "restricted"), 26, None),
    (W_("bf16-k48", 1, 300, 192, 48, "bf16", "restricted"), 27, None),
    (W_("bf16-k128-multi", 1, 1500, 2048, 128, "bf16", "restricted"), 28, None),
    (W_("bf16-k160-multi", 2, 4000, 480, 160, "bf16", "restricted"), 29, None),
    # float32-stored gradients on the tensor cores (split into bf16 hi + lo planes), with the
    # dx and dW kernels side by side
    (W_("bf16-k128-multi-g32", 1, 1500, 2048, 128, "bf16", "restricted"), 30, "f32"),
]


@pytest.mark.parametrize("wl,seed,grad", GEMM_CASES, ids=[c[0].name for c in GEMM_CASES])
def test_gate_proj_and_backward(wl, seed, grad):
    inp = generate(wl, seed, want_dlogits=True)
    sh = shape_for(wl, grad)
    d = {k: dev(v) for k, v in inp.items()}
    lr = torch.empty_like(d["x"])
    li = torch.empty_like(d["x"])
    ba = torch.randn(wl.W, generator=torch.Generator().manual_seed(seed)).mul_(0.1)
    bx = torch.randn(wl.W, generator=torch.Generator().manual_seed(seed + 1)).mul_(0.1)
    R.rglru_gate_proj(sh, d["x"], d["Wa"], dev(ba), d["Wx"], dev(bx), lr, li)
    o = oracle_inputs(inp)
    rl, ri = oracle.gate_proj(o["x"], o["Wa"], ba.double().numpy(), o["Wx"], bx.double().numpy())
    assert_close("lr", host(lr), rl, io=wl.io, kind="out")
    assert_close("li", host(li), ri, io=wl.io, kind="out")

    gd = _gdt(sh)
    dlr = inp["dlr"].to(gd)
    dli = inp["dli"].to(gd)
    dx0 = torch.randn(inp["x"].shape, generator=torch.Generator().manual_seed(seed + 2)).to(gd)
    dx = dev(dx0.clone())
    dWa = torch.empty(wl.nblk, wl.k, wl.k, dtype=torch.float32, device="cuda")
    dWx = torch.empty_like(dWa)
    dba = torch.empty(wl.W, dtype=torch.float32, device="cuda")
    dbx = torch.empty_like(dba)
    ws = R.alloc_workspace(sh)
    R.rglru_gate_proj_backward(sh, dev(dlr), dev(dli), d["x"], d["Wa"], d["Wx"], dx, dWa, dba,
                               dWx, dbx, ws)
    torch.cuda.synchronize()
    p = oracle.gate_proj_backward(o["x"], o["Wa"], o["Wx"], dlr.double().numpy(),
                                  dli.double().numpy(), dx_in=dx0.double().numpy())
    gst = "f32" if sh.grad == R.F32 else "bf16"
    assert_close("dx", host(dx), p["dx"], io=wl.io, kind="grad", stored=gst)
    for k, v in (("dWa", dWa), ("dWx", dWx), ("dba", dba), ("dbx", dbx)):
        assert_close(k, host(v), p[k], io=wl.io, kind="grad")


def test_gate_proj_backward_deterministic():
    """At a shape where the dx and dW kernels run side by side (the dW grid launched as a
    programmatic dependent of the dx grid), two calls give the same bits: dx per row tile and
    the dW partial sums in a fixed order do not depend on how the two grids overlap."""
    wl = W_("det-proj", 2, 1024, 2048, 128, "bf16", "restricted")
    inp = generate(wl, 45, want_dlogits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    outs = []
    for _ in range(2):
        dx = torch.zeros_like(d["x"])
        dWa = torch.empty(wl.nblk, wl.k, wl.k, dtype=torch.float32, device="cuda")
        dWx = torch.empty_like(dWa)
        dba = torch.empty(wl.W, dtype=torch.float32, device="cuda")
        dbx = torch.empty_like(dba)
        ws = R.alloc_workspace(sh)
        R.rglru_gate_proj_backward(sh, d["dlr"], d["dli"], d["x"], d["Wa"], d["Wx"], dx, dWa,
                                   dba, dWx, dbx, ws)
        outs.append((dx, dWa, dWx, dba, dbx))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


FUSED_CASES = [
    (WORKLOADS[1], 31, None),
    (W_("bf16-res-k128", 2, 100, 256, 128, "bf16", "restricted"), 32, None),
    (W_("bf16-res-k128-g32", 2, 100, 256, 128, "bf16", "restricted"), 32, "f32"),
    (W_("bf16-packed-k160", 2, 150, 320, 160, "bf16", "canonical", seg_len=(1, 60),
        continuation=True, h0_std=1.0), 33, "f32"),
    (W_("bf16-T1-k128", 2, 1, 128, 128, "bf16", "canonical", h0_std=1.0), 34, None),
    (W_("bf16-reset-k64", 1, 70, 128, 64, "bf16", "canonical", reset_p=0.05, reset_t0=True,
        h0_std=1.0), 35, None),
    # short memories: a^c down to 0.05, so many channels leave the near regime (la <= -1/8)
    # and the tensor-core kernels take their general path with the exponential decay
    (W_("bf16-far-k128", 2, 150, 256, 128, "bf16", "canonical", (0.05, 0.95), reset_p=0.05,
        h0_std=1.0), 36, "f32"),
    (W_("bf16-far-res-k128", 2, 130, 256, 128, "bf16", "restricted", (0.2, 0.9)), 37, None),
    # gate blocks the fused kernels do not take: tensor-core projections around the CUDA-core
    # scan, bf16-stored gradients
    (W_("bf16-res-k160", 2, 300, 480, 160, "bf16", "restricted"), 38, None),
    (W_("bf16-can-k96", 2, 200, 192, 96, "bf16", "canonical", reset_p=0.02, h0_std=1.0), 39,
     None),
]


def run_fused_gpu(wl, inp, sh, ba=None, bx=None):
    d = {k: dev(v) for k, v in inp.items()}
    ba = d["ba"] if ba is None else dev(ba)
    bx = d["bx"] if bx is None else dev(bx)
    y = torch.empty_like(d["x"])
    hT = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    saved = R.alloc_saved(sh)
    ws = R.alloc_workspace(sh)
    R.rglru_fused_forward(sh, d["x"], d["Wa"], ba, d["Wx"], bx, d["Lambda"], d["reset_mask"],
                          d["segment_pos"], d["h0"], y, hT, saved)
    out = {"y": y, "hT": hT}
    out["dx"] = torch.empty(d["x"].shape, dtype=_gdt(sh), device="cuda")
    for k in ("dWa", "dWx"):
        out[k] = torch.empty(wl.nblk, wl.k, wl.k, dtype=torch.float32, device="cuda")
    for k in ("dba", "dbx", "dLambda"):
        out[k] = torch.empty(wl.W, dtype=torch.float32, device="cuda")
    out["dh0"] = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    R.rglru_fused_backward(sh, d["dy"], d["dhT"], d["x"], d["Wa"], ba, d["Wx"], bx,
                           d["Lambda"], d["reset_mask"], d["segment_pos"], d["h0"], saved,
                           out["dx"], out["dWa"], out["dba"], out["dWx"], out["dbx"],
                           out["dLambda"], out["dh0"], ws)
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK
    return out


def check_fused(wl, inp, got, gst, ba=None, bx=None, sl=slice(None)):
    o = oracle_inputs(inp)
    ba = o["ba"] if ba is None else ba
    bx = o["bx"] if bx is None else bx
    mode = mode_id(wl)
    y, hT = oracle.fused_forward(mode, o["x"], o["Wa"], ba, o["Wx"], bx, o["Lambda"],
                                 o["reset_mask"], o["segment_pos"], o["h0"])
    g = oracle.fused_backward(mode, o["x"], o["Wa"], ba, o["Wx"], bx, o["Lambda"], o["dy"],
                              o["dhT"], o["reset_mask"], o["segment_pos"], o["h0"])
    assert_close("y", got["y"], y, io=wl.io, kind="out")
    assert_close("hT", got["hT"], hT, io=wl.io, kind="out")
    assert_close("dx", got["dx"], g["dx"], io=wl.io, kind="grad", stored=gst)
    for k in ("dWa", "dWx", "dba", "dbx", "dLambda", "dh0"):
        assert_close(k, got[k], g[k], io=wl.io, kind="grad")


def test_unfused_step_on_one_workspace():
    """The unfused training step on one workspace (scan backward, then the projection
    backward): the status word the scan leaves in the workspace survives the projection
    backward's partial sums, and those give bitwise the gradients of a run on a workspace of
    their own."""
    wl = W_("bf16-unfused", 2, 130, 256, 128, "bf16", "canonical", reset_p=0.05, h0_std=1.0)
    inp = generate(wl, 31, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    hT = torch.empty(wl.B, wl.W, device="cuda")
    dx, dlr, dli = (torch.empty_like(d["x"]) for _ in range(3))
    dL = torch.empty(wl.W, device="cuda")
    dh0 = torch.empty(wl.B, wl.W, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], d["reset_mask"],
                    d["segment_pos"], d["h0"], y, hT, saved)
    R.rglru_backward(sh, d["dy"], d["dhT"], d["x"], d["lr"], d["li"], d["Lambda"],
                     d["reset_mask"], d["segment_pos"], d["h0"], saved, dx, dlr, dli, dL, dh0, ws)
    grads = []
    for w in (ws, R.alloc_workspace(sh)):
        dxw = dx.clone()
        g = [torch.empty(wl.nblk, wl.k, wl.k, device="cuda") for _ in range(2)]
        b = [torch.empty(wl.W, device="cuda") for _ in range(2)]
        R.rglru_gate_proj_backward(sh, dlr, dli, d["x"], d["Wa"], d["Wx"], dxw, g[0], b[0], g[1],
                                   b[1], w)
        grads.append([dxw] + g + b)
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK
    for a, b in zip(*grads):
        assert torch.equal(a, b)


@pytest.mark.parametrize("wl,seed,grad", FUSED_CASES,
                         ids=[c[0].name + ("-g" + c[2] if c[2] else "") for c in FUSED_CASES])
def test_fused_forward_backward(wl, seed, grad):
    inp = generate(wl, seed)
    sh = shape_for(wl, grad)
    ba = torch.randn(wl.W, generator=torch.Generator().manual_seed(seed)).mul_(0.1)
    bx = torch.randn(wl.W, generator=torch.Generator().manual_seed(seed + 1)).mul_(0.1)
    got = {k: host(v) for k, v in run_fused_gpu(wl, inp, sh, ba, bx).items()}
    check_fused(wl, inp, got, "f32" if sh.grad == R.F32 else "bf16",
                ba.double().numpy(), bx.double().numpy())


def test_fused_path_names_the_kernels():
    """The fused calls run the one-kernel tensor-core pair for bf16 gate blocks of 128, the
    tensor-core projections around the CUDA-core scan for other bf16 gate blocks (multiples of
    16 up to 160), and the float32 SIMT projections for float32 I/O."""
    assert R.fused_path(R.make_shape(4, 2048, 2048, 16, R.BF16)).startswith("fused")
    p5 = R.fused_path(R.make_shape(8, 4096, 4000, 25, R.BF16))
    assert p5.startswith("composed") and "tcgen05" in p5
    assert "SIMT" in R.fused_path(R.make_shape(1, 64, 128, 2, R.F32))
    assert "SIMT" in R.fused_path(R.make_shape(1, 64, 8 * 24, 8, R.BF16))  # k = 24


def test_fused_forward_is_one_tensor_core_kernel():
    """For bf16 I/O with 128-wide gate blocks the fused forward is a single kernel launch (the
    tcgen05 kernel), not the composed projection + scan pair."""
    wl = W_("one-kernel", 1, 64, 256, 128, "bf16", "restricted")
    inp = generate(wl, 44)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    saved = R.alloc_saved(sh)
    n0 = R.rglru_kernel_launches()
    R.rglru_fused_forward(sh, d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], None,
                          None, None, y, None, saved)
    assert R.rglru_kernel_launches() - n0 == 1
    assert R.rglru_sync_status(saved) == R.OK


@pytest.mark.parametrize("case", ["restricted", "canonical"])
def test_fused_step_replayed_from_cuda_graph(case):
    """The fused forward and backward calls captured once in a CUDA graph (as the headline
    step is timed) and replayed twice: each replay clears its look-back slots itself, so both
    give bitwise the results of the calls issued directly, which match the oracle."""
    if case == "restricted":
        wl = W_("graph-res", 2, 260, 256, 128, "bf16", "restricted")
    else:
        wl = W_("graph-can", 2, 200, 256, 128, "bf16", "canonical", reset_p=0.02, h0_std=1.0)
    inp = generate(wl, 45)
    sh = shape_for(wl)
    direct = run_fused_gpu(wl, inp, sh)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    hT = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    out = {"y": y, "hT": hT, "dx": torch.empty(d["x"].shape, dtype=_gdt(sh), device="cuda")}
    for k in ("dWa", "dWx"):
        out[k] = torch.empty(wl.nblk, wl.k, wl.k, dtype=torch.float32, device="cuda")
    for k in ("dba", "dbx", "dLambda"):
        out[k] = torch.empty(wl.W, dtype=torch.float32, device="cuda")
    out["dh0"] = torch.empty(wl.B, wl.W, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    gs = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        R.rglru_fused_forward(sh, d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"],
                              d["reset_mask"], d["segment_pos"], d["h0"], y, hT, saved, gs)
        R.rglru_fused_backward(sh, d["dy"], d["dhT"], d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"],
                               d["Lambda"], d["reset_mask"], d["segment_pos"], d["h0"], saved,
                               out["dx"], out["dWa"], out["dba"], out["dWx"], out["dbx"],
                               out["dLambda"], out["dh0"], ws, gs)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert R.rglru_sync_status(saved) == R.OK
        assert R.rglru_sync_status(ws) == R.OK
        for k in direct:
            assert torch.equal(out[k], direct[k]), k
    check_fused(wl, inp, {k: host(v) for k, v in out.items()}, "bf16")


def test_fused_deterministic():
    wl = W_("det", 2, 300, 256, 128, "bf16", "canonical", reset_p=0.01, h0_std=1.0)
    inp = generate(wl, 41)
    sh = shape_for(wl)
    a = run_fused_gpu(wl, inp, sh)
    b = run_fused_gpu(wl, inp, sh)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_outputs_stay_in_bounds():
    """Canary: the elements just past every output buffer are never written."""
    wl = W_("canary", 1, 45, 72, 72, "bf16", "canonical", reset_p=0.1, h0_std=1.0)
    inp = generate(wl, 42, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    N = wl.B * wl.T * wl.W
    pad = 512
    sentinel = 12345.0

    def buf(n, dt):
        t = torch.full((n + pad,), sentinel, dtype=dt, device="cuda")
        return t, t[:n]

    yb, y = buf(N, torch.bfloat16)
    hb, hT = buf(wl.B * wl.W, torch.float32)
    saved = R.alloc_saved(sh)
    ws = R.alloc_workspace(sh)
    R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], d["reset_mask"], None, d["h0"],
                    y, hT, saved)
    bufs = [buf(N, torch.bfloat16) for _ in range(3)] + [buf(wl.W, torch.float32),
                                                          buf(wl.B * wl.W, torch.float32)]
    R.rglru_backward(sh, d["dy"], d["dhT"], d["x"], d["lr"], d["li"], d["Lambda"],
                     d["reset_mask"], None, d["h0"], saved, bufs[0][1], bufs[1][1], bufs[2][1],
                     bufs[3][1], bufs[4][1], ws)
    torch.cuda.synchronize()
    for full, n in [(yb, N), (hb, wl.B * wl.W)] + [(b[0], b[1].numel()) for b in bufs]:
        assert torch.all(full[n:] == torch.tensor(sentinel, dtype=full.dtype, device="cuda"))


def test_lookback_timeout_is_reported():
    """The CUDA-core scan (float32 I/O): a tile that never publishes makes its successor's
    bounded wait run out; the call still finishes and the status word reports the timeout.
    Afterwards the defaults are back."""
    wl = W_("timeout", 1, 128, 64, 64, "f32", "restricted")
    inp = generate(wl, 43, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    saved = R.alloc_saved(sh)
    R.rglru_debug_lookback(2000, 5)
    try:
        R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], None, None, None, y, None, saved)
        assert R.rglru_sync_status(saved) == R.ERR_TIMEOUT
    finally:
        R.rglru_debug_lookback(0, -1)
    R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], None, None, None, y, None, saved)
    assert R.rglru_sync_status(saved) == R.OK
    o = oracle_inputs(inp)
    yr, _ = oracle.forward(oracle.RESTRICTED, o["x"], o["lr"], o["li"], o["Lambda"])
    assert_close("y", host(y), yr, io="f32", kind="out")


@pytest.mark.parametrize("which", ["forward", "backward"])
def test_given_logits_lookback_timeout_is_reported(which):
    """rglru_forward / rglru_backward with bf16 I/O run the tensor-core scan kernels with the
    logits given: a tile that never publishes makes the later chunks' bounded look-back waits
    run out; the call finishes and the status word of its scratch reports the timeout.  One
    128-channel slice and 12 chunks, so every tile has a CTA of its own and the dropped tile
    (chunk 5) lies inside its successors' look-back windows."""
    wl = W_("timeout-lg", 1, 12 * 64, 128, 128, "bf16", "restricted")
    inp = generate(wl, 46, want_logits=True)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    dx, dlr, dli = (torch.empty_like(d["x"]) for _ in range(3))
    dL = torch.empty(wl.W, device="cuda")

    def fwd():
        R.rglru_forward(sh, d["x"], d["lr"], d["li"], d["Lambda"], None, None, None, y, None,
                        saved)

    def bwd():
        R.rglru_backward(sh, d["dy"], None, d["x"], d["lr"], d["li"], d["Lambda"], None, None,
                         None, saved, dx, dlr, dli, dL, None, ws)

    if which == "backward":
        fwd()
        assert R.rglru_sync_status(saved) == R.OK
    R.rglru_debug_lookback(2000, 5)
    try:
        (fwd if which == "forward" else bwd)()
        assert R.rglru_sync_status(saved if which == "forward" else ws) == R.ERR_TIMEOUT
    finally:
        R.rglru_debug_lookback(0, -1)
    fwd()
    bwd()
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK
    o = oracle_inputs(inp)
    yr, _ = oracle.forward(oracle.RESTRICTED, o["x"], o["lr"], o["li"], o["Lambda"])
    assert_close("y", host(y), yr, io="bf16", kind="out")


@pytest.mark.parametrize("which", ["forward", "backward"])
def test_fused_lookback_timeout_is_reported(which):
    """The fused tensor-core kernels: a tile that never publishes its aggregate and carry makes
    the later chunks' bounded look-back waits run out; the call finishes and the status word of
    its scratch reports the timeout.  One gate block of 128 channels and 12 chunks, so every
    tile has a CTA of its own and the dropped tile (chunk 5) lies inside its successors'
    look-back windows."""
    wl = W_("timeout-fused", 1, 12 * 64, 128, 128, "bf16", "restricted")
    inp = generate(wl, 45)
    sh = shape_for(wl)
    d = {k: dev(v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    saved = R.alloc_saved(sh)
    ws = R.alloc_workspace(sh)
    dx = torch.empty_like(d["x"])
    dW = [torch.empty(1, 128, 128, device="cuda") for _ in range(2)]
    dv = [torch.empty(128, device="cuda") for _ in range(3)]

    def fwd():
        R.rglru_fused_forward(sh, d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"], None,
                              None, None, y, None, saved)

    def bwd():
        R.rglru_fused_backward(sh, d["dy"], None, d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"],
                               d["Lambda"], None, None, None, saved, dx, dW[0], dv[0], dW[1],
                               dv[1], dv[2], None, ws)

    if which == "backward":
        fwd()
        assert R.rglru_sync_status(saved) == R.OK
    R.rglru_debug_lookback(2000, 5)
    try:
        (fwd if which == "forward" else bwd)()
        buf = saved if which == "forward" else ws
        assert R.rglru_sync_status(buf) == R.ERR_TIMEOUT
    finally:
        R.rglru_debug_lookback(0, -1)
    fwd()
    bwd()
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK


def test_invalid_arguments_rejected_on_gpu():
    wl = W_("bad", 1, 8, 64, 64, "bf16", "restricted")
    sh = shape_for(wl)
    x = torch.zeros(1, 8, 64, dtype=torch.bfloat16, device="cuda")
    L = torch.zeros(64, device="cuda")
    saved = R.alloc_saved(sh)
    rm = torch.zeros(1, 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(R.RglruError) as e:   # restricted mode takes no resets
        R.rglru_forward(sh, x, x, x, L, rm, None, None, x, None, saved)
    assert e.value.status == R.ERR_INVALID_ARG
    P = ctypes.c_void_p
    st = R.lib().rglru_forward(ctypes.byref(sh), P(x.data_ptr() + 2), P(x.data_ptr()),
                               P(x.data_ptr()), P(L.data_ptr()), None, None, None, P(x.data_ptr()),
                               None, P(saved.data_ptr()), None)
    assert st == R.ERR_INVALID_ARG   # misaligned x
