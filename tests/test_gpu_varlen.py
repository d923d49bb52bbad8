"""Packed variable-length sequences (rglru_fused_forward_varlen / _backward_varlen) against the
float64 oracle run on every sequence as a row of its own: sequence s continues from h0[s]
without a reset, its final state is hT[s], dhT[s] joins the gradient at its last token and
dh0[s] is its initial-state gradient; the parameter gradients are the sums over sequences.
Lengths include empty sequences (hT = h0, dh0 = dhT), a leading empty one (the next sequence
starts at token 0), a sequence of one token, and starts inside and across 64-token chunks;
bf16 I/O on the tensor-core kernels, float32 I/O on the CUDA-core scan."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.inputs import Workload, as_f64, generate

from helpers import assert_close, dev, host

pytestmark = pytest.mark.gpu

CASES = [
    ([0, 1, 0, 70, 64, 33, 0, 130, 5, 1], (0.9, 0.999), 41, "bf16", 256, 128),
    ([200, 3, 97], (0.05, 0.95), 42, "bf16", 256, 128),   # short memories: general decay too
    ([31, 1, 64, 129, 0, 2], (0.5, 0.999), 43, "f32", 256, 128),   # float32 dx
    # gate blocks of 160 (tensor-core projections around the packed scan; the last 128-channel
    # slice of W = 320 is partial) and of 48
    ([0, 1, 0, 70, 64, 33, 0, 130, 5, 1], (0.9, 0.999), 44, "bf16", 320, 160),
    ([95, 0, 3, 200], (0.5, 0.999), 45, "f32", 192, 48),
    # float32 I/O: the CUDA-core scan over the packed sequences (16-token chunks, so starts
    # fall at every offset within a chunk and inside both of its halves)
    ([0, 1, 0, 70, 64, 33, 0, 130, 5, 1], (0.9, 0.999), 46, "f32", 256, 128, "f32"),
    ([17, 8, 9, 1, 40, 0, 3], (0.05, 0.999), 47, "f32", 96, 24, "f32"),
    # long sequences: the look-back crosses many 16-token chunks inside each sequence (memories
    # of up to ~100 tokens: with longer ones the float32 sums over thousands of tokens alone
    # exceed the 1e-5 bound, on any float32 arithmetic)
    ([700, 1, 650, 0, 901], (0.5, 0.99), 48, "f32", 128, 64, "f32"),
]
CASES = [c if len(c) == 7 else c + ("bf16",) for c in CASES]


@pytest.mark.parametrize("lengths,u_range,seed,grad,W,k,io", CASES,
                         ids=["mixed", "far", "f32grad", "k160", "k48-f32grad", "f32io",
                              "f32io-k24-far", "f32io-long"])
def test_varlen_matches_per_sequence_oracle(lengths, u_range, seed, grad, W, k, io):
    T = int(sum(lengths))
    S = len(lengths)
    wl = Workload("varlen", 1, T, W, k, io, "canonical", u_range, h0_std=1.0)
    inp = generate(wl, seed)
    rng = np.random.default_rng(seed)
    h0s = torch.from_numpy(rng.standard_normal((S, W))).float()
    dhTs = torch.from_numpy(rng.standard_normal((S, W))).float()
    ba = torch.from_numpy(rng.normal(0.0, 0.1, W)).float()
    bx = torch.from_numpy(rng.normal(0.0, 0.1, W)).float()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)

    d = {n: dev(v) for n, v in inp.items() if isinstance(v, torch.Tensor)}
    gdt = R.BF16 if grad == "bf16" else R.F32
    sh = R.make_shape(1, T, W, W // k, R.BF16 if io == "bf16" else R.F32, gdt, R.CANONICAL)
    cu_d = torch.from_numpy(cu).cuda()
    y = torch.empty_like(d["x"])
    hT = torch.empty(S, W, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    R.rglru_fused_forward_varlen(sh, d["x"], d["Wa"], dev(ba), d["Wx"], dev(bx), d["Lambda"],
                                 cu_d, S, dev(h0s), y, hT, saved)
    dx = torch.empty(1, T, W, device="cuda", dtype=R.TORCH_DT[gdt])
    dWa = torch.empty(W // k, k, k, device="cuda")
    dWx = torch.empty_like(dWa)
    dba, dbx, dL = (torch.empty(W, device="cuda") for _ in range(3))
    dh0 = torch.empty(S, W, device="cuda")
    R.rglru_fused_backward_varlen(sh, d["dy"], dev(dhTs), d["x"], d["Wa"], dev(ba), d["Wx"],
                                  dev(bx), d["Lambda"], cu_d, S, dev(h0s), saved, dx, dWa, dba,
                                  dWx, dbx, dL, dh0, ws)
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK

    x, Wa, Wx, Lam, dy = (as_f64(inp[n]) for n in ("x", "Wa", "Wx", "Lambda", "dy"))
    ba64, bx64 = ba.double().numpy(), bx.double().numpy()
    h064, dhT64 = h0s.double().numpy(), dhTs.double().numpy()
    y_ref = np.zeros((1, T, W))
    hT_ref = np.zeros((S, W))
    dh0_ref = np.zeros((S, W))
    g_ref = {"dx": np.zeros((1, T, W)), "dWa": 0.0, "dWx": 0.0, "dba": 0.0, "dbx": 0.0,
             "dLambda": 0.0}
    for s in range(S):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            hT_ref[s] = h064[s]
            dh0_ref[s] = dhT64[s]
            continue
        ys, hs = oracle.fused_forward(oracle.CANONICAL, x[:, a:b], Wa, ba64, Wx, bx64, Lam,
                                      None, None, h064[s:s + 1])
        g = oracle.fused_backward(oracle.CANONICAL, x[:, a:b], Wa, ba64, Wx, bx64, Lam,
                                  dy[:, a:b], dhT64[s:s + 1], None, None, h064[s:s + 1])
        y_ref[:, a:b] = ys
        hT_ref[s] = hs[0]
        dh0_ref[s] = g["dh0"][0]
        g_ref["dx"][:, a:b] = g["dx"]
        for n in ("dWa", "dWx", "dba", "dbx", "dLambda"):
            g_ref[n] = g_ref[n] + g[n]
    assert_close("y", host(y), y_ref, io=io, kind="out")
    assert_close("hT", host(hT), hT_ref, io=io, kind="out")
    assert_close("dx", host(dx), g_ref["dx"], io=io, kind="grad", stored=grad)
    for n, got in (("dWa", dWa), ("dWx", dWx), ("dba", dba), ("dbx", dbx), ("dLambda", dL)):
        assert_close(n, host(got), g_ref[n], io=io, kind="grad")
    assert_close("dh0", host(dh0), dh0_ref, io=io, kind="grad")


def test_varlen_full_size_sampled_blocks():
    """The packed configuration the benchmark times: 8192 tokens in one row, W2048 in 16 gate
    blocks of 128, bf16, sequence lengths U[1, 2048] (the last one truncated), per-sequence h0
    and dhT.  Gate blocks are independent in every output, so the oracle run per sequence on
    the channels of one block is that block's exact reference; three blocks are compared."""
    from linear_recurrent_rnn_gb300.inputs import packed_lengths
    T, W, k = 8192, 2048, 128
    lengths = packed_lengths(5, T, 1, 2048)
    S = len(lengths)
    wl = Workload("varlen", 1, T, W, k, "bf16", "canonical", (0.9, 0.999))
    inp = generate(wl, 5)
    rng = np.random.default_rng(6)
    h0s = torch.from_numpy(rng.standard_normal((S, W)) * 0.5).float()
    dhTs = torch.from_numpy(rng.standard_normal((S, W))).float()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    d = {n: dev(v) for n, v in inp.items() if isinstance(v, torch.Tensor)}
    sh = R.make_shape(1, T, W, W // k, R.BF16, R.BF16, R.CANONICAL)
    cu_d = torch.from_numpy(cu).cuda()
    y = torch.empty_like(d["x"])
    hT = torch.empty(S, W, device="cuda")
    saved, ws = R.alloc_saved(sh), R.alloc_workspace(sh)
    R.rglru_fused_forward_varlen(sh, d["x"], d["Wa"], d["ba"], d["Wx"], d["bx"], d["Lambda"],
                                 cu_d, S, dev(h0s), y, hT, saved)
    dx = torch.empty_like(d["x"])
    dWa = torch.empty(W // k, k, k, device="cuda")
    dWx = torch.empty_like(dWa)
    dba, dbx, dL = (torch.empty(W, device="cuda") for _ in range(3))
    dh0 = torch.empty(S, W, device="cuda")
    R.rglru_fused_backward_varlen(sh, d["dy"], dev(dhTs), d["x"], d["Wa"], d["ba"], d["Wx"],
                                  d["bx"], d["Lambda"], cu_d, S, dev(h0s), saved, dx, dWa, dba,
                                  dWx, dbx, dL, dh0, ws)
    assert R.rglru_sync_status(saved) == R.OK
    assert R.rglru_sync_status(ws) == R.OK
    got = {n: host(t) for n, t in (("y", y), ("hT", hT), ("dx", dx), ("dWa", dWa), ("dWx", dWx),
                                   ("dba", dba), ("dbx", dbx), ("dLambda", dL), ("dh0", dh0))}
    for blk in (0, 7, 15):
        cs = slice(blk * k, (blk + 1) * k)
        x, dy = as_f64(inp["x"][..., cs]), as_f64(inp["dy"][..., cs])
        ba, bx, Lam = (as_f64(inp[n][cs]) for n in ("ba", "bx", "Lambda"))
        Wa, Wx = as_f64(inp["Wa"][blk:blk + 1]), as_f64(inp["Wx"][blk:blk + 1])
        h0, dhT = h0s[:, cs].double().numpy(), dhTs[:, cs].double().numpy()
        y_ref, dx_ref = np.zeros((1, T, k)), np.zeros((1, T, k))
        hT_ref, dh0_ref = np.zeros((S, k)), np.zeros((S, k))
        acc = {n: 0.0 for n in ("dWa", "dWx", "dba", "dbx", "dLambda")}
        for s in range(S):
            a, b = int(cu[s]), int(cu[s + 1])
            ys, hs = oracle.fused_forward(oracle.CANONICAL, x[:, a:b], Wa, ba, Wx, bx, Lam,
                                          None, None, h0[s:s + 1])
            g = oracle.fused_backward(oracle.CANONICAL, x[:, a:b], Wa, ba, Wx, bx, Lam,
                                      dy[:, a:b], dhT[s:s + 1], None, None, h0[s:s + 1])
            y_ref[:, a:b], dx_ref[:, a:b] = ys, g["dx"]
            hT_ref[s], dh0_ref[s] = hs[0], g["dh0"][0]
            for n in acc:
                acc[n] = acc[n] + g[n]
        tag = f"blk{blk} "
        assert_close(tag + "y", got["y"][..., cs], y_ref, io="bf16", kind="out")
        assert_close(tag + "hT", got["hT"][:, cs], hT_ref, io="bf16", kind="out")
        assert_close(tag + "dx", got["dx"][..., cs], dx_ref, io="bf16", kind="grad",
                     stored="bf16")
        assert_close(tag + "dWa", got["dWa"][blk:blk + 1], acc["dWa"], io="bf16", kind="grad")
        assert_close(tag + "dWx", got["dWx"][blk:blk + 1], acc["dWx"], io="bf16", kind="grad")
        for n in ("dba", "dbx", "dLambda"):
            assert_close(tag + n, got[n][cs], acc[n], io="bf16", kind="grad")
        assert_close(tag + "dh0", got["dh0"][:, cs], dh0_ref, io="bf16", kind="grad")
