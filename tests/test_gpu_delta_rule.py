"""GPU parity of the gated delta rule (delta_rule_forward / delta_rule_backward) with the
float64 oracle, element by element: o, the final states, and every gradient (dq, dk, dv, dg,
dbeta, dh0).

Tolerance, from the arithmetic: the kernels keep the state and every sum in float32 on the
same stored inputs as the oracle.  With unit keys and beta in [0, 1] the state map
S -> D (I - beta k k^T) S + ... does not expand, so rounding grows at most linearly in the
tokens: about Dk * 2^-24 per token (a 128-term dot product), 1e-4 over the short cases here and
1e-3 over 2048 tokens, as E = max |gpu - ref| / max(1, |ref|).  A bf16 output adds its own
rounding, half a bf16 ulp (2^-9 of |o|)."""
import numpy as np
import pytest
import torch

from oracle import delta_rule as D
from linear_recurrent_rnn_gb300 import librglru as R
from linear_recurrent_rnn_gb300.delta_inputs import DELTA_WORKLOADS, DeltaWorkload, as_f64, generate

pytestmark = pytest.mark.gpu


def err_E(got, ref):
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))) if ref.size else 0.0


def check(name, got, ref, tol):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    e = err_E(got, ref)
    assert e <= tol, f"{name}: E = {e:.3e} > {tol:.1e}"


def run_gpu(wl, inp, scale, v_first=False):
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    cu = d["cu_seqlens"]
    N = wl.B if cu is None else cu.numel() - 1
    sh = R.make_delta_shape(wl.B, wl.T, wl.Hk, wl.Hv, wl.Dk, wl.Dv,
                            R.F32 if wl.io == "f32" else R.BF16, wl.kda, v_first)
    st_shape = (N, wl.Hv, wl.Dv, wl.Dk) if v_first else (N, wl.Hv, wl.Dk, wl.Dv)
    h0 = d["h0"]
    dhT = d["dhT"]
    if v_first and h0 is not None:
        h0 = h0.transpose(-1, -2).contiguous()
        dhT = dhT.transpose(-1, -2).contiguous()
    o = torch.empty_like(d["v"])
    hT = torch.empty(st_shape, device="cuda")
    saved = torch.empty(max(1, R.delta_rule_saved_bytes(sh, N)), dtype=torch.uint8, device="cuda")
    R.delta_rule_forward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale, cu, N, h0, o, hT,
                         saved)
    out = {"o": o, "hT": hT}
    for n, like in (("dq", d["q"]), ("dk", d["k"]), ("dv", d["v"])):
        out[n] = torch.empty(like.shape, device="cuda")
    out["dg"] = torch.empty(d["g"].shape, device="cuda")
    out["dbeta"] = torch.empty(d["beta"].shape, device="cuda")
    out["dh0"] = torch.empty(st_shape, device="cuda")
    ws = torch.empty(max(1, R.delta_rule_workspace_bytes(sh)), dtype=torch.uint8, device="cuda")
    R.delta_rule_backward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale, cu, N, h0, saved,
                          d["do"], dhT, out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"],
                          out["dh0"], ws)
    torch.cuda.synchronize()
    res = {n: t.detach().cpu().double().numpy() for n, t in out.items()}
    if v_first:
        res["hT"] = np.swapaxes(res["hT"], -1, -2)
        res["dh0"] = np.swapaxes(res["dh0"], -1, -2)
    return res


def oracle_run(inp, scale):
    q, k, v, g, beta, do = (as_f64(inp[n]) for n in ("q", "k", "v", "g", "beta", "do"))
    h0, dhT = as_f64(inp["h0"]), as_f64(inp["dhT"])
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].numpy()
    o, fin = D.forward(q, k, v, g, beta, scale, h0, cu)
    gr = D.backward(q, k, v, g, beta, do, dhT, scale, h0, cu)
    return dict(o=o, hT=fin, **gr)


CASES = [
    # name, workload, seed, state_v_first
    ("gdn-f32-grouped-raggedDv", DeltaWorkload("a", 2, 100, 2, 4, 64, 48, "f32", h0_std=0.5), 1, False),
    ("kda-bf16-packed-vfirst", DeltaWorkload("b", 1, 74, 2, 2, 128, 128, "bf16", kda=True, h0_std=1.0,
                                             lengths=(0, 17, 1, 40, 16)), 2, True),
    ("gdn-bf16-Dk32-Dv8-noh0", DeltaWorkload("c", 2, 33, 1, 1, 32, 8, "bf16"), 3, False),
    ("gdn-f32-T1", DeltaWorkload("d", 1, 1, 1, 2, 64, 64, "f32", h0_std=1.0), 4, False),
    ("kda-f32-strong-decay", DeltaWorkload("e", 1, 50, 1, 1, 64, 40, "f32", kda=True,
                                           decay=(0.01, 0.5), h0_std=1.0), 5, False),
]


@pytest.mark.parametrize("name,wl,seed,v_first", CASES, ids=[c[0] for c in CASES])
def test_delta_rule_matches_oracle(name, wl, seed, v_first):
    inp = generate(wl, seed)
    scale = wl.Dk ** -0.5
    got = run_gpu(wl, inp, scale, v_first)
    ref = oracle_run(inp, scale)
    tol = 1e-4
    check("o", got["o"], ref["o"], tol + (2.0 ** -9 if wl.io == "bf16" else 0.0))
    for n in ("hT", "dq", "dk", "dv", "dg", "dbeta"):
        check(n, got[n], ref[n], tol)
    if inp["h0"] is not None:
        check("dh0", got["dh0"], ref["dh0"], tol)


def test_delta_rule_full_size_sampled_heads():
    """The timed configuration (B4 T2048, 16 heads of 128 x 128, bf16) on the GPU; heads are
    independent, so the oracle run on one batch row and one head is that slice's exact
    reference.  Two (row, head) pairs are compared element by element."""
    wl = DELTA_WORKLOADS["headline"].scaled(h0_std=0.5)
    inp = generate(wl, 11)
    scale = wl.Dk ** -0.5
    got = run_gpu(wl, inp, scale)
    for b, h in ((0, 0), (3, 13)):
        sl = {n: (None if t is None else (t[b:b + 1, :, h:h + 1] if n in ("q", "k", "v", "g", "beta", "do")
                                          else t[b:b + 1, h:h + 1])) for n, t in inp.items()
              if n != "cu_seqlens"}
        sl["cu_seqlens"] = None
        ref = oracle_run(sl, scale)
        check("o", got["o"][b:b + 1, :, h:h + 1], ref["o"], 1e-3 + 2.0 ** -9)
        check("hT", got["hT"][b:b + 1, h:h + 1], ref["hT"], 1e-3)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            check(n, got[n][b:b + 1, :, h:h + 1], ref[n], 1e-3)
        check("dh0", got["dh0"][b:b + 1, h:h + 1], ref["dh0"], 1e-3)


def test_decode_loop_reproduces_forward():
    """T = 1 calls with the states carried in place (hT = h0) reproduce the forward over the
    whole sequence, token by token (same float32 arithmetic per token: equal to rounding)."""
    wl = DeltaWorkload("dec", 2, 24, 2, 4, 64, 64, "f32", kda=True, h0_std=0.5)
    inp = generate(wl, 21)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    scale = wl.Dk ** -0.5
    full = R.make_delta_shape(wl.B, wl.T, wl.Hk, wl.Hv, wl.Dk, wl.Dv, R.F32, True)
    o = torch.empty_like(d["v"])
    hT = torch.empty_like(d["h0"])
    R.delta_rule_forward(full, d["q"], d["k"], d["v"], d["g"], d["beta"], scale, None, wl.B,
                         d["h0"], o, hT, None)
    one = R.make_delta_shape(wl.B, 1, wl.Hk, wl.Hv, wl.Dk, wl.Dv, R.F32, True)
    h = d["h0"].clone()
    outs = []
    for t in range(wl.T):
        sl = lambda x: x[:, t:t + 1].contiguous()
        ot = torch.empty_like(sl(d["v"]))
        R.delta_rule_forward(one, sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]),
                             scale, None, wl.B, h, ot, h, None)
        outs.append(ot)
    torch.cuda.synchronize()
    check("o", torch.cat(outs, 1).cpu().double().numpy(), o.cpu().double().numpy(), 1e-5)
    check("hT", h.cpu().double().numpy(), hT.cpu().double().numpy(), 1e-5)


def _padded(shape, dtype, pad=256, fill=12345.0):
    """A tensor view of `shape` inside a buffer with `pad` canary elements on both sides."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return buf, buf[pad:pad + n].view(shape)


def test_outputs_stay_in_bounds_and_runs_are_bitwise_equal():
    """Every output of the forward and the backward lives inside a buffer padded with canary
    values on both sides (packed sequences with an empty one, grouped heads, KDA, ragged Dv);
    no canary may change, and a second run must give bitwise the same outputs (fixed-order
    sums, including the cluster's rank-ordered exchange)."""
    wl = DeltaWorkload("cn", 1, 70, 2, 4, 64, 40, "f32", kda=True, h0_std=0.5,
                       lengths=(30, 0, 17, 23))
    inp = generate(wl, 31)
    d = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
    N = 4
    sh = R.make_delta_shape(wl.B, wl.T, wl.Hk, wl.Hv, wl.Dk, wl.Dv, R.F32, True)
    scale = wl.Dk ** -0.5
    runs = []
    for _ in range(2):
        bufs, outs = {}, {}
        for n, shape in (("o", d["v"].shape), ("hT", (N, wl.Hv, wl.Dk, wl.Dv)),
                         ("dq", d["q"].shape), ("dk", d["k"].shape), ("dv", d["v"].shape),
                         ("dg", d["g"].shape), ("dbeta", d["beta"].shape),
                         ("dh0", (N, wl.Hv, wl.Dk, wl.Dv))):
            bufs[n], outs[n] = _padded(shape, torch.float32)
        saved = torch.empty(R.delta_rule_saved_bytes(sh, N), dtype=torch.uint8, device="cuda")
        ws = torch.empty(max(1, R.delta_rule_workspace_bytes(sh)), dtype=torch.uint8, device="cuda")
        R.delta_rule_forward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale,
                             d["cu_seqlens"], N, d["h0"], outs["o"], outs["hT"], saved)
        R.delta_rule_backward(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], scale,
                              d["cu_seqlens"], N, d["h0"], saved, d["do"], d["dhT"], outs["dq"],
                              outs["dk"], outs["dv"], outs["dg"], outs["dbeta"], outs["dh0"], ws)
        torch.cuda.synchronize()
        for n, b in bufs.items():
            assert torch.all(b[:256] == 12345.0) and torch.all(b[-256:] == 12345.0), n
        runs.append({n: t.clone() for n, t in outs.items()})
    for n in runs[0]:
        assert torch.equal(runs[0][n], runs[1][n]), n
