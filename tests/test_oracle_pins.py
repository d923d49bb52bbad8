"""Pins for the float64 oracle (CPU only).

Each oracle function is pinned to something other than itself: closed forms with hand-fixed
gate values, special cases that reduce to a single library call, exact invariants of the
reset semantics, brute-force expansion on tiny inputs, central finite differences of the
forward for every gradient, and numpy's einsum for the projections.  The hand-fixed gate
values follow from the decay law log a = -8 r softplus(Lambda):

    Lambda = ln(2^(1/4) - 1)  =>  softplus(Lambda) = ln(2)/4
    lr = 0                    =>  r = 1/2, log a = -ln 2, a = 1/2, m = sqrt(3)/2
    li = 0                    =>  i = 1/2
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle

CAN, RES = oracle.CANONICAL, oracle.RESTRICTED
LAM_HALF = math.log(2.0 ** 0.25 - 1.0)   # softplus = ln2/4 -> a = 1/2 at r = 1/2


def rand_problem(rng, B, T, W, canonical=True, p_reset=0.2, h0=True):
    x = rng.standard_normal((B, T, W))
    lr = rng.standard_normal((B, T, W))
    li = rng.standard_normal((B, T, W))
    u = rng.uniform(0.5, 0.99, W)
    Lam = np.log(np.expm1(-np.log(u) / 8.0))
    rm = (rng.random((B, T)) < p_reset).astype(np.uint8) if canonical else None
    hh = rng.standard_normal((B, W)) if (h0 and canonical) else None
    return x, lr, li, Lam, rm, hh


# ---------------------------------------------------------------- forward: closed forms

def test_half_decay_closed_form():
    """a = 1/2, m = sqrt(3)/2, i = 1/2 by construction: h_t = 2^-(t+1) h0 + 2b(1 - 2^-(t+1)),
    b = sqrt(3)/4 x (geometric series)."""
    B, T, W = 2, 40, 3
    rng = np.random.default_rng(1)
    xc = rng.standard_normal((B, 1, W))
    x = np.repeat(xc, T, axis=1)
    z = np.zeros((B, T, W))
    Lam = np.full(W, LAM_HALF)
    h0 = rng.standard_normal((B, W))
    y, hT = oracle.forward(CAN, x, z, z, Lam, h0=h0)
    t = np.arange(T)[None, :, None]
    b = math.sqrt(3.0) / 4.0 * xc
    ref = 0.5 ** (t + 1) * h0[:, None, :] + 2.0 * b * (1.0 - 0.5 ** (t + 1))
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT, ref[:, -1], rtol=1e-13, atol=1e-14)
    # restricted mode: same with h0 = 0
    yr, _ = oracle.forward(RES, x, z, z, Lam)
    ref0 = 2.0 * b * (1.0 - 0.5 ** (t + 1))
    np.testing.assert_allclose(yr, ref0, rtol=1e-13, atol=1e-14)


def test_constant_gate_geometric_series():
    """Any constant gates, no resets: y_t = a^(t+1) h0 + b (1 - a^(t+1)) / (1 - a), with a and
    b read off the first two outputs of a zero-h0 run (the recurrence's structure is pinned,
    independently of the gate formula)."""
    rng = np.random.default_rng(2)
    B, T, W = 1, 64, 5
    col = lambda: np.repeat(rng.standard_normal((B, 1, W)), T, axis=1)
    x, lr, li = col(), col(), col()
    Lam = np.log(np.expm1(-np.log(rng.uniform(0.6, 0.99, W)) / 8.0))
    y0, _ = oracle.forward(CAN, x, lr, li, Lam)
    b = y0[:, 0, :]
    a = y0[:, 1, :] / b - 1.0
    h0 = rng.standard_normal((B, W))
    y, _ = oracle.forward(CAN, x, lr, li, Lam, h0=h0)
    t = np.arange(T)[None, :, None]
    ref = a[:, None] ** (t + 1) * h0[:, None] + b[:, None] * (1 - a[:, None] ** (t + 1)) / (1 - a[:, None])
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-12)


def test_zero_decay_gives_gated_input():
    """Lambda = 1e4, lr = 0: log a = -4e4, a = 0 exactly, m = 1, so y = sigmoid(li) x."""
    rng = np.random.default_rng(3)
    B, T, W = 2, 9, 4
    x, li = rng.standard_normal((B, T, W)), rng.standard_normal((B, T, W))
    z = np.zeros((B, T, W))
    Lam = np.full(W, 1e4)
    for mode in (CAN, RES):
        y, hT = oracle.forward(mode, x, z, li, Lam, h0=rng.standard_normal((B, W)) if mode == CAN else None)
        np.testing.assert_allclose(y, expit(li) * x, rtol=1e-15, atol=0)
    y, _ = oracle.forward(RES, x, z, z, Lam)
    assert np.array_equal(y, 0.5 * x)


def test_unit_decay_holds_state():
    """lr = -1e4: r = 0, a = 1, m = 0, so the state never changes: y == h0."""
    rng = np.random.default_rng(4)
    B, T, W = 2, 7, 3
    x, li = rng.standard_normal((B, T, W)), rng.standard_normal((B, T, W))
    lr = np.full((B, T, W), -1e4)
    Lam = rng.standard_normal(W)
    h0 = rng.standard_normal((B, W))
    y, hT = oracle.forward(CAN, x, lr, li, Lam, h0=h0)
    assert np.array_equal(y, np.repeat(h0[:, None], T, axis=1))
    assert np.array_equal(hT, h0)
    y, _ = oracle.forward(RES, x, lr, li, Lam)
    assert np.array_equal(y, np.zeros_like(y))


def test_brute_force_four_tokens():
    """T = 4 with per-token r in {1/2, 3/4, 1/4} (lr in {0, ln3, -ln3}) so a_t = 2^(-2 r_t);
    the expansion h_3 = a3a2a1a0 h0 + a3a2a1 b0 + a3a2 b1 + a3 b2 + b3 is written out."""
    rs = [0.5, 0.75, 0.25, 0.5]
    lr_vals = [0.0, math.log(3.0), -math.log(3.0), 0.0]
    li_vals = [0.0, math.log(3.0), 0.0, -math.log(3.0)]
    iv = [0.5, 0.75, 0.5, 0.25]
    xs = [1.5, -0.25, 2.0, 0.75]
    h0 = -0.6
    a = [2.0 ** (-2.0 * r) for r in rs]
    m = [math.sqrt(1.0 - ai * ai) for ai in a]
    b = [m[t] * iv[t] * xs[t] for t in range(4)]
    h = [a[0] * h0 + b[0]]
    h.append(a[1] * a[0] * h0 + a[1] * b[0] + b[1])
    h.append(a[2] * a[1] * a[0] * h0 + a[2] * a[1] * b[0] + a[2] * b[1] + b[2])
    h.append(a[3] * a[2] * a[1] * a[0] * h0 + a[3] * a[2] * a[1] * b[0] + a[3] * a[2] * b[1]
             + a[3] * b[2] + b[3])
    shp = (1, 4, 1)
    y, hT = oracle.forward(CAN, np.array(xs).reshape(shp), np.array(lr_vals).reshape(shp),
                           np.array(li_vals).reshape(shp), np.array([LAM_HALF]),
                           h0=np.array([[h0]]))
    np.testing.assert_allclose(y.ravel(), h, rtol=1e-14, atol=1e-15)
    # a reset at token 2 drops the state before it and uses m = 1
    rm = np.array([[0, 0, 1, 0]], dtype=np.uint8)
    y2, _ = oracle.forward(CAN, np.array(xs).reshape(shp), np.array(lr_vals).reshape(shp),
                           np.array(li_vals).reshape(shp), np.array([LAM_HALF]),
                           reset_mask=rm, h0=np.array([[h0]]))
    h2 = iv[2] * xs[2]
    h3 = a[3] * h2 + b[3]
    np.testing.assert_allclose(y2.ravel(), [h[0], h[1], h2, h3], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- reset semantics

def test_reset_cuts_history_bitwise():
    rng = np.random.default_rng(5)
    B, T, W, tr = 2, 12, 6, 5
    x, lr, li, Lam, _, h0 = rand_problem(rng, B, T, W)
    rm = np.zeros((B, T), np.uint8)
    rm[:, tr] = 1
    y, hT = oracle.forward(CAN, x, lr, li, Lam, reset_mask=rm, h0=h0)
    x2, lr2, li2 = x.copy(), lr.copy(), li.copy()
    x2[:, :tr] += rng.standard_normal((B, tr, W))
    lr2[:, :tr] -= 1.0
    li2[:, :tr] += 0.5
    y2, hT2 = oracle.forward(CAN, x2, lr2, li2, Lam, reset_mask=rm, h0=h0 + 3.0)
    assert np.array_equal(y[:, tr:], y2[:, tr:])
    assert np.array_equal(hT, hT2)
    assert not np.array_equal(y[:, :tr], y2[:, :tr])
    # gradients before the reset receive nothing from dy at/after it, nor from dhT
    dy = rng.standard_normal((B, T, W))
    g1 = oracle.backward(CAN, x, lr, li, Lam, dy, rng.standard_normal((B, W)), reset_mask=rm, h0=h0)
    dy2 = dy.copy()
    dy2[:, tr:] *= -3.0
    g2 = oracle.backward(CAN, x, lr, li, Lam, dy2, rng.standard_normal((B, W)), reset_mask=rm, h0=h0)
    for key in ("dx", "dlr", "dli"):
        assert np.array_equal(g1[key][:, :tr], g2[key][:, :tr])
    assert np.array_equal(g1["dh0"], g2["dh0"])


def test_segment_pos_equals_reset_mask():
    rng = np.random.default_rng(6)
    B, T, W = 2, 30, 4
    x, lr, li, Lam, _, h0 = rand_problem(rng, B, T, W)
    sp = np.zeros((B, T), np.int32)
    for b in range(B):
        p = 3 + b
        for t in range(T):
            if rng.random() < 0.15:
                p = 0
            sp[b, t] = p
            p += 1
    rm = (sp == 0).astype(np.uint8)
    ya, ha = oracle.forward(CAN, x, lr, li, Lam, segment_pos=sp, h0=h0)
    yb, hb = oracle.forward(CAN, x, lr, li, Lam, reset_mask=rm, h0=h0)
    assert np.array_equal(ya, yb) and np.array_equal(ha, hb)
    dy = rng.standard_normal((B, T, W))
    ga = oracle.backward(CAN, x, lr, li, Lam, dy, None, segment_pos=sp, h0=h0)
    gb = oracle.backward(CAN, x, lr, li, Lam, dy, None, reset_mask=rm, h0=h0)
    for k in ga:
        assert np.array_equal(ga[k], gb[k])


def test_restricted_equals_canonical_without_resets():
    rng = np.random.default_rng(7)
    B, T, W = 2, 17, 5
    x, lr, li, Lam, _, _ = rand_problem(rng, B, T, W)
    yc, hc = oracle.forward(CAN, x, lr, li, Lam)
    yr, hr = oracle.forward(RES, x, lr, li, Lam)
    assert np.array_equal(yc, yr) and np.array_equal(hc, hr)
    dy, dhT = rng.standard_normal((B, T, W)), rng.standard_normal((B, W))
    gc = oracle.backward(CAN, x, lr, li, Lam, dy, dhT)
    gr = oracle.backward(RES, x, lr, li, Lam, dy, dhT)
    for k in ("dx", "dlr", "dli", "dLambda"):
        assert np.array_equal(gc[k], gr[k])
    assert np.array_equal(gr["dh0"], np.zeros((B, W)))


def test_first_token_reset_difference():
    """Canonical with a reset only at t = 0 vs restricted: they differ only through the first
    write's multiplier, h^can_t - h^res_t = (prod_{s=1..t} a_s)(1 - m_0) i_0 x_0.  With the
    half-decay gates: = 2^-t (1 - sqrt(3)/2) x_0 / 2."""
    rng = np.random.default_rng(8)
    B, T, W = 1, 20, 3
    x = rng.standard_normal((B, T, W))
    z = np.zeros((B, T, W))
    Lam = np.full(W, LAM_HALF)
    rm = np.zeros((B, T), np.uint8)
    rm[:, 0] = 1
    yc, _ = oracle.forward(CAN, x, z, z, Lam, reset_mask=rm, h0=rng.standard_normal((B, W)))
    yr, _ = oracle.forward(RES, x, z, z, Lam)
    t = np.arange(T)[None, :, None]
    ref = 0.5 ** t * (1.0 - math.sqrt(3.0) / 2.0) * x[:, :1, :] / 2.0
    np.testing.assert_allclose(yc - yr, ref, rtol=1e-12, atol=1e-15)


def test_state_carry_split():
    """fwd(0:T) == fwd(t0:T, h0 = hT(fwd(0:t0))) when t0 is not a reset."""
    rng = np.random.default_rng(9)
    B, T, W, t0 = 2, 50, 4, 23
    x, lr, li, Lam, rm, h0 = rand_problem(rng, B, T, W, p_reset=0.05)
    rm[:, t0] = 0
    y, hT = oracle.forward(CAN, x, lr, li, Lam, reset_mask=rm, h0=h0)
    ya, ha = oracle.forward(CAN, x[:, :t0], lr[:, :t0], li[:, :t0], Lam, reset_mask=rm[:, :t0], h0=h0)
    yb, hb = oracle.forward(CAN, x[:, t0:], lr[:, t0:], li[:, t0:], Lam, reset_mask=rm[:, t0:], h0=ha)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(hb, hT, rtol=1e-14, atol=1e-14)


def test_dh0_zero_under_first_token_reset():
    rng = np.random.default_rng(10)
    B, T, W = 3, 11, 4
    x, lr, li, Lam, rm, h0 = rand_problem(rng, B, T, W)
    rm[:, 0] = 1
    g = oracle.backward(CAN, x, lr, li, Lam, rng.standard_normal((B, T, W)),
                        rng.standard_normal((B, W)), reset_mask=rm, h0=h0)
    assert np.array_equal(g["dh0"], np.zeros((B, W)))


# ---------------------------------------------------------------- backward: finite differences

def _loss_scan(mode, x, lr, li, Lam, rm, h0, dy, dhT):
    y, hT = oracle.forward(mode, x, lr, li, Lam, reset_mask=rm, h0=h0)
    L = float(np.sum(y * dy))
    if dhT is not None:
        L += float(np.sum(hT * dhT))
    return L


def _fd(f, arr, eps=1e-6):
    g = np.empty_like(arr)
    for idx in np.ndindex(arr.shape):
        old = arr[idx]
        h = eps * max(1.0, abs(old))
        arr[idx] = old + h
        fp = f()
        arr[idx] = old - h
        fm = f()
        arr[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("mode,T,W", [(CAN, 1, 8), (CAN, 2, 8), (CAN, 5, 8), (RES, 5, 8), (RES, 1, 8)])
def test_scan_backward_finite_differences(mode, T, W):
    rng = np.random.default_rng(100 + T + 10 * mode)
    B = 2
    x, lr, li, Lam, rm, h0 = rand_problem(rng, B, T, W, canonical=(mode == CAN), p_reset=0.3)
    dy = rng.standard_normal((B, T, W))
    dhT = rng.standard_normal((B, W))
    g = oracle.backward(mode, x, lr, li, Lam, dy, dhT, reset_mask=rm, h0=h0)
    f = lambda: _loss_scan(mode, x, lr, li, Lam, rm, h0, dy, dhT)
    for name, arr in (("dx", x), ("dlr", lr), ("dli", li), ("dLambda", Lam)):
        fd = _fd(f, arr)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-6 * max(1, np.abs(fd).max()),
                                   err_msg=name)
    if h0 is not None:
        fd = _fd(f, h0)
        np.testing.assert_allclose(g["dh0"], fd, rtol=1e-6, atol=1e-6, err_msg="dh0")


def test_scan_backward_fd_near_unit_decay():
    """a close to 1 (m small): the exact -a^2/m term of the multiplier's derivative."""
    rng = np.random.default_rng(11)
    B, T, W = 1, 6, 4
    x, lr, li, _, rm, h0 = rand_problem(rng, B, T, W, p_reset=0.0)
    Lam = np.log(np.expm1(-np.log(np.full(W, 0.9999)) / 8.0))
    lr[:] = -3.0
    dy = rng.standard_normal((B, T, W))
    g = oracle.backward(CAN, x, lr, li, Lam, dy, None, h0=h0)
    f = lambda: _loss_scan(CAN, x, lr, li, Lam, None, h0, dy, None)
    for name, arr in (("dlr", lr), ("dLambda", Lam), ("dx", x)):
        fd = _fd(f, arr, eps=1e-7)
        np.testing.assert_allclose(g[name], fd, rtol=2e-6, atol=1e-6 * max(1, np.abs(fd).max()),
                                   err_msg=name)


def test_fused_backward_finite_differences():
    rng = np.random.default_rng(12)
    B, T, nblk, k = 2, 4, 2, 4
    W = nblk * k
    x = rng.standard_normal((B, T, W))
    Wa = rng.standard_normal((nblk, k, k)) / math.sqrt(k)
    Wx = rng.standard_normal((nblk, k, k)) / math.sqrt(k)
    ba = rng.standard_normal(W) * 0.1
    bx = rng.standard_normal(W) * 0.1
    Lam = np.log(np.expm1(-np.log(rng.uniform(0.5, 0.99, W)) / 8.0))
    rm = np.zeros((B, T), np.uint8)
    rm[1, 2] = 1
    h0 = rng.standard_normal((B, W))
    dy = rng.standard_normal((B, T, W))
    dhT = rng.standard_normal((B, W))
    g = oracle.fused_backward(CAN, x, Wa, ba, Wx, bx, Lam, dy, dhT, reset_mask=rm, h0=h0)

    def f():
        y, hT = oracle.fused_forward(CAN, x, Wa, ba, Wx, bx, Lam, reset_mask=rm, h0=h0)
        return float(np.sum(y * dy) + np.sum(hT * dhT))

    for name, arr in (("dx", x), ("dWa", Wa), ("dWx", Wx), ("dba", ba), ("dbx", bx),
                      ("dLambda", Lam), ("dh0", h0)):
        fd = _fd(f, arr)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-6 * max(1, np.abs(fd).max()),
                                   err_msg=name)


# ---------------------------------------------------------------- projections: library matmul

def test_gate_proj_matches_einsum():
    rng = np.random.default_rng(13)
    B, T, nblk, k = 2, 7, 3, 16
    W = nblk * k
    x = rng.standard_normal((B, T, W))
    Wa, Wx = rng.standard_normal((2, nblk, k, k))
    ba, bx = rng.standard_normal((2, W))
    lr, li = oracle.gate_proj(x, Wa, ba, Wx, bx)
    xb = x.reshape(B, T, nblk, k)
    ref_r = np.einsum("btni,nij->btnj", xb, Wa).reshape(B, T, W) + ba
    ref_i = np.einsum("btni,nij->btnj", xb, Wx).reshape(B, T, W) + bx
    np.testing.assert_allclose(lr, ref_r, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(li, ref_i, rtol=1e-12, atol=1e-12)


def test_gate_proj_backward_matches_einsum():
    rng = np.random.default_rng(14)
    B, T, nblk, k = 2, 5, 3, 8
    W = nblk * k
    x, dlr, dli, dx0 = rng.standard_normal((4, B, T, W))
    Wa, Wx = rng.standard_normal((2, nblk, k, k))
    p = oracle.gate_proj_backward(x, Wa, Wx, dlr, dli, dx_in=dx0)
    xb = x.reshape(B, T, nblk, k)
    gr, gi = dlr.reshape(B, T, nblk, k), dli.reshape(B, T, nblk, k)
    ref_dx = dx0 + (np.einsum("btnj,nij->btni", gr, Wa) + np.einsum("btnj,nij->btni", gi, Wx)).reshape(B, T, W)
    np.testing.assert_allclose(p["dx"], ref_dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p["dWa"], np.einsum("btni,btnj->nij", xb, gr), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p["dWx"], np.einsum("btni,btnj->nij", xb, gi), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p["dba"], dlr.sum(axis=(0, 1)), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p["dbx"], dli.sum(axis=(0, 1)), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- the chunked scan's algebra

def _compose(p2, p1):
    """(A2, B2) o (A1, B1): apply map 1, then map 2 (h -> A h + B)."""
    return (p2[0] * p1[0], p2[0] * p1[1] + p2[1])


def _all_bracketings(items):
    if len(items) == 1:
        yield items[0]
        return
    for s in range(1, len(items)):
        for left in _all_bracketings(items[:s]):
            for right in _all_bracketings(items[s:]):
                yield _compose(right, left)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 7])
def test_affine_pair_composition_any_bracketing(T):
    """The exact chunked scan relies on (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2) being
    associative: every bracketing equals the serial recurrence h_t = a_t h_{t-1} + b_t."""
    rng = np.random.default_rng(20 + T)
    a = rng.uniform(0.0, 1.0, T)
    b = rng.standard_normal(T)
    h0 = rng.standard_normal()
    h = h0
    for t in range(T):
        h = a[t] * h + b[t]
    pairs = [(a[t], b[t]) for t in range(T)]
    for A, Bv in _all_bracketings(pairs):
        assert abs(A * h0 + Bv - h) <= 1e-15 * max(1.0, abs(h)) + 1e-15


def test_reverse_pair_composition_matches_serial_backward():
    """The backward's reverse scan g_t = dy_t + abar_{t+1} g_{t+1} written as a chunked
    composition (carry c_in -> c_out = abar_{t0} g_{t0}) equals the serial loop."""
    rng = np.random.default_rng(30)
    T, C = 23, 5
    abar = rng.uniform(0.0, 1.0, T)
    dy = rng.standard_normal(T)
    dhT = rng.standard_normal()
    g = np.empty(T)
    nxt = dhT
    for t in range(T - 1, -1, -1):
        g[t] = dy[t] + (nxt if t == T - 1 else abar[t + 1] * g[t + 1])
    # chunked: each chunk computes (A, Bv) with c_out = A c_in + Bv, then fix up
    c_in = dhT
    gc = np.empty(T)
    for s in reversed(range(0, T, C)):
        e = min(T, s + C)
        gl = np.empty(e - s)
        q = np.empty(e - s)
        acc_g, acc_q = 0.0, 1.0
        for t in range(e - 1, s - 1, -1):
            if t < e - 1:
                acc_g, acc_q = abar[t + 1] * acc_g, abar[t + 1] * acc_q
            acc_g += dy[t]
            gl[t - s], q[t - s] = acc_g, acc_q
        gc[s:e] = gl + q * c_in
        c_in = abar[s] * gc[s]
    np.testing.assert_allclose(gc, g, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- input generator

def test_lambda_placement():
    from linear_recurrent_rnn_gb300.inputs import lambda_for_decay
    u = np.array([0.9, 0.99, 0.999, 0.9999])
    lam = lambda_for_decay(u)
    # softplus via numpy's logaddexp (a library routine): 8 softplus(L) = -ln u
    np.testing.assert_allclose(8.0 * np.logaddexp(0.0, lam), -np.log(u), rtol=1e-12)
    np.testing.assert_allclose(lam, [-4.3232, -6.6790, -8.9866, -11.2897], atol=1e-3)
