"""Pins for the gated delta-rule oracle (CPU only).

Each oracle function is tied to something other than itself: closed forms of a single token
and of a write-free (beta = 0) sequence, exact retrieval and overwrite with orthonormal keys
(what distinguishes a delta rule from a plain linear-attention sum), the reductions of KDA
with equal per-key decays to GDN and of grouped heads to repeated keys, packing and splitting
invariants, the transposed state layout, and central finite differences for every gradient.
"""
import numpy as np
import pytest

from oracle import delta_rule as D


def rand(rng, B=2, T=7, Hk=1, Hv=2, Dk=4, Dv=3, kda=False, h0=True):
    q = rng.standard_normal((B, T, Hk, Dk))
    k = rng.standard_normal((B, T, Hk, Dk)) / np.sqrt(Dk)
    v = rng.standard_normal((B, T, Hv, Dv))
    beta = rng.uniform(0.1, 0.9, (B, T, Hv))
    g = np.log(rng.uniform(0.5, 1.0, (B, T, Hv, Dk) if kda else (B, T, Hv)))
    hh = rng.standard_normal((B, Hv, Dk, Dv)) if h0 else None
    return q, k, v, g, beta, hh


# ---------------------------------------------------------------- forward: closed forms

def test_single_token_from_zero_state():
    """T = 1 from S = 0: u = beta v, S = beta k v^T, o = scale beta (k . q) v."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, _ = rand(rng, B=1, T=1, Hk=1, Hv=1, Dk=5, Dv=3)
    o, fin = D.forward(q, k, v, g, beta, scale=0.7)
    b = beta[0, 0, 0]
    np.testing.assert_allclose(fin[0, 0], b * np.outer(k[0, 0, 0], v[0, 0, 0]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(o[0, 0, 0], 0.7 * b * (k[0, 0, 0] @ q[0, 0, 0]) * v[0, 0, 0],
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("kda", [False, True])
def test_no_write_is_pure_decay(kda):
    """beta = 0: nothing is written, S_t = prod_s D_s S_0, so o_t = scale (prod D) S_0^T q_t."""
    rng = np.random.default_rng(2)
    q, k, v, g, beta, h0 = rand(rng, B=1, T=6, Hk=1, Hv=1, Dk=4, Dv=3, kda=kda)
    beta[:] = 0.0
    o, fin = D.forward(q, k, v, g, beta, scale=1.0, initial_state=h0)
    cum = np.cumsum(g[0, :, 0], axis=0)  # [T] or [T, Dk]
    for t in range(6):
        d = np.exp(cum[t])
        St = (d[:, None] if kda else d) * h0[0, 0]
        np.testing.assert_allclose(o[0, t, 0], St.T @ q[0, t, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fin[0, 0], St, rtol=1e-12, atol=1e-14)


def test_exact_retrieval_and_overwrite():
    """g = 0, beta = 1, unit keys: a write makes S^T k = v exactly (the delta rule replaces the
    value stored under a key instead of adding to it).  Keys e0, e1, e0 with values v0, v1, v2:
    the final state holds v2 under e0 and v1 under e1, and a query e0 reads v2."""
    Dk, Dv = 3, 2
    e = np.eye(Dk)
    k = np.stack([e[0], e[1], e[0]])[None, :, None, :]
    v = np.array([[1.0, 2.0], [3.0, -1.0], [-4.0, 0.5]])[None, :, None, :]
    q = np.stack([e[1], e[1], e[0]])[None, :, None, :]
    g = np.zeros((1, 3, 1))
    beta = np.ones((1, 3, 1))
    o, fin = D.forward(q, k, v, g, beta, scale=1.0)
    np.testing.assert_array_equal(fin[0, 0][0], v[0, 2, 0])
    np.testing.assert_array_equal(fin[0, 0][1], v[0, 1, 0])
    np.testing.assert_array_equal(fin[0, 0][2], np.zeros(Dv))
    np.testing.assert_array_equal(o[0, 0, 0], np.zeros(Dv))      # e1 not written yet
    np.testing.assert_array_equal(o[0, 1, 0], v[0, 1, 0])
    np.testing.assert_array_equal(o[0, 2, 0], v[0, 2, 0])        # overwritten, not summed


def test_half_write_mixes_old_and_new():
    """beta = 1/2 on a repeated unit key: the stored value moves half way to the new one."""
    k = np.array([[1.0, 0.0], [1.0, 0.0]])[None, :, None, :]
    v = np.array([[2.0], [6.0]])[None, :, None, :]
    q = k.copy()
    g = np.zeros((1, 2, 1))
    beta = np.full((1, 2, 1), 0.5)
    o, fin = D.forward(q, k, v, g, beta, scale=1.0)
    assert o[0, 0, 0, 0] == 1.0          # half of 2
    assert o[0, 1, 0, 0] == 3.5          # 1 + (6 - 1) / 2
    assert fin[0, 0][0, 0] == 3.5


# ---------------------------------------------------------------- forward: invariants

def test_kda_with_equal_decays_is_gdn():
    rng = np.random.default_rng(3)
    q, k, v, g, beta, h0 = rand(rng, Dk=4)
    gk = np.repeat(g[..., None], 4, axis=-1)
    o1, f1 = D.forward(q, k, v, g, beta, initial_state=h0)
    o2, f2 = D.forward(q, k, v, gk, beta, initial_state=h0)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(f1, f2, rtol=1e-13, atol=1e-14)


def test_grouped_heads_equal_repeated_keys():
    """Hv = 2 Hk: value heads 2h, 2h + 1 read key head h, as with q and k repeated."""
    rng = np.random.default_rng(4)
    q, k, v, g, beta, h0 = rand(rng, Hk=2, Hv=4)
    o1, f1 = D.forward(q, k, v, g, beta, initial_state=h0)
    o2, f2 = D.forward(np.repeat(q, 2, axis=2), np.repeat(k, 2, axis=2), v, g, beta,
                       initial_state=h0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(f1, f2)


def test_packed_sequences_equal_separate_rows():
    rng = np.random.default_rng(5)
    lens = [3, 0, 5, 1]
    T = sum(lens)
    q, k, v, g, beta, _ = rand(rng, B=1, T=T, Hv=2)
    h0 = rng.standard_normal((4, 2, 4, 3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, fin = D.forward(q, k, v, g, beta, initial_state=h0, cu_seqlens=cu)
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        o_s, f_s = D.forward(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b],
                             initial_state=h0[s:s + 1])
        np.testing.assert_array_equal(o[:, a:b], o_s)
        np.testing.assert_array_equal(fin[s], f_s[0])
    np.testing.assert_array_equal(fin[1], h0[1])  # empty sequence: final = initial


def test_split_carries_the_state():
    rng = np.random.default_rng(6)
    q, k, v, g, beta, h0 = rand(rng, T=9, kda=True)
    o, fin = D.forward(q, k, v, g, beta, initial_state=h0)
    o1, f1 = D.forward(q[:, :4], k[:, :4], v[:, :4], g[:, :4], beta[:, :4], initial_state=h0)
    o2, f2 = D.forward(q[:, 4:], k[:, 4:], v[:, 4:], g[:, 4:], beta[:, 4:], initial_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(f2, fin, rtol=1e-14, atol=1e-14)


def test_value_first_state_layout_is_a_transpose():
    rng = np.random.default_rng(7)
    q, k, v, g, beta, h0 = rand(rng)
    o1, f1 = D.forward(q, k, v, g, beta, initial_state=h0)
    o2, f2 = D.forward(q, k, v, g, beta, initial_state=np.swapaxes(h0, -1, -2),
                       state_v_first=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(f1, np.swapaxes(f2, -1, -2))


# ---------------------------------------------------------------- backward: finite differences

def _loss(args, do, dfin, kw):
    o, fin = D.forward(*args, **kw)
    return np.sum(o * do) + np.sum(fin * dfin)


@pytest.mark.parametrize("kda,Hk,Hv,packed,v_first", [
    (False, 1, 1, False, False),
    (True, 1, 2, False, False),
    (False, 2, 4, True, False),
    (True, 1, 1, True, True),
])
def test_backward_matches_finite_differences(kda, Hk, Hv, packed, v_first):
    rng = np.random.default_rng(10 + kda + 2 * Hk + 4 * packed)
    B, T = (1, 6) if packed else (2, 5)
    q, k, v, g, beta, h0 = rand(rng, B=B, T=T, Hk=Hk, Hv=Hv, Dk=3, Dv=2, kda=kda)
    cu = np.array([0, 2, 2, 6]) if packed else None
    N = 3 if packed else B
    h0 = rng.standard_normal((N, Hv, 3, 2))
    if v_first:
        h0 = np.swapaxes(h0, -1, -2).copy()
    kw = dict(scale=0.8, cu_seqlens=cu, state_v_first=v_first)
    o, fin = D.forward(q, k, v, g, beta, initial_state=h0, **kw)
    do = rng.standard_normal(o.shape)
    dfin = rng.standard_normal(fin.shape)
    grads = D.backward(q, k, v, g, beta, do, dfin, initial_state=h0, **kw)
    names = ["q", "k", "v", "g", "beta", "h0"]
    arrays = [q, k, v, g, beta, h0]
    eps = 1e-6
    for name, arr in zip(names, arrays):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            keep = arr[i]
            arr[i] = keep + eps
            lp = _loss((q, k, v, g, beta), do, dfin, dict(kw, initial_state=h0))
            arr[i] = keep - eps
            lm = _loss((q, k, v, g, beta), do, dfin, dict(kw, initial_state=h0))
            arr[i] = keep
            num[i] = (lp - lm) / (2 * eps)
        got = grads["d" + name]
        np.testing.assert_allclose(got, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_backward_without_final_gradient_and_linearity():
    """dfinal = None is the zero gradient, and the gradients are linear in do."""
    rng = np.random.default_rng(20)
    q, k, v, g, beta, h0 = rand(rng, kda=True)
    o, fin = D.forward(q, k, v, g, beta, initial_state=h0)
    do = rng.standard_normal(o.shape)
    a = D.backward(q, k, v, g, beta, do, None, initial_state=h0)
    b = D.backward(q, k, v, g, beta, do, np.zeros_like(fin), initial_state=h0)
    c = D.backward(q, k, v, g, beta, 2.0 * do, None, initial_state=h0)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
        np.testing.assert_allclose(c[n], 2.0 * a[n], rtol=1e-13, atol=1e-14)
