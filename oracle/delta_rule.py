"""Gated delta rule oracle: TEST INFRASTRUCTURE ONLY.

A float64 CPU statement of the gated delta-rule recurrence (GDN: one scalar decay per value
head and token; KDA: one decay per key channel), forward and hand-derived backward, used to
check the CUDA library element by element.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; it shares no code with the CUDA library.

Passages followed ("linear_attention.reference" page, entry recurrent_delta_rule_reference):
the rule stepped one token at a time, with its decay one number per value head (GDN) or one
per key channel (KDA); inputs q, k [B, T, Hk, Dk],
v [B, T, Hv, Dv], beta [B, T, Hv], g [B, T, Hv] (GDN) or [B, T, Hv, Dk] (KDA); the state
[N, Hv, Dk, Dv] (key first) or [N, Hv, Dv, Dk] with state_v_first; the output and the final
state returned, with gradients through the initial state; gates given as natural logarithms;
q, k, v, beta taken as given (already normalised / activated); packed sequences by cu_seqlens.

The page prints no formula.  Readings taken (the plainest form of a gated delta rule, listed
with the other readings of the pages in the design notes):
  per sequence and value head h (key head h // (Hv / Hk)), per token t, S the [Dk, Dv] state:
    S' = D_t S                 D_t = exp(g_t) (GDN) or diag(exp(g_t)) (KDA)
    u  = beta_t (v_t - S'^T k_t)
    S  = S' + k_t u^T
    o_t = scale S^T q_t        scale = Dk ** -0.5 unless given
Backward (L = sum o do + sum S_final dS_final), per token in reverse, dS the gradient of S_t:
    dS += scale q do^T;  dq = scale S_t do
    dk = dS u;  du = dS^T k;  dS' = dS
    dbeta = du . (v - w) with w = S'^T k;  dv = beta du;  dw = -beta du
    dS' += k dw^T;  dk += S' dw
    GDN: dg = <dS', S'>;  KDA: dg_i = sum_j dS'_ij S'_ij;  dS_{t-1} = D_t dS'
and dh0 = dS after the sequence's first token.  dq, dk of a key head sum over its value heads.

Every function has pins in ``tests/test_delta_rule_oracle.py`` (closed forms, exact retrieval
and overwrite, invariants, central finite differences); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _sequences(B, T, cu_seqlens):
    """(row, start, end) of every sequence: the batch rows, or the packed ranges of row 0."""
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    assert B == 1 and cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    return [(0, int(cu[s]), int(cu[s + 1])) for s in range(len(cu) - 1)]


def _check(q, k, v, g, beta):
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T) and Hv % Hk == 0
    assert beta.shape == (B, T, Hv)
    kda = g.ndim == 4
    assert g.shape == ((B, T, Hv, Dk) if kda else (B, T, Hv))
    return B, T, Hk, Hv, Dk, Dv, kda


def _state_in(h, n, hv, Dk, Dv, v_first):
    if h is None:
        return np.zeros((Dk, Dv))
    s = np.asarray(h[n, hv], dtype=np.float64)
    return s.T.copy() if v_first else s.copy()


def forward(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
            state_v_first=False):
    """Returns (o [B, T, Hv, Dv], final_state [N, Hv, Dk, Dv] or [N, Hv, Dv, Dk])."""
    q, k, v, g, beta = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta))
    B, T, Hk, Hv, Dk, Dv, kda = _check(q, k, v, g, beta)
    scale = Dk ** -0.5 if scale is None else float(scale)
    seqs = _sequences(B, T, cu_seqlens)
    grp = Hv // Hk
    o = np.zeros((B, T, Hv, Dv))
    fin = np.zeros((len(seqs), Hv) + ((Dv, Dk) if state_v_first else (Dk, Dv)))
    for n, (b, t0, t1) in enumerate(seqs):
        for hv in range(Hv):
            hk = hv // grp
            S = _state_in(initial_state, n, hv, Dk, Dv, state_v_first)
            for t in range(t0, t1):
                a = np.exp(g[b, t, hv])
                S = a[:, None] * S if kda else a * S
                u = beta[b, t, hv] * (v[b, t, hv] - S.T @ k[b, t, hk])
                S = S + np.outer(k[b, t, hk], u)
                o[b, t, hv] = scale * (S.T @ q[b, t, hk])
            fin[n, hv] = S.T if state_v_first else S
    return o, fin


def backward(q, k, v, g, beta, do, dfinal=None, scale=None, initial_state=None,
             cu_seqlens=None, state_v_first=False):
    """Gradients of L = sum o do + sum final dfinal: dict of dq, dk [B, T, Hk, Dk], dv, dg, dbeta
    (the shapes of v, g, beta) and dh0 (the shape of the states)."""
    q, k, v, g, beta, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta, do))
    B, T, Hk, Hv, Dk, Dv, kda = _check(q, k, v, g, beta)
    scale = Dk ** -0.5 if scale is None else float(scale)
    seqs = _sequences(B, T, cu_seqlens)
    grp = Hv // Hk
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dh0 = np.zeros((len(seqs), Hv) + ((Dv, Dk) if state_v_first else (Dk, Dv)))
    for n, (b, t0, t1) in enumerate(seqs):
        for hv in range(Hv):
            hk = hv // grp
            # forward again, keeping every token's decayed state S', w and u
            S = _state_in(initial_state, n, hv, Dk, Dv, state_v_first)
            Sp, W, U = {}, {}, {}
            for t in range(t0, t1):
                a = np.exp(g[b, t, hv])
                S = a[:, None] * S if kda else a * S
                Sp[t] = S
                W[t] = S.T @ k[b, t, hk]
                U[t] = beta[b, t, hv] * (v[b, t, hv] - W[t])
                S = S + np.outer(k[b, t, hk], U[t])
            if dfinal is None:
                dS = np.zeros((Dk, Dv))
            else:
                dS = np.asarray(dfinal[n, hv], dtype=np.float64)
                dS = dS.T.copy() if state_v_first else dS.copy()
            for t in range(t1 - 1, t0 - 1, -1):
                kt, qt, dot = k[b, t, hk], q[b, t, hk], do[b, t, hv]
                St = Sp[t] + np.outer(kt, U[t])
                dq[b, t, hk] += scale * (St @ dot)
                dS = dS + scale * np.outer(qt, dot)
                dk_t = dS @ U[t]
                du = dS.T @ kt
                dSp = dS.copy()
                dbeta[b, t, hv] = du @ (v[b, t, hv] - W[t])
                dv[b, t, hv] = beta[b, t, hv] * du
                dw = -beta[b, t, hv] * du
                dSp += np.outer(kt, dw)
                dk_t += Sp[t] @ dw
                dk[b, t, hk] += dk_t
                a = np.exp(g[b, t, hv])
                if kda:
                    dg[b, t, hv] = np.sum(dSp * Sp[t], axis=1)
                    dS = a[:, None] * dSp
                else:
                    dg[b, t, hv] = np.sum(dSp * Sp[t])
                    dS = a * dSp
            dh0[n, hv] = dS.T if state_v_first else dS
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dh0": dh0}
