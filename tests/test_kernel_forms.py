"""The rearranged forms the kernels compute, restated in fp64 and held
against the oracle's rule, on CPU.

Decode step ("mstar PR #1139", "Why": the recurrent state update of one
token).  Each value row i of the state is updated on its own from two dot
products of the row, u_i = S_i·k̂ and w_i = S_i·q̂, and κ = k̂·q̂:

    c_i = β (v_i - α u_i),   S'_i = α S_i + c_i k̂,   o_i = α w_i + c_i κ

which is S' = α S (I - β k̂ k̂ᵀ) + β v k̂ᵀ and o = S' q̂.

Chunked prefill.  The pages name a chunked GDN path ("mstar PR #965", "Correctness"; "mstar PR
#1127": one GDN prefill kernel) but print no formula.  The tensor-core
prefill uses this regrouping, derived from the recurrence
S_t = α_t S_{t-1} + u_t k̂_tᵀ, u_t = β_t (v_t - α_t S_{t-1} k̂_t).  With G the
running sum of log α inside a chunk of C tokens:

    A[t][s] = β_t e^{G_t - G_s} k̂_t·k̂_s  (s < t),    T = (I + A)⁻¹
    P[t][s] = e^{G_t - G_s} q̂_t·k̂_s      (s ≤ t)
    E  = (Vᵀ - (S Kᵀ) diag(e^G)) diag(β),   Uᵀ = E Tᵀ
    Oᵀ = (S Qᵀ) diag(e^G) + Uᵀ Pᵀ
    S  ← e^{G_C} S + Uᵀ diag(e^{G_C - G}) K

Here the equations are restated in numpy, tokens as matrix rows, and held
against the oracle on small inputs: chunks of 4 and 8 tokens, whole chunks
and ragged tails, one-token sequences, grouped heads.  Planted mistakes in
the restatement (a dropped decay, a strict instead of an inclusive triangle,
a dropped β) must break the agreement, so the comparison can tell.
"""
import numpy as np
import pytest

import oracle


def test_decode_row_form_equals_the_rule():
    """The decode kernels' per-row form against the oracle's literal matrix
    form, on random heads, including the edge gates α = 1 and β = 0 or 1."""
    rng = np.random.default_rng(5)
    dk, dv = 16, 12
    for al, be in [(0.83, 0.37), (1.0, 0.0), (1.0, 1.0), (0.05, 0.99)]:
        S = rng.normal(0.0, 0.5, (dv, dk))
        qh = oracle.l2norm(rng.normal(0.0, 1.0, dk), scale=dk ** -0.5)
        kh = oracle.l2norm(rng.normal(0.0, 1.0, dk))
        v = rng.normal(0.0, 1.0, dv)
        S_ref, o_ref = oracle.rule(S, qh, kh, v, al, be)
        u, w, kappa = S @ kh, S @ qh, kh @ qh
        c = be * (v - al * u)
        S_new = al * S + np.outer(c, kh)
        o = al * w + c * kappa
        assert np.abs(S_new - S_ref).max() <= 1e-14 * max(1.0, np.abs(S_ref).max())
        assert np.abs(o - o_ref).max() <= 1e-14 * max(1.0, np.abs(o_ref).max())

HK, HV, DK, DV = 2, 4, 8, 6          # two value heads a qk head
LENS = [9, 16, 1, 0, 13]


def chunked_sequence(S, qh, kh, v, al, be, C, mistake=None):
    """One sequence, one value head: S [dv][dk], qh/kh [L][dk], v [L][dv],
    al/be [L].  Returns (final state, outputs [L][dv])."""
    S = S.copy()
    L = len(al)
    out = np.empty((L, S.shape[0]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        n = sl.stop - sl.start
        Q, K, V, bt = qh[sl], kh[sl], v[sl], be[sl]
        if mistake == "no_beta":
            bt = np.ones(n)
        G = np.cumsum(np.log(al[sl]))
        D = np.exp(G[:, None] - G[None, :])          # e^{G_t - G_s}
        A = np.tril(bt[:, None] * (D if mistake != "no_decay_in_A" else 1.0) * (K @ K.T), -1)
        P = np.tril(D * (Q @ K.T), -1 if mistake == "strict_P" else 0)
        T = np.linalg.inv(np.eye(n) + A)
        E = (V.T - (S @ K.T) * np.exp(G)[None, :]) * bt[None, :]
        Ut = E @ T.T
        out[sl] = ((S @ Q.T) * np.exp(G)[None, :] + Ut @ P.T).T
        S = np.exp(G[-1]) * S + (Ut * np.exp(G[-1] - G)[None, :]) @ K
    return S, out


def make_case(seed):
    rng = np.random.default_rng(seed)
    T = sum(LENS)
    nseq = len(LENS)
    cu = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32)
    q = rng.normal(0.0, 1.0, (T, HK, DK))
    k = rng.normal(0.0, 1.0, (T, HK, DK))
    v = rng.normal(0.0, 1.0, (T, HV, DV))
    a = rng.normal(0.0, 1.0, (T, HV))
    b = rng.normal(0.0, 1.0, (T, HV))
    A_log = np.log(rng.uniform(0.5, 4.0, HV))
    dt_bias = rng.normal(0.0, 0.5, HV)
    num_slots = 1 + 2 * nseq
    pool = np.zeros((num_slots, HV, DV, DK))
    pool[1:] = rng.normal(0.0, 0.5, (num_slots - 1, HV, DV, DK))
    rs = np.arange(1, nseq + 1, dtype=np.int32)
    ws = rs + nseq
    return cu, q, k, v, a, b, A_log, dt_bias, pool, rs, ws


def regrouped(case, C, mistake=None):
    cu, q, k, v, a, b, A_log, dt_bias, pool, rs, ws = case
    group = HV // HK
    states, out = {}, np.zeros((q.shape[0], HV, DV))
    for r in range(len(LENS)):
        t0, t1 = cu[r], cu[r + 1]
        for h in range(HV):
            g = h // group
            qh = np.array([oracle.l2norm(q[t, g], scale=DK ** -0.5) for t in range(t0, t1)]).reshape(-1, DK)
            kh = np.array([oracle.l2norm(k[t, g]) for t in range(t0, t1)]).reshape(-1, DK)
            al = np.array([oracle.alpha(A_log[h], a[t, h], dt_bias[h]) for t in range(t0, t1)])
            be = np.array([oracle.beta(b[t, h]) for t in range(t0, t1)])
            S, o = chunked_sequence(pool[rs[r], h], qh, kh, v[t0:t1, h], al, be, C, mistake)
            states[(r, h)] = S
            out[t0:t1, h] = o
    return states, out


def serial(case):
    cu, q, k, v, a, b, A_log, dt_bias, pool, rs, ws = case
    p = pool.copy()
    out, bad = oracle.prefill(cu, q, k, v, a, b, A_log, dt_bias, p, rs, write_slot=ws)
    assert bad == 0
    return p, out


def worst(case, C, mistake=None):
    p, o_ref = serial(case)
    states, out = regrouped(case, C, mistake)
    _, _, _, _, _, _, _, _, _, rs, ws = case
    err_s = max(np.abs(states[(r, h)] - p[ws[r], h]).max() / np.abs(p[ws[r], h]).max()
                for r in range(len(LENS)) for h in range(HV))
    err_o = np.abs(out - o_ref).max() / np.abs(o_ref).max()
    return err_s, err_o


@pytest.mark.parametrize("C", [4, 8])
def test_regrouping_equals_the_token_serial_rule(C):
    err_s, err_o = worst(make_case(7), C)
    assert err_s < 1e-12 and err_o < 1e-12, (err_s, err_o)


@pytest.mark.parametrize("mistake", ["no_decay_in_A", "strict_P", "no_beta"])
def test_planted_mistakes_are_caught(mistake):
    err_s, err_o = worst(make_case(7), 8, mistake)
    assert max(err_s, err_o) > 1e-3, (mistake, err_s, err_o)
