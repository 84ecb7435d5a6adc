"""Pins for the fp64 oracle: closed forms, special cases, a hand-worked example,
an unrolled product of transition matrices, library routines and brute force.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a swapped index or tap order) fails it.  The
rule and gates are the gated delta rule of a GDN decode step; the slot rules
follow the mstar PR #1139 page (section "What changed": twin slots, commit
swap, in place) and the PR #1127 / PR #965 pages (padding on the null slot).
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# gates
# --------------------------------------------------------------------------

def test_softplus_closed_forms(orc):
    assert orc.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    # softplus(ln(e - 1)) = ln(1 + e - 1) = 1
    assert orc.softplus(math.log(math.e - 1.0)) == pytest.approx(1.0, abs=1e-15)
    # softplus(x) - softplus(-x) = x for every x
    for x in (-7.5, -0.3, 0.9, 4.0, 19.0):
        assert orc.softplus(x) - orc.softplus(-x) == pytest.approx(x, abs=1e-13)
    # large x: the value is x itself; very negative x: e^x
    assert orc.softplus(50.0) == 50.0
    assert orc.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)


def test_alpha_closed_forms(orc):
    # exp(A_log) = 1, softplus(0) = ln 2  ->  alpha = exp(-ln 2) = 1/2
    assert orc.alpha(0.0, 0.0, 0.0) == pytest.approx(0.5, abs=1e-16)
    # the gate adds a and dt_bias before softplus
    assert orc.alpha(0.0, 1.25, -1.25) == pytest.approx(0.5, abs=1e-16)
    # exp(A_log) = 2, softplus(ln(e-1)) = 1  ->  alpha = e^-2
    assert orc.alpha(math.log(2.0), math.log(math.e - 1.0), 0.0) == pytest.approx(math.exp(-2.0), rel=1e-14)
    # A_log = -inf: no decay, alpha = 1 exactly
    assert orc.alpha(-math.inf, 0.3, -0.7) == 1.0
    assert orc.alpha(-math.inf, math.inf, 0.0) == 1.0
    # softplus -> inf with a finite rate: alpha = 0 exactly
    assert orc.alpha(0.0, math.inf, 0.0) == 0.0
    # decays more for a larger step size, always in (0, 1)
    vals = [orc.alpha(0.7, a, 0.1) for a in (-3.0, -1.0, 0.0, 1.0, 3.0)]
    assert all(0.0 < x < 1.0 for x in vals)
    assert all(x > y for x, y in zip(vals, vals[1:]))


def test_beta_closed_forms(orc):
    assert orc.beta(0.0) == 0.5
    assert orc.beta(math.log(3.0)) == pytest.approx(0.75, abs=1e-16)
    assert orc.beta(-math.log(3.0)) == pytest.approx(0.25, abs=1e-16)
    assert orc.beta(-math.inf) == 0.0
    assert orc.beta(math.inf) == 1.0


# --------------------------------------------------------------------------
# bfloat16 rounding (checked against torch's float32 -> bfloat16 conversion,
# which rounds to nearest even, and against hand-picked ties)
# --------------------------------------------------------------------------

def test_round_bf16_special_values(orc):
    one = 1.0
    assert orc.round_bf16([one + 2.0 ** -8])[0] == one                      # tie -> even (1)
    assert orc.round_bf16([one + 3 * 2.0 ** -8])[0] == one + 2.0 ** -6     # tie -> even (odd below)
    assert orc.round_bf16([one + 2.0 ** -8 + 2.0 ** -30])[0] == one + 2.0 ** -7  # past the tie
    assert orc.round_bf16([-(one + 2.0 ** -8)])[0] == -one
    assert orc.round_bf16([3.4e38])[0] == math.inf                         # past max + half spacing
    assert orc.round_bf16([3.39e38])[0] == 255.0 / 128.0 * 2.0 ** 127           # just above max: max
    tiny = 2.0 ** -133                                                     # smallest subnormal
    assert orc.round_bf16([tiny])[0] == tiny
    assert orc.round_bf16([1.5 * tiny])[0] == 2 * tiny                     # tie -> even
    assert orc.round_bf16([0.49 * tiny])[0] == 0.0
    assert orc.round_bf16([0.0])[0] == 0.0


def test_round_bf16_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x32 = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(500) * 1e-38).astype(np.float32),
        (rng.standard_normal(500) * 1e30).astype(np.float32),
    ])
    # exact ties: a bfloat16 value with the bit just below its last kept bit set
    bf = torch.from_numpy(x32[:1000]).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (bf.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x32 = np.concatenate([x32, ties])
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.round_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# L2 normalisation
# --------------------------------------------------------------------------

def test_l2norm(orc):
    y = orc.l2norm([3.0, 4.0], eps=0.0)
    assert y == pytest.approx([0.6, 0.8], abs=2e-16)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    y = orc.l2norm(x, eps=0.0, scale=1.0)
    assert np.linalg.norm(y) == pytest.approx(1.0, abs=1e-14)
    assert np.allclose(orc.l2norm(5.0 * x, eps=0.0), y, atol=1e-15, rtol=0)
    # eps sits inside the square root: |y| = |x| / sqrt(|x|^2 + eps)
    y = orc.l2norm([1.0, 0.0], eps=3.0)
    assert y == pytest.approx([0.5, 0.0], abs=1e-16)
    y = orc.l2norm(x, eps=0.0, scale=0.25)
    assert np.linalg.norm(y) == pytest.approx(0.25, abs=1e-14)


# --------------------------------------------------------------------------
# the rule, literal matrix form
# --------------------------------------------------------------------------

def test_rule_hand_worked_2x2(orc):
    g = _load("rule_2x2.json")
    for case in g["cases"]:
        S_new, o = orc.rule(g["S"], case["qhat"], g["khat"], g["v"], g["alpha"], g["beta"])
        assert np.allclose(S_new, g["S_new"], atol=1e-14, rtol=0)
        assert np.allclose(o, case["o"], atol=1e-14, rtol=0)


def _unit(rng, n):
    x = rng.standard_normal(n)
    return x / np.linalg.norm(x)


@pytest.mark.parametrize("dk,dv", [(4, 4), (16, 16), (8, 4), (4, 12)])
def test_rule_special_cases(orc, dk, dv):
    rng = np.random.default_rng(dk * 100 + dv)
    S = rng.standard_normal((dv, dk))
    q = _unit(rng, dk)
    k = _unit(rng, dk)
    v = rng.standard_normal(dv)
    # beta = 0, alpha = 1: the state is unchanged, bit for bit
    S1, o1 = orc.rule(S, q, k, v, 1.0, 0.0)
    assert np.array_equal(S1, S)
    assert np.allclose(o1, S @ q, atol=1e-13, rtol=0)
    # alpha = 1, beta = 1, unit k: the state now maps k to v
    S1, _ = orc.rule(S, q, k, v, 1.0, 1.0)
    assert np.allclose(S1 @ k, v, atol=1e-13, rtol=0)
    # general gates with unit k: S' k = alpha (1 - beta) S k + beta v
    for a_, b_ in ((0.3, 0.8), (0.9, 0.1), (0.55, 0.5)):
        S1, _ = orc.rule(S, q, k, v, a_, b_)
        assert np.allclose(S1 @ k, a_ * (1 - b_) * (S @ k) + b_ * v, atol=1e-13, rtol=0)
        # directions orthogonal to k are only decayed: S' x = alpha S x for x . k = 0
        x = rng.standard_normal(dk)
        x -= (x @ k) * k
        assert np.allclose(S1 @ x, a_ * (S @ x), atol=1e-13, rtol=0)
    # alpha = 0: the state is replaced by beta v k^T
    S1, _ = orc.rule(S, q, k, v, 0.0, 0.35)
    assert np.allclose(S1, 0.35 * np.outer(v, k), atol=1e-15, rtol=0)
    # the output reads the NEW state: o = S' q; with q = e_j it is column j of S'
    for j in (0, dk - 1):
        e = np.zeros(dk)
        e[j] = 1.0
        S1, o = orc.rule(S, e, k, v, 0.6, 0.4)
        assert np.array_equal(o, S1[:, j])


def test_rule_is_row_separable(orc):
    """With v = 0 the map S -> S' is linear; built column by column from basis
    matrices it equals I_dv (x) A^T on row-major vec(S), A = alpha (I - beta k k^T):
    each value row of the state is updated on its own."""
    rng = np.random.default_rng(3)
    dk, dv = 4, 3
    k = _unit(rng, dk)
    q = _unit(rng, dk)
    a_, b_ = 0.7, 0.45
    n = dv * dk
    T = np.zeros((n, n))
    for c in range(n):
        E = np.zeros(n)
        E[c] = 1.0
        S1, _ = orc.rule(E.reshape(dv, dk), q, k, np.zeros(dv), a_, b_)
        T[:, c] = S1.ravel()
    A = a_ * (np.eye(dk) - b_ * np.outer(k, k))
    assert np.allclose(T, np.kron(np.eye(dv), A.T), atol=1e-15, rtol=0)


@pytest.mark.parametrize("dk,dv", [(4, 4), (16, 16)])
def test_rule_unrolled_product(orc, dk, dv):
    """T recurrent steps equal the unrolled product of the transition matrices:
    S_T = S_0 A_1 ... A_T + sum_t beta_t v_t k_t^T A_{t+1} ... A_T,
    A_t = alpha_t (I - beta_t k_t k_t^T)."""
    rng = np.random.default_rng(11 + dk)
    T = 8
    S0 = rng.standard_normal((dv, dk)) * 0.1
    ks = [_unit(rng, dk) for _ in range(T)]
    vs = [rng.standard_normal(dv) for _ in range(T)]
    als = rng.uniform(0.2, 1.0, T)
    bes = rng.uniform(0.0, 1.0, T)
    q = _unit(rng, dk)
    S = S0
    for t in range(T):
        S, _ = orc.rule(S, q, ks[t], vs[t], als[t], bes[t])
    A = [als[t] * (np.eye(dk) - bes[t] * np.outer(ks[t], ks[t])) for t in range(T)]

    def prod(lo):
        P = np.eye(dk)
        for s in range(lo, T):
            P = P @ A[s]
        return P

    closed = S0 @ prod(0)
    for t in range(T):
        closed = closed + bes[t] * np.outer(vs[t], ks[t]) @ prod(t + 1)
    assert np.allclose(S, closed, atol=1e-12, rtol=0)


def test_head_basis_aligned_inputs(orc):
    """Raw inputs whose normalisation and gates are known in closed form:
    k along e_1 with length 5, q = (3, 4, 0, ...), exp(A_log) = 1 with
    a + dt_bias = 0 (alpha = 1/2), b = ln 3 (beta = 3/4)."""
    rng = np.random.default_rng(5)
    dk, dv = 8, 6
    S = rng.standard_normal((dv, dk))
    q = np.zeros(dk)
    q[0], q[1] = 3.0, 4.0
    k = np.zeros(dk)
    k[1] = 5.0
    v = rng.standard_normal(dv)
    S1, o = orc.head(S, q, k, v, a=0.4, b=math.log(3.0), A_log=0.0, dt_bias=-0.4)
    kn = 5.0 / math.sqrt(25.0 + 1e-6)          # |k^| slightly below 1 because of eps
    qs = 1.0 / math.sqrt(25.0 + 1e-6) / math.sqrt(dk)
    exp = 0.5 * S.copy()
    # only column 1 (the direction of k) feels the delta term
    exp[:, 1] = 0.5 * S[:, 1] * (1.0 - 0.75 * kn * kn) + 0.75 * v * kn
    assert np.allclose(S1, exp, atol=1e-14, rtol=0)
    assert np.allclose(o, (3.0 * exp[:, 0] + 4.0 * exp[:, 1]) * qs, atol=1e-14, rtol=0)


# --------------------------------------------------------------------------
# conv
# --------------------------------------------------------------------------

def test_conv_row_hand_worked(orc):
    g = _load("conv_row_w4.json")
    y, nw = orc.conv_row(g["win"], g["x"], g["w"], g["bias"], silu=False)
    assert np.array_equal(y, np.array(g["pre"]))
    assert np.array_equal(nw, np.array(g["new_win"]))
    y, _ = orc.conv_row(g["win"], g["x"], g["w"], None, silu=False)
    assert np.array_equal(y, np.array(g["pre"]) - np.array(g["bias"]))


def test_conv_row_taps_and_silu(orc):
    rng = np.random.default_rng(9)
    C, W = 5, 4
    win = rng.standard_normal((W - 1, C))
    x = rng.standard_normal(C)
    for tap in range(W):
        w = np.zeros((C, W))
        w[:, tap] = 1.0
        y, nw = orc.conv_row(win, x, w, np.zeros(C), silu=False)
        expect = x if tap == W - 1 else win[tap]            # tap W-1 is the current token
        assert np.array_equal(y, expect)
        assert np.array_equal(nw[:-1], win[1:]) and np.array_equal(nw[-1], x)
    # silu closed forms: silu(0) = 0, silu(ln 3) = (3/4) ln 3, silu(-ln 3) = -(1/4) ln 3
    w = np.zeros((3, W))
    w[:, W - 1] = 1.0
    xs = np.array([0.0, math.log(3.0), -math.log(3.0)])
    y, _ = orc.conv_row(np.zeros((W - 1, 3)), xs, w, None, silu=True)
    assert y == pytest.approx([0.0, 0.75 * math.log(3.0), -0.25 * math.log(3.0)], abs=1e-15)


def test_conv_sequence_equals_numpy_convolve(orc):
    """Feeding a token sequence one at a time through the decode conv (starting
    from a zero window) equals the causal part of numpy's full convolution."""
    rng = np.random.default_rng(13)
    C, W, T = 6, 4, 20
    w = rng.standard_normal((C, W))
    xs = rng.standard_normal((T, C))
    win = np.zeros((W - 1, C))
    ys = []
    for t in range(T):
        y, win = orc.conv_row(win, xs[t], w, None, silu=False)
        ys.append(y)
    ys = np.array(ys)
    for c in range(C):
        # y_t = sum_j w[j] x_{t-(W-1)+j}: the kernel reversed in np.convolve's convention
        ref = np.convolve(xs[:, c], w[c, ::-1])[:T]
        assert np.allclose(ys[:, c], ref, atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# pool / slot semantics
# --------------------------------------------------------------------------

def _pool_case(rng, rows=5, hk=2, hv=4, dk=8, dv=8, num_slots=12):
    pool = rng.standard_normal((num_slots, hv, dv, dk)) * 0.1
    pool[0] = 0.0
    q = rng.standard_normal((rows, hk, dk))
    k = rng.standard_normal((rows, hk, dk))
    v = rng.standard_normal((rows, hv, dv))
    a = rng.standard_normal((rows, hv))
    b = rng.standard_normal((rows, hv))
    A_log = rng.uniform(0, math.log(16), hv)
    dt_bias = rng.uniform(-1, 1, hv)
    return pool, q, k, v, a, b, A_log, dt_bias


def test_step_twin_and_in_place(orc):
    rng = np.random.default_rng(21)
    pool, q, k, v, a, b, A_log, dt_bias = _pool_case(rng)
    hk, hv = q.shape[1], pool.shape[1]
    rs = np.array([3, 0, 5, 1, 8], dtype=np.int32)      # row 1 is padding
    ws = np.array([4, 0, 6, 2, 9], dtype=np.int32)
    twin = pool.copy()
    out_t, bad = orc.step(q, k, v, a, b, A_log, dt_bias, twin, rs, ws, keep_in_place=False)
    assert bad == 0
    inpl = pool.copy()
    out_i, bad = orc.step(q, k, v, a, b, A_log, dt_bias, inpl, rs, ws, keep_in_place=True)
    assert bad == 0
    assert np.array_equal(out_t, out_i)                 # same values either way
    assert np.all(out_t[1] == 0.0)                      # padding row output is zero
    written = set(ws[ws > 0].tolist())
    for s in range(pool.shape[0]):
        if s not in written:                            # read slots and the null slot untouched
            assert np.array_equal(twin[s], pool[s]), s
    for r in range(len(rs)):
        if rs[r] == 0:
            continue
        assert np.array_equal(twin[ws[r]], inpl[rs[r]])
        for h in range(hv):
            g = h // (hv // hk)                         # v head h reads qk head h / (hv/hk)
            S1, o = orc.head(pool[rs[r], h], q[r, g], k[r, g], v[r, h], a[r, h], b[r, h],
                             A_log[h], dt_bias[h])
            assert np.array_equal(S1, twin[ws[r], h])
            assert np.array_equal(o, out_t[r, h])


def test_step_gqa_mapping_is_consecutive(orc):
    """Changing the q/k of qk head 1 changes v heads 2 and 3 only (group of 2)."""
    rng = np.random.default_rng(22)
    pool, q, k, v, a, b, A_log, dt_bias = _pool_case(rng, rows=2, hk=2, hv=4)
    rs = np.array([1, 2], dtype=np.int32)
    ws = np.array([3, 4], dtype=np.int32)
    p1 = pool.copy()
    o1, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p1, rs, ws)
    q2, k2 = q.copy(), k.copy()
    q2[:, 1] += 1.0
    k2[:, 1] -= 0.5
    p2 = pool.copy()
    o2, _ = orc.step(q2, k2, v, a, b, A_log, dt_bias, p2, rs, ws)
    assert np.array_equal(o1[:, :2], o2[:, :2])
    assert not np.allclose(o1[:, 2:], o2[:, 2:])
    assert np.array_equal(p1[3:5, :2], p2[3:5, :2])


def test_step_bad_slots_are_reported(orc):
    rng = np.random.default_rng(23)
    pool, q, k, v, a, b, A_log, dt_bias = _pool_case(rng, rows=3)
    rs = np.array([2, 99, 1], dtype=np.int32)           # row 1 reads past the pool
    ws = np.array([3, 4, 0], dtype=np.int32)            # row 2 would write the null slot
    p = pool.copy()
    out, bad = orc.step(q, k, v, a, b, A_log, dt_bias, p, rs, ws)
    assert bad == 2
    assert np.all(out[1:] == 0.0)
    assert np.array_equal(p[0], pool[0]) and np.array_equal(p[4], pool[4])


def test_twin_write_must_name_the_other_slot(orc):
    """A twin step writes the next state to the request's other slot; a twin
    row naming its read slot as write slot is rejected, in the rule and the conv."""
    rng = np.random.default_rng(26)
    pool, q, k, v, a, b, A_log, dt_bias = _pool_case(rng, rows=2)
    rs = np.array([2, 3], dtype=np.int32)
    ws = np.array([2, 4], dtype=np.int32)
    p = pool.copy()
    out, bad = orc.step(q, k, v, a, b, A_log, dt_bias, p, rs, ws)
    assert bad == 1 and np.all(out[0] == 0.0) and np.array_equal(p[2], pool[2])
    assert not np.array_equal(p[4], pool[4])
    p = pool.copy()
    _, bad = orc.step(q, k, v, a, b, A_log, dt_bias, p, rs, ws, keep_in_place=True)
    assert bad == 0
    cp = rng.standard_normal((6, 3, 8))
    y, bad = orc.conv_step(rng.standard_normal((2, 8)), cp, rs, ws, rng.standard_normal((8, 4)), None)
    assert bad == 1 and np.all(y[0] == 0.0)


def test_commit_swaps(orc):
    rs = np.array([1, 0, 5], dtype=np.int32)
    ws = np.array([2, 0, 6], dtype=np.int32)
    orc.commit(rs, ws)
    assert rs.tolist() == [2, 0, 6] and ws.tolist() == [1, 0, 5]


def test_conv_step_slots(orc):
    rng = np.random.default_rng(24)
    C, W, S = 10, 4, 7
    cp = rng.standard_normal((S, W - 1, C))
    cp[0] = 0.0
    x = rng.standard_normal((3, C))
    w = rng.standard_normal((C, W))
    bias = rng.standard_normal(C)
    rs = np.array([2, 0, 4], dtype=np.int32)
    ws = np.array([3, 0, 5], dtype=np.int32)
    twin = cp.copy()
    y_t, bad = orc.conv_step(x, twin, rs, ws, w, bias)
    assert bad == 0
    inpl = cp.copy()
    y_i, _ = orc.conv_step(x, inpl, rs, None, w, bias)
    assert np.array_equal(y_t, y_i) and np.all(y_t[1] == 0)
    for s in (0, 1, 2, 4, 6):
        assert np.array_equal(twin[s], cp[s])
    assert np.array_equal(twin[3], inpl[2]) and np.array_equal(twin[5], inpl[4])
    for r in (0, 2):
        y, nw = orc.conv_row(cp[rs[r]], x[r], w, bias, silu=True)
        assert np.array_equal(y, y_t[r]) and np.array_equal(nw, twin[ws[r]])


def test_layer_identity_conv_reduces_to_step(orc):
    """With the conv reduced to the identity (tap 3 = 1, no bias, no SiLU) and
    binary32-exact inputs, the layer is exactly the decode step on the split x."""
    rng = np.random.default_rng(25)
    hk, hv, dk, dv, W = 2, 4, 8, 8, 4
    C = 2 * hk * dk + hv * dv
    pool, _, _, _, a, b, A_log, dt_bias = _pool_case(rng, rows=3, hk=hk, hv=hv, dk=dk, dv=dv)
    x = rng.standard_normal((3, C)).astype(np.float32).astype(np.float64)
    cp = rng.standard_normal((pool.shape[0], W - 1, C))
    w = np.zeros((C, W))
    w[:, W - 1] = 1.0
    rs = np.array([1, 0, 2], dtype=np.int32)
    ws = np.array([3, 0, 4], dtype=np.int32)
    p1 = pool.copy()
    o1, _ = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p1, rs, ws, hk=hk,
                      act_bf16=False, silu=False)
    q = x[:, :hk * dk].reshape(3, hk, dk)
    k = x[:, hk * dk:2 * hk * dk].reshape(3, hk, dk)
    v = x[:, 2 * hk * dk:].reshape(3, hv, dv)
    p2 = pool.copy()
    o2, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p2, rs, ws)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)


# --------------------------------------------------------------------------
# the layer's composition: conv, rounding to the activation type, split, rule
# ("mstar PR #1139", "What changed": the decode conv, with its optional
# activation and its write slot, runs ahead of the GDN decode kernel)
# --------------------------------------------------------------------------

def _layer_case(rng, rows=3, hk=2, hv=4, dk=8, dv=8, W=4):
    C = 2 * hk * dk + hv * dv
    pool, _, _, _, a, b, A_log, dt_bias = _pool_case(rng, rows=rows, hk=hk, hv=hv, dk=dk, dv=dv)
    cp = rng.standard_normal((pool.shape[0], W - 1, C))
    cp[0] = 0.0
    w = np.zeros((C, W))
    w[:, W - 1] = 1.0                                   # identity taps: y = x before the activation
    return C, pool, cp, w, a, b, A_log, dt_bias


def _split(y, hk, hv, dk, dv):
    rows = y.shape[0]
    return (y[:, :hk * dk].reshape(rows, hk, dk), y[:, hk * dk:2 * hk * dk].reshape(rows, hk, dk),
            y[:, 2 * hk * dk:].reshape(rows, hv, dv))


def _bf16_grid_values(rng, shape):
    """Values with 8 significant bits (m * 2^(e-7), m in 129..255) and offsets of
    under 0.45 of their spacing: each rounds to the nearest bfloat16 value m * 2^(e-7)
    by construction, with no rounding routine involved."""
    m = rng.integers(129, 256, size=shape).astype(np.float64)
    e = rng.integers(-3, 3, size=shape)
    sign = np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    spacing = np.ldexp(1.0, e - 7)
    exact = sign * m * spacing
    off = rng.uniform(-0.45, 0.45, size=shape) * spacing
    off[np.abs(off) < 0.05 * spacing] = 0.25 * spacing[np.abs(off) < 0.05 * spacing]
    return exact, exact + off


def test_layer_rounds_the_conv_output_to_bf16(orc):
    """act_bf16: the conv output is rounded to bfloat16 before the rule.  With
    identity taps the layer must equal the step on the bfloat16 values the inputs
    round to (known by construction, plus hand-worked ties to even), and must
    differ from the step on the unrounded inputs."""
    rng = np.random.default_rng(41)
    hk, hv, dk, dv = 2, 4, 8, 8
    rows = 3
    C, pool, cp, w, a, b, A_log, dt_bias = _layer_case(rng, rows=rows, hk=hk, hv=hv, dk=dk, dv=dv)
    exact, x = _bf16_grid_values(rng, (rows, C))
    # hand-worked ties (bfloat16 spacing in [1, 2) is 2^-7): 1 + 2^-8 lies halfway
    # between 1 and 1 + 2^-7 and goes to the even 1; 1 + 3*2^-8 lies halfway between
    # 1 + 2^-7 and 1 + 2^-6 and goes to the even 1 + 2^-6; 1 + 2^-9 is below halfway
    x[0, :3] = [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -9]
    exact[0, :3] = [1.0, 1 + 2.0 ** -6, 1.0]
    rs = np.array([1, 0, 2], dtype=np.int32)
    ws = np.array([3, 0, 4], dtype=np.int32)
    p1 = pool.copy()
    o1, bad = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p1, rs, ws, hk=hk,
                        act_bf16=True, silu=False)
    assert bad == 0
    q, k, v = _split(exact, hk, hv, dk, dv)
    p2 = pool.copy()
    o2, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p2, rs, ws)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)
    q, k, v = _split(x, hk, hv, dk, dv)
    p3 = pool.copy()
    o3, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p3, rs, ws)
    assert not np.allclose(o1[[0, 2]], o3[[0, 2]], atol=1e-6, rtol=0)
    assert not np.allclose(p1, p3, atol=1e-7, rtol=0)


def test_layer_rounds_the_conv_output_to_f32(orc):
    """Without act_bf16 the conv output is rounded to binary32 (numpy's cast)."""
    rng = np.random.default_rng(42)
    hk, hv, dk, dv = 1, 2, 8, 8
    rows = 2
    C, pool, cp, w, a, b, A_log, dt_bias = _layer_case(rng, rows=rows, hk=hk, hv=hv, dk=dk, dv=dv)
    x = rng.standard_normal((rows, C)) * (1 + 2.0 ** -30)     # not binary32 values
    x32 = x.astype(np.float32).astype(np.float64)
    assert not np.array_equal(x, x32)
    rs = np.array([1, 2], dtype=np.int32)
    ws = np.array([3, 4], dtype=np.int32)
    p1 = pool.copy()
    o1, _ = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p1, rs, ws, hk=hk,
                      act_bf16=False, silu=False)
    q, k, v = _split(x32, hk, hv, dk, dv)
    p2 = pool.copy()
    o2, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p2, rs, ws)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)


def test_layer_forwards_silu(orc):
    """layer(silu=True) applies SiLU before the rounding and the rule.  With
    identity taps and x = ln m, SiLU gives the closed form ln(m) * m / (m + 1)
    (silu(ln 3) = 3/4 ln 3); rounded to binary32 (numpy) and to bfloat16 (torch)
    it must feed the step exactly."""
    rng = np.random.default_rng(43)
    hk, hv, dk, dv = 2, 2, 8, 8
    rows = 2
    C, pool, cp, w, a, b, A_log, dt_bias = _layer_case(rng, rows=rows, hk=hk, hv=hv, dk=dk, dv=dv)
    m = rng.uniform(0.05, 20.0, size=(rows, C))
    m[0, 0] = 3.0
    x = np.log(m)
    silu = x * m / (m + 1.0)
    assert silu[0, 0] == pytest.approx(0.75 * math.log(3.0), abs=1e-15)
    rs = np.array([1, 2], dtype=np.int32)
    ws = np.array([3, 4], dtype=np.int32)
    # binary32 activations
    p1 = pool.copy()
    o1, _ = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p1, rs, ws, hk=hk,
                      act_bf16=False, silu=True)
    y32 = silu.astype(np.float32).astype(np.float64)
    # the closed form and exp-based SiLU may differ in the last fp64 bits, which can
    # move a binary32 rounding only when the value sits on a midpoint: none here
    mid = np.abs(silu - y32) / np.maximum(np.abs(y32), 1e-300)
    assert np.all(np.abs(mid - 2.0 ** -24) > 1e-12)
    q, k, v = _split(y32, hk, hv, dk, dv)
    p2 = pool.copy()
    o2, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p2, rs, ws)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)
    # and without the activation the result differs
    p3 = pool.copy()
    o3, _ = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p3, rs, ws, hk=hk,
                      act_bf16=False, silu=False)
    assert not np.allclose(o1, o3, atol=1e-6, rtol=0)
    # bfloat16 activations (torch's round-to-nearest-even of the binary32 value;
    # the binary32 value is itself exact to 2^-24, far inside a bfloat16 spacing)
    torch = pytest.importorskip("torch")
    ybf = torch.from_numpy(y32).to(torch.bfloat16).to(torch.float64).numpy()
    p4 = pool.copy()
    o4, _ = orc.layer(x, cp.copy(), w, None, a, b, A_log, dt_bias, p4, rs, ws, hk=hk,
                      act_bf16=True, silu=True)
    q, k, v = _split(ybf, hk, hv, dk, dv)
    p5 = pool.copy()
    o5, _ = orc.step(q, k, v, a, b, A_log, dt_bias, p5, rs, ws)
    assert np.array_equal(o4, o5) and np.array_equal(p4, p5)


@pytest.mark.parametrize("keep_in_place", [False, True])
def test_layer_conv_window_goes_to_the_written_slot(orc, keep_in_place):
    """The layer's conv window follows its state: twin writes the new window
    [win[1], win[2], x] to the write slot and leaves the read slot alone; in
    place writes it back to the read slot and leaves the write slot alone."""
    rng = np.random.default_rng(44)
    hk, hv, dk, dv = 1, 2, 8, 8
    rows = 3
    C, pool, cp, w, a, b, A_log, dt_bias = _layer_case(rng, rows=rows, hk=hk, hv=hv, dk=dk, dv=dv)
    w = rng.standard_normal(w.shape) * 0.5              # any taps: the window is a plain copy
    x = rng.standard_normal((rows, C))
    rs = np.array([1, 0, 2], dtype=np.int32)
    ws = np.array([3, 0, 4], dtype=np.int32)
    c1 = cp.copy()
    p1 = pool.copy()
    orc.layer(x, c1, w, None, a, b, A_log, dt_bias, p1, rs, ws, hk=hk,
              keep_in_place=keep_in_place, act_bf16=False, silu=True)
    for r in (0, 2):
        new_win = np.concatenate([cp[rs[r], 1:], x[r][None]], axis=0)
        dst, other = (rs[r], ws[r]) if keep_in_place else (ws[r], rs[r])
        assert np.array_equal(c1[dst], new_win)
        assert np.array_equal(c1[other], cp[other])
        assert not np.array_equal(p1[dst], pool[dst])
        assert np.array_equal(p1[other], pool[other])
    for s in (0, 5, 6):
        assert np.array_equal(c1[s], cp[s]) and np.array_equal(p1[s], pool[s])
