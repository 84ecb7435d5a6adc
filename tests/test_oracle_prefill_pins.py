"""Pins for the oracle's many-tokens-a-sequence functions (prefill, speculative
verification, the conv over a sequence).

A prefill is the decode rule applied token after token ("mstar PR #1139",
section "Why": the rule is the recurrent state update; prefill keeps the state
in place), and verification keeps the state after every token ("What
changed": speculative decoding holds a state per token).  The checks: the
closed form of the unrolled product of transition matrices (numpy matrix
products, per token and at the end), the already pinned one-token step called
token by token, numpy's convolution for the conv, and the slot rules.
"""
import numpy as np
import pytest


def _unrolled(S0, ks, vs, als, bes):
    """States after each token from the closed form
    S_t = S_0 A_1..A_t + sum_{s<=t} beta_s v_s k_s^T A_{s+1}..A_t."""
    dk = S0.shape[1]
    A = [al * (np.eye(dk) - be * np.outer(k, k)) for k, al, be in zip(ks, als, bes)]
    out = []
    for t in range(len(ks)):
        def prod(lo, hi):
            P = np.eye(dk)
            for s in range(lo, hi):
                P = P @ A[s]
            return P
        S = S0 @ prod(0, t + 1)
        for s in range(t + 1):
            S = S + bes[s] * np.outer(vs[s], ks[s]) @ prod(s + 1, t + 1)
        out.append(S)
    return out


def _inputs(rng, T, hk, hv, dk, dv):
    return dict(q=rng.standard_normal((T, hk, dk)), k=rng.standard_normal((T, hk, dk)),
                v=rng.standard_normal((T, hv, dv)), a=rng.standard_normal((T, hv)),
                b=rng.standard_normal((T, hv)), A_log=rng.uniform(0, np.log(16), hv),
                dt_bias=rng.uniform(-1, 1, hv))


def _closed_form(orc, inp, S0, tokens, h, group):
    """(states after each token, outputs) of one sequence and value head."""
    g = h // group
    dk = inp["q"].shape[2]
    qh = [orc.l2norm(inp["q"][t, g], scale=1.0 / np.sqrt(dk)) for t in tokens]
    kh = [orc.l2norm(inp["k"][t, g]) for t in tokens]
    als = [orc.alpha(inp["A_log"][h], inp["a"][t, h], inp["dt_bias"][h]) for t in tokens]
    bes = [orc.beta(inp["b"][t, h]) for t in tokens]
    vs = [inp["v"][t, h] for t in tokens]
    Ss = _unrolled(S0, kh, vs, als, bes)
    return Ss, [S @ q for S, q in zip(Ss, qh)]


@pytest.mark.parametrize("hk,hv", [(1, 1), (1, 2)])
def test_prefill_twin_matches_unrolled_product(orc, hk, hv):
    """Four sequences: 5 tokens, padding (3 tokens), empty, 2 tokens; twin."""
    rng = np.random.default_rng(60 + hv)
    dk, dv = 4, 3
    cu = np.array([0, 5, 8, 8, 10], np.int32)
    T = int(cu[-1])
    inp = _inputs(rng, T, hk, hv, dk, dv)
    pool = rng.standard_normal((9, hv, dv, dk)) * 0.1
    pool[0] = 0.0
    start = pool.copy()
    rs = np.array([3, 0, 5, 1], np.int32)
    ws = np.array([7, 0, 2, 8], np.int32)
    out, bad = orc.prefill(cu, pool=pool, read_slot=rs, write_slot=ws, **inp)
    assert bad == 0
    group = hv // hk
    for r in range(4):
        toks = list(range(cu[r], cu[r + 1]))
        for h in range(hv):
            if rs[r] == 0:
                assert np.all(out[toks, h] == 0.0)
                continue
            if not toks:  # no tokens: the state moves to the write slot unchanged
                assert np.array_equal(pool[ws[r], h], start[rs[r], h])
                continue
            Ss, os = _closed_form(orc, inp, start[rs[r], h], toks, h, group)
            for i, t in enumerate(toks):
                assert np.allclose(out[t, h], os[i], atol=1e-12, rtol=0)
            assert np.allclose(pool[ws[r], h], Ss[-1], atol=1e-12, rtol=0)
            assert np.array_equal(pool[rs[r], h], start[rs[r], h])  # twin: read slot untouched
    untouched = [s for s in range(9) if s not in ws[rs > 0]]
    assert np.array_equal(pool[untouched], start[untouched])


def test_prefill_in_place_equals_decode_steps(orc):
    """A prefill in place equals the pinned one-token step called token by
    token (sequences of unequal length in a shuffled slot order)."""
    rng = np.random.default_rng(61)
    hk, hv, dk, dv = 2, 4, 8, 8
    lens = [4, 1, 6, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    inp = _inputs(rng, T, hk, hv, dk, dv)
    pool = rng.standard_normal((7, hv, dv, dk)) * 0.1
    pool[0] = 0.0
    ref = pool.copy()
    rs = np.array([6, 2, 1, 4], np.int32)
    out, bad = orc.prefill(cu, pool=pool, read_slot=rs, **inp)
    assert bad == 0
    for r, n in enumerate(lens):
        for i in range(n):
            t = cu[r] + i
            o, _ = orc.step(inp["q"][t:t + 1], inp["k"][t:t + 1], inp["v"][t:t + 1], inp["a"][t:t + 1],
                            inp["b"][t:t + 1], inp["A_log"], inp["dt_bias"], ref, rs[r:r + 1], None,
                            keep_in_place=True)
            assert np.array_equal(out[t], o[0])
    assert np.array_equal(pool, ref)


def test_verify_keeps_a_state_a_token(orc):
    """With token slots the state after token t lands in token_slot[t]; the
    read slot and the write slot stay as they were."""
    rng = np.random.default_rng(62)
    hk, hv, dk, dv = 1, 2, 4, 4
    cu = np.array([0, 3, 5], np.int32)
    T = 5
    inp = _inputs(rng, T, hk, hv, dk, dv)
    pool = rng.standard_normal((12, hv, dv, dk)) * 0.1
    pool[0] = 0.0
    start = pool.copy()
    rs = np.array([2, 9], np.int32)
    ts = np.array([4, 5, 6, 10, 11], np.int32)
    out, bad = orc.prefill(cu, pool=pool, read_slot=rs, write_slot=np.array([1, 3], np.int32),
                           token_slot=ts, **inp)
    assert bad == 0
    for r in range(2):
        toks = list(range(cu[r], cu[r + 1]))
        for h in range(hv):
            Ss, os = _closed_form(orc, inp, start[rs[r], h], toks, h, hv // hk)
            for i, t in enumerate(toks):
                assert np.allclose(pool[ts[t], h], Ss[i], atol=1e-12, rtol=0)
                assert np.allclose(out[t, h], os[i], atol=1e-12, rtol=0)
    for s in (1, 2, 3, 7, 8, 9):
        assert np.array_equal(pool[s], start[s])


def test_prefill_bad_slots(orc):
    rng = np.random.default_rng(63)
    hk, hv, dk, dv = 1, 1, 4, 4
    cu = np.array([0, 2, 4, 6], np.int32)
    inp = _inputs(rng, 6, hk, hv, dk, dv)
    pool = rng.standard_normal((6, hv, dv, dk))
    start = pool.copy()
    # twin: write slot equal to the read slot, write slot 0, read slot out of range
    out, bad = orc.prefill(cu, pool=pool, read_slot=np.array([1, 2, 9], np.int32),
                           write_slot=np.array([1, 0, 3], np.int32), **inp)
    assert bad == 3 and np.all(out == 0.0) and np.array_equal(pool, start)
    # verify: one token slot equal to the read slot spoils its whole sequence
    out, bad = orc.prefill(cu, pool=pool, read_slot=np.array([1, 2, 3], np.int32),
                           token_slot=np.array([4, 5, 2, 5, 4, 5], np.int32), **inp)
    assert bad == 1 and np.all(out[2:4] == 0.0) and np.any(out[:2] != 0.0)
    assert np.array_equal(pool[2], start[2])


def test_conv_prefill_equals_numpy_convolve(orc):
    """The conv over a sequence continues the window: the causal part of
    numpy's convolution of [window; tokens], the last W-1 inputs as the new
    window, and in verify mode the window after each token."""
    rng = np.random.default_rng(64)
    C, W = 5, 4
    lens = [6, 2, 0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    pool = rng.standard_normal((8, W - 1, C))
    start = pool.copy()
    rs = np.array([1, 4, 6], np.int32)
    ws = np.array([2, 5, 7], np.int32)
    y, bad = orc.conv_prefill(cu, x, pool, rs, ws, w, None, silu=False)
    assert bad == 0
    for r, n in enumerate(lens):
        seq = np.concatenate([start[rs[r]], x[cu[r]:cu[r + 1]]])  # oldest first
        for c in range(C):
            full = np.convolve(seq[:, c], w[c, ::-1])
            assert np.allclose(y[cu[r]:cu[r + 1], c], full[W - 1:W - 1 + n], atol=1e-13, rtol=0)
        assert np.array_equal(pool[ws[r]], seq[-(W - 1):])
        assert np.array_equal(pool[rs[r]], start[rs[r]])
    # verify mode: the window after each token, in six distinct token slots
    pool = start.copy()
    ts = np.array([2, 3, 4, 5, 6, 7], np.int32)
    cu1 = np.array([0, 6], np.int32)
    y1, bad = orc.conv_prefill(cu1, x[:6], pool, rs[:1], None, w, None, token_slot=ts, silu=False)
    assert bad == 0
    assert np.array_equal(y1, y[:6])
    seq = np.concatenate([start[rs[0]], x[:6]])
    for t in range(6):
        assert np.array_equal(pool[ts[t]], seq[t + 1:t + W])
    assert np.array_equal(pool[rs[0]], start[rs[0]])


def test_copy_slots_snapshot_and_fork(orc):
    """Snapshots and forks: a copied slot holds exactly the source's values,
    a copy there and back is the identity, copying the null slot zeroes the
    destination, slots outside the copies are untouched, bad pairs are
    skipped and counted."""
    rng = np.random.default_rng(65)
    pool = rng.standard_normal((9, 2, 3, 4))
    pool[0] = 0.0
    start = pool.copy()
    bad = orc.copy_slots(pool, [2, 5, 0], [7, 1, 8])
    assert bad == 0
    assert np.array_equal(pool[7], start[2]) and np.array_equal(pool[1], start[5])
    assert np.all(pool[8] == 0.0)
    for s in (0, 2, 3, 4, 5, 6):
        assert np.array_equal(pool[s], start[s])
    orc.copy_slots(pool, [7], [3])
    orc.copy_slots(pool, [3], [4])
    assert np.array_equal(pool[4], start[2])
    before = pool.copy()
    assert orc.copy_slots(pool, [1, 9, -1, 2], [0, 2, 3, 9]) == 4
    assert np.array_equal(pool, before)
