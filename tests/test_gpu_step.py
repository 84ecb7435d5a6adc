"""GPU parity of gdn_decode_step against the fp64 oracle, through the C ABI.

Workloads: the tiny check (4 rows, 2/2 heads, dk = dv = 16, fp32, 8 chained
twin steps), the 0.8B-shaped layer (64 rows, 16/16 heads, 128 x 128, bf16,
one step over every head and 256 chained steps on sampled heads), the
row-count / write-mode sweep (1..256 rows, twin and in place, 25% padding on
the null slot, 513 slots) and the 9B-shaped GQA layer (16 qk / 32 v heads).
Slot semantics follow the mstar PR #1139 page ("What changed": twin slots,
commit swap, in place; "Tests": a twin step touches no other slot) and the PR
#965 page (padding rows change no real row's result).

The oracle consumes only the generator's values and its own slot tables
(committed with the oracle's commit); GPU results are only ever compared.
"""
import math

import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import (STATE_TOL_CHAIN, STATE_TOL_ONE, assert_out_close, f64, pair,
                         state_rel_err, t, ti)

pytestmark = pytest.mark.gpu


class Case:
    """One layer's pool, parameters and slot tables: on the GPU, and as the
    exact values the oracle reads."""

    def __init__(self, gdn, shape: I.Shape, seed: int, num_slots: int, pad_frac=0.0):
        self.gdn, self.s = gdn, shape
        self.gen = I.Gen(seed)
        self.prm = self.gen.params(shape)
        self.pool_np = self.gen.state_pool(shape, num_slots)          # exact initial pool
        self.pool = gdn.GDNStatePool(num_slots, shape.hk, shape.hv, shape.dk, shape.dv, device="cuda",
                                     tensor=torch.from_numpy(self.pool_np.copy()).cuda())
        self.A_log = t(self.prm["A_log"])
        self.dt_bias = t(self.prm["dt_bias"])
        self.rs_np, self.ws_np = self.gen.slot_tables(shape.rows, num_slots, pad_frac)
        self.rs, self.ws = ti(self.rs_np), ti(self.ws_np)

    def draw(self):
        """(device inputs, exact inputs) for one step."""
        dev, ref = {}, {}
        for k, v in self.gen.step_inputs(self.s).items():
            dev[k], ref[k] = pair(v, self.s.dtype)
        return dev, ref

    def run(self, x, keep_in_place=False, out=None):
        return self.gdn.gdn_decode_step(x["q"], x["k"], x["v"], x["a"], x["b"], self.A_log, self.dt_bias,
                                        self.pool, self.rs, None if keep_in_place else self.ws, out=out,
                                        keep_in_place=keep_in_place)

    def snapshot(self):
        return self.pool.tensor.detach().cpu().numpy().copy()

    def oracle_head(self, orc, S, xr, r, h):
        g = h // (self.s.hv // self.s.hk)
        return orc.head(S, xr["q"][r, g], xr["k"][r, g], xr["v"][r, h], xr["a"][r, h], xr["b"][r, h],
                        self.prm["A_log"][h], self.prm["dt_bias"][h])


def check_one_step(orc, case: Case, keep_in_place=False):
    """One step from the generator's pool: every real head against the oracle,
    untouched slots bit-identical, padding outputs zero."""
    xd, xr = case.draw()
    out = case.run(xd, keep_in_place)
    torch.cuda.synchronize()
    after = case.snapshot()
    p_ref = case.pool_np.astype(np.float64)
    o_ref, bad = orc.step(xr["q"], xr["k"], xr["v"], xr["a"], xr["b"], case.prm["A_log"],
                          case.prm["dt_bias"], p_ref, case.rs_np, case.ws_np,
                          keep_in_place=keep_in_place)
    assert bad == 0
    assert_out_close(f64(out), o_ref, case.s.dtype)
    rs = case.rs_np
    ws = rs if keep_in_place else case.ws_np
    real = rs != 0
    err = state_rel_err(after[ws[real]], p_ref[ws[real]])
    assert err.max() <= STATE_TOL_ONE, f"state rel err {err.max():.3g}"
    untouched = np.setdiff1d(np.arange(after.shape[0]), ws[real])
    assert np.array_equal(after[untouched], case.pool_np[untouched])
    assert not after[0].any()
    assert not f64(out)[~real].any()
    return out, after


# ---------------------------------------------------------------------------

def test_tiny_chained_twin(gdn, orc):
    s = I.TINY
    case = Case(gdn, s, seed=0, num_slots=s.num_slots)
    ref_pool = case.pool_np.astype(np.float64)
    rs, ws = case.rs_np.copy(), case.ws_np.copy()
    for step in range(8):
        xd, xr = case.draw()
        out = case.run(xd)
        o_ref, bad = orc.step(xr["q"], xr["k"], xr["v"], xr["a"], xr["b"], case.prm["A_log"],
                              case.prm["dt_bias"], ref_pool, rs, ws)
        assert bad == 0
        assert_out_close(f64(out), o_ref, "f32", f"step {step} out")
        gdn.gdn_commit(case.rs, case.ws)
        orc.commit(rs, ws)
    torch.cuda.synchronize()
    assert np.array_equal(case.rs.cpu().numpy(), rs) and np.array_equal(case.ws.cpu().numpy(), ws)
    err = state_rel_err(case.snapshot()[rs], ref_pool[rs])
    assert err.max() <= STATE_TOL_ONE * 8, f"state rel err {err.max():.3g} after 8 steps"
    assert gdn.get_device_error() == 0


def test_qwen08b_one_step_every_head(gdn, orc):
    s = I.QWEN_08B
    check_one_step(orc, Case(gdn, s, seed=1, num_slots=s.num_slots))
    assert gdn.get_device_error() == 0


def test_qwen08b_in_place_one_step(gdn, orc):
    s = I.QWEN_08B
    check_one_step(orc, Case(gdn, s, seed=2, num_slots=s.num_slots), keep_in_place=True)
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_qwen08b_256_chained_steps(gdn, orc):
    """256 twin steps with a commit after each; sampled (row, head) pairs are
    followed by the oracle in fp64 the whole way."""
    s = I.QWEN_08B
    case = Case(gdn, s, seed=3, num_slots=s.num_slots)
    samples = [(0, 0), (0, 15), (63, 0), (63, 15), (17, 5), (40, 9), (31, 7), (5, 12)]
    rs, ws = case.rs_np.copy(), case.ws_np.copy()
    S = {(r, h): case.pool_np[rs[r], h].astype(np.float64) for r, h in samples}
    for step in range(256):
        xd, xr = case.draw()
        out = case.run(xd)
        o = f64(out) if (step % 32 == 0 or step == 255) else None
        for (r, h) in samples:
            S[(r, h)], o_ref = case.oracle_head(orc, S[(r, h)], xr, r, h)
            if o is not None:
                assert_out_close(o[r, h], o_ref, "bf16", f"step {step} out ({r},{h})")
        gdn.gdn_commit(case.rs, case.ws)
        orc.commit(rs, ws)
    torch.cuda.synchronize()
    assert np.array_equal(case.rs.cpu().numpy(), rs)
    final = case.snapshot()
    for (r, h) in samples:
        err = state_rel_err(final[rs[r], h], S[(r, h)])
        assert err <= STATE_TOL_CHAIN, f"({r},{h}) state rel err {err:.3g} after 256 steps"
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("rows", I.SWEEP_ROWS)
def test_sweep_rows_twin_vs_in_place(gdn, orc, rows):
    """Row-count / write-mode sweep: 25% padding rows on the null slot, random
    slot permutation of a 513-slot pool; twin and in place give bit-identical
    values, every slot outside the write set is untouched, sampled heads match
    the oracle."""
    s = I.QWEN_08B.with_(rows=rows)
    case = Case(gdn, s, seed=100 + rows, num_slots=I.SWEEP_SLOTS, pad_frac=0.25)
    before = case.pool_np
    xd, xr = case.draw()
    out_t = case.run(xd).clone()
    torch.cuda.synchronize()
    after_t = case.snapshot()
    case.pool.tensor.copy_(torch.from_numpy(before).cuda())
    out_i = case.run(xd, keep_in_place=True).clone()
    torch.cuda.synchronize()
    after_i = case.snapshot()
    rs, ws = case.rs_np, case.ws_np
    real = rs != 0
    assert torch.equal(out_t, out_i)
    assert np.array_equal(after_t[ws[real]], after_i[rs[real]])
    for after, wset in ((after_t, ws[real]), (after_i, rs[real])):
        untouched = np.setdiff1d(np.arange(before.shape[0]), wset)
        assert np.array_equal(after[untouched], before[untouched])
    assert not f64(out_t)[~real].any()
    rng = np.random.default_rng(rows)
    real_rows = np.nonzero(real)[0]
    o = f64(out_t)
    for r in rng.choice(real_rows, size=min(6, len(real_rows)), replace=False):
        for h in (0, s.hv - 1):
            S1, o_ref = case.oracle_head(orc, before[rs[r], h], xr, r, h)
            assert state_rel_err(after_t[ws[r], h], S1) <= STATE_TOL_ONE
            assert_out_close(o[r, h], o_ref, "bf16")
    assert gdn.get_device_error() == 0


def test_rows_independent_of_batch_and_padding(gdn):
    """A real row's output and next state do not depend on which other rows,
    or how many padding rows, share the launch (bit-exact)."""
    s = I.QWEN_08B
    case = Case(gdn, s, seed=7, num_slots=s.num_slots)
    xd, _ = case.draw()
    out_full = case.run(xd).clone()
    torch.cuda.synchronize()
    after_full = case.snapshot()
    pick = np.random.default_rng(0).choice(s.rows, size=10, replace=False)
    rows2 = 24
    pos = np.random.default_rng(1).choice(rows2, size=10, replace=False)
    rs2 = np.zeros(rows2, np.int32)
    ws2 = np.zeros(rows2, np.int32)
    rs2[pos], ws2[pos] = case.rs_np[pick], case.ws_np[pick]
    pos_t, pick_t = torch.from_numpy(pos).cuda(), torch.from_numpy(pick).cuda()
    x2 = {}
    for k, v in xd.items():
        z = torch.zeros((rows2,) + tuple(v.shape[1:]), dtype=v.dtype, device=v.device)
        z[pos_t] = v[pick_t]
        x2[k] = z
    case.pool.tensor.copy_(torch.from_numpy(case.pool_np).cuda())
    out2 = gdn.gdn_decode_step(x2["q"], x2["k"], x2["v"], x2["a"], x2["b"], case.A_log, case.dt_bias,
                               case.pool, ti(rs2), ti(ws2))
    torch.cuda.synchronize()
    after2 = case.snapshot()
    assert torch.equal(out2[pos_t], out_full[pick_t])
    assert np.array_equal(after2[case.ws_np[pick]], after_full[case.ws_np[pick]])


def test_graph_replay_equals_eager(gdn):
    """A captured step + commit, replayed, gives bit-identical results to eager calls."""
    s = I.QWEN_08B.with_(rows=16)
    case = Case(gdn, s, seed=8, num_slots=33)
    xd, _ = case.draw()
    out = torch.empty((s.rows, s.hv, s.dv), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        case.run(xd, out=out)
        gdn.gdn_commit(case.rs, case.ws)
    torch.cuda.synchronize()
    eager_pool, eager_out = case.snapshot(), out.clone()
    case.pool.tensor.copy_(torch.from_numpy(case.pool_np).cuda())
    case.rs.copy_(ti(case.rs_np))
    case.ws.copy_(ti(case.ws_np))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            case.run(xd, out=out)
            gdn.gdn_commit(case.rs, case.ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert np.array_equal(case.snapshot(), case.pool_np)      # capture ran nothing
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(case.snapshot(), eager_pool)
    assert torch.equal(out, eager_out)


def test_gates_special_cases(gdn, orc):
    """beta = 0 with alpha = 1 leaves the state bit-identical; alpha = 0 and
    beta = 1 match the oracle."""
    s = I.QWEN_08B.with_(rows=4)
    case = Case(gdn, s, seed=9, num_slots=9)
    before = case.pool_np
    xd, xr = case.draw()
    rs, ws = case.rs_np, case.ws_np
    # beta = 0 (b = -inf), alpha = 1 (A_log = -inf)
    case.A_log.fill_(-math.inf)
    case.run(dict(xd, b=torch.full_like(xd["b"], -math.inf)))
    torch.cuda.synchronize()
    assert np.array_equal(case.snapshot()[ws], before[rs])
    case.A_log.copy_(t(case.prm["A_log"]))
    # alpha = 0 (a = +inf with a finite A_log), then beta = 1 (b = +inf)
    for key in ("a", "b"):
        case.pool.tensor.copy_(torch.from_numpy(before).cuda())
        xd2 = dict(xd, **{key: torch.full_like(xd[key], math.inf)})
        xr2 = dict(xr, **{key: np.full_like(xr[key], math.inf)})
        out = case.run(xd2)
        torch.cuda.synchronize()
        after = case.snapshot()
        for r in range(s.rows):
            for h in (0, 7, 15):
                S1, o_ref = case.oracle_head(orc, before[rs[r], h], xr2, r, h)
                assert state_rel_err(after[ws[r], h], S1) <= STATE_TOL_ONE
                assert_out_close(f64(out)[r, h], o_ref, "bf16")


def test_bad_slots_set_the_device_error(gdn):
    s = I.QWEN_08B.with_(rows=4)
    case = Case(gdn, s, seed=10, num_slots=9)
    assert gdn.get_device_error() == 0
    rs, ws = case.rs_np.copy(), case.ws_np.copy()
    rs[1] = 9            # one past the pool
    ws[2] = rs[2]        # twin write onto its own read slot
    case.rs.copy_(ti(rs))
    case.ws.copy_(ti(ws))
    xd, _ = case.draw()
    out = case.run(xd)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == gdn.GDN_DEVERR_BAD_SLOT
    assert gdn.get_device_error() == 0                    # reading clears it
    after = case.snapshot()
    o = f64(out)
    assert not o[1].any() and not o[2].any()
    assert o[0].any() and o[3].any()
    untouched = np.setdiff1d(np.arange(9), [ws[0], ws[3]])
    assert np.array_equal(after[untouched], case.pool_np[untouched])


def test_zero_rows_and_all_padding(gdn):
    s = I.QWEN_08B.with_(rows=3)
    case = Case(gdn, s, seed=11, num_slots=9)
    xd, _ = case.draw()
    empty = {k: v[:0] for k, v in xd.items()}
    out = gdn.gdn_decode_step(empty["q"], empty["k"], empty["v"], empty["a"], empty["b"], case.A_log,
                              case.dt_bias, case.pool, case.rs[:0], case.ws[:0])
    assert out.shape[0] == 0
    zeros = torch.zeros(3, dtype=torch.int32, device="cuda")
    out = gdn.gdn_decode_step(xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], case.A_log, case.dt_bias,
                              case.pool, zeros, zeros)
    torch.cuda.synchronize()
    assert not f64(out).any()
    assert np.array_equal(case.snapshot(), case.pool_np)
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("rows", [64, 256])
def test_qwen9b_gqa_one_step(gdn, orc, rows):
    """16 qk heads shared by 32 value heads (consecutive pairs), 2R+1 slots."""
    s = I.QWEN_9B.with_(rows=rows)
    case = Case(gdn, s, seed=12 + rows, num_slots=2 * rows + 1)
    if rows == 64:
        check_one_step(orc, case)
    else:
        xd, xr = case.draw()
        out = case.run(xd)
        torch.cuda.synchronize()
        after = case.snapshot()
        rs, ws = case.rs_np, case.ws_np
        for r, h in [(0, 0), (0, 1), (128, 30), (255, 31), (77, 16), (200, 3)]:
            S1, o_ref = case.oracle_head(orc, case.pool_np[rs[r], h], xr, r, h)
            assert state_rel_err(after[ws[r], h], S1) <= STATE_TOL_ONE
            assert_out_close(f64(out)[r, h], o_ref, "bf16")
        untouched = np.setdiff1d(np.arange(after.shape[0]), ws)
        assert np.array_equal(after[untouched], case.pool_np[untouched])
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_qwen9b_128_chained_steps(gdn, orc):
    s = I.QWEN_9B
    case = Case(gdn, s, seed=13, num_slots=2 * s.rows + 1)
    samples = [(0, 0), (0, 1), (63, 31), (30, 14), (30, 15), (12, 22)]
    rs, ws = case.rs_np.copy(), case.ws_np.copy()
    S = {(r, h): case.pool_np[rs[r], h].astype(np.float64) for r, h in samples}
    for step in range(128):
        xd, xr = case.draw()
        case.run(xd)
        for (r, h) in samples:
            S[(r, h)], _ = case.oracle_head(orc, S[(r, h)], xr, r, h)
        gdn.gdn_commit(case.rs, case.ws)
        orc.commit(rs, ws)
    torch.cuda.synchronize()
    final = case.snapshot()
    for (r, h) in samples:
        assert state_rel_err(final[rs[r], h], S[(r, h)]) <= STATE_TOL_CHAIN
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 32), (256, 128), (128, 256), (16, 8)])
def test_other_head_sizes(gdn, orc, dk, dv):
    """Head sizes beyond the workloads: every supported dk, ragged dv chunks."""
    s = I.Shape(rows=5, hk=2, hv=4, dk=dk, dv=dv, dtype="bf16", num_slots=11)
    check_one_step(orc, Case(gdn, s, seed=dk + dv, num_slots=11, pad_frac=0.2))
    assert gdn.get_device_error() == 0
