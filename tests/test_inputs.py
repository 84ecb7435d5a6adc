"""The seeded input recipe (CPU): the same seed gives the same draws, and the
slot tables have the structure the kernels take as a precondition.  Padding
rows sit on the null slot 0 ("mstar PR #1127", "What changed": padding rows
address slot 0, which stays zero).  Real rows never share a slot, and a
twin row's write slot is no row's read slot, so no two rows touch one slot
("mstar PR #1139", "What changed": a request holds two slots)."""
import math

import numpy as np
import pytest

from gated_deltanet_decode_gb300 import inputs as I


def test_same_seed_same_draws():
    a, b = I.Gen(3), I.Gen(3)
    s = I.TINY
    for x, y in zip(a.step_inputs(s).values(), b.step_inputs(s).values()):
        assert np.array_equal(x, y)
    assert np.array_equal(a.state_pool(s), b.state_pool(s))
    assert not np.array_equal(I.Gen(4).state_pool(s), I.Gen(3).state_pool(s))


@pytest.mark.parametrize("rows,pad,twin", [(64, 0.25, True), (256, 0.25, False), (5, 0.0, True), (1, 0.5, True),
                                           (128, 0.1, True)])
def test_slot_tables(rows, pad, twin):
    g = I.Gen(11)
    num_slots = 2 * rows + 1
    rs, ws = g.slot_tables(rows, num_slots, pad_frac=pad, twin=twin)
    assert rs.dtype == np.int32 and ws.dtype == np.int32 and rs.shape == ws.shape == (rows,)
    padding = rs == 0
    assert padding.sum() == math.floor(pad * rows)
    assert np.all(ws[padding] == 0)                       # padding: both slots null
    real_r, real_w = rs[~padding], ws[~padding]
    assert np.all((real_r >= 1) & (real_r < num_slots)) and np.all((real_w >= 1) & (real_w < num_slots))
    assert len(set(real_r.tolist())) == len(real_r)       # no two rows read one slot
    assert len(set(real_w.tolist())) == len(real_w)       # nor write one
    if twin:
        assert not set(real_r.tolist()) & set(real_w.tolist())   # no write slot is a read slot
    else:
        assert np.array_equal(real_r, real_w)


def test_slot_tables_refuse_a_pool_too_small():
    with pytest.raises(ValueError):
        I.Gen(0).slot_tables(8, 16, twin=True)            # 16 slots needed, 15 usable


def test_seq_tables():
    g = I.Gen(12)
    lens = [6, 1, 0, 9, 4]
    cu, rs, ws, ts = g.seq_tables(lens, num_slots=64, n_pad=1)
    assert cu.tolist() == [0, 6, 7, 7, 16, 20]
    pad = rs == 0
    assert pad.sum() == 1 and np.all(ws[pad] == 0)
    used = []
    for r in range(len(lens)):
        tok = ts[cu[r]:cu[r + 1]]
        if pad[r]:
            assert np.all(tok == 0)
        else:
            used += [int(rs[r]), int(ws[r])] + tok.tolist()
    assert all(1 <= u < 64 for u in used) and len(set(used)) == len(used)   # every real slot distinct
    cu2, rs2, ws2, ts2 = I.Gen(12).seq_tables(lens, num_slots=64, n_pad=0, token_slots=False)
    assert not ts2.any() and np.all(rs2 > 0) and np.all(ws2 > 0)    # no padding, no token slots


def test_parameter_ranges_and_state_scale():
    g = I.Gen(5)
    s = I.QWEN_08B
    p = g.params(s)
    assert p["A_log"].shape == (s.hv,) and np.all((p["A_log"] >= 0) & (p["A_log"] < math.log(16.0)))
    assert np.all((p["dt_bias"] >= -1.0) & (p["dt_bias"] < 1.0))
    assert p["w"].shape == (s.channels, s.width) and p["bias"].shape == (s.channels,)
    pool = g.state_pool(I.TINY)
    assert not pool[0].any()                              # the null slot is zero
    assert abs(float(pool[1:].std()) - 0.1) < 0.01        # N(0, 0.1) elsewhere
    conv = g.conv_pool(I.TINY)
    assert not conv[0].any() and conv.shape == (I.TINY.num_slots, I.TINY.width - 1, I.TINY.channels)
