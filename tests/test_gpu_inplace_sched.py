"""GPU checks of the fused layer's in-place schedules.

With the state pool's in-place counters an in-place launch spreads a qk
head's items over the CTAs and the item that counts last writes the head's
new q/k conv window; without them each CTA takes whole qk heads.  Both give
the same values, bit for bit, over chained steps, and equal the twin write;
every counter is back at zero after each launch.  Shapes whose kept window
does not fit beside the kernel's ring keep the whole-head schedule even with
counters (dk = 256, width 3, bf16 here).  gdn_pool_zero_slots clears the
listed slots' counters.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import pair, t, ti

pytestmark = pytest.mark.gpu

GROUP4_F32 = I.Shape(rows=4, hk=2, hv=8, dk=64, dv=32, width=3, dtype="f32")
DK256_W3 = I.Shape(rows=4, hk=2, hv=4, dk=256, dv=64, width=3, dtype="bf16")


class Pools:
    """The same seeded layer three times: in place with counters, in place
    without, and twin."""

    def __init__(self, gdn, s: I.Shape, seed: int, pad_frac: float):
        self.gdn, self.s = gdn, s
        self.gen = I.Gen(seed)
        prm = self.gen.params(s)
        self.w, _ = pair(prm["w"], s.dtype)
        self.bias, _ = pair(prm["bias"], s.dtype)
        self.A_log, self.dt_bias = t(prm["A_log"]), t(prm["dt_bias"])
        n = 2 * s.rows + 1
        state = self.gen.state_pool(s, n)
        conv, _ = pair(self.gen.conv_pool(s, n), s.dtype)
        self.state0, self.conv0 = state, conv
        self.sets = {}
        for name, counters in (("fine", True), ("groups", False), ("twin", True)):
            pool = gdn.GDNStatePool(n, s.hk, s.hv, s.dk, s.dv, device="cuda",
                                    tensor=torch.from_numpy(state.copy()).cuda(), inplace_counters=counters)
            cp = gdn.ConvStatePool(n, s.channels, s.width, dtype=conv.dtype, device="cuda", tensor=conv.clone())
            self.sets[name] = (pool, cp)
        rs, ws = self.gen.slot_tables(s.rows, n, pad_frac)
        self.rs_np, self.ws_np = rs, ws
        self.rs, self.ws = ti(rs), ti(ws)

    def draw(self):
        return {k: pair(v, self.s.dtype)[0] for k, v in self.gen.layer_inputs(self.s).items()}

    def run(self, name, xd):
        pool, cp = self.sets[name]
        twin = name == "twin"
        return self.gdn.gdn_layer_decode(xd["x"], cp, self.w, self.bias, self.A_log, self.dt_bias, xd["a"],
                                         xd["b"], pool, self.rs, self.ws if twin else None,
                                         keep_in_place=not twin)


SHAPES = [
    (I.TINY, 1), (I.TINY, 4),
    (I.QWEN_08B, 1), (I.QWEN_08B, 2), (I.QWEN_08B, 5), (I.QWEN_08B, 16), (I.QWEN_08B, 64),
    (I.QWEN_9B, 1), (I.QWEN_9B, 16),
    (GROUP4_F32, 3),
    (DK256_W3, 4),
]


@pytest.mark.parametrize("shape,rows", SHAPES,
                         ids=[f"{'x'.join(map(str, (s.hk, s.hv, s.dk, s.dv, s.width)))}-{s.dtype}-r{r}"
                              for s, r in SHAPES])
def test_in_place_schedules_agree_over_chained_steps(gdn, shape, rows):
    s = shape.with_(rows=rows)
    P = Pools(gdn, s, seed=500 + rows, pad_frac=0.25 if rows >= 4 else 0.0)
    pf, cf = P.sets["fine"]
    pg, cg = P.sets["groups"]
    pt, ct = P.sets["twin"]
    real = torch.from_numpy(P.rs_np != 0).cuda()
    rs_l = torch.from_numpy(P.rs_np).long().cuda()[real]
    ws_l = torch.from_numpy(P.ws_np).long().cuda()[real]
    for step in range(3):
        xd = P.draw()
        o_f = P.run("fine", xd).clone()
        o_g = P.run("groups", xd).clone()
        if step == 0:
            o_t = P.run("twin", xd).clone()
        torch.cuda.synchronize()
        assert torch.equal(o_f, o_g), f"step {step}: outputs"
        assert torch.equal(pf.tensor, pg.tensor), f"step {step}: states"
        assert torch.equal(cf.tensor, cg.tensor), f"step {step}: conv windows"
        assert not pf.counters.any(), f"step {step}: counters left set"
        if step == 0:
            assert torch.equal(o_f, o_t)
            assert torch.equal(pf.tensor[rs_l], pt.tensor[ws_l])
            assert torch.equal(cf.tensor[rs_l], ct.tensor[ws_l])
        # the windows moved: a real row's newest column is this step's x
        x_new = xd["x"][real]
        assert torch.equal(cf.tensor[rs_l, s.width - 2], x_new)
    assert gdn.get_device_error() == 0


def test_zero_slots_clears_in_place_counters(gdn):
    s = I.QWEN_08B.with_(rows=4)
    pool = gdn.GDNStatePool(9, s.hk, s.hv, s.dk, s.dv, device="cuda")
    stride = pool.counters.numel() // 9
    assert stride == 16
    pool.counters.fill_(7)
    pool.zero_slots(ti(np.array([1, 3], np.int32)))
    torch.cuda.synchronize()
    c = pool.counters.view(9, stride)
    assert not c[1].any() and not c[3].any()
    keep = [i for i in range(9) if i not in (1, 3)]
    assert bool((c[keep] == 7).all())
    pool.counters.zero_()
    assert gdn.get_device_error() == 0
