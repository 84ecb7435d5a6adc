"""GPU parity of causal_conv1d_decode against the fp64 oracle, through the C ABI.

The decode conv is the conv state update for one token a row, with null
slots, strided rows, optional bias and activation, and a write slot that
leaves the read slot alone (mstar PR #1139, "What changed" and "Tests").
Windows are bit-exact; outputs are bit-exact after rounding, up to a
rounding-midpoint tie (see gpu_helpers).
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import check_conv_outputs, conv_magnitude, f64, pair, ti

pytestmark = pytest.mark.gpu


class ConvCase:
    def __init__(self, gdn, s: I.Shape, seed: int, num_slots: int, pad_frac=0.0):
        self.gdn, self.s = gdn, s
        self.gen = I.Gen(seed)
        prm = self.gen.params(s)
        self.w, self.w64 = pair(prm["w"], s.dtype)
        self.bias, self.bias64 = pair(prm["bias"], s.dtype)
        cp_dev, self.cp64 = pair(self.gen.conv_pool(s, num_slots), s.dtype)
        self.cp = gdn.ConvStatePool(num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda",
                                    tensor=cp_dev.contiguous())
        self.rs_np, self.ws_np = self.gen.slot_tables(s.rows, num_slots, pad_frac)
        self.rs, self.ws = ti(self.rs_np), ti(self.ws_np)

    def draw_x(self):
        return pair(self.gen.normal((self.s.rows, self.s.channels)), self.s.dtype)

    def pool(self):
        return f64(self.cp.tensor)


def run_and_check(orc, c: ConvCase, x, x64, twin=True, bias=True, silu=True):
    before = c.cp64.copy()
    out = c.gdn.causal_conv1d_decode(x, c.cp, c.rs, c.w, c.bias if bias else None,
                                     write_slot=c.ws if twin else None, silu=silu)
    torch.cuda.synchronize()
    ref_pool = before.copy()
    y, bad = orc.conv_step(x64, ref_pool, c.rs_np, c.ws_np if twin else None, c.w64,
                           c.bias64 if bias else None, silu=silu)
    assert bad == 0
    real = c.rs_np != 0
    mag = conv_magnitude(before[c.rs_np], x64, c.w64, c.bias64 if bias else None)
    flips = check_conv_outputs(orc, f64(out)[real], y[real], mag[real], c.s.dtype)
    assert not f64(out)[~real].any()
    assert np.array_equal(c.pool(), ref_pool)       # windows bit-exact, others untouched
    c.cp64 = ref_pool
    return out, flips


@pytest.mark.parametrize("shape", [I.TINY, I.QWEN_08B, I.QWEN_9B], ids=["tiny", "0.8b", "9b"])
@pytest.mark.parametrize("twin", [True, False], ids=["twin", "in_place"])
def test_conv_matches_oracle(gdn, orc, shape, twin):
    c = ConvCase(gdn, shape, seed=20, num_slots=2 * shape.rows + 1, pad_frac=0.25)
    x, x64 = c.draw_x()
    _, flips = run_and_check(orc, c, x, x64, twin=twin)
    assert flips.mean() < 1e-3
    assert gdn.get_device_error() == 0


def test_conv_twin_equals_in_place_and_leaves_read_slot(gdn):
    s = I.QWEN_08B
    c = ConvCase(gdn, s, seed=21, num_slots=s.num_slots)
    x, _ = c.draw_x()
    start = c.cp.tensor.clone()
    o_t = gdn.causal_conv1d_decode(x, c.cp, c.rs, c.w, c.bias, write_slot=c.ws).clone()
    after_t = c.cp.tensor.clone()
    c.cp.tensor.copy_(start)
    o_i = gdn.causal_conv1d_decode(x, c.cp, c.rs, c.w, c.bias).clone()
    after_i = c.cp.tensor.clone()
    assert torch.equal(o_t, o_i)
    rs, ws = torch.from_numpy(c.rs_np).long().cuda(), torch.from_numpy(c.ws_np).long().cuda()
    assert torch.equal(after_t[ws], after_i[rs])
    assert torch.equal(after_t[rs], start[rs])             # the read slot is left alone


def test_conv_strided_rows_no_bias_no_activation(gdn, orc):
    s = I.QWEN_08B.with_(rows=9)
    c = ConvCase(gdn, s, seed=22, num_slots=19, pad_frac=0.3)
    wide_np = c.gen.normal((s.rows, s.channels + 64))
    wide, wide64 = pair(wide_np, s.dtype)
    x, x64 = wide[:, :s.channels], wide64[:, :s.channels]
    assert x.stride(0) == s.channels + 64
    run_and_check(orc, c, x, x64, twin=True, bias=False, silu=False)
    # identity taps, no bias, no activation: the output is x itself, bit for bit
    w_id = np.zeros((s.channels, s.width), np.float32)
    w_id[:, -1] = 1.0
    c.w, c.w64 = pair(w_id, s.dtype)
    out = gdn.causal_conv1d_decode(x, c.cp, c.rs, c.w, None, write_slot=c.ws, silu=False)
    real = torch.from_numpy(c.rs_np != 0).cuda()
    assert torch.equal(out[real], x[real])


@pytest.mark.parametrize("width", [2, 3])
def test_conv_other_widths(gdn, orc, width):
    s = I.QWEN_08B.with_(rows=6, width=width)
    c = ConvCase(gdn, s, seed=23 + width, num_slots=13)
    x, x64 = c.draw_x()
    run_and_check(orc, c, x, x64)


def test_conv_chained_twin_steps(gdn, orc):
    """8 chained steps with the commit swapping the slot tables."""
    s = I.TINY
    c = ConvCase(gdn, s, seed=24, num_slots=s.num_slots)
    for _ in range(8):
        x, x64 = c.draw_x()
        run_and_check(orc, c, x, x64)
        gdn.gdn_commit(c.rs, c.ws)
        orc.commit(c.rs_np, c.ws_np)
    torch.cuda.synchronize()
    assert np.array_equal(c.rs.cpu().numpy(), c.rs_np)


def test_conv_bad_slot(gdn):
    s = I.QWEN_08B.with_(rows=3)
    c = ConvCase(gdn, s, seed=25, num_slots=7)
    rs = c.rs_np.copy()
    rs[1] = 99
    c.rs.copy_(ti(rs))
    x, _ = c.draw_x()
    before = c.cp.tensor.clone()
    out = gdn.causal_conv1d_decode(x, c.cp, c.rs, c.w, c.bias, write_slot=c.ws)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == gdn.GDN_DEVERR_BAD_SLOT
    assert not out[1].any() and out[0].any()
    assert torch.equal(c.cp.tensor[c.ws_np[1]], before[c.ws_np[1]])
