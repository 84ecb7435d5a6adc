"""GPU checks of the many-tokens-a-sequence calls (gdn_prefill, gdn_verify,
causal_conv1d_prefill).

1. Each token's output and every state equal, bit for bit, the same tokens
   fed one gdn_decode_step (or causal_conv1d_decode) at a time: in place,
   twin (final state in the write slot, read slot untouched), and verify
   (the state after token t in token_slot[t]).
2. They match the fp64 oracle's prefill: outputs within the output
   tolerance, states within the chained-state tolerance, conv windows
   bit-exact, conv outputs as in the decode conv check.
3. Padding sequences and empty sequences touch nothing; bad slots and bad
   token ranges skip the sequence and set the device error word.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import (STATE_TOL_CHAIN, assert_out_close, check_conv_outputs, f64, pair,
                         state_rel_err, t, ti)

pytestmark = pytest.mark.gpu


class Case:
    """Packed sequences with their inputs, a state pool and a conv pool."""

    def __init__(self, gdn, s: I.Shape, lens, seed: int, n_pad: int = 1, token_slots: bool = True):
        self.gdn, self.s, self.lens = gdn, s, list(lens)
        gen = I.Gen(seed)
        T = int(sum(lens))
        self.T = T
        self.num_slots = 1 + 2 * len(lens) + (T if token_slots else 0)
        prm = gen.params(s)
        self.prm = prm
        self.w, self.w64 = pair(prm["w"], s.dtype)
        self.bias, self.bias64 = pair(prm["bias"], s.dtype)
        self.A_log, self.dt_bias = t(prm["A_log"]), t(prm["dt_bias"])
        self.cu_np, self.rs_np, self.ws_np, self.ts_np = gen.seq_tables(lens, self.num_slots, n_pad,
                                                                        token_slots=token_slots)
        self.cu, self.rs, self.ws, self.ts = ti(self.cu_np), ti(self.rs_np), ti(self.ws_np), ti(self.ts_np)
        self.pool_np = gen.state_pool(s, self.num_slots)
        cp_dev, self.cp64 = pair(gen.conv_pool(s, self.num_slots), s.dtype)
        self.cp_start = cp_dev.clone()
        self.pool = gdn.GDNStatePool(self.num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                                     tensor=torch.from_numpy(self.pool_np.copy()).cuda())
        self.cp = gdn.ConvStatePool(self.num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda",
                                    tensor=cp_dev)
        self.dev, self.ref = {}, {}
        for k, v in gen.step_inputs(s.with_(rows=T)).items():
            self.dev[k], self.ref[k] = pair(v, s.dtype)
        self.x, self.x64 = pair(gen.layer_inputs(s.with_(rows=T))["x"], s.dtype)

    def reset(self):
        self.pool.tensor.copy_(torch.from_numpy(self.pool_np).cuda())
        self.cp.tensor.copy_(self.cp_start)

    def step_rows(self, i):
        """Token i of every sequence as one decode step: (token index per row,
        read slots with 0 for sequences that have no token i)."""
        idx = np.zeros(len(self.lens), dtype=np.int64)
        rs = np.zeros(len(self.lens), dtype=np.int32)
        for r, n in enumerate(self.lens):
            if i < n and self.rs_np[r] != 0:
                idx[r] = self.cu_np[r] + i
                rs[r] = self.rs_np[r]
        return idx, rs

    def decode_reference(self, snapshots=False):
        """Outputs [T] and final pool from token-by-token decode steps in place
        (optionally the pool after each step)."""
        g, s = self.gdn, self.s
        out = torch.zeros((self.T, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device="cuda")
        snaps = []
        for i in range(max(self.lens, default=0)):
            idx, rs = self.step_rows(i)
            it = torch.from_numpy(idx).cuda()
            o = g.gdn_decode_step(*(self.dev[k][it].contiguous() for k in ("q", "k", "v", "a", "b")),
                                  self.A_log, self.dt_bias, self.pool, ti(rs), None, keep_in_place=True)
            real = torch.from_numpy(rs != 0).cuda()
            out[it[real]] = o[real]
            if snapshots:
                snaps.append(self.pool.tensor.clone())
        torch.cuda.synchronize()
        return out, self.pool.tensor.clone(), snaps

    def prefill(self, keep_in_place=False):
        return self.gdn.gdn_prefill(self.dev["q"], self.dev["k"], self.dev["v"], self.dev["a"], self.dev["b"],
                                    self.A_log, self.dt_bias, self.pool, self.cu, self.rs,
                                    None if keep_in_place else self.ws, keep_in_place=keep_in_place)

    def verify(self):
        return self.gdn.gdn_verify(self.dev["q"], self.dev["k"], self.dev["v"], self.dev["a"], self.dev["b"],
                                   self.A_log, self.dt_bias, self.pool, self.cu, self.rs, self.ts)


SHAPES = [(I.TINY, [8, 3, 0, 5, 2]), (I.QWEN_08B, [6, 1, 0, 9, 4]), (I.QWEN_9B, [5, 0, 7, 2])]
IDS = ["tiny", "0.8b", "9b"]


@pytest.mark.parametrize("shape,lens", SHAPES, ids=IDS)
def test_prefill_equals_decode_steps(gdn, shape, lens):
    c = Case(gdn, shape, lens, seed=70)
    ref_out, ref_pool, _ = c.decode_reference()
    real = c.rs_np != 0
    # in place
    c.reset()
    out = c.prefill(keep_in_place=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(c.pool.tensor, ref_pool)
    # twin: the final state in the write slot, everything else untouched
    c.reset()
    out = c.prefill()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    start = torch.from_numpy(c.pool_np).cuda()
    rs = torch.from_numpy(c.rs_np[real]).long().cuda()
    ws = torch.from_numpy(c.ws_np[real]).long().cuda()
    assert torch.equal(c.pool.tensor[ws], ref_pool[rs])
    others = torch.ones(c.num_slots, dtype=torch.bool, device="cuda")
    others[ws] = False
    assert torch.equal(c.pool.tensor[others], start[others])
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape,lens", SHAPES, ids=IDS)
def test_verify_keeps_the_decode_states(gdn, shape, lens):
    c = Case(gdn, shape, lens, seed=71)
    ref_out, _, snaps = c.decode_reference(snapshots=True)
    c.reset()
    out = c.verify()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    start = torch.from_numpy(c.pool_np).cuda()
    written = torch.zeros(c.num_slots, dtype=torch.bool, device="cuda")
    for r, n in enumerate(lens):
        if c.rs_np[r] == 0:
            continue
        for i in range(n):
            ts = int(c.ts_np[c.cu_np[r] + i])
            assert torch.equal(c.pool.tensor[ts], snaps[i][int(c.rs_np[r])]), f"sequence {r} token {i}"
            written[ts] = True
    assert torch.equal(c.pool.tensor[~written], start[~written])  # read slots included
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape,lens", [(I.TINY, [8, 3, 0, 5, 2]), (I.QWEN_08B, [24, 0, 16])],
                         ids=["tiny", "0.8b"])
@pytest.mark.parametrize("mode", ["twin", "verify"])
def test_prefill_matches_oracle(gdn, orc, shape, lens, mode):
    c = Case(gdn, shape, lens, seed=72)
    out = c.verify() if mode == "verify" else c.prefill()
    torch.cuda.synchronize()
    pool = c.pool_np.astype(np.float64).copy()
    o_ref, bad = orc.prefill(c.cu_np, c.ref["q"], c.ref["k"], c.ref["v"], c.ref["a"], c.ref["b"],
                             c.prm["A_log"], c.prm["dt_bias"], pool, c.rs_np,
                             write_slot=None if mode == "verify" else c.ws_np,
                             token_slot=c.ts_np if mode == "verify" else None)
    assert bad == 0
    assert_out_close(f64(out), o_ref, shape.dtype)
    got = c.pool.tensor.cpu().numpy()
    slots = (c.ts_np[c.ts_np > 0] if mode == "verify" else c.ws_np[c.rs_np > 0])
    for sl in slots:
        for h in range(shape.hv):
            err = state_rel_err(got[sl, h], pool[sl, h])
            assert err <= STATE_TOL_CHAIN, f"slot {sl} head {h}: {err:.3g}"
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape,lens", [(I.TINY, [8, 3, 0, 5, 2]), (I.QWEN_08B, [6, 1, 0, 9, 4])],
                         ids=["tiny", "0.8b"])
def test_conv_prefill_equals_decode_conv_and_oracle(gdn, orc, shape, lens):
    c = Case(gdn, shape, lens, seed=73)
    g = gdn
    C = shape.channels
    # token by token through causal_conv1d_decode, in place
    ref = torch.zeros((c.T, C), dtype=I.torch_dtype(shape.dtype), device="cuda")
    snaps = []
    for i in range(max(lens)):
        idx, rs = c.step_rows(i)
        it = torch.from_numpy(idx).cuda()
        y = g.causal_conv1d_decode(c.x[it].contiguous(), c.cp, ti(rs), c.w, c.bias)
        real = torch.from_numpy(rs != 0).cuda()
        ref[it[real]] = y[real]
        snaps.append(c.cp.tensor.clone())
    ref_cp = c.cp.tensor.clone()
    real = c.rs_np != 0
    # twin
    c.reset()
    y = g.causal_conv1d_prefill(c.x, c.cp, c.cu, c.rs, c.w, c.bias, write_slot=c.ws)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    rs = torch.from_numpy(c.rs_np[real]).long().cuda()
    ws = torch.from_numpy(c.ws_np[real]).long().cuda()
    assert torch.equal(c.cp.tensor[ws], ref_cp[rs])
    assert torch.equal(c.cp.tensor[rs], c.cp_start[rs])
    # the oracle: windows bit-exact, outputs as in the decode conv check
    cp64 = c.cp64.copy()
    y_exact, bad = orc.conv_prefill(c.cu_np, c.x64, cp64, c.rs_np, c.ws_np, c.w64, c.bias64)
    assert bad == 0
    mag, _ = orc.conv_prefill(c.cu_np, np.abs(c.x64), np.abs(c.cp64), c.rs_np, c.ws_np, np.abs(c.w64),
                              np.abs(c.bias64), silu=False)
    check_conv_outputs(orc, f64(y), y_exact, mag, shape.dtype)
    assert np.array_equal(f64(c.cp.tensor), cp64)
    # in place: the same outputs, the new window back in the read slot
    c.reset()
    y = g.causal_conv1d_prefill(c.x, c.cp, c.cu, c.rs, c.w, c.bias)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert torch.equal(c.cp.tensor[rs], ref_cp[rs])
    # verify: the window after each token in its token slot
    c.reset()
    y = g.causal_conv1d_prefill(c.x, c.cp, c.cu, c.rs, c.w, c.bias, token_slot=c.ts)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    for r, n in enumerate(lens):
        if c.rs_np[r] == 0:
            continue
        for i in range(n):
            ts = int(c.ts_np[c.cu_np[r] + i])
            assert torch.equal(c.cp.tensor[ts], snaps[i][int(c.rs_np[r])])
    assert gdn.get_device_error() == 0


def test_prefill_bad_slots_and_ranges(gdn):
    s = I.TINY
    c = Case(gdn, s, [4, 3, 5], seed=74, n_pad=0)
    start = torch.from_numpy(c.pool_np).cuda()
    # a token slot equal to the sequence's read slot spoils that sequence only
    ts = c.ts_np.copy()
    ts[c.cu_np[1]] = c.rs_np[1]
    c.ts = ti(ts)
    out = c.verify()
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    assert not out[c.cu_np[1]:c.cu_np[2]].any()
    assert out[c.cu_np[0]:c.cu_np[1]].any()
    for tok in range(c.cu_np[1], c.cu_np[2]):
        assert torch.equal(c.pool.tensor[int(ts[tok])], start[int(ts[tok])])
    # a token range past total_tokens is bad; the other sequences run
    c.reset()
    cu = c.cu_np.copy()
    cu[3] = c.T + 5
    c.cu = ti(cu)
    out = c.gdn.gdn_prefill(c.dev["q"], c.dev["k"], c.dev["v"], c.dev["a"], c.dev["b"], c.A_log,
                            c.dt_bias, c.pool, c.cu, c.rs, c.ws)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    assert torch.equal(c.pool.tensor[int(c.ws_np[2])], start[int(c.ws_np[2])])
    assert not torch.equal(c.pool.tensor[int(c.ws_np[0])], start[int(c.ws_np[0])])
    # empty and padding sequences: a twin empty sequence moves its state unchanged
    c.reset()
    c2 = Case(gdn, s, [0, 2], seed=75, n_pad=0)
    c2.prefill()
    torch.cuda.synchronize()
    start2 = torch.from_numpy(c2.pool_np).cuda()
    assert torch.equal(c2.pool.tensor[int(c2.ws_np[0])], start2[int(c2.rs_np[0])])
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 32), (256, 128), (16, 8), (128, 256)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_other_head_sizes(gdn, dk, dv, dtype):
    """Every head size the kernels are built for: prefill in place and
    verification equal token-by-token decode steps, bit for bit."""
    s = I.Shape(rows=1, hk=2, hv=4, dk=dk, dv=dv, width=4, dtype=dtype, num_slots=0)
    c = Case(gdn, s, [5, 0, 3, 7], seed=76)
    ref_out, ref_pool, snaps = c.decode_reference(snapshots=True)
    c.reset()
    out = c.prefill(keep_in_place=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(c.pool.tensor, ref_pool)
    c.reset()
    out = c.verify()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    for r, n in enumerate(c.lens):
        if c.rs_np[r] == 0:
            continue
        for i in range(n):
            assert torch.equal(c.pool.tensor[int(c.ts_np[c.cu_np[r] + i])], snaps[i][int(c.rs_np[r])])
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_prefill_256_tokens_matches_oracle(gdn, orc):
    """A 256-token prefill (0.8B shape, twin) against the fp64 oracle: every
    output within the bf16 tolerance and every final state within the
    chained-state tolerance of 256 steps."""
    s = I.QWEN_08B
    c = Case(gdn, s, [256, 0, 3], seed=77, n_pad=0)
    out = c.prefill()
    torch.cuda.synchronize()
    pool = c.pool_np.astype(np.float64).copy()
    o_ref, bad = orc.prefill(c.cu_np, c.ref["q"], c.ref["k"], c.ref["v"], c.ref["a"], c.ref["b"],
                             c.prm["A_log"], c.prm["dt_bias"], pool, c.rs_np, write_slot=c.ws_np)
    assert bad == 0
    assert_out_close(f64(out), o_ref, s.dtype)
    got = c.pool.tensor.cpu().numpy()
    for sl in c.ws_np:
        for h in range(s.hv):
            err = state_rel_err(got[sl, h], pool[sl, h])
            assert err <= STATE_TOL_CHAIN, f"slot {sl} head {h}: {err:.3g}"
    assert gdn.get_device_error() == 0


def test_step_and_prefill_with_pinned_host_activations(gdn):
    """gdn_decode_step and gdn_prefill read q, k, v, a, b and write their
    outputs in pinned host memory too, with the values of device buffers."""
    s = I.QWEN_08B
    c = Case(gdn, s, [5, 0, 3, 7], seed=78)
    c.reset()
    ref = c.prefill(keep_in_place=True).clone()
    torch.cuda.synchronize()
    ref_pool = c.pool.tensor.clone()
    c.reset()
    h = {k: c.dev[k].cpu().pin_memory() for k in ("q", "k", "v", "a", "b")}
    hout = torch.empty(ref.shape, dtype=ref.dtype).pin_memory()
    gdn.gdn_prefill(h["q"], h["k"], h["v"], h["a"], h["b"], c.A_log, c.dt_bias, c.pool, c.cu, c.rs, None,
                    out=hout, keep_in_place=True)
    torch.cuda.synchronize()
    assert torch.equal(hout, ref.cpu()) and torch.equal(c.pool.tensor, ref_pool)
    # one decode step over the first token of every sequence
    c.reset()
    idx, rs = c.step_rows(0)
    it = torch.from_numpy(idx).cuda()
    dev_in = [c.dev[k][it].contiguous() for k in ("q", "k", "v", "a", "b")]
    o_ref = gdn.gdn_decode_step(*dev_in, c.A_log, c.dt_bias, c.pool, ti(rs), None, keep_in_place=True).clone()
    torch.cuda.synchronize()
    p_ref = c.pool.tensor.clone()
    c.reset()
    host_in = [t_.cpu().pin_memory() for t_ in dev_in]
    hout = torch.empty(o_ref.shape, dtype=o_ref.dtype).pin_memory()
    gdn.gdn_decode_step(*host_in, c.A_log, c.dt_bias, c.pool, ti(rs), None, out=hout, keep_in_place=True)
    torch.cuda.synchronize()
    assert torch.equal(hout, o_ref.cpu()) and torch.equal(c.pool.tensor, p_ref)
    assert gdn.get_device_error() == 0
