"""GPU checks of the fused conv + GDN layer (gdn_layer_decode).

1. The fused kernel equals causal_conv1d_decode followed by gdn_decode_step,
   bit for bit (outputs, state pool, conv pool), twin and in place, for the
   tiny, 0.8B- and 9B-shaped layers.
2. It matches the fp64 oracle's layer: outputs within the bf16 tolerance,
   conv windows and untouched slots bit-exact, every head's state within
   1e-5.  Where the GPU's fp32 conv landed on the other side of a bf16
   rounding midpoint (accepted by the conv check), the oracle takes that
   other rounding of its own exact value; everything else is the oracle's.
   The 0.8B layer is also chained 256 steps (commit in the launch) against
   the oracle on sampled rows, states within 1e-3 at the end.
3. In place (clustered launch) equals twin, bit for bit.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import (STATE_TOL_CHAIN, STATE_TOL_ONE, assert_out_close, f64,
                         oracle_layer_on_gpu_roundings, pair, state_rel_err, t, ti)

pytestmark = pytest.mark.gpu


class LayerCase:
    def __init__(self, gdn, s: I.Shape, seed: int, num_slots: int, pad_frac=0.0):
        self.gdn, self.s = gdn, s
        self.gen = I.Gen(seed)
        prm = self.gen.params(s)
        self.prm = prm
        self.w, self.w64 = pair(prm["w"], s.dtype)
        self.bias, self.bias64 = pair(prm["bias"], s.dtype)
        self.A_log, self.dt_bias = t(prm["A_log"]), t(prm["dt_bias"])
        self.pool_np = self.gen.state_pool(s, num_slots)
        cp_dev, self.cp64 = pair(self.gen.conv_pool(s, num_slots), s.dtype)
        self.cp_start = cp_dev.clone()
        self.pool = gdn.GDNStatePool(num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                                     tensor=torch.from_numpy(self.pool_np.copy()).cuda())
        self.cp = gdn.ConvStatePool(num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda",
                                    tensor=cp_dev)
        self.rs_np, self.ws_np = self.gen.slot_tables(s.rows, num_slots, pad_frac)
        self.rs, self.ws = ti(self.rs_np), ti(self.ws_np)

    def draw(self):
        dev, ref = {}, {}
        for k, v in self.gen.layer_inputs(self.s).items():
            dev[k], ref[k] = pair(v, self.s.dtype)
        return dev, ref

    def reset(self):
        self.pool.tensor.copy_(torch.from_numpy(self.pool_np).cuda())
        self.cp.tensor.copy_(self.cp_start)

    def fused(self, xd, keep_in_place=False):
        return self.gdn.gdn_layer_decode(xd["x"], self.cp, self.w, self.bias, self.A_log, self.dt_bias,
                                         xd["a"], xd["b"], self.pool, self.rs,
                                         None if keep_in_place else self.ws, keep_in_place=keep_in_place)

    def unfused(self, xd, keep_in_place=False):
        s = self.s
        y = self.gdn.causal_conv1d_decode(xd["x"], self.cp, self.rs, self.w, self.bias,
                                          write_slot=None if keep_in_place else self.ws)
        nq = s.hk * s.dk
        q = y[:, :nq].contiguous()
        k = y[:, nq:2 * nq].contiguous()
        v = y[:, 2 * nq:].contiguous()
        out = self.gdn.gdn_decode_step(q, k, v, xd["a"], xd["b"], self.A_log, self.dt_bias, self.pool,
                                       self.rs, None if keep_in_place else self.ws,
                                       keep_in_place=keep_in_place)
        return out, y


@pytest.mark.parametrize("shape", [I.TINY, I.QWEN_08B, I.QWEN_9B], ids=["tiny", "0.8b", "9b"])
@pytest.mark.parametrize("keep_in_place", [False, True], ids=["twin", "in_place"])
def test_fused_equals_unfused(gdn, shape, keep_in_place):
    c = LayerCase(gdn, shape, seed=30, num_slots=2 * shape.rows + 1, pad_frac=0.25)
    xd, _ = c.draw()
    o_f = c.fused(xd, keep_in_place).clone()
    torch.cuda.synchronize()
    pool_f, cp_f = c.pool.tensor.clone(), c.cp.tensor.clone()
    c.reset()
    o_u, _ = c.unfused(xd, keep_in_place)
    torch.cuda.synchronize()
    assert torch.equal(o_f, o_u)
    assert torch.equal(pool_f, c.pool.tensor)
    assert torch.equal(cp_f, c.cp.tensor)
    assert gdn.get_device_error() == 0


def test_in_place_equals_twin(gdn):
    s = I.QWEN_9B
    c = LayerCase(gdn, s, seed=31, num_slots=2 * s.rows + 1, pad_frac=0.1)
    xd, _ = c.draw()
    o_t = c.fused(xd).clone()
    torch.cuda.synchronize()
    pool_t, cp_t = c.pool.tensor.clone(), c.cp.tensor.clone()
    c.reset()
    o_i = c.fused(xd, keep_in_place=True).clone()
    torch.cuda.synchronize()
    rs = torch.from_numpy(c.rs_np).long().cuda()
    ws = torch.from_numpy(c.ws_np).long().cuda()
    real = rs != 0
    assert torch.equal(o_t, o_i)
    assert torch.equal(pool_t[ws[real]], c.pool.tensor[rs[real]])
    assert torch.equal(cp_t[ws[real]], c.cp.tensor[rs[real]])
    # twin left every read slot alone
    assert torch.equal(pool_t[rs[real]], torch.from_numpy(c.pool_np).cuda()[rs[real]])
    assert torch.equal(cp_t[rs[real]], c.cp_start[rs[real]])


@pytest.mark.parametrize("shape", [I.TINY, I.QWEN_08B, I.QWEN_9B], ids=["tiny", "0.8b", "9b"])
@pytest.mark.parametrize("keep_in_place", [False, True], ids=["twin", "in_place"])
def test_fused_matches_oracle(gdn, orc, shape, keep_in_place):
    s = shape
    c = LayerCase(gdn, s, seed=32, num_slots=2 * s.rows + 1, pad_frac=0.25)
    xd, xr = c.draw()
    # the GPU's conv outputs, the selector of its rounding at midpoints: the standalone
    # conv equals the fused kernel's bit for bit (test_fused_equals_unfused)
    y_gpu = f64(gdn.causal_conv1d_decode(xd["x"], c.cp, c.rs, c.w, c.bias,
                                         write_slot=None if keep_in_place else c.ws))
    c.reset()
    out = c.fused(xd, keep_in_place)
    torch.cuda.synchronize()
    pool_gpu = c.pool.tensor.cpu().numpy()
    cp_gpu = f64(c.cp.tensor)
    p_ref = c.pool_np.astype(np.float64)
    cp_ref = c.cp64.copy()
    o_ref, flips = oracle_layer_on_gpu_roundings(orc, y_gpu, xr, cp_ref, c.w64, c.bias64, c.prm["A_log"],
                                                 c.prm["dt_bias"], p_ref, c.rs_np, c.ws_np, s,
                                                 keep_in_place=keep_in_place)
    assert_out_close(f64(out), o_ref, s.dtype)
    assert np.array_equal(cp_gpu, cp_ref)
    real = c.rs_np != 0
    dst = c.rs_np if keep_in_place else c.ws_np
    for r in np.nonzero(real)[0]:
        err = state_rel_err(pool_gpu[dst[r]], p_ref[dst[r]])
        assert (err <= STATE_TOL_ONE).all(), f"row {r}: state rel err {err.max():.3g}"
    # every slot the step does not write is bit-identical, the null slot included
    untouched = np.setdiff1d(np.arange(c.pool_np.shape[0]), dst[real])
    assert np.array_equal(pool_gpu[untouched], c.pool_np[untouched])
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_fused_qwen08b_256_chained_steps_with_commit(gdn, orc):
    """The 0.8B-shaped layer (64 rows, bf16), 256 chained twin steps of
    gdn_layer_decode with the commit in its launch.  Sampled rows are followed
    through the oracle's layer the whole way (windows and states in fp64, the
    GPU's rounding choice taken only at accepted bf16 midpoints); their outputs
    are checked every step and their states are held to the chained tolerance
    at the end, their windows bit-exact."""
    s = I.QWEN_08B
    c = LayerCase(gdn, s, seed=37, num_slots=s.num_slots)
    sample = np.array([0, 17, 40, 63])
    p_ref = c.pool_np.astype(np.float64)
    cp_ref = c.cp64.copy()
    rs, ws = c.rs_np.copy(), c.ws_np.copy()
    n_flips = 0
    for step in range(256):
        xd, xr = c.draw()
        # the standalone conv writes the very window the fused step writes next
        y_gpu = f64(gdn.causal_conv1d_decode(xd["x"], c.cp, c.rs, c.w, c.bias, write_slot=c.ws))
        out = gdn.gdn_layer_decode(xd["x"], c.cp, c.w, c.bias, c.A_log, c.dt_bias, xd["a"], xd["b"], c.pool,
                                   c.rs, c.ws, commit=True)
        sub = {k: v[sample] for k, v in xr.items()}
        o_ref, flips = oracle_layer_on_gpu_roundings(orc, y_gpu[sample], sub, cp_ref, c.w64, c.bias64,
                                                     c.prm["A_log"], c.prm["dt_bias"], p_ref, rs[sample],
                                                     ws[sample], s)
        n_flips += int(flips.sum())
        assert_out_close(f64(out)[sample], o_ref, s.dtype, f"step {step}")
        orc.commit(rs, ws)
    torch.cuda.synchronize()
    assert np.array_equal(c.rs.cpu().numpy(), rs) and np.array_equal(c.ws.cpu().numpy(), ws)
    pool_gpu = c.pool.tensor.cpu().numpy()
    cp_gpu = f64(c.cp.tensor)
    for r in sample:
        err = state_rel_err(pool_gpu[rs[r]], p_ref[rs[r]])
        assert (err <= STATE_TOL_CHAIN).all(), f"row {r}: state rel err {err.max():.3g} after 256 steps"
        assert np.array_equal(cp_gpu[rs[r]], cp_ref[rs[r]])
    print(f"bf16 midpoint choices taken from the GPU over 256 steps: {n_flips}")
    assert gdn.get_device_error() == 0


def test_fused_tiny_chained_vs_oracle(gdn, orc):
    """8 chained twin steps of the fp32 tiny layer against the oracle's layer."""
    s = I.TINY
    c = LayerCase(gdn, s, seed=33, num_slots=s.num_slots)
    p_ref = c.pool_np.astype(np.float64)
    cp_ref = c.cp64.copy()
    rs, ws = c.rs_np.copy(), c.ws_np.copy()
    for step in range(8):
        xd, xr = c.draw()
        out = c.fused(xd)
        o_ref, bad = orc.layer(xr["x"], cp_ref, c.w64, c.bias64, xr["a"], xr["b"], c.prm["A_log"],
                               c.prm["dt_bias"], p_ref, rs, ws, hk=s.hk, act_bf16=False)
        assert bad == 0
        assert_out_close(f64(out), o_ref, "f32", f"step {step}")
        gdn.gdn_commit(c.rs, c.ws)
        orc.commit(rs, ws)
    torch.cuda.synchronize()
    pool_gpu = c.pool.tensor.cpu().numpy()
    assert state_rel_err(pool_gpu[rs], p_ref[rs]).max() <= 8 * STATE_TOL_ONE
    # fp32 windows: the shift copies values, so they match the oracle's exactly
    assert np.array_equal(f64(c.cp.tensor), cp_ref)


def test_repeated_launches_reuse_the_work_counters(gdn):
    """With many items a CTA the kernels hand out the tail of their work
    through the pool's pair of work counters and leave it at zero when they
    end: launch after launch on one pool (twin, in place, twin, fused and
    unfused) writes every output and gives identical values."""
    s = I.QWEN_08B.with_(rows=256)
    c = LayerCase(gdn, s, seed=33, num_slots=2 * s.rows + 1, pad_frac=0.1)
    xd, _ = c.draw()
    out = torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device="cuda")
    runs = []
    for keep_in_place in (False, True, False, False):
        c.reset()
        out.fill_(float("nan"))
        gdn.gdn_layer_decode(xd["x"], c.cp, c.w, c.bias, c.A_log, c.dt_bias, xd["a"], xd["b"], c.pool,
                             c.rs, None if keep_in_place else c.ws, out=out, keep_in_place=keep_in_place)
        torch.cuda.synchronize()
        runs.append((keep_in_place, out.clone(), c.pool.tensor.clone()))
    for _ in range(2):
        c.reset()
        o_u, _ = c.unfused(xd)
        torch.cuda.synchronize()
        runs.append((False, o_u.clone(), c.pool.tensor.clone()))
    o0, p0 = runs[0][1], runs[0][2]
    assert not torch.isnan(o0.float()).any()
    for keep_in_place, o, p in runs[1:]:
        assert torch.equal(o, o0)
        if not keep_in_place:
            assert torch.equal(p, p0)
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape", [I.TINY, I.QWEN_08B, I.QWEN_08B.with_(rows=256), I.QWEN_9B],
                         ids=["tiny", "0.8b", "0.8b-256rows", "9b"])
def test_fused_commit_equals_layer_then_commit(gdn, shape):
    """gdn_layer_decode_commit gives the values of gdn_layer_decode followed by
    gdn_commit, bit for bit, and leaves the slot tables swapped; two steps in
    a row read the committed tables."""
    c = LayerCase(gdn, shape, seed=34, num_slots=2 * shape.rows + 1, pad_frac=0.25)
    steps = [c.draw()[0] for _ in range(2)]
    rs0, ws0 = c.rs.clone(), c.ws.clone()
    ref = []
    for xd in steps:
        o = c.fused(xd).clone()
        gdn.gdn_commit(c.rs, c.ws)
        torch.cuda.synchronize()
        ref.append((o, c.rs.clone(), c.ws.clone()))
    ref_pool, ref_cp = c.pool.tensor.clone(), c.cp.tensor.clone()
    c.reset()
    c.rs.copy_(rs0)
    c.ws.copy_(ws0)
    for (o_ref, rs_ref, ws_ref), xd in zip(ref, steps):
        o = gdn.gdn_layer_decode(xd["x"], c.cp, c.w, c.bias, c.A_log, c.dt_bias, xd["a"], xd["b"], c.pool,
                                 c.rs, c.ws, commit=True).clone()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(c.rs, rs_ref) and torch.equal(c.ws, ws_ref)
    assert torch.equal(c.pool.tensor, ref_pool)
    assert torch.equal(c.cp.tensor, ref_cp)
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_claim_counters_under_repetition_and_two_streams(gdn):
    """The claimed tail and its counter reset, over and over: 40 launches of
    the fused layer with its commit (256 rows, where half of the work is
    claimed) give identical outputs and states every time; and two pools
    driven from two streams at once, each with its own counters, give what
    they give one after the other."""
    s = I.QWEN_08B.with_(rows=256)
    cases = [LayerCase(gdn, s, seed=35 + i, num_slots=2 * s.rows + 1, pad_frac=0.1) for i in range(2)]
    inputs = [c.draw()[0] for c in cases]

    def run(c, xd, stream=None):
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            return gdn.gdn_layer_decode(xd["x"], c.cp, c.w, c.bias, c.A_log, c.dt_bias, xd["a"], xd["b"],
                                        c.pool, c.rs, c.ws, commit=True)

    # one after the other: the reference
    refs = []
    for c, xd in zip(cases, inputs):
        c.reset()
        rs0, ws0 = c.rs.clone(), c.ws.clone()
        o = run(c, xd).clone()
        torch.cuda.synchronize()
        refs.append((o, c.pool.tensor.clone(), c.cp.tensor.clone(), c.rs.clone(), c.ws.clone()))
        c.rs.copy_(rs0)
        c.ws.copy_(ws0)
    c0, xd0 = cases[0], inputs[0]
    rs0, ws0 = c0.rs.clone(), c0.ws.clone()
    for rep in range(40):
        c0.reset()
        c0.rs.copy_(rs0)
        c0.ws.copy_(ws0)
        o = run(c0, xd0)
        torch.cuda.synchronize()
        assert torch.equal(o, refs[0][0]), f"launch {rep}"
        assert torch.equal(c0.pool.tensor, refs[0][1]), f"launch {rep}"
        assert torch.equal(c0.rs, refs[0][3]) and torch.equal(c0.ws, refs[0][4]), f"launch {rep}"
    # both pools at once, on two streams
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(10):
        for c in cases:
            c.reset()
        cases[0].rs.copy_(rs0)
        cases[0].ws.copy_(ws0)
        rs1, ws1 = refs[1][4], refs[1][3]  # the second case's tables before its commit
        cases[1].rs.copy_(rs1)
        cases[1].ws.copy_(ws1)
        torch.cuda.synchronize()
        outs = [run(c, xd, st) for c, xd, st in zip(cases, inputs, streams)]
        torch.cuda.synchronize()
        for i, (c, o) in enumerate(zip(cases, outs)):
            assert torch.equal(o, refs[i][0]), f"pool {i}, round {rep}"
            assert torch.equal(c.pool.tensor, refs[i][1]), f"pool {i}, round {rep}"
            assert torch.equal(c.cp.tensor, refs[i][2]), f"pool {i}, round {rep}"
    assert gdn.get_device_error() == 0


def test_activations_in_pinned_host_memory(gdn):
    """x, a, b and the output may live in pinned host memory: the fused layer
    (with its commit) reads and writes them across the host link and gives
    the values it gives with device buffers, bit for bit."""
    s = I.QWEN_08B
    c = LayerCase(gdn, s, seed=36, num_slots=2 * s.rows + 1, pad_frac=0.25)
    xd, _ = c.draw()
    rs0, ws0 = c.rs.clone(), c.ws.clone()
    ref = gdn.gdn_layer_decode(xd["x"], c.cp, c.w, c.bias, c.A_log, c.dt_bias, xd["a"], xd["b"], c.pool,
                               c.rs, c.ws, commit=True).clone()
    torch.cuda.synchronize()
    ref_pool, ref_cp, ref_rs = c.pool.tensor.clone(), c.cp.tensor.clone(), c.rs.clone()
    c.reset()
    c.rs.copy_(rs0)
    c.ws.copy_(ws0)
    hx, ha, hb = (xd[k].cpu().pin_memory() for k in ("x", "a", "b"))
    hout = torch.full(ref.shape, float("nan"), dtype=ref.dtype).pin_memory()
    gdn.gdn_layer_decode(hx, c.cp, c.w, c.bias, c.A_log, c.dt_bias, ha, hb, c.pool, c.rs, c.ws, out=hout,
                         commit=True)
    torch.cuda.synchronize()
    assert torch.equal(hout, ref.cpu())
    assert torch.equal(c.pool.tensor, ref_pool) and torch.equal(c.cp.tensor, ref_cp)
    assert torch.equal(c.rs, ref_rs)
    with pytest.raises(ValueError):
        gdn.gdn_layer_decode(xd["x"].cpu(), c.cp, c.w, c.bias, c.A_log, c.dt_bias, ha, hb, c.pool, c.rs,
                             c.ws)  # plain (pageable) host memory is refused
    assert gdn.get_device_error() == 0
