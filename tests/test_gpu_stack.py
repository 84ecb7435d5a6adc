"""The decode-stack stand-in: 18 GDN layers of the 0.8B shape run back to back
per step (fused conv + rule), 128 rows, a 257-slot state pool and conv pool per
layer, twin slots with one commit per step shared by all layers, and the rows'
request order re-permuted every 16 steps with 10% padding rows.

Checks: a CUDA-graph replay of whole steps equals eager execution bit for bit;
with fp32 activations (no bf16 rounding at the conv boundary) sampled
(layer, request, head) states follow the fp64 oracle's layer through the
chained steps within the chained-state tolerance; every slot outside the
write set is untouched.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import STATE_TOL_CHAIN, assert_out_close, f64, pair, state_rel_err, t, ti

pytestmark = pytest.mark.gpu

ROWS = 128
PAD = 0.10


class Stack:
    """Layers sharing one slot table; requests keep their two slots while
    their row position moves."""

    def __init__(self, gdn, layers: int, dtype: str, seed: int):
        self.gdn = gdn
        self.s = I.STACK.with_(dtype=dtype)
        self.gen = I.Gen(seed)
        s = self.s
        self.layers = []
        for _ in range(layers):
            prm = self.gen.params(s)
            L = {"prm": prm, "pool_np": self.gen.state_pool(s), "cp_np": self.gen.conv_pool(s)}
            L["w"], L["w64"] = pair(prm["w"], dtype)
            L["bias"], L["bias64"] = pair(prm["bias"], dtype)
            L["A_log"], L["dt_bias"] = t(prm["A_log"]), t(prm["dt_bias"])
            cp_dev, L["cp64"] = pair(L["cp_np"], dtype)
            L["pool"] = gdn.GDNStatePool(s.num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                                         tensor=torch.from_numpy(L["pool_np"].copy()).cuda())
            L["cp"] = gdn.ConvStatePool(s.num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda",
                                        tensor=cp_dev.clone())
            L["out"] = torch.empty((ROWS, s.hv, s.dv), dtype=I.torch_dtype(dtype), device="cuda")
            self.layers.append(L)
        n_real = ROWS - int(PAD * ROWS)
        perm = self.gen.rng.permutation(np.arange(1, s.num_slots, dtype=np.int32))
        self.req_rs = perm[:n_real].copy()          # each request's two slots
        self.req_ws = perm[n_real:2 * n_real].copy()
        self.rs = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
        self.ws = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
        self.x = torch.empty((len(self.layers), ROWS, s.channels), dtype=I.torch_dtype(dtype), device="cuda")
        self.a = torch.empty((len(self.layers), ROWS, s.hv), dtype=I.torch_dtype(dtype), device="cuda")
        self.b = torch.empty_like(self.a)

    def place(self):
        """New row order: padding rows at random positions, requests shuffled."""
        n_real = len(self.req_rs)
        pos = self.gen.rng.permutation(ROWS)[:n_real]
        order = self.gen.rng.permutation(n_real)
        rs = np.zeros(ROWS, np.int32)
        ws = np.zeros(ROWS, np.int32)
        rs[pos] = self.req_rs[order]
        ws[pos] = self.req_ws[order]
        self.rs.copy_(ti(rs))
        self.ws.copy_(ti(ws))
        self.row_req = np.full(ROWS, -1)
        self.row_req[pos] = order
        return rs, ws

    def draw(self):
        """This step's inputs for every layer; returns their exact values."""
        ex = []
        for li in range(len(self.layers)):
            inp = self.gen.layer_inputs(self.s.with_(rows=ROWS))
            d = {}
            for k in ("x", "a", "b"):
                dev, d[k] = pair(inp[k], self.s.dtype)
                getattr(self, k)[li].copy_(dev)
            ex.append(d)
        return ex

    def step(self, fused_commit=False):
        """All layers, then the commit (with fused_commit, inside the last
        layer's launch)."""
        n = len(self.layers)
        for li, L in enumerate(self.layers):
            self.gdn.gdn_layer_decode(self.x[li], L["cp"], L["w"], L["bias"], L["A_log"], L["dt_bias"],
                                      self.a[li], self.b[li], L["pool"], self.rs, self.ws, out=L["out"],
                                      commit=fused_commit and li == n - 1)
        if not fused_commit:
            self.gdn.gdn_commit(self.rs, self.ws)
        # the commit swaps every request's two slots; keep the host copy in step
        self.req_rs, self.req_ws = self.req_ws, self.req_rs


@pytest.mark.parametrize("fused_commit", [False, True], ids=["commit_kernel", "commit_in_last_layer"])
def test_stack_graph_replay_equals_eager(gdn, fused_commit):
    """Eager steps (separate commit) against graph replays of steps whose
    commit is a separate kernel or folded into the last layer's launch."""
    torch.manual_seed(0)
    st = Stack(gdn, layers=18, dtype="bf16", seed=40)
    st.place()
    st.draw()
    snap0 = [(L["pool"].tensor.clone(), L["cp"].tensor.clone()) for L in st.layers]
    rs0, ws0 = st.rs.clone(), st.ws.clone()
    for _ in range(4):
        st.step()  # (host bookkeeping of request slots is not used by this test)
    torch.cuda.synchronize()
    eager = [(L["pool"].tensor.clone(), L["cp"].tensor.clone(), L["out"].clone()) for L in st.layers]
    eager_rs = st.rs.clone()
    for (p0, c0), L in zip(snap0, st.layers):
        L["pool"].tensor.copy_(p0)
        L["cp"].tensor.copy_(c0)
    st.rs.copy_(rs0)
    st.ws.copy_(ws0)
    st.step(fused_commit)  # warm-up of every launch path before capture (error word lookup, attributes)
    for (p0, c0), L in zip(snap0, st.layers):
        L["pool"].tensor.copy_(p0)
        L["cp"].tensor.copy_(c0)
    st.rs.copy_(rs0)
    st.ws.copy_(ws0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st.step(fused_commit)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.rs, eager_rs)
    for (pe, ce, oe), L in zip(eager, st.layers):
        assert torch.equal(L["pool"].tensor, pe)
        assert torch.equal(L["cp"].tensor, ce)
        assert torch.equal(L["out"], oe)
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_stack_chained_parity_fp32(gdn, orc):
    """64 steps of the stack (18 layers) with fp32 activations; the oracle
    follows two layers' sampled (request, head) states through every step,
    including the re-permutations of the row order every 16 steps."""
    st = Stack(gdn, layers=18, dtype="f32", seed=41)
    s = st.s
    follow = [0, 17]
    req_heads = [(0, 0), (5, 7), (57, 15), (100, 3)]
    # oracle-side state per (layer, request, head) and conv window per (layer, request)
    S = {(li, rq, h): st.layers[li]["pool_np"][st.req_rs[rq], h].astype(np.float64)
         for li in follow for rq, h in req_heads}
    Wn = {(li, rq): st.layers[li]["cp64"][st.req_rs[rq]].copy() for li in follow for rq, _ in req_heads}
    for step in range(64):
        if step % 16 == 0:
            st.place()
        ex = st.draw()
        st.step()
        for li in follow:
            L = st.layers[li]
            for rq in {rq for rq, _ in req_heads}:
                r = int(np.nonzero(st.row_req == rq)[0][0])
                # one row of the oracle's layer on this request's own fp64 state and window
                x = ex[li]["x"][r:r + 1]
                cp = np.zeros((3, 3, s.channels))
                cp[1] = Wn[(li, rq)]
                pool = np.zeros((3, s.hv, s.dv, s.dk))
                for h in range(s.hv):
                    key = (li, rq, h)
                    if key in S:
                        pool[1, h] = S[key]
                o, bad = orc.layer(x, cp, L["w64"], L["bias64"], ex[li]["a"][r:r + 1], ex[li]["b"][r:r + 1],
                                   L["prm"]["A_log"], L["prm"]["dt_bias"], pool, np.array([1], np.int32),
                                   np.array([2], np.int32), hk=s.hk, act_bf16=False)
                assert bad == 0
                Wn[(li, rq)] = cp[2].copy()
                for h in range(s.hv):
                    if (li, rq, h) in S:
                        S[(li, rq, h)] = pool[2, h].copy()
                        if step % 16 == 15:
                            assert_out_close(f64(L["out"][r, h]), o[0, h], "f32", f"step {step} layer {li}")
    torch.cuda.synchronize()
    req_rs = st.req_rs
    rs_gpu = st.rs.cpu().numpy()
    assert np.array_equal(np.sort(rs_gpu[rs_gpu > 0]), np.sort(req_rs))
    for li in follow:
        pool = st.layers[li]["pool"].tensor.cpu().numpy()
        for rq, h in req_heads:
            err = state_rel_err(pool[req_rs[rq], h], S[(li, rq, h)])
            assert err <= STATE_TOL_CHAIN, f"layer {li} request {rq} head {h}: {err:.3g}"
    assert gdn.get_device_error() == 0
