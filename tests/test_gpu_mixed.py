"""GPU checks of the decode half of a mixed step (gdn_layer_decode_bucket):
the launch covers the bucket, a device-side count says how many leading rows
decode ("mstar PR #965", section "What changed").

1. Rows below the count equal gdn_layer_decode over those rows alone, bit for
   bit; rows past it have zero outputs and their slots, windows and table
   entries stay as they were, although they name real slots.
2. With the commit in the launch, only the decoded rows' tables swap.
3. One captured launch serves every count (the count is read on the device).
4. The decoded rows match the fp64 oracle's layer on the same rows (tiny fp32,
   and the 0.8B and 9B shapes in bf16 with 48 of 64 rows decoding).
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import (STATE_TOL_ONE, assert_out_close, f64, oracle_layer_on_gpu_roundings, pair,
                         state_rel_err, t, ti)

pytestmark = pytest.mark.gpu


class Bucket:
    def __init__(self, gdn, s: I.Shape, seed: int):
        self.gdn, self.s = gdn, s
        gen = I.Gen(seed)
        self.num_slots = 2 * s.rows + 1
        prm = gen.params(s)
        self.prm = prm
        self.w, self.w64 = pair(prm["w"], s.dtype)
        self.bias, self.bias64 = pair(prm["bias"], s.dtype)
        self.A_log, self.dt_bias = t(prm["A_log"]), t(prm["dt_bias"])
        self.pool_np = gen.state_pool(s, self.num_slots)
        cp_dev, self.cp64 = pair(gen.conv_pool(s, self.num_slots), s.dtype)
        self.cp_start = cp_dev.clone()
        self.pool = gdn.GDNStatePool(self.num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                                     tensor=torch.from_numpy(self.pool_np.copy()).cuda())
        self.cp = gdn.ConvStatePool(self.num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda",
                                    tensor=cp_dev)
        # every row of the bucket names real slots: the rows past the count are prefill rows
        self.rs_np, self.ws_np = gen.slot_tables(s.rows, self.num_slots)
        self.rs, self.ws = ti(self.rs_np), ti(self.ws_np)
        self.dev, self.ref = {}, {}
        for k, v in gen.layer_inputs(s).items():
            self.dev[k], self.ref[k] = pair(v, s.dtype)

    def reset(self):
        self.pool.tensor.copy_(torch.from_numpy(self.pool_np).cuda())
        self.cp.tensor.copy_(self.cp_start)
        self.rs.copy_(ti(self.rs_np))
        self.ws.copy_(ti(self.ws_np))

    def bucket(self, n, out=None, commit=False):
        d = self.dev
        return self.gdn.gdn_layer_decode_bucket(d["x"], self.cp, self.w, self.bias, self.A_log, self.dt_bias,
                                                d["a"], d["b"], self.pool, self.rs, self.ws, n, out=out,
                                                commit=commit)

    def leading(self, k):
        d = self.dev
        return self.gdn.gdn_layer_decode(d["x"][:k].contiguous(), self.cp, self.w, self.bias, self.A_log,
                                         self.dt_bias, d["a"][:k].contiguous(), d["b"][:k].contiguous(),
                                         self.pool, self.rs[:k].contiguous(), self.ws[:k].contiguous())


@pytest.mark.parametrize("shape", [I.TINY, I.QWEN_08B], ids=["tiny", "0.8b"])
def test_bucket_equals_leading_rows(gdn, shape):
    c = Bucket(gdn, shape, seed=80)
    for k in sorted({0, 1, shape.rows // 2 + 1, shape.rows}):
        c.reset()
        ref = c.leading(k).clone() if k else None
        torch.cuda.synchronize()
        ref_pool, ref_cp = c.pool.tensor.clone(), c.cp.tensor.clone()
        c.reset()
        out = c.bucket(ti(np.array([k], np.int32)))
        torch.cuda.synchronize()
        if k:
            assert torch.equal(out[:k], ref)
        assert not out[k:].any()
        assert torch.equal(c.pool.tensor, ref_pool), f"k={k}"
        assert torch.equal(c.cp.tensor, ref_cp), f"k={k}"
        assert torch.equal(c.rs, ti(c.rs_np)) and torch.equal(c.ws, ti(c.ws_np))
    assert gdn.get_device_error() == 0


def test_bucket_commit_swaps_only_decoded_rows(gdn):
    s = I.QWEN_08B
    c = Bucket(gdn, s, seed=81)
    k = 23
    c.reset()
    ref = c.leading(k).clone()
    torch.cuda.synchronize()
    ref_pool = c.pool.tensor.clone()
    c.reset()
    out = c.bucket(ti(np.array([k], np.int32)), commit=True)
    torch.cuda.synchronize()
    assert torch.equal(out[:k], ref) and not out[k:].any()
    assert torch.equal(c.pool.tensor, ref_pool)
    rs, ws = c.rs.cpu().numpy(), c.ws.cpu().numpy()
    assert np.array_equal(rs[:k], c.ws_np[:k]) and np.array_equal(ws[:k], c.rs_np[:k])
    assert np.array_equal(rs[k:], c.rs_np[k:]) and np.array_equal(ws[k:], c.ws_np[k:])
    assert gdn.get_device_error() == 0


def test_bucket_graph_replay_serves_every_count(gdn):
    s = I.QWEN_08B
    c = Bucket(gdn, s, seed=82)
    n = ti(np.array([s.rows], np.int32))
    out = torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device="cuda")
    c.reset()
    c.bucket(n, out=out)  # warm-up of the launch path before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            c.bucket(n, out=out)
    torch.cuda.current_stream().wait_stream(side)
    for k in (5, 40, 0, s.rows):
        c.reset()
        n.fill_(k)
        g.replay()
        torch.cuda.synchronize()
        got, got_pool = out.clone(), c.pool.tensor.clone()
        c.reset()
        ref = c.bucket(ti(np.array([k], np.int32)))
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"k={k}"
        assert torch.equal(got_pool, c.pool.tensor), f"k={k}"
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape,k", [(I.TINY.with_(rows=6), 4), (I.QWEN_08B, 48), (I.QWEN_9B, 48)],
                         ids=["tiny", "0.8b", "9b"])
def test_bucket_matches_oracle(gdn, orc, shape, k):
    """The decoded rows of a bucket match the oracle's layer over those rows
    (every head's state within 1e-5, outputs within the activation tolerance,
    windows bit-exact); the rows past the count are left alone."""
    s = shape
    c = Bucket(gdn, s, seed=83)
    c.reset()
    # the GPU's conv outputs (rounding choices at midpoints) for the decoded rows: the
    # standalone conv writes the windows the bucket launch writes next
    d = c.dev
    y_gpu = f64(gdn.causal_conv1d_decode(d["x"][:k].contiguous(), c.cp, c.rs[:k].contiguous(), c.w, c.bias,
                                         write_slot=c.ws[:k].contiguous()))
    out = c.bucket(ti(np.array([k], np.int32)))
    torch.cuda.synchronize()
    pool = c.pool_np.astype(np.float64).copy()
    cp = c.cp64.copy()
    sub = {name: v[:k] for name, v in c.ref.items()}
    o_ref, _ = oracle_layer_on_gpu_roundings(orc, y_gpu, sub, cp, c.w64, c.bias64, c.prm["A_log"],
                                             c.prm["dt_bias"], pool, c.rs_np[:k], c.ws_np[:k], s)
    assert_out_close(f64(out[:k]), o_ref, s.dtype)
    assert not out[k:].any()
    got = c.pool.tensor.cpu().numpy()
    for r in range(k):
        err = state_rel_err(got[c.ws_np[r]], pool[c.ws_np[r]])
        assert (err <= STATE_TOL_ONE).all(), f"row {r}: state rel err {err.max():.3g}"
    assert np.array_equal(f64(c.cp.tensor), cp)
    for r in range(k, s.rows):
        assert np.array_equal(got[c.ws_np[r]], c.pool_np[c.ws_np[r]])
        assert np.array_equal(got[c.rs_np[r]], c.pool_np[c.rs_np[r]])
    assert gdn.get_device_error() == 0
