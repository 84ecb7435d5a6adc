"""The bounded-wait failure path on the GPU, with no fault: a kernel waits on
a shared-memory barrier that nothing arrives at, through the same bounded wait
every kernel uses, with a short time limit; the wait gives up, the device
error word reads the timeout, and the context keeps serving calls -- the next
fused layer call still matches the oracle."""
import time

import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import STATE_TOL_ONE, assert_out_close, f64, pair, state_rel_err, t, ti

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_survives(gdn, orc):
    gdn.get_device_error()                                    # start from a clear word
    for limit_us in (1000, 200000):
        t0 = time.perf_counter()
        gdn.selftest_wait_timeout(limit_us)
        assert gdn.get_device_error() == gdn.GDN_DEVERR_TIMEOUT  # synchronises
        waited = time.perf_counter() - t0
        # the wait ends on its clock: not before the limit, and soon after it
        assert limit_us * 1e-6 <= waited < limit_us * 1e-6 + 2.0, f"{limit_us} us limit: waited {waited:.3f} s"
    assert gdn.get_device_error() == gdn.GDN_DEVERR_NONE      # read and cleared
    with pytest.raises(gdn.GDNError):
        gdn.selftest_wait_timeout(0)                          # refused on the host
    # the same context runs the next calls normally: a fused layer step of the
    # tiny fp32 workload against the oracle's layer
    s = I.TINY
    gen = I.Gen(90)
    prm = gen.params(s)
    w, w64 = pair(prm["w"], s.dtype)
    bias, bias64 = pair(prm["bias"], s.dtype)
    pool_np = gen.state_pool(s, s.num_slots)
    cp_dev, cp64 = pair(gen.conv_pool(s, s.num_slots), s.dtype)
    pool = gdn.GDNStatePool(s.num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                            tensor=torch.from_numpy(pool_np.copy()).cuda())
    cp = gdn.ConvStatePool(s.num_slots, s.channels, s.width, dtype=cp_dev.dtype, device="cuda", tensor=cp_dev)
    rs_np, ws_np = gen.slot_tables(s.rows, s.num_slots)
    xd, xr = {}, {}
    for k, v in gen.layer_inputs(s).items():
        xd[k], xr[k] = pair(v, s.dtype)
    out = gdn.gdn_layer_decode(xd["x"], cp, w, bias, t(prm["A_log"]), t(prm["dt_bias"]), xd["a"], xd["b"],
                               pool, ti(rs_np), ti(ws_np))
    torch.cuda.synchronize()
    p_ref = pool_np.astype(np.float64)
    o_ref, bad = orc.layer(xr["x"], cp64, w64, bias64, xr["a"], xr["b"], prm["A_log"], prm["dt_bias"], p_ref,
                           rs_np, ws_np, hk=s.hk, act_bf16=False)
    assert bad == 0
    assert_out_close(f64(out), o_ref, s.dtype)
    got = pool.tensor.cpu().numpy()
    assert (state_rel_err(got[ws_np], p_ref[ws_np]) <= STATE_TOL_ONE).all()
    assert np.array_equal(f64(cp.tensor), cp64)
    assert gdn.get_device_error() == gdn.GDN_DEVERR_NONE
