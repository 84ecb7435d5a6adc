"""gdn_layer_decode_noalloc through the C ABI: the same results as
gdn_layer_decode, bit for bit, on two calls in a row.

The entry point serves callers that may not allocate device memory (engines
that hand all of it to their own allocator up front); its two work counters
live in a fixed array in the library's module memory.  The shapes give the
kernel a dozen or more items a CTA, so the launch hands out the tail of its
work through those counters; the second call only gets every item if the
first left its scratch slot at zero.  Both ends of the array are used, the
second call must not change the device's free memory, and two calls on
neighbouring slots run at once on two streams (a slot whose counters
overlapped its neighbour's would lose items).
"""
import ctypes

import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import pair, t, ti

pytestmark = pytest.mark.gpu


def _call(L, name, c, xd, out, keep_in_place, extra=()):
    P = lambda v: ctypes.c_void_p(v.data_ptr()) if v is not None else None
    args = [P(xd["x"]), c["cp"].handle, P(c["w"]), P(c["bias"]), 1, P(c["A_log"]), P(c["dt_bias"]),
            P(xd["a"]), P(xd["b"]), c["pool"].handle, P(c["rs"]), None if keep_in_place else P(c["ws"]),
            P(out), xd["x"].shape[0], int(keep_in_place), *extra, c["dtype_code"],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]
    rc = getattr(L, name)(*args)
    assert rc == 0, L.gdn_last_error()


def _case(gdn, s, seed):
    gen = I.Gen(seed)
    num_slots = 2 * s.rows + 1
    prm = gen.params(s)
    c = {"dtype_code": gdn.GDN_BF16 if s.dtype == "bf16" else gdn.GDN_F32}
    c["w"], _ = pair(prm["w"], s.dtype)
    c["bias"], _ = pair(prm["bias"], s.dtype)
    c["A_log"], c["dt_bias"] = t(prm["A_log"]), t(prm["dt_bias"])
    c["pool0"] = torch.from_numpy(gen.state_pool(s, num_slots)).cuda()
    c["cp0"], _ = pair(gen.conv_pool(s, num_slots), s.dtype)
    c["pool"] = gdn.GDNStatePool(num_slots, s.hk, s.hv, s.dk, s.dv, device="cuda", tensor=c["pool0"].clone())
    c["cp"] = gdn.ConvStatePool(num_slots, s.channels, s.width, dtype=c["cp0"].dtype, device="cuda",
                                tensor=c["cp0"].clone())
    rs, ws = gen.slot_tables(s.rows, num_slots, 0.25)
    c["rs"], c["ws"] = ti(rs), ti(ws)
    xd = {k: pair(v, s.dtype)[0] for k, v in gen.layer_inputs(s).items()}
    return c, xd


def _reset(c):
    c["pool"].tensor.copy_(c["pool0"])
    c["cp"].tensor.copy_(c["cp0"])


@pytest.mark.parametrize("scratch_slot", [0, 63], ids=["slot0", "slot63"])
@pytest.mark.parametrize("shape", [I.QWEN_08B.with_(rows=256), I.QWEN_9B], ids=["0.8b-256rows", "9b-64rows"])
@pytest.mark.parametrize("keep_in_place", [False, True], ids=["twin", "in_place"])
def test_noalloc_equals_layer_decode_twice(gdn, shape, keep_in_place, scratch_slot):
    L = gdn.load()
    assert scratch_slot < gdn.GDN_NOALLOC_SCRATCH_SLOTS
    c, xd = _case(gdn, shape, seed=50)
    s = shape
    ref = torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device="cuda")
    _reset(c)
    _call(L, "gdn_layer_decode", c, xd, ref, keep_in_place)
    torch.cuda.synchronize()
    ref_pool, ref_cp = c["pool"].tensor.clone(), c["cp"].tensor.clone()
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    free = []
    for call in range(2):
        _reset(c)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _call(L, "gdn_layer_decode_noalloc", c, xd, outs[call], keep_in_place, extra=(scratch_slot,))
        torch.cuda.synchronize()
        free.append((free_before, torch.cuda.mem_get_info()[0]))  # read before any comparison allocates
        assert torch.equal(outs[call], ref), f"call {call}: outputs differ"
        assert torch.equal(c["pool"].tensor, ref_pool), f"call {call}: state pools differ"
        assert torch.equal(c["cp"].tensor, ref_cp), f"call {call}: conv pools differ"
    # the second call (the first did the one-time set-up) takes no device memory
    assert free[1][1] == free[1][0], f"free device memory went from {free[1][0]} to {free[1][1]} bytes"
    code = ctypes.c_int(-1)
    assert L.gdn_get_device_error(ctypes.byref(code), None) == 0
    assert code.value == 0


def test_noalloc_neighbouring_slots_at_once(gdn):
    """Two calls on two pools, on two streams at once, with scratch slots 0 and
    1 (then 62 and 63): each gives what gdn_layer_decode gives alone."""
    L = gdn.load()
    s = I.QWEN_08B.with_(rows=256)
    cases = [_case(gdn, s, seed=51 + i) for i in range(2)]
    refs = []
    for c, xd in cases:
        ref = torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device="cuda")
        _reset(c)
        _call(L, "gdn_layer_decode", c, xd, ref, False)
        torch.cuda.synchronize()
        refs.append((ref, c["pool"].tensor.clone(), c["cp"].tensor.clone()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for slots in ((0, 1), (62, 63), (1, 0)):
        outs = []
        for c, _ in cases:
            _reset(c)
        torch.cuda.synchronize()
        for (c, xd), st, slot in zip(cases, streams, slots):
            out = torch.full_like(refs[0][0], float("nan"))
            with torch.cuda.stream(st):
                _call(L, "gdn_layer_decode_noalloc", c, xd, out, False, extra=(slot,))
            outs.append(out)
        torch.cuda.synchronize()
        for i, ((c, _), out) in enumerate(zip(cases, outs)):
            assert torch.equal(out, refs[i][0]), f"slots {slots}, case {i}: outputs differ"
            assert torch.equal(c["pool"].tensor, refs[i][1]), f"slots {slots}, case {i}: state pools differ"
            assert torch.equal(c["cp"].tensor, refs[i][2]), f"slots {slots}, case {i}: conv pools differ"
    code = ctypes.c_int(-1)
    assert L.gdn_get_device_error(ctypes.byref(code), None) == 0
    assert code.value == 0
