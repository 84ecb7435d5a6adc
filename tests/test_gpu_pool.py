"""GPU checks of the pools, commit, slot validation and the traffic probes,
through the C ABI.  Release and rollback zero both of a request's slots
(mstar PR #1139, "Tests"); the probes move a step's state bytes without
arithmetic (mstar PR #1139, "Numbers")."""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_decode_gb300 as G
from gated_deltanet_decode_gb300 import _lib
from gpu_helpers import ti

pytestmark = pytest.mark.gpu


def test_library_owned_pools(gdn):
    L = _lib.load()
    h = ctypes.c_void_p()
    assert L.gdn_state_pool_create(5, _lib.gdn_dims(2, 4, 32, 16), None, ctypes.byref(h)) == 0
    n = 5 * 4 * 16 * 32
    buf = torch.empty(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    assert rt.cudaMemcpy(buf.data_ptr(), L.gdn_pool_data(h), n * 4, 3) == 0   # device to device
    assert not buf.any()                                  # zero-filled
    assert L.gdn_state_pool_destroy(h) == 0
    c = ctypes.c_void_p()
    assert L.conv_state_pool_create(3, 64, 4, 1, None, ctypes.byref(c)) == 0
    assert L.conv_pool_num_slots(c) == 3
    assert L.conv_state_pool_destroy(c) == 0


def test_zero_slots(gdn):
    pool = G.GDNStatePool(6, 2, 2, 16, 16, device="cuda",
                          tensor=torch.randn(6, 2, 16, 16, device="cuda"))
    cp = G.ConvStatePool(6, 96, 4, dtype=torch.bfloat16, device="cuda",
                         tensor=torch.randn(6, 3, 96, device="cuda").bfloat16())
    before, cbefore = pool.tensor.clone(), cp.tensor.clone()
    slots = ti(np.array([2, 4]))
    pool.zero_slots(slots)
    cp.zero_slots(slots)
    torch.cuda.synchronize()
    for s in range(6):
        if s in (2, 4):
            assert not pool.tensor[s].any() and not cp.tensor[s].any()
        else:
            assert torch.equal(pool.tensor[s], before[s]) and torch.equal(cp.tensor[s], cbefore[s])
    pool.zero_slots(ti(np.array([7])))
    assert gdn.get_device_error() == G.GDN_DEVERR_BAD_SLOT


def test_commit_swaps_on_device(gdn):
    rs = ti(np.array([1, 0, 5, 7]))
    ws = ti(np.array([2, 0, 6, 8]))
    G.gdn_commit(rs, ws)
    assert rs.tolist() == [2, 0, 6, 8] and ws.tolist() == [1, 0, 5, 7]


def test_validate_slots(gdn):
    G.gdn_validate_slots(ti(np.array([1, 0, 3])), ti(np.array([2, 0, 4])), 5)
    G.gdn_validate_slots(ti(np.array([1, 0, 3])), None, 5, keep_in_place=True)
    bad_tables = [
        ([1, 2], [3, 3]),      # two rows write one slot
        ([1, 2], [2, 3]),      # row 0 writes what row 1 reads
        ([1, 9], [2, 3]),      # out of range
        ([1, 2], [1, 3]),      # twin write onto its own read slot
        ([1, 2], [0, 3]),      # real row writing the null slot
        ([1, 1], [2, 3]),      # two rows read one slot
    ]
    for rs, ws in bad_tables:
        with pytest.raises(G.GDNError) as e:
            G.gdn_validate_slots(ti(np.array(rs)), ti(np.array(ws)), 5)
        assert e.value.code == 5


def test_probes_move_the_bytes(gdn):
    torch.manual_seed(0)
    pool = G.GDNStatePool(9, 2, 4, 128, 128, device="cuda",
                          tensor=torch.randn(9, 4, 128, 128, device="cuda"))
    start = pool.tensor.clone()
    rs, ws = ti(np.array([1, 3, 0, 5])), ti(np.array([2, 4, 0, 6]))
    G.probe_traffic(pool, rs, ws, G.GDN_PROBE_TWIN)
    torch.cuda.synchronize()
    assert torch.equal(pool.tensor[[2, 4, 6]], start[[1, 3, 5]])
    assert torch.equal(pool.tensor[[0, 1, 3, 5, 7, 8]], start[[0, 1, 3, 5, 7, 8]])
    pool.tensor.copy_(start)
    G.probe_traffic(pool, rs, None, G.GDN_PROBE_INPLACE)
    G.probe_traffic(pool, rs, None, G.GDN_PROBE_READ)
    torch.cuda.synchronize()
    assert torch.equal(pool.tensor, start)
    G.probe_traffic(pool, rs, ws, G.GDN_PROBE_WRITE)
    torch.cuda.synchronize()
    assert not pool.tensor[[2, 4, 6]].any()
    assert torch.equal(pool.tensor[[0, 1, 3, 5, 7, 8]], start[[0, 1, 3, 5, 7, 8]])
    assert gdn.get_device_error() == 0


def test_copy_slots_snapshot_restore_and_bad_pairs(gdn, orc):
    """Snapshots and forks: copies are exact (the oracle's copy of the same
    pool), a snapshot taken before a decode step restores the state, bad
    pairs are skipped and set the device error word."""
    import numpy as np
    import torch
    from gated_deltanet_decode_gb300 import inputs as I
    s = I.QWEN_08B.with_(rows=8)
    gen = I.Gen(90)
    n_slots = 40
    pool_np = gen.state_pool(s, n_slots)
    pool = gdn.GDNStatePool(n_slots, s.hk, s.hv, s.dk, s.dv, device="cuda",
                            tensor=torch.from_numpy(pool_np.copy()).cuda())
    cp_np = gen.conv_pool(s, n_slots).astype(np.float32)
    cp = gdn.ConvStatePool(n_slots, s.channels, s.width, dtype=torch.float32, device="cuda",
                           tensor=torch.from_numpy(cp_np.copy()).cuda())
    src = np.array([3, 7, 0, 12], np.int32)
    dst = np.array([20, 21, 22, 23], np.int32)
    ts, td = (torch.from_numpy(a).cuda() for a in (src, dst))
    pool.copy_slots(ts, td)
    cp.copy_slots(ts, td)
    torch.cuda.synchronize()
    ref = pool_np.astype(np.float64)
    assert orc.copy_slots(ref, src, dst) == 0
    assert np.array_equal(pool.tensor.cpu().numpy().astype(np.float64), ref)
    ref_cp = cp_np.astype(np.float64)
    orc.copy_slots(ref_cp, src, dst)
    assert np.array_equal(cp.tensor.cpu().numpy().astype(np.float64), ref_cp)
    # snapshot, one decode step in place, restore: the state is back
    rows = np.array([3, 7, 12, 5], np.int32)
    snap = np.array([30, 31, 32, 33], np.int32)
    tr, tsn = (torch.from_numpy(a).cuda() for a in (rows, snap))
    before = pool.tensor.clone()
    pool.copy_slots(tr, tsn)
    inp = gen.step_inputs(s.with_(rows=4))
    q, k, v, a, b = (I.to_torch(inp[n], s.dtype, "cuda") for n in ("q", "k", "v", "a", "b"))
    prm = gen.params(s)
    gdn.gdn_decode_step(q, k, v, a, b, I.to_torch(prm["A_log"], "f32", "cuda"),
                        I.to_torch(prm["dt_bias"], "f32", "cuda"), pool, tr, None, keep_in_place=True)
    torch.cuda.synchronize()
    assert not torch.equal(pool.tensor[tr.long()], before[tr.long()])
    pool.copy_slots(tsn, tr)
    torch.cuda.synchronize()
    assert torch.equal(pool.tensor[tr.long()], before[tr.long()])
    assert gdn.get_device_error() == 0
    # bad pairs: a destination on the null slot, a source past the pool
    now = pool.tensor.clone()
    pool.copy_slots(torch.tensor([4, 99], dtype=torch.int32, device="cuda"),
                    torch.tensor([0, 25], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    assert torch.equal(pool.tensor, now)
