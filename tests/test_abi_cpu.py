"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA.

No call here reaches the GPU: every call either fails validation or has
nothing to launch (rows == 0), and pools wrap fake (never dereferenced)
addresses.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn_decode.h")

EINVAL, ENOMEM, EUNSUPPORTED = 1, 2, 4
FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def L():
    from gated_deltanet_decode_gb300 import _lib
    return _lib.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(n for n in names if not n.startswith("_")))


def test_header_declarations_are_exported(L):
    from gated_deltanet_decode_gb300 import _lib
    declared = _declared()
    assert len(declared) >= 20
    assert sorted(_lib.EXPORTS) == declared
    for name in declared:
        assert hasattr(L, name), f"{name} not exported"
    assert L.gdn_abi_version() >= 1


def _dims(hk=2, hv=2, dk=16, dv=16):
    from gated_deltanet_decode_gb300._lib import gdn_dims
    return gdn_dims(hk, hv, dk, dv)


def _wrap(L, num_slots=9, **kw):
    h = ctypes.c_void_p()
    rc = L.gdn_state_pool_wrap(FAKE, num_slots, _dims(**kw), ctypes.byref(h))
    return rc, h


def test_state_pool_wrap_validation(L):
    h = ctypes.c_void_p()
    assert L.gdn_state_pool_wrap(None, 9, _dims(), ctypes.byref(h)) == EINVAL
    assert b"NULL" in L.gdn_last_error()
    assert L.gdn_state_pool_wrap(FAKE + 4, 9, _dims(), ctypes.byref(h)) == EINVAL  # misaligned
    assert _wrap(L, num_slots=0)[0] == EINVAL
    assert _wrap(L, hk=3, hv=4)[0] == EINVAL          # hv % hk != 0
    assert _wrap(L, dk=48)[0] == EUNSUPPORTED
    assert _wrap(L, dv=12)[0] == EUNSUPPORTED          # dv % 8
    rc, h = _wrap(L, num_slots=5, hk=2, hv=4, dk=64, dv=32)
    assert rc == 0 and h.value
    assert L.gdn_pool_num_slots(h) == 5
    d = L.gdn_pool_dims(h)
    assert (d.hk, d.hv, d.dk, d.dv) == (2, 4, 64, 32)
    assert L.gdn_pool_data(h) == FAKE
    assert L.gdn_state_pool_destroy(h) == 0            # wrapped: frees the handle only
    assert L.gdn_state_pool_destroy(None) == 0


def test_inplace_counters_size_and_attach(L):
    """One 32-bit counter per (slot, qk head), a slot's row padded to 16 bytes;
    attaching checks the pool, the alignment and the size and makes no CUDA
    call (a fake, never dereferenced address is accepted)."""
    n = L.gdn_pool_inplace_counter_bytes
    assert n(9, _dims(hk=2, hv=2)) == 9 * 4 * 4           # hk 2 -> 4 counters a slot
    assert n(129, _dims(hk=16, hv=16, dk=128, dv=128)) == 129 * 16 * 4
    assert n(3, _dims(hk=5, hv=10)) == 3 * 8 * 4           # hk 5 -> 8
    assert n(0, _dims()) == 0 and n(9, _dims(dk=48)) == 0  # bad arguments
    rc, h = _wrap(L, num_slots=9, hk=2, hv=2)
    assert rc == 0
    need = n(9, _dims(hk=2, hv=2))
    a = L.gdn_pool_attach_inplace_counters
    assert a(None, FAKE, need) == EINVAL
    assert a(h, FAKE + 4, need) == EINVAL                    # misaligned
    assert b"aligned" in L.gdn_last_error()
    assert a(h, FAKE, need - 1) == EINVAL                    # short
    assert a(h, FAKE, need) == 0
    assert a(h, FAKE + 4096, need + 64) == 0                 # replaced
    assert a(h, None, 0) == 0                                # detached
    assert L.gdn_state_pool_destroy(h) == 0


def test_state_pool_handle_limit(L):
    """Every state pool handle holds one pair of work counters from a fixed
    table; handles beyond GDN_MAX_POOLS fail with GDN_ENOMEM and destroyed
    handles give their pair back."""
    from gated_deltanet_decode_gb300._lib import GDN_MAX_POOLS
    handles = []
    try:
        while len(handles) <= GDN_MAX_POOLS:
            rc, h = _wrap(L)
            if rc:
                break
            handles.append(h)
        assert rc == ENOMEM and b"state pools" in L.gdn_last_error()
        assert GDN_MAX_POOLS - 64 <= len(handles) <= GDN_MAX_POOLS
        assert L.gdn_state_pool_destroy(handles.pop()) == 0
        rc, h = _wrap(L)
        assert rc == 0
        handles.append(h)
    finally:
        for h in handles:
            assert L.gdn_state_pool_destroy(h) == 0
    rc, h = _wrap(L)
    assert rc == 0 and L.gdn_state_pool_destroy(h) == 0


def test_conv_pool_wrap_validation(L):
    h = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 5, 0, ctypes.byref(h)) == EUNSUPPORTED  # width
    assert L.conv_state_pool_wrap(FAKE, 9, 100, 4, 0, ctypes.byref(h)) == EINVAL       # channels % 8
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 4, 7, ctypes.byref(h)) == EINVAL        # dtype
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 4, 1, ctypes.byref(h)) == 0
    assert L.conv_pool_num_slots(h) == 9 and L.conv_pool_data(h) == FAKE
    assert L.conv_state_pool_destroy(h) == 0


def test_step_argument_checks(L):
    rc, pool = _wrap(L)
    assert rc == 0
    P = FAKE
    args = dict(q=P, k=P, v=P, a=P, b=P, A_log=P, dt_bias=P, pool=pool, rs=P, ws=P, out=P,
                rows=4, heads=2, inplace=0, dtype=0)

    def call(**over):
        x = dict(args, **over)
        return L.gdn_decode_step(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                                 x["pool"], x["rs"], x["ws"], x["out"], x["rows"], x["heads"],
                                 x["inplace"], x["dtype"], None)

    assert call(pool=None) == EINVAL
    assert call(rows=-1) == EINVAL
    assert call(dtype=5) == EINVAL
    assert call(heads=3) == EINVAL and b"heads" in L.gdn_last_error()
    assert call(q=None) == EINVAL
    assert call(ws=None) == EINVAL                      # twin needs a write table
    assert call(a=None) == EINVAL
    assert call(q=P + 8) == EINVAL and b"aligned" in L.gdn_last_error()
    assert call(rows=0) == 0                            # nothing to launch
    assert call(rows=0, ws=None, inplace=1) == 0
    L.gdn_state_pool_destroy(pool)


def test_layer_and_conv_argument_checks(L):
    rc, pool = _wrap(L, hk=2, hv=2, dk=16, dv=16)
    cp = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 4, 0, ctypes.byref(cp)) == 0
    bad_cp = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 9, 88, 4, 0, ctypes.byref(bad_cp)) == 0
    P = FAKE

    def layer(cpool, rows=4, inplace=0, dtype=0, x=P, w=P, pool_=pool):
        return L.gdn_layer_decode(x, cpool, w, None, 1, P, P, P, P, pool_, P, P, P, rows, inplace,
                                  dtype, None)

    assert layer(None) == EINVAL
    assert layer(bad_cp) == EINVAL and b"channels" in L.gdn_last_error()
    assert layer(cp, dtype=1) == EINVAL                 # dtype differs from the conv pool's
    assert layer(cp, x=None) == EINVAL
    assert layer(cp, rows=0) == 0
    assert layer(cp, x=P + 8) == EINVAL                 # bulk-copy sources must be 16-byte aligned
    assert layer(cp, w=P + 4) == EINVAL
    # a wide qk group (16 value heads of dv = 512 sharing one qk head) is accepted
    rc, big = _wrap(L, num_slots=3, hk=1, hv=16, dk=16, dv=512)
    assert rc == 0
    cbig = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 3, 2 * 16 + 16 * 512, 4, 0, ctypes.byref(cbig)) == 0
    assert layer(cbig, rows=0, inplace=1, pool_=big) == 0

    def conv(stride=96, x=P, out=P, rows=2, dtype=0):
        return L.causal_conv1d_decode(x, stride, cp, P, None, P, None, 1, out, rows, dtype, None)

    assert conv(stride=90) == EINVAL                    # shorter than a row
    assert conv(stride=100) == EINVAL                   # not a multiple of 8
    assert conv(x=P + 8) == EINVAL                      # misaligned
    assert conv(out=None) == EINVAL
    assert conv(dtype=1) == EINVAL
    assert conv(rows=0) == 0
    # layer + commit in one launch: twin only, so the write table is required
    def layer_c(cpool, rows=4, ws=P):
        return L.gdn_layer_decode_commit(P, cpool, P, None, 1, P, P, P, P, pool, P, ws, P, rows, 0, None)

    assert layer_c(cp, ws=None) == EINVAL
    assert layer_c(bad_cp) == EINVAL and b"channels" in L.gdn_last_error()
    assert layer_c(cp, rows=0) == 0
    # a bucket's decode half: a device row count, and commit only with twin slots
    def layer_b(n=P, inplace=0, commit=0, rows=4):
        return L.gdn_layer_decode_bucket(P, cp, P, None, 1, P, P, P, P, pool, P, P, P, rows, n, inplace,
                                         commit, 0, None)

    assert layer_b(n=None) == EINVAL and b"n_decode" in L.gdn_last_error()
    assert layer_b(inplace=1, commit=1) == EINVAL
    assert layer_b(rows=0) == 0
    # the no-allocation variant: same checks, plus its scratch slot
    from gated_deltanet_decode_gb300._lib import GDN_NOALLOC_SCRATCH_SLOTS

    def layer_na(cpool, slot, rows=4, x=P):
        return L.gdn_layer_decode_noalloc(x, cpool, P, None, 1, P, P, P, P, pool, P, P, P, rows, 0, slot,
                                          0, None)

    assert layer_na(cp, GDN_NOALLOC_SCRATCH_SLOTS) == EINVAL and b"scratch" in L.gdn_last_error()
    assert layer_na(cp, -1) == EINVAL
    assert layer_na(bad_cp, 0) == EINVAL and b"channels" in L.gdn_last_error()
    assert layer_na(cp, 0, x=P + 8) == EINVAL
    assert layer_na(cp, GDN_NOALLOC_SCRATCH_SLOTS - 1, rows=0) == 0
    for h in (cp, bad_cp, cbig):
        L.conv_state_pool_destroy(h)
    L.gdn_state_pool_destroy(pool)
    L.gdn_state_pool_destroy(big)


def test_small_entry_points_checks(L):
    assert L.gdn_commit(None, None, 0, None) == 0
    assert L.gdn_commit(None, FAKE, 3, None) == EINVAL
    assert L.gdn_commit(FAKE, FAKE, -1, None) == EINVAL
    assert L.gdn_validate_slots(FAKE, None, 0, 9, 0, None) == 0
    assert L.gdn_validate_slots(FAKE, None, 2, 9, 0, None) == EINVAL
    assert L.gdn_get_device_error(None, None) == EINVAL
    rc, pool = _wrap(L)
    assert L.gdn_probe_traffic(pool, FAKE, FAKE, 4, 9, None, None) == EINVAL
    assert L.gdn_probe_traffic(pool, FAKE, None, 4, 0, None, None) == EINVAL
    assert L.gdn_probe_traffic(pool, FAKE, FAKE, 0, 0, None, None) == 0
    assert L.gdn_pool_zero_slots(pool, None, 0, None) == 0
    assert L.gdn_pool_zero_slots(pool, None, 2, None) == EINVAL
    assert L.gdn_pool_zero_slots(None, FAKE, 2, None) == EINVAL
    L.gdn_state_pool_destroy(pool)


def test_prefill_argument_checks(L):
    """gdn_prefill, gdn_verify and causal_conv1d_prefill reject bad arguments
    on the host and return at once when there is nothing to launch."""
    rc, pool = _wrap(L, hk=2, hv=2, dk=16, dv=16)
    assert rc == 0
    cp = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 4, 0, ctypes.byref(cp)) == 0
    P = FAKE

    def prefill(nseq=2, T=5, pool_=pool, ws=P, inplace=0, dtype=0, q=P):
        return L.gdn_prefill(q, P, P, P, P, P, P, pool_, P, P, ws, P, nseq, T, inplace, dtype, None)

    assert prefill(pool_=None) == EINVAL
    assert prefill(nseq=-1) == EINVAL
    assert prefill(T=-1) == EINVAL
    assert prefill(dtype=3) == EINVAL
    assert prefill(ws=None) == EINVAL and b"write_slot" in L.gdn_last_error()
    assert prefill(q=P + 8) == EINVAL and b"aligned" in L.gdn_last_error()
    assert prefill(nseq=0) == 0
    assert prefill(nseq=0, ws=None, inplace=1) == 0

    def verify(nseq=2, T=5, ts=P):
        return L.gdn_verify(P, P, P, P, P, P, P, pool, P, P, ts, P, nseq, T, 0, None)

    assert verify(ts=None) == EINVAL and b"token_slot" in L.gdn_last_error()
    assert verify(T=0, ts=None) == 0      # no token, no state to keep
    assert verify(nseq=0) == 0

    def conv(nseq=2, T=5, cpool=cp, x=P, dtype=0):
        return L.causal_conv1d_prefill(x, cpool, P, P, None, None, P, None, 1, P, nseq, T, dtype, None)

    assert conv(cpool=None) == EINVAL
    assert conv(dtype=1) == EINVAL and b"dtype" in L.gdn_last_error()
    assert conv(x=P + 4) == EINVAL
    assert conv(x=None) == EINVAL
    assert conv(nseq=0) == 0
    L.conv_state_pool_destroy(cp)
    L.gdn_state_pool_destroy(pool)


def test_prefill_chunked_argument_checks(L):
    """gdn_prefill_chunked: built for dk = dv = 128 only (unsupported shapes
    are refused before anything else); bf16 activations need a 128-byte
    aligned workspace of gdn_prefill_chunked_workspace_bytes; otherwise
    gdn_prefill's checks."""
    import ctypes
    P = FAKE
    rc, small = _wrap(L, hk=2, hv=2, dk=16, dv=16)
    assert rc == 0
    rc, pool = _wrap(L, hk=2, hv=4, dk=128, dv=128)
    assert rc == 0
    need = L.gdn_prefill_chunked_workspace_bytes(2, 5, 4)
    # one unit per chunk start, ceil(T / 64) + nseq units a value head, whole 128-byte blocks
    assert need > 0 and need % (3 * 4) == 0 and (need // 12) % 128 == 0
    assert L.gdn_prefill_chunked_workspace_bytes(2, 640, 4) == need // 3 * (10 + 2)
    assert L.gdn_prefill_chunked_workspace_bytes(0, 5, 4) == 0

    def chunked(nseq=2, T=5, pool_=pool, ws=P, inplace=0, dtype=1, q=P, work=P, work_bytes=None):
        wb = need if work_bytes is None else work_bytes
        return L.gdn_prefill_chunked(q, P, P, P, P, P, P, pool_, P, P, ws, P, nseq, T, inplace, work,
                                     ctypes.c_size_t(wb), dtype, None)

    assert chunked(pool_=small) == EUNSUPPORTED and b"128" in L.gdn_last_error()
    assert chunked(pool_=None) == EINVAL
    assert chunked(nseq=-1) == EINVAL
    assert chunked(dtype=3) == EINVAL
    assert chunked(ws=None) == EINVAL and b"write_slot" in L.gdn_last_error()
    assert chunked(work=None) == EINVAL and b"workspace" in L.gdn_last_error()
    assert chunked(work_bytes=need - 16) == EINVAL and b"workspace" in L.gdn_last_error()
    assert chunked(work=P + 64) == EINVAL and b"128-byte" in L.gdn_last_error()
    assert chunked(q=P + 8) == EINVAL and b"aligned" in L.gdn_last_error()
    assert chunked(nseq=0) == 0
    assert chunked(nseq=0, ws=None, inplace=1, work=None, work_bytes=0) == 0
    L.gdn_state_pool_destroy(small)
    L.gdn_state_pool_destroy(pool)


def test_copy_slots_argument_checks(L):
    rc, pool = _wrap(L)
    assert rc == 0
    cp = ctypes.c_void_p()
    assert L.conv_state_pool_wrap(FAKE, 9, 96, 4, 0, ctypes.byref(cp)) == 0
    assert L.gdn_pool_copy_slots(None, FAKE, FAKE, 1, None) == EINVAL
    assert L.gdn_pool_copy_slots(pool, FAKE, FAKE, -1, None) == EINVAL
    assert L.gdn_pool_copy_slots(pool, None, FAKE, 1, None) == EINVAL
    assert L.gdn_pool_copy_slots(pool, None, None, 0, None) == 0
    assert L.conv_pool_copy_slots(None, FAKE, FAKE, 1, None) == EINVAL
    assert L.conv_pool_copy_slots(cp, FAKE, None, 2, None) == EINVAL
    assert L.conv_pool_copy_slots(cp, None, None, 0, None) == 0
    L.conv_state_pool_destroy(cp)
    L.gdn_state_pool_destroy(pool)


def test_binding_accepts_only_device_or_pinned_pointers():
    """The binding hands the library a device pointer, or a page-locked host
    pointer where the call allows activations in host memory; pageable host
    memory is refused on the host."""
    import torch
    from gated_deltanet_decode_gb300 import _ptr
    with pytest.raises(ValueError, match="pinned host memory"):
        _ptr(torch.zeros(4), "x", host_ok=True)
    with pytest.raises(ValueError, match="must be a CUDA tensor$"):
        _ptr(torch.zeros(4), "x")
    assert _ptr(None, "x", host_ok=True) is None


def test_prefill_chunked_workspace_holds_every_chunk(L):
    """The chunked prefill's workspace: sequence s's chunk j (64 tokens a
    chunk) lives in unit cu_seqlens[s] // 64 + s + j of each value head.  For
    random nondecreasing cu_seqlens the units of all chunks are distinct and
    lie inside the size gdn_prefill_chunked_workspace_bytes reports."""
    import numpy as np
    block = L.gdn_prefill_chunked_workspace_bytes(1, 1, 1) // 2  # one sequence of one token: 2 units
    assert block > 0 and block % 128 == 0
    rng = np.random.default_rng(5)
    for _ in range(200):
        nseq = int(rng.integers(1, 12))
        lens = rng.integers(0, 300, size=nseq)
        lens[rng.random(nseq) < 0.2] = 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        T = int(cu[-1])
        hv = int(rng.integers(1, 5))
        units = L.gdn_prefill_chunked_workspace_bytes(nseq, T, hv) // (hv * block)
        seen = set()
        for s in range(nseq):
            for j in range((int(lens[s]) + 63) // 64):
                u = int(cu[s]) // 64 + s + j
                assert u not in seen and 0 <= u < units, (cu.tolist(), s, j, u, units)
                seen.add(u)
