"""GB300 (sm_103a) Gated DeltaNet decode: Python binding of the C ABI.

The functions here only marshal torch tensors (device pointers, sizes, the
current CUDA stream) into calls of ``libgdn_decode.so``; every step of the
decode path runs in the library's CUDA kernels.  The names follow the C ABI
(``include/gdn_decode.h``):

  GDNStatePool / ConvStatePool   slot-indexed pools (slot 0 = null slot)
  causal_conv1d_decode           depthwise causal conv, one token a row
  gdn_decode_step                gated delta rule per row and value head
  gdn_layer_decode               both in one kernel
  gdn_commit                     twin-slot commit (swap read/write slots)

The operation is the decode step of "mstar PR #1139" ("Why": the GDN rule is
the recurrent state update of one token a row; "What changed": twin slots,
the decode-only conv), with padding on the null slot of "mstar PR #1127".
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import (GDN_BF16, GDN_DEVERR_BAD_SLOT, GDN_DEVERR_NONE, GDN_DEVERR_TIMEOUT, GDN_F32,
                   GDN_NOALLOC_SCRATCH_SLOTS,
                   GDN_PROBE_INPLACE, GDN_PROBE_READ, GDN_PROBE_TWIN, GDN_PROBE_WRITE, gdn_dims)

__all__ = [
    "GDNError", "load", "lib_path", "GDNStatePool", "ConvStatePool", "causal_conv1d_decode",
    "gdn_decode_step", "gdn_layer_decode", "gdn_layer_decode_noalloc", "gdn_commit", "gdn_validate_slots",
    "gdn_prefill", "gdn_prefill_chunked", "gdn_prefill_chunked_workspace_bytes", "gdn_verify", "causal_conv1d_prefill", "gdn_layer_decode_bucket",
    "get_device_error", "selftest_wait_timeout", "probe_traffic", "GDN_F32", "GDN_BF16", "GDN_DEVERR_NONE",
    "GDN_DEVERR_BAD_SLOT", "GDN_DEVERR_TIMEOUT", "GDN_PROBE_TWIN", "GDN_PROBE_INPLACE", "GDN_PROBE_READ",
    "GDN_PROBE_WRITE", "GDN_NOALLOC_SCRATCH_SLOTS",
]


class GDNError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[gdn status {code}] {msg}")
        self.code = code


def load():
    return _lib.load()


def lib_path() -> str:
    return _lib.lib_path()


def _check(rc: int):
    if rc != 0:
        msg = _lib.load().gdn_last_error().decode(errors="replace")
        raise GDNError(rc, msg)


_DTYPES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}


def _dtype_code(t: torch.dtype) -> int:
    if t not in _DTYPES:
        raise TypeError(f"activation dtype must be float32 or bfloat16, got {t}")
    return _DTYPES[t]


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t: Optional[torch.Tensor], what: str, dtype=None, device=None, contiguous=True, host_ok=False):
    """Device pointer of a tensor.  With host_ok, a page-locked (pinned) host
    tensor is accepted too: under unified addressing its pointer is valid on
    the device, and the kernels read or write it across the host link."""
    if t is None:
        return None
    if not t.is_cuda:
        if host_ok and t.is_pinned():
            if dtype is not None and t.dtype != dtype:
                raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
            if contiguous and not t.is_contiguous():
                raise ValueError(f"{what} must be contiguous")
            return t.data_ptr()
        raise ValueError(f"{what} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if device is not None and t.device != device:
        raise ValueError(f"{what} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _numel(t: torch.Tensor, n: int, what: str):
    if t.numel() != n:
        raise ValueError(f"{what} has {t.numel()} elements, expected {n}")


class GDNStatePool:
    """Recurrent state pool [num_slots][hv][dv][dk] fp32 in torch-owned memory.

    The library wraps the tensor (it never frees it).  Slot 0 is the null slot.
    The pool also holds its in-place counters (`inplace_counters`, zeroed
    int32 device memory the library's in-place layer launches schedule with);
    `inplace_counters=False` leaves them out, and in-place launches then give
    each CTA whole qk heads.
    """

    def __init__(self, num_slots: int, hk: int, hv: int, dk: int, dv: int, device=None,
                 tensor: Optional[torch.Tensor] = None, inplace_counters: bool = True):
        L = _lib.load()
        device = torch.device(device if device is not None else "cuda")
        if tensor is None:
            tensor = torch.zeros((num_slots, hv, dv, dk), dtype=torch.float32, device=device)
        if tuple(tensor.shape) != (num_slots, hv, dv, dk) or tensor.dtype != torch.float32:
            raise ValueError("state tensor must be float32 [num_slots][hv][dv][dk]")
        self.tensor = tensor
        self.num_slots, self.hk, self.hv, self.dk, self.dv = num_slots, hk, hv, dk, dv
        h = ctypes.c_void_p()
        _check(L.gdn_state_pool_wrap(_ptr(tensor, "state"), num_slots, gdn_dims(hk, hv, dk, dv),
                                     ctypes.byref(h)))
        self._h = h
        self.counters = None
        if inplace_counters:
            nbytes = L.gdn_pool_inplace_counter_bytes(num_slots, gdn_dims(hk, hv, dk, dv))
            self.counters = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=tensor.device)
            _check(L.gdn_pool_attach_inplace_counters(h, _ptr(self.counters, "in-place counters"),
                                                      self.counters.numel() * 4))

    @property
    def handle(self):
        return self._h

    def zero_slots(self, slots: torch.Tensor):
        _check(_lib.load().gdn_pool_zero_slots(self._h, _ptr(slots, "slots", torch.int32),
                                               slots.numel(), _stream(self.tensor.device)))

    def copy_slots(self, src: torch.Tensor, dst: torch.Tensor):
        """Slot dst[i] receives a copy of slot src[i] (snapshots, forks)."""
        _numel(dst, src.numel(), "dst")
        _check(_lib.load().gdn_pool_copy_slots(self._h, _ptr(src, "src", torch.int32),
                                               _ptr(dst, "dst", torch.int32), src.numel(),
                                               _stream(self.tensor.device)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _lib.load().gdn_state_pool_destroy(h)
            except Exception:
                pass
            self._h = None


class ConvStatePool:
    """Conv window pool [num_slots][width-1][channels] in the activation dtype."""

    def __init__(self, num_slots: int, channels: int, width: int, dtype=torch.bfloat16, device=None,
                 tensor: Optional[torch.Tensor] = None):
        L = _lib.load()
        device = torch.device(device if device is not None else "cuda")
        if tensor is None:
            tensor = torch.zeros((num_slots, width - 1, channels), dtype=dtype, device=device)
        if tuple(tensor.shape) != (num_slots, width - 1, channels) or tensor.dtype != dtype:
            raise ValueError("conv tensor must be [num_slots][width-1][channels] of the given dtype")
        self.tensor = tensor
        self.num_slots, self.channels, self.width, self.dtype = num_slots, channels, width, dtype
        h = ctypes.c_void_p()
        _check(L.conv_state_pool_wrap(_ptr(tensor, "conv state"), num_slots, channels, width,
                                      _dtype_code(dtype), ctypes.byref(h)))
        self._h = h

    @property
    def handle(self):
        return self._h

    def zero_slots(self, slots: torch.Tensor):
        _check(_lib.load().conv_pool_zero_slots(self._h, _ptr(slots, "slots", torch.int32),
                                                slots.numel(), _stream(self.tensor.device)))

    def copy_slots(self, src: torch.Tensor, dst: torch.Tensor):
        """Slot dst[i] receives a copy of slot src[i] (snapshots, forks)."""
        _numel(dst, src.numel(), "dst")
        _check(_lib.load().conv_pool_copy_slots(self._h, _ptr(src, "src", torch.int32),
                                                _ptr(dst, "dst", torch.int32), src.numel(),
                                                _stream(self.tensor.device)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                _lib.load().conv_state_pool_destroy(h)
            except Exception:
                pass
            self._h = None


def causal_conv1d_decode(x: torch.Tensor, conv_pool: ConvStatePool, slot_idx: torch.Tensor,
                         w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                         out: Optional[torch.Tensor] = None, write_slot: Optional[torch.Tensor] = None,
                         silu: bool = True) -> torch.Tensor:
    """Conv state update for one token a row. x: [rows][C] (row stride allowed)."""
    rows, C = x.shape
    dt = conv_pool.dtype
    dev = conv_pool.tensor.device
    if x.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    if out is None:
        out = torch.empty((rows, C), dtype=dt, device=dev)
    _numel(slot_idx, rows, "slot_idx")
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    _check(_lib.load().causal_conv1d_decode(
        _ptr(x, "x", dt, dev, contiguous=False), x.stride(0), conv_pool.handle,
        _ptr(slot_idx, "slot_idx", torch.int32, dev), _ptr(write_slot, "write_slot", torch.int32, dev),
        _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev), int(bool(silu)),
        _ptr(out, "out", dt, dev, host_ok=True), rows, _dtype_code(dt), _stream(dev)))
    return out


def gdn_decode_step(q, k, v, a, b, A_log, dt_bias, pool: GDNStatePool, read_slot, write_slot=None,
                    out: Optional[torch.Tensor] = None, keep_in_place: bool = False) -> torch.Tensor:
    """Gated delta rule for one token a row. q,k: [rows][hk][dk]; v: [rows][hv][dv]; a,b: [rows][hv].
    q, k, v, a, b and out may be pinned host tensors (read and written across the host link)."""
    rows = q.shape[0]
    dt = q.dtype
    dev = pool.tensor.device
    _numel(q, rows * pool.hk * pool.dk, "q")
    _numel(k, rows * pool.hk * pool.dk, "k")
    _numel(v, rows * pool.hv * pool.dv, "v")
    _numel(a, rows * pool.hv, "a")
    _numel(b, rows * pool.hv, "b")
    _numel(A_log, pool.hv, "A_log")
    _numel(dt_bias, pool.hv, "dt_bias")
    _numel(read_slot, rows, "read_slot")
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    if out is None:
        out = torch.empty((rows, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, rows * pool.hv * pool.dv, "out")
    _check(_lib.load().gdn_decode_step(
        _ptr(q, "q", dt, dev, host_ok=True), _ptr(k, "k", dt, dev, host_ok=True),
        _ptr(v, "v", dt, dev, host_ok=True), _ptr(a, "a", dt, dev, host_ok=True),
        _ptr(b, "b", dt, dev, host_ok=True), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), pool.handle,
        _ptr(read_slot, "read_slot", torch.int32, dev), _ptr(write_slot, "write_slot", torch.int32, dev),
        _ptr(out, "out", dt, dev, host_ok=True), rows, pool.hv, int(bool(keep_in_place)), _dtype_code(dt),
        _stream(dev)))
    return out


def _prefill_checks(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot):
    T = q.shape[0]
    nseq = cu_seqlens.numel() - 1
    if nseq < 0:
        raise ValueError("cu_seqlens needs nseq + 1 entries")
    _numel(q, T * pool.hk * pool.dk, "q")
    _numel(k, T * pool.hk * pool.dk, "k")
    _numel(v, T * pool.hv * pool.dv, "v")
    _numel(a, T * pool.hv, "a")
    _numel(b, T * pool.hv, "b")
    _numel(A_log, pool.hv, "A_log")
    _numel(dt_bias, pool.hv, "dt_bias")
    _numel(read_slot, nseq, "read_slot")
    return T, nseq


def gdn_prefill(q, k, v, a, b, A_log, dt_bias, pool: GDNStatePool, cu_seqlens, read_slot, write_slot=None,
                out: Optional[torch.Tensor] = None, keep_in_place: bool = False) -> torch.Tensor:
    """The rule over many tokens a sequence (packed, token-major: q,k [T][hk][dk],
    v [T][hv][dv], a,b [T][hv]; sequence r is tokens cu_seqlens[r]..cu_seqlens[r+1]).
    The final state goes to write_slot (twin) or back to read_slot (in place)."""
    T, nseq = _prefill_checks(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot)
    dt, dev = q.dtype, pool.tensor.device
    if write_slot is not None:
        _numel(write_slot, nseq, "write_slot")
    if out is None:
        out = torch.empty((T, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, T * pool.hv * pool.dv, "out")
    _check(_lib.load().gdn_prefill(
        _ptr(q, "q", dt, dev, host_ok=True), _ptr(k, "k", dt, dev, host_ok=True), _ptr(v, "v", dt, dev, host_ok=True), _ptr(a, "a", dt, dev, host_ok=True),
        _ptr(b, "b", dt, dev, host_ok=True), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), pool.handle,
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, dev), _ptr(read_slot, "read_slot", torch.int32, dev),
        _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), nseq, T,
        int(bool(keep_in_place)), _dtype_code(dt), _stream(dev)))
    return out


def gdn_prefill_chunked_workspace_bytes(nseq: int, total_tokens: int, hv: int) -> int:
    """Bytes of the device workspace gdn_prefill_chunked needs for bf16 activations."""
    return int(_lib.load().gdn_prefill_chunked_workspace_bytes(int(nseq), int(total_tokens), int(hv)))


def gdn_prefill_chunked(q, k, v, a, b, A_log, dt_bias, pool: GDNStatePool, cu_seqlens, read_slot,
                        write_slot=None, out: Optional[torch.Tensor] = None,
                        keep_in_place: bool = False, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """gdn_prefill's operation in chunks of 64 tokens on the tensor cores
    (dk = dv = 128): the same arguments and slot semantics, results within
    about 1e-5 relative of gdn_prefill instead of bit-identical.  Its
    activations must be device memory.  bf16 activations use a device
    workspace (a uint8 tensor of at least gdn_prefill_chunked_workspace_bytes;
    allocated here when none is given)."""
    T, nseq = _prefill_checks(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot)
    dt, dev = q.dtype, pool.tensor.device
    if write_slot is not None:
        _numel(write_slot, nseq, "write_slot")
    if out is None:
        out = torch.empty((T, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, T * pool.hv * pool.dv, "out")
    need = gdn_prefill_chunked_workspace_bytes(nseq, T, pool.hv) if dt == torch.bfloat16 else 0
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the pool's device")
        ws_ptr, ws_bytes = ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()
    _check(_lib.load().gdn_prefill_chunked(
        _ptr(q, "q", dt, dev), _ptr(k, "k", dt, dev),
        _ptr(v, "v", dt, dev), _ptr(a, "a", dt, dev),
        _ptr(b, "b", dt, dev), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), pool.handle,
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, dev), _ptr(read_slot, "read_slot", torch.int32, dev),
        _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev), nseq, T,
        int(bool(keep_in_place)), ws_ptr, ctypes.c_size_t(ws_bytes), _dtype_code(dt), _stream(dev)))
    return out


def gdn_verify(q, k, v, a, b, A_log, dt_bias, pool: GDNStatePool, cu_seqlens, read_slot, token_slot,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """As gdn_prefill, but the state after token t goes to token_slot[t] (a
    state a token) and the read slot is left alone."""
    T, nseq = _prefill_checks(q, k, v, a, b, A_log, dt_bias, pool, cu_seqlens, read_slot)
    dt, dev = q.dtype, pool.tensor.device
    _numel(token_slot, T, "token_slot")
    if out is None:
        out = torch.empty((T, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, T * pool.hv * pool.dv, "out")
    _check(_lib.load().gdn_verify(
        _ptr(q, "q", dt, dev, host_ok=True), _ptr(k, "k", dt, dev, host_ok=True), _ptr(v, "v", dt, dev, host_ok=True), _ptr(a, "a", dt, dev, host_ok=True),
        _ptr(b, "b", dt, dev, host_ok=True), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), pool.handle,
        _ptr(cu_seqlens, "cu_seqlens", torch.int32, dev), _ptr(read_slot, "read_slot", torch.int32, dev),
        _ptr(token_slot, "token_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), nseq, T,
        _dtype_code(dt), _stream(dev)))
    return out


def causal_conv1d_prefill(x, conv_pool: ConvStatePool, cu_seqlens, read_slot, w, bias, write_slot=None,
                          token_slot=None, out: Optional[torch.Tensor] = None, silu: bool = True) -> torch.Tensor:
    """The conv over many tokens a sequence: x [T][C] packed token-major; the
    window continues from read_slot and ends in write_slot (None: in place), or
    with token_slot [T] the window after each token goes to its slot."""
    T = x.shape[0]
    C = conv_pool.channels
    nseq = cu_seqlens.numel() - 1
    dt, dev = x.dtype, conv_pool.tensor.device
    _numel(x, T * C, "x")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    _numel(read_slot, nseq, "read_slot")
    if write_slot is not None:
        _numel(write_slot, nseq, "write_slot")
    if token_slot is not None:
        _numel(token_slot, T, "token_slot")
    if out is None:
        out = torch.empty((T, C), dtype=dt, device=dev)
    _numel(out, T * C, "out")
    _check(_lib.load().causal_conv1d_prefill(
        _ptr(x, "x", dt, dev, host_ok=True), conv_pool.handle, _ptr(cu_seqlens, "cu_seqlens", torch.int32, dev),
        _ptr(read_slot, "read_slot", torch.int32, dev), _ptr(write_slot, "write_slot", torch.int32, dev),
        _ptr(token_slot, "token_slot", torch.int32, dev), _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev),
        int(bool(silu)), _ptr(out, "out", dt, dev, host_ok=True), nseq, T, _dtype_code(dt), _stream(dev)))
    return out


def gdn_layer_decode(x, conv_pool: ConvStatePool, w, bias, A_log, dt_bias, a, b, pool: GDNStatePool,
                     read_slot, write_slot=None, out: Optional[torch.Tensor] = None,
                     keep_in_place: bool = False, silu: bool = True, commit: bool = False) -> torch.Tensor:
    """Fused conv + gated delta rule. x: [rows][2*hk*dk + hv*dv] packed q|k|v.
    With commit (twin only) the slot tables are swapped in the same launch
    (gdn_layer_decode_commit)."""
    if commit and (keep_in_place or write_slot is None):
        raise ValueError("commit needs twin slots (a write_slot table, keep_in_place False)")
    rows = x.shape[0]
    dt = x.dtype
    dev = pool.tensor.device
    C = 2 * pool.hk * pool.dk + pool.hv * pool.dv
    _numel(x, rows * C, "x")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    _numel(a, rows * pool.hv, "a")
    _numel(b, rows * pool.hv, "b")
    _numel(A_log, pool.hv, "A_log")
    _numel(dt_bias, pool.hv, "dt_bias")
    _numel(read_slot, rows, "read_slot")
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    if out is None:
        out = torch.empty((rows, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, rows * pool.hv * pool.dv, "out")
    args = (_ptr(x, "x", dt, dev, host_ok=True), conv_pool.handle, _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev),
            int(bool(silu)), _ptr(A_log, "A_log", torch.float32, dev),
            _ptr(dt_bias, "dt_bias", torch.float32, dev), _ptr(a, "a", dt, dev, host_ok=True), _ptr(b, "b", dt, dev, host_ok=True),
            pool.handle, _ptr(read_slot, "read_slot", torch.int32, dev),
            _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), rows)
    if commit:
        _check(_lib.load().gdn_layer_decode_commit(*args, _dtype_code(dt), _stream(dev)))
    else:
        _check(_lib.load().gdn_layer_decode(*args, int(bool(keep_in_place)), _dtype_code(dt), _stream(dev)))
    return out


def gdn_layer_decode_noalloc(x, conv_pool: ConvStatePool, w, bias, A_log, dt_bias, a, b,
                             pool: GDNStatePool, read_slot, write_slot, out: torch.Tensor,
                             keep_in_place: bool = False, silu: bool = True,
                             scratch_slot: int = 0) -> torch.Tensor:
    """gdn_layer_decode with its work counters in the library's fixed scratch
    slot `scratch_slot` instead of the pool's; allocates nothing, so `out`
    is required."""
    rows = x.shape[0]
    dt = x.dtype
    dev = pool.tensor.device
    C = 2 * pool.hk * pool.dk + pool.hv * pool.dv
    _numel(x, rows * C, "x")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    _numel(a, rows * pool.hv, "a")
    _numel(b, rows * pool.hv, "b")
    _numel(A_log, pool.hv, "A_log")
    _numel(dt_bias, pool.hv, "dt_bias")
    _numel(read_slot, rows, "read_slot")
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    _numel(out, rows * pool.hv * pool.dv, "out")
    _check(_lib.load().gdn_layer_decode_noalloc(
        _ptr(x, "x", dt, dev, host_ok=True), conv_pool.handle, _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev),
        int(bool(silu)), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), _ptr(a, "a", dt, dev, host_ok=True), _ptr(b, "b", dt, dev, host_ok=True),
        pool.handle, _ptr(read_slot, "read_slot", torch.int32, dev),
        _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), rows,
        int(bool(keep_in_place)), int(scratch_slot), _dtype_code(dt), _stream(dev)))
    return out


def gdn_layer_decode_bucket(x, conv_pool: ConvStatePool, w, bias, A_log, dt_bias, a, b, pool: GDNStatePool,
                            read_slot, write_slot, n_decode: torch.Tensor, out: Optional[torch.Tensor] = None,
                            keep_in_place: bool = False, commit: bool = False,
                            silu: bool = True) -> torch.Tensor:
    """The decode half of a mixed step: the launch covers the bucket (x's rows);
    only rows below the device int32 n_decode are decoded, the rest are left
    alone (outputs zero).  With commit (twin only) the decoded rows' tables are
    swapped in the same launch."""
    if commit and (keep_in_place or write_slot is None):
        raise ValueError("commit needs twin slots (a write_slot table, keep_in_place False)")
    rows = x.shape[0]
    dt = x.dtype
    dev = pool.tensor.device
    C = 2 * pool.hk * pool.dk + pool.hv * pool.dv
    _numel(x, rows * C, "x")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    for tname, tt, n in (("a", a, rows * pool.hv), ("b", b, rows * pool.hv), ("A_log", A_log, pool.hv),
                         ("dt_bias", dt_bias, pool.hv), ("read_slot", read_slot, rows), ("n_decode", n_decode, 1)):
        _numel(tt, n, tname)
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    if out is None:
        out = torch.empty((rows, pool.hv, pool.dv), dtype=dt, device=dev)
    _numel(out, rows * pool.hv * pool.dv, "out")
    _check(_lib.load().gdn_layer_decode_bucket(
        _ptr(x, "x", dt, dev, host_ok=True), conv_pool.handle, _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev),
        int(bool(silu)), _ptr(A_log, "A_log", torch.float32, dev),
        _ptr(dt_bias, "dt_bias", torch.float32, dev), _ptr(a, "a", dt, dev, host_ok=True), _ptr(b, "b", dt, dev, host_ok=True),
        pool.handle, _ptr(read_slot, "read_slot", torch.int32, dev),
        _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), rows,
        _ptr(n_decode, "n_decode", torch.int32, dev), int(bool(keep_in_place)), int(bool(commit)),
        _dtype_code(dt), _stream(dev)))
    return out


def gdn_commit(read_slot: torch.Tensor, write_slot: torch.Tensor) -> None:
    """Swap the read and write slot tables on the device (twin-slot commit)."""
    n = read_slot.numel()
    _numel(write_slot, n, "write_slot")
    dev = read_slot.device
    _check(_lib.load().gdn_commit(_ptr(read_slot, "read_slot", torch.int32, dev),
                                  _ptr(write_slot, "write_slot", torch.int32, dev), n, _stream(dev)))


def gdn_validate_slots(read_slot: torch.Tensor, write_slot: Optional[torch.Tensor], num_slots: int,
                       keep_in_place: bool = False) -> None:
    """Debug check of the slot tables (synchronises). Raises GDNError on a violation."""
    dev = read_slot.device
    _check(_lib.load().gdn_validate_slots(_ptr(read_slot, "read_slot", torch.int32, dev),
                                          _ptr(write_slot, "write_slot", torch.int32, dev),
                                          read_slot.numel(), num_slots, int(bool(keep_in_place)),
                                          _stream(dev)))


def get_device_error(device=None) -> int:
    """Read and clear the sticky device error word of `device` (synchronises)."""
    device = torch.device(device if device is not None else "cuda")
    code = ctypes.c_int(0)
    with torch.cuda.device(device):
        _check(_lib.load().gdn_get_device_error(ctypes.byref(code), _stream(device)))
    return code.value


def selftest_wait_timeout(limit_us: int = 1000, device=None) -> None:
    """Run a kernel whose bounded wait cannot end (it gives up after
    `limit_us` microseconds); afterwards the device error word reads
    GDN_DEVERR_TIMEOUT.  Asynchronous."""
    device = torch.device(device if device is not None else "cuda")
    with torch.cuda.device(device):
        _check(_lib.load().gdn_selftest_wait_timeout(int(limit_us), _stream(device)))


def probe_traffic(pool: GDNStatePool, read_slot: torch.Tensor, write_slot: Optional[torch.Tensor],
                  mode: int, sink: Optional[torch.Tensor] = None) -> None:
    """Move a step's state bytes with no arithmetic (roofline probe)."""
    dev = read_slot.device
    _check(_lib.load().gdn_probe_traffic(pool.handle, _ptr(read_slot, "read_slot", torch.int32, dev),
                                         _ptr(write_slot, "write_slot", torch.int32, dev),
                                         read_slot.numel(), mode,
                                         _ptr(sink, "sink", torch.float32, dev), _stream(dev)))


class PreparedCall:
    """A validated C-ABI call with its pointer arguments bound once.

    Calling it launches the same entry point again on the same buffers and
    stream, without re-marshalling the tensors: a decode loop (or a graph
    capture) then costs one ctypes call per launch.  The tensors must stay
    alive and keep their addresses while the call is used.
    """

    def __init__(self, fn_name: str, args: tuple, keep: tuple):
        self._fn = getattr(_lib.load(), fn_name)
        self._args = args
        self._keep = keep  # hold references to the tensors whose pointers are bound

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc:
            _check(rc)


def prepare_layer_decode(x, conv_pool: ConvStatePool, w, bias, A_log, dt_bias, a, b, pool: GDNStatePool,
                         read_slot, write_slot, out, keep_in_place: bool = False, silu: bool = True,
                         stream: Optional[torch.cuda.Stream] = None, commit: bool = False) -> PreparedCall:
    """gdn_layer_decode (or, with commit, gdn_layer_decode_commit) bound to
    fixed buffers (validated here, once)."""
    if commit and (keep_in_place or write_slot is None):
        raise ValueError("commit needs twin slots (a write_slot table, keep_in_place False)")
    rows = x.shape[0]
    dt = x.dtype
    dev = pool.tensor.device
    C = 2 * pool.hk * pool.dk + pool.hv * pool.dv
    _numel(x, rows * C, "x")
    _numel(w, C * conv_pool.width, "w")
    if bias is not None:
        _numel(bias, C, "bias")
    for tname, tt, n in (("a", a, rows * pool.hv), ("b", b, rows * pool.hv), ("A_log", A_log, pool.hv),
                         ("dt_bias", dt_bias, pool.hv), ("read_slot", read_slot, rows),
                         ("out", out, rows * pool.hv * pool.dv)):
        _numel(tt, n, tname)
    if write_slot is not None:
        _numel(write_slot, rows, "write_slot")
    s = (stream or torch.cuda.current_stream(dev)).cuda_stream
    args = (_ptr(x, "x", dt, dev, host_ok=True), conv_pool.handle, _ptr(w, "w", dt, dev), _ptr(bias, "bias", dt, dev),
            int(bool(silu)), _ptr(A_log, "A_log", torch.float32, dev),
            _ptr(dt_bias, "dt_bias", torch.float32, dev), _ptr(a, "a", dt, dev, host_ok=True), _ptr(b, "b", dt, dev, host_ok=True),
            pool.handle, _ptr(read_slot, "read_slot", torch.int32, dev),
            _ptr(write_slot, "write_slot", torch.int32, dev), _ptr(out, "out", dt, dev, host_ok=True), rows)
    if commit:
        args += (_dtype_code(dt), s)
    else:
        args += (int(bool(keep_in_place)), _dtype_code(dt), s)
    return PreparedCall("gdn_layer_decode_commit" if commit else "gdn_layer_decode", args,
                        (x, conv_pool, w, bias, A_log, dt_bias, a, b, pool, read_slot, write_slot, out))


def prepare_commit(read_slot: torch.Tensor, write_slot: torch.Tensor,
                   stream: Optional[torch.cuda.Stream] = None) -> PreparedCall:
    """gdn_commit bound to fixed slot tables."""
    n = read_slot.numel()
    _numel(write_slot, n, "write_slot")
    dev = read_slot.device
    s = (stream or torch.cuda.current_stream(dev)).cuda_stream
    args = (_ptr(read_slot, "read_slot", torch.int32, dev), _ptr(write_slot, "write_slot", torch.int32, dev),
            n, s)
    return PreparedCall("gdn_commit", args, (read_slot, write_slot))


__all__ += ["PreparedCall", "prepare_layer_decode", "prepare_commit"]
