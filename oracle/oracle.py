"""ctypes wrapper around ``gdn_oracle.c`` (plain C, fp64).

Test infrastructure, not product code.  Only ``tests/``, the smoke check and
the benchmark's CPU-baseline leg may call it.  It shares no code with the CUDA
path; arrays go in and out as float64 numpy arrays (int32 for slot tables).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, special cases, a hand-worked example
(``tests/golden/rule_2x2.json``), an unrolled product of transition matrices
and brute force on tiny inputs; ``layer``'s composition (the conv output
rounded to the activation type by construction-known values and hand-worked
ties, the SiLU forwarded through closed forms, the window written to the slot
its state goes to) by the layer pins there; ``prefill`` and ``conv_prefill`` by
``tests/test_oracle_prefill_pins.py`` (the unrolled product per token, the
pinned one-token step token by token, numpy's convolution).  Planted mistakes
in ``tests/test_oracle_mutations.py`` show the pins are sharp.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

__all__ = [
    "build", "lib", "softplus", "alpha", "beta", "round_bf16", "l2norm", "rule", "head",
    "conv_row", "step", "conv_step", "layer", "prefill", "conv_prefill", "copy_slots", "commit",
    "max_threads",
]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) unless an up-to-date build exists."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_D = ctypes.c_double
_I = ctypes.c_int
_P = ctypes.c_void_p


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # GDN_ORACLE_LIB points at another build of the same source; the
            # mutation test uses it to load copies with planted mistakes.
            override = os.environ.get("GDN_ORACLE_LIB")
            L = ctypes.CDLL(override if override else build())
            L.gdn_oracle_softplus.restype = _D
            L.gdn_oracle_softplus.argtypes = [_D]
            L.gdn_oracle_alpha.restype = _D
            L.gdn_oracle_alpha.argtypes = [_D, _D, _D]
            L.gdn_oracle_beta.restype = _D
            L.gdn_oracle_beta.argtypes = [_D]
            L.gdn_oracle_round_bf16.restype = _D
            L.gdn_oracle_round_bf16.argtypes = [_D]
            L.gdn_oracle_round_bf16_array.restype = None
            L.gdn_oracle_round_bf16_array.argtypes = [_P, _P, ctypes.c_long]
            L.gdn_oracle_round_f32.restype = _D
            L.gdn_oracle_round_f32.argtypes = [_D]
            L.gdn_oracle_l2norm.restype = None
            L.gdn_oracle_l2norm.argtypes = [_P, _I, _D, _D, _P]
            L.gdn_oracle_rule.restype = None
            L.gdn_oracle_rule.argtypes = [_I, _I, _P, _P, _P, _P, _D, _D, _P, _P]
            L.gdn_oracle_head.restype = None
            L.gdn_oracle_head.argtypes = [_I, _I, _P, _P, _P, _P, _D, _D, _D, _D, _P, _P]
            L.gdn_oracle_conv_row.restype = None
            L.gdn_oracle_conv_row.argtypes = [_I, _I, _P, _P, _P, _P, _I, _P, _P]
            L.gdn_oracle_step.restype = _I
            L.gdn_oracle_step.argtypes = [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _I, _P, _I]
            L.gdn_oracle_conv_step.restype = _I
            L.gdn_oracle_conv_step.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P]
            L.gdn_oracle_layer.restype = _I
            L.gdn_oracle_layer.argtypes = [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P,
                                           _P, _P, _P, _P, _P, _P, _I, _I, _P, _I]
            L.gdn_oracle_prefill.restype = _I
            L.gdn_oracle_prefill.argtypes = [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _P, _P, _P, _P, _I]
            L.gdn_oracle_conv_prefill.restype = _I
            L.gdn_oracle_conv_prefill.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I,
                                                  _P]
            L.gdn_oracle_copy_slots.restype = _I
            L.gdn_oracle_copy_slots.argtypes = [_I, ctypes.c_long, _P, _P, _P, _I]
            L.gdn_oracle_commit.restype = None
            L.gdn_oracle_commit.argtypes = [_I, _P, _P]
            L.gdn_oracle_max_threads.restype = _I
            L.gdn_oracle_max_threads.argtypes = []
            _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data


def softplus(x: float) -> float:
    return lib().gdn_oracle_softplus(float(x))


def alpha(A_log: float, a: float, dt_bias: float) -> float:
    return lib().gdn_oracle_alpha(float(A_log), float(a), float(dt_bias))


def beta(b: float) -> float:
    return lib().gdn_oracle_beta(float(b))


def round_bf16(x) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().gdn_oracle_round_bf16_array(_ptr(x), _ptr(y), x.size)
    return y


def l2norm(x, eps: float = 1e-6, scale: float = 1.0) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().gdn_oracle_l2norm(_ptr(x), x.size, eps, scale, _ptr(y))
    return y


def rule(S, qhat, khat, v, alpha_: float, beta_: float):
    """Literal matrix form for one head. S: [dv][dk]. Returns (S_new, o)."""
    S = _f64(S)
    dv, dk = S.shape
    qhat, khat, v = _f64(qhat), _f64(khat), _f64(v)
    assert qhat.shape == (dk,) and khat.shape == (dk,) and v.shape == (dv,)
    S_new = np.empty_like(S)
    o = np.empty(dv)
    lib().gdn_oracle_rule(dk, dv, _ptr(S), _ptr(qhat), _ptr(khat), _ptr(v), float(alpha_),
                          float(beta_), _ptr(S_new), _ptr(o))
    return S_new, o


def head(S, q, k, v, a: float, b: float, A_log: float, dt_bias: float):
    """One (row, value head) from raw q/k/v and gate inputs. Returns (S_new, o)."""
    S = _f64(S)
    dv, dk = S.shape
    q, k, v = _f64(q), _f64(k), _f64(v)
    assert q.shape == (dk,) and k.shape == (dk,) and v.shape == (dv,)
    S_new = np.empty_like(S)
    o = np.empty(dv)
    lib().gdn_oracle_head(dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v), float(a), float(b),
                          float(A_log), float(dt_bias), _ptr(S_new), _ptr(o))
    return S_new, o


def conv_row(win, x, w, bias, silu: bool = True):
    """One row of the decode conv. win: [W-1][C], x: [C], w: [C][W]. Returns (y, new_win)."""
    win, x, w = _f64(win), _f64(x), _f64(w)
    C, W = w.shape
    assert win.shape == (W - 1, C) and x.shape == (C,)
    bias = None if bias is None else _f64(bias)
    y = np.empty(C)
    new_win = np.empty_like(win)
    lib().gdn_oracle_conv_row(C, W, _ptr(win), _ptr(x), _ptr(w), _ptr(bias), int(bool(silu)),
                              _ptr(y), _ptr(new_win))
    return y, new_win


def step(q, k, v, a, b, A_log, dt_bias, pool, read_slot, write_slot, keep_in_place=False,
         nthreads: int = 0):
    """Decode step over an fp64 pool [num_slots][hv][dv][dk], updated in place.

    Returns (out [rows][hv][dv], bad_rows).
    """
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    num_slots, hv, dv, dk = pool.shape
    rows, hk = q.shape[0], q.shape[1]
    rs = _i32(read_slot)
    ws = _i32(write_slot if write_slot is not None else read_slot)
    out = np.empty((rows, hv, dv))
    bad = lib().gdn_oracle_step(rows, hk, hv, dk, dv, num_slots, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(pool),
                                _ptr(rs), _ptr(ws), int(bool(keep_in_place)), _ptr(out),
                                int(nthreads))
    return out, bad


def conv_step(x, conv_pool, read_slot, write_slot, w, bias, silu: bool = True):
    """Decode conv over an fp64 conv pool [num_slots][W-1][C], updated in place.

    write_slot None means in place.  Returns (y [rows][C], bad_rows).
    """
    x, w = _f64(x), _f64(w)
    assert conv_pool.dtype == np.float64 and conv_pool.flags.c_contiguous
    num_slots = conv_pool.shape[0]
    rows, C = x.shape
    W = w.shape[1]
    bias = None if bias is None else _f64(bias)
    rs = _i32(read_slot)
    ws = None if write_slot is None else _i32(write_slot)
    y = np.empty((rows, C))
    bad = lib().gdn_oracle_conv_step(rows, C, W, num_slots, _ptr(x), _ptr(conv_pool), _ptr(rs),
                                     _ptr(ws), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(y))
    return y, bad


def layer(x, conv_pool, w, bias, a, b, A_log, dt_bias, pool, read_slot, write_slot, hk: int,
          keep_in_place=False, act_bf16=True, silu=True, nthreads: int = 0):
    """Conv, rounding to the activation type, split, decode step. Pools update in place.

    Returns (out [rows][hv][dv], bad_rows).
    """
    x, w, a, b = _f64(x), _f64(w), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    bias = None if bias is None else _f64(bias)
    num_slots, hv, dv, dk = pool.shape
    rows = x.shape[0]
    W = w.shape[1]
    assert conv_pool.dtype == np.float64 and pool.dtype == np.float64
    rs = _i32(read_slot)
    ws = _i32(write_slot if write_slot is not None else read_slot)
    out = np.empty((rows, hv, dv))
    bad = lib().gdn_oracle_layer(rows, hk, hv, dk, dv, W, num_slots, _ptr(x), _ptr(conv_pool),
                                 _ptr(w), _ptr(bias), int(bool(silu)), _ptr(a), _ptr(b),
                                 _ptr(A_log), _ptr(dt_bias), _ptr(pool), _ptr(rs), _ptr(ws),
                                 int(bool(keep_in_place)), int(bool(act_bf16)), _ptr(out),
                                 int(nthreads))
    return out, bad


def prefill(cu_seqlens, q, k, v, a, b, A_log, dt_bias, pool, read_slot, write_slot=None,
            token_slot=None, nthreads: int = 0):
    """Many tokens a sequence over an fp64 pool [num_slots][hv][dv][dk],
    updated in place.  q, k: [T][hk][dk]; v: [T][hv][dv]; a, b: [T][hv].
    write_slot None: in place; token_slot ([T]): a state a token (verify).

    Returns (out [T][hv][dv], bad_sequences).
    """
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    num_slots, hv, dv, dk = pool.shape
    T, hk = q.shape[0], q.shape[1]
    cu = _i32(cu_seqlens)
    nseq = cu.shape[0] - 1
    assert cu[0] == 0 and cu[-1] == T
    rs = _i32(read_slot)
    ws = None if write_slot is None else _i32(write_slot)
    ts = None if token_slot is None else _i32(token_slot)
    out = np.empty((T, hv, dv))
    bad = lib().gdn_oracle_prefill(nseq, hk, hv, dk, dv, num_slots, _ptr(cu), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(pool), _ptr(rs),
                                   _ptr(ws), _ptr(ts), _ptr(out), int(nthreads))
    return out, bad


def conv_prefill(cu_seqlens, x, conv_pool, read_slot, write_slot, w, bias, token_slot=None,
                 silu: bool = True):
    """Causal conv over many tokens a sequence, on an fp64 conv pool
    [num_slots][W-1][C] updated in place.  x: [T][C].  write_slot None: in
    place; token_slot ([T]): a window a token.  Returns (y [T][C], bad)."""
    x, w = _f64(x), _f64(w)
    assert conv_pool.dtype == np.float64 and conv_pool.flags.c_contiguous
    num_slots = conv_pool.shape[0]
    T, C = x.shape
    W = w.shape[1]
    bias = None if bias is None else _f64(bias)
    cu = _i32(cu_seqlens)
    nseq = cu.shape[0] - 1
    assert cu[0] == 0 and cu[-1] == T
    rs = _i32(read_slot)
    ws = None if write_slot is None else _i32(write_slot)
    ts = None if token_slot is None else _i32(token_slot)
    y = np.empty((T, C))
    bad = lib().gdn_oracle_conv_prefill(nseq, C, W, num_slots, _ptr(cu), _ptr(x), _ptr(conv_pool), _ptr(rs),
                                        _ptr(ws), _ptr(ts), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(y))
    return y, bad


def copy_slots(pool, src, dst) -> int:
    """Copy slot src[i] to slot dst[i] of an fp64 pool [num_slots][...] in
    place; returns the number of bad pairs (skipped)."""
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    num_slots = pool.shape[0]
    slot_elems = int(np.prod(pool.shape[1:]))
    s, d = _i32(src), _i32(dst)
    assert s.shape == d.shape
    return lib().gdn_oracle_copy_slots(num_slots, slot_elems, _ptr(pool), _ptr(s), _ptr(d), int(s.shape[0]))


def commit(read_slot: np.ndarray, write_slot: np.ndarray) -> None:
    assert read_slot.dtype == np.int32 and write_slot.dtype == np.int32
    lib().gdn_oracle_commit(read_slot.size, _ptr(read_slot), _ptr(write_slot))


def max_threads() -> int:
    return lib().gdn_oracle_max_threads()
