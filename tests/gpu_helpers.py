"""Helpers for the GPU parity tests: move seeded inputs into torch tensors,
run the oracle on the same values, and compare.

The oracle side only ever sees the generator's values (rounded to the
activation dtype on the CPU) and its own slot tables; nothing the CUDA path
computed is fed to it.

Tolerances (written here, used by every parity test):
  * state, one step:        per (row, value head) max|S_gpu - S_ref| / max|S_ref| <= 1e-5
  * state, chained steps:   the same ratio <= 1e-3 after 256 (or 128) steps
  * bf16 outputs:           |o_gpu - o_ref| <= 2e-2 + 1e-2 |o_ref| elementwise
  * fp32 outputs:           |o_gpu - o_ref| <= 1e-5 + 1e-5 |o_ref|
  * slots, conv windows:    bit-exact
  * conv outputs:           bit-exact after rounding to the activation type,
                            except where the exact value lies within the fp32
                            evaluation error of a rounding midpoint; there either
                            neighbour is accepted (both are correct roundings)
"""
from __future__ import annotations

import numpy as np
import torch

from gated_deltanet_decode_gb300 import inputs as I

STATE_TOL_ONE = 1e-5
STATE_TOL_CHAIN = 1e-3
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL, F32_RTOL = 1e-5, 1e-5
# fp32 evaluation of one conv channel: a handful of roundings of terms bounded
# by `mag`, and SiLU's slope is below 1.1; 2^-20 leaves a wide margin.
CONV_EVAL_REL = 2.0 ** -20

DEV = "cuda"


def pair(a: np.ndarray, dtype: str = "f32"):
    """(device tensor, exact float64 values): rounding happens once, on the CPU."""
    cpu = I.to_torch(a, dtype, "cpu")
    return cpu.to(DEV), I.as_f64(cpu)


def t(a: np.ndarray, dtype: str = "f32") -> torch.Tensor:
    return I.to_torch(a, dtype, DEV)


def ti(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a.astype(np.int32))).to(DEV)


def f64(x: torch.Tensor) -> np.ndarray:
    return I.as_f64(x)


def state_rel_err(S_gpu: np.ndarray, S_ref: np.ndarray) -> np.ndarray:
    """Per-head max|diff| / max|ref| over the trailing [dv][dk] axes."""
    d = np.abs(S_gpu.astype(np.float64) - S_ref).reshape(*S_ref.shape[:-2], -1).max(-1)
    m = np.abs(S_ref).reshape(*S_ref.shape[:-2], -1).max(-1)
    return d / np.maximum(m, 1e-30)


def assert_out_close(o_gpu: np.ndarray, o_ref: np.ndarray, dtype: str, what: str = "out"):
    atol, rtol = (BF16_ATOL, BF16_RTOL) if dtype == "bf16" else (F32_ATOL, F32_RTOL)
    err = np.abs(o_gpu - o_ref)
    bad = err > atol + rtol * np.abs(o_ref)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance, "
                           f"worst {err.max():.3g}")


def conv_magnitude(win: np.ndarray, x: np.ndarray, w: np.ndarray, bias) -> np.ndarray:
    """|bias| + sum |w_j * window_j| + |w_last * x| per (row, channel): the scale of the
    terms an fp32 evaluation of the conv rounds.  win: [rows][W-1][C], x: [rows][C]."""
    W = w.shape[1]
    mag = np.abs(w[:, W - 1])[None, :] * np.abs(x)
    for j in range(W - 1):
        mag = mag + np.abs(w[:, j])[None, :] * np.abs(win[:, j, :])
    if bias is not None:
        mag = mag + np.abs(bias)[None, :]
    return mag


def check_conv_outputs(orc, y_gpu: np.ndarray, y_exact: np.ndarray, mag: np.ndarray, dtype: str):
    """Compare conv outputs; returns the boolean mask of accepted rounding flips."""
    tol = CONV_EVAL_REL * (mag + np.abs(y_exact))
    if dtype == "f32":
        err = np.abs(y_gpu - y_exact)
        assert (err <= tol).all(), f"conv f32 outputs off by up to {err.max():.3g}"
        return np.zeros(y_gpu.shape, dtype=bool)
    ref = orc.round_bf16(y_exact)
    flip = y_gpu != ref
    if flip.any():
        mid = 0.5 * (y_gpu[flip] + ref[flip])
        near = np.abs(y_exact[flip] - mid) <= tol[flip]
        adjacent = np.abs(y_gpu[flip] - ref[flip]) <= np.abs(ref[flip]) * 2.0 ** -7 + 2.0 ** -133
        assert (near & adjacent).all(), (
            f"{(~(near & adjacent)).sum()} conv outputs differ from the oracle's rounding "
            "away from a rounding midpoint")
    return flip


def bf16_other_neighbour(y_exact: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """The bfloat16 value next to `ref` on the side of `y_exact` (ref being the
    oracle's rounding of y_exact): the other correct rounding when y_exact sits
    on a rounding midpoint.  Formed from the oracle's values alone."""
    y_exact = np.asarray(y_exact, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    r32 = ref.astype(np.float32)
    bits = r32.view(np.uint32).astype(np.int64)
    away = (y_exact > ref) != np.signbit(r32)            # the neighbour is farther from zero
    out = (bits + np.where(away, 0x10000, -0x10000)).astype(np.uint32).view(np.float32)
    out = out.astype(np.float64)
    zero = ref == 0.0
    out[zero] = np.copysign(2.0 ** -133, y_exact[zero])
    return out


def oracle_layer_on_gpu_roundings(orc, y_gpu, xr, cp_ref, w64, bias64, A_log, dt_bias, pool_ref, rs, ws,
                                  s, keep_in_place=False, silu=True):
    """The oracle's layer (conv, rounding to the activation type, split, rule:
    the composition gdn_oracle_layer performs) on `rows = len(rs)` rows, where
    each bf16 rounding of the conv output is the oracle's own except at the
    channels where the GPU's conv (y_gpu, its fp32 evaluation rounded) took the
    other neighbour of a rounding midpoint and check_conv_outputs accepted it:
    there the oracle uses that other neighbour, formed from its own exact value.
    The GPU's value only selects; every input of the rule is the oracle's.
    Updates cp_ref and pool_ref; returns (o_ref, flips)."""
    rs = np.asarray(rs, dtype=np.int32)
    ws = np.asarray(ws, dtype=np.int32)
    real = rs != 0
    mag = conv_magnitude(cp_ref[rs], xr["x"], w64, bias64)
    y_exact, bad = orc.conv_step(xr["x"], cp_ref, rs, None if keep_in_place else ws, w64, bias64, silu=silu)
    assert bad == 0
    flips = np.zeros(y_exact.shape, dtype=bool)
    if s.dtype == "bf16":
        ref = orc.round_bf16(y_exact)
        flips[real] = check_conv_outputs(orc, y_gpu[real], y_exact[real], mag[real], "bf16")
        y_sel = ref.copy()
        if flips.any():
            y_sel[flips] = bf16_other_neighbour(y_exact[flips], ref[flips])
        assert np.array_equal(y_sel[real], y_gpu[real])
    else:
        check_conv_outputs(orc, y_gpu[real], y_exact[real], mag[real], "f32")
        y_sel = y_exact.astype(np.float32).astype(np.float64)
    rows = y_sel.shape[0]
    nq = s.hk * s.dk
    q = y_sel[:, :nq].reshape(rows, s.hk, s.dk)
    k = y_sel[:, nq:2 * nq].reshape(rows, s.hk, s.dk)
    v = y_sel[:, 2 * nq:].reshape(rows, s.hv, s.dv)
    o_ref, bad = orc.step(q, k, v, xr["a"], xr["b"], A_log, dt_bias, pool_ref, rs, ws,
                          keep_in_place=keep_in_place)
    assert bad == 0
    return o_ref, flips
