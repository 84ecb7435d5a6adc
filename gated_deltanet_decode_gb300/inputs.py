"""Seeded synthetic inputs for the GDN decode step.

Shared by the tests, the smoke check and the benchmark; it holds none of the
method's arithmetic, only shapes, distributions and slot tables.  Every draw
comes from numpy's PCG64 (``np.random.default_rng(seed)``) in the order the
functions below document; values are drawn in float32 and rounded to the
activation dtype when they are moved into torch tensors.

Distributions (synthetic stand-ins for the decode workloads of the Qwen3.5
models the GDN decode pages serve): q, k, v, a, b and the packed conv input
x ~ N(0, 1); A_log ~ U(0, ln 16); dt_bias ~ U(-1, 1); conv taps ~ N(0, 0.5);
conv bias ~ N(0, 0.1); initial state ~ N(0, 0.1) in every non-null slot;
initial conv window ~ N(0, 1) (past inputs); slot 0 is zero.  N(0, s) names
the standard deviation s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, Optional

import numpy as np


@dataclass(frozen=True)
class Shape:
    rows: int
    hk: int
    hv: int
    dk: int
    dv: int
    width: int = 4
    dtype: str = "bf16"      # activation dtype: "bf16" or "f32"
    num_slots: int = 0

    @property
    def channels(self) -> int:
        return 2 * self.hk * self.dk + self.hv * self.dv

    def with_(self, **kw) -> "Shape":
        return replace(self, **kw)


# The workloads, by what they are.
TINY = Shape(rows=4, hk=2, hv=2, dk=16, dv=16, width=4, dtype="f32", num_slots=9)
QWEN_08B = Shape(rows=64, hk=16, hv=16, dk=128, dv=128, width=4, dtype="bf16", num_slots=129)
QWEN_9B = Shape(rows=64, hk=16, hv=32, dk=128, dv=128, width=4, dtype="bf16", num_slots=129)
SWEEP_ROWS = (1, 4, 16, 64, 128, 256)
SWEEP_SLOTS = 513
STACK_LAYERS = 18
STACK = Shape(rows=128, hk=16, hv=16, dk=128, dv=128, width=4, dtype="bf16", num_slots=257)


class Gen:
    """One seeded stream of draws."""

    def __init__(self, seed: int = 0):
        self.rng = np.random.default_rng(seed)

    def normal(self, shape, std: float = 1.0) -> np.ndarray:
        return (self.rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)

    def uniform(self, lo: float, hi: float, shape) -> np.ndarray:
        return self.rng.uniform(lo, hi, shape).astype(np.float32)

    # -- per-layer parameters: A_log, dt_bias, conv taps, conv bias (this order)
    def params(self, s: Shape) -> Dict[str, np.ndarray]:
        return {
            "A_log": self.uniform(0.0, math.log(16.0), (s.hv,)),
            "dt_bias": self.uniform(-1.0, 1.0, (s.hv,)),
            "w": self.normal((s.channels, s.width), 0.5),
            "bias": self.normal((s.channels,), 0.1),
        }

    # -- per-step inputs of the unfused rule: q, k, v, a, b (this order)
    def step_inputs(self, s: Shape) -> Dict[str, np.ndarray]:
        return {
            "q": self.normal((s.rows, s.hk, s.dk)),
            "k": self.normal((s.rows, s.hk, s.dk)),
            "v": self.normal((s.rows, s.hv, s.dv)),
            "a": self.normal((s.rows, s.hv)),
            "b": self.normal((s.rows, s.hv)),
        }

    # -- per-step inputs of the fused layer: x, a, b (this order)
    def layer_inputs(self, s: Shape) -> Dict[str, np.ndarray]:
        return {
            "x": self.normal((s.rows, s.channels)),
            "a": self.normal((s.rows, s.hv)),
            "b": self.normal((s.rows, s.hv)),
        }

    def state_pool(self, s: Shape, num_slots: Optional[int] = None) -> np.ndarray:
        n = num_slots or s.num_slots
        pool = self.normal((n, s.hv, s.dv, s.dk), 0.1)
        pool[0] = 0.0
        return pool

    def conv_pool(self, s: Shape, num_slots: Optional[int] = None) -> np.ndarray:
        n = num_slots or s.num_slots
        cp = self.normal((n, s.width - 1, s.channels), 1.0)
        cp[0] = 0.0
        return cp

    def slot_tables(self, rows: int, num_slots: int, pad_frac: float = 0.0, twin: bool = True):
        """(read_slot, write_slot) int32 [rows].

        floor(pad_frac * rows) rows, at random positions, are padding (both
        slots 0).  Real rows take distinct slots from a random permutation of
        1..num_slots-1: the first n_real for reading, the next n_real for
        writing (twin) -- or write == read (in place)."""
        n_pad = int(math.floor(pad_frac * rows))
        n_real = rows - n_pad
        need = 2 * n_real if twin else n_real
        if need > num_slots - 1:
            raise ValueError(f"{rows} rows need {need} slots, the pool has {num_slots - 1}")
        perm = self.rng.permutation(np.arange(1, num_slots, dtype=np.int32))
        pad_rows = self.rng.choice(rows, size=n_pad, replace=False) if n_pad else np.array([], int)
        real = np.ones(rows, dtype=bool)
        real[pad_rows] = False
        rs = np.zeros(rows, dtype=np.int32)
        ws = np.zeros(rows, dtype=np.int32)
        rs[real] = perm[:n_real]
        ws[real] = perm[n_real:2 * n_real] if twin else perm[:n_real]
        return rs, ws

    def seq_tables(self, lens, num_slots: int, n_pad: int = 0, token_slots: bool = True):
        """Packed sequences of the given lengths for the many-token calls:
        (cu_seqlens [nseq+1], read_slot [nseq], write_slot [nseq],
        token_slot [T]), int32.

        n_pad sequences, at random positions, are padding (slots 0, token
        slots 0).  Real sequences take distinct slots from a random
        permutation of 1..num_slots-1: reads first, then writes, then (with
        token_slots) one slot a token of the real sequences, for a state a
        token; without, token_slot is all zeros."""
        lens = np.asarray(lens, dtype=np.int64)
        nseq = len(lens)
        cu = np.zeros(nseq + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        pad = np.zeros(nseq, dtype=bool)
        if n_pad:
            pad[self.rng.choice(nseq, size=n_pad, replace=False)] = True
        n_real = int((~pad).sum())
        n_tok = int(lens[~pad].sum()) if token_slots else 0
        need = 2 * n_real + n_tok
        if need > num_slots - 1:
            raise ValueError(f"the sequences need {need} slots, the pool has {num_slots - 1}")
        perm = self.rng.permutation(np.arange(1, num_slots, dtype=np.int32))
        rs = np.zeros(nseq, dtype=np.int32)
        ws = np.zeros(nseq, dtype=np.int32)
        rs[~pad] = perm[:n_real]
        ws[~pad] = perm[n_real:2 * n_real]
        ts = np.zeros(int(cu[-1]), dtype=np.int32)
        nxt = 2 * n_real
        for r in range(nseq if token_slots else 0):
            if not pad[r]:
                ts[cu[r]:cu[r + 1]] = perm[nxt:nxt + lens[r]]
                nxt += int(lens[r])
        return cu, rs, ws, ts


# ---------------------------------------------------------------------------
# torch helpers (plumbing only)
# ---------------------------------------------------------------------------

def torch_dtype(name: str):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def to_torch(a: np.ndarray, dtype: str = "f32", device="cpu"):
    """numpy float32 -> torch tensor of the activation dtype (round to nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.int32:
        return t.to(device)
    return t.to(torch_dtype(dtype)).to(device)


def as_f64(t) -> np.ndarray:
    """The exact values a tensor holds, as float64 numpy (what the oracle consumes)."""
    return t.detach().to("cpu").double().numpy()
