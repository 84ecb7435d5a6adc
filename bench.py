#!/usr/bin/env python
"""Benchmark of the GDN decode layer on GB300.

Workload (default): the 0.8B-shaped single layer -- 64 rows, 16 qk / 16 value
heads, dk = dv = 128, 6144 conv channels of width 4, bf16 activations, fp32
state, 129-slot pools, twin slots.  One step is one fused conv + GDN layer
decode with the twin commit folded into the same launch
(gdn_layer_decode_commit), through the C ABI.  Four independent layer instances (pools, parameters, inputs) are
used in rotation, so that a step never finds the state it reads in L2 (the
four state pools hold 4 x 135 MB against a 126 MB L2).

Prints one JSON line: whole-job GB/s of algorithmic bytes, µs per layer,
the roofline of the layer kernel, an end-to-end figure through host buffers,
the clocks seen during the timed region and the fp64 oracle timed on the
host cores.  `--impl reference` times the oracle itself on the same workload.

The traffic probes (the same state reads and writes with no arithmetic,
read-only and write-only) follow the pages' own roofline measurement of the
step ("mstar PR #1139", "Numbers").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode layer: achieved HBM GB/s (% of 8 TB/s) and µs/layer at 64 rows"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
NSETS = 4
KERNEL_SOURCES = ["gated_deltanet_decode_gb300/csrc/gdn_stream.cu",
                  "gated_deltanet_decode_gb300/csrc/gdn_device.cuh",
                  "gated_deltanet_decode_gb300/csrc/gdn_ptx.cuh"]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "gdn_layer_decode_qwen08b_rows64_steady_traffic.md")


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def layer_bytes(s, real_rows: int) -> int:
    """Bytes one gdn_layer_decode launch must move at least.

    Per real row: the state read and written (2 * hv * dv * dk * 4), the conv
    window read and written (2 * (W-1) * C * e), the token x (C * e), the gates'
    inputs a and b (2 * hv * e).  Per row: the output (hv * dv * e) and two slot
    ids.  Per launch: conv taps and bias ((W + 1) * C * e), A_log and dt_bias.
    """
    e = 2 if s.dtype == "bf16" else 4
    C = s.channels
    per_real = (2 * s.hv * s.dv * s.dk * 4 + 2 * (s.width - 1) * C * e + C * e + 2 * s.hv * e)
    per_row = s.hv * s.dv * e + 2 * 4
    per_launch = (s.width + 1) * C * e + 2 * s.hv * 4
    return real_rows * per_real + s.rows * per_row + per_launch


def commit_bytes(rows: int) -> int:
    return rows * 4 * 4  # read and write both tables


# ---------------------------------------------------------------------------
# peaks, traffic, clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor rate, TFLOP/s: the measured burst figure, else the
    fallback of one earlier GB300 measurement."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def chunked_mma_flops(lens, hv: int, bf16_inputs: bool = True) -> float:
    """Tensor-core flops gdn_prefill_chunked issues (dk = dv = 128, chunks of
    64 tokens).  bf16 inputs (the tcgen05 kernel, M = 128 products of
    K = 16): [K|Q] K^T (8, N = 64, exact), S [K|Q]^T (2 x 8, N = 128: head
    and tail of S against exact K|Q), E T^T and U P^T (3 x 4 each, N = 64:
    hi*hi, hi*lo, lo*hi), the state update (2 x 4, N = 128), plus the blocks
    of T below the diagonal on mma.sync (96 m16n8k16).  fp32 inputs (the
    mma.sync kernel, every operand split, three m16n8k16 a product): the 40
    8-column tiles of the lower blocks of K K^T and Q K^T, T's blocks, and
    per 16 state rows S K^T and S Q^T, E T^T and U^T P^T, and the update."""
    if bf16_inputs:
        fma = (8 * 128 * 64 + 16 * 128 * 128 + 12 * 128 * 64 + 12 * 128 * 64 + 8 * 128 * 128) * 16
        per_chunk = 2 * fma + 96 * 4096
    else:
        per_chunk = (40 * 8 * 3 + 96 + 8 * (2 * 8 * 8 * 3 + 2 * 8 * 4 * 3 + 16 * 4 * 3)) * 4096
    chunks = sum((n + 63) // 64 for n in lens)
    return float(per_chunk * chunks * hv)


def kernel_source_sha() -> str:
    """Hash of the layer kernel's code: its sources with comments, blank lines
    and surrounding whitespace removed, so that editing a comment does not
    disown a profile taken on the same code."""
    import re
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            line = line.split("//", 1)[0].strip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per launch of the layer kernel from the committed ncu summary,
    or None when the summary is missing or the kernel changed since."""
    try:
        fields = {}
        with open(TRAFFIC_SUMMARY) as f:
            for line in f:
                key = line.strip().lstrip("-* `")
                if ":" in key and key.startswith(("traffic_per_launch_bytes", "source_sha256")):
                    k, v = key.split(":", 1)
                    fields[k.strip().strip("`")] = v.strip().strip("` ")
        if fields.get("source_sha256") != kernel_source_sha():
            return None
        return int(fields["traffic_per_launch_bytes"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def count(self) -> int:
        return len(self.lines)

    def wait_first(self, timeout_s: float = 3.0) -> None:
        """Return once the sampler has written a line (nvidia-smi takes a moment to start)."""
        t_end = time.perf_counter() + timeout_s
        while self.proc is not None and not self.lines and time.perf_counter() < t_end:
            time.sleep(0.01)

    def stop(self, since: int = 0):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[since:]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def build_sets(G, I, s, device, nsets, pad_frac=0.0):
    import torch
    sets = []
    for i in range(nsets):
        gen = I.Gen(1000 + i)
        prm = gen.params(s)
        inp = gen.layer_inputs(s)
        dt = s.dtype
        st = {
            "pool": G.GDNStatePool(s.num_slots, s.hk, s.hv, s.dk, s.dv, device=device,
                                   tensor=torch.from_numpy(gen.state_pool(s)).to(device)),
            "cp": G.ConvStatePool(s.num_slots, s.channels, s.width, dtype=I.torch_dtype(dt), device=device,
                                  tensor=I.to_torch(gen.conv_pool(s), dt, device)),
            "w": I.to_torch(prm["w"], dt, device),
            "bias": I.to_torch(prm["bias"], dt, device),
            "A_log": I.to_torch(prm["A_log"], "f32", device),
            "dt_bias": I.to_torch(prm["dt_bias"], "f32", device),
            "x": I.to_torch(inp["x"], dt, device),
            "a": I.to_torch(inp["a"], dt, device),
            "b": I.to_torch(inp["b"], dt, device),
            "out": torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(dt), device=device),
        }
        rs, ws = gen.slot_tables(s.rows, s.num_slots, pad_frac)
        st["rs"] = torch.from_numpy(rs).to(device)
        st["ws"] = torch.from_numpy(ws).to(device)
        st["layer"] = G.prepare_layer_decode(st["x"], st["cp"], st["w"], st["bias"], st["A_log"],
                                             st["dt_bias"], st["a"], st["b"], st["pool"], st["rs"], st["ws"],
                                             st["out"])
        st["layer_ip"] = G.prepare_layer_decode(st["x"], st["cp"], st["w"], st["bias"], st["A_log"],
                                                st["dt_bias"], st["a"], st["b"], st["pool"], st["rs"], None,
                                                st["out"], keep_in_place=True)
        st["commit"] = G.prepare_commit(st["rs"], st["ws"])
        st["layer_commit"] = G.prepare_layer_decode(st["x"], st["cp"], st["w"], st["bias"], st["A_log"],
                                                    st["dt_bias"], st["a"], st["b"], st["pool"], st["rs"],
                                                    st["ws"], st["out"], commit=True)
        sets.append(st)
    return sets


def time_calls(calls, n, device):
    """Mean µs per call of `n` back-to-back calls cycling through `calls`."""
    import torch
    stream = torch.cuda.current_stream(device)
    for i in range(2 * len(calls)):
        calls[i % len(calls)]()
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n):
        calls[i % len(calls)]()
    b.record(stream)
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) * 1e3 / n


def run_unfused(G, I, device, n=400):
    """The two calls the fused layer replaces, 0.8B shape, 64 rows, twin:
    causal_conv1d_decode over the packed q|k|v channels, then gdn_decode_step
    on q, k, v of the same shapes (four instances in rotation)."""
    import torch
    s = I.QWEN_08B
    dt = s.dtype
    sets = []
    for i in range(NSETS):
        gen = I.Gen(4000 + i)
        prm = gen.params(s)
        st = {"pool": G.GDNStatePool(s.num_slots, s.hk, s.hv, s.dk, s.dv, device=device,
                                     tensor=torch.from_numpy(gen.state_pool(s)).to(device)),
              "cp": G.ConvStatePool(s.num_slots, s.channels, s.width, dtype=I.torch_dtype(dt), device=device,
                                    tensor=I.to_torch(gen.conv_pool(s), dt, device)),
              "w": I.to_torch(prm["w"], dt, device), "bias": I.to_torch(prm["bias"], dt, device),
              "A_log": I.to_torch(prm["A_log"], "f32", device), "dt_bias": I.to_torch(prm["dt_bias"], "f32", device),
              "x": I.to_torch(gen.layer_inputs(s)["x"], dt, device)}
        for k, v in gen.step_inputs(s).items():
            st[k] = I.to_torch(v, dt, device)
        rs, ws = gen.slot_tables(s.rows, s.num_slots)
        st["rs"], st["ws"] = torch.from_numpy(rs).to(device), torch.from_numpy(ws).to(device)
        st["y"] = torch.empty((s.rows, s.channels), dtype=I.torch_dtype(dt), device=device)
        st["o"] = torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(dt), device=device)
        stream = torch.cuda.current_stream(device).cuda_stream
        code = G.GDN_BF16 if dt == "bf16" else G.GDN_F32
        st["conv"] = G.PreparedCall("causal_conv1d_decode",
                                    (st["x"].data_ptr(), s.channels, st["cp"].handle, st["rs"].data_ptr(),
                                     st["ws"].data_ptr(), st["w"].data_ptr(), st["bias"].data_ptr(), 1,
                                     st["y"].data_ptr(), s.rows, code, stream), (st,))
        st["step"] = G.PreparedCall("gdn_decode_step",
                                    (st["q"].data_ptr(), st["k"].data_ptr(), st["v"].data_ptr(),
                                     st["a"].data_ptr(), st["b"].data_ptr(), st["A_log"].data_ptr(),
                                     st["dt_bias"].data_ptr(), st["pool"].handle, st["rs"].data_ptr(),
                                     st["ws"].data_ptr(), st["o"].data_ptr(), s.rows, s.hv, 0, code, stream), (st,))
        sets.append(st)

    def both(st):
        st["conv"]()
        st["step"]()
    conv_us = time_calls([st["conv"] for st in sets], n, device)
    step_us = time_calls([st["step"] for st in sets], n, device)
    pair_us = time_calls([lambda st=st: both(st) for st in sets], n, device)
    state = s.rows * s.hv * s.dv * s.dk * 4 * 2
    res = {"workload": "0.8B-shaped conv then rule as two calls, 64 rows, twin",
           "conv_us": round(conv_us, 2), "step_us": round(step_us, 2), "pair_us": round(pair_us, 2),
           "step_GBs": round(state / step_us / 1e3, 1),
           "pair_GBs_of_layer_bytes": round(layer_bytes(s, s.rows) / pair_us / 1e3, 1)}
    del sets
    torch.cuda.empty_cache()
    return res


def run_extras(G, I, device, n=400):
    """The other workloads, timed on the same terms (four instances in rotation,
    back-to-back launches): the rows x write-mode sweep, the 9B-shaped GQA layer
    and the 18-layer decode stack (eager and CUDA-graph replay)."""
    import torch
    res = {}
    sweep = {}
    for rows in I.SWEEP_ROWS:
        sh = I.QWEN_08B.with_(rows=rows, num_slots=I.SWEEP_SLOTS)
        sets = build_sets(G, I, sh, device, NSETS, pad_frac=0.25)
        real = rows - int(math.floor(0.25 * rows))
        nb = layer_bytes(sh, real)
        tw = time_calls([st["layer"] for st in sets], n, device)
        ip = time_calls([st["layer_ip"] for st in sets], n, device)
        # chained and warm: one instance, each step reading what the one before
        # wrote (twin with the commit in the launch, or in place), so whatever
        # of the state L2 still holds is reused
        tw_w = time_calls([sets[0]["layer_commit"]], n, device)
        ip_w = time_calls([sets[0]["layer_ip"]], n, device)
        sweep[str(rows)] = {"real_rows": real, "twin_us": round(tw, 2), "in_place_us": round(ip, 2),
                            "twin_GBs": round(nb / tw / 1e3, 1), "in_place_GBs": round(nb / ip / 1e3, 1),
                            "twin_chained_warm_us": round(tw_w, 2), "in_place_chained_warm_us": round(ip_w, 2)}
        del sets
        torch.cuda.empty_cache()
    res["sweep_rows_write_mode"] = {"workload": "0.8B-shaped fused layer, 25% padding rows on the null "
                                                "slot, 513-slot pools, twin vs in place; cold = four "
                                                "instances in rotation, chained warm = one instance "
                                                "stepping on its own output", "rows": sweep}
    gqa = {}
    for rows in (64, 256):
        sh = I.QWEN_9B.with_(rows=rows, num_slots=2 * rows + 1)
        sets = build_sets(G, I, sh, device, NSETS)
        nb = layer_bytes(sh, rows)
        tw = time_calls([st["layer"] for st in sets], n // 2, device)
        gqa[str(rows)] = {"twin_us": round(tw, 2), "GBs": round(nb / tw / 1e3, 1),
                          "frac_of_measured_peak": round(nb / tw / 1e3 / hbm_peak()[0], 4)}
        del sets
        torch.cuda.empty_cache()
    res["qwen9b_gqa"] = {"workload": "9B-shaped fused layer: 16 qk / 32 v heads, 2R+1 slots, twin",
                         "rows": gqa}
    res["unfused_calls"] = run_unfused(G, I, device)
    res["decode_stack"] = run_stack(G, I, device)
    res["many_tokens"] = run_many_tokens(G, I, device)
    return res


def fp32_alu_peak_tflops() -> float:
    """FP32 FMA rate from the unit counts and the SM clock: 128 FP32 lanes an
    SM, 2 flops an FMA, at the measured maximum SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except (OSError, ValueError):
        pass
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def run_many_tokens(G, I, device, n=20):
    """Prefill (the rule over many tokens, in place), verification (a state a
    token) and the conv over a sequence, 0.8B-shaped, bf16 activations."""
    import torch
    res = {}
    s = I.QWEN_08B
    sets = []
    for i, (nseq, tok) in enumerate([(8, 512)] * 2):
        gen = I.Gen(2000 + i)
        lens = [tok] * nseq
        T = nseq * tok
        cu, rs, ws, _ = gen.seq_tables(lens, 2 * nseq + 1, token_slots=False)
        prm = gen.params(s)
        inp = gen.step_inputs(s.with_(rows=T))
        st = {k: I.to_torch(v, s.dtype, device) for k, v in inp.items()}
        st["x"] = I.to_torch(gen.layer_inputs(s.with_(rows=T))["x"], s.dtype, device)
        st["w"] = I.to_torch(prm["w"], s.dtype, device)
        st["bias"] = I.to_torch(prm["bias"], s.dtype, device)
        st["A_log"] = I.to_torch(prm["A_log"], "f32", device)
        st["dt_bias"] = I.to_torch(prm["dt_bias"], "f32", device)
        st["pool"] = G.GDNStatePool(2 * nseq + 1, s.hk, s.hv, s.dk, s.dv, device=device,
                                    tensor=torch.from_numpy(gen.state_pool(s, 2 * nseq + 1)).to(device))
        st["cp"] = G.ConvStatePool(2 * nseq + 1, s.channels, s.width, dtype=I.torch_dtype(s.dtype),
                                   device=device, tensor=I.to_torch(gen.conv_pool(s, 2 * nseq + 1), s.dtype, device))
        st["cu"], st["rs"] = torch.from_numpy(cu).to(device), torch.from_numpy(rs).to(device)
        st["out"] = torch.empty((T, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device=device)
        st["y"] = torch.empty((T, s.channels), dtype=I.torch_dtype(s.dtype), device=device)
        sets.append(st)
    nseq, tok = 8, 512
    T = nseq * tok

    def prefill(st):
        G.gdn_prefill(st["q"], st["k"], st["v"], st["a"], st["b"], st["A_log"], st["dt_bias"], st["pool"],
                      st["cu"], st["rs"], None, out=st["out"], keep_in_place=True)

    def conv(st):
        G.causal_conv1d_prefill(st["x"], st["cp"], st["cu"], st["rs"], st["w"], st["bias"], out=st["y"])

    us = time_calls([lambda st=st: prefill(st) for st in sets], n, device)
    flops = 6.0 * s.dk * s.dv * s.hv * T  # per token and head: S.k, S.q, the update
    peak = fp32_alu_peak_tflops()
    res["prefill"] = {"workload": f"0.8B-shaped rule, {nseq} sequences x {tok} tokens, in place",
                      "us": round(us, 1), "tokens_per_s": round(T / (us * 1e-6), 1),
                      "roofline": {"bound": "alu", "achieved": round(flops / (us * 1e-6) / 1e12, 3),
                                   "peak": round(peak, 1), "unit": "TFLOP/s",
                                   "frac": round(flops / (us * 1e-6) / 1e12 / peak, 4),
                                   "peak_kind": "fp32 FMA lanes x 2 x max SM clock"}}
    # the same prefill in chunks on the tensor cores
    def prefill_chunked(st):
        G.gdn_prefill_chunked(st["q"], st["k"], st["v"], st["a"], st["b"], st["A_log"], st["dt_bias"],
                              st["pool"], st["cu"], st["rs"], None, out=st["out"], keep_in_place=True)

    us_c = time_calls([lambda st=st: prefill_chunked(st) for st in sets], n, device)
    mma = chunked_mma_flops([tok] * nseq, s.hv)
    tpeak, tkind = bf16_peak()
    res["prefill_chunked"] = {
        "workload": f"0.8B-shaped rule, {nseq} sequences x {tok} tokens, in place, chunks of 64 on the tensor cores (tcgen05, state in TMEM)",
        "us": round(us_c, 1), "tokens_per_s": round(T / (us_c * 1e-6), 1),
        "speedup_vs_token_serial": round(us / us_c, 2),
        "roofline": {"bound": "tensor", "achieved": round(mma / (us_c * 1e-6) / 1e12, 2), "peak": tpeak,
                     "peak_kind": f"{tkind} dense bf16", "unit": "TFLOP/s",
                     "frac": round(mma / (us_c * 1e-6) / 1e12 / tpeak, 4),
                     "flops_per_launch": mma}}
    cb = 2.0 * T * s.channels * 2 + 2 * nseq * (s.width - 1) * s.channels * 2
    us = time_calls([lambda st=st: conv(st) for st in sets], n, device)
    res["conv_prefill"] = {"workload": f"0.8B-shaped conv, {nseq} sequences x {tok} tokens, in place",
                           "us": round(us, 1), "GBs": round(cb / us / 1e3, 1)}
    del sets
    torch.cuda.empty_cache()
    # verification: 64 rows, 4 draft tokens each, a state a token
    rows, tok = 64, 4
    vsets = []
    for i in range(NSETS):
        gen = I.Gen(3000 + i)
        T = rows * tok
        num_slots = 2 * rows + T + 1
        cu, rs, _, ts = gen.seq_tables([tok] * rows, num_slots)
        prm = gen.params(s)
        st = {k: I.to_torch(v, s.dtype, device) for k, v in gen.step_inputs(s.with_(rows=T)).items()}
        st["A_log"] = I.to_torch(prm["A_log"], "f32", device)
        st["dt_bias"] = I.to_torch(prm["dt_bias"], "f32", device)
        st["pool"] = G.GDNStatePool(num_slots, s.hk, s.hv, s.dk, s.dv, device=device,
                                    tensor=torch.from_numpy(gen.state_pool(s, num_slots)).to(device))
        st["cu"], st["rs"], st["ts"] = (torch.from_numpy(a).to(device) for a in (cu, rs, ts))
        st["out"] = torch.empty((T, s.hv, s.dv), dtype=I.torch_dtype(s.dtype), device=device)
        vsets.append(st)

    def verify(st):
        G.gdn_verify(st["q"], st["k"], st["v"], st["a"], st["b"], st["A_log"], st["dt_bias"], st["pool"],
                     st["cu"], st["rs"], st["ts"], out=st["out"])

    us = time_calls([lambda st=st: verify(st) for st in vsets], 200, device)
    vb = rows * s.hv * s.dv * s.dk * 4 * (1 + tok)  # one state read, one state written a token
    res["verify"] = {"workload": f"0.8B-shaped rule, {rows} rows x {tok} draft tokens, a state a token",
                     "us": round(us, 2), "GBs": round(vb / us / 1e3, 1),
                     "frac_of_measured_peak": round(vb / us / 1e3 / hbm_peak()[0], 4)}
    del vsets
    torch.cuda.empty_cache()
    return res


def run_stack(G, I, device, layers=18, steps=64):
    """18 fused layers of the 0.8B shape per step, 128 rows with 10% padding,
    257-slot pools per layer, one commit per step (in the last layer's launch), the rows' request order
    re-permuted (a 1 KB host-to-device table copy) every 16 steps."""
    import numpy as np
    import torch
    s = I.STACK
    gen = I.Gen(77)
    # everything runs on one stream, which the graph capture also uses (the
    # prepared calls are bound to the stream current when they are prepared)
    stream = torch.cuda.Stream(device)
    stream.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(stream):
        return _run_stack(G, I, device, s, gen, stream, layers, steps)


def _run_stack(G, I, device, s, gen, stream, layers, steps):
    import numpy as np
    import torch
    dt = s.dtype
    Ls = []
    for _ in range(layers):
        prm = gen.params(s)
        inp = gen.layer_inputs(s)
        Ls.append({
            "pool": G.GDNStatePool(s.num_slots, s.hk, s.hv, s.dk, s.dv, device=device,
                                   tensor=torch.from_numpy(gen.state_pool(s)).to(device)),
            "cp": G.ConvStatePool(s.num_slots, s.channels, s.width, dtype=I.torch_dtype(dt), device=device,
                                  tensor=I.to_torch(gen.conv_pool(s), dt, device)),
            "w": I.to_torch(prm["w"], dt, device), "bias": I.to_torch(prm["bias"], dt, device),
            "A_log": I.to_torch(prm["A_log"], "f32", device), "dt_bias": I.to_torch(prm["dt_bias"], "f32", device),
            "x": I.to_torch(inp["x"], dt, device), "a": I.to_torch(inp["a"], dt, device),
            "b": I.to_torch(inp["b"], dt, device),
            "out": torch.empty((s.rows, s.hv, s.dv), dtype=I.torch_dtype(dt), device=device)})
    n_real = s.rows - int(0.10 * s.rows)
    perm = gen.rng.permutation(np.arange(1, s.num_slots, dtype=np.int32))
    req = [perm[:n_real].copy(), perm[n_real:2 * n_real].copy()]
    rs = torch.zeros(s.rows, dtype=torch.int32, device=device)
    ws = torch.zeros(s.rows, dtype=torch.int32, device=device)
    tables = []
    for k in range(steps // 16 + 1):  # pinned host tables for each re-permutation
        pos = gen.rng.permutation(s.rows)[:n_real]
        order = gen.rng.permutation(n_real)
        tr = np.zeros(s.rows, np.int32)
        tw = np.zeros(s.rows, np.int32)
        # after 16 steps (an even number of commits) every request is back on its first slot
        tr[pos] = req[0][order]
        tw[pos] = req[1][order]
        tables.append((torch.from_numpy(tr).pin_memory(), torch.from_numpy(tw).pin_memory()))
    # the last layer of the step commits the shared slot tables in its own launch
    calls = [G.prepare_layer_decode(L["x"], L["cp"], L["w"], L["bias"], L["A_log"], L["dt_bias"], L["a"], L["b"],
                                    L["pool"], rs, ws, L["out"], commit=li == len(Ls) - 1)
             for li, L in enumerate(Ls)]

    def one_step():
        for c in calls:
            c()

    def run(replay):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            if i % 16 == 0:
                tr, tw = tables[i // 16]
                rs.copy_(tr, non_blocking=True)
                ws.copy_(tw, non_blocking=True)
            replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) * 1e3 / steps

    rs.copy_(tables[0][0])
    ws.copy_(tables[0][1])
    one_step()
    torch.cuda.synchronize(device)
    eager_us = run(one_step)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        one_step()
    torch.cuda.synchronize(device)
    graph_us = run(g.replay)
    step_bytes = layers * layer_bytes(s, n_real) + commit_bytes(s.rows)
    if G.get_device_error(device) != 0:
        raise RuntimeError("device error in the decode stack")
    res = {"workload": f"{layers} fused layers (0.8B shape) per step, {s.rows} rows with 10% padding, "
                       f"{s.num_slots}-slot pools, commit per step, re-permuted every 16 steps, {steps} steps",
           "eager_us_per_step": round(eager_us, 1), "graph_us_per_step": round(graph_us, 1),
           "eager_GBs": round(step_bytes / eager_us / 1e3, 1), "graph_GBs": round(step_bytes / graph_us / 1e3, 1),
           "us_per_layer_graph": round(graph_us / layers, 2)}
    del Ls, calls, g
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, device):
    import torch
    import gated_deltanet_decode_gb300 as G
    from gated_deltanet_decode_gb300 import inputs as I

    s = I.QWEN_08B
    G.load()
    sets = build_sets(G, I, s, device, NSETS)
    stream = torch.cuda.current_stream(device)
    real_rows = s.rows
    lb = layer_bytes(s, real_rows)
    step_bytes = lb + commit_bytes(s.rows)

    # twin: the step is the layer with the commit in its launch; in place: the
    # in-place layer (nothing to commit)
    twin = args.write_mode == "twin"
    step_key, layer_key = ("layer_commit", "layer") if twin else ("layer_ip", "layer_ip")
    if not twin:
        step_bytes = lb
    # the clock sampler starts before any GPU work, so that it is running (and
    # sampling) through the warm-up and the timed regions that follow
    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    # priming: one call of each kind (lazy set-up: kernel attributes, symbols)
    for st in sets:
        st[step_key]()
        st[layer_key]()
        st["layer"]()
        st["commit"]()
    torch.cuda.synchronize(device)
    if G.get_device_error(device) != 0:
        raise RuntimeError("device error during priming")

    K, W = args.steps, args.warmup
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks.wait_first()
    n_clk = clocks.count() # the clock record starts with the warm-up
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    host0 = time.perf_counter()
    # W untimed warm-up steps, enqueued right ahead of the timed region so that
    # the GPU does not idle before it: the first timed step follows a running
    # step, as every later one does.  Then the timed region: K steps (fused layer
    # with the commit in the same launch), events only at the ends so
    # consecutive kernels keep their programmatic-launch overlap.  The instances
    # rotate throughout, so no step reads state the step before it wrote.
    for i in range(W):
        sets[i % NSETS][step_key]()
    t0.record(stream)
    for i in range(K):
        sets[(W + i) % NSETS][step_key]()
    t1.record(stream)
    host_enqueue_s = time.perf_counter() - host0
    # The same step keeps the GPU under the same load, untimed, until the clock
    # sampler (one sample per 100 ms) has recorded it three times (at most 1 s):
    # a short timed region falls between samples, this window surrounds it.
    t_clk = time.perf_counter() + 1.0
    i = W + K
    while clocks.count() < n_clk + 3 and time.perf_counter() < t_clk:
        for _ in range(50):
            sets[i % NSETS][step_key]()
            i += 1
        torch.cuda.synchronize(device)
    torch.cuda.synchronize(device)
    # second timed region: the layer kernel alone, back to back, for its
    # average launch duration (the roofline's denominator)
    KL = max(K // 2, 100)
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for i in range(KL):
        sets[i % NSETS][layer_key]()
    l1.record(stream)
    torch.cuda.synchronize(device)
    # the same step as two launches (gdn_layer_decode, then gdn_commit), for comparison
    KS = max(K // 4, 100)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(KS):
        st = sets[i % NSETS]
        st["layer"]()
        st["commit"]()
    s1.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop(since=n_clk)
    clk["window"] = ("nvidia-smi every 100 ms from the warm-up through the timed region and the same "
                     "step run on untimed until three samples had been taken")
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    layer_mean_ms = l0.elapsed_time(l1) / KL
    if G.get_device_error(device) != 0:
        raise RuntimeError("device error during the timed region")

    if world > 1:
        total_ms = max_over_ranks(total_ms, device)

    ms_per_step = total_ms / K
    value = world * step_bytes * K / (total_ms * 1e-3) / 1e9
    achieved = lb / (layer_mean_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    # end to end through host buffers: inputs in pinned host memory, output read
    # back to pinned host memory, every step.  The headline form leaves them
    # there and the kernel moves them across the host link itself (the public
    # API takes pinned host activations); the copy-engine form uploads and reads
    # back with cudaMemcpyAsync on copy streams.
    KE = max(K, 200) if K < 2000 else 2000
    e2e_copies = run_e2e(G, I, s, sets, device, KE, step_bytes)
    e2e = run_e2e_zero_copy(G, s, sets, device, KE, step_bytes) if twin else e2e_copies
    probes = run_probes(G, s, sets, device, min(K, 2000))
    del sets
    torch.cuda.empty_cache()
    extras = run_extras(G, I, device) if not args.no_extras else {}

    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(s, world, args.write_mode),
        "us_per_layer": round(layer_mean_ms * 1e3, 3),
        "layer_timing": f"{KL} back-to-back gdn_layer_decode launches over the {NSETS} instances, "
                        "CUDA events at both ends",
        "us_per_step": round(ms_per_step * 1e3, 3),
        "us_per_step_two_launches": round(s0.elapsed_time(s1) * 1e3 / KS, 3),
        "pct_of_8TBps": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "rows_heads_per_s": round(world * s.rows * s.hv * K / (total_ms * 1e-3), 1),
        "algorithmic_bytes_per_step": step_bytes,
        "host_enqueue_s": round(host_enqueue_s, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": f"gdn_layer_decode (gdn_stream_kernel, fused layer, {args.write_mode.replace('_', ' ')})",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic() if twin else None,
            "algorithmic_bytes_per_launch": lb,
            "frac_of_same_bytes_vendor_copy": round(achieved / probes["vendor_copy_same_bytes"]["GB/s"], 4),
        },
        "e2e": e2e,
        "e2e_copies": e2e_copies,
        "probes": probes,
        **extras,
        "gpu_launches": K,
        "clocks": clk,
    }
    return res


def run_probes(G, s, sets, device, K):
    """GB/s of the traffic probes over the same rotation: the state bytes of a
    step moved with no arithmetic (twin copy, in-place read-modify-write,
    read only, write only)."""
    import torch
    stream = torch.cuda.current_stream(device)
    state = s.rows * s.hv * s.dv * s.dk * 4
    res = {}
    for name, mode, nbytes in (("twin_copy", G.GDN_PROBE_TWIN, 2 * state),
                               ("in_place_rmw", G.GDN_PROBE_INPLACE, 2 * state),
                               ("read_only", G.GDN_PROBE_READ, state),
                               ("write_only", G.GDN_PROBE_WRITE, state)):
        calls = [G.PreparedCall("gdn_probe_traffic",
                                (st["pool"].handle, st["rs"].data_ptr(), st["ws"].data_ptr(), s.rows, mode,
                                 None, stream.cuda_stream), (st,)) for st in sets]

        def go(i):
            calls[i % NSETS]()
        for i in range(8):
            go(i)
        torch.cuda.synchronize(device)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K):
            go(i)
        t1.record(stream)
        torch.cuda.synchronize(device)
        us = t0.elapsed_time(t1) * 1e3 / K
        res[name] = {"us": round(us, 3), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1)}
    # the vendor's device-to-device copy (torch copy_) of the same state bytes,
    # rotated over as many buffer pairs: what a copy of this size reaches
    src = [torch.empty(state // 4, dtype=torch.float32, device=device).uniform_() for _ in range(NSETS)]
    dst = [torch.empty_like(x) for x in src]
    for i in range(8):
        dst[i % NSETS].copy_(src[i % NSETS])
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        dst[i % NSETS].copy_(src[i % NSETS])
    t1.record(stream)
    torch.cuda.synchronize(device)
    us = t0.elapsed_time(t1) * 1e3 / K
    res["vendor_copy_same_bytes"] = {"us": round(us, 3), "GB/s": round(2 * state / (us * 1e-6) / 1e9, 1)}
    del src, dst
    # the probes wrote the pools; the layer kernel's values are not reused after this
    return res


def run_e2e(G, I, s, sets, device, K, step_bytes):
    """The step through host buffers, as a serving loop would run it: every
    step copies its inputs (x, a, b, packed in one pinned host arena) to the
    device in one copy, runs the layer with its commit, and reads the output
    back to pinned host memory.  Uploads and read-backs run on two copy
    streams, ordered against the launches by events, so step i+1's upload
    overlaps step i's kernel; every byte still crosses the link inside the
    timed region."""
    import torch
    compute = torch.cuda.current_stream(device)
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)

    def aligned(n):
        return (n + 15) // 16 * 16

    e2e_sets = []
    for st in sets:
        parts = [st[k] for k in ("x", "a", "b")]
        offs, total = [], 0
        for t_ in parts:
            offs.append(total)
            total += aligned(t_.numel() * t_.element_size())
        h = torch.empty(total, dtype=torch.uint8).pin_memory()
        d = torch.empty(total, dtype=torch.uint8, device=device)
        views = {}
        for name, t_, o in zip(("x", "a", "b"), parts, offs):
            nb = t_.numel() * t_.element_size()
            h[o:o + nb].copy_(t_.reshape(-1).view(torch.uint8).cpu())
            views[name] = d[o:o + nb].view(t_.dtype).view(t_.shape)
        out_h = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
        call = G.prepare_layer_decode(views["x"], st["cp"], st["w"], st["bias"], st["A_log"], st["dt_bias"],
                                      views["a"], views["b"], st["pool"], st["rs"], st["ws"], st["out"],
                                      stream=compute, commit=True)
        e2e_sets.append({"h": h, "d": d, "out_h": out_h, "out": st["out"], "call": call,
                         "consumed": torch.cuda.Event(), "read": torch.cuda.Event(),
                         "uploaded": torch.cuda.Event()})
    n = len(e2e_sets)

    def step(i):
        e = e2e_sets[i % n]
        if i >= n:
            up.wait_event(e["consumed"])       # the kernel that read this arena is done
        with torch.cuda.stream(up):
            e["d"].copy_(e["h"], non_blocking=True)
        e["uploaded"].record(up)
        compute.wait_event(e["uploaded"])
        if i >= n:
            compute.wait_event(e["read"])      # the output buffer has been read back
        e["call"]()
        e["consumed"].record(compute)
        down.wait_event(e["consumed"])
        with torch.cuda.stream(down):
            e["out_h"].copy_(e["out"], non_blocking=True)
        e["read"].record(down)

    for i in range(2 * n):
        step(i)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    up.wait_event(t0)
    for i in range(K):
        step(2 * n + i)
    down.wait_event(e2e_sets[(2 * n + K - 1) % n]["read"])
    t1.record(down)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / K
    h2d = e2e_sets[0]["h"].numel()
    d2h = e2e_sets[0]["out_h"].numel() * e2e_sets[0]["out_h"].element_size()
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 6),
            "steps": K, "copies": "one packed upload and one read-back a step, on copy streams overlapping "
                                  "the previous step's kernel"}


def run_e2e_zero_copy(G, s, sets, device, K, step_bytes):
    """The step with its inputs and output left in pinned host memory: the
    kernel reads x, a and b and writes the output across the host link
    (zero-copy), so no separate copy runs; every byte still crosses the link
    inside the timed region."""
    import torch
    compute = torch.cuda.current_stream(device)
    calls, keep = [], []
    for st in sets:
        hx, ha, hb = (st[k].cpu().pin_memory() for k in ("x", "a", "b"))
        hout = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
        calls.append(G.prepare_layer_decode(hx, st["cp"], st["w"], st["bias"], st["A_log"], st["dt_bias"],
                                            ha, hb, st["pool"], st["rs"], st["ws"], hout, stream=compute,
                                            commit=True))
        keep.append((hx, ha, hb, hout))
    for i in range(8):
        calls[i % len(calls)]()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # a few untimed steps right ahead of the timed ones, so that the first timed
    # step follows a running step as every later one does
    for i in range(4):
        calls[i % len(calls)]()
    t0.record(compute)
    for i in range(K):
        calls[(4 + i) % len(calls)]()
    t1.record(compute)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / K
    hx, ha, hb, hout = keep[0]
    h2d = sum(t.numel() * t.element_size() for t in (hx, ha, hb))
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": hout.numel() * hout.element_size(), "ms_per_step": round(ms, 6),
            "steps": K, "how": "x, a, b and the output in pinned host memory, read and written by the "
                              "kernel across the host link; no separate copies"}


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_layer_sample(s, rows: int, seed: int = 7):
    """Inputs for the oracle on `rows` rows of the workload (fp64, rounded to
    the activation dtype like the GPU's)."""
    import numpy as np
    from gated_deltanet_decode_gb300 import inputs as I
    sub = s.with_(rows=rows, num_slots=2 * rows + 1)
    gen = I.Gen(seed)
    prm = gen.params(sub)
    inp = gen.layer_inputs(sub)
    rnd = lambda a: I.as_f64(I.to_torch(a, sub.dtype, "cpu"))  # noqa: E731
    rs, ws = gen.slot_tables(rows, sub.num_slots)
    return {
        "s": sub, "w": rnd(prm["w"]), "bias": rnd(prm["bias"]), "A_log": prm["A_log"].astype(np.float64),
        "dt_bias": prm["dt_bias"].astype(np.float64), "x": rnd(inp["x"]), "a": rnd(inp["a"]),
        "b": rnd(inp["b"]), "pool": gen.state_pool(sub).astype(np.float64),
        "cp": rnd(gen.conv_pool(sub)), "rs": rs, "ws": ws,
    }


def time_oracle_step(orc, d, nthreads: int) -> float:
    t = time.perf_counter()
    orc.layer(d["x"], d["cp"], d["w"], d["bias"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"],
              d["rs"], d["ws"], hk=d["s"].hk, act_bf16=d["s"].dtype == "bf16", nthreads=nthreads)
    orc.commit(d["rs"], d["ws"])
    return time.perf_counter() - t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(budget_s: float = 12.0):
    """The oracle as it stands, on all host cores, over the full 64-row step of
    the workload, repeated while the budget lasts (at least once)."""
    import oracle as orc
    from gated_deltanet_decode_gb300 import inputs as I
    s = I.QWEN_08B
    cores = host_cores()
    d = oracle_layer_sample(s, s.rows)
    times = []
    t_end = time.perf_counter() + budget_s
    while not times or time.perf_counter() < t_end:
        times.append(time_oracle_step(orc, d, cores))
    per = statistics.median(times)
    # the same oracle on one thread: one 8-row step (an eighth of the workload)
    d1 = oracle_layer_sample(s, 8)
    one = time_oracle_step(orc, d1, 1) * (s.rows / 8)
    return {"value": round(layer_bytes(s, s.rows) / per / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(times)} full 64-row steps of the workload (fp64 oracle layer + commit), "
                      f"median {per * 1e3:.1f} ms per step",
            "one_thread": {"value": round(layer_bytes(s, s.rows) / one / 1e9, 4), "unit": "GB/s",
                           "sample": "one 8-row step on one thread, scaled to 64 rows"}}


def workload_config(s, world: int, mode: str = "twin") -> dict:
    """The bench's workload, as both arms report it."""
    slots = ("twin slots, commit each step (in the layer's launch)" if mode == "twin"
             else "state updated in place")
    return {
        "workload": "0.8B-shaped GDN decode layer: fused conv+rule, 64 rows, 16 qk/16 v heads, "
                    "dk=dv=128, 6144 conv channels width 4, bf16 activations, fp32 state, "
                    f"129-slot pools, {slots}",
        "rows": s.rows, "hk": s.hk, "hv": s.hv, "dk": s.dk, "dv": s.dv, "conv_width": s.width,
        "activations": s.dtype, "num_slots": s.num_slots, "mode": mode,
        "l2": f"inputs larger than L2: {NSETS} layer instances in rotation "
              f"({NSETS} x {s.num_slots * s.hv * s.dv * s.dk * 4 / 1e6:.0f} MB of state)",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def run_reference(args, budget_s: float = 150.0):
    """--impl reference: the oracle itself on all host cores, as the cpu_baseline
    leg runs it.  A step is the full 64-row step of the workload (fp64 oracle
    layer + commit) when (warmup + steps) of them fit the time budget, else the
    leading rows of it, the most that fit (all 16 head pairs of each row, so the
    cores have (row, head) units to share)."""
    import oracle as orc
    from gated_deltanet_decode_gb300 import inputs as I
    s = I.QWEN_08B
    cores = host_cores()
    d = oracle_layer_sample(s, s.rows)
    t64 = time_oracle_step(orc, d, cores)            # calibration, untimed
    n = args.steps + args.warmup
    rows = s.rows
    while rows > 1 and n * t64 * rows / s.rows > budget_s:
        rows //= 2
    if rows != s.rows:
        d = oracle_layer_sample(s, rows)
    for _ in range(args.warmup):
        time_oracle_step(orc, d, cores)
    t = time.perf_counter()
    for _ in range(args.steps):
        time_oracle_step(orc, d, cores)
    el = time.perf_counter() - t
    bytes_per = layer_bytes(s.with_(rows=rows), rows) + commit_bytes(rows)
    value = bytes_per * args.steps / el / 1e9
    sample = (f"{rows} of the 64 rows of the workload per step, all 16 qk/v head pairs "
              f"(fp64 oracle layer + commit), {cores} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(I.QWEN_08B, 1),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true",
                    help="omit the sweep, 9B and decode-stack workloads (reported beside the headline)")
    ap.add_argument("--write-mode", choices=["twin", "in_place"], default="twin",
                    help="the timed step's state write: twin slots with the commit (default) or in place")
    ap.add_argument("--many-tokens-only", action="store_true",
                    help="time only the prefill, verification and sequence-conv workloads (one GPU) "
                         "and print their JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.many_tokens_only:
        import gated_deltanet_decode_gb300 as G
        from gated_deltanet_decode_gb300 import inputs as I
        G.load()
        if rank == 0:
            print(json.dumps(run_many_tokens(G, I, device)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    res = run_ours(args, rank, world, device)
    if rank == 0:
        if world == 1:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
