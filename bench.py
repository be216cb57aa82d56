#!/usr/bin/env python
"""Benchmark of the Q4_0 / Q8_0 block-quantised products on GB300.

One step = one pass over every kernel of the hot path, each at the workload
size of the pages' models (synthetic, seeded data of those shapes):

  gemv   Q4_0 5120x5120, 1 column, y = y0 + W x           (decode projection)
  lmhead Q8_0 248320x5120, 1 column                       (LM head)
  twins  Q4_0 17408x5120, 8 columns                       (speculative verify)
  gateup Q4_0 2 x 17408x5120, 16 columns, h = SiLU(g) * u (prefill FFN, fused)
  down   Q4_0 5120x17408, 16 columns, y = y0 + W h        (prefill FFN down)
  moe    Q8_0 256 experts x top-8 + shared, 8 columns     (MoE layer)

Metric: weight-stream GB/s = algorithmic weight bytes (quants + f16 scales of
every matrix read in the step; routed experts only for the MoE) / step time.
All weights are resident in HBM before timing; each step streams ~1.8 GB of
distinct weights, far more than the 129 MB L2, so no step finds the previous
step's weights in L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4_0/Q8_0 GEMV weight-stream GB/s & % of GB300 HBM peak at 1/8/16 columns"
UNIT = "GB/s"
WORKLOAD = ("hot-path pass: Q4_0 GEMV 5120x5120 C=1 +y0; Q8_0 LM head 248320x5120 C=1; "
            "Q4_0 twins 17408x5120 C=8; Q4_0 FFN gate/up 2x17408x5120 C=16 (SiLU*up, f16 h) "
            "+ down 5120x17408 C=16 +y0; Q8_0 MoE 256 experts top-8 + shared, ffn 512, "
            "hidden 2048, C=8")
KERNELS = ("gemv", "lmhead", "twins", "gateup", "down", "moe")


def lmhead_traffic(rows: int):
    """DRAM bytes per LM-head launch from the committed ncu record
    (profiles/lmhead_q8_gemv_traffic.json), scaled to `rows`; None when the
    kernel's sources changed since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "lmhead_q8_gemv_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    h = hashlib.sha256()
    for f in rec["sources"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != rec["sources_sha256"]:
        return None
    return rec["traffic_bytes_per_row"] * rows


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------- workload
def make_workload(seed: int = 0, only=None) -> dict:
    """All host-side inputs of one step (numpy), drawn once; `only` names one
    call of the step whose inputs alone are drawn (the same values)."""
    w = {}
    need = {"gemv": ("gemv",), "lmhead": ("lmhead",), "twins": ("twins",),
            "gateup": ("ffn",), "down": ("ffn",), "moe": ("moe",)}
    keep = need.get(only) if only else None
    if keep is None or "gemv" in keep:
        w["gemv"] = synth.q4_gemv_residual(seed)
    if keep is None or "lmhead" in keep:
        w["lmhead"] = synth.lm_head(seed + 1)
    if keep is None or "twins" in keep:
        w["twins"] = synth.twins(17408, 8, seed + 2)
    if keep is None or "ffn" in keep:
        w["ffn"] = synth.prefill_ffn(seed + 3)
    if keep is None or "moe" in keep:
        w["moe"] = synth.moe_layer(8, seed + 4)
    return w


def activation_bytes() -> dict:
    """Algorithmic bytes of a step's activations, residuals and outputs per
    call (what each kernel must read or write besides weights): x f16 read,
    y0 f32 read, y f32 or h f16 written; the FFN's h is written by gate/up and
    read by down; the MoE reads x, the ids and routing weights, writes y and
    writes then reads its h (f16 [cols][top-k + 1][ffn])."""
    f16, f32, i32 = 2, 4, 4
    return {
        "gemv": 5120 * f16 + 5120 * f32 + 5120 * f32,
        "lmhead": 5120 * f16 + 248320 * f32,
        "twins": 8 * 5120 * f16 + 8 * 17408 * f32,
        "gateup": 16 * 5120 * f16 + 16 * 17408 * f16,
        "down": 16 * 17408 * f16 + 16 * 5120 * f32 + 16 * 5120 * f32,
        "moe": 8 * 2048 * f16 + 8 * 8 * (i32 + f32) + 8 * 2048 * f32 + 2 * 8 * 9 * 512 * f16,
    }


def weight_bytes(w: dict, uniq_count: int) -> dict:
    wb = {}
    wb["gemv"] = synth.weight_bytes(synth.Q4_0, 5120, 5120)
    wb["lmhead"] = synth.weight_bytes(synth.Q8_0, w["lmhead"]["rows"], 5120)
    wb["twins"] = synth.weight_bytes(synth.Q4_0, 17408, 5120)
    wb["gateup"] = 2 * synth.weight_bytes(synth.Q4_0, 17408, 5120)
    wb["down"] = synth.weight_bytes(synth.Q4_0, 5120, 17408)
    m = w["moe"]
    per_expert = 3 * synth.weight_bytes(synth.Q8_0, m["ffn"], m["hidden"])
    wb["moe"] = (uniq_count + 1) * per_expert  # routed experts read once + shared
    return wb


# --------------------------------------------------------------- GPU arm
class GpuStep:
    """Device-resident buffers and the six calls of one step."""

    def __init__(self, w: dict, torch, only=None):
        import gemm_q4_q8_gb300 as qg
        self.qg = qg
        self.torch = torch
        t = torch
        self.w = w

        def d(a):
            return t.from_numpy(np.ascontiguousarray(a)).cuda()

        def dq(qtype, q, scl):
            # load-time repack on the GPU: GGUF blocks -> the library's layout
            rows, nb = scl.shape
            blocks = d(synth.to_gguf_blocks(qtype, q, scl))
            qd = t.empty(q.shape, dtype=t.uint8, device="cuda")
            sd = t.empty(scl.shape, dtype=t.int16, device="cuda")
            qg.qrepack(qtype, blocks, rows, nb * 32, qd, sd)
            t.cuda.synchronize()
            del blocks
            return qd, sd

        def want(*names):
            return only is None or only in names

        g, l, tw, f, m = (w.get("gemv"), w.get("lmhead"), w.get("twins"), w.get("ffn"),
                          w.get("moe"))
        if want("gemv"):
            self.g_q, self.g_s = dq(synth.Q4_0, g["q"], g["scl"])
        if want("lmhead"):
            self.l_q, self.l_s = dq(synth.Q8_0, l["q"], l["scl"])
        if want("twins"):
            self.t_q, self.t_s = dq(synth.Q4_0, tw["q"], tw["scl"])
        if want("gateup"):
            self.f_qg, self.f_sg = dq(f["qtype"], f["qg"], f["sg"])
            self.f_qu, self.f_su = dq(f["qtype"], f["qu"], f["su"])
        if want("down"):
            self.f_qd, self.f_sd = dq(f["qtype"], f["qd"], f["sd"])
        if want("moe"):
            self.m = {}
            for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
                self.m[a], self.m[b] = dq(m["qtype"], m[a], m[b])
            self.m_sh = {}
            for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
                self.m_sh[a], self.m_sh[b] = dq(m["qtype"], m["shared"][a], m["shared"][b])
            ws = qg.qmoe_workspace_bytes(m["n_expert"], m["ffn"], m["hidden"], m["ncols"], m["topk"])
            self.m_ws = t.empty(ws, dtype=t.uint8, device="cuda")
            self.m_err = t.zeros(1, dtype=t.int32, device="cuda")
            self.m_uniq = t.empty(m["ncols"] * m["topk"], dtype=t.int32, device="cuda")

        # Per-step inputs and outputs. Each direction is one flat buffer (every
        # tensor a 256-byte aligned view into it), so a step moves its inputs
        # up in one copy and its outputs down in one copy. Two device sets: the
        # end-to-end loop copies one set while the kernels work on the other.
        self.host_in = {}
        if g is not None:
            self.host_in.update({"g_x": g["x"].view(np.int16), "g_y0": g["y0"]})
        if l is not None:
            self.host_in["l_x"] = l["x"].view(np.int16)
        if tw is not None:
            self.host_in["t_x"] = tw["x"].view(np.int16)
        if f is not None:
            self.host_in.update({"f_x": f["x"].view(np.int16), "f_y0": f["y0"]})
        if m is not None:
            self.host_in.update({"m_x": m["x"].view(np.int16), "m_ids": m["ids"], "m_rw": m["rw"]})
        tdt = {np.dtype(np.int16): t.int16, np.dtype(np.float32): t.float32,
               np.dtype(np.int32): t.int32}
        in_specs = [(k, v.shape, tdt[v.dtype]) for k, v in self.host_in.items()]
        out_specs = []
        if g is not None:
            out_specs.append(("g_y", (1, g["scl"].shape[0]), t.float32))
        if l is not None:
            out_specs.append(("l_y", (1, l["scl"].shape[0]), t.float32))
        if tw is not None:
            out_specs.append(("t_y", (8, tw["scl"].shape[0]), t.float32))
        if f is not None:
            out_specs += [("f_h", (16, 17408), t.float16), ("f_y", (16, 5120), t.float32)]
        if m is not None:
            out_specs.append(("m_y", (8, 2048), t.float32))

        def layout(specs):
            offs, off = {}, 0
            for k, shape, dt in specs:
                nbytes = int(np.prod(shape)) * t.empty((), dtype=dt).element_size()
                offs[k] = (off, nbytes, shape, dt)
                off = (off + nbytes + 255) // 256 * 256
            return offs, max(off, 256)

        def views(flat, offs):
            return {k: flat[o:o + n].view(dt).view(shape) for k, (o, n, shape, dt) in offs.items()}
        in_offs, in_total = layout(in_specs)
        out_offs, out_total = layout(out_specs)
        self.pin_in_flat = t.zeros(in_total, dtype=t.uint8).pin_memory()
        for k, v in views(self.pin_in_flat, in_offs).items():
            v.copy_(t.from_numpy(np.ascontiguousarray(self.host_in[k])))
        self.pin_out_flat = t.zeros(out_total, dtype=t.uint8).pin_memory()
        self.pin_out = views(self.pin_out_flat, out_offs)
        self.din_flat = [self.pin_in_flat.cuda() for _ in range(2)]
        self.dout_flat = [t.zeros(out_total, dtype=t.uint8, device="cuda") for _ in range(2)]
        self.din_sets = [views(fl, in_offs) for fl in self.din_flat]
        self.out_sets = [views(fl, out_offs) for fl in self.dout_flat]
        self.din, self.out = self.din_sets[0], self.out_sets[0]
        self.copy_stream = None

    def call(self, name: str, stream, buf: int = 0):
        qg, m = self.qg, self.w.get("moe")
        din, o = self.din_sets[buf], self.out_sets[buf]

        def x16(key):
            return din[key].view(self.torch.float16)
        if name == "gemv":
            qg.qgemv_q4_0(self.g_q, self.g_s, x16("g_x"), o["g_y"], din["g_y0"], stream)
        elif name == "lmhead":
            qg.qgemv_q8_0(self.l_q, self.l_s, x16("l_x"), o["l_y"], None, stream)
        elif name == "twins":
            qg.qgemv_q4_0(self.t_q, self.t_s, x16("t_x"), o["t_y"], None, stream)
        elif name == "gateup":
            qg.qffn_gate_up_silu(qg.Q4_0, self.f_qg, self.f_sg, self.f_qu, self.f_su,
                                 x16("f_x"), o["f_h"], stream)
        elif name == "down":
            qg.qgemm_cols(qg.Q4_0, self.f_qd, self.f_sd, o["f_h"], o["f_y"], din["f_y0"], stream)
        elif name == "moe":
            mm = self.m
            qg.qmoe_experts(qg.Q8_0, mm["qg"], mm["sg"], mm["qu"], mm["su"], mm["qd"], mm["sd"],
                            m["n_expert"], m["ffn"], m["hidden"], din["m_ids"],
                            din["m_rw"], x16("m_x"), o["m_y"], self.m_ws, y0=None,
                            shared=self.m_sh, err_flag=self.m_err, uniq_ids_out=self.m_uniq,
                            stream=stream)

    def step(self, stream, events=None, buf: int = 0):
        for i, name in enumerate(KERNELS):
            if events is not None:
                events[i].record(stream)
            self.call(name, stream, buf)
        if events is not None:
            events[len(KERNELS)].record(stream)

    def step_e2e(self, stream, i: int):
        """Step i end to end: its inputs go up from pinned host memory, the six
        calls run, its outputs come down to pinned host memory. Uploads and
        downloads run on two copy streams of their own (one in-order copy
        stream would queue step i+1's upload behind step i's download, and so
        behind step i's kernels), with device buffer set i % 2, so step i+1's
        upload and step i's download overlap the kernels of the neighbouring
        step; events keep every buffer's writes and reads in order."""
        t = self.torch
        if self.copy_stream is None:
            self.copy_stream = (t.cuda.Stream(), t.cuda.Stream())  # uploads, downloads
            self.ev = {k: [t.cuda.Event(), t.cuda.Event()] for k in ("up", "run", "down")}
            self.used = [False, False]
        (us, ds), b = self.copy_stream, i % 2
        ev = self.ev
        with t.cuda.stream(us):
            if i == 0:
                us.wait_stream(stream)           # the timed region starts before the first upload
            if self.used[b]:
                us.wait_event(ev["run"][b])      # step i-2 has finished reading set b
            self.din_flat[b].copy_(self.pin_in_flat, non_blocking=True)
            ev["up"][b].record(us)
        stream.wait_event(ev["up"][b])
        if self.used[b]:
            stream.wait_event(ev["down"][b])     # step i-2's outputs have left set b
        self.step(stream, buf=b)
        ev["run"][b].record(stream)
        with t.cuda.stream(ds):
            ds.wait_event(ev["run"][b])
            self.pin_out_flat.copy_(self.dout_flat[b], non_blocking=True)
            ev["down"][b].record(ds)
        self.used[b] = True

    def e2e_join(self, stream):
        """Make `stream` wait for every copy issued so far."""
        if self.copy_stream is not None:
            for cs in self.copy_stream:
                stream.wait_stream(cs)

    def e2e_bytes(self):
        """Bytes of the one upload and the one download of a step (the flat
        buffers: the tensors plus their alignment padding)."""
        return self.pin_in_flat.numel(), self.pin_out_flat.numel()


# -------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock, its maximum and the clock-event reasons of one GPU, read (never
    set) from two sources at once: `nvidia-smi -lms 50` and, every ~1 ms, NVML
    itself (libnvidia-ml, which ships with the driver), so that a timed region
    of a few milliseconds still holds samples."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits (nvml.h) of the reasons the record keeps
    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (time, sm, max, reasons set, source)
        self.proc = None
        self.thread = None
        self.nvml_thread = None
        self._halt = threading.Event()

    def start(self):
        self.nvml_thread = threading.Thread(target=self._nvml_loop, daemon=True)
        self.nvml_thread.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        if self.proc is not None:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        t0 = time.time()
        while (not self.samples and time.time() - t0 < 5 and
               (self.proc is not None or self.nvml_thread.is_alive())):
            time.sleep(0.02)

    def _nvml_loop(self):
        import ctypes as C
        try:
            lib = C.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        if lib.nvmlInit_v2() != 0:
            return
        try:
            h = C.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(C.c_uint(self.index), C.byref(h)) != 0:
                return
            reasons_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or
                          getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None))
            clock_sm = C.c_int(1)  # NVML_CLOCK_SM
            sm, mx, rs = C.c_uint(), C.c_uint(), C.c_ulonglong()
            if lib.nvmlDeviceGetMaxClockInfo(h, clock_sm, C.byref(mx)) != 0:
                return
            while not self._halt.is_set():
                if lib.nvmlDeviceGetClockInfo(h, clock_sm, C.byref(sm)) == 0:
                    reasons = set()
                    if reasons_fn is not None and reasons_fn(h, C.byref(rs)) == 0:
                        reasons = {n for bit, n in self.NVML_REASONS.items() if rs.value & bit}
                    self.samples.append((time.time(), float(sm.value), float(mx.value), reasons,
                                         "nvml"))
                time.sleep(0.001)
        finally:
            lib.nvmlShutdown()

    def _read(self):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.time(), sm, mx, reasons, "nvidia-smi"))

    def stop(self):
        self._halt.set()
        if self.nvml_thread is not None:
            self.nvml_thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = None
        if not inside:
            inside = [s for s in self.samples if t0 - 0.3 <= s[0] <= t1 + 0.3]
            note = "no sample inside the timed region; nearest samples within 0.3 s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "neither nvidia-smi nor NVML answered"}
        reasons = sorted(set().union(*[s[3] for s in inside]))
        d = {"sm_mhz": statistics.median(s[1] for s in inside),
             "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
             "samples": len(inside),
             "samples_by_source": {src: sum(1 for s in inside if s[4] == src)
                                   for src in ("nvml", "nvidia-smi")}}
        if note:
            d["note"] = note
        return d


# ---------------------------------------------------------- CPU oracle
def oracle_step_estimate(w: dict, frac: float, nthreads: int, h_for_down: np.ndarray) -> dict:
    """Time the oracle on every matrix of the step (frac = 1: all rows, measured,
    nothing scaled), or on an evenly spaced fraction of the rows of every dense
    matrix, each part's time scaled to its whole matrix: returns {kernel:
    seconds for the full kernel}. The MoE layer always runs whole."""
    import oracle
    oracle.build()
    est = {}

    def rows_sel(rows):
        if frac >= 1.0:
            return None, 1.0
        n = max(1, int(round(rows * frac)))
        return np.linspace(0, rows - 1, n).astype(np.int64), n / rows

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    g = w["gemv"]
    sel, f = rows_sel(5120)
    est["gemv"] = timed(lambda: oracle.matmul(g["qtype"], g["q"], g["scl"], g["x"], g["y0"],
                                              rows_sel=sel, nthreads=nthreads)) / f
    l = w["lmhead"]
    sel, f = rows_sel(l["rows"])
    est["lmhead"] = timed(lambda: oracle.matmul(l["qtype"], l["q"], l["scl"], l["x"], None,
                                                rows_sel=sel, nthreads=nthreads)) / f
    tw = w["twins"]
    sel, f = rows_sel(17408)
    est["twins"] = timed(lambda: oracle.matmul(tw["qtype"], tw["q"], tw["scl"], tw["x"], None,
                                               rows_sel=sel, nthreads=nthreads)) / f
    ff = w["ffn"]
    sel, f = rows_sel(17408)
    # the oracle's fused gate/up computes every row; time it on a row slice
    if sel is None:
        qg_s, sg_s, qu_s, su_s = ff["qg"], ff["sg"], ff["qu"], ff["su"]
    else:
        qg_s, sg_s = ff["qg"][sel], ff["sg"][sel]
        qu_s, su_s = ff["qu"][sel], ff["su"][sel]
    est["gateup"] = timed(lambda: oracle.ffn_gate_up_silu(ff["qtype"], qg_s, sg_s, qu_s, su_s,
                                                          ff["x"], nthreads=nthreads)) / f
    sel, f = rows_sel(5120)
    est["down"] = timed(lambda: oracle.matmul(ff["qtype"], ff["qd"], ff["sd"], h_for_down,
                                              ff["y0"], rows_sel=sel, nthreads=nthreads)) / f
    m = w["moe"]
    est["moe"] = timed(lambda: oracle.moe(m, nthreads=nthreads))
    return est


def oracle_h_for_down() -> np.ndarray:
    """f16 h [16][17408] fed to the oracle's down projection when it is timed
    (the values do not change its work)."""
    g = synth.rng(77)
    return (g.standard_normal((16, 17408)) * 0.05).astype(np.float16).view(np.uint16)


def cpu_baseline(w: dict, wb: dict, passes: int = 2) -> dict:
    """The oracle as it stands, timed on the whole step (every matrix, every
    row, the whole MoE layer) on all host cores, `passes` times."""
    nthreads = os.cpu_count() or 1
    h = oracle_h_for_down()
    times = []
    parts = {}
    for _ in range(passes):
        est = oracle_step_estimate(w, 1.0, nthreads, h)
        times.append(sum(est.values()))
        parts = est
    step_s = float(np.mean(times))
    return {
        "value": sum(wb.values()) / step_s / 1e9,
        "unit": UNIT,
        "cores": nthreads,
        "kind": "oracle",
        "sample": (f"f64 C oracle with {nthreads} threads on the whole step (every row of every "
                   f"matrix, the whole MoE layer), {passes} passes, measured (nothing scaled); "
                   "value = step weight bytes / mean pass time"),
        "cpu": platform.processor() or platform.machine(),
        "step_s": step_s,
        "part_s": {k: round(v, 4) for k, v in parts.items()},
    }


# ------------------------------------------------------------------ main
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(v: float, world: int, torch, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(step_bytes: float, region_ms: float, steps: int, world: int, torch,
                   device) -> tuple:
    """(ms per step, GB/s) of the whole job: the slowest rank's timed region
    sets the step time; every rank streamed `step_bytes` per step."""
    ms_per_step = max_over_ranks(region_ms, world, torch, device) / steps
    return ms_per_step, world * step_bytes / (ms_per_step * 1e-3) / 1e9


def run_case(args):
    """Profiling target: one call of the step, `--steps` times back to back, at
    full size or with its matrix cut to `--case-rows` rows; prints nothing but
    'ok'. For ncu captures of a single kernel on a case smaller than the step."""
    import torch
    import gemm_q4_q8_gb300 as qg
    from gemm_q4_q8_gb300 import build
    build.build()
    if args.case in EXTRA_CASES:
        return run_extra_case(args, torch, qg)
    w = make_workload(0, only=args.case)
    if args.case_rows:
        for key in ("gemv", "lmhead", "twins"):
            if key not in w:
                continue
            c = w[key]
            r = min(args.case_rows, c["scl"].shape[0])
            c["q"], c["scl"] = c["q"][:r], c["scl"][:r]
            if c.get("y0") is not None:
                c["y0"] = c["y0"][:, :r]
            c["rows"] = r
    gs = GpuStep(w, torch, only=args.case)
    stream = torch.cuda.current_stream()
    for _ in range(args.steps):
        gs.call(args.case, stream)
    torch.cuda.synchronize()
    print("ok", args.case)
    return 0


# The next steps around the step's calls, as single-kernel profiling targets
# at their config sizes: greedy argmax and top-40 over one column of 248,320
# logits; the MoE router (256 x 2048 f32, top-8) on one column; the small
# Q8_0 decode GEMV (2048 x 2048, one column, CUDA-core kernel), which the step
# does not contain; a tall Q4_0 / Q8_0 matrix (--case-rows rows, default
# 65,536, by 5,120; --case-cols columns, default 8), where the tensor-core
# kernel streams long enough to show its steady state; and the MoE layer at one
# column (the staged down kernel), cycling through its config's id sets.
EXTRA_CASES = ("argmax", "topk40", "router", "q8gemv2048", "q4tall", "q8tall", "moe1", "moe16")


def run_extra_case(args, torch, qg):
    g = synth.rng(11)
    stream = torch.cuda.current_stream()
    if args.case in ("argmax", "topk40"):
        x = torch.from_numpy(g.standard_normal((1, 248320)).astype(np.float32)).cuda()
        k = 1 if args.case == "argmax" else 40
        idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
        val = torch.empty((1, k), dtype=torch.float32, device="cuda")
        for _ in range(args.steps):
            if args.case == "argmax":
                qg.qargmax_f32(x, idx[:, 0], val[:, 0], stream)
            else:
                qg.qtopk_f32(x, k, idx, val, stream)
    elif args.case in ("q4tall", "q8tall"):
        qt = synth.Q4_0 if args.case == "q4tall" else synth.Q8_0
        c = synth.gemv_case(qt, args.case_rows or 65536, 5120, args.case_cols or 8,
                            residual=False, seed=5)
        blocks = torch.from_numpy(synth.to_gguf_blocks(qt, c["q"], c["scl"])).cuda()
        q = torch.empty(c["q"].shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(c["scl"].shape, dtype=torch.int16, device="cuda")
        qg.qrepack(qt, blocks, c["rows"], c["k"], q, sc)
        x = torch.from_numpy(c["x"].view(np.int16)).cuda().view(torch.float16)
        y = torch.empty((c["ncols"], c["rows"]), dtype=torch.float32, device="cuda")
        fn = qg.qgemv_q4_0 if qt == synth.Q4_0 else qg.qgemv_q8_0
        for _ in range(args.steps):
            fn(q, sc, x, y, None, stream)
    elif args.case in ("moe1", "moe16"):
        ct = ConfigTimer(torch, qg, None, None)
        name = "q8_moe_c1" if args.case == "moe1" else "q8_moe_c16"
        cfg = next(c for c in CONFIGS if c[0] == name)
        calls = ct.build(*cfg, False)[0]
        for i in range(args.steps):
            calls[i % len(calls)](stream)
    elif args.case == "q8gemv2048":
        c = synth.small_q8_gemv()
        blocks = torch.from_numpy(synth.to_gguf_blocks(c["qtype"], c["q"], c["scl"])).cuda()
        q = torch.empty(c["q"].shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(c["scl"].shape, dtype=torch.int16, device="cuda")
        qg.qrepack(c["qtype"], blocks, c["rows"], c["k"], q, sc)
        x = torch.from_numpy(c["x"].view(np.int16)).cuda().view(torch.float16)
        y = torch.empty((1, c["rows"]), dtype=torch.float32, device="cuda")
        for _ in range(args.steps):
            qg.qgemv_q8_0(q, sc, x, y, None, stream)
    else:
        w = torch.from_numpy((g.standard_normal((256, 2048)) * 0.02).astype(np.float32)).cuda()
        x = torch.from_numpy(synth.draw_x(g, 1, 2048).view(np.int16)).cuda().view(torch.float16)
        ids = torch.empty((1, 8), dtype=torch.int32, device="cuda")
        rw = torch.empty((1, 8), dtype=torch.float32, device="cuda")
        for _ in range(args.steps):
            qg.qmoe_router(w, x, 8, ids, rw, stream=stream)
    torch.cuda.synchronize()
    print("ok", args.case)
    return 0


# ------------------------------------------------------------ per-config
CONFIGS = (
    # name, kind, qtype, rows, k, ncols, residual
    ("q8_gemv_2048_c1", "gemv", synth.Q8_0, 2048, 2048, 1, False),
    ("q4_gemv_5120_c1_y0", "gemv", synth.Q4_0, 5120, 5120, 1, True),
    ("q8_lmhead_248320_c1", "gemv", synth.Q8_0, 248320, 5120, 1, False),
    ("q4_lmhead_248320_c1", "gemv", synth.Q4_0, 248320, 5120, 1, False),
    ("q4_twins_5120_c2", "gemv", synth.Q4_0, 5120, 5120, 2, False),
    ("q4_twins_5120_c4", "gemv", synth.Q4_0, 5120, 5120, 4, False),
    ("q4_twins_5120_c8", "gemv", synth.Q4_0, 5120, 5120, 8, False),
    ("q4_twins_17408_c2", "gemv", synth.Q4_0, 17408, 5120, 2, False),
    ("q4_twins_17408_c4", "gemv", synth.Q4_0, 17408, 5120, 4, False),
    ("q4_twins_17408_c8", "gemv", synth.Q4_0, 17408, 5120, 8, False),
    ("q8_twins_17408_c8", "gemv", synth.Q8_0, 17408, 5120, 8, False),
    ("q4_ffn_gateup_17408_c16", "gateup", synth.Q4_0, 17408, 5120, 16, False),
    ("q4_ffn_down_5120x17408_c16_y0", "cols", synth.Q4_0, 5120, 17408, 16, True),
    ("q8_moe_c1", "moe", synth.Q8_0, 0, 0, 1, False),
    ("q8_moe_c8", "moe", synth.Q8_0, 0, 0, 8, False),
    ("q8_moe_c16", "moe", synth.Q8_0, 0, 0, 16, False),
    # sampling over LM-head logits (next steps after the LM head): rows = n, k = top-k
    ("argmax_lmhead_248320_c1", "argmax", None, 248320, 1, 1, False),
    ("argmax_lmhead_248320_c8", "argmax", None, 248320, 1, 8, False),
    ("topk40_lmhead_248320_c1", "topk", None, 248320, 40, 1, False),
    ("topk40_lmhead_248320_c8", "topk", None, 248320, 40, 8, False),
    # MoE router (f32 [256, 2048] router weights) + top-8 + softmax: rows = experts
    ("router_256x2048_top8_c1", "router", None, 256, 2048, 1, False),
    ("router_256x2048_top8_c8", "router", None, 256, 2048, 8, False),
    ("router_256x2048_top8_c16", "router", None, 256, 2048, 16, False),
)
# The configs the default bench line reports (the workload's configs at every
# column count it names); --configs times all of CONFIGS.
DEFAULT_CONFIGS = ("q8_gemv_2048_c1", "q4_gemv_5120_c1_y0", "q8_lmhead_248320_c1",
                   "q4_twins_5120_c2", "q4_twins_5120_c4", "q4_twins_5120_c8",
                   "q4_twins_17408_c2", "q4_twins_17408_c4", "q4_twins_17408_c8",
                   "q8_twins_17408_c8", "q4_ffn_gateup_17408_c16",
                   "q4_ffn_down_5120x17408_c16_y0", "q8_moe_c1", "q8_moe_c8", "q8_moe_c16")
L2_BYTES = 129 * 2**20


class ConfigTimer:
    """Each config of the workload alone: CUDA-graph replays of back-to-back
    calls that cycle through enough distinct weight copies (>= 4x L2, at most
    16, or one copy when a single one is larger) that L2 holds none of them;
    MoE calls cycle through 8 id sets. 20 warm-up calls; per replay, the mean
    call time; median and p10/p90 over the replays.

    Device matrices come from the step's own buffers where the step has the
    same matrix (rotating copies are device-to-device clones of it); the rest
    are drawn with the same distributions and repacked on the GPU."""

    def __init__(self, torch, qg, gs, w):
        self.t, self.qg, self.gs, self.w = torch, qg, gs, w
        self.stream = torch.cuda.current_stream()

    def d(self, a):
        return self.t.from_numpy(np.ascontiguousarray(a)).cuda()

    def dq(self, qtype, q, scl):
        t = self.t
        rows, nb = scl.shape
        blocks = self.d(synth.to_gguf_blocks(qtype, q, scl))
        qd = t.empty(q.shape, dtype=t.uint8, device="cuda")
        sd = t.empty(scl.shape, dtype=t.int16, device="cuda")
        self.qg.qrepack(qtype, blocks, rows, nb * 32, qd, sd)
        t.cuda.synchronize()
        return qd, sd

    def host_matrices(self, kind, qt, rows, k):
        """Host (quants, scales) of the config's matrices, from the workload
        when it holds that matrix; None when it must be drawn."""
        w = self.w
        if w is None:
            return None
        if kind == "gateup" and (qt, rows, k) == (synth.Q4_0, 17408, 5120) and "ffn" in w:
            f = w["ffn"]
            return [(f["qg"], f["sg"]), (f["qu"], f["su"])]
        if kind == "cols" and (qt, rows, k) == (synth.Q4_0, 5120, 17408) and "ffn" in w:
            return [(w["ffn"]["qd"], w["ffn"]["sd"])]
        if kind == "gemv":
            for key in ("gemv", "lmhead", "twins"):
                c = w.get(key)
                if c is not None and (c["qtype"], c["scl"].shape[0], c["k"]) == (qt, rows, k):
                    return [(c["q"], c["scl"])]
        return None

    def device_matrix(self, kind, qt, rows, k, mats):
        """Device copies of the config's matrices: the step's own when it has
        them, else repacked from `mats`."""
        gs = self.gs
        if gs is not None:
            if kind == "gateup" and hasattr(gs, "f_qg") and (qt, rows, k) == (synth.Q4_0, 17408, 5120):
                return [(gs.f_qg, gs.f_sg), (gs.f_qu, gs.f_su)]
            if kind == "cols" and hasattr(gs, "f_qd") and (qt, rows, k) == (synth.Q4_0, 5120, 17408):
                return [(gs.f_qd, gs.f_sd)]
            if kind == "gemv":
                for key, attr in (("gemv", "g"), ("lmhead", "l"), ("twins", "t")):
                    c = self.w.get(key) if self.w else None
                    if (c is not None and hasattr(gs, attr + "_q") and
                            (c["qtype"], c["scl"].shape[0], c["k"]) == (qt, rows, k)):
                        return [(getattr(gs, attr + "_q"), getattr(gs, attr + "_s"))]
        return [self.dq(qt, q, sc) for (q, sc) in mats]

    def build(self, name, kind, qt, rows, k, ncols, residual, with_oracle):
        """(calls, weight bytes, total bytes, oracle fns or None, oracle row
        fraction, extra keys) of one config."""
        t, qg = self.t, self.qg
        g = synth.rng(1)
        calls = []
        ncores = os.cpu_count() or 1
        o_fn, o_frac = None, 1.0
        import oracle
        if kind in ("argmax", "topk"):
            n, kk = rows, k
            xs_np = [g.standard_normal((ncols, n)).astype(np.float32) for _ in range(4)]
            xs_d = [self.d(a) for a in xs_np]
            ib = t.empty((ncols, kk), dtype=t.int32, device="cuda")
            vb = t.empty((ncols, kk), dtype=t.float32, device="cuda")
            for a in xs_d:
                if kind == "argmax":
                    calls.append(lambda s, a=a: qg.qargmax_f32(a, ib[:, 0], vb[:, 0], s))
                else:
                    calls.append(lambda s, a=a: qg.qtopk_f32(a, kk, ib, vb, s))
            wbytes = ncols * n * 4  # logits read (no weights)
            tbytes = wbytes + ncols * kk * 8  # + indices and values written
            if with_oracle:
                o_fn = {th: ((lambda: oracle.argmax(xs_np[0])) if kind == "argmax"
                             else (lambda: oracle.topk(xs_np[0], kk))) for th in (1, ncores)}
            extra = {"bytes_are": "logits read", "k": kk}
        elif kind == "router":
            E, hid = rows, k
            wr_np = [(g.standard_normal((E, hid)) * 0.02).astype(np.float32) for _ in range(4)]
            x_np = synth.draw_x(g, ncols, hid)
            wr = [self.d(a) for a in wr_np]
            x = self.d(x_np.view(np.int16)).view(t.float16)
            ib = t.empty((ncols, 8), dtype=t.int32, device="cuda")
            rb = t.empty((ncols, 8), dtype=t.float32, device="cuda")
            for a in wr:
                calls.append(lambda s, a=a: qg.qmoe_router(a, x, 8, ib, rb, stream=s))
            wbytes = E * hid * 4  # f32 router weights
            tbytes = wbytes + ncols * hid * 2 + ncols * 8 * 8  # + x, ids and weights out

            def o_router(i=0):
                lg, _ = oracle.router_logits(wr_np[i], x_np)
                _, v = oracle.topk(lg.astype(np.float32), 8)
                return [oracle.softmax(r) for r in v]
            if with_oracle:
                o_fn = {th: o_router for th in (1, ncores)}
            extra = {"bytes_are": "f32 router weights", "topk": 8}
        elif kind == "moe":
            gs = self.gs
            m_host = self.w["moe"] if (self.w is not None and "moe" in self.w) else synth.moe_layer(8, seed=2)
            if gs is not None and hasattr(gs, "m"):
                dm, sh = gs.m, gs.m_sh
            else:
                dm, sh = {}, {}
                for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
                    dm[a], dm[b] = self.dq(qt, m_host[a], m_host[b])
                    sh[a], sh[b] = self.dq(qt, m_host["shared"][a], m_host["shared"][b])
            E, ffn, hid = m_host["n_expert"], m_host["ffn"], m_host["hidden"]
            ws = t.empty(qg.qmoe_workspace_bytes(E, ffn, hid, ncols, 8), dtype=t.uint8,
                         device="cuda")
            gi = synth.rng(9)
            idn = [np.stack([gi.choice(E, 8, replace=False) for _ in range(ncols)]).astype(np.int32)
                   for _ in range(8)]
            x_np = synth.draw_x(gi, ncols, hid)
            _, rw_np = synth.draw_routing(gi, ncols, E, 8)
            uniq = float(np.mean([len(np.unique(i)) for i in idn]))
            wbytes = (uniq + 1) * 3 * synth.weight_bytes(qt, ffn, hid)
            # + x, y, ids, rw, and h (f16 [ncols][9][512]) written then read
            tbytes = wbytes + ncols * hid * (2 + 4) + ncols * 8 * 8 + 2 * ncols * 9 * ffn * 2
            ids = [self.d(i) for i in idn]
            rw, x = self.d(rw_np), self.d(x_np.view(np.int16)).view(t.float16)
            y = t.empty((ncols, hid), dtype=t.float32, device="cuda")
            for i in range(8):
                calls.append(lambda s, i=i: qg.qmoe_experts(
                    qt, dm["qg"], dm["sg"], dm["qu"], dm["su"], dm["qd"], dm["sd"], E, ffn, hid,
                    ids[i], rw, x, y, ws, shared=sh, stream=s))
            if with_oracle:
                mc = dict(m_host, ncols=ncols, ids=idn[0], rw=rw_np, x=x_np, y0=None)
                o_fn = {th: (lambda th=th: oracle.moe(mc, nthreads=th)) for th in (1, ncores)}
            extra = {"distinct_experts_mean": uniq}
        else:
            nmat = 2 if kind == "gateup" else 1
            wb1 = nmat * synth.weight_bytes(qt, rows, k)
            ncopy = int(min(16, max(1, np.ceil(4 * L2_BYTES / wb1))))
            mats = self.host_matrices(kind, qt, rows, k)
            if mats is None:
                mats = [synth.draw_matrix(g, qt, rows, k) for _ in range(nmat)]
            x_np = synth.draw_x(g, ncols, k)
            y0_np = synth.draw_y0(g, ncols, rows) if residual else None
            first = self.device_matrix(kind, qt, rows, k, mats)
            dev_mats = [first] + [[(a.clone(), sa.clone()) for (a, sa) in first]
                                  for _ in range(ncopy - 1)]
            x = self.d(x_np.view(np.int16)).view(t.float16)
            y0 = self.d(y0_np) if residual else None
            if kind == "gateup":
                h = t.empty((ncols, rows), dtype=t.float16, device="cuda")
                for c in range(ncopy):
                    (a, sa), (b, sb) = dev_mats[c]
                    calls.append(lambda s, a=a, sa=sa, b=b, sb=sb: qg.qffn_gate_up_silu(
                        qt, a, sa, b, sb, x, h, s))
            else:
                y = t.empty((ncols, rows), dtype=t.float32, device="cuda")
                fn = qg.qgemm_cols if kind == "cols" else (
                    qg.qgemv_q4_0 if qt == synth.Q4_0 else qg.qgemv_q8_0)
                for c in range(ncopy):
                    (a, sa), = dev_mats[c]
                    if kind == "cols":
                        calls.append(lambda s, a=a, sa=sa: fn(qt, a, sa, x, y, y0, s))
                    else:
                        calls.append(lambda s, a=a, sa=sa: fn(a, sa, x, y, y0, s))
            wbytes = wb1
            # + x read, y (f32) or h (f16) written, y0 read
            out_b = ncols * rows * (2 if kind == "gateup" else 4)
            tbytes = wbytes + ncols * k * 2 + out_b + (ncols * rows * 4 if residual else 0)
            if with_oracle:
                # the oracle runs on an evenly spaced row sample of about 25 M
                # weights (the whole matrix when it is smaller), scaled to all rows
                n_s = max(1, min(rows, int(25e6 / (nmat * k))))
                sel = np.linspace(0, rows - 1, n_s).astype(np.int64)
                o_frac = n_s / rows
                if kind == "gateup":
                    (q1, s1), (q2, s2) = mats
                    o_fn = {th: (lambda th=th: oracle.ffn_gate_up_silu(
                        qt, q1[sel], s1[sel], q2[sel], s2[sel], x_np, nthreads=th))
                        for th in (1, ncores)}
                else:
                    (q1, s1), = mats
                    o_fn = {th: (lambda th=th: oracle.matmul(qt, q1, s1, x_np, y0_np, rows_sel=sel,
                                                           nthreads=th)) for th in (1, ncores)}
            extra = {"weight_copies": ncopy}
        return calls, wbytes, tbytes, o_fn, o_frac, extra

    def time_calls(self, calls):
        """Per-call µs of back-to-back graph replays: (median, p10, p90, calls timed)."""
        t = self.t
        reps = max(len(calls), 16)
        gcap = t.cuda.Stream()
        with t.cuda.stream(gcap):
            for i in range(20):
                calls[i % len(calls)](gcap)
        t.cuda.synchronize()
        graph = t.cuda.CUDAGraph()
        with t.cuda.graph(graph, stream=gcap):
            for i in range(reps):
                calls[i % len(calls)](gcap)
        for _ in range(3):
            graph.replay()
        t.cuda.synchronize()
        nrep = max(13, -(-200 // reps))
        evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True))
               for _ in range(nrep)]
        for e0, e1 in evs:
            e0.record(self.stream)
            graph.replay()
            e1.record(self.stream)
        t.cuda.synchronize()
        per_call = np.array([e0.elapsed_time(e1) * 1e3 / reps for e0, e1 in evs])
        del graph
        return (float(np.median(per_call)), float(np.percentile(per_call, 10)),
                float(np.percentile(per_call, 90)), int(nrep * reps))

    def run(self, names, with_oracle, peak, peak_kind):
        """One dict per config name (in CONFIGS order)."""
        out = []
        ncores = os.cpu_count() or 1
        for name, kind, qt, rows, k, ncols, residual in CONFIGS:
            if name not in names:
                continue
            calls, wbytes, tbytes, o_fn, o_frac, extra = self.build(
                name, kind, qt, rows, k, ncols, residual, with_oracle)
            med, p10, p90, ncalls = self.time_calls(calls)
            line = {"config": name, "us_median": med, "us_p10": p10, "us_p90": p90,
                    "timed_calls": ncalls, "weight_bytes": wbytes, "total_bytes": tbytes,
                    "GBps": wbytes / (med * 1e-6) / 1e9,
                    "frac_of_measured_hbm": wbytes / (med * 1e-6) / 1e9 / peak,
                    "peak_kind": peak_kind,
                    "frac_of_8TBps_nominal": wbytes / (med * 1e-6) / 8e12}
            if o_fn is not None:
                def oracle_us(fn):
                    t0 = time.perf_counter()
                    fn()
                    return (time.perf_counter() - t0) / o_frac * 1e6
                line.update({"oracle_us_1thread": oracle_us(o_fn[1]),
                             "oracle_us_all_threads": oracle_us(o_fn[ncores]),
                             "oracle_threads": ncores,
                             "oracle_sample": ("whole layer" if kind == "moe" else
                                               f"{o_frac:.3f} of the rows, scaled")})
            line.update(extra)
            out.append(line)
            del calls
            self.t.cuda.empty_cache()
        return out


def run_configs(args):
    """Every config of CONFIGS alone (ConfigTimer), with the oracle's time per
    call beside it (rows sampled and scaled; 1 thread and all host threads).
    One JSON line per config."""
    import torch
    import gemm_q4_q8_gb300 as qg
    import oracle
    from gemm_q4_q8_gb300 import build
    build.build()
    oracle.build()
    peak, peak_kind = peaks()
    names = [c[0] for c in CONFIGS if not args.config_filter or args.config_filter in c[0]]
    w = make_workload(0)
    gs = GpuStep(w, torch)
    for line in ConfigTimer(torch, qg, gs, w).run(names, True, peak, peak_kind):
        print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    """The oracle timed on this host's cores (the reference arm of this tier)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = make_workload(0)
    uniq = len(np.unique(w["moe"]["ids"]))
    wb = weight_bytes(w, uniq)
    frac = args.ref_frac
    nthreads = os.cpu_count() or 1
    h = oracle_h_for_down()
    for _ in range(args.warmup):
        oracle_step_estimate(w, frac, nthreads, h)
    times = []
    for _ in range(args.steps):
        est = oracle_step_estimate(w, frac, nthreads, h)
        times.append(sum(est.values()))
    step_s = float(np.mean(times))
    value = sum(wb.values()) / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                         "sample": ("each step one whole pass of the oracle over the step "
                                    "(every row of every matrix, the whole MoE layer), measured"
                                    if frac >= 1.0 else
                                    f"{frac:.4f} of the rows of every dense matrix per step, "
                                    "whole MoE layer; times scaled to full matrices")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # default: 1000 device steps (~0.3 s timed, several clock samples); the
    # reference arm's steps are whole oracle passes of ~1.2 s each, so 20 there
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ref-frac", type=float, default=1.0,
                    help="fraction of the rows the reference arm's oracle runs (1: all)")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=KERNELS + EXTRA_CASES, default=None,
                    help="profiling target: run only this call (see run_case)")
    ap.add_argument("--case-rows", type=int, default=0)
    ap.add_argument("--case-cols", type=int, default=0)
    ap.add_argument("--configs", action="store_true",
                    help="time every workload config alone (one JSON line each)")
    ap.add_argument("--config-filter", default="")
    args = ap.parse_args(argv)
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else (200 if args.case else 1000)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    if args.configs:
        return run_configs(args)

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from gemm_q4_q8_gb300 import build
    build.build()
    import gemm_q4_q8_gb300 as qg

    w = make_workload(0)
    uniq = len(np.unique(w["moe"]["ids"]))
    wb = weight_bytes(w, uniq)
    step_bytes = sum(wb.values())
    gs = GpuStep(w, torch)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        gs.step(stream)
    torch.cuda.synchronize()

    # The step is captured once into a CUDA graph (the library's calls are
    # capture-safe: no allocation, no synchronisation) and the timed region
    # replays it, so no per-call host work sits between the kernels.
    cap = torch.cuda.Stream()
    step_graph = torch.cuda.CUDAGraph()
    l_before = qg.qg_kernel_launches()
    with torch.cuda.graph(step_graph, stream=cap):
        gs.step(cap)
    launches_per_step = qg.qg_kernel_launches() - l_before
    # Each call also gets a graph of its own, for the per-kernel breakdown:
    # replayed back to back with a CUDA event between consecutive graphs.
    graphs = []
    for name in KERNELS:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            gs.call(name, cap)
        graphs.append(g)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step_graph.replay()
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()

    # ---- device-resident timed region: whole-step graph replays
    clk = ClockSampler(local)
    clk.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    launches = launches_per_step * args.steps
    if world > 1:
        torch.distributed.barrier()
    # A second window of about a second of back-to-back step replays (not part
    # of the timed region), so the clock record has samples under this load
    # however short the timed region is.
    n_sus = int(max(1, min(20000, 1.0 / max(e0.elapsed_time(e1) * 1e-3 / args.steps, 1e-6))))
    t_sus0 = time.time()
    for i in range(n_sus):
        step_graph.replay()
    torch.cuda.synchronize()
    t_sus1 = time.time()
    clk.stop()
    ms_per_step, value = whole_job_rate(step_bytes, e0.elapsed_time(e1), args.steps, world,
                                        torch, device)

    # ---- per-kernel breakdown: per-call graphs with events between them
    nb_steps = max(3, min(args.steps, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)]
          for _ in range(nb_steps)]
    for i in range(nb_steps):
        for j, g in enumerate(graphs):
            ev[i][j].record(stream)
            g.replay()
        ev[i][len(KERNELS)].record(stream)
    torch.cuda.synchronize()
    per_kernel_ms = {name: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1])
                                          for i in range(nb_steps)]))
                     for j, name in enumerate(KERNELS)}

    # ---- end to end through the public API from pinned host buffers
    e2e_steps = max(3, min(args.steps, 100))
    for i in range(2):
        gs.step_e2e(stream, i)
    gs.e2e_join(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(e2e_steps):
        gs.step_e2e(stream, i)
    gs.e2e_join(stream)   # the last step's outputs are on the host before f1
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, torch, device) / e2e_steps
    bi, bo = gs.e2e_bytes()
    # the outputs that reached the host equal the device-resident step's, bit for bit
    # (same inputs, deterministic kernels)
    e2e_match = all(torch.equal(gs.pin_out[k], v.cpu()) for k, v in gs.out_sets[0].items())

    peak, peak_kind = peaks()
    lm_ms = per_kernel_ms["lmhead"]
    achieved = wb["lmhead"] / (lm_ms * 1e-3) / 1e9
    breakdown = {}
    for name in KERNELS:
        gbs = wb[name] / (per_kernel_ms[name] * 1e-3) / 1e9
        breakdown[name] = {"us": per_kernel_ms[name] * 1e3, "weight_bytes": wb[name],
                           "GBps": gbs, "frac_of_measured_hbm": gbs / peak}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "weights": "Q4_0/Q8_0 blocks, f16 scales",
                   "activations": "f16", "accumulate": "f32",
                   "step_weight_bytes": step_bytes,
                   "step_total_bytes": step_bytes + sum(activation_bytes().values()),
                   "moe_unique_experts": uniq,
                   "l2": "inputs larger than L2: each step streams ~1.8 GB of distinct weights "
                         "(L2 is 129 MB), so no step finds the previous step's weights in L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "lmhead (qgemv_q8_0, 248320x5120, 1 column)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": lmhead_traffic(w["lmhead"]["rows"]),
                     "traffic_note": "dram read+write bytes per launch, ncu capture of a "
                                     "65,536-row cut scaled by rows (committed LM-head "
                                     "capture summary under profiles/)"},
        "breakdown": breakdown,
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": e2e_ms, "outputs_match_device_step": bool(e2e_match)},
        "gpu_launches": int(launches),
        "timing": "value: one CUDA graph per step (all calls), replayed back to back; "
                  "breakdown: one graph per call, replayed back to back with a CUDA event "
                  "between consecutive graphs (includes each graph's launch gap); e2e: eager "
                  "calls, every step's inputs uploaded from and outputs downloaded to pinned "
                  "host memory on a copy stream (two device buffer sets, so one step's copies "
                  "overlap the neighbouring step's kernels), all inside the timed region",
        "clocks": clk.summary(t_wall0, t_wall1),
        "clocks_sustained": dict(clk.summary(t_sus0, t_sus1), steps=n_sus,
                                 note="untimed window of back-to-back step replays right "
                                      "after the timed region"),
    }
    if rank == 0 and not args.no_per_config:
        # every workload config alone, graph replays over rotating weight copies
        del graphs
        torch.cuda.empty_cache()
        pc = ConfigTimer(torch, qg, gs, w).run(DEFAULT_CONFIGS, False, peak, peak_kind)
        line["per_config"] = {
            d["config"]: {"us": round(d["us_median"], 3), "us_p10": round(d["us_p10"], 3),
                          "us_p90": round(d["us_p90"], 3), "weight_bytes": d["weight_bytes"],
                          "GBps": round(d["GBps"], 1),
                          "frac_of_measured_hbm": round(d["frac_of_measured_hbm"], 4)}
            for d in pc}
        line["per_config_timing"] = ("each config alone: CUDA-graph replays of back-to-back "
                                     "calls cycling through distinct weight copies (>= 4x L2, "
                                     "at most 16; one when a copy is larger) and 8 MoE id sets; "
                                     "median per call over >= 13 replays")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, wb)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
