"""Benchmark of the MoE expert layer on GB300: one JSON line on rank 0.

A step is one pass of the whole layer over one batch: route, dispatch, gate_up GEMM + SwiGLU,
down GEMM (and the shared expert's two GEMMs when the workload has one), combine - the same
C-ABI calls moe_forward makes, issued one by one so CUDA events between them time each kernel
family on the stream it runs on. Inputs are seeded synthetic tensors resident in HBM before the
timed region; a 256 MB write (twice the L2) precedes every timed step, outside its events, so
no step finds the previous step's weights or activations in L2.

The headline line is the Mixtral-shaped layer (the default --config); `per_config` adds, from
the same run, every other workload: gpt-oss-shaped, Llama-4-Scout-shaped with its shared expert,
the decode batches T = 1, 8 and 64 (µs per layer against HBM bandwidth) and the tiny fp32 layer,
each with its stage times, the roofline of its dominant kernel and its own CPU-oracle sample.

e2e: the same metric through moe_forward with host buffers: every step copies x and the logits
from pinned host memory, runs the layer, and copies the output back.

--impl reference: the CPU oracle (float64 numpy, the test reference) timed on the host cores
on a bounded token sample of the same workload.

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own GPU (weak scaling, no
collective on the data path); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MoE layer tokens/s & expert-GEMM TFLOP/s on 1 GB300; decode µs/layer vs HBM "
          "GB/s")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral_8x7b")
    ap.add_argument("--T", type=int, default=None, help="override the token count")
    ap.add_argument("--E", type=int, default=None,
                    help="override the expert count (smaller cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=None, help="tokens in the CPU sample")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the selected workload only (no per_config object)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the timed region runs.
    Read-only NVML queries every 2 ms (libnvidia-ml through ctypes); nvidia-smi as a fallback."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.index = index
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._proc = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, h, reasons_fn

    def _loop_nvml(self):
        import ctypes
        lib, h, reasons_fn = self._nvml
        c, m = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0 and \
                    reasons_fn(h, ctypes.byref(m)) == 0:
                self.samples.append((float(c.value), int(m.value)))
            time.sleep(self.period)

    def _loop_smi(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                self.max_mhz = float(parts[1])
                mask = int(parts[2], 16)
                self.samples.append((float(parts[0]), mask))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        try:
            self._nvml = self._nvml_open()
        except OSError:
            self._nvml = None
        if self._nvml is not None:
            self._t = threading.Thread(target=self._loop_nvml, daemon=True)
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self._t = threading.Thread(target=self._loop_smi, daemon=True)
            except OSError:
                self._t = None
        if self._t is not None:
            self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, mask in self.samples:
            for bit, name in self.REASONS.items():
                if mask & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(v for v, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# ------------------------------------------------------------------------------------------------
# CPU oracle on a token sample (the baseline and the reference arm)
# ------------------------------------------------------------------------------------------------
def cpu_oracle_run(cfg, inp_host, tokens):
    """The oracle's whole layer on the first `tokens` tokens; returns wall seconds."""
    import numpy as np

    from oracle import moe_oracle as o

    class Widen:
        def __init__(self, t):
            self.t = t

        def __len__(self):
            return self.t.shape[0]

        def __getitem__(self, e):
            return self.t[e].double().numpy()

    x = inp_host["x"][:tokens].double().numpy()
    logits = inp_host["logits"][:tokens].numpy()
    sh = inp_host.get("w_shared_gate_up")
    t0 = time.perf_counter()
    o.forward(x, logits, Widen(inp_host["w_gate_up"]), Widen(inp_host["w_down"]), cfg.k,
              cfg.score_fn, cfg.renormalize, cfg.scale_input, True,
              None if sh is None else sh.double().numpy(),
              None if sh is None else inp_host["w_shared_down"].double().numpy())
    return time.perf_counter() - t0


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


def default_sample(cfg):
    # about 10-30 s of the oracle on a 16-core host: it sustains roughly 300 GFLOP/s of float64
    # matrix products there, plus the per-expert widening of the weights
    per_token = 6.0 * cfg.d * cfg.I * cfg.k + 6.0 * cfg.d * cfg.I_shared
    return int(max(8, min(cfg.T, 3e12 / per_token)))


def host_inputs(cfg, dev_inputs):
    out = {}
    for k_, v in dev_inputs.items():
        out[k_] = None if v is None else v.cpu()
    return out


# ------------------------------------------------------------------------------------------------
# source file of each grouped GEMM kernel (traffic.json is keyed by it)
GEMM_SOURCES = {"tc_grouped_gemm": "gemm_tc.cu", "tc_grouped_gemm_2sm": "gemm_tc_2sm.cu",
                "tc_grouped_gemm_swap": "gemm_tc_swap.cu",
                "tc_grouped_gemm_swap_pair": "gemm_tc_swap_pair.cu"}


def traffic_for(kernel_file: str, workload: str):
    """DRAM bytes per launch of the kernel on this workload from the committed ncu summary, if it
    was taken on the current source of the kernel (matching sha256), else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "routing_dispatch_grouped_gb300", "csrc", kernel_file)
    if not os.path.exists(p) or not os.path.exists(src):
        return None, None
    with open(p) as f:
        d = json.load(f)
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    ent = d.get(kernel_file)
    if not ent or ent.get("sha256") != h:
        return None, None
    return ent.get("by_workload", {}).get(workload), ent


def reduce_max(x: float, device) -> float:
    """Maximum of a per-rank float over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_tokens(T: int, rank: int, world: int):
    """Token range [a, b) of one rank when a batch is split across ranks."""
    per = (T + world - 1) // world
    a = min(T, rank * per)
    return a, min(T, a + per)


def decode_name(T):
    return f"decode_T{T}"


def workload_config(name, T=None, E=None):
    """The synth workload of a bench name (decode_T<n> = the decode shape at T = n)."""
    from routing_dispatch_grouped_gb300 import synth
    if name.startswith("decode_T"):
        T = int(name[len("decode_T"):]) if T is None else T
        name = "decode"
    cfg = synth.CONFIGS[name]
    if T is not None:
        cfg = cfg.with_T(T)
    if E is not None:
        cfg = dataclasses.replace(cfg, E=E, name=f"{cfg.name}@E{E}")
    return cfg


def fp32_alu_peak_tflops(sm_max_mhz):
    """FP32 FMA peak of the GPU: 152 SMs x 128 FP32 lanes x 2 FLOP per FMA x the maximum SM
    clock (the tiny fp32 layer runs on the FP32 pipes)."""
    return 152 * 128 * 2 * sm_max_mhz * 1e6 / 1e12


class Layer:
    """One workload on the device: inputs, packed weights, workspaces and the timed forms."""

    def __init__(self, cfg, dev, steps, warmup, world):
        import torch

        from routing_dispatch_grouped_gb300 import moe, synth
        self.cfg, self.dev, self.steps, self.warmup, self.world = cfg, dev, steps, warmup, world
        self.moe = moe
        self.inp = synth.make_inputs(cfg, dev)
        T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
        # expert weights are repacked once, as at model load (moe_pack_weights); bf16 layers
        self.packed = cfg.dtype == torch.bfloat16
        self.wts = {}
        for n_ in ("w_gate_up", "w_down", "w_shared_gate_up", "w_shared_down"):
            w_ = self.inp[n_]
            if w_ is not None and self.packed:
                w_ = moe.pack_weights(w_, moe.W_GATE_UP if "gate_up" in n_ else moe.W_DOWN)
            self.wts[n_] = w_
        torch.cuda.synchronize()
        self.flags = (moe.RENORMALIZE if cfg.renormalize else 0) | (
            moe.SCALE_INPUT if cfg.scale_input else 0)
        dt = cfg.dtype
        self.stream = torch.cuda.current_stream(dev)
        self.ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.out = torch.empty(T, d, dtype=dt, device=dev)
        self.ws = torch.empty(moe.moe_forward_workspace_size(T, d, E, k, I, Is, dt),
                              dtype=torch.uint8, device=dev)
        self.v = moe.forward_workspace_views(self.ws, T, d, E, k, I, Is, dt)
        self.dws = torch.empty(moe.moe_dispatch_workspace_size(T, E, k), dtype=torch.uint8,
                               device=dev)
        self.gws = torch.empty(256, dtype=torch.uint8, device=dev)
        # between timed steps: write a buffer twice the L2 size so no step finds the previous
        # step's weights or activations cached (decode touches less than the L2 holds)
        self.l2_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.stages = ["route", "dispatch", "gate_up", "down"] + (
            ["shared_gate_up", "shared_down"] if Is else []) + ["combine"]

    def flush_l2(self):
        self.l2_buf.fill_(1)

    def events(self, n):
        import torch
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def step(self, ev=None):
        """The layer as its separate C-ABI calls, with an event after each."""
        moe, cfg, inp, v, wts, st = self.moe, self.cfg, self.inp, self.v, self.wts, self.stream

        def mark(i):
            if ev is not None:
                ev[i].record(st)
        k, E, Is = cfg.k, cfg.E, cfg.I_shared
        mark(0)
        moe.moe_route(inp["logits"], k, cfg.score_fn, cfg.renormalize, self.ids, self.w, st)
        mark(1)
        disp = {n: v[n] for n in ("counts", "offsets", "sorted_to_slot", "slot_to_sorted",
                                  "x_sorted")}
        moe.moe_dispatch(self.ids, E, x=inp["x"], workspace=self.dws, out=disp, stream=st)
        mark(2)
        moe.moe_gate_up(v["x_sorted"], v["offsets"], wts["w_gate_up"], v["sorted_to_slot"],
                        self.w, cfg.scale_input, h=v["h"], workspace=self.gws, stream=st)
        mark(3)
        moe.moe_down(v["h"], v["offsets"], wts["w_down"], y_sorted=v["y_sorted"],
                     workspace=self.gws, stream=st)
        mark(4)
        i = 5
        if Is:
            sgu, sdn = wts["w_shared_gate_up"], wts["w_shared_down"]
            moe.moe_gate_up(inp["x"], None, sgu if self.packed else sgu.unsqueeze(0),
                            h=v["h_shared"], workspace=self.gws, stream=st)
            mark(i)
            moe.moe_down(v["h_shared"], None, sdn if self.packed else sdn.unsqueeze(0),
                         y_sorted=v["y_shared"], workspace=self.gws, stream=st)
            mark(i + 1)
            i += 2
        moe.moe_combine(v["y_sorted"], v["slot_to_sorted"], k, cfg.dtype,
                        topk_weights=None if cfg.scale_input else self.w,
                        y_shared=v["y_shared"] if Is else None, out=self.out, stream=st)
        mark(i)

    def fwd(self, st_):
        cfg, wts = self.cfg, self.wts
        self.moe.moe_forward(self.inp["x"], self.inp["logits"], wts["w_gate_up"], wts["w_down"],
                             cfg.k, cfg.score_fn, self.flags, wts["w_shared_gate_up"],
                             wts["w_shared_down"], out=self.out, topk_ids=self.ids,
                             topk_weights=self.w, workspace=self.ws, stream=st_)

    def timed(self, fn):
        """Mean ms of fn() over the timed steps, each between its own events, L2 flushed
        before each (max over ranks)."""
        import torch
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        self.barrier()
        evs = [self.events(2) for _ in range(self.steps)]
        for a_, b_ in evs:
            self.flush_l2()
            a_.record(self.stream)
            fn()
            b_.record(self.stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
        return reduce_max(ms, self.dev) if self.world > 1 else ms

    def run_staged(self):
        import torch
        moe = self.moe
        for _ in range(max(self.warmup, 3)):
            self.step()
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(self.gws) == 0
        assert moe.moe_read_device_status(self.dws) == 0
        nev = len(self.stages) + 1
        events = [self.events(nev) for _ in range(self.steps)]
        self.barrier()
        torch.cuda.synchronize()
        with ClockSampler(self.dev.index) as clocks:
            for s_ in range(self.steps):
                self.flush_l2()
                self.step(events[s_])
            torch.cuda.synchronize()
        self.barrier()
        per_stage = {name: [] for name in self.stages}
        step_ms = []
        for ev in events:
            for i, name in enumerate(self.stages):
                per_stage[name].append(ev[i].elapsed_time(ev[i + 1]))
            step_ms.append(ev[0].elapsed_time(ev[-1]))
        self.per_stage = per_stage
        self.staged_ms = statistics.mean(step_ms)
        if self.world > 1:
            self.staged_ms = reduce_max(self.staged_ms, self.dev)
        self.staged_clocks = clocks.summary()

    def run_graph(self):
        """moe_forward captured once as a CUDA graph and replayed: the headline timed region."""
        import torch
        dev, stream = self.dev, self.stream
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            self.fwd(cap)  # first call on this stream outside capture
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(graph, stream=cap):
                self.fwd(cap)
        stream.wait_stream(cap)
        for _ in range(max(self.warmup, 3)):
            graph.replay()
        torch.cuda.synchronize()
        self.barrier()
        torch.cuda.synchronize()
        g_ev = [self.events(2) for _ in range(self.steps)]
        with ClockSampler(dev.index) as gclocks:
            for a_, b_ in g_ev:
                self.flush_l2()
                a_.record(stream)
                graph.replay()
                b_.record(stream)
            torch.cuda.synchronize()
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in g_ev)
        self.graph_ms = reduce_max(ms, dev) if self.world > 1 else ms
        self.graph_clocks = gclocks.summary()
        assert self.moe.moe_read_device_status(self.ws) == 0
        del graph

    def run_mx_decode(self, tc=False):
        """The MX layer on MXFP4 weights captured as a CUDA graph and replayed with L2 flushed,
        as the bf16 layer is timed: µs per layer and the touched experts' MX bytes (codes and
        scales) per second. tc=False: moe_forward_mx (first-version layout, warp-level MMAs);
        tc=True: moe_forward_mx_tc (tensor-core layout, block-scaled tcgen05 MMAs)."""
        import torch
        cfg, moe, dev, stream = self.cfg, self.moe, self.dev, self.stream
        T, d, E, k, I = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I
        quant = moe.quantize_weights_mx_tc if tc else moe.quantize_weights_mx
        mgu = quant(self.inp["w_gate_up"], moe.W_GATE_UP)
        mdn = quant(self.inp["w_down"], moe.W_DOWN)
        size = moe.moe_forward_mx_tc_workspace_size if tc else moe.moe_forward_mx_workspace_size
        ws = torch.empty(size(T, d, E, k, I, 0), dtype=torch.uint8, device=dev)
        out, ids, w = torch.empty_like(self.out), torch.empty_like(self.ids), torch.empty_like(self.w)
        layer = moe.moe_forward_mx_tc if tc else moe.moe_forward_mx

        def fwd(s_):
            layer(self.inp["x"], self.inp["logits"], mgu, mdn, k, cfg.score_fn, self.flags,
                  out=out, topk_ids=ids, topk_weights=w, workspace=ws, stream=s_)
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            fwd(cap)
            torch.cuda.current_stream().synchronize()
            with torch.cuda.graph(graph, stream=cap):
                fwd(cap)
        stream.wait_stream(cap)
        for _ in range(max(self.warmup, 3)):
            graph.replay()
        torch.cuda.synchronize()
        evs = [self.events(2) for _ in range(self.steps)]
        for a_, b_ in evs:
            self.flush_l2()
            a_.record(stream)
            graph.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
        ms = reduce_max(ms, dev) if self.world > 1 else ms
        distinct = int(torch.unique(ids).numel())
        touched = (mgu.data.numel() + mdn.data.numel()) * distinct // E
        del graph
        kernels = moe.moe_forward_mx_tc_kernel_count(T, d, k, I, 0) if tc else 1
        path = ("moe_forward_mx_tc: one cooperative kernel, the touched experts' MXFP4 codes "
                "times x and h in MXFP8 on the block-scaled tensor cores "
                "(tcgen05.mma.kind::mxf8f6f4.block_scale, weights as M, tokens as N)"
                if tc and kernels == 1 else
                f"moe_forward_mx_tc: {kernels} kernels (block-scaled tensor-core GEMMs)" if tc else
                "moe_forward_mx: one cooperative kernel streaming the touched experts' "
                "MXFP4 codes and scales (x and h rounded to MXFP8 in the kernel)")
        return {"us_per_layer": round(ms * 1e3, 2), "distinct_experts": distinct,
                "weight_bytes_touched": touched,
                "weight_gbs": round(touched / (ms * 1e-3) / 1e9, 1),
                "path": path,
                "time": "CUDA-graph replay, events on the launching stream, L2 flushed before "
                        "every replay"}

    def run_e2e(self):
        import torch
        cfg, moe, wts = self.cfg, self.moe, self.wts
        T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
        self.x_h = self.inp["x"].cpu().pin_memory()
        self.lg_h = self.inp["logits"].cpu().pin_memory()
        self.out_h = torch.empty(T, d, dtype=cfg.dtype).pin_memory()
        hws = torch.empty(moe.moe_forward_host_workspace_size(T, d, E, k, I, Is, cfg.dtype),
                          dtype=torch.uint8, device=self.dev)

        def e2e_step():
            # moe_forward_host: the kernels read the pinned x and logits and write the pinned
            # output in place
            moe.moe_forward_host(self.x_h, self.lg_h, wts["w_gate_up"], wts["w_down"], k,
                                 cfg.score_fn, self.flags, wts["w_shared_gate_up"],
                                 wts["w_shared_down"], out=self.out_h, workspace=hws,
                                 stream=self.stream, device=self.dev)

        self.e2e_ms = self.timed(e2e_step)
        del hws

    def e2e_entry(self):
        T = self.cfg.T
        return {"value": round(T * self.world / (self.e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "ms_per_step": round(self.e2e_ms, 4),
                "h2d_bytes_per_step": self.x_h.numel() * self.x_h.element_size()
                + self.lg_h.numel() * self.lg_h.element_size(),
                "d2h_bytes_per_step": self.out_h.numel() * self.out_h.element_size(),
                "path": "moe_forward_host on pinned host x, logits and out: the kernels read x "
                        "and the logits and write out across NVLink-C2C (x staged by one copy "
                        "when a shared expert runs), all on the timed stream"}

    def roofline(self):
        """Roofline of the dominant kernel: the gate_up grouped GEMM (2/3 of the expert FLOPs)
        for prefill layers; the whole layer against HBM for decode batches; the FP32 pipes for
        the fp32 layer."""
        import torch
        cfg, moe, v = self.cfg, self.moe, self.v
        T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
        R = T * k
        pk, pk_src = peaks()
        ps = self.per_stage
        gu_ms = statistics.mean(ps["gate_up"])
        dn_ms = statistics.mean(ps["down"])
        gu_flops, dn_flops = 4.0 * d * I * R, 2.0 * d * I * R
        sh_flops, sh_ms = 0.0, 0.0
        if Is:
            sh_flops = 6.0 * d * Is * T
            sh_ms = statistics.mean(ps["shared_gate_up"]) + statistics.mean(ps["shared_down"])
        self.experts_ms = gu_ms + dn_ms + sh_ms
        self.expert_tflops = (gu_flops + dn_flops + sh_flops) / (self.experts_ms * 1e-3) / 1e12
        ach = gu_flops / (gu_ms * 1e-3) / 1e12
        if cfg.dtype != torch.bfloat16:
            peak = fp32_alu_peak_tflops(pk.get("sm_max_mhz", 2070.0))
            return {"bound": "alu", "kernel": "simt_grouped_gemm<gate_up>",
                    "achieved": round(ach, 3), "peak": round(peak, 1), "unit": "TFLOP/s",
                    "frac": round(ach / peak, 5), "traffic": None,
                    "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x max SM clock",
                    "note": "correctness workload (0.1 GFLOP): launch-bound, no target"}
        gu_kernel = moe.moe_gemm_kernel_name(moe.W_GATE_UP, R, E)
        traffic, _ = traffic_for(GEMM_SOURCES.get(gu_kernel, ""), cfg.name)
        roof = {"bound": "tensor", "kernel": f"{gu_kernel}<gate_up>", "achieved": round(ach, 1),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops"], 4), "traffic": traffic,
                "peak_source": f"{pk_src} bf16_tflops (burst)",
                "frac_of_sustained": round(ach / pk.get("bf16_tflops_sustained",
                                                        pk["bf16_tflops"]), 4),
                "algorithmic_flops": gu_flops,
                "time": "gate_up stage of the staged loop (events around the call, L2 flushed)"}
        if cfg.name.startswith("decode"):
            # decode streams weights: the bound is HBM. Algorithmic bytes of one layer = the
            # distinct experts' weights (3 d I bf16 each) + x, logits, ids/weights and out,
            # over the whole layer's replay time (the fused kernel, or the chain)
            n_touched = int((v["counts"] > 0).sum().item())
            layer_bytes = (n_touched * 3.0 * d * I * 2 + T * d * 2 * 2 + T * E * 4 + T * k * 8)
            ach_gbs = layer_bytes / (self.graph_ms * 1e-3) / 1e9
            fused = moe.moe_forward_kernel_count(T, k, Is, cfg.dtype) == 1
            traffic, _ = traffic_for("decode_fused.cu", cfg.name) if fused else (None, None)
            roof = {"bound": "hbm",
                    "kernel": ("decode layer: decode_fused_kernel (route, dispatch, experts, "
                               "combine)" if fused else
                               "decode layer: route/dispatch chain + grouped GEMMs + combine"),
                    "achieved": round(ach_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(ach_gbs / pk["hbm_gbs"], 4), "traffic": traffic,
                    "peak_source": f"{pk_src} hbm_gbs",
                    "algorithmic_bytes": int(layer_bytes), "distinct_experts": n_touched,
                    "time": "whole-layer graph replay (per-step events, L2 flushed between "
                            "steps)"}
        return roof

    def kernels(self):
        cfg = self.cfg
        return self.moe.moe_forward_kernel_count(cfg.T, cfg.k, cfg.I_shared, cfg.dtype)

    def run_mx_tc(self):
        """The MX layer on the block-scaled tensor cores (MXFP4 weights quantised once at load
        into the tensor-core layout, x and h MXFP8): moe_forward_mx_tc timed whole, and its
        x rounding and two GEMMs timed on their own; L2 flushed before each step."""
        import torch
        cfg, moe, inp = self.cfg, self.moe, self.inp
        T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
        R = T * k
        q = {n_: (moe.quantize_weights_mx_tc(inp[n_], moe.W_GATE_UP if "gate_up" in n_
                                             else moe.W_DOWN) if inp[n_] is not None else None)
             for n_ in ("w_gate_up", "w_down", "w_shared_gate_up", "w_shared_down")}
        ws = torch.empty(moe.moe_forward_mx_tc_workspace_size(T, d, E, k, I, Is),
                         dtype=torch.uint8, device=self.dev)
        out = torch.empty_like(self.out)

        def layer():
            moe.moe_forward_mx_tc(inp["x"], inp["logits"], q["w_gate_up"], q["w_down"], k,
                                  cfg.score_fn, self.flags, q["w_shared_gate_up"],
                                  q["w_shared_down"], out=out, topk_ids=self.ids,
                                  topk_weights=self.w, workspace=ws, stream=self.stream)

        layer_ms = self.timed(layer)
        assert moe.moe_read_device_status(ws) == 0
        v = moe.mx_tc_workspace_views(ws, T, d, E, k, I, Is)
        gws = torch.zeros(256, dtype=torch.uint8, device=self.dev)
        rows_ms = self.timed(lambda: moe.mx_tc_rows(
            inp["x"], self.ids, v["slot_to_sorted"], v["offsets"], E, v["x_codes"], v["x_sf"],
            stream=self.stream))
        gu_ms = self.timed(lambda: moe.moe_gate_up_mx_tc(
            v["x_codes"], v["x_sf"], v["offsets"], q["w_gate_up"], R, v["h_codes"], v["h_sf"],
            v["sorted_to_slot"], self.w, cfg.scale_input, gws, self.stream))
        dn_ms = self.timed(lambda: moe.moe_down_mx_tc(
            v["h_codes"], v["h_sf"], v["offsets"], q["w_down"], R, v["y_sorted"], gws,
            self.stream))
        assert moe.moe_read_device_status(gws) == 0
        pk, pk_src = peaks()
        fp8_peak = 2.0 * pk["bf16_tflops"]   # dense FP8 = 2 x bf16 (nominal 4.5 / 2.25 PFLOP/s)
        # DRAM traffic of the gate_up launch: captured on the Mixtral shape cut to E=4, T=2048
        # (a few GB on the device). The full Mixtral launch (E=8, T=4096) doubles each part of
        # it: the weights (with E) and the x and h rows (with T), so the capture is scaled x2
        traffic = None
        small, _ = traffic_for("gemm_mx_tc.cu", "mixtral_8x7b@T2048@E4")
        if small is not None and cfg.name == "mixtral_8x7b":
            traffic = int(small * 2)
        gu_tf = 4.0 * d * I * R / (gu_ms * 1e-3) / 1e12
        dn_tf = 2.0 * d * I * R / (dn_ms * 1e-3) / 1e12
        wb = sum(v_.data.numel() for v_ in q.values() if v_ is not None)
        bf = sum(inp[n_].numel() * 2 for n_ in q if inp[n_] is not None)
        res = {"ms_per_step": round(layer_ms, 4),
               "tokens_per_s": round(T * self.world / (layer_ms * 1e-3), 1),
               "stages_ms": {"x_to_mxfp8_rows": round(rows_ms, 4), "gate_up": round(gu_ms, 4),
                             "down": round(dn_ms, 4)},
               "roofline": {"bound": "tensor", "kernel": "tc_mx_gemm<gate_up>",
                            "achieved": round(gu_tf, 1), "peak": round(fp8_peak, 1),
                            "unit": "TFLOP/s", "frac": round(gu_tf / fp8_peak, 4),
                            "traffic": traffic,
                            "traffic_source": "ncu on E=4, T=2048 scaled x2 (weights, x and h "
                                              "all double)" if traffic is not None else None,
                            "peak_source": f"{pk_src} bf16_tflops (burst) x 2, the nominal "
                                           "FP8 / bf16 dense ratio"},
               "down_tflops": round(dn_tf, 1),
               "weight_bytes": wb, "weight_bytes_bf16": bf,
               "path": "tcgen05.mma.kind::mxf8f6f4.block_scale: E4M3 x E2M1 codes with E8M0 "
                       "block scales applied by the tensor cores (nothing dequantized)",
               # route(+dispatch indices when R <= 1024), x rows, gate_up, down, combine; the
               # dispatch's histogram, scan and rank above 1024 slots; two for a shared expert
               "kernels_per_step": 5 + (2 if Is else 0) + (0 if R <= 1024 else 3),
               "time": "events around each call, L2 flushed before each step"}
        del q, ws, v
        return res


# the workload statement's 60% bars (SURVEY-style targets), by bench name
TARGETS = {"mixtral_8x7b": ("experts_ms", 2.49), "gpt_oss_120b": ("experts_ms", 1.40),
           "llama4_scout": ("experts_ms", 7.10), "decode_T1": ("us_per_layer", 18.8),
           "decode_T8": ("us_per_layer", 121.0), "decode_T64": ("us_per_layer", 296.0)}
PER_CONFIG = ["tiny_fp32", "mixtral_8x7b", "gpt_oss_120b", "llama4_scout", "decode_T1",
              "decode_T8", "decode_T64"]


def config_entry(L, name, cpu):
    """The per_config object of one workload (staged stages, graph-replayed layer, e2e,
    roofline of its dominant kernel, CPU oracle sample)."""
    cfg = L.cfg
    roof = L.roofline()
    ent = {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k, "I": cfg.I,
           "I_shared": cfg.I_shared,
           "dtype": "bf16" if L.packed else "f32",
           "tokens_per_s": round(cfg.T * L.world / (L.graph_ms * 1e-3), 1),
           "ms_per_step": round(L.graph_ms, 4), "us_per_layer": round(L.graph_ms * 1e3, 2),
           "experts_ms": round(L.experts_ms, 4),
           "expert_gemm_tflops": round(L.expert_tflops, 1),
           "stages_ms": {n: round(statistics.mean(vv), 4) for n, vv in L.per_stage.items()},
           "roofline": roof, "e2e": L.e2e_entry(), "gpu_launches_per_step": L.kernels(),
           "clocks": L.graph_clocks}
    tgt = TARGETS.get(name)
    if tgt is not None:
        key, bar = tgt
        ent["target"] = {"quantity": key, "bar": bar, "met": ent[key] <= bar}
    if cpu is not None:
        ent["cpu_baseline"] = cpu
    return ent


def cpu_sample_entry(cfg, L, n):
    n = min(n, cfg.T)
    hi = host_inputs(cfg, L.inp)
    secs = cpu_oracle_run(cfg, hi, n)
    return {"value": round(n / secs, 2), "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"first {n} of {cfg.T} tokens, whole layer, float64 numpy ({secs:.1f} s)"}


def run_ours(args, rank, world):
    import torch

    from routing_dispatch_grouped_gb300 import moe, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = workload_config(args.config, args.T, args.E)
    moe.lib()
    L = Layer(cfg, dev, args.steps, args.warmup, world)
    T, d, E, k, I, Is = cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.I_shared
    R = T * k
    dt = cfg.dtype
    inp, wts, stream, flags = L.inp, L.wts, L.stream, L.flags
    ids, w, out = L.ids, L.w, L.out
    flush_l2 = L.flush_l2

    L.run_staged()
    # the product call: moe_forward issued from the host every step ...
    forward_ms = L.timed(lambda: L.fwd(stream))
    # ... and captured once as a CUDA graph and replayed (no host launch cost; the form a
    # decode loop runs in). This is the timed region of the headline value.
    L.run_graph()
    graph_ms = L.graph_ms
    # end to end through moe_forward with host buffers
    L.run_e2e()

    # the router from hidden states (logits = x W_r + b and the top-k in one kernel): the step
    # before the layer, timed on its own (not part of the layer's timed region above)
    w_r = synth.make_router_weight(cfg, dev)
    b_r = synth.router_bias(cfg, device=dev)
    b_r = None if b_r is None else b_r.to(torch.float32).contiguous()
    lg_r = torch.empty(T, E, dtype=torch.float32, device=dev)
    router_hidden_ms = L.timed(lambda: moe.moe_route_hidden(
        inp["x"], w_r, k, cfg.score_fn, cfg.renormalize, bias=b_r, logits=lg_r, topk_ids=ids,
        topk_weights=w, stream=stream))
    # training step of the same layer (not part of the headline value): moe_forward_train, which
    # keeps what the backward reads, then moe_backward (dx, both weight gradients in fp32, the
    # routing-weight and logit gradients), each step with its own events, L2 flushed before it
    bwd = None
    if not cfg.name.startswith("decode"):
        tflags = flags & ~moe.FUSE_COMBINE_WEIGHT
        dout = synth.normal((T, d), dt, 0, "dout", 1.0, device=dev)
        fws = torch.empty(moe.moe_forward_train_workspace_size(T, d, E, k, I, Is, dt),
                          dtype=torch.uint8, device=dev)

        def train_fwd():
            moe.moe_forward_train(inp["x"], inp["logits"], wts["w_gate_up"], wts["w_down"], k,
                                  cfg.score_fn, tflags, wts["w_shared_gate_up"],
                                  wts["w_shared_down"], out=out, topk_ids=ids, topk_weights=w,
                                  workspace=fws, stream=stream)

        train_fwd()
        grads = moe.moe_backward(dout, inp["x"], inp["logits"], wts["w_gate_up"], wts["w_down"],
                                 k, ids, w, fws, cfg.score_fn, tflags, wts["w_shared_gate_up"],
                                 wts["w_shared_down"], stream=stream)
        bws = grads["workspace"]

        def train_bwd():
            moe.moe_backward(dout, inp["x"], inp["logits"], wts["w_gate_up"], wts["w_down"], k,
                             ids, w, fws, cfg.score_fn, tflags, wts["w_shared_gate_up"],
                             wts["w_shared_down"], out=grads, workspace=bws, stream=stream)

        for _ in range(3):
            train_fwd()
            train_bwd()
        torch.cuda.synchronize()
        t_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                for _ in range(args.steps)]
        for ev in t_ev:
            flush_l2()
            ev[0].record(stream)
            train_fwd()
            ev[1].record(stream)
            train_bwd()
            ev[2].record(stream)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(bws) == 0
        tf_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in t_ev)
        tb_ms = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in t_ev)
        if world > 1:
            tf_ms, tb_ms = reduce_max(tf_ms, dev), reduce_max(tb_ms, dev)
        bwd_flops = 2.0 * (6.0 * d * I * R + 6.0 * d * Is * T)  # dgrad + wgrad of each GEMM
        pk_b, pk_b_src = peaks()
        b_tf = bwd_flops / (tb_ms * 1e-3) / 1e12
        # the same backward with the weight gradients rounded once to bf16 (MOE_WGRAD_BF16)
        tb16_ms = None
        if dt == torch.bfloat16:
            g16 = moe.moe_backward(dout, inp["x"], inp["logits"], wts["w_gate_up"],
                                   wts["w_down"], k, ids, w, fws, cfg.score_fn,
                                   tflags | moe.WGRAD_BF16, wts["w_shared_gate_up"],
                                   wts["w_shared_down"], workspace=bws, stream=stream)

            def train_bwd16():
                moe.moe_backward(dout, inp["x"], inp["logits"], wts["w_gate_up"], wts["w_down"],
                                 k, ids, w, fws, cfg.score_fn, tflags | moe.WGRAD_BF16,
                                 wts["w_shared_gate_up"], wts["w_shared_down"], out=g16,
                                 workspace=bws, stream=stream)

            for _ in range(3):
                train_bwd16()
            b_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                    for _ in range(args.steps)]
            for ev in b_ev:
                flush_l2()
                ev[0].record(stream)
                train_bwd16()
                ev[1].record(stream)
            torch.cuda.synchronize()
            assert moe.moe_read_device_status(bws) == 0
            tb16_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in b_ev)
            if world > 1:
                tb16_ms = reduce_max(tb16_ms, dev)
            del g16
        bwd = {"backward_ms": round(tb_ms, 4), "backward_tflops": round(b_tf, 1),
               "backward_frac_of_peak": round(b_tf / pk_b["bf16_tflops"], 4)
               if dt == torch.bfloat16 else None,
               "peak_source": f"{pk_b_src} bf16_tflops (burst)",
               "forward_train_ms": round(tf_ms, 4),
               "train_step_ms": round(tf_ms + tb_ms, 4),
               "train_tokens_per_s": round(T * world / ((tf_ms + tb_ms) * 1e-3), 1),
               "backward_kernels": moe.moe_backward_kernel_count(T, k, Is, tflags, True),
               "outputs": "dx, fp32 dW_gate_up/dW_down (and shared), d topk_weights, d logits",
               "backward_bf16_wgrad_ms": None if tb16_ms is None else round(tb16_ms, 4),
               "backward_bf16_wgrad_tflops": None if tb16_ms is None else
               round(bwd_flops / (tb16_ms * 1e-3) / 1e12, 1),
               "time": "per-step events around each call, L2 flushed before each step"}
        del grads, bws, fws

    # the MX form of the same layer (MXFP4 expert weights quantised once at load, MXFP8 x and
    # h): moe_forward_mx with per-step events, L2 flushed before each step (not part of the
    # headline value)
    mxr = None
    if dt == torch.bfloat16:
        mxw = {n_: (moe.quantize_weights_mx(inp[n_], moe.W_GATE_UP if "gate_up" in n_
                                            else moe.W_DOWN) if inp[n_] is not None else None)
               for n_ in ("w_gate_up", "w_down", "w_shared_gate_up", "w_shared_down")}
        mws = torch.empty(moe.moe_forward_mx_workspace_size(T, d, E, k, I, Is),
                          dtype=torch.uint8, device=dev)

        def mx_fwd():
            moe.moe_forward_mx(inp["x"], inp["logits"], mxw["w_gate_up"], mxw["w_down"], k,
                               cfg.score_fn, flags, mxw["w_shared_gate_up"],
                               mxw["w_shared_down"], out=out, topk_ids=ids, topk_weights=w,
                               workspace=mws, stream=stream)

        for _ in range(3):
            mx_fwd()
        torch.cuda.synchronize()
        m_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        for a_, b_ in m_ev:
            flush_l2()
            a_.record(stream)
            mx_fwd()
            b_.record(stream)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(mws) == 0
        mx_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in m_ev)
        if world > 1:
            mx_ms = reduce_max(mx_ms, dev)
        mx_bytes = sum(v_.data.numel() for v_ in mxw.values() if v_ is not None)
        bf_bytes = sum(inp[n_].numel() * 2 for n_ in mxw if inp[n_] is not None)
        mxr = {"ms_per_step": round(mx_ms, 4),
               "tokens_per_s": round(T * world / (mx_ms * 1e-3), 1),
               "weight_bytes": mx_bytes, "weight_bytes_bf16": bf_bytes,
               "path": ("one-kernel decode layer streaming the MXFP4 codes (x and h rounded "
                        "to MXFP8 in the kernel, f16 MMAs on the element values rescaled per "
                        "32-row K block)" if moe.moe_forward_kernel_count(T, k, Is, dt) == 1
                        else "x and h rounded to MXFP8; the touched experts' MXFP4 weights "
                        "dequantized to bf16 (exact) for the bf16 tensor-core GEMMs"),
               "time": "per-step events around moe_forward_mx, L2 flushed before each step"}
        del mxw, mws
        if d % 32 == 0 and I % 32 == 0 and Is % 32 == 0:
            mxr = {"tensor_core": L.run_mx_tc(), "dequantized_or_decode": mxr}

    roof = L.roofline()
    tokens_per_s = T * world / (graph_ms * 1e-3)
    res = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(graph_ms, 4), "higher_is_better": True, "scaling": "weak",
        "timing": "CUDA-graph replay of moe_forward, events on the launching stream",
        "us_per_layer": round(graph_ms * 1e3, 2),
        "vs_baseline": None, "dtype": "bf16" if dt == torch.bfloat16 else "f32",
        "data": "synthetic (seeded counter-based generator; shapes of the workload)",
        "config": {"workload": cfg.name, "T": T, "d": d, "E": E, "k": k, "I": I,
                   "I_shared": Is, "seed": cfg.seed,
                   "weights": "repacked once at load (moe_pack_weights)" if L.packed
                   else "layout of the pages",
                   "l2": "flushed before every timed step (256 MB write, outside the events)",
                   "headline": "value, roofline, e2e and cpu_baseline are this workload's; "
                               "per_config holds every workload of the same run"},
        "roofline": roof,
        "expert_gemm_tflops": round(L.expert_tflops, 1),
        "experts_ms": round(L.experts_ms, 4),
        "stages_ms": {n: round(statistics.mean(vv), 4) for n, vv in L.per_stage.items()},
        "staged_calls_ms_per_step": round(L.staged_ms, 4),
        "forward_call_ms": round(forward_ms, 4),
        "router_from_hidden_ms": round(router_hidden_ms, 4),
        "training": bwd,
        "mx": mxr,
        "e2e": L.e2e_entry(),
        "gpu_launches": args.steps * L.kernels(),
        "clocks": L.graph_clocks,
        "clocks_staged": L.staged_clocks,
    }
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_sample_entry(cfg, L, args.cpu_sample or default_sample(cfg))
        res["cpu_baseline"] = cpu

    if not args.no_per_config:
        # every workload in the same run: the headline's own entry, then the others one at a
        # time (each freed before the next is built)
        per = {}
        head = args.config if args.config.startswith("decode_T") or args.T is None else None
        small = rank == 0 and world == 1 and not args.no_cpu_baseline
        for name in PER_CONFIG:
            if name == head and args.E is None:
                per[name] = config_entry(L, name, cpu)
                if isinstance(mxr, dict) and "tensor_core" in mxr:
                    per[name]["mx_tensor_core"] = mxr["tensor_core"]
                if name.startswith("decode") and moe.moe_forward_kernel_count(T, k, Is, dt) == 1:
                    per[name]["mx_decode"] = L.run_mx_decode()
                if name.startswith("decode") and L.packed:
                    per[name]["mx_tc_decode"] = L.run_mx_decode(tc=True)
                continue
            c_ = workload_config(name)
            Lc = Layer(c_, dev, args.steps, args.warmup, world)
            Lc.run_staged()
            Lc.run_graph()
            Lc.run_e2e()
            mx_tc = Lc.run_mx_tc() if Lc.packed and not name.startswith("decode") else None
            # a shorter CPU sample per extra workload (about a third of the headline's)
            cs = cpu_sample_entry(c_, Lc, max(8, default_sample(c_) // 3)) if small else None
            per[name] = config_entry(Lc, name, cs)
            if mx_tc is not None:
                per[name]["mx_tensor_core"] = mx_tc
            if (name.startswith("decode") and Lc.packed and
                    moe.moe_forward_kernel_count(c_.T, c_.k, c_.I_shared, c_.dtype) == 1):
                per[name]["mx_decode"] = Lc.run_mx_decode()
            if name.startswith("decode") and Lc.packed:
                per[name]["mx_tc_decode"] = Lc.run_mx_decode(tc=True)
            del Lc
            torch.cuda.empty_cache()
        res["per_config"] = per
    return res


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is the whole layer on a token sample."""
    import torch

    from routing_dispatch_grouped_gb300 import synth

    cfg = workload_config(args.config, args.T, args.E)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = host_inputs(cfg, synth.make_inputs(cfg, dev))
    n = args.cpu_sample or max(8, default_sample(cfg) // max(1, args.steps + args.warmup) * 2)
    n = min(n, cfg.T)
    for _ in range(args.warmup):
        cpu_oracle_run(cfg, inp, n)
    secs = [cpu_oracle_run(cfg, inp, n) for _ in range(args.steps)]
    ms = 1e3 * sum(secs) / len(secs)
    val = n / (ms * 1e-3)
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                                        "E": cfg.E, "k": cfg.k, "I": cfg.I,
                                        "I_shared": cfg.I_shared},
        "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"first {n} of {cfg.T} tokens per step, whole layer"},
        "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
