#!/usr/bin/env python
"""Benchmark of the DSpark per-cycle hot path on GB300.

One step = one decoding cycle of the workload: the gamma-step Markov draft
(fused bias contraction + exact softmax normaliser + the two-level sample --
16-entry blocks raced on their masses, the entry by inverse CDF -- + confidence,
per step) followed by verification of every drafted token of the
flattened batch (the qwen4b workload verifies all R * (gamma + 1) rows; workloads
with a profiled SPS table also run the prefix scheduler and verify only the
scheduled rows).

Prints ONE JSON line (rank 0).  `value` is drafted-and-verified tokens per second
of device time, R * gamma / (T_draft + T_schedule + T_verify), summed over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dspark|reference]
                  [--workload qwen4b|heavy|prod|rnn|tiny|sts_fit|train_loss]

`--workload sts_fit` times the confidence calibration instead (Module D's
sequential temperature scaling on a held-out set of draft blocks): one step is
one full fit, and `value` is (block, position, temperature) evaluations per
second.

`--workload sched_profile` profiles SPS(B) from a stand-in target forward (two bf16
GEMM layers at d = 2560, timed over B = 16..8704) and runs the prefix scheduler on
that measured table for R = 16..512 requests of gamma = 16 (with and without the
early-stop break): `value` is the expected throughput Theta of the no-break
schedule at R = 256, and the line carries the verify budget per request against
load (the production section's Figure 8 mechanism, reproduced qualitatively).

`--workload train_loss` times the drafter's training losses and their gradient
(Module F, eqs. 8-12) on 64 blocks x 8 positions over V = 151936 (bf16 logits):
one step is one call, and `value` is positions per second.

`--impl reference` times the CPU oracle (the plain single-threaded checker) on a
bounded sample of requests of the same workload; it is the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_drafter_markov_gb300 import _lib as dsp  # noqa: E402
from speculative_decoding_drafter_markov_gb300 import workloads as W  # noqa: E402

METRIC = "drafted tok/s (R·γ) + verified tok/s at 1 GB300; % of HBM/TC roofline"
L2_FLUSH_BYTES = 256 << 20


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dspark", choices=["dspark", "reference"])
    ap.add_argument("--workload", default="prod",
                    choices=sorted(W.WORKLOADS) + ["sts_fit", "train_loss", "sched_profile"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return world, rank, local


def aggregate_ranks(local_ms, local_units, world, device):
    """Whole-job figures of a weak-scaling run: the timed span is the maximum
    over ranks, the work is every rank's (each rank runs its own replica of the
    workload).  Returns (max_ms, units per second summed over ranks)."""
    total_ms = float(local_ms)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, world * local_units / (total_ms / 1e3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def _workload_desc(wl):
    return (f"{wl.name}: R={wl.R} gamma={wl.gamma} V={wl.V} r={wl.r} d={wl.d} {wl.dtype} "
            f"{wl.head} head, scheduler={wl.sched}")


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region: NVML through
    ctypes every ~1 ms in a background thread (the device matched by UUID), else
    nvidia-smi at its fastest interval."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        self.dev = device_index
        self.samples, self.max_mhz, self.reasons = [], None, set()
        self.nvml, self.handle, self.thread, self.proc = None, None, None, None
        self.stop_flag = False
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + uuid)
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.nvml, self.handle, self.ct = lib, h, ctypes
        except (OSError, AttributeError, RuntimeError):
            self.nvml = None

    def _poll(self):
        ct, lib, h = self.ct, self.nvml, self.handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, ct.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.001)

    def start(self):
        import threading
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join()
            src = "nvml"
        elif self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                parts = [q.strip() for q in line.split(",")]
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue
                for name, val in zip(names, parts[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)
            src = "nvidia-smi"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"]}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": src}


class Cycle:
    """Preallocated buffers and the enqueue order of one decoding cycle."""

    def __init__(self, wl, seed, device):
        self.wl = wl
        self.dev = device
        inp = W.draft_inputs(wl, seed=seed, device=device)
        self.inp = inp
        R, gm, V = wl.R, wl.gamma, wl.V
        self.out = {"x": torch.empty((R, gm), dtype=torch.int32, device=device),
                    "logq": torch.empty((R, gm), dtype=torch.float32, device=device),
                    "lse": torch.empty((R, gm), dtype=torch.float32, device=device),
                    "c": torch.empty((R, gm), dtype=torch.float32, device=device)}
        self.rnn = wl.head == "rnn"
        if self.rnn:
            r = wl.r
            self.out["A"] = torch.empty((R, gm, r), dtype=torch.float32, device=device)
            self.out["s_out"] = torch.empty((R, r), dtype=torch.float32, device=device)
            ws_bytes = dsp.draft_rnn_workspace_size(inp["U"], inp["h"], inp["W1"], inp["W2t"],
                                                    inp["W"], inp["w"], inp["anchor"])
        else:
            ws_bytes = dsp.draft_markov_workspace_size(inp["U"], inp["h"], inp["W1"], inp["W2t"],
                                                       inp["w"], inp["anchor"])
        self.ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
        # verification batch: every drafted token (no scheduler), or the capacity
        # R (gamma + 1) with the scheduler's device-side row count
        self.sched = wl.sched != "none"
        cap = R * (gm + 1)
        ell_all = np.full(R, gm)
        self.tags = torch.as_tensor(W.tags_from_ell(ell_all), device=device)
        self.T = W.target_logits(wl, inp["U"], inp["U_bonus"], W.tags_from_ell(ell_all), seed=seed)
        assert self.T.shape[0] == cap
        if self.sched:
            B_min, _ = wl.B_range
            self.B_min = B_min
            self.sps = torch.as_tensor(W.sps_table(wl, seed), device=device)
            self.K_hist = [torch.full((1,), -1, dtype=torch.int32, device=device) for _ in range(3)]
            self.N_dev = torch.empty(1, dtype=torch.int32, device=device)
            self.tags_sched = torch.empty((cap, 2), dtype=torch.int32, device=device)
            self.sched_out = {"ell": torch.empty(R, dtype=torch.int32, device=device),
                              "K_out": self.K_hist[0],
                              "theta_best": torch.empty(1, dtype=torch.float64, device=device)}
        self.vout = {"n_accept": torch.empty(R, dtype=torch.int32, device=device),
                     "out_tokens": torch.empty((R, gm + 1), dtype=torch.int32, device=device),
                     "next_anchor": torch.empty(R, dtype=torch.int32, device=device)}
        if self.sched:
            # target rows of the scheduled batch are gathered from the full grid
            # (a stand-in for the target forward; not part of the timed stages)
            self.T_sched = torch.empty_like(self.T)
        nbytes = dsp.verify_workspace_size(self.T, self.tags, inp["anchor"], self.out["x"],
                                           self.out["logq"], self.out["lse"], inp["U"], inp["W1"],
                                           inp["W2t"], A=self.out.get("A"))
        self.vws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        # library kernels per cycle: the gamma draft steps in one launch (the RNN
        # head's state updates inside it), after the RNN head's h projection (a
        # tensor-core GEMM); schedule + build_tags; verify (init, phase 1, phase 2
        # with the draw)
        n_draft = 2 if self.rnn else 1
        self.launches_per_cycle = n_draft + 3 + (2 if self.sched else 0)

    def draft(self, cycle):
        i = self.inp
        if self.rnn:
            dsp.draft_rnn(i["U"], i["h"], i["W1"], i["W2t"], i["W"], i["w"], i["anchor"],
                          out=self.out, ws=self.ws, seed=1234, cycle=cycle)
        else:
            dsp.draft_markov(i["U"], i["h"], i["W1"], i["W2t"], i["w"], i["anchor"],
                             out=self.out, ws=self.ws, seed=1234, cycle=cycle)

    def schedule(self, cycle):
        if not self.sched:
            return
        mode = dsp.SCHED_ASYNC if self.wl.sched == "async" else dsp.SCHED_SYNC
        k_in = self.K_hist[(cycle + 1) % 3] if mode == dsp.SCHED_ASYNC else None
        self.sched_out["K_out"] = self.K_hist[cycle % 3]
        dsp.schedule(self.out["c"], self.sps, self.B_min, mode=mode, K_in=k_in, out=self.sched_out)
        dsp.build_tags(self.sched_out["ell"], self.wl.gamma, tags=self.tags_sched, N_out=self.N_dev)

    def target(self):
        """Target logits of the scheduled rows (harness stand-in for the target model)."""
        if self.sched:
            t = self.tags_sched.long()
            torch.index_select(self.T, 0, t[:, 0] * (self.wl.gamma + 1) + t[:, 1], out=self.T_sched)

    def verify(self, cycle):
        i = self.inp
        tags = self.tags_sched if self.sched else self.tags
        N_dev = self.N_dev if self.sched else None
        T = self.T_sched if self.sched else self.T
        dsp.verify(T, tags, i["anchor"], self.out["x"], self.out["logq"], self.out["lse"],
                   i["U"], i["W1"], i["W2t"], A=self.out.get("A"), N_dev=N_dev, seed=1234,
                   cycle=cycle, out=self.vout, ws=self.vws)

    def verified_tokens(self):
        if self.sched:
            return int(self.sched_out["ell"].sum().item())
        return self.wl.R * self.wl.gamma


# DRAM bytes (read + write) of one launch as ncu measured them, recorded with
# the SHA-256 of the kernel's sources at the time of the capture: a figure is
# used only while the sources still hash the same (else the traffic is null)
NCU_DRAM_FILE = os.path.join(ROOT, "profiles", "ncu_dram_bytes.txt")
KERNEL_SOURCES = {
    "draft_step_tc": ["draft_tc.cu", "tc_pipe.cuh", "tc.cuh", "common.cuh", "kernels.h", "rnn_step.cuh"],
    "train_loss_resident": ["train_loss.cu", "common.cuh"],
    "verify_phase2_tc": ["verify_tc.cu", "verify_common.cuh", "tc_pipe.cuh", "tc.cuh", "common.cuh",
                         "kernels.h"],
}


def kernel_source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_drafter_markov_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """(bytes per launch, note): the recorded ncu DRAM bytes of `kernel` at
    `workload` if they were taken on the current sources, else (None, why)."""
    want = kernel_source_hash(kernel)
    try:
        lines = open(NCU_DRAM_FILE).read().splitlines()
    except OSError:
        return None, "no ncu record"
    for line in lines:
        f = line.split()
        if len(f) >= 5 and not line.startswith("#") and f[0] == kernel and f[1] == workload:
            if f[2] == want:
                return int(f[3]) + int(f[4]), f"ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch ({f[5] if len(f) > 5 else 'full size'})"
            return None, "kernel changed since the last ncu capture"
    return None, "no ncu capture at this workload"


def draft_step_bytes(wl, with_w2=True):
    """Algorithmic bytes of one draft step: U_k rows, W_2 streamed once, the
    gathered W_1 rows, h_k and w (fp32)."""
    es = 4 if wl.dtype == "f32" else 2
    w2 = wl.V * wl.r if with_w2 else 0
    return (wl.R * wl.V + w2 + wl.R * wl.r + wl.R * wl.d) * es + (wl.d + wl.r) * 4


def draft_cycle_bytes_strict(wl):
    """The stricter per-cycle count: W_2 read from memory once for all gamma steps."""
    es = 4 if wl.dtype == "f32" else 2
    return wl.gamma * draft_step_bytes(wl, with_w2=False) + wl.V * wl.r * es


def verify_cycle_bytes(wl, rows, rejected, reread=True):
    """Algorithmic bytes of one verification: the target rows of the batch read
    once (phase 1: log-sum-exp and acceptance), then the base row U_{n+1} of
    each rejected request (the residual needs q) and W_2 once (phase 2).  With
    `reread`, phase 2 also reads each request's target row at its rejected or
    bonus position a second time: the residual max(0, p - q) needs that row's
    log-sum-exp, which only phase 1's full pass over the row gives."""
    es = 4 if wl.dtype == "f32" else 2
    return (rows * wl.V + (wl.R * wl.V if reread else 0) + rejected * wl.V + wl.V * wl.r) * es


def _verify_roofline(wl, verified, rejected, steps, t_verify_ms, hbm):
    """The verification stage (init, phase 1, phase 2) against the HBM copy
    bandwidth, from the mean rows and rejected requests per cycle (None when the
    timings are unusable)."""
    rows = wl.R + verified / steps
    nbytes = verify_cycle_bytes(wl, rows, rejected / steps)
    us = 1e3 * statistics.mean(t_verify_ms) if t_verify_ms else 0.0
    if not us > 0.0 or not hbm:
        return None
    achieved = nbytes / (us * 1e-6) / 1e9
    strict = verify_cycle_bytes(wl, rows, rejected / steps, reread=False) / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "algorithmic_bytes_per_cycle": nbytes, "rows_per_cycle": rows,
            "bytes_rule": "target rows once (phase 1); phase 2 reads each request's rejected/bonus target "
                          "row again (its residual needs the row's log-sum-exp first), the U_{n+1} rows of "
                          "rejected requests and W_2 once",
            "frac_strict": strict / hbm,
            "strict_rule": "as bytes_rule without phase 2's second read of the target rows",
            "timing": "CUDA events around the whole verify call"}


def bind_to_gpu_cpus(device_index):
    """Restrict this process to the host CPUs NVML reports as local to the GPU,
    so pinned host buffers (allocated after this) sit on the GPU's NUMA node.
    Reads the device's affinity only; returns a short description."""
    try:
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return "unchanged (nvmlInit failed)"
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            return "unchanged (no NVML handle)"
        n_words = 16  # 64-bit words: up to 1024 CPUs
        words = (ctypes.c_ulong * n_words)()
        if lib.nvmlDeviceGetCpuAffinity(h, n_words, words) != 0:
            return "unchanged (no CPU affinity)"
        cpus = {64 * i + b for i in range(n_words) for b in range(64) if (words[i] >> b) & 1}
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return "unchanged (empty CPU set)"
        os.sched_setaffinity(0, cpus)
        return f"{len(cpus)} CPUs local to the GPU (NVML)"
    except (OSError, AttributeError, RuntimeError) as e:
        return f"unchanged ({type(e).__name__})"


def run_dspark(args, world, rank, local):
    torch.cuda.set_device(local)
    host_binding = bind_to_gpu_cpus(local)
    dev = torch.device("cuda", local)
    wl = W.WORKLOADS[args.workload]
    cyc = Cycle(wl, seed=1000 + rank, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    gm = wl.gamma

    def one_cycle(c, ev=None):
        cyc.draft(c)
        if ev is not None:
            ev["d"].record(stream)
        cyc.schedule(c)
        if ev is not None:
            ev["s"].record(stream)
        cyc.target()
        if ev is not None:
            ev["g"].record(stream)
        cyc.verify(c)

    for c in range(args.warmup):
        flush.zero_()
        one_cycle(c)
    torch.cuda.synchronize()

    mk = lambda: torch.cuda.Event(enable_timing=True)
    events = [{"a": mk(), "b": mk(), "d": mk(), "s": mk(), "g": mk()} for _ in range(args.steps)]
    clocks = ClockSampler(local)
    accepted_dev = torch.zeros((), dtype=torch.int64, device=dev)  # sum of (n_accept + 1)
    rejected_dev = torch.zeros((), dtype=torch.int64, device=dev)  # requests with n_accept < l
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    verified = 0
    for s in range(args.steps):
        flush.zero_()  # L2 flush between timed iterations (outside the timed span)
        # a ~1 ms GPU spin (outside the span) lets the host enqueue the whole
        # cycle first, so the span holds device work, not Python launch latency
        torch.cuda._sleep(2_000_000)
        ev = events[s]
        ev["a"].record(stream)
        one_cycle(args.warmup + s, ev)
        ev["b"].record(stream)
        accepted_dev += cyc.vout["n_accept"].sum() + wl.R  # outside the timed span
        rejected_dev += (cyc.vout["n_accept"] < (cyc.sched_out["ell"] if cyc.sched else gm)).sum()
        if cyc.sched:
            torch.cuda.synchronize()
            verified += cyc.verified_tokens()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    if not cyc.sched:
        verified = args.steps * wl.R * gm
    t_draft = [e["a"].elapsed_time(e["d"]) for e in events]  # ms
    t_sched = [e["d"].elapsed_time(e["s"]) for e in events]
    t_verify = [e["g"].elapsed_time(e["b"]) for e in events]
    # cycle time without the harness's target-row gather
    t_cycle = [a + b + c for a, b, c in zip(t_draft, t_sched, t_verify)]
    drafted = args.steps * wl.R * gm
    total_ms, value = aggregate_ranks(sum(t_cycle), drafted, world, dev)
    accepted = int(accepted_dev.item())
    rejected = int(rejected_dev.item())

    hbm, tc, peak_kind = _peaks()
    draft_us = 1e3 * statistics.mean(t_draft)
    bytes_launch = gm * draft_step_bytes(wl)  # W_2 counted once per step
    if cyc.rnn:  # + the recurrent projection W [3r, 2r + d], read once per cycle
        bytes_launch += 3 * wl.r * (2 * wl.r + wl.d) * 2
    achieved = bytes_launch / (draft_us * 1e-6) / 1e9
    strict = draft_cycle_bytes_strict(wl) / (draft_us * 1e-6) / 1e9
    draft_traffic = (ncu_traffic("draft_step_tc", wl.name) if not cyc.rnn
                     else (None, "RNN head: the stage is two launches (h projection, steps)"))
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->f32" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": _workload_desc(wl),
                   "verify_rows": "all R*(gamma+1)" if not cyc.sched else "scheduled",
                   "l2": "256 MB buffer written between timed steps; U and T also exceed L2",
                   "host": "each timed cycle is enqueued behind a ~1 ms GPU spin (outside the span)",
                   "host_binding": host_binding,
                   "parallelism": f"replicas x{world} (requests independent)"},
        "drafted_tok_s": world * drafted / (sum(t_draft) / 1e3),
        "verified_tok_s": world * verified / ((sum(t_sched) + sum(t_verify)) / 1e3),
        "accepted_tok_s": world * accepted / (total_ms / 1e3),
        "mean_tau": accepted / (args.steps * wl.R),
        "mean_ell": verified / (args.steps * wl.R),
        "stage_us": {"draft": draft_us,
                     "draft_step": draft_us / gm,
                     "schedule": 1e3 * statistics.mean(t_sched),
                     "verify": 1e3 * statistics.mean(t_verify)},
        "roofline": {"kernel": (f"draft: h projection, step 1 state update, {gm} x draft_step_tc "
                                "(each ending with the next step's state update)"
                                if cyc.rnn else
                                f"draft_step_tc: the {gm} draft steps of a cycle in one launch "
                                "(fused contraction + epilogue + row merge per step)"),
                     "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes_per_launch": bytes_launch,
                     "bytes_rule": "per step: U_k + W_2 + W_1 rows + h_k + w; x gamma steps",
                     "timing": "CUDA events around the whole draft call",
                     "traffic": draft_traffic[0], "traffic_source": draft_traffic[1]},
        "roofline_w2_once_per_cycle": {"achieved": strict, "peak": hbm, "unit": "GB/s",
                                       "frac": strict / hbm,
                                       "algorithmic_bytes_per_launch": draft_cycle_bytes_strict(wl)},
        "roofline_verify": _verify_roofline(wl, verified, rejected, args.steps, t_verify, hbm),
        "gpu_launches": args.steps * cyc.launches_per_cycle,
        "clocks": clk,
    }
    line["diagnostics"] = acceptance_diagnostics(cyc)
    if not args.no_e2e:
        line["e2e"] = run_e2e(cyc, args, stream, flush)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=12.0)
    return line, rank


def acceptance_diagnostics(cyc, cycles=16):
    """Per-position conditional acceptance and the acceptance-length histogram of
    `cycles` further decoding cycles (untimed), counted on the GPU by
    dspark_accept_stats from each cycle's verification outcome."""
    wl = cyc.wl
    counters = None
    for c in range(cycles):
        cyc.draft(20_000 + c)
        cyc.schedule(20_000 + c)
        cyc.target()
        cyc.verify(20_000 + c)
        ell = cyc.sched_out["ell"] if cyc.sched else None
        counters = dsp.accept_stats(cyc.vout["n_accept"], wl.gamma, ell=ell, counters=counters)
    torch.cuda.synchronize()
    reached = counters["reached"].cpu().numpy()
    accepted = counters["accepted"].cpu().numpy()
    tau = counters["tau_hist"].cpu().numpy()
    cond = [round(float(a) / float(r), 4) if r > 0 else None for a, r in zip(accepted, reached)]
    return {"cycles": cycles, "conditional_acceptance": cond, "reached": reached.tolist(),
            "tau_hist": tau.tolist(),
            "mean_tau": float((tau * np.arange(1, len(tau) + 1)).sum() / max(1, tau.sum()))}


def run_e2e(cyc, args, stream, flush):
    """Same cycle through the public API from pinned host buffers: every step the
    H2D copy of that step's inputs (base logits, hidden states, anchors, target
    logits) and the D2H read of its results are inside the timed span.  The
    copies run on a second stream into two device input buffers, so step s + 1's
    inputs travel while step s computes (the double buffering a serving loop
    would use); the span runs from before step 0's copy to after the last read."""
    wl = cyc.wl
    keys = ("U", "h", "anchor")
    host_in = {k: cyc.inp[k].cpu().pin_memory() for k in keys}
    host_T = cyc.T.cpu().pin_memory()
    host_out = {k: torch.empty_like(v, device="cpu").pin_memory()
                for k, v in (("out_tokens", cyc.vout["out_tokens"]),
                             ("n_accept", cyc.vout["n_accept"]), ("c", cyc.out["c"]))}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + host_T.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    # two device input sets: set 0 is the cycle's own, set 1 a copy of its shapes
    sets = [(dict(cyc.inp), cyc.T),
            ({**cyc.inp, **{k: torch.empty_like(cyc.inp[k]) for k in keys}}, torch.empty_like(cyc.T))]
    copy_stream = torch.cuda.Stream()  # one stream: more streams measured no faster (~206 GB/s H2D)
    n = max(3, min(args.steps, 10))
    total = 0.0
    for rep in range(2):  # the first pass warms up the copy path
        mk = lambda: torch.cuda.Event(enable_timing=False)
        copied = [mk() for _ in range(n)]
        done = [mk() for _ in range(n)]
        flush.zero_()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)

        def enqueue_copy(step):
            inp, T = sets[step % 2]
            copy_stream.wait_event(a)
            if step >= 2:
                copy_stream.wait_event(done[step - 2])  # that buffer's last reader
            with torch.cuda.stream(copy_stream):
                for k in keys:
                    inp[k].copy_(host_in[k], non_blocking=True)
                T.copy_(host_T, non_blocking=True)
            copied[step].record(copy_stream)

        enqueue_copy(0)
        for step in range(n):
            if step + 1 < n:
                enqueue_copy(step + 1)
            cyc.inp, cyc.T = sets[step % 2]
            stream.wait_event(copied[step])
            cyc.draft(10_000 + step)
            cyc.schedule(10_000 + step)
            cyc.target()
            cyc.verify(10_000 + step)
            host_out["out_tokens"].copy_(cyc.vout["out_tokens"], non_blocking=True)
            host_out["n_accept"].copy_(cyc.vout["n_accept"], non_blocking=True)
            host_out["c"].copy_(cyc.out["c"], non_blocking=True)
            done[step].record(stream)
        b.record(stream)
        torch.cuda.synchronize()
        total = a.elapsed_time(b)
    cyc.inp, cyc.T = sets[0]
    return {"value": n * wl.R * wl.gamma / (total / 1e3), "unit": "tok/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipeline": "step s+1's H2D copies on a second stream during step s (two device input buffers)"}


def _oracle_sample(wl, n_req, seed=0):
    """Host inputs of `n_req` requests of the workload (same shapes per request)."""
    import dataclasses
    sub = dataclasses.replace(wl, R=n_req)
    inp = W.draft_inputs(sub, seed=seed, device="cpu")
    to_np = W.bf16_bits
    h = {k: to_np(v) for k, v in inp.items() if k not in ("U_bonus",)}
    ell = np.full(n_req, wl.gamma)
    tags = W.tags_from_ell(ell)
    T = to_np(W.target_logits(sub, inp["U"], inp["U_bonus"], tags, seed=seed))
    return h, tags, T


def _oracle_cycle(orc, h, tags, T, cycle):
    d = orc.draft_markov(h["U"], h["h"], h["W1"], h["W2t"], h["w"], h["anchor"], seed=1234,
                         cycle=cycle)
    orc.verify(T, tags, h["anchor"], d["x"], d["logq"].astype(np.float32),
               d["lse"].astype(np.float32), h["U"], h["W1"], h["W2t"], seed=1234, cycle=cycle)


def cpu_baseline(wl, budget_s=12.0):
    """The oracle as it stands, one host core, on a bounded sample of requests of
    the same workload (full vocabulary, full gamma, verify all): drafted and
    verified tokens per second, extrapolated per request."""
    import oracle as orc
    orc.build()
    h, tags, T = _oracle_sample(wl, 1)
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_cycle(orc, h, tags, T, done)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 64:
            break
    return {"value": done * wl.gamma / el, "unit": "tok/s", "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{done} request-cycles of {wl.name} (full V={wl.V}, gamma={wl.gamma}, "
                      f"verify all), single-threaded C oracle, {el:.1f} s"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on each step's bounded sample (one request),
    same metric and unit."""
    if rank != 0:
        return None
    import oracle as orc
    orc.build()
    wl = W.WORKLOADS[args.workload]
    h, tags, T = _oracle_sample(wl, 1)
    for c in range(args.warmup):
        _oracle_cycle(orc, h, tags, T, c)
    t0 = time.perf_counter()
    for s in range(args.steps):
        _oracle_cycle(orc, h, tags, T, args.warmup + s)
    el = time.perf_counter() - t0
    value = args.steps * wl.gamma / el
    return {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": _workload_desc(wl), "sample": "1 request per step"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "host_cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"1 request per step of {wl.name}, {args.steps} steps"},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- calibration fit
# held-out set: 65,536 draft blocks of gamma = 16 (e.g. 512 requests x 128 cycles),
# 256 temperatures on [0.05, 12.8], 15 ECE bins
STS = {"M": 65536, "gamma": 16, "G": 256, "n_bins": 15}
STS_METRIC = "STS calibration fit: (block, position, temperature) evaluations/s at 1 GB300"
# special-function throughput on GB300, measured with a throughput probe of
# independent chains: ex2.approx 32 and rcp.approx 16 results per SM per clock.
# One evaluation takes one of each: 1/32 + 1/16 = 3/32 SM-cycles.
EVALS_PER_SM_CLK = 32.0 / 3.0


def _sts_inputs(seed):
    s, n = W.calibration_set(STS["M"], STS["gamma"], seed=seed,
                             T_true=np.linspace(1.2, 2.4, STS["gamma"]))
    grid = np.linspace(0.05, 12.8, STS["G"]).astype(np.float32)
    return s, n, grid


def _sts_desc():
    return (f"sts_fit: M={STS['M']} blocks x gamma={STS['gamma']} positions, G={STS['G']} "
            f"temperatures, {STS['n_bins']} bins")


def _sts_cpu(budget_s=12.0, M=4096):
    """The oracle's fit on the first M blocks of the same set, per evaluation."""
    import oracle as orc
    orc.build()
    s, n, grid = _sts_inputs(11)
    s, n = s[:M], n[:M]
    done, t0 = 0, time.perf_counter()
    while True:
        orc.sts_fit(s, n, grid, n_bins=STS["n_bins"])
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 8:
            break
    evals = done * M * STS["gamma"] * STS["G"]
    return {"value": evals / el, "unit": "eval/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} fits of the first {M} blocks of the set (gamma={STS['gamma']}, "
                      f"G={STS['G']}), single-threaded C oracle, {el:.1f} s"}


def run_sts_fit(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s, n, grid = _sts_inputs(11 + rank)
    logit = torch.as_tensor(s, device=dev)
    n_acc = torch.as_tensor(n, device=dev)
    grid_d = torch.as_tensor(grid, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    fit = lambda: dsp.sts_fit(logit, n_acc, grid_d, n_bins=STS["n_bins"], ws=ws)
    for _ in range(args.warmup):
        flush.zero_()
        fit()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for a, b in ev:
        flush.zero_()  # the inputs (4.5 MB) fit in L2: flushed between timed fits
        torch.cuda._sleep(2_000_000)
        a.record(stream)
        fit()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    times = [a.elapsed_time(b) for a, b in ev]
    evals = STS["M"] * STS["gamma"] * STS["G"]
    total_ms, value = aggregate_ranks(sum(times), args.steps * evals, world, dev)
    fit_us = 1e3 * statistics.mean(times)
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0
    peak = sm * EVALS_PER_SM_CLK * mhz * 1e6 / 1e9  # G eval/s
    achieved = evals / (fit_us * 1e-6) / 1e9
    line = {
        "metric": STS_METRIC, "value": value, "unit": "eval/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded held-out blocks with a known acceptance temperature)",
        "config": {"workload": _sts_desc(),
                   "l2": "256 MB buffer written between timed fits (the inputs fit in L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"kernel": f"sts_fit_kernel: one cooperative launch, {STS['gamma']} positions",
                     "bound": "alu", "achieved": achieved, "peak": peak, "unit": "G eval/s",
                     "frac": achieved / peak,
                     "peak_kind": (f"MUFU: {sm} SMs x 32/3 evaluations per clock (one ex2 at "
                                   f"32/clk, one rcp at 16/clk, measured) x {mhz:.0f} MHz (sampled)"),
                     "timing": "CUDA events around the whole fit (memset + one cooperative launch)",
                     "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if not args.no_e2e:
        h_s = torch.as_tensor(s).pin_memory()
        h_n = torch.as_tensor(n).pin_memory()
        h_T = torch.empty(STS["gamma"], dtype=torch.float32).pin_memory()
        h_e = torch.empty(STS["gamma"], dtype=torch.float64).pin_memory()
        tot = 0.0
        for i in range(args.steps + 2):
            a, b = mk(), mk()
            a.record(stream)
            logit.copy_(h_s, non_blocking=True)
            n_acc.copy_(h_n, non_blocking=True)
            out = fit()
            h_T.copy_(out["T"], non_blocking=True)
            h_e.copy_(out["ece"], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                tot += a.elapsed_time(b)
        line["e2e"] = {"value": args.steps * evals / (tot / 1e3), "unit": "eval/s",
                       "h2d_bytes_per_step": int(s.nbytes + n.nbytes),
                       "d2h_bytes_per_step": STS["gamma"] * 12}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _sts_cpu()
    return line, rank


def run_sts_reference(args, world, rank):
    if rank != 0:
        return None
    cpu = _sts_cpu(budget_s=max(1.0, 1.5 * args.steps))
    evals = STS["M"] * STS["gamma"] * STS["G"]
    return {"metric": STS_METRIC, "value": cpu["value"], "unit": "eval/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * evals / cpu["value"],
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": {"workload": _sts_desc(), "sample": cpu["sample"]},
            "cpu_baseline": cpu,
            "e2e": {"value": cpu["value"], "unit": "eval/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


TRAIN = {"B": 64, "gamma": 8, "V": 151936}
TRAIN_METRIC = "drafter training losses + gradient: positions/s at 1 GB300; % of HBM roofline"


def _train_desc():
    return (f"train_loss: B={TRAIN['B']} blocks x gamma={TRAIN['gamma']} positions, V={TRAIN['V']}, "
            f"bf16 draft and target logits, fp32 gradient")


def _train_bytes():
    N, V = TRAIN["B"] * TRAIN["gamma"], TRAIN["V"]
    return 2 * N * V * 2 + N * V * 4 + N * (4 + 4 + 4 + 24)  # logits read once, gradient written


def _train_cpu(budget_s=12.0, n_blocks=1):
    """The oracle (losses + gradient) on the first n_blocks blocks, per position."""
    import oracle as orc
    orc.build()
    inp = W.train_loss_inputs(n_blocks, TRAIN["gamma"], TRAIN["V"], seed=21, device="cpu")
    zd, zt = W.bf16_bits(inp["zd"]), W.bf16_bits(inp["zt"])
    xs, sv = inp["xs"].numpy(), inp["s"].numpy()
    done, t0 = 0, time.perf_counter()
    while True:
        orc.train_losses(zd, zt, xs, sv, TRAIN["gamma"], want_grad=True)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 50:
            break
    pos = done * n_blocks * TRAIN["gamma"]
    return {"value": pos / el, "unit": "positions/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} calls on {n_blocks} block(s) of the workload (gamma={TRAIN['gamma']}, "
                      f"V={TRAIN['V']}, losses and gradient), single-threaded C oracle, {el:.1f} s"}


def run_train_loss(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g = TRAIN["gamma"]
    inp = W.train_loss_inputs(TRAIN["B"], g, TRAIN["V"], seed=21 + rank, device=dev)
    N = TRAIN["B"] * g
    grad = torch.empty((N, TRAIN["V"]), dtype=torch.float32, device=dev)
    loss = torch.empty(4, dtype=torch.float64, device=dev)
    call = lambda: dsp.train_losses(inp["zd"], inp["zt"], inp["xs"], inp["s"], g, want_grad=True)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for a, b in ev:
        flush.zero_()
        torch.cuda._sleep(2_000_000)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    times = [a.elapsed_time(b) for a, b in ev]
    total_ms, value = aggregate_ranks(sum(times), args.steps * N, world, dev)
    call_us = 1e3 * statistics.mean(times)
    achieved = _train_bytes() / (call_us * 1e-6) / 1e9
    peak, _, peak_src = _peaks()
    train_traffic = ncu_traffic("train_loss_resident", "train_loss")
    line = {
        "metric": TRAIN_METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->f32",
        "data": "synthetic (seeded draft and target logits of the draft workloads' distribution)",
        "config": {"workload": _train_desc(),
                   "l2": "256 MB buffer written between timed calls; the logits (311 MB) exceed L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"kernel": "train_loss_resident: one launch, clusters of 8 CTAs each holding 1/8 of a row "
                               "pair in shared memory (memset of the 4 totals before it)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_src} copy bandwidth",
                     "algorithmic_bytes_per_launch": _train_bytes(),
                     "bytes_rule": "draft and target logits read once, fp32 gradient written once",
                     "timing": "CUDA events around the whole call", "traffic": train_traffic[0],
                     "traffic_source": train_traffic[1]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if not args.no_e2e:
        h_d, h_t = inp["zd"].cpu().pin_memory(), inp["zt"].cpu().pin_memory()
        h_loss = torch.empty(4, dtype=torch.float64).pin_memory()
        tot = 0.0
        for i in range(args.steps + 2):
            a, b = mk(), mk()
            a.record(stream)
            inp["zd"].copy_(h_d, non_blocking=True)
            inp["zt"].copy_(h_t, non_blocking=True)
            out = call()
            h_loss.copy_(out["loss"], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                tot += a.elapsed_time(b)
        line["e2e"] = {"value": args.steps * N / (tot / 1e3), "unit": "positions/s",
                       "h2d_bytes_per_step": int(h_d.numel() * 2 + h_t.numel() * 2), "d2h_bytes_per_step": 32}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _train_cpu()
    return line, rank


def run_train_reference(args, world, rank):
    if rank != 0:
        return None
    cpu = _train_cpu(budget_s=max(1.0, 1.5 * args.steps))
    N = TRAIN["B"] * TRAIN["gamma"]
    return {"metric": TRAIN_METRIC, "value": cpu["value"], "unit": "positions/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * N / cpu["value"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": {"workload": _train_desc(), "sample": cpu["sample"]},
            "cpu_baseline": cpu,
            "e2e": {"value": cpu["value"], "unit": "positions/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


SCHED_PROFILE = {"gamma": 16, "R": [16, 32, 64, 128, 256, 512], "d": 2560, "layers": 2, "step": 8}
SCHED_METRIC = "scheduler on a profiled SPS(B) table: expected throughput Theta (tok/s) at R=256, gamma=16"


def run_sched_profile(args, world, rank, local):
    """Profile SPS(B) from the stand-in target forward, then schedule on it."""
    from speculative_decoding_drafter_markov_gb300 import sps as sps_mod
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = SCHED_PROFILE
    g = cfg["gamma"]
    B_min, B_max = min(cfg["R"]), max(cfg["R"]) * (g + 1)
    fwd = W.stand_in_target(d=cfg["d"], layers=cfg["layers"], max_B=B_max, device=dev, seed=rank)
    t0 = time.perf_counter()
    table = sps_mod.profile_sps(fwd, B_min, B_max, step=cfg["step"], reps=3)
    prof_s = time.perf_counter() - t0
    t_d = torch.as_tensor(table, device=dev)
    curve = []
    for R in cfg["R"]:
        c_d = torch.as_tensor(W.confidences(R, g, seed=1000 + R), device=dev)
        brk = dsp.schedule(c_d, t_d, B_min, mode=dsp.SCHED_SYNC)
        nob = dsp.schedule(c_d, t_d, B_min, mode=dsp.SCHED_ASYNC, K_in=brk["K_out"])
        torch.cuda.synchronize()
        curve.append({"R": R, "ell_break": float(brk["ell"].float().mean()),
                      "ell_nobreak": float(nob["ell"].float().mean()),
                      "theta_break": float(brk["theta_best"][0]), "theta_nobreak": float(nob["theta_best"][0])})
    at = next(p for p in curve if p["R"] == 256)
    # where the measured curve falls: the largest one-step drops of SPS(B)
    drops = np.argsort(table[1:] / table[:-1])[:4]
    line = {
        "metric": SCHED_METRIC, "value": at["theta_nobreak"], "unit": "tok/s", "n_gpus": world,
        "steps": 1, "warmup": 0, "ms_per_step": 1e3 * prof_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic confidences; SPS(B) measured on this GPU",
        "config": {"workload": (f"sched_profile: stand-in target {cfg['layers']} x (bf16 GEMM [B,{cfg['d']}]x"
                                f"[{cfg['d']},{3 * cfg['d']}] + [B,{3 * cfg['d']}]x[{3 * cfg['d']},{cfg['d']}]), "
                                f"B={B_min}..{B_max} every {cfg['step']}; R={cfg['R']}, gamma={g}"),
                   "parallelism": f"replicas x{world}"},
        "theta_break_at_256": at["theta_break"],
        "budget_vs_load": curve,
        "sps_table": {"B_min": B_min, "B_max": B_max, "sps_at_B_min": float(table[0]),
                      "sps_at_B_max": float(table[-1]),
                      "largest_drops_at_B": [int(B_min + 1 + i) for i in drops],
                      "profile_seconds": prof_s},
        "gpu_launches": 2 * len(cfg["R"]),
    }
    return line, rank


def main():
    args = _args()
    world, rank, local = _dist()
    if args.workload == "sched_profile":
        if args.impl == "reference":
            line = None if rank != 0 else {"impl": "reference", "unavailable":
                                           "the profiled table is a measurement of this GPU; no CPU counterpart"}
        else:
            line, rank = run_sched_profile(args, world, rank, local)
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.workload in ("sts_fit", "train_loss"):
        sts = args.workload == "sts_fit"
        if args.impl == "reference":
            line = run_sts_reference(args, world, rank) if sts else run_train_reference(args, world, rank)
        else:
            line, rank = (run_sts_fit if sts else run_train_loss)(args, world, rank, local)
        if line is not None and rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line, rank = run_dspark(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
