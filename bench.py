#!/usr/bin/env python3
"""Benchmark of the WKV operator on one or more B300 GPUs (one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line on rank 0.  A step is one pass of the training hot path
over one batch of seeded synthetic input already resident in HBM: the
forward call (which also writes the chunk checkpoints) followed by the
backward call (gradients of w, u, k, v), for the named workload (default
``l1b5``: B=16, T=4096, C=2048, fp32, one layer of a 1.5B-class model, the
largest forward+backward shape).  Other workloads: ``tiny``, ``l169m``
(B=8 T=1024 C=768, one layer of a 169M RWKV-4), ``long`` (forward only,
bf16 k/v, B=1 T=131072 C=2560), ``decode`` / ``decode_bf16`` (one fused
decode step of L=32 layers, B=256, C=4096, fp32 / bf16 token inputs, state
carried across steps), and the pointwise neighbours ``shift``, ``cmix``,
``l169m_bf16``, ``l169m_gated``.

Timing: W untimed warm-up steps; then the step (the forward call, then the
backward call) is captured once as a CUDA graph (as a training loop would run
it; ``--no-graph`` calls the API every step instead) and K steps replay it.
L2 is flushed before every timed step, outside the step's CUDA-event pair: a
write of twice its size, then a read of another buffer of twice its size, so
that the lines the write left dirty are written back before the step and not
during it.  The value is the elements of all ranks over the max over ranks of
the summed per-step device times.  For the roofline entry the dominant call
is timed in K more steps, the forward and backward calls replayed as graphs
of their own with CUDA events around the dominant one on the launching
stream.  SM clocks and
clock-event reasons are sampled (NVML, else nvidia-smi) during the timed steps.

``--impl reference`` times the float64 CPU oracle (oracle/) on this
machine's host cores instead: each step is a bounded sample of the same
workload (a subset of channels), so the whole run ends within minutes.
Under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "WKV fwd+bwd B·T·C elements/s and achieved HBM GB/s fraction on 1 B300"
METRIC_FWD = "WKV forward B·T·C elements/s and achieved HBM GB/s fraction on 1 B300"
METRIC_DEC = "WKV decode step L·B·C elements/s and achieved HBM GB/s fraction on 1 B300"
METRIC_SHIFT = "token shift fwd+bwd B·T·C elements/s and achieved HBM GB/s fraction on 1 B300"
METRIC_CMIX = "channel-mix pointwise fwd+bwd B·T·C elements/s and achieved HBM GB/s fraction on 1 B300"
METRIC_GATED = "gated WKV sigmoid(r)*wkv fwd+bwd B·T·C elements/s and achieved HBM GB/s fraction on 1 B300"

# Algorithmic HBM bytes per element (what the method must move with the
# separate forward / backward calls; O(1/chunk) checkpoint and workspace
# traffic excluded).
BYTES_FWD_F32 = 12   # read k, v; write y
BYTES_FWD_BF16 = 8   # read bf16 k, v; write fp32 y
BYTES_BWD = 20       # read k, v, gy; write gk, gv
BYTES_BWD_BF16 = 14  # read bf16 k, v, gy; write fp32 gk, gv
BYTES_DECODE = 60    # read x, x_prev, r, k, v; read+write num, den, pp; write y, xk, xv, xr
BYTES_DECODE_BF16 = 50  # the same with bf16 x, x_prev, r, k, v
BYTES_SHIFT_FWD = 16  # read x; write xk, xv, xr
BYTES_SHIFT_BWD = 20  # read x, gxk, gxv, gxr; write gx
BYTES_SQRELU_FWD = 8    # read k; write max(k, 0)^2                 (per hidden element)
BYTES_SQRELU_BWD = 12   # read k, ga; write gk                      (per hidden element)
BYTES_CMIX_GATE_FWD = 12  # read r, vk; write out
BYTES_CMIX_GATE_BWD = 20  # read r, vk, gout; write gr, gvk
BYTES_FWD_GATED = 16  # read k, v, r; write sigmoid(r) * wkv
BYTES_BWD_GATED = 28  # read k, v, r, gout; write gk, gv, gr

REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default depends on the workload)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="l1b5", choices=["tiny", "l169m", "l1b5", "long", "l169m_bf16",
                                                             "l169m_gated", "decode", "decode_bf16", "shift",
                                                             "cmix"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-graph", action="store_true",
                    help="call the API every step instead of replaying CUDA graphs of the calls")
    ap.add_argument("--scan-mode", default="auto", choices=["auto", "chunked", "sequential"],
                    help="scan strategy of the forward/backward calls (default: the library's choice by shape)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


DEFAULT_STEPS = {"tiny": 2000, "l169m": 4000, "l1b5": 200, "long": 200, "l169m_bf16": 4000, "l169m_gated": 4000,
                 "decode": 256, "decode_bf16": 256, "shift": 200, "cmix": 1000}
DECODE_WORKLOADS = ("decode", "decode_bf16")


# ------------------------------------------------------------------ ranks
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks of a float (host value; torch.distributed for N > 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate(per_rank_seconds: float, units_per_rank: float, world: int, device=None):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    t = reduce_max(per_rank_seconds, world, device)
    return world * units_per_rank / t, t


# ----------------------------------------------------------------- clocks
class CtypesNvml:
    """The few read-only NVML calls the clock sampler makes, through ctypes
    on the driver's libnvidia-ml.so.1: for hosts where the pynvml module is
    not installed.  `lib` stands in for the library in host tests."""

    NVML_CLOCK_SM = 1  # nvmlClockType_t: the SM clock domain

    def __init__(self, lib=None):
        import ctypes

        self._c = ctypes
        self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        self._check(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    @staticmethod
    def _check(status, what):
        if status != 0:
            raise RuntimeError(f"{what} returned NVML status {status}")

    def nvmlInit(self):
        pass  # initialised in the constructor

    def nvmlDeviceGetHandleByIndex(self, index):
        h = self._c.c_void_p()
        self._check(self.lib.nvmlDeviceGetHandleByIndex_v2(self._c.c_uint(index), self._c.byref(h)),
                    "nvmlDeviceGetHandleByIndex_v2")
        return h

    def _clock(self, fn, name, h, domain):
        v = self._c.c_uint()
        self._check(fn(h, self._c.c_int(domain), self._c.byref(v)), name)
        return v.value

    def nvmlDeviceGetClockInfo(self, h, domain):
        return self._clock(self.lib.nvmlDeviceGetClockInfo, "nvmlDeviceGetClockInfo", h, domain)

    def nvmlDeviceGetMaxClockInfo(self, h, domain):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo, "nvmlDeviceGetMaxClockInfo", h, domain)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if fn is None:  # the older name of the same call
            fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = self._c.c_ulonglong()
        self._check(fn(h, self._c.byref(v)), "nvmlDeviceGetCurrentClocksEventReasons")
        return v.value


class ClockSampler:
    """Samples the SM clock and clock-event reasons during a timed region
    (read only): through NVML (the pynvml module, else the driver's NVML
    library through ctypes) every 2 ms, else by running
    ``nvidia-smi --query-gpu=... -lms 10`` and reading its output."""

    NAMES = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
        0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
        0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.002):
        self.index = index
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.source = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.nv = None
        errors = []
        for source in ("nvml", "nvml (ctypes)"):
            try:
                if source == "nvml":
                    import pynvml as nv

                    nv.nvmlInit()
                else:
                    nv = CtypesNvml()
                self.h = nv.nvmlDeviceGetHandleByIndex(index)
                self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(self.h, nv.NVML_CLOCK_SM)
                self.nv, self.source = nv, source
                break
            except Exception as e:
                errors.append(f"{source}: {e}")
        self.error = "; ".join(errors) or None

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(float(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)))
                mask = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self.NAMES.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            self._stop.wait(self.period)

    def _run_smi(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append(float(parts[0]))
                self.max_mhz = float(parts[1])
                mask = int(parts[2], 16)
            except ValueError:
                continue
            for bit, name in self.NAMES.items():
                if mask & bit:
                    self.reasons.add(name)
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 parts[3:7]):
                if val.lower() == "active":
                    self.reasons.add(name)

    def __enter__(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
            return self
        import subprocess

        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "10"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError as e:
            self.error = f"{self.error}; nvidia-smi: {e}"
            return self
        self._thread = threading.Thread(target=self._run_smi, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0:  # first sample before the timed region
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "source": self.source,
                    "error": self.error}
        reasons = sorted(self.reasons - {"gpu_idle"})
        out = {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": reasons,
               "samples": len(self.samples), "source": self.source}
        if self.source == "nvidia-smi" and self.error:
            out["nvml_error"] = self.error[:160]
        return out

    def rejected(self) -> bool:
        s = self.summary()
        if any(r in s["reasons"] for r in REJECT_REASONS):
            return True
        # clocks stuck well below max with no reason: a leftover clock lock
        return bool(s["sm_mhz"] and s["sm_max_mhz"] and s["sm_mhz"] < 0.6 * s["sm_max_mhz"] and not s["reasons"])


# ---------------------------------------------------------------- helpers
# The source files each kernel is compiled from (its .cu file and the
# headers that file includes): a traffic record stays valid while these are
# unchanged.
_HEADERS = ("wkv_common.cuh", "wkv_internal.h")
KERNEL_FILES = {
    "seq_": ("wkv_seq.cu", "wkv_adjoint.cuh", "wkv_pipe.cuh") + _HEADERS,
    "decode_kernel": ("wkv_decode.cu",) + _HEADERS,
    "shift_": ("wkv_shift.cu",) + _HEADERS,
    "cmix_kernel": ("wkv_cmix.cu",) + _HEADERS,
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the sources of `kernel` (by its name's prefix), or of every
    file under csrc/ when the kernel is None or unlisted."""
    h = hashlib.sha256()
    csrc = ROOT / "rwkv_linear_attention_backward_b300" / "csrc"
    files = next((f for pre, f in KERNEL_FILES.items() if kernel and kernel.startswith(pre)), None)
    paths = sorted(csrc.glob("*")) if files is None else [csrc / n for n in sorted(files)]
    for p in paths:
        h.update(p.name.encode())
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    f = ROOT / "profiles" / "ncu_traffic.json"
    if not f.exists():
        return None
    try:
        rec = json.loads(f.read_text()).get(f"{kernel}@{workload}")
    except ValueError:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# ------------------------------------------------------------- ours: setup
class TrainingRun:
    def __init__(self, name: str, device):
        import torch
        from rwkv_linear_attention_backward_b300 import binding, inputs

        self.torch, self.wkv = torch, binding
        self.wl = inputs.WORKLOADS[name]
        wl = self.wl
        self.host = inputs.workload_inputs(name)  # (w, u, k, v, gy[, r]) on the CPU
        self.dev = tuple(t.to(device).contiguous() for t in self.host)
        B, T, C = wl.B, wl.T, wl.C
        self.elements = wl.elements
        self.y = torch.empty(B, T, C, device=device)
        self.ckpt = torch.empty(binding.checkpoint_floats(B, T, C), device=device)
        self.gw = torch.empty(C, device=device)
        self.gu = torch.empty(C, device=device)
        self.gk = torch.empty(B, T, C, device=device)
        self.gv = torch.empty(B, T, C, device=device)
        self.gr = torch.empty(B, T, C, device=device) if wl.gated else None
        self.ws_f = binding.Workspace(binding.forward_workspace_bytes(B, T, C), device)
        self.ws_b = binding.Workspace(binding.backward_workspace_bytes(B, T, C), device)
        kv_bytes = BYTES_FWD_BF16 if wl.kv_dtype == "bf16" else BYTES_FWD_F32
        bwd_bytes = BYTES_BWD_BF16 if wl.kv_dtype == "bf16" else BYTES_BWD
        if wl.gated:
            assert wl.kv_dtype == "f32"
            kv_bytes, bwd_bytes = BYTES_FWD_GATED, BYTES_BWD_GATED
        self.bytes_fwd = kv_bytes * self.elements
        self.bytes_bwd = bwd_bytes * self.elements if wl.backward else 0
        self.launches_per_step = 1 + (2 if wl.backward else 0)
        from rwkv_linear_attention_backward_b300 import binding

        self.strategy = binding.scan_strategy(wl.B, wl.T, wl.C)
        if self.strategy == "sequential":
            self.dominant = "seq_bwd_kernel" if wl.backward else "seq_fwd_kernel"
        else:
            self.dominant = "bwd_scan_kernel" if wl.backward else "fwd_scan_kernel"
        self.dominant_bytes = self.bytes_bwd if wl.backward else self.bytes_fwd

    def _forward(self):
        w, u, k, v = self.dev[:4]
        if self.wl.gated:
            self.wkv.forward_gated(w, u, k, v, self.dev[5], out=self.y, ckpt=self.ckpt, workspace=self.ws_f)
        else:
            self.wkv.forward(w, u, k, v, y=self.y, ckpt=self.ckpt, workspace=self.ws_f)

    def _backward(self):
        w, u, k, v, gy = self.dev[:5]
        if self.wl.gated:
            self.wkv.backward_gated(w, u, k, v, self.dev[5], gy, ckpt=self.ckpt, gw=self.gw, gu=self.gu, gk=self.gk,
                                    gv=self.gv, gr=self.gr, workspace=self.ws_b)
        else:
            self.wkv.backward(w, u, k, v, gy, ckpt=self.ckpt, gw=self.gw, gu=self.gu, gk=self.gk, gv=self.gv,
                              workspace=self.ws_b)

    def capture(self):
        """CUDA graphs of the forward and the backward call on the run's
        buffers (after warm-up: per-device set-up stays out of the capture),
        replayed by the timed steps as a training loop would."""
        torch = self.torch
        self.g_fwd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_fwd):
            self._forward()
        self.g_bwd = None
        self.g_step = self.g_fwd
        if self.wl.backward:
            self.g_bwd = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_bwd):
                self._backward()
            self.g_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.g_step):
                self._forward()
                self._backward()
        torch.cuda.synchronize()

    def step(self, ev=None):
        graphs = getattr(self, "g_fwd", None) is not None
        if graphs and ev is None:
            self.g_step.replay()  # the whole step as one graph
            return
        self.g_fwd.replay() if graphs else self._forward()
        if self.wl.backward:
            if ev is not None:
                ev[0].record()
            self.g_bwd.replay() if graphs else self._backward()
            if ev is not None:
                ev[1].record()

    def step_dominant_events(self, ev):
        """A step with the dominant call bracketed by the events `ev`."""
        if self.wl.backward:
            self.step(ev)
        else:
            ev[0].record()
            self.g_fwd.replay() if getattr(self, "g_fwd", None) is not None else self._forward()
            ev[1].record()

    def check(self):
        self.wkv.workspace_check(self.ws_f)
        self.wkv.workspace_check(self.ws_b)

    # end to end through the public API with host buffers
    def e2e_setup(self):
        """Pinned host buffers and two device slots of inputs and outputs
        (slot 0: the timed run's own buffers)."""
        torch = self.torch
        self.pin_in = tuple(t.pin_memory() for t in self.host)
        self._slots = [(self.dev, tuple(self._outputs()))]
        self._slots.append((tuple(torch.empty_like(t) for t in self.dev),
                            tuple(torch.empty_like(t) for t in self._outputs())))
        self.pin_out = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in self._outputs())
                        for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for t in self.pin_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.pin_out[0])

    def _outputs(self):
        grads = [self.gk, self.gv, self.gw, self.gu] + ([self.gr] if self.wl.gated else [])
        return [self.y] + (grads if self.wl.backward else [])

    def e2e_inputs(self, k):
        return self._slots[k][0]

    def e2e_compute(self, k):
        """The step's calls on slot k's inputs into slot k's outputs."""
        dev, outs = self._slots[k]
        self.dev = dev
        self.y = outs[0]
        if self.wl.backward:
            self.gk, self.gv, self.gw, self.gu = outs[1:5]
            if self.wl.gated:
                self.gr = outs[5]
        self._forward()
        if self.wl.backward:
            self._backward()
        return outs


class DecodeRun:
    def __init__(self, device, name="decode"):
        import torch
        from rwkv_linear_attention_backward_b300 import binding, inputs

        self.torch, self.wkv = torch, binding
        D = inputs.DECODES[name]
        self.D = D
        L, B, C = D.L, D.B, D.C
        self.elements = D.elements_per_step
        self.params = tuple(t.to(device) for t in inputs.decode_params(L, C, seed=D.seed, d_lo=D.d_lo, d_hi=D.d_hi))
        self.pool = inputs.decode_pool(L, B, C, seed=D.seed, n_sets=16, device=device, token_dtype=D.token_dtype)
        self.state = tuple(t.to(device) for t in inputs.initial_state(L, B, C))
        self.out = tuple(torch.empty(L, B, C, device=device) for _ in range(4))
        self.t = 0
        self.bytes_fwd = (BYTES_DECODE_BF16 if D.token_dtype == "bf16" else BYTES_DECODE) * self.elements
        self.bytes_bwd = 0
        self.launches_per_step = 1
        self.dominant = "decode_kernel_vec4<__nv_bfloat16>" if D.token_dtype == "bf16" else "decode_kernel_vec4<float>"
        self.dominant_bytes = self.bytes_fwd

    def step(self, ev=None):
        x, xp, r, k, v = self.pool[self.t % len(self.pool)]
        mk, mv, mr, w, u = self.params
        y, xk, xv, xr = self.out
        if ev is not None:
            ev[0].record()
        self.wkv.decode_step(x, xp, mk, mv, mr, r, k, v, w, u, *self.state, y=y, xk=xk, xv=xv, xr=xr)
        if ev is not None:
            ev[1].record()
        self.t += 1

    step_dominant_events = step

    def capture(self):
        pass  # one launch per step, on a rotating input set: called directly

    def check(self):
        pass

    def e2e_setup(self):
        torch = self.torch
        self.pin_in = tuple(t.to("cpu").pin_memory() for t in self.pool[0])
        self._slots = [(self.pool[0], self.out[0]), (self.pool[1], torch.empty_like(self.out[0]))]
        self.pin_out = [(torch.empty(self.out[0].shape, pin_memory=True),) for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for t in self.pin_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.pin_out[0])

    def e2e_inputs(self, k):
        return self._slots[k][0]

    def e2e_compute(self, k):
        (x, xp, r, kk, v), y = self._slots[k]
        mk, mv, mr, w, u = self.params
        _, xk, xv, xr = self.out
        self.wkv.decode_step(x, xp, mk, mv, mr, r, kk, v, w, u, *self.state, y=y, xk=xk, xv=xv, xr=xr)
        return (y,)


class ShiftRun:
    """A step is the token shift's forward and backward calls (the training
    path's mix of each token with the previous one)."""

    def __init__(self, device):
        import torch
        from rwkv_linear_attention_backward_b300 import binding, inputs

        self.torch, self.wkv = torch, binding
        S = inputs.SHIFT
        self.S = S
        B, T, C = S.B, S.T, S.C
        self.elements = S.elements
        self.host = inputs.shift_inputs(B, T, C, seed=S.seed)
        self.dev = tuple(t.to(device).contiguous() for t in self.host)
        self.out = tuple(torch.empty(B, T, C, device=device) for _ in range(3))
        self.ws = binding.Workspace(binding._lib.wkv_token_shift_backward_workspace_bytes(B, T, C), device)
        self.bytes_fwd = BYTES_SHIFT_FWD * self.elements
        self.bytes_bwd = BYTES_SHIFT_BWD * self.elements
        self.launches_per_step = 3
        self.dominant = "shift_bwd_kernel"
        self.dominant_bytes = self.bytes_bwd

    def _forward(self):
        x, x0, mk, mv, mr = self.dev[:5]
        self.wkv.token_shift(x, x0, mk, mv, mr, xk=self.out[0], xv=self.out[1], xr=self.out[2])

    def _backward(self):
        return self.wkv.token_shift_backward(*self.dev, workspace=self.ws)

    def step(self, ev=None):
        self._forward()
        if ev is not None:
            ev[0].record()
        self._backward()
        if ev is not None:
            ev[1].record()

    step_dominant_events = step

    def capture(self):
        pass  # two API calls per step

    def check(self):
        pass

    def e2e_setup(self):
        torch = self.torch
        self.pin_in = tuple(t.pin_memory() for t in self.host)
        self._slots = [(self.dev, self.out), (tuple(torch.empty_like(t) for t in self.dev),
                                              tuple(torch.empty_like(t) for t in self.out))]
        self.pin_out = [tuple(torch.empty(self.S.B, self.S.T, self.S.C, pin_memory=True) for _ in range(4))
                        for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for t in self.pin_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.pin_out[0])

    def e2e_inputs(self, k):
        return self._slots[k][0]

    def e2e_compute(self, k):
        self.dev, self.out = self._slots[k]
        self._forward()
        gx = self._backward()[0]  # allocated by the call: the copy-out stream marks its use
        return self.out + (gx,)


# --------------------------------------------------------------- ours: run
class CmixRun:
    """A step is channel mixing's four pointwise calls: the squared ReLU
    and the gate forward, then the gate's and the squared ReLU's backward
    (the projections between them are the caller's matmuls, not timed)."""

    def __init__(self, device):
        import torch
        from rwkv_linear_attention_backward_b300 import binding, inputs

        self.torch, self.wkv = torch, binding
        M = inputs.CMIX
        self.M = M
        self.elements = M.elements
        self.host = inputs.cmix_inputs(M.B, M.T, M.C, M.H, seed=M.seed)
        self.dev = tuple(t.to(device).contiguous() for t in self.host)
        k, _, r, _, _ = self.dev
        self.out = (torch.empty_like(k), torch.empty_like(r), torch.empty_like(r), torch.empty_like(r),
                    torch.empty_like(k))  # a, out, gr, gvk, gk
        hid = M.B * M.T * M.H
        self.bytes_fwd = BYTES_SQRELU_FWD * hid + BYTES_CMIX_GATE_FWD * self.elements
        self.bytes_bwd = BYTES_SQRELU_BWD * hid + BYTES_CMIX_GATE_BWD * self.elements
        self.launches_per_step = 4
        self.dominant = "cmix_kernel<1, 4> (squared-ReLU backward)"
        self.dominant_bytes = BYTES_SQRELU_BWD * hid

    def _forward(self):
        k, _, r, vk, _ = self.dev
        self.wkv.channel_mix_sqrelu(k, out=self.out[0])
        self.wkv.channel_mix_gate(r, vk, out=self.out[1])

    def _gate_backward(self):
        _, _, r, vk, gout = self.dev
        self.wkv.channel_mix_gate_backward(r, vk, gout, gr=self.out[2], gvk=self.out[3])

    def _sqrelu_backward(self):
        k, ga = self.dev[:2]
        self.wkv.channel_mix_sqrelu_backward(k, ga, gk=self.out[4])

    def step(self, ev=None):
        self._forward()
        self._gate_backward()
        if ev is not None:
            ev[0].record()
        self._sqrelu_backward()
        if ev is not None:
            ev[1].record()

    step_dominant_events = step

    def capture(self):
        pass  # four API calls per step

    def check(self):
        pass

    def e2e_setup(self):
        torch = self.torch
        self.pin_in = tuple(t.pin_memory() for t in self.host)
        self._slots = [(self.dev, self.out), (tuple(torch.empty_like(t) for t in self.dev),
                                              tuple(torch.empty_like(t) for t in self.out))]
        self.pin_out = [tuple(torch.empty(t.shape, pin_memory=True) for t in self.out) for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for t in self.pin_in)
        self.d2h = sum(t.numel() * t.element_size() for t in self.pin_out[0])

    def e2e_inputs(self, k):
        return self._slots[k][0]

    def e2e_compute(self, k):
        self.dev, self.out = self._slots[k]
        self._forward()
        self._gate_backward()
        self._sqrelu_backward()
        return self.out


def time_steps(run, steps: int, flush, stream):
    """Per-step device times (s) of `steps` steps, L2 flushed before each;
    then, in `steps` more steps, the dominant call's per-launch times."""
    torch = run.torch
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ev_dom = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush()
        ev_step[i][0].record(stream)
        run.step()
        ev_step[i][1].record(stream)
    for i in range(steps):
        flush()
        run.step_dominant_events(ev_dom[i])
    torch.cuda.synchronize()
    step_s = [a.elapsed_time(b) / 1e3 for a, b in ev_step]
    dom_s = [a.elapsed_time(b) / 1e3 for a, b in ev_dom]
    return step_s, dom_s


def cpu_baseline(workload: str, target_s: float = 12.0):
    """Time the float64 oracle (recurrent forward + adjoint backward, or the
    decode step) on this host's cores on a bounded sample of the workload:
    a subset of channels (decode: of batch rows), grown until about
    target_s of CPU work."""
    import numpy as np

    import oracle
    from rwkv_linear_attention_backward_b300 import inputs

    o = oracle.load()
    if workload in DECODE_WORKLOADS:
        D = inputs.DECODES[workload]
        L, B, C = D.L, D.B, D.C
        params = [p.numpy() for p in inputs.decode_params(L, C, seed=D.seed, d_lo=D.d_lo, d_hi=D.d_hi)]
        rows = 16
        x, xp, r, k, v = (t.float().numpy()[:, :rows] for t in
                          inputs.decode_step_inputs(L, B, C, seed=D.seed, step=0, token_dtype=D.token_dtype))
        st = [t.numpy()[:, :rows] for t in inputs.initial_state(L, B, C)]
        done, t0, steps = 0, time.perf_counter(), 0
        while time.perf_counter() - t0 < target_s:
            y, *st, _, _, _ = o.decode_step(x, xp, *params[:3], r, k, v, *params[3:], *st)
            done += L * rows * C
            steps += 1
        el = time.perf_counter() - t0
        return {"value": done / el, "unit": "elements/s", "cores": o.num_threads(), "kind": "oracle",
                "sample": f"decode step on batch rows 0..{rows - 1} of {B} (all {L} layers, all {C} channels), "
                          f"{steps} steps in {el:.1f} s"}
    if workload == "shift":
        return _shift_oracle_timing(o, target_s)
    if workload == "cmix":
        return _cmix_oracle_timing(o, target_s)
    wl = inputs.WORKLOADS[workload]
    w, u, k, v, gy, *r = inputs.workload_inputs(workload)
    r = r[0] if r else None
    C = wl.C
    nchan = C
    # calibrate on a few channels, then size the sample for ~target_s
    cs = np.arange(min(8, C))
    t0 = time.perf_counter()
    _oracle_pass(o, wl, w, u, k, v, gy, cs, r)
    per_chan = (time.perf_counter() - t0) / len(cs)
    nchan = int(max(1, min(C, target_s / max(per_chan, 1e-9) / 2)))
    cs = np.linspace(0, C - 1, nchan).astype(int)
    reps, done, t0 = 0, 0, time.perf_counter()
    while True:
        _oracle_pass(o, wl, w, u, k, v, gy, cs, r)
        reps += 1
        done += wl.B * wl.T * len(cs)
        if time.perf_counter() - t0 >= target_s or reps >= 50:
            break
    el = time.perf_counter() - t0
    what = _oracle_what(wl)
    return {"value": done / el, "unit": "elements/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"{what} on {len(cs)} of {C} channels (all B={wl.B}, T={wl.T}), {reps} pass(es) in {el:.1f} s"}


def _shift_oracle_timing(o, target_s):
    """The oracle's token shift forward + backward on batch row 0 of the
    shift workload, repeated for about target_s."""
    from rwkv_linear_attention_backward_b300 import inputs

    S = inputs.SHIFT
    x, x0, mk, mv, mr, gk, gv, gr = (t.numpy() for t in inputs.shift_inputs(1, S.T, S.C, seed=S.seed))
    reps, done, t0 = 0, 0, time.perf_counter()
    while True:
        o.token_shift(x, x0, mk, mv, mr)
        o.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
        reps += 1
        done += S.T * S.C
        if time.perf_counter() - t0 >= target_s or reps >= 200:
            break
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "elements/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"token shift forward + backward on one batch row (T={S.T}, C={S.C}) of {S.B}, "
                      f"{reps} pass(es) in {el:.1f} s"}


def _cmix_oracle_timing(o, target_s):
    """The oracle's channel-mix steps (forward and backward) on batch row 0
    of the cmix workload, repeated for about target_s."""
    from rwkv_linear_attention_backward_b300 import inputs

    M = inputs.CMIX
    k, ga, r, vk, gout = (t.numpy() for t in inputs.cmix_inputs(1, M.T, M.C, M.H, seed=M.seed))
    reps, done, t0 = 0, 0, time.perf_counter()
    while True:
        _cmix_oracle_pass(o, k, ga, r, vk, gout)
        reps += 1
        done += M.T * M.C
        if time.perf_counter() - t0 >= target_s or reps >= 200:
            break
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "elements/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"channel-mix squared ReLU + gate, forward and backward, on one batch row (T={M.T}, "
                      f"C={M.C}, H={M.H}) of {M.B}, {reps} pass(es) in {el:.1f} s"}


def _cmix_oracle_pass(o, k, ga, r, vk, gout):
    o.sqrelu(k)
    o.cmix_gate(r, vk)
    o.cmix_gate_backward(r, vk, gout)
    o.sqrelu_backward(k, ga)


def _oracle_pass(o, wl, w, u, k, v, gy, cs, r=None):
    ks, vs = k[:, :, cs], v[:, :, cs]
    if wl.gated:
        rs = r[:, :, cs]
        o.forward_gated_recurrent(w[cs], u[cs], ks, vs, rs)
        o.backward_gated(w[cs], u[cs], ks, vs, rs, gy[:, :, cs])
        return
    o.forward_recurrent(w[cs], u[cs], ks, vs)
    if wl.backward:
        o.backward_adjoint(w[cs], u[cs], ks, vs, gy[:, :, cs])


def _oracle_what(wl):
    if wl.gated:
        return "gated recurrent forward + gated adjoint backward"
    return "recurrent forward + adjoint backward" if wl.backward else "recurrent forward"


def run_ours(args):
    import torch

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    from rwkv_linear_attention_backward_b300 import build

    build.build()
    if args.scan_mode != "auto":
        from rwkv_linear_attention_backward_b300 import binding

        binding.set_scan_mode(args.scan_mode)
    steps = args.steps or DEFAULT_STEPS[args.workload]
    if args.workload in DECODE_WORKLOADS:
        run = DecodeRun(device, args.workload)
    elif args.workload == "shift":
        run = ShiftRun(device)
    elif args.workload == "cmix":
        run = CmixRun(device)
    else:
        run = TrainingRun(args.workload, device)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    scratch = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=device)
    evict = torch.ones_like(scratch)
    evict_sum = torch.empty((), dtype=torch.float32, device=device)

    def flush():
        # a write larger than L2, then a read of as much other memory: the
        # read evicts the lines the write left dirty (their write-back happens
        # here, not in the step) and leaves L2 holding none of the step's data
        scratch.fill_(1.0)
        torch.sum(evict, dim=0, out=evict_sum)

    for _ in range(args.warmup):
        flush()
        run.step()
    torch.cuda.synchronize()
    run.check()
    if not args.no_graph:
        run.capture()
        for _ in range(2):
            flush()
            run.step()
        torch.cuda.synchronize()
        run.check()

    attempts = []
    for attempt in range(2):
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(device.index) as clocks:
            step_s, dom_s = time_steps(run, steps, flush, stream)
        torch.cuda.synchronize()
        barrier(world)
        attempts.append((step_s, dom_s, clocks))
        if not clocks.rejected():
            break
    step_s, dom_s, clocks = attempts[-1]
    run.check()

    total = sum(step_s)
    value, tmax = aggregate(total, run.elements * steps, world, device)
    ms_per_step = 1e3 * tmax / steps
    peak, peak_kind = peaks()
    dom_avg = sum(dom_s) / len(dom_s)
    achieved = run.dominant_bytes / dom_avg / 1e9
    step_bytes = run.bytes_fwd + run.bytes_bwd
    if args.workload in DECODE_WORKLOADS:
        wl_cfg = {"workload": args.workload, "L": run.D.L, "B": run.D.B, "C": run.D.C,
                  "token_inputs": run.D.token_dtype, "state": "fp32"}
    elif args.workload == "shift":
        wl_cfg = {"workload": "shift", "B": run.S.B, "T": run.S.T, "C": run.S.C, "pass": "forward+backward"}
    elif args.workload == "cmix":
        wl_cfg = {"workload": "cmix", "B": run.M.B, "T": run.M.T, "C": run.M.C, "H": run.M.H,
                  "pass": "forward+backward of the squared ReLU [B,T,H] and the gate [B,T,C]"}
    else:
        wl_cfg = {"workload": args.workload, "B": run.wl.B, "T": run.wl.T, "C": run.wl.C,
                  "kv_dtype": run.wl.kv_dtype, "pass": "forward+backward" if run.wl.backward else "forward"}
        if run.wl.gated:
            wl_cfg["output"] = "sigmoid(r) * wkv, the gate fused into the forward and backward kernels"
    pointwise = DECODE_WORKLOADS + ("shift", "cmix")
    wl_cfg.update({"launch": "api calls per step" if (args.no_graph or args.workload in pointwise) else
                   "one CUDA graph of the step's calls, captured once and replayed per step",
                   "l2": "flushed before every timed step (write of 2x L2, then a read of another 2x L2 buffer)",
                   "parallelism": f"replicas x{world}",
                   "scan_mode": args.scan_mode,
                   "strategy": getattr(run, "strategy", "n/a"),
                   "checkpoints": "forward writes chunk checkpoints, backward reads them"
                   if args.workload not in pointwise else "n/a"})
    metric = {"long": METRIC_FWD, "decode": METRIC_DEC, "decode_bf16": METRIC_DEC, "shift": METRIC_SHIFT,
              "cmix": METRIC_CMIX,
              "l169m_gated": METRIC_GATED}.get(args.workload, METRIC)
    out = {
        "metric": metric,
        "value": value,
        "unit": "elements/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; see rwkv_linear_attention_backward_b300/inputs.py)",
        "config": wl_cfg,
        "achieved_hbm_gbs": step_bytes * steps / total / 1e9,
        "hbm_frac": step_bytes * steps / total / 1e9 / peak,
        "roofline": {
            "kernel": run.dominant,
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": ncu_traffic(run.dominant, args.workload),
            "algorithmic_bytes_per_launch": run.dominant_bytes,
            "launch_ms": dom_avg * 1e3,
        },
        "gpu_launches": run.launches_per_step * steps,
        "gpu_launches_roofline_pass": run.launches_per_step * steps,  # the dominant call's own K steps
        "clocks": clocks.summary(),
    }
    if len(attempts) > 1:
        out["clocks"]["remeasured"] = True
    if not args.no_e2e:
        out["e2e"] = e2e(run, steps=max(3, min(steps, 50)), world=world, device=device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def e2e(run, steps: int, world: int = 1, device=None):
    """Same metric through the public API with pinned host buffers: every
    step copies its inputs host->device, runs the step's calls and copies
    its results device->host.  Steps are pipelined as a training loop's
    data path would be: copies in on one stream, the calls on a second,
    copies out on a third, over two slots of device buffers, so step i+1's
    inputs and step i-1's results cross the host link (both directions at
    once) while step i computes.  The time is the whole sequence's, from the
    first copy in to the last copy out; with several ranks (each its own
    GPU and buffers) the value is all ranks' elements over the slowest
    rank's time."""
    torch = run.torch
    run.e2e_setup()
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def issue(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[k])  # step i-2 has read slot k's inputs
            for d, h in zip(run.e2e_inputs(k), run.pin_in):
                d.copy_(h, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[k])
            if i >= 2:
                s_comp.wait_event(ev_out[k])  # step i-2's results have left slot k
            outs = run.e2e_compute(k)
            ev_comp[k].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            for h, d in zip(run.pin_out[k], outs):
                d.record_stream(s_out)
                h.copy_(d, non_blocking=True)
            ev_out[k].record(s_out)

    def sequence(n):
        for i in range(n):
            issue(i)
        cur = torch.cuda.current_stream()
        for e in ev_out[:min(n, 2)]:
            cur.wait_event(e)

    sequence(2)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    sequence(steps)
    b.record()
    torch.cuda.synchronize()
    value, _ = aggregate(a.elapsed_time(b) / 1e3, run.elements * steps, world, device)
    return {"value": value, "unit": "elements/s", "h2d_bytes_per_step": run.h2d,
            "d2h_bytes_per_step": run.d2h, "steps": steps,
            "pipeline": "copies in, calls and copies out on three streams over two buffer slots"}


# -------------------------------------------------------------- reference
def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from rwkv_linear_attention_backward_b300 import inputs

    steps = args.steps or DEFAULT_STEPS[args.workload]
    total_budget = 120.0  # seconds for warm-up + timed steps together
    per_step = total_budget / (steps + args.warmup)
    o = oracle.load()
    if args.workload in DECODE_WORKLOADS:
        D = inputs.DECODES[args.workload]
        L, B, C = D.L, D.B, D.C
        params = [p.numpy() for p in inputs.decode_params(L, C, seed=D.seed, d_lo=D.d_lo, d_hi=D.d_hi)]
        x, xp, r, k, v = (t.float().numpy() for t in
                          inputs.decode_step_inputs(L, B, C, seed=D.seed, step=0, token_dtype=D.token_dtype))
        t0 = time.perf_counter()
        o.decode_step(x[:, :1], xp[:, :1], *params[:3], r[:, :1], k[:, :1], v[:, :1], *params[3:],
                      *[t.numpy()[:, :1] for t in inputs.initial_state(L, 1, C)])
        per_row = time.perf_counter() - t0
        rows = int(max(1, min(B, per_step / max(per_row, 1e-9))))
        st = [t.numpy()[:, :rows] for t in inputs.initial_state(L, B, C)]

        def one():
            nonlocal st
            y, *st, _, _, _ = o.decode_step(x[:, :rows], xp[:, :rows], *params[:3], r[:, :rows], k[:, :rows],
                                            v[:, :rows], *params[3:], *st)
            return L * rows * C

        sample = f"decode step on batch rows 0..{rows - 1} of {B} (all {L} layers, {C} channels)"
        metric = METRIC_DEC
    elif args.workload == "shift":
        S = inputs.SHIFT
        x, x0, mk, mv, mr, gk, gv, gr = (t.numpy() for t in inputs.shift_inputs(1, S.T, S.C, seed=S.seed))

        def one():
            o.token_shift(x, x0, mk, mv, mr)
            o.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
            return S.T * S.C

        sample = f"token shift forward + backward on one batch row (T={S.T}, C={S.C}) of {S.B}"
        metric = METRIC_SHIFT
    elif args.workload == "cmix":
        M = inputs.CMIX
        k, ga, r, vk, gout = (t.numpy() for t in inputs.cmix_inputs(1, M.T, M.C, M.H, seed=M.seed))

        def one():
            _cmix_oracle_pass(o, k, ga, r, vk, gout)
            return M.T * M.C

        sample = f"channel-mix squared ReLU + gate, forward and backward, on one batch row (T={M.T}, C={M.C}, " \
                 f"H={M.H}) of {M.B}"
        metric = METRIC_CMIX
    else:
        wl = inputs.WORKLOADS[args.workload]
        w, u, k, v, gy, *r = inputs.workload_inputs(args.workload)
        r = r[0] if r else None
        cs = np.arange(min(4, wl.C))
        t0 = time.perf_counter()
        _oracle_pass(o, wl, w, u, k, v, gy, cs, r)
        per_chan = (time.perf_counter() - t0) / len(cs)
        nchan = int(max(1, min(wl.C, per_step / max(per_chan, 1e-9))))
        cs = np.linspace(0, wl.C - 1, nchan).astype(int)

        def one():
            _oracle_pass(o, wl, w, u, k, v, gy, cs, r)
            return wl.B * wl.T * len(cs)

        sample = f"{_oracle_what(wl)} on {len(cs)} of {wl.C} channels (all B={wl.B}, T={wl.T})"
        metric = METRIC_GATED if wl.gated else (METRIC if wl.backward else METRIC_FWD)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    done = sum(one() for _ in range(steps))
    el = time.perf_counter() - t0
    value = done / el
    if args.workload in DECODE_WORKLOADS:
        cfg = {"workload": args.workload}
    elif args.workload == "shift":
        cfg = {"workload": "shift", "B": inputs.SHIFT.B, "T": inputs.SHIFT.T, "C": inputs.SHIFT.C}
    elif args.workload == "cmix":
        cfg = {"workload": "cmix", "B": inputs.CMIX.B, "T": inputs.CMIX.T, "C": inputs.CMIX.C, "H": inputs.CMIX.H}
    else:
        cfg = {"workload": args.workload, "B": inputs.WORKLOADS[args.workload].B,
               "T": inputs.WORKLOADS[args.workload].T, "C": inputs.WORKLOADS[args.workload].C}
    out = {
        "impl": "reference",
        "metric": metric,
        "value": value,
        "unit": "elements/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * el / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; see rwkv_linear_attention_backward_b300/inputs.py)",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
