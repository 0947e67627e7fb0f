"""Benchmark of the exact-attention forward path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline: attention forward TFLOPS on the long causal prefill workload (B = 2, H = 32,
N = 8192, d = 128, bf16, causal), FLOPs = 4 * Nq * Nk * d per (batch, head), halved for
causal.  One step = one fa_fwd call over that whole workload with inputs resident in HBM
(402 MB of Q/K/V, larger than the 129 MB L2).  The same JSON line also carries:
  roofline      the prefill kernel against the measured dense bf16 peak
  e2e           the same metric through the public call with pinned host buffers, the
                host->device copies of Q/K/V and the device->host copy of O/LSE timed
  cpu_baseline  the fp64 oracle on a bounded sample of rows, on this host's cores
  extra         the other workloads (dense 2k, GQA 16k causal, split-KV decode) and the
                variants (fp16, sliding window, softcap + ALiBi, backward, windowed and
                paged decode with append + rotary) measured the same way, decode against
                HBM bandwidth
Under torchrun (N > 1) every rank runs the full workload on its own GPU (weak scaling;
the (batch, head) units are independent, so there is no collective on the data path);
the step time is the max over ranks.
`--impl reference` times the fp64 CPU oracle instead (rank 0 only).
`--backward` makes the timed step the backward pass (fa_bwd) of the chosen dense workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "causal8k"
METRIC = "attention fwd TFLOPS (bf16 causal N=8192 d=128) & % of GB300 BF16 peak"
BWD_METRIC = "attention bwd TFLOPS (dQ, dK, dV; 2.5 x forward FLOPs) & % of GB300 BF16 peak"
L2_BYTES = 129 * 1024 * 1024


def flops(w) -> float:
    f = 4.0 * w.Nq * w.Nk * w.d * w.B * w.Hq
    return f / 2 if w.causal else f


def window_pairs(Nq, Nk, wl, wr) -> int:
    """Number of (query, key) pairs a sliding window (wl, wr) leaves visible (bottom-right
    positions, negative bound = unbounded)."""
    import numpy as np
    pos = np.arange(Nq, dtype=np.int64) + (Nk - Nq)
    lo = np.maximum(pos - wl, 0) if wl >= 0 else np.zeros_like(pos)
    hi = np.minimum(pos + wr, Nk - 1) if wr >= 0 else np.full_like(pos, Nk - 1)
    return int(np.maximum(hi - lo + 1, 0).sum())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm": float(p["hbm_gbs"]), "basis": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "basis": "fallback"}


def source_hash(files) -> str:
    """sha256[:12] of the kernel sources with comments and blank lines removed, so that
    a recorded capture stays valid across edits that change no code."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:12]


PREFILL_SRC = ["exact_attention_81_gb300/csrc/fa_prefill.cu", "exact_attention_81_gb300/csrc/ptx.cuh"]
DECODE_SRC = ["exact_attention_81_gb300/csrc/fa_decode.cu", "exact_attention_81_gb300/csrc/ptx.cuh"]


def profiled_traffic(kernel: str, src_files, workload: str):
    """DRAM bytes per launch recorded under profiles/ for this kernel, or None when no
    capture exists for the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    want = source_hash(src_files)
    pat = re.compile(r"^\|\s*" + re.escape(kernel) + r"\s*\|\s*" + re.escape(workload) +
                     r"\s*\|\s*([0-9a-f]+)\s*\|\s*([0-9.eE+]+)\s*\|")
    for line in open(path):
        m = pat.match(line.strip())
        if m and m.group(1) == want:
            return float(m.group(2))
    return None


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, power, clock-event
    reasons), or None attributes when the library is missing."""

    # clock-event reason bits (nvml.h: nvmlClocksEventReason*)
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, index: int, pci_bus_id: str | None = None):
        import ctypes
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            # the CUDA device by its PCI address (NVML numbers GPUs its own way), else by index
            if not pci_bus_id or lib.nvmlDeviceGetHandleByPciBusId_v2(
                    pci_bus_id.encode(), ctypes.byref(h)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                    return
            self.lib, self.h, self.ct = lib, h, ctypes
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = reasons or lib.nvmlDeviceGetCurrentClocksThrottleReasons
            v = ctypes.c_uint()
            self.max_mhz = (float(v.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(v))
                            == 0 else None)
            self.ok = True
        except Exception:
            self.ok = False

    def sample(self):
        """(sm MHz, power W, reason bits) now."""
        ct = self.ct
        mhz, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))  # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(bits))
        return float(mhz.value), mw.value / 1000.0, int(bits.value)


def _pci_bus_id(index: int):
    """PCI address of CUDA device `index` in NVML's form, or None."""
    try:
        import torch
        p = torch.cuda.get_device_properties(index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


class ClockSampler:
    """SM clock and clock-event reasons sampled in the background while the timed region
    runs: NVML every millisecond (so that a timed region of a few tens of milliseconds
    still gets tens of samples), else nvidia-smi every 25 ms."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (time, sm MHz, max MHz, set of reasons)
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.nvml = _Nvml(index, _pci_bus_id(index))
        self.source = "nvml 1 ms" if self.nvml.ok else "nvidia-smi 25 ms"

    def start(self):
        if self.nvml.ok:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        names = _Nvml.REASONS
        while not self.stop_flag.is_set():
            try:
                mhz, _, bits = self.nvml.sample()
            except Exception:
                break
            self.samples.append((time.time(), mhz, self.nvml.max_mhz or mhz,
                                 {n for n, b in names.items() if bits & b}))
            time.sleep(0.001)

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 10:
                continue
            try:
                mhz, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            self.samples.append((time.time(), mhz, mx,
                                 {n for n, v in zip(names, parts[6:10])
                                  if v.lower().startswith("active")}))

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = list(self.samples)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "window": "none", "source": self.source}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed"
        if not inside:
            after = [r for r in rows if r[0] >= t0]
            inside = after[:2] if after else rows[-2:]
            window = "nearest"
        mhz = sorted(r[1] for r in inside)
        reasons = set()
        for r in inside:
            reasons |= r[3]
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "sm_min_mhz": mhz[0], "reasons": sorted(reasons), "samples": len(inside),
                "window": window, "source": self.source}


# ----------------------------------------------------------------------------- GPU arm

DECODE_METRIC = "split-KV decode GB/s (bf16, KV cache read once) & % of GB300 HBM bandwidth"


def max_over_ranks(ms: float, dist, device) -> float:
    """Step time of the job: the slowest rank's (identity without a process group)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_workload(w, world: int, rank: int):
    """The rank's part of a workload under head sharding (strong scaling): the kv heads are
    cut into `world` contiguous ranges, each rank taking its kv heads and the query heads that
    read them (the (batch, head) units are independent, so no collective is needed and each
    GPU holds only its own K/V).  The rank draws its inputs with its own seed.  Requires Hkv
    to be a multiple of world."""
    import dataclasses
    if world == 1:
        return w
    if w.Hkv % world != 0:
        raise ValueError(f"{w.name}: {w.Hkv} kv heads do not split over {world} ranks")
    return dataclasses.replace(w, Hq=w.Hq // world, Hkv=w.Hkv // world,
                               seed=w.seed + 7919 * rank)


def job_value(work_per_rank: float, ms_step: float, world: int, scale: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes `work_per_rank`
    units per step; the job's step takes the slowest rank's time."""
    return world * work_per_rank / (ms_step * 1e-3) / scale


class DenseCase:
    """One fa_fwd call over a dense workload; work = FLOPs."""

    def __init__(self, w, dev, softcap=0.0, alibi=False):
        import torch
        from exact_attention_81_gb300.inputs import workload_inputs
        self.w = w
        self.q, self.k, self.v = workload_inputs(w, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        self.work = flops(w)
        self.launches = 1
        # score modifiers (softcap, ALiBi with the geometric slopes 2^(-8 (h + 1) / H))
        self.mods = {}
        if softcap > 0.0:
            self.mods["softcap"] = softcap
        if alibi:
            self.mods["alibi_slopes"] = torch.tensor(
                [2.0 ** (-8.0 * (h + 1) / w.Hq) for h in range(w.Hq)], dtype=torch.float32,
                device=dev)

    def step(self):
        import exact_attention_81_gb300 as fa
        fa.fa_fwd(self.q, self.k, self.v, causal=self.w.causal, out=self.out, lse=self.lse,
                  **self.mods)

    def e2e(self):
        """Pinned host Q/K/V copied in, O/LSE copied out, every step, through fa_fwd_host
        (copies of one query range overlap the computation of the previous one)."""
        import torch
        import exact_attention_81_gb300 as fa
        hq, hk, hv = (t.cpu().pin_memory() for t in (self.q, self.k, self.v))
        ho = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        hl = torch.empty(self.lse.shape, dtype=self.lse.dtype, pin_memory=True)
        bufs = tuple(torch.empty_like(t) for t in (self.q, self.k, self.v, self.out, self.lse))

        def run():
            fa.fa_fwd_host(hq, hk, hv, causal=self.w.causal, out=ho, lse=hl,
                           device_buffers=bufs, chunks=8, device=self.q.device)
        h2d = (self.q.numel() + self.k.numel() + self.v.numel()) * 2
        d2h = self.out.numel() * 2 + self.lse.numel() * 4
        return run, h2d, d2h

    def describe(self, pk, ms_step, world):
        w = self.w
        tf = self.work / (ms_step * 1e-3) / 1e12
        io = (self.q.numel() + self.k.numel() + self.v.numel()) * 2
        kernel = f"prefill_kernel<{w.d},{str(w.causal).lower()}>"
        mods = []
        if "softcap" in self.mods:
            mods.append(f"softcap {self.mods['softcap']:g}")
        if "alibi_slopes" in self.mods:
            mods.append("ALiBi 2^(-8(h+1)/H)")
        if mods:
            kernel = f"prefill_kernel<{w.d},{str(w.causal).lower()},{'+'.join(mods)}>"
        return {
            "metric": METRIC, "unit": "TFLOPS",
            "value": round(job_value(self.work, ms_step, world, 1e12), 2),
            "config": {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} Nq=Nk={w.Nq} "
                                   f"d={w.d} causal={w.causal} bf16",
                       "batch": w.B, "heads": w.Hq, "seq_len": w.Nq, "head_dim": w.d,
                       "causal": w.causal,
                       "parallelism": f"replicas x{world} (independent heads)",
                       "l2": f"inputs {io / 1e6:.0f} MB > L2 {L2_BYTES / 1e6:.0f} MB, no flush",
                       **({"modifiers": ", ".join(mods)} if mods else {})},
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16"],
                         "unit": "TFLOP/s", "frac": round(tf / pk["bf16"], 4),
                         "traffic": profiled_traffic(kernel, PREFILL_SRC, w.name),
                         "peak_basis": f"{pk['basis']} bf16 dense (burst)",
                         "kernel": f"{kernel} (one launch per step)"},
        }

    def e2e_value(self, ms, world):
        return round(job_value(self.work, ms, world, 1e12), 2), "TFLOPS"


BWD_SRC = ["exact_attention_81_gb300/csrc/fa_backward.cu", "exact_attention_81_gb300/csrc/ptx.cuh"]


class BwdCase(DenseCase):
    """One fa_bwd call (D preprocessing, bwd_kernel, dQ conversion) on the forward output of
    a dense workload; work = the five matmuls' FLOPs, 2.5 x the forward's."""

    def __init__(self, w, dev):
        super().__init__(w, dev)
        import torch
        import exact_attention_81_gb300 as fa
        g = torch.Generator(device=dev).manual_seed(w.seed + 9)
        self.do = torch.randn(self.q.shape, device=dev, generator=g).to(torch.bfloat16)
        fa.fa_fwd(self.q, self.k, self.v, causal=w.causal, out=self.out, lse=self.lse)
        self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
        self.ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Nq, w.Hq, w.d),
                              dtype=torch.uint8, device=dev)
        self.work = 2.5 * flops(w)
        self.launches = 3

    def step(self):
        import exact_attention_81_gb300 as fa
        fa.fa_bwd(self.q, self.k, self.v, self.out, self.lse, self.do, causal=self.w.causal,
                  dq=self.dq, dk=self.dk, dv=self.dv, workspace=self.ws)

    def e2e(self):
        """Pinned host Q/K/V/O/LSE/dO copied in, dQ/dK/dV copied out, every step."""
        import torch
        import exact_attention_81_gb300 as fa
        srcs = (self.q, self.k, self.v, self.out, self.lse, self.do)
        hosts = [t.cpu().pin_memory() for t in srcs]
        devs = [torch.empty_like(t) for t in srcs]
        outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for t in (self.dq, self.dk, self.dv)]

        def run():
            for dst, h in zip(devs, hosts):
                dst.copy_(h, non_blocking=True)
            fa.fa_bwd(*devs, causal=self.w.causal, dq=self.dq, dk=self.dk, dv=self.dv,
                      workspace=self.ws)
            for h, t in zip(outs, (self.dq, self.dk, self.dv)):
                h.copy_(t, non_blocking=True)
        h2d = sum(t.numel() * t.element_size() for t in srcs)
        d2h = sum(t.numel() * t.element_size() for t in (self.dq, self.dk, self.dv))
        return run, h2d, d2h

    def describe(self, pk, ms_step, world):
        d = super().describe(pk, ms_step, world)
        w = self.w
        tf = self.work / (ms_step * 1e-3) / 1e12
        kern = f"bwd_kernel<{w.d},{str(w.causal).lower()}>"
        d["metric"] = BWD_METRIC
        d["roofline"] = {
            "bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": round(tf / pk["bf16"], 4),
            "traffic": profiled_traffic(kern, BWD_SRC, w.name),
            "peak_basis": f"{pk['basis']} bf16 dense (burst)",
            "kernel": f"{kern} + preprocessing + dQ conversion (3 launches per step; achieved "
                      "uses the step time)"}
        return d


class DecodeCase:
    """One fa_fwd_kvcache call (split-KV decode + combine); work = bytes of the visible
    K/V prefix, Q, O and LSE (the split partials are overhead, not counted)."""

    def __init__(self, w, dev, e4m3=False):
        import torch
        import exact_attention_81_gb300 as fa
        from exact_attention_81_gb300.inputs import kvcache_workload_inputs
        self.w = w
        self.e4m3 = e4m3
        self.q, self.kc, self.vc, self.lens = kvcache_workload_inputs(w, device=dev)
        self.dk = self.dv = None
        if e4m3:  # the caches divided by a per-(batch, kv head) factor, rounded to E4M3
            g8 = torch.Generator(device="cpu").manual_seed(w.seed + 100)
            fk, fv = (0.25 * (1.0 + 0.5 * torch.rand((w.B, w.Hkv), generator=g8))
                      for _ in range(2))
            caches = []
            for c, f in ((self.kc, fk), (self.vc, fv)):
                c8 = torch.zeros(c.shape, dtype=torch.uint8, device=dev)
                for b in range(w.B):
                    n = int(self.lens[b].item())
                    c8[b, :n] = (c[b, :n].float() / f[b].to(dev)[None, :, None]).to(
                        torch.float8_e4m3fn).view(torch.uint8)
                caches.append(c8.view(torch.float8_e4m3fn))
            self.kc, self.vc = caches
            self.dk, self.dv = fk.float().to(dev), fv.float().to(dev)
        self.ws = torch.empty(fa.fa_fwd_kvcache_workspace_size(w.B, w.Hq, w.Nk, w.d, 0),
                              dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        kv = int(self.lens.long().sum().item()) * w.Hkv * w.d * (1 if e4m3 else 2) * 2
        self.work = kv + self.q.numel() * 2 * 2 + self.lse.numel() * 4
        self.launches = 2

    def _call(self, q):
        import exact_attention_81_gb300 as fa
        if self.e4m3:
            fa.fa_fwd_kvcache_fp8(q, self.kc, self.vc, self.lens, k_descale=self.dk,
                                  v_descale=self.dv, workspace=self.ws, out=self.out,
                                  lse=self.lse)
        else:
            fa.fa_fwd_kvcache(q, self.kc, self.vc, self.lens, workspace=self.ws, out=self.out,
                              lse=self.lse)

    def step(self):
        self._call(self.q)

    def e2e(self):
        """The cache is resident state; each step copies the new queries in and the
        output and LSE back."""
        import torch
        import exact_attention_81_gb300 as fa
        hq = self.q.cpu().pin_memory()
        ho = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        hl = torch.empty(self.lse.shape, dtype=self.lse.dtype, pin_memory=True)
        dq = torch.empty_like(self.q)

        def run():
            dq.copy_(hq, non_blocking=True)
            self._call(dq)
            ho.copy_(self.out, non_blocking=True)
            hl.copy_(self.lse, non_blocking=True)
        return run, self.q.numel() * 2, self.out.numel() * 2 + self.lse.numel() * 4

    def describe(self, pk, ms_step, world):
        w = self.w
        gbs = self.work / (ms_step * 1e-3) / 1e9
        return {
            "metric": DECODE_METRIC, "unit": "GB/s",
            "value": round(job_value(self.work, ms_step, world, 1e9), 1),
            "config": {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} cache={w.Nk} "
                                   f"d={w.d} lengths U[{w.Nk // 32},{w.Nk}] "
                                   + ("bf16 query, E4M3 cache" if self.e4m3 else "bf16"),
                       "batch": w.B, "heads": w.Hq, "kv_heads": w.Hkv, "cache_len": w.Nk,
                       "head_dim": w.d, "parallelism": f"replicas x{world}",
                       "l2": f"K/V read {self.work / 1e9:.2f} GB > L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                         "traffic": None if self.e4m3 else profiled_traffic(
                             f"decode_kernel<{w.d},{w.Hq // w.Hkv}>", DECODE_SRC, w.name),
                         "peak_basis": f"{pk['basis']} copy bandwidth",
                         "kernel": f"decode_kernel<{w.d},{w.Hq // w.Hkv}"
                                   + (",e4m3" if self.e4m3 else "") + "> + combine_kernel"},
        }

    def e2e_value(self, ms, world):
        return round(job_value(self.work, ms, world, 1e9), 1), "GB/s"


def run_ours(args, rank, world, dist):
    import torch
    import exact_attention_81_gb300 as fa
    from exact_attention_81_gb300.inputs import WORKLOADS

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()
    w_job = WORKLOADS[args.workload]
    w = shard_workload(w_job, world, rank) if args.shard else w_job
    if w.kind == "kvcache":
        case = DecodeCase(w, dev, e4m3=args.kv_e4m3)
    else:
        case = BwdCase(w, dev) if args.backward else DenseCase(w, dev, args.softcap, args.alibi)
    fa.set_cta_pairs(args.cta_pairs)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        case.step()
    st = fa.get_last_device_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device error during warm-up: {fa.status_string(st)}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        case.step()
    ev1.record(stream)
    barrier()
    t_wall1 = time.time()
    ms_total = ev0.elapsed_time(ev1)
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    st = fa.get_last_device_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device error in the timed region: {fa.status_string(st)}")
    ms_step = max_over_ranks(ms_total / args.steps, dist, dev)

    # e2e through the public call with pinned host buffers.
    e2e_run, h2d, d2h = case.e2e()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(3):
        e2e_run()
    barrier()
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_run()
    ev1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / e2e_steps, dist, dev)
    e2e_val, e2e_unit = case.e2e_value(e2e_ms, world)

    d = case.describe(pk, ms_step, world)
    if args.shard:  # every rank computed 1 / world of the one workload
        d["config"]["parallelism"] = (f"kv heads sharded x{world} (each GPU holds its own "
                                      "heads' K/V; no collective on the data path)")
        d["config"]["workload"] += f" (this rank: Hq={w.Hq} Hkv={w.Hkv})"
    result = {
        "metric": d["metric"], "value": d["value"], "unit": d["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded iid N(0,1) bf16)", "config": d["config"],
        "roofline": d["roofline"],
        "e2e": {"value": e2e_val, "unit": e2e_unit, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * case.launches,
        "clocks": clocks,
    }
    if not args.no_extra:
        result["extra"] = extra_workloads(args, dev, pk, world, dist)
    if rank == 0 and not args.no_cpu_baseline and not args.kv_e4m3:
        if w.kind == "kvcache":
            result["cpu_baseline"] = cpu_baseline_decode(case, args.cpu_seconds)
        elif args.backward:
            result["cpu_baseline"] = cpu_baseline_bwd(case, args.cpu_seconds)
        else:
            result["cpu_baseline"] = cpu_baseline(w, case.q, case.k, case.v, args.cpu_seconds)
    return result


def cpu_baseline_bwd(case, seconds):
    """The fp64 oracle's backward on a bounded sample: whole heads of batch 0, one after
    the other, until `seconds` of CPU time have been spent."""
    import oracle.oracle as ORACLE
    w = case.w
    threads = os.cpu_count() or 1
    fl, dt, heads = 0.0, 0.0, 0
    while dt < seconds and heads < w.Hkv:
        g = heads
        G = w.Hq // w.Hkv
        q, do = (t[0:1, :, g * G:(g + 1) * G].contiguous().cpu() for t in (case.q, case.do))
        k, v = (t[0:1, :, g:g + 1].contiguous().cpu() for t in (case.k, case.v))
        t0 = time.time()
        ORACLE.attention_bwd(q, k, v, do, w.scale, w.causal, nthreads=threads)
        dt += time.time() - t0
        fl += 2.5 * 4.0 * w.Nq * w.Nk * w.d * G / (2 if w.causal else 1)
        heads += 1
    return {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"backward of {heads} kv head(s) of batch 0 of {w.name} "
                      f"(fp64, {dt:.1f} s)"}


def cpu_baseline_decode(case, seconds):
    """The fp64 oracle on a bounded sample of the decode workload's batch entries."""
    import math
    import numpy as np
    import oracle.oracle as ORACLE
    w = case.w
    threads = os.cpu_count() or 1
    lens = case.lens.cpu()
    scale = float(np.float32(1 / math.sqrt(w.d)))
    nb = 1
    while True:
        sel = list(range(nb))
        top = int(lens[:nb].max())
        q = case.q[:nb].cpu()
        kc = case.kc[:nb, :top].cpu()
        vc = case.vc[:nb, :top].cpu()
        t0 = time.time()
        ORACLE.attention_kvcache(q, kc, vc, lens[:nb], scale, nthreads=threads)
        dt = time.time() - t0
        if dt >= seconds / 4 or nb >= w.B:
            break
        nb = min(w.B, nb * 2)
    byts = int(lens[:nb].long().sum()) * w.Hkv * w.d * 4
    return {"value": byts / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{nb} of {w.B} batch entries of {w.name} (fp64, {dt:.1f} s)"}


def time_calls(fn, steps, stream, warm=3):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def extra_workloads(args, dev, pk, world, dist):
    import torch
    import exact_attention_81_gb300 as fa
    from exact_attention_81_gb300.inputs import WORKLOADS, kvcache_workload_inputs, workload_inputs
    stream = torch.cuda.current_stream()
    res = {}
    # the width-128 forward on CTA pairs (cta_group::2), next to the default single-CTA kernel
    for name in ("causal8k", "dense2k", "gqa16k"):
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        o = torch.empty_like(q)
        l = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        fa.set_cta_pairs(True)
        try:
            ms = time_calls(lambda: fa.fa_fwd(q, k, v, causal=w.causal, out=o, lse=l),
                            max(10, args.steps // 4), stream)
        finally:
            fa.set_cta_pairs(False)
        tf = flops(w) / (ms * 1e-3) / 1e12
        res[name + "_cta_pairs"] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                                    "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
        del q, k, v, o, l
    for name in ("dense2k", "gqa16k", "causal8k_d256"):
        w = WORKLOADS[name]
        q, k, v = workload_inputs(w, device=dev)
        o = torch.empty_like(q)
        l = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        ms = time_calls(lambda: fa.fa_fwd(q, k, v, causal=w.causal, out=o, lse=l),
                        max(10, args.steps // 4), stream)
        tf = flops(w) / (ms * 1e-3) / 1e12
        res[name] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                     "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
        del q, k, v, o, l
    # variants of the headline workload: fp16 inputs, a 4096-key sliding window, softcap +
    # ALiBi (FLOPs: 4 d per visible (query, key) pair; the causal convention N^2/2 otherwise)
    w = WORKLOADS["causal8k"]
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / w.Hq) for h in range(w.Hq)],
                          dtype=torch.float32, device=dev)
    for name, dtype, kw, work in [
            ("causal8k_fp16", torch.float16, {}, flops(w)),
            ("causal8k_window4096", torch.bfloat16, {"window_size": (4096, 0)},
             4.0 * w.d * w.B * w.Hq * window_pairs(w.Nq, w.Nk, 4096, 0)),
            ("causal8k_alibi", torch.bfloat16, {"alibi_slopes": slopes}, flops(w)),
            ("causal8k_softcap", torch.bfloat16, {"softcap": 30.0}, flops(w)),
            ("causal8k_softcap_alibi", torch.bfloat16,
             {"softcap": 30.0, "alibi_slopes": slopes}, flops(w))]:
        q, k, v = workload_inputs(w, device=dev, dtype=dtype)
        o = torch.empty_like(q)
        l = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        ms = time_calls(lambda: fa.fa_fwd(q, k, v, causal=True, out=o, lse=l, **kw),
                        max(10, args.steps // 4), stream)
        tf = work / (ms * 1e-3) / 1e12
        res[name] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                     "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
        del q, k, v, o, l
    # FP8 (E4M3) inputs on the headline shape; peak: the measured bf16 peak times the
    # nominal fp8 / bf16 ratio of the part (4.5 / 2.25 PFLOP/s dense)
    from exact_attention_81_gb300.inputs import fp8_inputs
    q8, k8, v8, dq8, dk8, dv8 = fp8_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, w.seed, device=dev)
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device=dev)
    l = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    ws8 = torch.empty(fa.fa_fwd_fp8_workspace_size(w.B, w.Nk, w.Hkv, w.d), dtype=torch.uint8,
                      device=dev)
    ms = time_calls(lambda: fa.fa_fwd_fp8(q8, k8, v8, causal=True, q_descale=dq8, k_descale=dk8,
                                          v_descale=dv8, out=o, lse=l, workspace=ws8),
                    max(10, args.steps // 4), stream)
    tf = flops(w) / (ms * 1e-3) / 1e12
    res["causal8k_fp8"] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                           "frac_of_fp8_peak": round(tf / (2.0 * pk["bf16"]), 4),
                           "peak_basis": "2 x measured bf16 (nominal fp8 / bf16 ratio)",
                           "gpu_launches_per_call": 2}
    del q8, k8, v8, o, l, ws8
    # backward pass of the headline workload (FLOPs: five matmuls, 2.5 x the forward)
    w = WORKLOADS["causal8k"]
    q, k, v = workload_inputs(w, device=dev)
    do = torch.randn(q.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(9))
    do = do.to(torch.bfloat16)
    o, l = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Nq, w.Hq, w.d), dtype=torch.uint8,
                      device=dev)
    ms = time_calls(lambda: fa.fa_bwd(q, k, v, o, l, do, causal=True, dq=dq, dk=dk, dv=dv,
                                      workspace=bws), max(10, args.steps // 4), stream)
    tf = 2.5 * flops(w) / (ms * 1e-3) / 1e12
    res["causal8k_backward"] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                                "frac_of_bf16_peak": round(tf / pk["bf16"], 4),
                                "gpu_launches_per_call": 3}
    ms = time_calls(lambda: fa.fa_bwd(q, k, v, o, l, do, causal=True, dq=dq, dk=dk, dv=dv,
                                      workspace=bws, deterministic=True),
                    max(10, args.steps // 4), stream)
    tf = 2.5 * flops(w) / (ms * 1e-3) / 1e12
    res["causal8k_backward_deterministic"] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                                              "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
    # backward with the modifiers (FLOPs: 10 d per visible pair; the causal convention else)
    for name, kw, work in [
            ("causal8k_backward_window4096", {"window_size": (4096, 0)},
             10.0 * w.d * w.B * w.Hq * window_pairs(w.Nq, w.Nk, 4096, 0)),
            ("causal8k_backward_alibi", {"alibi_slopes": slopes}, 2.5 * flops(w)),
            ("causal8k_backward_softcap_alibi", {"softcap": 30.0, "alibi_slopes": slopes},
             2.5 * flops(w))]:
        o, l = fa.fa_fwd(q, k, v, causal=True, **kw)
        ms = time_calls(lambda: fa.fa_bwd(q, k, v, o, l, do, causal=True, dq=dq, dk=dk, dv=dv,
                                          workspace=bws, **kw), max(10, args.steps // 4), stream)
        tf = work / (ms * 1e-3) / 1e12
        res[name] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                     "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
    del q, k, v, do, o, l, dq, dk, dv, bws
    # backward at head dimension 256 (the wide kernel: units per d half, 64-query steps;
    # FLOPs as above: the algorithmic five matmuls, not the recomputed S and dP of the
    # second d half)
    w = WORKLOADS["causal8k_d256"]
    q, k, v = workload_inputs(w, device=dev)
    do = torch.randn(q.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(9))
    do = do.to(torch.bfloat16)
    o, l = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Nq, w.Hq, w.d), dtype=torch.uint8,
                      device=dev)
    ms = time_calls(lambda: fa.fa_bwd(q, k, v, o, l, do, causal=True, dq=dq, dk=dk, dv=dv,
                                      workspace=bws), max(10, args.steps // 4), stream)
    tf = 2.5 * flops(w) / (ms * 1e-3) / 1e12
    res["causal8k_d256_backward"] = {"ms": round(ms, 4), "TFLOPS": round(tf, 2),
                                     "frac_of_bf16_peak": round(tf / pk["bf16"], 4),
                                     "gpu_launches_per_call": 3}
    del q, k, v, do, o, l, dq, dk, dv, bws
    w = WORKLOADS["decode"]
    q, kc, vc, lens = kvcache_workload_inputs(w, device=dev)
    ws = torch.empty(fa.fa_fwd_kvcache_workspace_size(w.B, w.Hq, w.Nk, w.d, 0), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(q)
    l = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ms = time_calls(lambda: fa.fa_fwd_kvcache(q, kc, vc, lens, workspace=ws, out=o, lse=l),
                    max(20, args.steps // 2), stream)
    kv_bytes = int(lens.long().sum().item()) * w.Hkv * w.d * 2 * 2
    io_bytes = q.numel() * 2 * 2 + l.numel() * 4
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    res["decode"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "algorithmic_bytes": kv_bytes + io_bytes,
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                                  "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                                  "traffic": profiled_traffic("decode_kernel<128,4>", DECODE_SRC,
                                                              "decode"),
                                  "peak_basis": f"{pk['basis']} copy bandwidth"},
                     "gpu_launches_per_call": 2}
    ms = time_calls(lambda: fa.fa_fwd_kvcache(q, kc, vc, lens, workspace=ws, out=o, lse=l,
                                              window_size=(4095, -1)),
                    max(20, args.steps // 2), stream)
    kv_bytes = int(lens.clamp(max=4096).long().sum().item()) * w.Hkv * w.d * 2 * 2
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    res["decode_window4096"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                "algorithmic_bytes": kv_bytes + io_bytes,
                                "frac_of_hbm": round(gbs / pk["hbm"], 4)}
    # the decode workload as a paged cache (pages of 256 rows in shuffled order over the same
    # memory), one appended token per sequence with rotary on the query and the new key
    page = 256
    nblk = w.Nk // page
    perm = torch.randperm(w.B * nblk, generator=torch.Generator().manual_seed(7))
    table = perm.reshape(w.B, nblk).to(torch.int32).to(dev)
    kp = kc.view(w.B * nblk, page, w.Hkv, w.d)
    vp = vc.view(w.B * nblk, page, w.Hkv, w.d)
    lens_a = lens.clamp(max=w.Nk - 1)
    kn = torch.randn((w.B, 1, w.Hkv, w.d), device=dev).to(torch.bfloat16)
    vn = torch.randn((w.B, 1, w.Hkv, w.d), device=dev).to(torch.bfloat16)
    ang = torch.arange(w.Nk, device=dev, dtype=torch.float64)[:, None] * \
        10000.0 ** (-torch.arange(w.d // 2, device=dev, dtype=torch.float64) / (w.d // 2))
    cos, sin = ang.cos().float().contiguous(), ang.sin().float().contiguous()
    ms = time_calls(lambda: fa.fa_fwd_kvcache(q, kp, vp, lens_a, workspace=ws, out=o, lse=l,
                                              k_new=kn, v_new=vn, rotary_cos=cos,
                                              rotary_sin=sin, block_table=table),
                    max(20, args.steps // 2), stream)
    kv_bytes = int((lens_a.long() + 1).sum().item()) * w.Hkv * w.d * 2 * 2
    new_bytes = 2 * kn.numel() * 2 * 2  # new rows read and written
    gbs = (kv_bytes + io_bytes + new_bytes) / (ms * 1e-3) / 1e9
    res["decode_paged_append_rotary"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                         "algorithmic_bytes": kv_bytes + io_bytes + new_bytes,
                                         "frac_of_hbm": round(gbs / pk["hbm"], 4),
                                         "gpu_launches_per_call": 3}
    # the decode workload over E4M3 caches: the bf16 caches divided by a per-(batch, kv head)
    # factor and rounded to float8_e4m3fn on the device (input preparation, untimed)
    g8 = torch.Generator(device="cpu").manual_seed(w.seed + 100)
    fk, fv = (0.25 * (1.0 + 0.5 * torch.rand((w.B, w.Hkv), generator=g8)) for _ in range(2))
    kc8 = torch.empty(kc.shape, dtype=torch.float8_e4m3fn, device=dev)
    vc8 = torch.empty(vc.shape, dtype=torch.float8_e4m3fn, device=dev)
    for b in range(w.B):
        n = int(lens[b].item())
        kc8[b].view(torch.uint8).fill_(0)
        vc8[b].view(torch.uint8).fill_(0)
        kc8[b, :n] = (kc[b, :n].float() / fk[b].to(dev)[None, :, None]).to(torch.float8_e4m3fn)
        vc8[b, :n] = (vc[b, :n].float() / fv[b].to(dev)[None, :, None]).to(torch.float8_e4m3fn)
    dk8, dv8 = fk.float().to(dev), fv.float().to(dev)
    del kp, vp
    ms_bf16 = res["decode"]["ms"]
    ms = time_calls(lambda: fa.fa_fwd_kvcache_fp8(q, kc8, vc8, lens, k_descale=dk8, v_descale=dv8,
                                                  workspace=ws, out=o, lse=l),
                    max(20, args.steps // 2), stream)
    kv_bytes = int(lens.long().sum().item()) * w.Hkv * w.d * 1 * 2
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    res["decode_fp8"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                         "algorithmic_bytes": kv_bytes + io_bytes,
                         "frac_of_hbm": round(gbs / pk["hbm"], 4),
                         "speedup_vs_bf16_cache": round(ms_bf16 / ms, 3),
                         "gpu_launches_per_call": 2}
    del q, kc, vc, kc8, vc8, lens, ws, o, l, kn, vn
    # decode at head dimension 256 (width-256 instance, 3 ring slots)
    w = WORKLOADS["decode_d256"]
    q, kc, vc, lens = kvcache_workload_inputs(w, device=dev)
    ws = torch.empty(fa.fa_fwd_kvcache_workspace_size(w.B, w.Hq, w.Nk, w.d, 0), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(q)
    l = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ms = time_calls(lambda: fa.fa_fwd_kvcache(q, kc, vc, lens, workspace=ws, out=o, lse=l),
                    max(20, args.steps // 2), stream)
    kv_bytes = int(lens.long().sum().item()) * w.Hkv * w.d * 2 * 2
    io_bytes = q.numel() * 2 * 2 + l.numel() * 4
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    res["decode_d256"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                          "algorithmic_bytes": kv_bytes + io_bytes,
                          "frac_of_hbm": round(gbs / pk["hbm"], 4)}
    del q, kc, vc, lens, ws, o, l
    st = fa.get_last_device_error()
    if st != fa.FA_OK:
        raise RuntimeError(f"device error in extra workloads: {fa.status_string(st)}")
    return res


# ----------------------------------------------------------------------------- oracle arm

def cpu_sample_rows(w, n, seed=123):
    import numpy as np
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, w.B, n), rng.integers(0, w.Hq, n),
                     rng.integers(0, w.Nq, n)], axis=1).astype(np.int32)
    return rows


def rows_flops(w, rows) -> float:
    import numpy as np
    i = rows[:, 2].astype(np.float64)
    keys = np.minimum(i + 1 + (w.Nk - w.Nq), w.Nk) if w.causal else np.full_like(i, w.Nk)
    # 4 * d per visible key: the causal-halved convention of the headline metric
    return float(np.sum(4.0 * w.d * keys))


def cpu_baseline(w, q, k, v, seconds):
    """The fp64 oracle, as it stands, on a bounded sample of query rows of the workload."""
    import oracle.oracle as ORACLE
    hq, hk, hv = q.cpu(), k.cpu(), v.cpu()
    threads = os.cpu_count() or 1
    n = 32
    while True:  # calibrate on a small sample, then time one sample of ~`seconds`
        rows = cpu_sample_rows(w, n)
        t0 = time.time()
        ORACLE.attention_rows(hq, hk, hv, rows, w.scale, w.causal, nthreads=threads)
        dt = time.time() - t0
        if dt >= 0.5 or n >= 1 << 20:
            break
        n *= 4
    n = max(n, int(n * seconds / max(dt, 1e-3)))
    rows = cpu_sample_rows(w, n, seed=7)
    t0 = time.time()
    ORACLE.attention_rows(hq, hk, hv, rows, w.scale, w.causal, nthreads=threads)
    dt = time.time() - t0
    tflops = rows_flops(w, rows) / dt / 1e12
    return {"value": tflops, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"{n} random query rows of {w.name} (fp64, {dt:.1f} s)"}


def run_reference_decode(args, w):
    """The fp64 oracle on a few batch entries of the decode workload per step."""
    import math
    import numpy as np
    import oracle.oracle as ORACLE
    from exact_attention_81_gb300.inputs import kvcache_workload_entry
    threads = os.cpu_count() or 1
    scale = float(np.float32(1 / math.sqrt(w.d)))
    steps = []
    for s in range(args.warmup + args.steps):
        b = s % w.B
        q, kc, vc, n = kvcache_workload_entry(w, b)
        t0 = time.time()
        ORACLE.attention_kvcache(q, kc, vc, [n], scale, nthreads=threads)
        dt = time.time() - t0
        if s >= args.warmup:
            steps.append((n * w.Hkv * w.d * 4, dt))
    value = sum(x for x, _ in steps) / sum(t for _, t in steps) / 1e9
    return {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(t for _, t in steps) / len(steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1) bf16)",
        "config": {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} cache={w.Nk} "
                               f"d={w.d} lengths U[{w.Nk // 32},{w.Nk}] bf16"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"one batch entry of {w.name} per step (fp64)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_reference(args, w):
    import numpy as np
    import oracle.oracle as ORACLE
    from exact_attention_81_gb300.inputs import workload_inputs
    if w.kind == "kvcache":
        return run_reference_decode(args, w)
    q, k, v = workload_inputs(w, device="cpu")
    threads = os.cpu_count() or 1
    # size one step so that warm-up + timed steps stay within a few minutes
    n = 64
    while True:
        rows = cpu_sample_rows(w, n)
        t0 = time.time()
        ORACLE.attention_rows(q, k, v, rows, w.scale, w.causal, nthreads=threads)
        dt = time.time() - t0
        if dt >= 0.5 or n >= 1 << 20:
            break
        n *= 2
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = max(16, int(n * min(4.0, per_step_budget / max(dt, 1e-3))))
    steps = []
    for s in range(args.warmup + args.steps):
        rows = cpu_sample_rows(w, n, seed=1000 + s)
        t0 = time.time()
        ORACLE.attention_rows(q, k, v, rows, w.scale, w.causal, nthreads=threads)
        dt = time.time() - t0
        if s >= args.warmup:
            steps.append((rows_flops(w, rows), dt))
    total_f = sum(f for f, _ in steps)
    total_t = sum(t for _, t in steps)
    value = total_f / total_t / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_t / len(steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1) bf16)",
        "config": {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} Nq=Nk={w.Nq} "
                               f"d={w.d} causal={w.causal} bf16"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{n} random query rows of {w.name} per step (fp64)"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (fa_bwd) of the dense workload instead")
    ap.add_argument("--kv-e4m3", action="store_true",
                    help="decode workloads: E4M3 caches (fa_fwd_kvcache_fp8) instead of bf16")
    ap.add_argument("--shard", action="store_true",
                    help="N > 1: split the one workload's kv heads over the ranks (strong "
                         "scaling) instead of running it whole on every rank (weak scaling)")
    ap.add_argument("--softcap", type=float, default=0.0,
                    help="dense forward workloads: softcap the scores (tanh, this cap)")
    ap.add_argument("--alibi", action="store_true",
                    help="dense forward workloads: ALiBi bias, slopes 2^(-8 (h + 1) / H)")
    ap.add_argument("--cta-pairs", action="store_true",
                    help="dense forward workloads: run the forward on CTA pairs (cta_group::2)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    from exact_attention_81_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w)), flush=True)
        return

    import __graft_entry__
    __graft_entry__.build()
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    result = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
