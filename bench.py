#!/usr/bin/env python
"""Throughput of the multi-head attention forward on GB300, one JSON line.

Metric: MHA forward TFLOP/s (bf16 causal, 1 x GB300) and % of the dense-BF16
peak.  FLOPs per step follow itwiki.kr "멀티 헤드 어텐션", 매개변수와 계산량:
8 T D^2 for the projections plus 4 T^2 D for scores and weighted sum, the
latter halved under the causal mask, per batch element.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     # the fp64 CPU oracle as the reference arm
  python bench.py --variant NAME           # a variant (gqa4, mqa, gated, residual, decode-*)

One step = one mha_forward of the whole workload (three kernels: QKV GEMM,
fused attention, output GEMM) on inputs already resident in HBM; L2 is flushed
(a 256 MiB write) before every timed step, outside the events that time it.
Before each timed loop the stream spins on the GPU long enough for the host to
queue all K steps, so the events time the GPU's work rather than the host's
launch latency.
Under torchrun each rank runs an independent replica (the layer does not
shard: there is no exchange step), the timed region is bracketed by a barrier
and a device synchronise, and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from transformer_head_scaled_02_gb300 import workloads as wl  # noqa: E402

METRIC = "MHA forward TFLOP/s (bf16 causal, 1×GB300) and % of dense-BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "c3_bf16_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# GPU clock cycles the stream spins (torch.cuda._sleep) per queued step before a timed loop, so
# that the host has queued every step's launches before the GPU reaches the first event: the
# events then time the GPU work, not the gaps left while Python prepares the next launch
PREQUEUE_CYCLES_PER_STEP = 200_000
# batch chunks of the end-to-end (host buffers) measurement; each chunk's copies overlap the
# other chunks' kernels (three: the library cuts 1 + 2 + 1 for c3, 4 + 8 + 4 for c5)
E2E_CHUNKS = 3


# ---------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
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


def kernel_source_hash(fname: str) -> str:
    with open(os.path.join(ROOT, "transformer_head_scaled_02_gb300", "csrc", fname), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_file: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_sha256_16") != kernel_source_hash(src_file):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """Polls SM clock, max clock, power and clock-event reasons through NVML
    (read-only queries) every few ms on a background thread."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting"}

    def __init__(self, device_index: int = 0, period_s: float = 0.005):
        self.period = period_s
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.dev = ctypes.c_void_p()
            handle_found = False
            try:
                import torch
                pr = torch.cuda.get_device_properties(device_index)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
                handle_found = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.dev)) == 0
            except Exception:
                handle_found = False
            if not handle_found and self.nvml.nvmlDeviceGetHandleByIndex_v2(
                    device_index, ctypes.byref(self.dev)) != 0:
                return
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            self.ok = False

    def _poll(self):
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk))
            self.nvml.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(pw))
            self._reasons_fn(self.dev, ctypes.byref(rs))
            self.samples.append((time.time(), int(clk.value), pw.value / 1000.0, int(rs.value)))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "NVML not available"}
        s = [x for x in self.samples if self.t0 <= x[0] <= self.t1] or self.samples
        reasons = set()
        for _, _, _, r in s:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[1] for x in s) if s else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(s),
                "power_w_max": max(x[2] for x in s) if s else None}


# ---------------------------------------------------------------------------- our arm

def to_device(a, dtype_name, torch):
    import numpy as np
    if a is None:
        return None
    if dtype_name == "bf16":
        return torch.from_numpy(wl.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def cpu_baseline(w, budget_s: float = 15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: the first nb
    batches and, of each, the first T' query rows (for causal self-attention the outputs of
    those rows depend on nothing else).  The sample grows (rows first, then batches, up to
    the whole workload) until one run takes about a quarter of budget_s or more."""
    import oracle
    oracle.build()
    x = wl.make_inputs(w)

    def run(nb, tp):
        t0 = time.perf_counter()
        if w.cross:
            L = None if x["kv_lengths"] is None else x["kv_lengths"][:nb]
            oracle.mha_forward(x["X_q"][:nb, :tp], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h,
                               w.d_k, w.d_v, Xkv=x["X_kv"][:nb], causal=w.causal, kv_lengths=L)
        else:
            oracle.mha_forward(x["X_q"][:nb, :tp], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h,
                               w.d_k, w.d_v, causal=w.causal)
        return time.perf_counter() - t0

    nb, tp = 1, min(w.T_q, 64)
    dt = run(nb, tp)
    while dt < budget_s / 4 and (tp < w.T_q or nb < w.B):
        if tp < w.T_q:
            tp = min(w.T_q, tp * 2)
        else:
            nb = min(w.B, nb * 2)
        dt = run(nb, tp)
    sw = wl.custom("sample", B=nb, T_q=tp, T_kv=w.T_kv if w.cross else tp, D=w.D, h=w.h,
                   d_k=w.d_k, d_v=w.d_v, dtype=w.dtype, causal=w.causal, cross=w.cross)
    f = wl.flops(sw)["total"]
    whole = nb == w.B and tp == w.T_q
    what = ("the whole workload" if whole else
            f"batches 0..{nb - 1}, first {tp} of {w.T_q} query rows of {w.name}")
    return {"value": f / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{what} ({'all ' + str(w.T_kv) + ' keys' if w.cross else 'causal prefix'}), "
                      f"fp64, {dt:.2f} s"}


def measure_workload(w, K, warmup, torch, dev, world, flush, sampler=None):
    """Time workload w: K steps of mha_forward (each bracketed by events, L2 flushed before
    it), then the same launches with events between them (per-kernel durations), then the
    host-buffer forward through the C ABI.  Returns the figures of one JSON line."""
    from transformer_head_scaled_02_gb300 import Mha
    x = wl.make_inputs(w)
    d = {k: to_device(v, w.dtype, torch) for k, v in x.items() if k != "kv_lengths"}
    kvl = None if x["kv_lengths"] is None else torch.from_numpy(x["kv_lengths"]).cuda()
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    layer = Mha(w.D, w.h, w.d_k, w.d_v, dtype=tdt)
    out = torch.empty((w.B, w.T_q, w.D), dtype=tdt, device=dev)

    def forward():
        layer.forward(d["X_q"], d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"], X_kv=d["X_kv"],
                      causal=w.causal, kv_lengths=kvl, out=out)

    for _ in range(warmup):
        forward()
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError(f"{w.name}: device status not clean after warm-up")

    # ---------------- timed region: K steps, each timed by events, L2 flushed between
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.05)
    wall0 = time.perf_counter()
    torch.cuda._sleep(PREQUEUE_CYCLES_PER_STEP * K)
    for k in range(K):
        flush.zero_()
        ev[k][0].record()
        forward()
        ev[k][1].record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    if sampler is not None:
        sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / K
    if layer.status() != 0:
        raise RuntimeError(f"{w.name}: device status reports an error after the timed region")

    fl = wl.flops(w, x["kv_lengths"])
    # with key padding, only the valid keys count: the padded ones need neither projection nor
    # attention, and the kernels skip them (the nominal count is reported beside it)
    step_flops = fl.get("alg_total", fl["total"])
    flops_counted = "algorithmic (valid keys only)" if "alg_total" in fl else "nominal"
    value = world * step_flops / (ms_per_step / 1e3) / 1e12

    # ---------------- per-kernel durations: the same launches, events between them
    sf = wl.step_flops(w)
    names = ["qkv_proj", "attention", "out_proj"]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    Wqkv, bqkv = d["W_qkv"], d["b_qkv"]
    hq, hv = w.h * w.d_k, w.h * w.d_v
    ncols = 2 * hq + hv
    ocat = torch.empty((w.B, w.T_q, hv), dtype=tdt, device=dev)
    torch.cuda.synchronize()
    torch.cuda._sleep(PREQUEUE_CYCLES_PER_STEP * K)
    if not w.cross:
        qkv = torch.empty((w.B, w.T_q, ncols), dtype=tdt, device=dev)
        X2 = d["X_q"].view(-1, w.D)
        for k in range(K):
            flush.zero_()
            e = kev[k]
            e[0].record()
            layer.linear(X2, Wqkv, bqkv, out=qkv.view(-1, ncols))
            e[1].record()
            layer.attention(qkv[..., :hq], qkv[..., hq:2 * hq], qkv[..., 2 * hq:], causal=w.causal,
                            out=ocat)
            e[2].record()
            layer.linear(ocat.view(-1, hv), d["W_o"], d["b_o"], out=out.view(-1, w.D))
            e[3].record()
        torch.cuda.synchronize()
        per_kernel = {n: statistics.mean(kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(K))
                      for i, n in enumerate(names)}
    else:
        # cross-attention: the key/value and query projections in one launch (as the forward
        # runs them, rows past the key lengths not projected), attention, output projection,
        # each timed alone
        hk = w.h * w.d_k
        qb = torch.empty((w.B, w.T_q, hq), dtype=tdt, device=dev)
        kvb = torch.empty((w.B, w.T_kv, hk + hv), dtype=tdt, device=dev)
        Xq2, Xkv2 = d["X_q"].view(-1, w.D), d["X_kv"].view(-1, w.D)
        bq = None if bqkv is None else bqkv[:hq]
        bkv = None if bqkv is None else bqkv[hq:]
        for k in range(K):
            flush.zero_()
            e = kev[k]
            e[0].record()
            layer.linear_pair(Xkv2, Wqkv[:, hq:], bkv, Xq2, Wqkv[:, :hq], bq, seg_len=kvl,
                              seg_rows=w.T_kv if kvl is not None else 0,
                              out=kvb.view(-1, hk + hv), out2=qb.view(-1, hq))
            e[1].record()
            layer.attention(qb, kvb[..., :hk], kvb[..., hk:], causal=w.causal, kv_lengths=kvl,
                            out=ocat)
            e[2].record()
            layer.linear(ocat.view(-1, hv), d["W_o"], d["b_o"], out=out.view(-1, w.D))
            e[3].record()
        torch.cuda.synchronize()
        per_kernel = {n: statistics.mean(kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(K))
                      for i, n in enumerate(["kv_q_proj", "attention", "out_proj"])}
        # FLOPs per launch; with key lengths the kernels visit only the L_b valid keys of each
        # batch (the key/value projection skips whole 256-row blocks past them)
        L = float(w.B * w.T_kv)
        if x["kv_lengths"] is not None:
            import numpy as np
            L = float(np.sum(np.asarray(x["kv_lengths"], dtype=np.float64)))
        sf = dict(sf, kv_q_proj=2.0 * w.D * w.B * w.T_q * hq + 2.0 * w.D * L * (hk + hv),
                  attention=2.0 * w.h * w.T_q * L * (w.d_k + w.d_v) * (0.5 if w.causal else 1.0))

    # ---------------- end to end through the public API, host buffers in and out
    xh = d["X_q"].cpu().pin_memory()
    xkvh = None if d["X_kv"] is None else d["X_kv"].cpu().pin_memory()
    yh = torch.empty(out.shape, dtype=tdt).pin_memory()
    Ke = min(K, 50)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Ke)]
    barrier(world)
    torch.cuda.synchronize()
    e2e_chunks = min(E2E_CHUNKS, w.B)

    def forward_host():
        layer.forward_host(xh, d["W_qkv"], d["b_qkv"], d["W_o"], d["b_o"], out=yh, X_kv=xkvh,
                           causal=w.causal, kv_lengths=kvl, chunks=e2e_chunks)

    for _ in range(2):
        forward_host()
    torch.cuda.synchronize()
    torch.cuda._sleep(PREQUEUE_CYCLES_PER_STEP * Ke)
    for k in range(Ke):
        flush.zero_()
        eev[k][0].record()
        forward_host()
        eev[k][1].record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in eev), world, dev) / Ke
    h2d = xh.numel() * xh.element_size() + (0 if xkvh is None else xkvh.numel() * xkvh.element_size())
    d2h = yh.numel() * yh.element_size()

    pk, pk_src = peaks()
    top = max(per_kernel, key=per_kernel.get)
    src = "attn_bf16.cu" if top == "attention" else "gemm_bf16.cu"
    if w.dtype == "f32":
        src = "simt_f32.cu"
    ach = sf[top] / (per_kernel[top] / 1e3) / 1e12
    if w.dtype == "f32":
        # fp32 runs as FFMA on the CUDA cores: SMs x 128 fp32 lanes x 2 FLOP x max SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = float(pk.get("sm_max_mhz", 2070.0))
        peak = round(sms * 128 * 2 * mhz * 1e6 / 1e12, 1)
        bound, peak_source = "alu", f"derived fp32 FFMA: {sms} SMs x 128 lanes x 2 x {mhz:.0f} MHz"
    else:
        peak = pk["bf16_tflops"]
        bound, peak_source = "tensor", f"{pk_src} bf16 dense (burst)"
    roofline = {"kernel": top, "bound": bound, "achieved": round(ach, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "traffic": recorded_traffic(top, w.name, src),
                "peak_source": peak_source,
                "per_kernel_ms": {k: round(v, 4) for k, v in per_kernel.items()},
                "per_kernel_frac_of_peak": {k: round(sf[k] / (v / 1e3) / 1e12 / peak, 4)
                                            for k, v in per_kernel.items()}}
    return {
        "workload": w, "value": value, "ms_per_step": ms_per_step, "step_flops": step_flops,
        "flops_counted": flops_counted, "nominal_flops": fl["total"], "roofline": roofline,
        "e2e": {"value": round(world * step_flops / (e2e_ms / 1e3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "chunks": e2e_chunks,
                "note": "mha_forward_host through the C ABI: pinned host X in and Y out, the batch "
                        "in chunks whose host-device copies overlap the kernels; weights resident"},
        "launches_per_step": launches_per_step(w), "wall": wall, "peak": pk["bf16_tflops"],
        "step_ms": step_stats(step_ms),
        # the step's algorithmic HBM bytes (X in, Q/K/V and Ocat written and read back, Y out,
        # the weights once; nominal key counts) over its time, against the measured copy rate
        "hbm": {"algorithmic_bytes_per_step": wl.hbm_bytes(w),
                "achieved_gbs": round(world * wl.hbm_bytes(w) / (ms_per_step / 1e3) / 1e9, 1),
                "peak_gbs": pk["hbm_gbs"],
                "frac": round(wl.hbm_bytes(w) / (ms_per_step / 1e3) / 1e9 / pk["hbm_gbs"], 4)},
        "peak_source": pk_src,
    }


def launches_per_step(w) -> int:
    """Kernels one forward launches: projections (self-attention: one; cross-attention: the
    key/value and query projections in one launch for bf16 when both have more than 128 rows,
    else two; a gate block one more), attention, output projection."""
    if not w.cross:
        return 3
    paired = w.dtype == "bf16" and w.B * w.T_q > 128 and w.B * w.T_kv > 128
    return (1 if paired else 2) + (1 if getattr(w, "gated", False) else 0) + 2


def step_stats(step_ms) -> dict:
    """Median and p10 / p90 of the timed steps (this rank's), in ms."""
    import numpy as np
    a = np.asarray(step_ms, dtype=np.float64)
    return {"p10": round(float(np.percentile(a, 10)), 4), "median": round(float(np.median(a)), 4),
            "p90": round(float(np.percentile(a, 90)), 4)}


# the other bf16 workloads, timed in the same process after the headline one and reported
# under "other_workloads" of the same line
EXTRA_WORKLOADS = ["c4_bf16_causal_long", "c5_bf16_cross"]


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__ as g
    g.build_library()

    w = wl.WORKLOADS[args.workload]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(torch.cuda.current_device())
    r = measure_workload(w, args.steps, args.warmup, torch, dev, world, flush, sampler)
    K = args.steps
    pk = r["peak"]
    line = {
        "metric": METRIC, "value": round(r["value"], 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) weights; no dataset)",
        "config": {"workload": w.name, "B": w.B, "T_q": w.T_q, "T_kv": w.T_kv, "D": w.D,
                   "h": w.h, "d_k": w.d_k, "d_v": w.d_v, "causal": w.causal, "cross": w.cross,
                   "flops_per_step": r["step_flops"], "flops_counted": r["flops_counted"],
                   "nominal_flops_per_step": r["nominal_flops"],
                   "frac_of_peak": round(r["value"] / world / pk, 4),
                   "peak_tflops": pk, "peak_source": r["peak_source"],
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": r["roofline"],
        "e2e": r["e2e"],
        "gpu_launches": r["launches_per_step"] * K,
        "step_ms": r["step_ms"],
        "hbm": r["hbm"],
        "clocks": sampler.summary(),
        "wall_s_timed_region": round(r["wall"], 3),
    }
    if world == 1 and not args.no_other_workloads:
        others = {}
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            ow = wl.WORKLOADS[name]
            s2 = ClockSampler(torch.cuda.current_device())
            o = measure_workload(ow, K, args.warmup, torch, dev, world, flush, s2)
            others[name] = {
                "value": round(o["value"], 2), "unit": UNIT, "ms_per_step": round(o["ms_per_step"], 4),
                "frac_of_peak": round(o["value"] / pk, 4), "flops_per_step": o["step_flops"],
                "flops_counted": o["flops_counted"], "nominal_flops_per_step": o["nominal_flops"],
                "config": {"B": ow.B, "T_q": ow.T_q, "T_kv": ow.T_kv, "D": ow.D, "h": ow.h,
                           "d_k": ow.d_k, "causal": ow.causal, "cross": ow.cross},
                "roofline": o["roofline"], "e2e": o["e2e"], "step_ms": o["step_ms"], "hbm": o["hbm"],
                "clocks": s2.summary(), "steps": K, "warmup": args.warmup}
        line["other_workloads"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_baseline_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- variants

# The variants of itwiki.kr "멀티 헤드 어텐션", 추론 비용과 변형 and the residual of
# iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", section 14, measured on the
# c3 layer shape (B=4, T=2048, D=1024, h=16, d=64, causal), and the KV-cache decode step on a
# cache larger than L2.  Each prints its own JSON line; the default run prints none of them.
VARIANTS = {
    "residual": dict(h_kv=16, gated=False, residual=True),
    "gqa4": dict(h_kv=4, gated=False, residual=False),
    "mqa": dict(h_kv=1, gated=False, residual=False),
    "gated": dict(h_kv=16, gated=True, residual=False),
    "decode-mha": dict(decode=True, h_kv=16),
    "decode-gqa4": dict(decode=True, h_kv=4),
    "decode-mqa": dict(decode=True, h_kv=1),
    "decode-proj": dict(decode_proj=True),
}
DECODE_SHAPE = dict(B=32, T_q=1, T_max=8192, h=16, d=128)


def _timed_steps(torch, fn, flush, K, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda._sleep(PREQUEUE_CYCLES_PER_STEP * K)
    for k in range(K):
        flush.zero_()
        ev[k][0].record()
        fn()
        ev[k][1].record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / K


def run_variant(args):
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__ as g
    g.build_library()
    from transformer_head_scaled_02_gb300 import Mha
    v = VARIANTS[args.variant]
    pk, pk_src = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(0)

    def bf(shape, seed, scale=1.0):
        return to_device(wl.random_tensor(shape, seed, "bf16", scale), "bf16", torch)

    if v.get("decode_proj"):
        # the projections of the same decode step: B new tokens (one per sequence) through
        # W_qkv and, with the residual, through W_O; weights read once per step
        c = DECODE_SHAPE
        M, D = c["B"] * c["T_q"], c["h"] * c["d"]
        layer = Mha(D, c["h"], c["d"], c["d"], dtype=torch.bfloat16)
        layer.ensure_workspace(1, 1, 1)
        X = bf((M, D), 1)
        Wqkv, bqkv = bf((D, 3 * D), 2, 0.02), bf((3 * D,), 3, 0.02)
        Oc = bf((M, D), 4)
        Wo, bo = bf((D, D), 5, 0.02), bf((D,), 6, 0.02)
        qkv = torch.empty((M, 3 * D), dtype=torch.bfloat16, device=dev)
        Y = torch.empty((M, D), dtype=torch.bfloat16, device=dev)

        def fn():
            layer.linear(X, Wqkv, bqkv, out=qkv)
            layer.linear(Oc, Wo, bo, out=Y, residual=X)
        sampler.start()
        ms = _timed_steps(torch, fn, flush, args.steps, args.warmup)
        sampler.stop()
        if layer.status() != 0:
            raise RuntimeError("device status reports an error")
        weights = 2.0 * (D * 3 * D + D * D)
        small = 2.0 * (3 * D + D + M * D * 3 + M * 3 * D + M * D)   # biases, X twice, Ocat, outputs
        gbs = (weights + small) / (ms / 1e3) / 1e9
        line = {"metric": "MHA decode step projections: weight read bandwidth", "value": round(gbs, 1),
                "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) activations, N(0, 0.02^2) weights)",
                "config": {"variant": args.variant, "rows": M, "D": D, "qkv": [M, D, 3 * D],
                           "out_with_residual": [M, D, D], "weight_bytes": weights,
                           "l2": "flushed before every timed step"},
                "roofline": {"kernel": "gemm_bf16_splitk_kernel x 2", "bound": "hbm", "achieved": round(gbs, 1),
                             "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                             "peak_source": f"{pk_src} HBM copy"},
                "gpu_launches": 2 * args.steps, "clocks": sampler.summary()}
        print(json.dumps(line), flush=True)
        return

    if v.get("decode"):
        c = DECODE_SHAPE
        B, Tq, Tm, h, d, hkv = c["B"], c["T_q"], c["T_max"], c["h"], c["d"], v["h_kv"]
        layer = Mha(h * d, h, d, d, dtype=torch.bfloat16, h_kv=hkv)
        Q = bf((B, Tq, h * d), 1)
        Kc = bf((B, Tm, hkv * d), 2)
        Vc = bf((B, Tm, hkv * d), 3)
        lens = torch.full((B,), Tm, dtype=torch.int32, device=dev)
        O = torch.empty((B, Tq, h * d), dtype=torch.bfloat16, device=dev)
        fn = lambda: layer.decode(Q, Kc, Vc, lens, out=O)  # noqa: E731
        sampler.start()
        ms = _timed_steps(torch, fn, flush, args.steps, args.warmup)
        sampler.stop()
        if layer.status() != 0:
            raise RuntimeError("device status reports an error")
        cache = 2.0 * B * Tm * hkv * 2 * d          # K and V cache rows read once
        small = 2.0 * (Q.numel() + O.numel())
        gbs = (cache + small) / (ms / 1e3) / 1e9
        line = {"metric": "MHA decode step: KV-cache read bandwidth", "value": round(gbs, 1),
                "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) cache and queries)",
                "config": {"variant": args.variant, "B": B, "T_q": Tq, "T_max": Tm, "h": h, "h_kv": hkv,
                           "d": d, "cache_lengths": "all T_max", "cache_bytes": cache,
                           "l2": "flushed before every timed step"},
                "roofline": {"kernel": "decode_tc_kernel + decode_merge_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                             "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                             "peak_source": f"{pk_src} HBM copy"},
                "gpu_launches": 2 * args.steps, "clocks": sampler.summary()}
        print(json.dumps(line), flush=True)
        return

    B, T, D, h, d = 4, 2048, 1024, 16, 64
    hkv, gated, resid = v["h_kv"], v["gated"], v["residual"]
    layer = Mha(D, h, d, d, dtype=torch.bfloat16, h_kv=hkv, gated=gated)
    width = layer.proj_width
    X = bf((B, T, D), 1)
    Wqkv = bf((D, width), 2, 0.02)
    bqkv = bf((width,), 3, 0.02)
    Wo = bf((h * d, D), 4, 0.02)
    bo = bf((D,), 5, 0.02)
    out = torch.empty((B, T, D), dtype=torch.bfloat16, device=dev)
    fn = lambda: layer.forward(X, Wqkv, bqkv, Wo, bo, causal=True, out=out,  # noqa: E731
                               residual=X if resid else None)
    sampler.start()
    ms = _timed_steps(torch, fn, flush, args.steps, args.warmup)
    sampler.stop()
    if layer.status() != 0:
        raise RuntimeError("device status reports an error")
    proj = 2.0 * B * T * D * width + 2.0 * B * T * h * d * D
    attn = 2.0 * B * h * T * T * 2 * d * 0.5
    tf = (proj + attn) / (ms / 1e3) / 1e12
    # per-kernel durations of the same three launches, events between them
    hq, hk, hvv = h * d, hkv * d, hkv * d
    qkv = torch.empty((B, T, width), dtype=torch.bfloat16, device=dev)
    ocat = torch.empty((B, T, h * d), dtype=torch.bfloat16, device=dev)
    gview = qkv[..., hq + hk + hvv:] if gated else None
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        e = kev[k]
        e[0].record()
        layer.linear(X.view(-1, D), Wqkv, bqkv, out=qkv.view(-1, width))
        e[1].record()
        layer.attention(qkv[..., :hq], qkv[..., hq:hq + hk], qkv[..., hq + hk:hq + hk + hvv], causal=True,
                        out=ocat, G=gview)
        e[2].record()
        layer.linear(ocat.view(-1, h * d), Wo, bo, out=out.view(-1, D),
                     residual=X.view(-1, D) if resid else None)
        e[3].record()
    torch.cuda.synchronize()
    names = ["qkv_proj", "attention", "out_proj"]
    per_kernel = {n: statistics.mean(kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(args.steps))
                  for i, n in enumerate(names)}
    kflops = {"qkv_proj": 2.0 * B * T * D * width, "attention": attn, "out_proj": 2.0 * B * T * h * d * D}
    top = max(per_kernel, key=per_kernel.get)
    ach = kflops[top] / (per_kernel[top] / 1e3) / 1e12
    roofline = {"kernel": top, "bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4),
                "peak_source": f"{pk_src} bf16 dense (burst)",
                "per_kernel_ms": {k2: round(v2, 4) for k2, v2 in per_kernel.items()},
                "per_kernel_frac_of_peak": {k2: round(kflops[k2] / (v2 / 1e3) / 1e12 / pk["bf16_tflops"], 4)
                                            for k2, v2 in per_kernel.items()}}
    line = {"metric": f"MHA forward TFLOP/s, {args.variant} variant (bf16 causal, 1×GB300)",
            "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) weights)",
            "config": {"variant": args.variant, "B": B, "T": T, "D": D, "h": h, "h_kv": hkv, "d": d,
                       "gated": gated, "residual": resid, "proj_width": width,
                       "flops_per_step": proj + attn, "frac_of_peak": round(tf / pk["bf16_tflops"], 4),
                       "l2": "flushed before every timed step"},
            "roofline": roofline,
            "gpu_launches": 3 * args.steps, "clocks": sampler.summary()}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle on the host cores, each step a bounded sample of the workload
    (batch 0, a prefix of T' query rows), T' sized so the whole run takes about
    --reference-seconds."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    x = wl.make_inputs(w)

    def step(tp):
        t0 = time.perf_counter()
        if w.cross:
            L = None if x["kv_lengths"] is None else x["kv_lengths"][:1]
            oracle.mha_forward(x["X_q"][:1, :tp], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h,
                               w.d_k, w.d_v, Xkv=x["X_kv"][:1], causal=w.causal, kv_lengths=L)
        else:
            oracle.mha_forward(x["X_q"][:1, :tp], x["W_qkv"], x["b_qkv"], x["W_o"], x["b_o"], w.h,
                               w.d_k, w.d_v, causal=w.causal)
        return time.perf_counter() - t0

    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    tp = 16
    dt = step(tp)
    while tp < w.T_q and dt * 2 < per_step:
        tp = min(w.T_q, tp * 2)
        dt = step(tp)
    for _ in range(args.warmup):
        step(tp)
    times = [step(tp) for _ in range(args.steps)]
    sw = wl.custom("sample", B=1, T_q=tp, T_kv=w.T_kv if w.cross else tp, D=w.D, h=w.h, d_k=w.d_k,
                   d_v=w.d_v, dtype=w.dtype, causal=w.causal, cross=w.cross)
    f = wl.flops(sw)["total"]
    ms = 1e3 * sum(times) / len(times)
    value = f / (ms / 1e3) / 1e12
    sample = (f"batch 0, first {tp} of {w.T_q} query rows of {w.name} per step, fp64 oracle "
              f"on {oracle.max_threads()} host threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample_rows": tp},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only --workload (by default c4 and c5 follow in the same run)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--variant", choices=sorted(VARIANTS), default=None,
                    help="measure a variant (grouped heads, gate, residual, decode) instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.variant is not None:
        run_variant(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
