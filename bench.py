"""Benchmark of the QLoRA NF4 linear-layer hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (one "step"): forward + backward of the seven Llama-3-8B
projection shapes (q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096,
down 4096x14336), every base weight NF4 + double-quantised, LoRA r=16
alpha=32, 2048 tokens per projection, bf16 activations.  Metric: fused QLoRA
forward+backward TFLOP/s (algorithmic flops 2MNK + 2Mr(K+N) forward and
2MNK + 2MNr + 2MrK + 2MrK + 2MNr backward).  All inputs are seeded synthetic
tensors resident in HBM before timing; the per-step working set (~0.7 GB)
is far larger than the 126 MB L2.

The same JSON line also carries sub-measurements of the other hot-path
rows: the q_proj 4096x4096 forward at 2048 tokens (TFLOP/s), the decode
GEMV on the 14336x4096 gate projection at 1/4/16 tokens (GB/s of packed
4-bit weights, rotating over 8 weight copies so L2 cannot hold them), the
bulk NF4+DQ quantisation of 136 4096x14336 matrices (GB/s), and
dequantisation (GB/s).

--impl reference times the CPU oracle (the reference arm):
each step runs the oracle's forward + backward on a 4-token sample of one
projection of the same workload, cycling over the seven shapes.

Multi-GPU: replicas only.  Every rank runs the same per-GPU workload (no
data-path collective); timing is bracketed by a barrier and
torch.cuda.synchronize() and the maximum over ranks is reported; value is
the sum of the work of all ranks divided by that time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "fused QLoRA fwd+bwd TFLOP/s at M=2048; decode GEMV GB/s; NF4 quantise GB/s"
UNIT = "TFLOP/s"
M_TOKENS = 2048
RANK_R, ALPHA = 16, 32.0
LAYERS = [("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096),
          ("o_proj", 4096, 4096), ("gate_proj", 14336, 4096), ("up_proj", 14336, 4096),
          ("down_proj", 4096, 14336)]
KERNELS_PER_LAYER_STEP = 7  # fwd: LoRA pre-pass, GEMM; bwd: transposes, dY pre-pass, dX GEMM, dB, dA


def fwd_flops(M, N, K, r):
    return 2 * M * N * K + 2 * M * r * (K + N)


def bwd_flops(M, N, K, r):
    return 2 * M * N * K + 2 * M * N * r + 2 * M * r * K + 2 * M * r * K + 2 * M * N * r


# ----------------------------------------------------------------- dist glue
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def maybe_init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, ws: int, device) -> float:
    """Maximum of a per-rank float over all ranks (identity at world size 1)."""
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and throttle reasons of one GPU through NVML."""

    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index: int, period_s: float = 0.02):
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._h = None
        self.error = None
        try:
            import pynvml
            pynvml.nvmlInit()
            props = torch.cuda.get_device_properties(device_index)
            uuid = str(props.uuid)
            cands = [uuid, "GPU-" + uuid] if not uuid.startswith("GPU-") else [uuid]
            for u in cands:
                try:
                    self._h = pynvml.nvmlDeviceGetHandleByUUID(u)
                    break
                except Exception:  # noqa: BLE001
                    continue
            if self._h is None:
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id,
                                             props.pci_device_id)
                self._h = pynvml.nvmlDeviceGetHandleByPciBusId(bus)
            self._nv = pynvml
            self._reasons_fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception as e:  # noqa: BLE001
            self._h = None
            self.error = f"{type(e).__name__}: {e}"
            try:
                u = str(torch.cuda.get_device_properties(device_index).uuid)
                self._smi_id = u if u.startswith("GPU-") else "GPU-" + u
            except Exception:  # noqa: BLE001
                self._smi_id = str(device_index)

    def _run_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        cmd = ["nvidia-smi", "-i", self._smi_id, f"--query-gpu={q}", "--format=csv,noheader,nounits",
               f"-lms={max(20, int(self.period * 1000))}"]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                          text=True)
        except Exception as e:  # noqa: BLE001
            self.error = f"nvidia-smi: {e}"
            return
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                self.samples.append(float(parts[0]))
                self.max_mhz = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[2:6]):
                if val.lower() == "active":
                    self.reasons.add(name)

    def _run(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                bits = self._reasons_fn(self._h)
                for name, mask in self.REASONS.items():
                    if bits & mask:
                        self.reasons.add(name)
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def __enter__(self):
        self._proc = None
        target = self._run if self._h is not None else self._run_smi
        self._t = threading.Thread(target=target, daemon=True)
        self._t.start()
        if self._h is None:
            time.sleep(0.3)  # let nvidia-smi start sampling
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0, "error": self.error}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self._h is not None else "nvidia-smi"}


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def profile_traffic(kernel_tag: str, source_file: str):
    """DRAM bytes per launch of a kernel from the committed ncu figures in
    profiles/traffic.json ({tag: {"bytes_per_launch", "source_sha16", ...}}),
    or None when absent or when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    entry = json.load(open(p)).get(kernel_tag)
    if not entry:
        return None
    sha = hashlib.sha256(open(source_file, "rb").read()).hexdigest()[:16]
    return float(entry["bytes_per_launch"]) if entry.get("source_sha16") == sha else None


def pick_tensor_peak(peaks: dict, clocks: dict):
    """Dense bf16 peak for a kernel timed in this run: the sustained figure
    when the run's own clock record shows the power cap (or SM clocks well
    below max), else the burst figure."""
    reasons = set(clocks.get("reasons") or [])
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    low = mhz is not None and mx and mhz < 0.95 * float(mx)
    if "sw_power_cap" in reasons or low:
        why = "sw_power_cap seen" if "sw_power_cap" in reasons else f"SM clock {mhz} of {mx} MHz"
        return peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), \
            f"bf16_tflops_sustained ({why} during the timed region)"
    return peaks["bf16_tflops"], (f"bf16_tflops burst (SM clock {mhz} of {mx} MHz, no power cap "
                                  "during the timed region)")


def gen_bf16(shape, std, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


# --------------------------------------------------------------- our arm
def run_ours(args, ws_n, rank, device):
    from bit_nf4_quantized_35_b300 import build as libbuild
    libbuild.build()
    from bit_nf4_quantized_35_b300 import capi

    capi.load()
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    M = M_TOKENS
    layers = []
    for li, (name, N, K) in enumerate(LAYERS):
        W = gen_bf16((N, K), 0.02, 100 + li, device)
        q = capi.quantize_nf4(W)
        del W
        L = {
            "name": name, "N": N, "K": K, "q": q,
            "A": gen_bf16((RANK_R, K), 0.01, 200 + li, device),
            "B": gen_bf16((N, RANK_R), 0.01, 300 + li, device),
            "x": gen_bf16((M, K), 1.0, 400 + li, device),
            "dY": gen_bf16((M, N), 1.0, 500 + li, device),
            "t": torch.empty((M, RANK_R), dtype=torch.float32, device=device),
            "y": torch.empty((M, N), dtype=torch.bfloat16, device=device),
            "dX": torch.empty((M, K), dtype=torch.bfloat16, device=device),
            "dA": torch.empty((RANK_R, K), dtype=torch.float32, device=device),
            "dB": torch.empty((N, RANK_R), dtype=torch.float32, device=device),
            "ws": capi.Workspace(M, N, K, RANK_R, device=device),
        }
        layers.append(L)
    torch.cuda.synchronize()

    def layer_fwd(L):
        capi.linear_fwd(L["q"], L["x"], L["A"], L["B"], ALPHA, L["ws"], y=L["y"], t_save=L["t"])

    def layer_bwd(L):
        capi.linear_bwd(L["q"], L["x"], L["dY"], L["A"], L["B"], ALPHA, L["ws"], t_saved=L["t"],
                        dX=L["dX"], dA=L["dA"], dB=L["dB"])

    step_flops = sum(fwd_flops(M, L["N"], L["K"], RANK_R) + bwd_flops(M, L["N"], L["K"], RANK_R)
                     for L in layers)
    fwd_gemm_flops = sum(fwd_flops(M, L["N"], L["K"], RANK_R) for L in layers)

    for _ in range(args.warmup):
        for L in layers:
            layer_fwd(L)
            layer_bwd(L)
    torch.cuda.synchronize()

    # --- timed region: K steps, events around each forward (one GEMM launch)
    ev_pairs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in layers] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device)
    barrier(ws_n)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with sampler:
        start.record(stream)
        for s in range(args.steps):
            for li, L in enumerate(layers):
                e0, e1 = ev_pairs[s][li]
                e0.record(stream)
                layer_fwd(L)
                e1.record(stream)
                layer_bwd(L)
        end.record(stream)
        torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(ws_n)
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, ws_n, device)
    ms_step = ms_total / args.steps
    value = sum_over_ranks(step_flops * args.steps, ws_n, device) / (ms_total * 1e-3) / 1e12
    # Per-layer forward GEMM launch times (each forward call is one GEMM launch).
    layer_ms = [sum(ev_pairs[s][li][0].elapsed_time(ev_pairs[s][li][1]) for s in range(args.steps))
                / args.steps for li in range(len(layers))]
    fwd_ms = sum(layer_ms)
    gi = [L["name"] for L in layers].index("gate_proj")
    gate_flops = fwd_flops(M, layers[gi]["N"], layers[gi]["K"], RANK_R)
    gemm_achieved = gate_flops / (layer_ms[gi] * 1e-3) / 1e12  # TFLOP/s, gate_proj forward
    clocks = sampler.summary()

    # --- e2e: host buffers through the C ABI, copies inside the timed region
    e2e_steps = max(3, min(args.steps, 20))
    host = []
    for L in layers:
        host.append({
            "x": L["x"].cpu().pin_memory(), "dY": L["dY"].cpu().pin_memory(),
            "y": torch.empty_like(L["y"], device="cpu").pin_memory(),
            "dX": torch.empty_like(L["dX"], device="cpu").pin_memory(),
            "dA": torch.empty_like(L["dA"], device="cpu").pin_memory(),
            "dB": torch.empty_like(L["dB"], device="cpu").pin_memory(),
        })
    h2d = sum(h["x"].numel() * 2 + h["dY"].numel() * 2 for h in host)
    d2h = sum(h["y"].numel() * 2 + h["dX"].numel() * 2 + h["dA"].numel() * 4 +
              h["dB"].numel() * 4 for h in host)

    # Inputs go up on one copy stream while earlier layers compute (a training
    # loop prefetching its next batch) and every result (y, dX, dA, dB) comes
    # back on another: layer i's compute waits for its inputs and for the
    # previous step's read-back of its outputs; the next step's copies into
    # layer i's input buffers wait until this step's layer i is done with them.
    up_stream = torch.cuda.Stream(device=device)
    down_stream = torch.cuda.Stream(device=device)
    ready = [torch.cuda.Event() for _ in layers]
    inputs_free = [torch.cuda.Event() for _ in layers]
    computed = [torch.cuda.Event() for _ in layers]
    outputs_free = [torch.cuda.Event() for _ in layers]

    def e2e_step(start=None):
        if start is not None:
            up_stream.wait_event(start)  # the timed region opens before the first copy
        for i, (L, h) in enumerate(zip(layers, host)):
            up_stream.wait_event(inputs_free[i])
            with torch.cuda.stream(up_stream):
                L["x"].copy_(h["x"], non_blocking=True)
                L["dY"].copy_(h["dY"], non_blocking=True)
            ready[i].record(up_stream)
        for i, (L, h) in enumerate(zip(layers, host)):
            stream.wait_event(ready[i])
            stream.wait_event(outputs_free[i])
            layer_fwd(L)
            layer_bwd(L)
            inputs_free[i].record(stream)
            computed[i].record(stream)
            down_stream.wait_event(computed[i])
            with torch.cuda.stream(down_stream):
                for k in ("y", "dX", "dA", "dB"):
                    h[k].copy_(L[k], non_blocking=True)
            outputs_free[i].record(down_stream)

    e2e_step()
    torch.cuda.synchronize()
    barrier(ws_n)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for k in range(e2e_steps):
        e2e_step(s0 if k == 0 else None)
    stream.wait_stream(down_stream)
    s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s0.elapsed_time(s1), ws_n, device)
    e2e_value = sum_over_ranks(step_flops * e2e_steps, ws_n, device) / (e2e_ms * 1e-3) / 1e12

    rows = sub_benchmarks(capi, layers, device, stream, args) if not args.no_rows else {}

    peaks, peak_src = measured_peaks()
    peak, peak_kind = pick_tensor_peak(peaks, clocks)
    traffic = profile_traffic("qlora_gemm_kernel<false>:gate_proj_14336x4096_M2048",
                              os.path.join(ROOT, "bit_nf4_quantized_35_b300", "csrc",
                                            "gemm_tc.cu"))
    out = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "llama3_8b_7proj_fwd_bwd_M2048_r16_nf4dq",
            "global_batch": M_TOKENS * ws_n,
            "tokens_per_gpu": M_TOKENS,
            "projections": [f"{n}:{N}x{K}" for n, N, K in LAYERS],
            "r": RANK_R, "alpha": ALPHA, "block": 64, "dq_group": 256,
            "parallelism": f"replicas x{ws_n}",
            "l2": "per-step working set ~0.7 GB >> 126 MB L2 (no flush needed)",
            "wall_s_timed": round(t_wall, 3),
        },
        "roofline": {
            "kernel": "qlora_gemm_kernel<false> (fused NF4 dequant + tcgen05 GEMM + LoRA) on "
                      "gate_proj 14336x4096 at M=2048: CUDA events around each gate forward "
                      "call of the timed steps, which is the t = x.A^T pre-pass (about 4% of "
                      "it) and this GEMM launch; flops are the whole call's",
            "flops_per_launch": gate_flops,
            "avg_launch_ms": round(layer_ms[gi], 4),
            "bound": "tensor",
            "achieved": round(gemm_achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_src} {peak_kind}",
            "unit": "TFLOP/s",
            "frac": round(gemm_achieved / peak, 4),
            "traffic": traffic,
        },
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": "x, dY up from pinned host buffers; y, dX (bf16), dA, dB (fp32) "
                          "back to pinned host buffers, on two copy streams overlapped with "
                          "compute"},
        "gpu_launches": KERNELS_PER_LAYER_STEP * len(layers) * args.steps,
        "fwd_gemm_per_layer": {L["name"]: {"ms": round(ms, 4), "tflops": round(
            fwd_flops(M, L["N"], L["K"], RANK_R) / (ms * 1e-3) / 1e12, 1)}
            for L, ms in zip(layers, layer_ms)},
        "fwd_gemm_all_layers_tflops": round(fwd_gemm_flops / (fwd_ms * 1e-3) / 1e12, 1),
        "clocks": clocks,
        "rows": rows,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(tokens=16, layers_subset=None)
        if not args.no_rows:
            out["cpu_baseline"]["rows"] = oracle_rows()
    return out


def time_graph(fn, iters, stream):
    """Capture `iters` calls of fn into a CUDA graph and time one replay."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(iters):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(5):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return best / iters  # ms per call


def sub_benchmarks(capi, layers, device, stream, args):
    rows = {}
    peaks, _ = measured_peaks()
    hbm = peaks["hbm_gbs"]
    # q_proj forward, M = 2048 (prefill / training forward of a 4096x4096 projection)
    L = layers[0]
    s = torch.cuda.Stream(device=device)
    with torch.cuda.stream(s):
        ms = time_graph(lambda i: capi.linear_fwd(L["q"], L["x"], L["A"], L["B"], ALPHA, L["ws"],
                                                  y=L["y"], t_save=L["t"], stream=s), 20, s)
    fl = fwd_flops(M_TOKENS, 4096, 4096, RANK_R)
    peak = peaks["bf16_tflops"]
    rows["qproj_fwd_M2048"] = {"ms": round(ms, 4), "tflops": round(fl / ms / 1e9, 2),
                               "frac_of_bf16_burst_peak": round(fl / ms / 1e9 / peak, 4)}
    # decode GEMV on gate 14336x4096, 8 rotating weight copies (> L2)
    N, K = 14336, 4096
    copies = []
    for c in range(8):
        copies.append(capi.quantize_nf4(gen_bf16((N, K), 0.02, 600 + c, device)))
    A = gen_bf16((RANK_R, K), 0.01, 700, device)
    B = gen_bf16((N, RANK_R), 0.01, 701, device)
    packed_bytes = N * K // 2
    for Mg in (1, 4, 16):
        x = gen_bf16((Mg, K), 1.0, 800 + Mg, device)
        y = torch.empty((Mg, N), dtype=torch.bfloat16, device=device)
        t = torch.empty((Mg, RANK_R), dtype=torch.float32, device=device)
        ws = capi.Workspace(Mg, N, K, RANK_R, device=device)
        call = lambda i: capi.linear_fwd(copies[i % 8], x, A, B, ALPHA, ws, y=y, t_save=t,
                                         stream=s)
        with torch.cuda.stream(s):
            ms = time_graph(call, 64, s)
            # the same 64 calls launched one by one from the host: the difference is the
            # per-call launch overhead that the graph replay hides
            for i in range(8):
                call(i)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(s)
            for i in range(64):
                call(i)
            ev1.record(s)
        torch.cuda.synchronize()
        eager_ms = ev0.elapsed_time(ev1) / 64
        gbs = packed_bytes / (ms * 1e-3) / 1e9
        rows[f"gemv_gate_M{Mg}"] = {"us": round(ms * 1e3, 2), "packed_GBps": round(gbs, 1),
                                    "frac_of_hbm": round(gbs / hbm, 4),
                                    "eager_us": round(eager_ms * 1e3, 2),
                                    "launch_overhead_us": round((eager_ms - ms) * 1e3, 2)}
    del copies
    # bulk quantisation: 136 x (4096 x 14336) bf16 -> NF4 + DQ (streamed in chunks of 8)
    nmat = 136 if not args.quick else 16
    Rq, Cq = 4096, 14336
    chunk = 8
    mats = [gen_bf16((Rq, Cq), 0.02, 1000 + i, device) for i in range(chunk)]
    outs = [capi.NF4Weight.empty(Rq, Cq, device) for _ in range(chunk)]
    for m in mats:  # outliers: 0.1% of entries -> +-10 sigma
        g = torch.Generator(device=device)
        g.manual_seed(12345)
        mask = torch.rand(m.shape, generator=g, device=device) < 1e-3
        sign = torch.where(torch.rand(m.shape, generator=g, device=device) < 0.5, -0.2, 0.2)
        m[mask] = sign[mask].to(torch.bfloat16)
    for i in range(chunk):  # warm-up: one call per matrix
        capi.quantize_nf4(mats[i], out=outs[i])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(nmat):
        capi.quantize_nf4(mats[i % chunk], out=outs[i % chunk])
    e1.record()
    torch.cuda.synchronize()
    qms = e0.elapsed_time(e1)
    nw = nmat * Rq * Cq
    bytes_total = nw * (2 + 0.5 + 1 / 64 + 4 / 16384)
    rows["quantize_bulk"] = {"matrices": nmat, "weights": nw, "ms": round(qms, 3),
                             "GBps_total": round(bytes_total / (qms * 1e-3) / 1e9, 1),
                             "GBps_input": round(nw * 2 / (qms * 1e-3) / 1e9, 1),
                             "frac_of_hbm": round(bytes_total / (qms * 1e-3) / 1e9 / hbm, 4),
                             "note": "8 distinct 117 MB matrices cycled (> L2)"}
    # dequantisation to bf16 of the same matrices
    outw = torch.empty((Rq, Cq), dtype=torch.bfloat16, device=device)
    for i in range(3):  # warm-up
        capi.dequant(outs[i], out=outw)
    e0.record()
    for i in range(32):
        capi.dequant(outs[i % chunk], out=outw)
    e1.record()
    torch.cuda.synchronize()
    dms = e0.elapsed_time(e1) / 32
    db = Rq * Cq * (0.5 + 1 / 64 + 4 / 16384 + 2)
    rows["dequant_4096x14336"] = {"us": round(dms * 1e3, 1),
                                  "GBps": round(db / (dms * 1e-3) / 1e9, 1),
                                  "frac_of_hbm": round(db / (dms * 1e-3) / 1e9 / hbm, 4)}
    del mats, outs, outw
    torch.cuda.empty_cache()
    # adapter merge bf16(W_hat + alpha/r B A) of the gate and up projections, alternating
    mg = [L for L in layers if L["name"] in ("gate_proj", "up_proj")]
    mo = [torch.empty((L["N"], L["K"]), dtype=torch.bfloat16, device=device) for L in mg]
    for i in range(3):
        capi.merge_lora(mg[i % 2]["q"], mg[i % 2]["A"], mg[i % 2]["B"], ALPHA, out=mo[i % 2])
    torch.cuda.synchronize()
    e0.record()
    for i in range(20):
        capi.merge_lora(mg[i % 2]["q"], mg[i % 2]["A"], mg[i % 2]["B"], ALPHA, out=mo[i % 2])
    e1.record()
    torch.cuda.synchronize()
    mms = e0.elapsed_time(e1) / 20
    Nm, Km = mg[0]["N"], mg[0]["K"]
    mb = Nm * Km * (0.5 + 1 / 64 + 4 / 16384 + 2) + RANK_R * (Nm + Km) * 2
    rows["merge_14336x4096"] = {"us": round(mms * 1e3, 1), "GBps": round(mb / (mms * 1e-3) / 1e9, 1),
                                "frac_of_hbm": round(mb / (mms * 1e-3) / 1e9 / hbm, 4),
                                "note": "gate and up weights alternated (147 MB per call pair > L2)"}
    del mo
    rows["llama3_7proj_fwd_bwd_M8192"] = layer_set_at(capi, layers, 8192, device, stream,
                                                      steps=3 if args.quick else 6)
    rows["llama3_7proj_fwd_bwd_dropout0.1_M2048"] = dropout_step(capi, layers, device, stream,
                                                                 steps=5 if args.quick else 20)
    return rows


def dropout_step(capi, layers, device, stream, steps, p=0.1):
    """The headline step with LoRA dropout p on every projection: per layer
    and step, the keep mask is drawn (Philox, in the timed region), the
    forward and backward take it (fp32 dX)."""
    M = M_TOKENS
    dx32 = [torch.empty((M, L["K"]), dtype=torch.float32, device=device) for L in layers]
    masks = [torch.empty((M, capi.dropout_mask_words(L["K"])), dtype=torch.int32, device=device)
             for L in layers]

    def step(si, ev=None):
        for li, L in enumerate(layers):
            mk = capi.dropout_mask(1000 * si + li, p, M, L["K"], out=masks[li])
            capi.linear_fwd(L["q"], L["x"], L["A"], L["B"], ALPHA, L["ws"], y=L["y"],
                            t_save=L["t"], dropout=(mk, p))
            capi.linear_bwd(L["q"], L["x"], L["dY"], L["A"], L["B"], ALPHA, L["ws"],
                            t_saved=L["t"], dX=dx32[li], dA=L["dA"], dB=L["dB"],
                            dropout=(mk, p))

    for si in range(3):
        step(si)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for si in range(steps):
        step(si)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    total = sum(fwd_flops(M, L["N"], L["K"], RANK_R) + bwd_flops(M, L["N"], L["K"], RANK_R)
                for L in layers)
    return {"p": p, "steps": steps, "ms_per_step": round(ms, 4),
            "tflops": round(total / (ms * 1e-3) / 1e12, 2),
            "note": "mask drawn per layer per step inside the timed region; dX in fp32"}


def layer_set_at(capi, layers, M, device, stream, steps):
    """Forward + backward of the seven projections at M tokens (the layer set
    as its workload states it: 4 x 2048 tokens), per layer and in total."""
    bufs = []
    for li, L in enumerate(layers):
        N, K = L["N"], L["K"]
        bufs.append({
            "x": gen_bf16((M, K), 1.0, 900 + li, device),
            "dY": gen_bf16((M, N), 1.0, 950 + li, device),
            "t": torch.empty((M, RANK_R), dtype=torch.float32, device=device),
            "y": torch.empty((M, N), dtype=torch.bfloat16, device=device),
            "dX": torch.empty((M, K), dtype=torch.bfloat16, device=device),
            "dA": torch.empty((RANK_R, K), dtype=torch.float32, device=device),
            "dB": torch.empty((N, RANK_R), dtype=torch.float32, device=device),
            "ws": capi.Workspace(M, N, K, RANK_R, device=device),
        })

    def run(L, b, ev=None):
        if ev:
            ev[0].record(stream)
        capi.linear_fwd(L["q"], b["x"], L["A"], L["B"], ALPHA, b["ws"], y=b["y"], t_save=b["t"])
        if ev:
            ev[1].record(stream)
        capi.linear_bwd(L["q"], b["x"], b["dY"], L["A"], L["B"], ALPHA, b["ws"], t_saved=b["t"],
                        dX=b["dX"], dA=b["dA"], dB=b["dB"])
        if ev:
            ev[2].record(stream)

    for _ in range(3):
        for L, b in zip(layers, bufs):
            run(L, b)
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in layers]
           for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in range(steps):
        for li, (L, b) in enumerate(zip(layers, bufs)):
            run(L, b, evs[st][li])
    e1.record(stream)
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / steps
    total = sum(fwd_flops(M, L["N"], L["K"], RANK_R) + bwd_flops(M, L["N"], L["K"], RANK_R)
                for L in layers)
    per = {}
    for li, L in enumerate(layers):
        f = sum(evs[st][li][0].elapsed_time(evs[st][li][1]) for st in range(steps)) / steps
        bw = sum(evs[st][li][1].elapsed_time(evs[st][li][2]) for st in range(steps)) / steps
        per[L["name"]] = {
            "fwd_ms": round(f, 4), "bwd_ms": round(bw, 4),
            "fwd_tflops": round(fwd_flops(M, L["N"], L["K"], RANK_R) / (f * 1e-3) / 1e12, 1),
            "bwd_tflops": round(bwd_flops(M, L["N"], L["K"], RANK_R) / (bw * 1e-3) / 1e12, 1)}
    del bufs
    torch.cuda.empty_cache()
    return {"tokens": M, "steps": steps, "ms_per_step": round(ms_step, 4),
            "tflops": round(total / (ms_step * 1e-3) / 1e12, 2), "per_layer": per}


def oracle_rows():
    """The oracle, as it stands, timed on the host cores for the other rows
    of the line: with one thread and with all of them, on the workloads the
    GPU rows run (samples where stated)."""
    import numpy as np
    from bit_nf4_quantized_35_b300 import inputs
    from oracle import oracle

    oracle.build()
    ncores = oracle.num_threads()
    out = {"cores_all": ncores}

    def timed(fn):
        res = {}
        for tag, n in (("1_thread", 1), ("all_cores", ncores)):
            oracle.set_num_threads(n)
            t0 = time.perf_counter()
            fn()
            res[tag] = time.perf_counter() - t0
        oracle.set_num_threads(ncores)
        return res

    # decode GEMV on gate 14336x4096: the oracle dequantises the packed weight
    # and runs the fp64 forward (GB/s of packed weights, as the GPU row)
    N, K = 14336, 4096
    W = inputs.normal((N, K), inputs.STD_W, inputs.SEED_W).float().numpy()
    q = oracle.quantize_nf4(W, 64, 256, want_idx=False)
    A = inputs.normal((RANK_R, K), inputs.STD_LORA, inputs.SEED_A).float().numpy()
    B = inputs.normal((N, RANK_R), inputs.STD_LORA, inputs.SEED_B).float().numpy()
    for Mg in (1, 4, 16):
        x = inputs.normal((Mg, K), 1.0, inputs.SEED_X).float().numpy()
        t = timed(lambda: oracle.linear_fwd(x, oracle.dequant_f32(q), A, B, ALPHA))
        out[f"gemv_gate_M{Mg}"] = {k: {"s": round(v, 3), "packed_GBps": round(
            N * K / 2 / v / 1e9, 3)} for k, v in t.items()}
    # adapter merge of the gate weight (the bytes of the GPU row)
    wg = oracle.dequant_f32(q)
    mbytes = N * K * (0.5 + 1 / 64 + 4 / 16384 + 2) + RANK_R * (N + K) * 2
    t = timed(lambda: oracle.merge_bf16(wg, A, B, ALPHA))
    out["merge_14336x4096"] = {k: {"s": round(v, 3), "GBps": round(mbytes / v / 1e9, 3)}
                               for k, v in t.items()}
    # dequantisation of one 4096x14336 matrix
    Wb = inputs.bulk_matrix(0).float().numpy()
    qb = oracle.quantize_nf4(Wb, 64, 256, want_idx=False)
    db = 4096 * 14336 * (0.5 + 1 / 64 + 4 / 16384 + 2)
    t = timed(lambda: oracle.dequant_bf16(qb))
    out["dequant_4096x14336"] = {k: {"s": round(v, 3), "GBps": round(db / v / 1e9, 3)}
                                 for k, v in t.items()}
    # bulk quantisation: one of the 136 matrices (with its outliers)
    qbytes = 4096 * 14336 * (2 + 0.5 + 1 / 64 + 4 / 16384)
    t = timed(lambda: oracle.quantize_nf4(Wb, 64, 256, want_idx=False))
    out["quantize_bulk"] = {k: {"s": round(v, 3), "GBps": round(qbytes / v / 1e9, 3)}
                            for k, v in t.items()}
    out["quantize_bulk"]["sample"] = "1 of the 136 4096x14336 matrices (bulk matrix 0)"
    # q_proj 4096x4096 forward at 2048 tokens: in full on all cores; on one
    # thread 64 of the tokens (rows are independent), the full time scaled x32
    shape = inputs.QPROJ_2048
    d = inputs.linear_inputs(shape, with_dy=False)
    wq = oracle.dequant_f32(oracle.quantize_nf4(d["W"].float().numpy(), 64, 256, want_idx=False))
    xq, Aq, Bq = d["x"].float().numpy(), d["A"].float().numpy(), d["B"].float().numpy()
    fl = fwd_flops(2048, 4096, 4096, RANK_R)
    oracle.set_num_threads(1)
    t0 = time.perf_counter()
    oracle.linear_fwd(xq, wq, Aq, Bq, shape.alpha, rows=np.arange(64, dtype=np.int64))
    t1 = (time.perf_counter() - t0) * 2048 / 64
    oracle.set_num_threads(ncores)
    t0 = time.perf_counter()
    oracle.linear_fwd(xq, wq, Aq, Bq, shape.alpha)
    ta = time.perf_counter() - t0
    out["qproj_fwd_M2048"] = {
        "1_thread": {"s": round(t1, 2), "tflops": round(fl / t1 / 1e12, 6),
                     "sample": "64 of the 2048 tokens, time scaled x32"},
        "all_cores": {"s": round(ta, 2), "tflops": round(fl / ta / 1e12, 6),
                      "sample": "all 2048 tokens"}}
    # the 256x256 single layer (r = 8, 4 tokens), forward + backward in full
    s1 = inputs.SINGLE_256
    d1 = {k: v.float().numpy() for k, v in inputs.linear_inputs(s1).items()}
    w1 = oracle.dequant_f32(oracle.quantize_nf4(d1["W"], 64, 256, want_idx=False))
    t = timed(lambda: (oracle.linear_fwd(d1["x"], w1, d1["A"], d1["B"], s1.alpha),
                       oracle.linear_bwd(d1["x"], d1["dY"], w1, d1["A"], d1["B"], s1.alpha)))
    out["single_256_fwd_bwd"] = {k: {"s": round(v, 5)} for k, v in t.items()}
    return out


# ------------------------------------------------------- oracle (CPU) arm
def oracle_sample_step(layer_idx: int, tokens: int):
    """Oracle forward + backward of `tokens` tokens of one projection.
    Returns (flops, seconds)."""
    import numpy as np
    from bit_nf4_quantized_35_b300 import inputs
    from oracle import oracle

    name, N, K = LAYERS[layer_idx]
    key = (layer_idx, tokens)
    cache = oracle_sample_step.cache
    if key not in cache:
        shape = inputs.LinearShape(name, N=N, K=K, M=tokens, r=RANK_R, alpha=ALPHA)
        d = inputs.linear_inputs(shape, seed_offset=10 * layer_idx)
        q = oracle.quantize_nf4(d["W"].float().numpy(), 64, 256, want_idx=False)
        cache[key] = (d["x"].float().numpy(), d["dY"].float().numpy(), oracle.dequant_f32(q),
                      d["A"].float().numpy(), d["B"].float().numpy())
    x, dY, w, A, B = cache[key]
    t0 = time.perf_counter()
    oracle.linear_fwd(x, w, A, B, ALPHA)
    oracle.linear_bwd(x, dY, w, A, B, ALPHA)
    dt = time.perf_counter() - t0
    return fwd_flops(tokens, N, K, RANK_R) + bwd_flops(tokens, N, K, RANK_R), dt


oracle_sample_step.cache = {}


def cpu_baseline(tokens=16, layers_subset=None):
    from oracle import oracle
    idx = layers_subset if layers_subset is not None else range(len(LAYERS))
    fl = sec = 0.0
    for li in idx:
        f, s = oracle_sample_step(li, tokens)
        fl += f
        sec += s
    return {"value": round(fl / sec / 1e12, 6), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"oracle fp64 forward+backward of {tokens} tokens of each of the 7 "
                      f"projections ({fl / 1e9:.1f} GFLOP, {sec:.1f} s)"}


def run_reference(args, ws_n, rank):
    if rank != 0:
        return None
    from oracle import oracle
    oracle.build()
    tokens = 4
    for i in range(args.warmup):
        oracle_sample_step(i % len(LAYERS), tokens)
    fl = sec = 0.0
    t0 = time.perf_counter()
    for s in range(args.steps):
        f, dt = oracle_sample_step(s % len(LAYERS), tokens)
        fl += f
        sec += dt
    wall = time.perf_counter() - t0
    value = fl / sec / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "llama3_8b_7proj_fwd_bwd_M2048_r16_nf4dq",
                   "sample": f"{tokens} tokens of one projection per step, cycling the 7 shapes",
                   "wall_s": round(wall, 2)},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{tokens} tokens per step, one projection per step"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_case(args):
    """One kernel case, args.steps launches after args.warmup, for profilers:
    gemm_fwd / gemm_dx on the 14336x4096 gate projection at 2048 tokens,
    gemv on the same weight at --M tokens, quantise (bf16 or fp32 weight) /
    dequantise / adapter merge of one 14336x4096 matrix, the backward with
    LoRA dropout (p = 0.1, mask drawn each call) at 2048 tokens."""
    from bit_nf4_quantized_35_b300 import build as libbuild
    libbuild.build()
    from bit_nf4_quantized_35_b300 import capi
    dev = 0
    N, K = 14336, 4096
    M = M_TOKENS if args.only.startswith(("gemm", "dropout")) else args.M
    W = gen_bf16((N, K), 0.02, 100, dev)
    q = capi.quantize_nf4(W)
    A = gen_bf16((RANK_R, K), 0.01, 200, dev)
    B = gen_bf16((N, RANK_R), 0.01, 300, dev)
    x = gen_bf16((M, K), 1.0, 400, dev)
    dY = gen_bf16((M, N), 1.0, 500, dev)
    t = torch.empty((M, RANK_R), dtype=torch.float32, device=dev)
    ws = capi.Workspace(M, N, K, RANK_R, device=dev)
    out_q = capi.NF4Weight.empty(N, K, dev)
    out_w = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    W32 = W.float() if args.only == "quantize_f32" else None
    mask = torch.empty((M, capi.dropout_mask_words(K)), dtype=torch.int32, device=dev)
    fns = {
        "gemm_fwd": lambda: capi.linear_fwd(q, x, A, B, ALPHA, ws, y_dtype=torch.bfloat16,
                                            t_save=t),
        "gemm_dx": lambda: capi.linear_bwd(q, x, dY, A, B, ALPHA, ws, t_saved=t,
                                           dx_dtype=torch.bfloat16),
        "gemv": lambda: capi.linear_fwd(q, x, A, B, ALPHA, ws, y_dtype=torch.bfloat16, t_save=t),
        "quantize": lambda: capi.quantize_nf4(W, out=out_q),
        "quantize_f32": lambda: capi.quantize_nf4(W32, out=out_q),
        "dequant": lambda: capi.dequant(q, out=out_w),
        "merge": lambda: capi.merge_lora(q, A, B, ALPHA, out=out_w),
        "dropout_bwd": lambda: capi.linear_bwd(
            q, x, dY, A, B, ALPHA, ws, t_saved=t, dropout=(
                capi.dropout_mask(7, 0.1, M, K, out=mask), 0.1)),
    }
    capi.linear_fwd(q, x, A, B, ALPHA, ws, t_save=t)
    fn = fns[args.only]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"case": args.only, "M": M, "ms_per_call": e0.elapsed_time(e1) / args.steps,
                      "status": ws.device_status()}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="smaller sub-benchmarks")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row sub-benchmarks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["gemm_fwd", "gemm_dx", "gemv", "quantize",
                                       "quantize_f32", "dequant", "merge", "dropout_bwd"],
                    help="run one kernel case a few times and exit (for profiling)")
    ap.add_argument("--M", type=int, default=1, help="tokens for --only gemv")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    ws_n, rank, local = dist_info()
    if args.only:
        run_case(args)
        return
    if args.impl == "reference":
        maybe_init_dist(ws_n, "gloo")
        out = run_reference(args, ws_n, rank)
    else:
        maybe_init_dist(ws_n, "nccl")
        out = run_ours(args, ws_n, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
