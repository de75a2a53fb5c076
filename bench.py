"""Attention fwd+bwd throughput on GB300 through the C ABI (libfa.so).

One step = one forward (fa_fwd) and one backward (fa_bwd_preprocess, then
fa_bwd_grads for dK, dV and dQ) over one batch of the workload, inputs
resident in HBM.
FLOP convention: forward 4*B*H*Nq*Nk*d, backward 2.5x that, both halved when
causal.  L2 (129 MB) is flushed by writing a 512 MiB buffer between timed
steps; each step is timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step).  Under torchrun every rank runs
the same per-GPU workload (independent batch*head units, no collective on the
data path): weak scaling; rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s and % of GB300 bf16 tensor peak on 1 GPU"
DEFAULT_WORKLOAD = "bench_b8_n4096_d64_causal"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"bf16_tflops": j["bf16_tflops"], "bf16_tflops_sustained": j.get("bf16_tflops_sustained"),
                "hbm_gbs": j["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """SM clocks and throttle reasons sampled while the timed region runs.

    Reads NVML through ctypes every millisecond (read-only queries), falling
    back to `nvidia-smi -lms 50` when libnvidia-ml cannot be loaded.
    """
    HW_SLOWDOWN, SW_POWER_CAP, SW_THERMAL, HW_THERMAL = 0x8, 0x4, 0x20, 0x40

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []           # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.stop = threading.Event()
        self.nvml = None
        self.proc = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM = 1
            self.max_mhz = float(mx.value)
        self.reasons_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                           or lib.nvmlDeviceGetCurrentClocksThrottleReasons)
        self.nvml, self.h = lib, h
        return True

    def _poll_nvml(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.reasons_fn(self.h, ctypes.byref(rs))
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def _read_smi(self):
        for line in self.proc.stdout:
            r = [x.strip() for x in line.split(",")]
            try:
                mask = 0
                for bit, v in zip((self.HW_SLOWDOWN, self.HW_THERMAL, self.SW_THERMAL, self.SW_POWER_CAP), r[3:7]):
                    if v.lower() == "active":
                        mask |= bit
                self.samples.append((float(r[0]), mask))
                self.max_mhz = float(r[1])
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        try:
            ok = self._nvml_open()
        except OSError:
            ok = False
        if ok:
            self.t = threading.Thread(target=self._poll_nvml, daemon=True)
            self.t.start()
            while not self.samples and self.t.is_alive():
                time.sleep(0.001)
            return self
        try:
            q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read_smi, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if hasattr(self, "t"):
            self.t.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        names = {self.HW_SLOWDOWN: "hw_slowdown", self.HW_THERMAL: "hw_thermal_slowdown",
                 self.SW_THERMAL: "sw_thermal_slowdown", self.SW_POWER_CAP: "sw_power_cap"}
        mask = 0
        for _, m in self.samples:
            mask |= m
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(v for k, v in names.items() if mask & k), "samples": len(self.samples),
                "source": "nvml" if self.nvml else "nvidia-smi"}


# ---------------------------------------------------------------------------- CPU oracle timing

def oracle_sample(w, budget_s: float, max_units=None):
    """Time the oracle on whole batch*head units of the workload until ~budget_s has passed."""
    import oracle
    from tiled_attention_04_gb300 import inputs
    Q, K, V, dO = inputs.make_inputs(w)
    fwd, bwd = w.flops()
    per_unit = (fwd + bwd) / w.BH
    units, t = 0, 0.0
    limit = max_units or w.BH
    while units < limit and (t < budget_s or units == 0):
        b = units % w.BH
        t0 = time.perf_counter()
        oracle.attn_bwd_ref(Q.exact[b:b + 1], K.exact[b:b + 1], V.exact[b:b + 1], dO.exact[b:b + 1],
                            w.scale, w.causal)
        t += time.perf_counter() - t0
        units += 1
    try:
        from threadpoolctl import threadpool_info
        cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=os.cpu_count())
    except Exception:
        cores = os.cpu_count()
    return {"value": per_unit * units / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{units} of {w.BH} batch*head units of {w.name} (full rows, fwd+bwd), {t:.1f} s"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    steps = []
    for i in range(args.warmup + args.steps):
        r = oracle_sample(w, budget_s=0.0, max_units=1)
        if i >= args.warmup:
            steps.append(r)
    v = statistics.mean(s["value"] for s in steps)
    per_unit_flop = sum(w.flops()) / w.BH
    ms = per_unit_flop / (v * 1e12) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "kind": "oracle", "cores": steps[-1]["cores"],
                             "sample": f"1 of {w.BH} batch*head units of {w.name} per step (fwd+bwd)"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest per-rank value of x (the job takes as long as its slowest rank)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def config_of(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "seq_len": w.N, "head_dim": w.d, "causal": w.causal,
            "input_dtype": w.dtype, "l2": "flushed between timed steps (512 MiB write)"}


# ---------------------------------------------------------------------------- GPU arm

def kernel_flops(w, path):
    """Algorithmic FLOP per launch of each kernel, by the FLOP convention above.

    The backward's algorithmic count (2.5x the forward: the five N x N x d
    matmuls dS recomputation aside) is credited to the launch that forms the
    gradients.  Both kernel families execute more than that -- the dK/dV pass
    recomputes S and dP and forms dV and dK (four matmuls), the dQ pass
    recomputes S and dP again and forms dQ (three) -- so the tensor pipes run
    at 3.5/2.5 = 1.4x the achieved rate reported for fa_bwd_grads.
    """
    f = 4.0 * w.BH * w.N * w.N * w.d * (0.5 if w.causal else 1.0)   # two N x N x d matmuls
    return {"fwd": f, "bwd_pre": 0.0, "bwd_grads": 2.5 * f}


# matmul FLOP per launch that the kernels actually execute (recomputation included)
EXECUTED_FACTOR = {"fwd": 1.0, "bwd_pre": 0.0, "bwd_grads": 3.5 / 2.5}


# DRAM bytes (read + write) per launch of the dominant kernel, from one
# `ncu --set full` capture of the current kernels (profiles/fa_tc_kernels_*.md);
# None where no capture of the current build exists for that workload.
NCU_TRAFFIC = {
    ("bench_b8_n4096_d64_causal", "fwd"): 12625664,
    ("bench_b8_n4096_d64_causal", "bwd_grads"): 17095168,
    ("long_n16384_d128_causal", "fwd"): 12634624,
    ("long_n16384_d128_causal", "bwd_grads"): 16977664,
}


def run_gpu(args, w, rank, world):
    import torch

    from tiled_attention_04_gb300 import binding, build, inputs
    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.lib()
    tens = inputs.make_inputs(w)
    Qd, Kd, Vd, dOd = (inputs.to_torch(t, dev) for t in tens)
    host = [inputs.to_torch(t).pin_memory() for t in tens]
    O = torch.empty_like(Qd)
    L = torch.empty(Qd.shape[:-1], dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Qd), torch.empty_like(Kd), torch.empty_like(Vd)
    ws = binding.alloc_workspace(Qd, Kd, w.causal)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    path = binding.path_name(w.N, w.N, w.d, w.causal, binding.dtype_code(Qd))
    kf = kernel_flops(w, path)
    fwd_f, bwd_f = w.flops()

    def launch_step():   # forward + backward in one library call (fa_fwd_bwd: three kernels)
        binding.fa_fwd_bwd(Qd, Kd, Vd, dOd, is_causal=w.causal, O=O, L=L, dQ=dQ, dK=dK, dV=dV, workspace=ws)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        launch_step()
    torch.cuda.synchronize()
    if binding.fa_get_device_status() != binding.FA_OK:
        raise RuntimeError("device status not ok after warm-up")

    # timed region: one event pair per step, so that each kernel may be scheduled
    # onto SMs the previous one has vacated (programmatic dependent launch)
    evs = [(ev(), ev()) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for a, b in evs:
            flush.fill_(1.0)
            a.record(stream)
            launch_step()
            b.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total = [a.elapsed_time(b) for a, b in evs]
    step_ms = max_over_ranks(sum(total) / len(total), world, dev)

    # fwd / bwd split: the same steps with one more event, between fa_fwd and the
    # backward (preprocessing + gradients, still overlapped by dependent launch)
    nb = min(args.steps, 50)
    split = {"fwd": [], "bwd": []}
    sevs = [[ev() for _ in range(3)] for _ in range(nb)]
    for e in sevs:
        flush.fill_(1.0)
        e[0].record(stream)
        binding.fa_fwd(Qd, Kd, Vd, is_causal=w.causal, O=O, L=L)
        e[1].record(stream)
        binding.fa_bwd_preprocess(O, dOd, L, Qd, Kd, w.causal, ws)
        binding.fa_bwd_grads(Qd, Kd, Vd, dOd, L, dQ, dK, dV, w.causal, ws)
        e[2].record(stream)
    torch.cuda.synchronize()
    for e in sevs:
        split["fwd"].append(e[0].elapsed_time(e[1]))
        split["bwd"].append(e[1].elapsed_time(e[2]))

    # per-kernel durations (roofline of the dominant kernel): an event between every
    # two kernels, which serialises them
    names = ["fwd", "bwd_pre", "bwd_grads"]
    per = {n: [] for n in names}
    kevs = [[ev() for _ in range(4)] for _ in range(nb)]
    for e in kevs:
        flush.fill_(1.0)
        e[0].record(stream)
        binding.fa_fwd(Qd, Kd, Vd, is_causal=w.causal, O=O, L=L)
        e[1].record(stream)
        binding.fa_bwd_preprocess(O, dOd, L, Qd, Kd, w.causal, ws)
        e[2].record(stream)
        binding.fa_bwd_grads(Qd, Kd, Vd, dOd, L, dQ, dK, dV, w.causal, ws)
        e[3].record(stream)
    torch.cuda.synchronize()
    for e in kevs:
        for i, n in enumerate(names):
            per[n].append(e[i].elapsed_time(e[i + 1]))
    if binding.fa_get_device_status() != binding.FA_OK:
        raise RuntimeError("device status not ok after timed steps")

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs from pinned host memory, runs fa_fwd_bwd and copies O, L, dQ, dK,
    # dV back.  Three buffer sets, each step captured once as a CUDA graph and the
    # graphs replayed in turn on three streams, so the copies of two steps overlap the
    # kernels of a third (as a data loader would); per-step work is unchanged.  The
    # copy engines move about 190 GB/s each way from pinned memory here, so with the
    # short steps the copies, not the kernels, set this number; a third set hides
    # the copy-in of one step behind the copy-out of another (two sets left the
    # batch-8 step at 157 us against 130 us with three; a fourth adds nothing, and
    # splitting the copies over parallel graph branches was slower).
    def make_set():
        dev_in = [torch.empty_like(x) for x in (Qd, Kd, Vd, dOd)]
        o, l_ = torch.empty_like(O), torch.empty_like(L)
        g = [torch.empty_like(x) for x in (dQ, dK, dV)]
        outs = [o, l_, *g]
        return {"in": dev_in, "out": outs, "ws": binding.alloc_workspace(Qd, Kd, w.causal),
                "host_out": [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]}

    n_sets = 3
    sets = [make_set() for _ in range(n_sets)]
    h2d = sum(x.numel() * x.element_size() for x in host)
    d2h = sum(x.numel() * x.element_size() for x in sets[0]["host_out"])

    def e2e_step(st):
        q, k, v, g = st["in"]
        o, l_, dq, dk, dv = st["out"]
        for dst, src in zip(st["in"], host):
            dst.copy_(src, non_blocking=True)
        binding.fa_fwd_bwd(q, k, v, g, is_causal=w.causal, O=o, L=l_, dQ=dq, dK=dk, dV=dv, workspace=st["ws"])
        for dst, src in zip(st["host_out"], st["out"]):
            dst.copy_(src, non_blocking=True)

    streams = [torch.cuda.Stream() for _ in range(n_sets)]
    e2e_method = (f"{n_sets} CUDA graphs of (H2D inputs, fa_fwd_bwd, D2H outputs) replayed in turn on "
                  f"{n_sets} streams")
    graphs = []
    try:
        for st, sm in zip(sets, streams):
            sm.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(sm):
                for _ in range(2):
                    e2e_step(st)
            sm.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=sm):
                e2e_step(st)
            graphs.append(g)
    except Exception as exc:   # capture refused: the same steps issued eagerly on the streams
        graphs = []
        e2e_method = f"eager on {n_sets} streams in turn (graph capture failed: {type(exc).__name__})"
    torch.cuda.synchronize()

    def run_e2e(n):
        cur = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for sm in streams:
            sm.wait_stream(cur)
        for i in range(n):
            sm = streams[i % n_sets]
            with torch.cuda.stream(sm):
                if graphs:
                    graphs[i % n_sets].replay()
                else:
                    e2e_step(sets[i % n_sets])
        for sm in streams:
            cur.wait_stream(sm)
        b.record(cur)
        b.synchronize()
        return a.elapsed_time(b) / n

    run_e2e(max(4, args.warmup))
    n_e2e = max(4, min(args.steps, 100))
    e2e_ms = max_over_ranks(run_e2e(n_e2e), world, dev)
    if binding.fa_get_device_status() != binding.FA_OK:
        raise RuntimeError("device status not ok after the end-to-end steps")

    if rank != 0:
        return
    pk = peaks()
    avg = {n: sum(v) / len(v) for n, v in per.items()}
    dom = max(names, key=lambda n: avg[n])
    dom_tf = kf[dom] / (avg[dom] * 1e-3) / 1e12
    value = world * (fwd_f + bwd_f) / (step_ms * 1e-3) / 1e12
    fwd_ms = sum(split["fwd"]) / nb
    bwd_ms = sum(split["bwd"]) / nb
    fwd_tf = fwd_f / (fwd_ms * 1e-3) / 1e12
    bwd_tf = bwd_f / (bwd_ms * 1e-3) / 1e12
    launches_per_step = 3 if path == "tc" else 4
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w),
        "frac_of_peak": round(value / world / pk["bf16_tflops"], 4),
        "fwd": {"ms": round(fwd_ms, 5), "tflops": round(fwd_tf, 2), "frac": round(fwd_tf / pk["bf16_tflops"], 4)},
        "bwd": {"ms": round(bwd_ms, 5), "tflops": round(bwd_tf, 2), "frac": round(bwd_tf / pk["bf16_tflops"], 4),
                "kernels_ms": {n: round(avg[n], 5) for n in names[1:]}},
        "breakdown": f"fwd and bwd from {nb} further steps with an event between fa_fwd and the backward; "
                     "kernels_ms and the roofline from another pass with an event between every two kernels",
        "path": path,
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(dom_tf, 2), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(dom_tf / pk["bf16_tflops"], 4),
                     "traffic": NCU_TRAFFIC.get((w.name, dom)),
                     "executed_tflops": round(dom_tf * EXECUTED_FACTOR[dom], 2),
                     "peak_source": f"{pk['source']} bf16 dense burst"},
        "e2e": {"value": round(world * (fwd_f + bwd_f) / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": n_e2e, "method": e2e_method,
                "l2": "not flushed: each step's inputs are rewritten by its own host-to-device copy"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = oracle_sample(w, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from tiled_attention_04_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, w, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
