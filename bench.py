#!/usr/bin/env python3
"""Throughput of the S_up (FO) calibration pass for one layer.

A step is one affinity_up(FO) call over one batch of T synthetic tokens of a
Qwen3-0.6B-shaped layer (by default): fp16 operand staging, the fold of
W_o^(h) diag(gamma) [W_g | W_u], the operating-point + per-head tensor-core
kernel, and the deterministic reductions.  Inputs are resident in HBM when
the timed region starts; they are larger than L2 (402 MB of a and x per
step), so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle on a token sample

Under torchrun (N > 1) every rank processes its own token batch (weak
scaling, no collective in the timed region); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "calibration tokens/sec for S^up fo affinity per layer; % of GB300 bf16 tensor peak"


def fo_flops(s) -> dict:
    """Algorithmic flops (multiply-add = 2) of the S_up FO pass."""
    fold = 2 * 2 * s.I * s.D * s.H * s.dh            # [Wg;Wu] diag(gamma) Wo^(h): (2I x D)(D x H dh)
    gate_up = 2 * s.T * s.D * 2 * s.I                  # (gamma x / r) [Wg;Wu]^T
    heads = 2 * s.T * s.H * s.dh * 2 * s.I             # a_h M_h for gate and up
    return {"fold": fold, "gate_up": gate_up, "heads": heads, "total": fold + gate_up + heads,
            "tile_kernel": gate_up + heads}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the FO tile kernel, from an ncu capture of this bench's workload; valid only
# while the kernel sources hash to the recorded value (otherwise null).
KERNEL_SOURCES = ("tile_kernel.cu", "tile_kernel.cuh", "sm103_primitives.cuh", "scales.cuh", "launch.cuh")
MOMENT_SOURCES = ("moment_kernel.cu", "moment_kernel.cuh", "sm103_primitives.cuh", "scales.cuh", "launch.cuh")
TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (1 pass), third FO launch of
    # `python bench.py --steps 2 --warmup 3 --no-cpu-baseline --e2e-steps 0`: 460.04 + 50.02 MB
    ("qwen3_0p6b_layer", "fo", 65536): {"bytes": 510.06e6, "src": "4a7405103e25fb79"},
}


def moment_launches(shape) -> int:
    """Kernels of one ADD call in the second-moment form: 1/r, the weight staging and
    restaging, the Gram pass, its reduction and fallback, the quadratic forms, the finish,
    and the fold -- two launches when some of its units run before the Gram pass (those
    past its last whole round of one unit per SM, or AFFINITY_FOLD_EARLY of them)."""
    import torch
    i_pad = -(-shape.I // 256) * 256
    units = 2 * (i_pad // 128) * -(-(shape.H * shape.dh) // 256)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    early = int(os.environ.get("AFFINITY_FOLD_EARLY", "-1"))
    if early < 0:
        early = units % sms if units > sms else 0
    return 9 if min(early, units) in (0, units) else 10


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "transformer_sharding_affinity_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, mode: str, T: int):
    rec = TRAFFIC.get((workload, mode, T))
    if rec is None or rec["src"] != kernel_source_hash(MOMENT_SOURCES if mode == "add" else KERNEL_SOURCES):
        return None
    return rec["bytes"]


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class _Nvml:
    """The few read-only NVML queries the clock record needs, through ctypes
    (no Python NVML package on the GPU host).  Reads clocks, power and the
    clock-event reasons; changes no setting."""
    SM = 1   # NVML_CLOCK_SM
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, cuda_index: int):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        ok = False
        try:   # the CUDA device by UUID (CUDA and NVML may number devices differently)
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(cuda_index).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(lib.nvmlDeviceGetMaxClockInfo, self.SM)

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        if fn(self.dev, *args, self.c.byref(v)) != 0:
            return None
        return v.value

    def sample(self):
        r = self.c.c_ulonglong()
        self.reasons_fn(self.dev, self.c.byref(r))
        return (self._uint(self.lib.nvmlDeviceGetClockInfo, self.SM),
                [n for bit, n in self.REASONS.items() if r.value & bit],
                self._uint(self.lib.nvmlDeviceGetPowerUsage))


class ClockSampler:
    """SM clock, power and throttle reasons sampled while the timed region runs:
    NVML polled every millisecond or so (the default timed region lasts tens of
    milliseconds), else nvidia-smi every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_s: float = 0.001):
        self.gpu = gpu_index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.lines = []
        self.samples = []      # (sm_mhz, reasons, power_mw) from NVML
        self.stop = threading.Event()

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.gpu)
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        except Exception:
            self.nvml = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _poll(self):
        while not self.stop.is_set():
            self.samples.append(self.nvml.sample())
            time.sleep(self.period)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml is not None:
            self.t.join(timeout=5)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.nvml is not None:
            sm = [c for c, _, _ in self.samples if c is not None]
            reasons = sorted({n for _, rs, _ in self.samples for n in rs})
            pw = [p for _, _, p in self.samples if p is not None]
            return {"sm_mhz": float(np.median(sm)) if sm else None,
                    "sm_mhz_min": float(min(sm)) if sm else None, "sm_max_mhz": self.nvml.max_mhz,
                    "reasons": reasons, "samples": len(sm),
                    "power_w_max": max(pw) / 1e3 if pw else None, "source": "NVML"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


def cpu_oracle_rate(shape, layer, budget_s: float = 10.0, max_tokens: int | None = None) -> dict:
    """Time the fp64 oracle (as it stands) on the first tokens of the same layer."""
    from oracle import affinity_oracle as O
    cores = len(os.sched_getaffinity(0))

    def run(n):
        t0 = time.perf_counter()
        O.s_up(layer["a"][:n], layer["x"][:n], layer["Wo"], layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"],
               shape.H, shape.G, shape.dh, shape.eps, "fo")
        return time.perf_counter() - t0

    n0 = 32
    t_probe = run(n0)
    n = int(max(n0, min(shape.T, n0 * budget_s / max(t_probe, 1e-6))))
    if max_tokens:
        n = min(n, max_tokens)
    t = run(n)
    return {"value": n / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle, FO S_up over all {shape.I} neurons for the first {n} of {shape.T} tokens "
                      f"({t:.1f} s wall, numpy BLAS threads over {cores} host cores)"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args) -> None:
    from transformer_sharding_affinity_gb300 import workloads as W
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    shape = W.CONFIGS[args.workload]
    sample = W.make_layer(shape.scaled(T=max(64, args.ref_tokens)))
    tok = sample["a"].shape[0]
    from oracle import affinity_oracle as O
    for _ in range(args.warmup):
        O.s_up(sample["a"][:8], sample["x"][:8], sample["Wo"], sample["gamma"], sample["Wg"], sample["Wu"],
               sample["Wd"], shape.H, shape.G, shape.dh, shape.eps, "fo")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.s_up(sample["a"], sample["x"], sample["Wo"], sample["gamma"], sample["Wg"], sample["Wu"], sample["Wd"],
               shape.H, shape.G, shape.dh, shape.eps, "fo")
    dt = time.perf_counter() - t0
    v = tok * args.steps / dt
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "T": shape.T, "D": shape.D, "H": shape.H, "G": shape.G,
                       "d_head": shape.dh, "I": shape.I, "mode": "fo"},
            "tokens_per_step": tok,
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: fp64 oracle FO S_up over all {shape.I} neurons for {tok} tokens "
                                       f"of the {args.workload} workload"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_layout(args) -> None:
    """Layout search on a 28-layer Qwen3-shaped stack of seeded unit-mass
    affinity matrices: the GPU neuron step for all layers in one launch
    (CUDA events) and the whole alternating search from the contiguous layout
    (wall clock, including the host head steps)."""
    import torch
    from transformer_sharding_affinity_gb300 import binding as B
    from transformer_sharding_affinity_gb300 import stack as ST
    from transformer_sharding_affinity_gb300 import workloads as W

    B.load()
    shape = W.CONFIGS["qwen3_0p6b_stack"]
    N, G, I, L = W.STACK_LAYERS, shape.G, shape.I, 4
    rng = np.random.Generator(np.random.PCG64(shape.seed))
    S_up = [rng.gamma(0.5, size=(G, I)).astype(np.float32) for _ in range(N)]
    S_dn = [rng.gamma(0.5, size=(I, G)).astype(np.float32) for _ in range(N - 1)]
    up = [B.unit_mass(s) for s in S_up]
    dn = [B.unit_mass(s) for s in S_dn]
    hc = np.stack([ST.contiguous_map(G, L)] * N)
    # neuron step of every layer at once on M built by the gain kernel
    d_up = torch.from_numpy(np.stack(up)).cuda()
    d_dn = torch.from_numpy(np.stack(dn)).cuda()
    M = torch.empty(N, I, L, dtype=torch.float64, device="cuda")
    nu = torch.empty(N, I, dtype=torch.int32, device="cuda")
    val = torch.empty(N, dtype=torch.float64, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")

    def neuron_step():
        for i in range(N):
            B.neuron_gain(d_up[i], d_dn[i] if i + 1 < N else None, hc[i], hc[i + 1] if i + 1 < N else None, L, M[i])
        B.assign_neurons(M, L, nu, val, ws)

    for _ in range(args.warmup):
        neuron_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        neuron_step()
    e1.record()
    torch.cuda.synchronize()
    step_ms = e0.elapsed_time(e1) / args.steps
    st = B.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}: {B.strerror(st)}")
    ST.optimise(up, dn, L)    # warm
    t0 = time.perf_counter()
    res = ST.optimise(up, dn, L)
    # the paper's run also scores eight random balanced layouts (seeds 1000..1007)
    J_random = []
    for seed in range(1000, 1008):
        r = np.random.default_rng(seed)
        J_random.append(B.objective(up, dn, [r.permutation(ST.contiguous_map(G, L)) for _ in range(N)],
                                    [r.permutation(ST.contiguous_map(I, L)) for _ in range(N)]))
    opt_s = time.perf_counter() - t0
    J0 = B.objective(up, dn, hc, np.stack([ST.contiguous_map(I, L)] * N))
    line = {"metric": "layout search: balanced neuron step for every layer of a 28-layer stack",
            "value": N / (step_ms * 1e-3), "unit": "layers/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "none",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "qwen3_0p6b_stack unit-mass affinities (gamma(0.5) draws)", "N": N, "G": G,
                       "I": I, "L": L},
            "roofline": {"bound": "latency", "note": "one 1024-thread CTA per layer; M (I*L*8 B) re-read "
                                                     "from L1 on every dual-ascent iteration"},
            "optimise": {"seconds": opt_s, "sweeps": res.sweeps, "J_contiguous": J0, "J": res.J,
                         "J_random_mean": float(np.mean(J_random)),
                         "note": "seconds include scoring eight random layouts"},
            "gpu_launches": N + 1}
    if not args.no_cpu_baseline:
        from oracle import assignment as A
        M0 = A.neuron_gain(up[0], hc[0], L, dn[0], hc[1])
        t0 = time.perf_counter()
        A.best_balanced_neurons(M0)
        t = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": "layers/s", "cores": 1, "kind": "oracle",
                                "sample": f"scipy linear_sum_assignment on the {I}x{I} replicated-slot matrix of "
                                          f"layer 0 ({t:.2f} s)"}
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_0p6b_layer")
    ap.add_argument("--mode", default="fo", choices=["fo", "add", "loo", "down"])
    ap.add_argument("--add-form", default="moment", choices=["moment", "direct"],
                    help="ADD through each head's second moment (d_head <= 128) or the direct contraction")
    ap.add_argument("--e2e-steps", type=int, default=200,
                    help="at least this many end-to-end steps (0: skip); more when --min-load-s asks for it")
    ap.add_argument("--min-load-s", type=float, default=5.0,
                    help="run the end-to-end loop for about this long, so that a clock sampler polling "
                         "every few hundred ms sees the GPU under load many times")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling runs on a smaller case)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step in a CUDA graph and time its replays")
    ap.add_argument("--path", default="scores", choices=["scores", "layout"],
                    help="scores: the S_up calibration pass (default); layout: the layout search")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        run_reference(args)
        return
    if args.path == "layout":
        run_layout(args)
        return

    import torch
    from transformer_sharding_affinity_gb300 import binding as B
    from transformer_sharding_affinity_gb300 import device as DV
    from transformer_sharding_affinity_gb300 import workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    B.load()

    base = W.CONFIGS[args.workload]
    if args.tokens:
        base = base.scaled(T=args.tokens)
    shape = base.scaled(seed=base.seed + 1000 * rank)     # each rank: its own token batch
    down = args.mode == "down"
    keys = DV.DOWN_KEYS if down else DV.UP_KEYS
    layer = W.make_layer(shape, with_next=down)
    host = {k: DV.host_tensor(layer, k, shape.dtype).pin_memory() for k in keys}
    dev = {k: v.to("cuda") for k, v in host.items()}
    moment = args.mode == "add" and args.add_form == "moment" and shape.dh <= 128
    direct_add = args.mode == "add" and not moment
    d = B.dims(shape.T, shape.D, shape.H, shape.G, shape.dh, shape.I, shape.eps,
               flags=B.AFF_FLAG_ADD_DIRECT if direct_add else 0)
    mode = 0 if down else B.MODES[args.mode]
    work = torch.empty(B.workspace_size(d, mode, down=down), dtype=torch.uint8, device="cuda")
    S = torch.empty((shape.I, shape.G) if down else (shape.G, shape.I), device="cuda")
    stream = torch.cuda.current_stream()

    def call(t):
        if down:
            B.affinity_down(t["x"], t["gamma"], t["Wg"], t["Wu"], t["Wd"], t["gamma_next"], t["Wq_next"],
                            t["Wk_next"], t["Wv_next"], d, S, work, stream)
        else:
            B.affinity_up(t["a"], t["x"], t["Wo"], t["gamma"], t["Wg"], t["Wu"], t["Wd"], d, mode, S, None, work,
                          stream)

    ev_k0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_k1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in ev_k0 + ev_k1:
        e.record()
    torch.cuda.synchronize()

    def step(i=None, bufs=dev):
        if i is not None:
            B.set_timing_events(ev_k0[i], ev_k1[i])
        call(bufs)
        if i is not None:
            B.set_timing_events(None, None)

    for _ in range(args.warmup):
        step()
    st = B.device_status(work)
    if st != 0:
        raise RuntimeError(f"device status {st}: {B.strerror(st)}")
    graph = None
    kern_direct = []
    if args.graph:
        # the dominant kernel's time comes from direct calls (events recorded inside a
        # graph are not timing events); the timed loop then replays one captured step
        for i in range(min(args.steps, 20)):
            step(i)
        torch.cuda.synchronize()
        kern_direct = [ev_k0[i].elapsed_time(ev_k1[i]) for i in range(min(args.steps, 20))]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            stream = torch.cuda.current_stream()
            call(dev)
        stream = torch.cuda.current_stream()
        for _ in range(args.warmup):
            graph.replay()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0.record()
        for i in range(args.steps):
            if graph is None:
                step(i)
            else:
                graph.replay()
        t1.record()
        torch.cuda.synchronize()

    if ws > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    kern_ms = float(np.mean(kern_direct if graph is not None else
                            [a.elapsed_time(b) for a, b in zip(ev_k0, ev_k1)]))
    st = B.device_status(work)
    if st != 0:
        raise RuntimeError(f"device status {st}: {B.strerror(st)}")
    if ws > 1:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / args.steps

    # End to end: every step copies all of its inputs from pinned host memory,
    # calls affinity_up and reads S back to pinned host memory.  Two input
    # buffer sets let the copy of step i+1 (on a copy stream) overlap the
    # compute of step i; a buffer set is refilled only after the step that
    # read it has finished.
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    S_host = torch.empty(tuple(S.shape), pin_memory=True)
    bufs = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = 0
    if args.e2e_steps > 0:
        # an end-to-end step takes ~1.1-1.2x the device step
        n_e2e = max(args.e2e_steps, min(100000, int(math.ceil(args.min_load_s * 1e3 / (1.15 * ms_step)))))
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks_e2e:
        e0.record(stream)
        copy_stream.wait_stream(stream)
        for i in range(n_e2e):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(free[j])
                for k in keys:
                    bufs[j][k].copy_(host[k], non_blocking=True)
                ready[j].record(copy_stream)
            stream.wait_event(ready[j])
            step(bufs=bufs[j])
            free[j].record(stream)
            S_host.copy_(S, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e if n_e2e > 0 else float("nan")

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    pk = peaks()
    fl = fo_flops(shape)
    heads = 2 * shape.T * shape.H * shape.dh * 2 * shape.I
    if args.mode == "fo":
        flops_per_step, tile_flops = fl["total"], fl["tile_kernel"]
    elif moment:   # fold, C_h = sum_t a~ a~^T, then m^T C_h m (hi and lo halves of C_h)
        tile_flops = 2 * shape.T * shape.H * shape.dh ** 2
        flops_per_step = fl["fold"] + tile_flops + 2 * 2 * 2 * shape.I * shape.H * shape.dh ** 2
    elif args.mode == "add":
        flops_per_step, tile_flops = fl["fold"] + heads, heads
    elif args.mode == "loo":   # the FO-shaped pass plus c_h / r = (a_h / r) Wo^(h)^T for the rms of x - c_h
        flops_per_step = fl["total"] + 2 * shape.T * shape.H * shape.dh * shape.D
        tile_flops = fl["tile_kernel"]
    else:   # down: gate/up GEMM for alpha, x' = x + alpha Wd^T, ||W^qkv_g (gamma' * w^d_k)||^2 (hi + lo)
        tile_flops = fl["gate_up"]
        flops_per_step = tile_flops + 2 * shape.T * shape.I * shape.D + \
            2 * 2 * (shape.H + 2 * shape.G) * shape.dh * shape.D * shape.I
    achieved = tile_flops / (kern_ms * 1e-3) / 1e12
    tokens = shape.T * ws
    if moment:
        # the Gram pass reads every token's a~ once (fp16): HBM-bound
        gram_bytes = shape.T * shape.H * shape.dh * 2
        gbs = gram_bytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "moment_kernel<GRAM> (C_h = sum_t a~_t a~_t^T, tcgen05)",
                "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                "peak_source": pk["source"] + " HBM copy bandwidth", "kernel_ms": kern_ms,
                "algorithmic_bytes_per_launch": gram_bytes, "algorithmic_flops_per_launch": tile_flops,
                "traffic": measured_traffic(args.workload, args.mode, shape.T)}
    else:
        roof = {"bound": "tensor",
                "kernel": ("affinity_tile_kernel<ALPHA> (gate/up GEMM, alpha = silu(g) u)" if down else
                           f"affinity_tile_kernel<{args.mode.upper()}> (operating point + per-head contraction)"),
                "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                "frac_sustained": achieved / pk["bf16_tflops_sustained"] if pk["bf16_tflops_sustained"] else None,
                "peak_source": pk["source"] + " bf16 dense (fp16 runs at the bf16 rate)",
                "kernel_ms": kern_ms, "algorithmic_flops_per_launch": tile_flops,
                "traffic": measured_traffic(args.workload, "add_direct" if direct_add else args.mode, shape.T)}
    line = {
        "metric": METRIC, "value": tokens / (ms_step * 1e-3), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16 operands, fp32 accumulate (bf16 inputs)",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": shape.T, "D": shape.D, "H": shape.H, "G": shape.G,
                   "d_head": shape.dh, "I": shape.I, "mode": args.mode,
                   **({"add_form": "moment" if moment else "direct"} if args.mode == "add" else {}),
                   "parallelism": f"dp{ws} (token shards)",
                   "launch": "CUDA graph replay of one step" if graph is not None else "direct calls",
                   "l2": "inputs larger than L2 (a + x = %.0f MB per step); no flush" %
                         ((shape.T * (shape.H * shape.dh + shape.D) * 2) / 2**20)},
        "step_flops": flops_per_step,
        "step_tflops": flops_per_step / (ms_step * 1e-3) / 1e12,
        "step_frac_of_peak": flops_per_step / (ms_step * 1e-3) / 1e12 / pk["bf16_tflops"],
        "roofline": roof,
        "gpu_launches": (moment_launches(shape) if moment else
                         {"fo": 8, "add": 7, "loo": 10, "down": 10}[args.mode]) * args.steps,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": shape.G * shape.I * 4, "ms_per_step": e2e_ms, "steps": n_e2e,
                "clocks": clocks_e2e.summary()},
        "clocks": clocks.summary(),
    }
    if down:
        line["metric"] = "calibration tokens/sec for S^down affinity per layer; % of GB300 bf16 tensor peak"
    if not args.no_cpu_baseline and ws == 1 and not down:
        line["cpu_baseline"] = cpu_oracle_rate(shape, layer, args.cpu_budget)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
