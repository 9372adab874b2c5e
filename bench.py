"""Benchmark of the W4A16 GEMM on GB300: one JSON line on rank 0.

Default workload (the metric's headline configuration): the Llama-3-8B decode
linear layers -- qkv (4096x6144), o_proj (4096x4096), gate_up (4096x28672),
down (14336x4096) -- at M in {1, 8, 16, 32}, g = 128.  One step = those 16
GEMMs, each with its own packed weights, X and Y (453 MB of distinct packed
weights per step, more than the 129 MB L2, so every step streams its weights
from HBM).  A step is captured once as a CUDA graph and replayed.

  value     = algorithmic bytes of the step / device time per step (GB/s),
              summed over all ranks (replicas) for --gpus N.
  roofline  = the decode kernel against the measured HBM copy bandwidth.
  e2e       = the same metric end to end: per step every X copied in from
              pinned host memory, the GEMMs through the public call, every Y
              copied back to pinned host memory, one synchronisation.
  cpu_baseline = the fp64 oracle on a bounded column sample of the same
              workload, extrapolated to the full step, on the host cores.

  detail    = every configuration of the metric (workloads 0-4: the 1x4096x4096
              GEMM, the 8B decode and prefill shapes, the 70B shapes, the
              group-size/outlier stress shapes), each GEMM in steady state
              with its own roofline; the 8B layer linears per M and for
              M <= 16 together; the prefill step (TFLOP/s against the burst
              tensor peak).  --no-detail skips it.

--workload prefill runs the Llama-3-8B prefill shapes (M in {128,1024,4096},
TFLOP/s of the tensor-memory kernel against the measured tensor peak) instead.
--impl reference times the oracle as the reference arm: the whole workload per
step when the run fits its time budget, else a labelled column sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM GB/s (M≤32) & TFLOP/s (M≥128), % of roofline, Llama-3 shapes"
WORKLOADS = {
    "decode": {"idx": 1, "unit": "GB/s", "bound": "hbm",
               "name": "llama3-8b decode linears: qkv/o_proj/gate_up/down x M in {1,8,16,32}, g=128"},
    "prefill": {"idx": 2, "unit": "TFLOP/s", "bound": "tensor",
                "name": "llama3-8b prefill linears: qkv/o_proj/gate_up/down x M in {128,1024,4096}, g=128"},
}
KERNEL_SOURCES = {"decode": ["decode.cu", "tm_common.cuh"], "tc": ["tc.cu", "tm_common.cuh"],
                  "kv": ["kv.cu", "tm_common.cuh"], "w8": ["w8a8.cu", "tm_common.cuh"],
                  "rtn": ["quant.cu", "tm_common.cuh"]}


# ----------------------------------------------------------------- helpers ---

def algorithmic_bytes(M, K, N, g):
    G = K // g
    return K * N // 2 + G * N * 2 + G * N // 2 + 2 * M * K + 2 * M * N


def flops(M, K, N):
    return 2 * M * N * K


def rtn_bytes(K, N, g):
    """RTN quantisation: read fp16 W; write one code and, per (group, column), one
    zero byte and one fp16 scale."""
    G = K // g
    return 2 * K * N + K * N + G * N + 2 * G * N


def kv_cache_bytes(B, L, Hkv, D, bits):
    """K and V of B sequences of L tokens: codes plus an fp16 scale and a uint8
    zero per (token, head)."""
    return 2 * B * L * Hkv * (D * bits // 8 + 3)


def w8a8_bytes(M, K, N):
    """One W8A8 layer: the quantiser reads fp16 X and writes int8 X and s_x; the
    GEMM reads the int8 weights, their fp32 scales, int8 X and s_x, writes fp16 Y."""
    return (2 * M * K + M * K + 4 * M) + (K * N + 4 * N + M * K + 4 * M + 2 * M * N)


def workload_config(kind, world=1):
    """The `config` object both arms print: the workload and its sizes only."""
    from w4a16_quantized_gemm_gb300 import synth
    cases = synth.workload(WORKLOADS[kind]["idx"])
    return {"workload": WORKLOADS[kind]["name"], "gemms_per_step": len(cases),
            "bytes_per_step": sum(algorithmic_bytes(c.M, c.K, c.N, c.g) for c in cases),
            "flops_per_step": sum(flops(c.M, c.K, c.N) for c in cases),
            "l2": "inputs larger than L2: every GEMM of a step has its own weights (>129 MB per step)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def roofline_entry(nbytes, nflops, seconds, peaks, tensor_peak="bf16_tflops"):
    """Roofline of one timed unit: the bound is whichever of bytes / HBM and
    flops / tensor peak takes longer; achieved is that quantity per second."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = nflops / (peaks[tensor_peak] * 1e12)
    if t_hbm >= t_tc:
        ach, peak, unit, bound = nbytes / seconds / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
    else:
        ach, peak, unit, bound = nflops / seconds / 1e12, peaks[tensor_peak], "TFLOP/s", "tensor"
    return {"bound": bound, "achieved": round(ach, 1), "peak": peak, "unit": unit, "frac": round(ach / peak, 4),
            "peak_source": peaks["source"] + (" (sustained)" if tensor_peak.endswith("sustained") else "")}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "of measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "of fallback"}


def kernel_hash(kind):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "w4a16_quantized_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(kind, workload):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    or None when there is none or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kind}_kernel_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    d = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                d[k.strip()] = v.strip()
    if d.get("kernel_source_sha") != kernel_hash(kind):
        return None
    try:
        return float(d["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value, world):
    """Max over ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units, world, t_max_s):
    """Whole-job throughput: units every rank processed / slowest rank's time."""
    return per_rank_units * world / t_max_s


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- GPU arm ---

class Workload:
    def __init__(self, kind, device, copies=1):
        import numpy as np
        import torch

        from w4a16_quantized_gemm_gb300 import binding, synth

        self.kind = kind
        self.cases = synth.workload(WORKLOADS[kind]["idx"])
        self.items = []
        weights_cache = {}
        for c in self.cases:
            key = (c.K, c.N, c.g)
            if key not in weights_cache:
                weights_cache[key] = synth.weights(c.K, c.N, c.g)
            q, z, s, _ = weights_cache[key]
            qd = torch.from_numpy(q).to(device)
            zd = torch.from_numpy(z).to(device)
            sd = torch.from_numpy(s.view(np.uint16)).to(device).view(torch.float16)
            w = binding.pack(qd, zd, sd, c.g)
            del qd, zd, sd
            Xh = synth.activations(c.M, c.K, None, 0, tag=f"/N{c.N}/g{c.g}")
            X = torch.from_numpy(Xh.view(np.uint16)).to(device).view(torch.float16)
            Y = torch.empty((c.M, c.N), dtype=torch.float16, device=device)
            self.items.append({"case": c, "w": w, "X": X, "Y": Y, "Xh": Xh,
                               "bytes": algorithmic_bytes(c.M, c.K, c.N, c.g), "flops": flops(c.M, c.K, c.N),
                               "plan": binding.plan(w, c.M)})
        self.step_bytes = sum(i["bytes"] for i in self.items)
        self.step_flops = sum(i["flops"] for i in self.items)
        self.weight_bytes = sum(i["w"].nbytes for i in self.items)

    def runs(self):
        """The step's products as launches: consecutive products with the same
        M <= 32 (the four linears of a layer at one batch size) share one
        grouped launch; every other product is a launch of its own."""
        from w4a16_quantized_gemm_gb300 import binding
        out = []
        for it in self.items:
            M = it["case"].M
            last = out[-1] if out else None
            if (last and M <= 32 and last[0]["case"].M == M and last[0]["case"].g == it["case"].g
                    and len(last) < binding.GROUP_MAX):
                last.append(it)
            else:
                out.append([it])
        return out

    def launch_all(self, stream, grouped=True, concurrent=True):
        """One step: the grouped launches of runs() (grouped=False: every
        product launched on its own), on two streams (concurrent): the step's
        products are independent, so one launch's start-up and tail overlap
        another's.  Decode: the runs by M, largest with smallest -- M = 32 and
        1 on the launching stream, 16 and 8 on the second.  Prefill: the
        products under 60 GFLOP (every M = 128 one, qkv and o_proj at
        M = 1024: bound by their weight stream or a badly filled wave) on the
        second stream, the others largest first on the launching one.  The
        second stream joins the first before the step ends.  Returns the
        number of kernel launches."""
        import torch

        from w4a16_quantized_gemm_gb300 import binding
        runs = self.runs() if grouped else [[it] for it in self.items]
        main, side = split_lanes(runs, self.kind) if concurrent else (runs, [])
        if side:
            if not hasattr(self, "_side"):
                self._side = torch.cuda.Stream(stream.device)
            start = torch.cuda.Event()
            start.record(stream)
            self._side.wait_event(start)
        n = 0
        for st, group in ((stream, main), (getattr(self, "_side", None), side)):
            for run in group:
                if len(run) > 1:
                    binding.gemm_grouped([(it["X"], it["w"], it["Y"], False) for it in run], stream=st)
                else:
                    binding.gemm(run[0]["X"], run[0]["w"], out=run[0]["Y"], stream=st)
                n += binding.last_launch_count()
        if side:
            done = torch.cuda.Event()
            done.record(self._side)
            stream.wait_event(done)
        return n


def split_lanes(runs, kind):
    """The two streams of a step's launches (launching stream, second stream).
    Decode: the runs by M, the j-th largest with the j-th smallest on lane j % 2
    (M = 32 and 1 on the launching stream, 16 and 8 on the second).  Prefill:
    the products under 60 GFLOP on the second stream, the others largest
    first on the launching one.  Anything else: one stream."""
    if kind == "decode" and len(runs) > 1:
        order = sorted(range(len(runs)), key=lambda i: -runs[i][0]["case"].M)
        lanes = [[], []]
        for j in range((len(order) + 1) // 2):
            ids = [order[j]] + ([order[-1 - j]] if len(order) - 1 - j != j else [])
            lanes[j % 2].extend(runs[i] for i in ids)
        return lanes[0], lanes[1]
    if kind == "prefill":
        small = [flops(r[0]["case"].M, r[0]["case"].K, r[0]["case"].N) < 60e9 for r in runs]
        return [r for r, f in zip(runs, small) if not f][::-1], [r for r, f in zip(runs, small) if f]
    return runs, []


def run_gpu(args, rank, world, local):
    import torch

    from w4a16_quantized_gemm_gb300 import binding

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    wl = Workload(args.workload, device)
    spec = WORKLOADS[args.workload]
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()

    # capture one step as a graph
    with torch.cuda.stream(stream):
        wl.launch_all(stream)  # warm the kernels (attributes, module load) before capture
    stream.synchronize()
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=stream):
        launches_per_step = wl.launch_all(torch.cuda.current_stream())


    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_plain.replay()
    stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    t_sampler0 = time.time()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for k in range(args.steps):
            g_plain.replay()
            evs[k + 1].record(stream)
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = [evs[k].elapsed_time(evs[k + 1]) for k in range(args.steps)]
    t_total_ms = evs[0].elapsed_time(evs[-1])
    # keep the same load running until the sampler has seen >= 1.5 s of it
    extra = 0
    with torch.cuda.stream(stream):
        while time.time() - t_sampler0 < 1.5:
            for _ in range(200):
                g_plain.replay()
                extra += 1
            stream.synchronize()
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = f"timed region + {extra} untimed steps of the same workload"

    t_max_s = reduce_max(t_total_ms / 1e3, world)

    step_s = statistics.mean(step_ms) * 1e-3
    # Every configuration of the metric, each GEMM in steady state and the
    # step-level figures (not the headline value; see config_detail).
    detail = [] if args.no_detail else config_detail(wl, stream, peaks, args)

    if spec["unit"] == "GB/s":
        per_rank_units = wl.step_bytes * args.steps / 1e9
        achieved = wl.step_bytes / step_s / 1e9
        peak = peaks["hbm_gbs"]
        traffic = read_traffic("decode", "llama3_8b_decode")
        unit_kernel = "GB/s"
    else:
        per_rank_units = wl.step_flops * args.steps / 1e12
        achieved = wl.step_flops / step_s / 1e12
        peak = peaks["bf16_tflops"]  # a ms-scale step: the burst peak
        traffic = read_traffic("tc", "llama3_8b_prefill")
        unit_kernel = "TFLOP/s"
    value = aggregate(per_rank_units, world, t_max_s)

    e2e = run_e2e(wl, args, spec) if rank == 0 else None
    cpu = cpu_baseline(wl, args.cpu_seconds) if (rank == 0 and world == 1 and not args.no_cpu) else None

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": spec["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max_s * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(args.workload, world),
        "launch": f"one CUDA graph per step ({launches_per_step} kernel nodes for {len(wl.items)} products, "
                  f"programmatic dependent launch"
                  + ("; the products of one M (a layer's four linears, independent inputs) share one grouped "
                     "launch, tm_w4a16_gemm_grouped" if launches_per_step < len(wl.items) else "")
                  + ("; the launches on two streams (independent products): M = 32 and 1 on the launching "
                     "stream, 16 and 8 on a second, joined before the step ends" if wl.kind == "decode" else "")
                  + ("; the products under 60 GFLOP (M = 128, qkv and o_proj at M = 1024) on a second stream "
                     "beside the others, joined before the step ends" if wl.kind == "prefill" else "")
                  + f"); {wl.weight_bytes} bytes of distinct packed weights per step; fp32 accumulation",
        "roofline": {"bound": spec["bound"], "achieved": round(achieved, 2), "peak": peak,
                     "unit": unit_kernel, "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": peaks["source"],
                     "kernel": "decode_kernel" if spec["bound"] == "hbm" else "tc_kernel",
                     "basis": "algorithmic units of the step's launches / mean step time of the timed "
                              "region (CUDA events around each graph replay, the step's streams joined "
                              "before its closing event); the launches overlap (programmatic dependent "
                              "launch, and two streams where the step uses them), so the step time stands "
                              "for their combined duration",
                     "launches_per_step": launches_per_step},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "detail": detail,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def _time_graph(launch, stream, reps):
    """Capture ``launch(stream)`` as one CUDA graph, replay it once untimed,
    then ``reps`` times between CUDA events on ``stream``: ms per replay."""
    import torch
    with torch.cuda.stream(stream):
        launch(stream)  # outside capture: attributes, module load
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        launch(torch.cuda.current_stream())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del g
    return ms


def _pack_copies(key, device, min_bytes):
    """Distinct packed copies of one synthetic weight (q, z, s of the case's
    recipe) until together they exceed ``min_bytes`` (> L2)."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth
    K, N, g, stress = key
    q, z, s, sal = synth.weights(K, N, g, stress)
    qd = torch.from_numpy(q).to(device)
    zd = torch.from_numpy(z).to(device)
    sd = torch.from_numpy(s.view(np.uint16)).to(device).view(torch.float16)
    copies = [binding.pack(qd, zd, sd, g)]
    while len(copies) * copies[0].nbytes < min_bytes:
        copies.append(binding.pack(qd, zd, sd, g))
    del qd, zd, sd
    return copies, sal


def _decode_step_at_m(wl, M, stream, peaks, rounds=3, grouped=False):
    """The four Llama-3-8B layers of the headline workload at one M (qkv,
    o_proj, gate_up, down: one decoder layer's linears at batch M), on
    `rounds` distinct copies of their weights (> L2 together): launched one by
    one in order, or (grouped) as one grouped launch per copy."""
    from w4a16_quantized_gemm_gb300 import binding
    items = [it for it in wl.items if it["case"].M == M]
    sets = [[it["w"] for it in items]]
    for _ in range(rounds - 1):
        sets.append([])
        for it in items:
            q, z, s_ = it["w"].unpack()
            sets[-1].append(binding.pack(q, z, s_, it["case"].g))
            del q, z, s_

    def launch(st):
        for ws in sets:
            if grouped:
                binding.gemm_grouped([(it["X"], w, it["Y"], False) for it, w in zip(items, ws)], stream=st)
            else:
                for it, w in zip(items, ws):
                    binding.gemm(it["X"], w, out=it["Y"], stream=st)
    ms = _time_graph(launch, stream, 10) / rounds
    plan = binding.plan_grouped(sets[0], M) if grouped else None
    for ws in sets[1:]:
        for w in ws:
            w.free()
    nbytes = sum(it["bytes"] for it in items)
    nflops = sum(it["flops"] for it in items)
    how = "one grouped launch" if grouped else "four launches"
    e = {"config": 1, "step": f"llama3-8b layer linears at M={M}, {how}", "M": M, "grouped": grouped,
         "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes,
         "roofline": roofline_entry(nbytes, nflops, ms * 1e-3, peaks)}
    if plan:
        e["plan"] = plan
    return e


def _decode_step_concurrent(wl, stream, peaks, rounds=3):
    """The headline step with its four M values as four independent chains
    (each the layer linears qkv, o_proj, gate_up, down in order, on `rounds`
    weight copies), one stream each, forked and joined inside one graph: how
    far the per-launch start-up of one chain hides under the others."""
    import torch

    from w4a16_quantized_gemm_gb300 import binding
    Ms = sorted({it["case"].M for it in wl.items})
    chains = {}
    extra = []
    for M in Ms:
        items = [it for it in wl.items if it["case"].M == M]
        sets = [[it["w"] for it in items]]
        for _ in range(rounds - 1):
            sets.append([])
            for it in items:
                q, z, s_ = it["w"].unpack()
                sets[-1].append(binding.pack(q, z, s_, it["case"].g))
                extra.append(sets[-1][-1])
                del q, z, s_
        chains[M] = (items, sets)
    side = [torch.cuda.Stream(stream.device) for _ in Ms]

    def launch(st):
        start = torch.cuda.Event()
        start.record(st)
        for k, M in enumerate(Ms):
            side[k].wait_event(start)
            items, sets = chains[M]
            for ws in sets:
                for it, w in zip(items, ws):
                    binding.gemm(it["X"], w, out=it["Y"], stream=side[k])
            done = torch.cuda.Event()
            done.record(side[k])
            st.wait_event(done)
    ms = _time_graph(launch, stream, 10) / rounds
    for w in extra:
        w.free()
    return {"config": 1, "step": "llama3-8b decode step with its four M values as four concurrent chains "
                                 "(one stream each; each chain qkv, o_proj, gate_up, down in order)",
            "us": round(ms * 1e3, 2), "GB/s": round(wl.step_bytes / (ms * 1e-3) / 1e9, 1),
            "roofline": roofline_entry(wl.step_bytes, wl.step_flops, ms * 1e-3, peaks)}


def _prefill_step(device, stream, peaks, steps):
    """Workload 2 as one step (the 12 prefill GEMMs, each with its own weights)
    captured as a graph: TFLOP/s against the burst tensor peak."""
    wl = Workload("prefill", device)
    ms = _time_graph(lambda st: wl.launch_all(st), stream, steps)
    for it in wl.items:
        it["w"].free()
    return {"config": 2, "step": WORKLOADS["prefill"]["name"], "us": round(ms * 1e3, 1),
            "TFLOP/s": round(wl.step_flops / (ms * 1e-3) / 1e12, 1), "flops": wl.step_flops,
            "roofline": roofline_entry(wl.step_bytes, wl.step_flops, ms * 1e-3, peaks)}


def config_detail(wl, stream, peaks, args, min_bytes=300e6, reps=5):
    """Every configuration of the metric (workloads 0-4), each GEMM in steady
    state: launched back to back (programmatic dependent launch) on enough
    distinct copies of its packed weights to exceed L2, captured as one graph;
    time per launch = replay time / copies, with its own roofline (burst
    tensor peak: every replay lasts milliseconds at most).  Then the step-level
    figures: the headline workload's layer linears per M (and M <= 16
    together), and the prefill step of workload 2."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth
    device = wl.items[0]["X"].device
    out = []
    groups = {}
    for ci in range(5):
        for c in synth.workload(ci):
            groups.setdefault((c.K, c.N, c.g, c.stress), []).append((ci, c))
    for key, cases in groups.items():
        copies, sal = _pack_copies(key, device, min_bytes)
        for ci, c in cases:
            Xh = synth.activations(c.M, c.K, sal, 0, tag=f"/N{c.N}/g{c.g}" + ("/stress" if c.stress else ""))
            X = torch.from_numpy(Xh.view(np.uint16)).to(device).view(torch.float16)
            Y = torch.empty((c.M, c.N), dtype=torch.float16, device=device)

            def launch(st, X=X, Y=Y):
                for w in copies:
                    binding.gemm(X, w, out=Y, stream=st)
            ms = _time_graph(launch, stream, reps) / len(copies)
            nb, nf = algorithmic_bytes(c.M, c.K, c.N, c.g), flops(c.M, c.K, c.N)
            out.append({"config": ci, "gemm": c.name, "M": c.M, "us": round(ms * 1e3, 2),
                        "GB/s": round(nb / (ms * 1e-3) / 1e9, 1), "TFLOP/s": round(nf / (ms * 1e-3) / 1e12, 1),
                        "plan": binding.plan(copies[0], c.M), "roofline": roofline_entry(nb, nf, ms * 1e-3, peaks)})
            del X, Y
        for w in copies:
            w.free()
        del copies
        torch.cuda.empty_cache()
    dwl = wl if wl.kind == "decode" else Workload("decode", device)  # the step figures are the decode workload's
    for grouped in (True, False):
        steps = [_decode_step_at_m(dwl, M, stream, peaks, grouped=grouped) for M in (1, 8, 16, 32)]
        out.extend(steps)
        small = [e for e in steps if e["M"] <= 16]
        nb = sum(e["bytes"] for e in small)
        t = sum(e["us"] for e in small) * 1e-6
        how = "one grouped launch per M" if grouped else "one launch per GEMM"
        out.append({"config": 1, "step": f"llama3-8b layer linears at M in {{1,8,16}} (the decode target's range), "
                                         f"{how}", "grouped": grouped,
                    "us": round(t * 1e6, 2), "GB/s": round(nb / t / 1e9, 1),
                    "roofline": roofline_entry(nb, 0, t, peaks)})
    for grouped, what in ((False, "the 16 GEMMs launched one by one on one stream (16 launches)"),
                          (True, "one grouped launch per M on one stream (4 launches)")):
        ms = _time_graph(lambda st: dwl.launch_all(st, grouped=grouped, concurrent=False), stream, 20)
        out.append({"config": 1, "step": f"llama3-8b decode step, {what}",
                    "us": round(ms * 1e3, 2), "GB/s": round(dwl.step_bytes / (ms * 1e-3) / 1e9, 1),
                    "roofline": roofline_entry(dwl.step_bytes, dwl.step_flops, ms * 1e-3, peaks)})
    out.append(_decode_step_concurrent(dwl, stream, peaks))
    out.append(_prefill_step(device, stream, peaks, max(5, min(args.steps, 50))))
    return out


def run_e2e(wl, args, spec):
    """Public call with host buffers: tm_w4a16_gemm_host_batch (every GEMM's X
    in one copy from pinned host memory, the step's products in order, every Y
    back in one copy to pinned host memory), host wall clock.  Consecutive
    steps alternate between two streams, each with its own pinned and device
    buffers, so that one step's copies overlap the other's products; a stream
    is synchronised before its buffers are reused (two steps later) and once
    more at the end, so every step's copies in and out lie inside the timed
    region.  The first step's results are compared bit for bit with the
    device-resident run's outputs."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding

    Ms = [int(it["Xh"].shape[0]) for it in wl.items]
    batches = [binding.HostBatch([it["w"] for it in wl.items], Ms) for _ in range(2)]
    for b in batches:
        for i, it in enumerate(wl.items):
            b.x(i).copy_(torch.from_numpy(it["Xh"].view(np.uint16)).view(torch.float16))
    h2d = batches[0].X_host.numel() * 2
    d2h = batches[0].Y_host.numel() * 2
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    batches[0].run(streams[0])  # waits for the stream
    # the device-resident step's own launches, now (the detail figures rewrite Y with other settings)
    with torch.cuda.stream(streams[1]):
        wl.launch_all(streams[1])
    streams[1].synchronize()
    same = all(torch.equal(batches[0].y(i).view(torch.int16), it["Y"].cpu().view(torch.int16))
               for i, it in enumerate(wl.items))

    def run(n):
        for k in range(n):
            j = k & 1
            streams[j].synchronize()  # step k - 2 (its copy out included) is done: reuse its buffers
            batches[j].run(streams[j], sync=False)
        for st in streams:
            st.synchronize()

    steps = max(3, min(args.steps, 200))
    run(4)
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    # the same calls one step at a time on one stream, synchronised after each
    t1 = time.perf_counter()
    for _ in range(steps):
        batches[0].run(streams[0])
    dt1 = time.perf_counter() - t1
    units = (wl.step_bytes / 1e9) if spec["unit"] == "GB/s" else (wl.step_flops / 1e12)
    return {"value": round(units * steps / dt, 2), "unit": spec["unit"], "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(dt * 1e3 / steps, 3),
            "bitwise_equal_to_device_run": same,
            "serial_one_stream": {"value": round(units * steps / dt1, 2), "ms_per_step": round(dt1 * 1e3 / steps, 3)},
            "timing": "host wall clock; per step one tm_w4a16_gemm_host_batch call (every X in one copy from "
                      "pinned host memory, the GEMMs, every Y out in one copy to pinned host memory); steps "
                      "alternate between two streams with their own buffers, so a step's copies -- and its "
                      "products -- overlap the other stream's; each stream is synchronised before its buffers "
                      "are reused and at the end.  serial_one_stream: the same calls one step at a time"}


# ------------------------------------------------------------ CPU baseline ---

def _oracle_sample(cases_weights, cols, threads):
    """Time the oracle on the first `cols` columns of every GEMM; returns
    (seconds, extrapolated seconds for the full step)."""
    import numpy as np

    import oracle
    t_sample = 0.0
    t_full = 0.0
    for (c, q, z, s, X) in cases_weights:
        n = min(c.N, cols)
        qs, zs, ss = (np.ascontiguousarray(a[:, :n]) for a in (q, z, s))
        t0 = time.perf_counter()
        oracle.gemm(X, qs, zs, ss, c.g, threads=threads)
        dt = time.perf_counter() - t0
        t_sample += dt
        t_full += dt * c.N / n
    return t_sample, t_full


def _cases_with_weights(kind):
    from w4a16_quantized_gemm_gb300 import synth
    out = []
    cache = {}
    for c in synth.workload(WORKLOADS[kind]["idx"]):
        key = (c.K, c.N, c.g)
        if key not in cache:
            cache[key] = synth.weights(c.K, c.N, c.g)
        q, z, s, _ = cache[key]
        X = synth.activations(c.M, c.K, None, 0, tag=f"/N{c.N}/g{c.g}")
        out.append((c, q, z, s, X))
    return out


def _calibrated_cols(cw, budget_s, threads):
    t, _ = _oracle_sample(cw, 16, threads)
    cols = int(16 * budget_s / max(t, 1e-6))
    return max(16, min(cols // 16 * 16, max(c.N for (c, *_rest) in cw)))


def cpu_baseline(wl, budget_s):
    import oracle
    threads = oracle.default_threads()
    cw = _cases_with_weights(wl.kind)
    cols = _calibrated_cols(cw, budget_s, threads)
    t_sample, t_full = _oracle_sample(cw, cols, threads)
    spec = WORKLOADS[wl.kind]
    units = wl.step_bytes / 1e9 if spec["unit"] == "GB/s" else wl.step_flops / 1e12
    return {"value": round(units / t_full, 4), "unit": spec["unit"], "cores": threads, "kind": "oracle",
            "sample": f"every GEMM of one step on its first {cols} output columns (all M rows, full K); "
                      f"{t_sample:.1f} s measured, scaled by N/{cols} per GEMM to a full step "
                      f"({t_full:.1f} s)",
            "config0_one_thread": config0_one_thread()}


def config0_one_thread():
    """The oracle on workload 0 (one 1x4096x4096 GEMM, g = 128) in full, one
    thread: the single-core baseline of the smallest configuration."""
    import oracle
    from w4a16_quantized_gemm_gb300 import synth
    c = synth.workload(0)[0]
    p = synth.case_problem(c)
    oracle.gemm(p.X, p.q, p.z, p.s, c.g, threads=1)  # warm (page in, first call)
    t0 = time.perf_counter()
    oracle.gemm(p.X, p.q, p.z, p.s, c.g, threads=1)
    dt = time.perf_counter() - t0
    nb = algorithmic_bytes(c.M, c.K, c.N, c.g)
    return {"gemm": c.name, "ms": round(dt * 1e3, 2), "GB/s": round(nb / dt / 1e9, 4), "cores": 1}


def run_reference(args, rank, world):
    """The reference arm: the oracle as it stands, on the host cores.  Each
    step is the whole workload when that fits the run's time budget (every
    GEMM of the step in full); otherwise every GEMM on its first C output
    columns, C chosen for the budget, and the line says so.  ms_per_step and
    value are what was measured on the work that ran."""
    if rank != 0:
        return
    import oracle
    spec = WORKLOADS[args.workload]
    threads = oracle.default_threads()
    cw = _cases_with_weights(args.workload)
    budget_s = 150.0  # the whole --steps/--warmup run
    full_cols = max(c.N for (c, *_r) in cw)
    t_probe, t_full_est = _oracle_sample(cw, 64, threads)
    steps_total = args.steps + args.warmup
    if t_full_est * steps_total <= budget_s:
        cols = full_cols
    else:
        cols = max(16, int(full_cols * budget_s / (t_full_est * steps_total)) // 16 * 16)
    for _ in range(args.warmup):
        _oracle_sample(cw, cols, threads)
    t_run = 0.0
    for _ in range(args.steps):
        a, _b = _oracle_sample(cw, cols, threads)
        t_run += a
    done_bytes = sum(algorithmic_bytes(c.M, c.K, min(c.N, cols), c.g) for (c, *_r) in cw)
    done_flops = sum(flops(c.M, c.K, min(c.N, cols)) for (c, *_r) in cw)
    units = done_bytes / 1e9 if spec["unit"] == "GB/s" else done_flops / 1e12
    value = units * args.steps / t_run
    if cols >= full_cols:
        sample = "every step the whole workload (every GEMM in full)"
    else:
        sample = (f"every step each GEMM on its first {cols} output columns (all M rows, full K): "
                  f"{done_bytes} algorithmic bytes per step, value = those bytes / measured time")
    cfg = workload_config(args.workload)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": spec["unit"],
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(t_run * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
           "cpu_baseline": {"value": round(value, 4), "unit": spec["unit"], "cores": threads, "kind": "oracle",
                            "sample": sample, "config0_one_thread": config0_one_thread()},
           "e2e": {"value": round(value, 4), "unit": spec["unit"], "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_rtn(args, rank, world, local):
    """--workload rtn: round-to-nearest INT4 quantisation (tm_quantize_rtn) of
    the four Llama-3-8B linear weights (fp16 in; codes, zeros, scales out), one
    step = the four layers, graph-replayed; GB/s of algorithmic bytes against
    the measured HBM copy bandwidth."""
    import ctypes

    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    peaks = load_peaks()
    g = 128
    layers = []
    for name, (K, N) in synth.LLAMA3_8B.items():
        Wh = synth.fp16_weights(K, N, g)
        W = torch.from_numpy(Wh.view(np.uint16)).to(device).view(torch.float16)
        q = torch.empty((K, N), dtype=torch.uint8, device=device)
        z = torch.empty((K // g, N), dtype=torch.uint8, device=device)
        sc = torch.empty((K // g, N), dtype=torch.float16, device=device)
        layers.append({"name": name, "K": K, "N": N, "Wh": Wh, "W": W, "q": q, "z": z, "s": sc,
                       "bytes": rtn_bytes(K, N, g)})
    step_bytes = sum(L["bytes"] for L in layers)
    lib = binding.load()
    stream = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)

    def quantize(L, st):
        r = lib.tm_quantize_rtn(L["W"].data_ptr(), L["K"], L["N"], g, L["q"].data_ptr(), L["z"].data_ptr(),
                                L["s"].data_ptr(), ctypes.c_void_p(st.cuda_stream))
        if r != 0:
            raise RuntimeError(f"tm_quantize_rtn failed: {r}")

    # The four layers are independent: gate_up and o_proj on the launching
    # stream, down and qkv on a second one, joined before the step ends, so
    # that one layer's wave tail overlaps another's launch.
    by = {L["name"]: L for L in layers}

    def launch_all(st):
        start = torch.cuda.Event()
        start.record(st)
        side.wait_event(start)
        for a, b in (("gate_up", "down"), ("o_proj", "qkv")):
            quantize(by[a], st)
            quantize(by[b], side)
        done = torch.cuda.Event()
        done.record(side)
        st.wait_event(done)

    with torch.cuda.stream(stream):
        launch_all(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch_all(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_sampler0 = time.time()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for _ in range(args.steps):
            graph.replay()
        evs[1].record(stream)
    stream.synchronize()
    t_ms = evs[0].elapsed_time(evs[1])
    with torch.cuda.stream(stream):
        while time.time() - t_sampler0 < 1.5:
            for _ in range(50):
                graph.replay()
            stream.synchronize()
    clocks = sampler.stop()
    t_max_s = reduce_max(t_ms / 1e3, world)
    value = aggregate(step_bytes * args.steps / 1e9, world, t_max_s)
    achieved = step_bytes / (t_ms / 1e3 / args.steps) / 1e9

    e2e = None
    cpu = None
    if rank == 0:
        # public call with host buffers: pinned W in, quantise, codes/zeros/scales out
        hostW = [torch.from_numpy(L["Wh"].view(np.uint16)).view(torch.float16).pin_memory() for L in layers]
        outs = [(torch.empty(tuple(L["q"].shape), dtype=torch.uint8, pin_memory=True),
                 torch.empty(tuple(L["z"].shape), dtype=torch.uint8, pin_memory=True),
                 torch.empty(tuple(L["s"].shape), dtype=torch.float16, pin_memory=True)) for L in layers]
        h2d = sum(w.numel() * 2 for w in hostW)
        d2h = sum(a.numel() * a.element_size() for o in outs for a in o)
        steps = max(3, min(args.steps, 20))
        t0 = time.perf_counter()
        for _ in range(steps):
            for w, o in zip(hostW, outs):
                qd, zd, sd = binding.quantize_rtn(w.to(device, non_blocking=True), g)
                o[0].copy_(qd, non_blocking=True)
                o[1].copy_(zd, non_blocking=True)
                o[2].copy_(sd, non_blocking=True)
            torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        e2e = {"value": round(step_bytes / 1e9 * steps / dt, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(dt * 1e3 / steps, 3),
               "timing": "host wall clock; W copied in, quantised, codes/zeros/scales copied out"}
        if world == 1 and not args.no_cpu:
            import oracle.rtn as rtn_oracle  # the CPU baseline leg only
            t0 = time.perf_counter()
            for L in layers:
                rtn_oracle.quantize(L["Wh"], g)
            t_cpu = time.perf_counter() - t0
            cpu = {"value": round(step_bytes / 1e9 / t_cpu, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"the whole step (four layers, numpy binary32 on one core), {t_cpu:.1f} s"}
    out = {
        "metric": "RTN INT4 quantisation GB/s (fp16 weights in, codes/zeros/scales out), Llama-3-8B linears",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max_s * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "rtn: qkv/o_proj/gate_up/down fp16 weights, g=128", "launches_per_step": len(layers),
                   "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2 (698 MB of fp16 weights per step)"},
        "launch": "one CUDA graph per step: gate_up then o_proj on the launching stream, down then qkv on a "
                  "second stream (independent layers), joined before the step ends",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": read_traffic("rtn", "llama3_8b_rtn"),
                     "peak_source": peaks["source"], "kernel": "rtn_tma_kernel",
                     "basis": "algorithmic bytes of the step's four launches / mean step time (CUDA events "
                              "around graph replays); traffic = DRAM bytes per launch, the mean over the "
                              "step's four launches"},
        "gpu_launches": len(layers) * args.steps, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_silu(args, rank, world, local):
    """--workload silu: the Llama-3-8B gate_up layer (4096 x 28672, g=128) with
    the fused silu(gate) * up epilogue (tm_w4a16_gemm_silu_mul) at the decode
    sizes M in {1, 8, 16, 32}, one step = the four launches, graph-replayed;
    GB/s of algorithmic bytes (W4 weights, X in, H out) against the measured
    HBM bandwidth.  `unfused_ms_per_step` times the same step as GEMM + a
    separate torch silu-mul pass, for context."""
    import numpy as np
    import torch
    import torch.nn.functional as F

    from w4a16_quantized_gemm_gb300 import binding, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    peaks = load_peaks()
    K, N, g = synth.LLAMA3_8B["gate_up"][0], synth.LLAMA3_8B["gate_up"][1], 128
    q, z, s, _ = synth.weights(K, N, g)
    items = []
    Ms = (1, 8, 16, 32)
    for M in Ms:
        w = binding.pack(torch.from_numpy(q).to(device), torch.from_numpy(z).to(device),
                         torch.from_numpy(s.view(np.uint16)).to(device).view(torch.float16), g)
        X = torch.from_numpy(synth.activations(M, K, tag=f"/silu/M{M}").view(np.uint16)).to(device).view(torch.float16)
        items.append({"M": M, "w": w, "X": X, "H": torch.empty((M, N // 2), dtype=torch.float16, device=device),
                      "Y": torch.empty((M, N), dtype=torch.float16, device=device),
                      "bytes": K * N // 2 + (K // g) * N * 5 // 2 + 2 * M * K + 2 * M * (N // 2)})
    step_bytes = sum(it["bytes"] for it in items)
    stream = torch.cuda.Stream(device)

    # The four batch sizes are independent products: one stream each, joined
    # before the step ends.
    sides = [torch.cuda.Stream(device) for _ in items[1:]]

    def fused(st):
        start = torch.cuda.Event()
        start.record(st)
        for sd in sides:
            sd.wait_event(start)
        for it, sd in zip(items, [st] + sides):
            binding.gemm_silu_mul(it["X"], it["w"], out=it["H"], stream=sd)
        for sd in sides:
            done = torch.cuda.Event()
            done.record(sd)
            st.wait_event(done)

    def unfused(st):
        for it in items:
            binding.gemm(it["X"], it["w"], out=it["Y"], stream=st)
            y = it["Y"].view(it["M"], N // 8, 2, 4)
            it["H"].view(it["M"], N // 8, 4).copy_(F.silu(y[:, :, 0, :].float()).mul_(y[:, :, 1, :].float()))

    def timed(fn, steps):
        with torch.cuda.stream(stream):
            fn(stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fn(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graph.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1), graph

    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    t_ms, graph = timed(fused, args.steps)
    with torch.cuda.stream(stream):
        while time.time() - t0 < 1.5:
            for _ in range(50):
                graph.replay()
            stream.synchronize()
    clocks = sampler.stop()
    t_unfused, _ = timed(unfused, args.steps)
    t_max_s = reduce_max(t_ms / 1e3, world)
    value = aggregate(step_bytes * args.steps / 1e9, world, t_max_s)
    achieved = step_bytes / (t_ms / 1e3 / args.steps) / 1e9
    out = {
        "metric": "fused gate_up + silu*mul W4A16 GB/s, Llama-3-8B gate_up (4096 x 28672), M in {1,8,16,32}",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max_s * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "silu: gate_up with fused silu(gate)*up epilogue", "launches_per_step": len(items),
                   "bytes_per_step": step_bytes, "unfused_ms_per_step": round(t_unfused / args.steps, 4),
                   "unfused": "the same GEMMs writing Y [M][N], then torch silu-mul on the interleaved halves",
                   "l2": "each GEMM has its own packed weights (235 MB per step > 129 MB L2)"},
        "launch": "one CUDA graph per step: the four batch sizes (independent products) on four streams, "
                  "joined before the step ends (the unfused figure: one stream)",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "peak_source": peaks["source"], "kernel": "decode_kernel / tc_kernel (fused epilogue)"},
        "gpu_launches": len(items) * args.steps, "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_kv(args, rank, world, local):
    """--workload kv: decode attention over a low-bit KV cache
    (tm_kv_decode_attention), Llama-3-8B heads (32 query / 8 KV heads, D = 128),
    32 sequences x 4096 cached tokens, one step = the int8 and the int4 cache
    (two launches on two streams), graph-replayed; GB/s of algorithmic bytes
    (codes, scales and zeros of K and V, Q in, out) against the measured HBM
    bandwidth."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    peaks = load_peaks()
    Bsz, L, Hq, Hkv, D = 32, 4096, 32, 8, 128
    lens = torch.full((Bsz,), L, dtype=torch.int32, device=device)
    Q = torch.from_numpy(synth.normal64("kvbench/Q", 1, Bsz * Hq * D).reshape(Bsz, Hq, D)
                         .astype(np.float16).view(np.uint16)).to(device).view(torch.float16)
    caches = []
    for bits in (8, 4):
        # the head-major cache order [B][Hkv][L][D]
        K = torch.randn((Bsz, Hkv, L, D), generator=torch.Generator(device=device).manual_seed(bits),
                        device=device, dtype=torch.float32).half()
        V = torch.randn((Bsz, Hkv, L, D), generator=torch.Generator(device=device).manual_seed(100 + bits),
                        device=device, dtype=torch.float32).half()
        vq = binding.kv_quantize(V, bits)
        caches.append((bits, binding.kv_quantize(K, bits), (binding.kv_pack_v(vq[0], bits), vq[1], vq[2]),
                       torch.empty((Bsz, Hq, D), dtype=torch.float16, device=device), vq[0]))
        del K, V
    step_bytes = sum(kv_cache_bytes(Bsz, L, Hkv, D, bits) for bits in (8, 4)) + 2 * 2 * Bsz * Hq * D * 2
    stream = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)

    # The two caches are independent: the int4 attention (bound by the
    # instructions it issues) on the launching stream and the int8 attention
    # (bound by HBM) on a second stream, joined before the step ends -- each
    # fills SM slots the other leaves idle (256 (sequence, KV head) CTAs each
    # on 304 slots).
    def launch_all(st):
        start = torch.cuda.Event()
        start.record(st)
        side.wait_event(start)
        for bits, kq, vq, out, _ in sorted(caches, key=lambda c: c[0]):
            binding.kv_decode_attention(Q, kq, vq, lens, bits, out=out, stream=st if bits == 4 else side)
        done = torch.cuda.Event()
        done.record(side)
        st.wait_event(done)

    with torch.cuda.stream(stream):
        launch_all(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch_all(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    t_ms = e0.elapsed_time(e1)
    with torch.cuda.stream(stream):
        while time.time() - t0 < 1.5:
            for _ in range(50):
                graph.replay()
            stream.synchronize()
    clocks = sampler.stop()
    t_max_s = reduce_max(t_ms / 1e3, world)
    value = aggregate(step_bytes * args.steps / 1e9, world, t_max_s)
    achieved = step_bytes / (t_ms / 1e3 / args.steps) / 1e9
    # each cache format on its own (one launch a step): the step above overlaps the two
    per_format = []
    for bits, kq, vq, out_, _ in caches:
        def one(st, bits=bits, kq=kq, vq=vq, out_=out_):
            binding.kv_decode_attention(Q, kq, vq, lens, bits, out=out_, stream=st)
        ms = _time_graph(one, stream, max(10, min(args.steps, 100)))
        nb = kv_cache_bytes(Bsz, L, Hkv, D, bits) + 2 * Bsz * Hq * D * 2
        per_format.append({"bits": bits, "us": round(ms * 1e3, 2), "GB/s": round(nb / (ms * 1e-3) / 1e9, 1),
                           "frac": round(nb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)})
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        # the fp64 oracle on the whole step (dequantise both caches, attention),
        # repeated for at least 10 s
        import oracle.kv as kv_oracle  # the CPU baseline leg only
        host = [(bits, [t.cpu().numpy() for t in kq], [vcodes.cpu().numpy(), vq[1].cpu().numpy(), vq[2].cpu().numpy()])
                for bits, kq, vq, _, vcodes in caches]
        q64 = Q.float().cpu().numpy().astype(np.float64)
        lens_np = np.full(Bsz, L)
        reps, ts, cs = 0, time.perf_counter(), time.process_time()
        while reps == 0 or time.perf_counter() - ts < 10.0:
            for bits, (kc, ks, kz), (vc, vs, vz) in host:
                Kd = np.swapaxes(kv_oracle.dequantize(kc, ks.view(np.float16), kz, bits), 1, 2)
                Vd = np.swapaxes(kv_oracle.dequantize(vc, vs.view(np.float16), vz, bits), 1, 2)
                kv_oracle.decode_attention(q64, Kd, Vd, lens_np)
                del Kd, Vd
            reps += 1
        wall = time.perf_counter() - ts
        t_step = wall / reps
        used = max(1, round((time.process_time() - cs) / wall))  # BLAS threads numpy actually kept busy
        cpu = {"value": round(step_bytes / 1e9 / t_step, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"the whole step (both caches, all 32 sequences: fp64 dequantisation and attention, "
                         f"numpy), {reps} repetition(s) in {t_step * reps:.1f} s"}
    out = {
        "metric": "low-bit KV decode attention GB/s, Llama-3-8B heads (32q/8kv, D=128), 32 seqs x 4096 tokens, "
                  "int8 + int4 caches",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max_s * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "kv: decode attention, B=32, L=4096, Hq=32, Hkv=8, D=128, int8 and int4",
                   "launches_per_step": 2, "bytes_per_step": step_bytes,
                   "streams": "int4 on the launching stream, int8 on a second stream (independent caches)",
                   "l2": f"inputs larger than L2 ({step_bytes / 1e6:.0f} MB of cache per step)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": read_traffic("kv", "llama3_8b_kv"),
                     "peak_source": peaks["source"], "kernel": "kv_attn_tc_kernel"},
        "gpu_launches": 2 * args.steps, "clocks": clocks, "cpu_baseline": cpu,
        "detail": per_format,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_w8a8(args, rank, world, local, prefill=False):
    """--workload w8a8 / w8a8_prefill: the W8A8 path on the four Llama-3-8B
    linear shapes -- per GEMM, the per-token activation quantiser
    (tm_w8a8_quantize_act) then the GEMM (tm_w8a8_gemm) -- at the decode sizes
    M in {1, 8, 16, 32} (GB/s of algorithmic bytes against the measured HBM
    bandwidth) or the prefill sizes M in {128, 1024, 4096} (TFLOP/s against
    the measured bf16 peak: the products run on fp16 tensor cores).  One step =
    every (shape, M) pair, each with its own packed weights, graph-replayed."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    binding.load()
    peaks = load_peaks()
    Ms = (128, 1024, 4096) if prefill else (1, 8, 16, 32)
    # the activation codes: fp16 integers (TMA-staged X, tm_w8a8_gemm_f16) for
    # prefill, int8 (the decode kernel's operand) for decode, unless forced
    codes = args.w8_codes if args.w8_codes != "auto" else ("f16" if prefill else "int8")
    host = {}
    items = []
    for name in ("qkv", "o_proj", "gate_up", "down"):
        K, N = synth.LLAMA3_8B[name]
        Wh = (synth.normal64(f"w8bench/W/{name}", K, N) * 0.02).astype(np.float16)
        W = torch.from_numpy(Wh.view(np.uint16)).to(device).view(torch.float16)
        qd, sd = binding.w8_quantize_weight(W)  # the per-channel quantiser on the GPU
        del W
        host[name] = Wh
        for M in Ms:
            X = torch.from_numpy(synth.activations(M, K, tag=f"/w8/{name}/M{M}").view(np.uint16)).to(device)
            X = X.view(torch.float16)
            items.append({"name": name, "M": M, "K": K, "N": N, "w": binding.pack_w8(qd, sd), "X": X,
                          "xq": torch.empty((M, K), dtype=torch.int8 if codes == "int8" else torch.float16,
                                            device=device),
                          "sx": torch.empty((M,), dtype=torch.float32, device=device),
                          "Y": torch.empty((M, N), dtype=torch.float16, device=device),
                          "bytes": w8a8_bytes(M, K, N),
                          "flops": 2 * M * K * N})
        del qd, sd
    step_bytes = sum(it["bytes"] for it in items)
    step_flops = sum(it["flops"] for it in items)
    weight_bytes = sum(it["w"].nbytes for it in items)
    stream = torch.cuda.Stream(device)

    # The step's products are independent: the activation quantisers run on a
    # second stream, each GEMM waiting only for its own quantiser, so that a
    # quantiser (HBM-bound) overlaps the GEMMs before it (tensor-bound in
    # prefill); the second stream joins the first before the step ends.
    side = torch.cuda.Stream(device)
    lane2 = torch.cuda.Stream(device)
    # The GEMMs on two lanes as in the W4A16 steps: decode M = 16 and 8, or
    # the prefill products under 60 GFLOP, on a second GEMM stream.
    second = [(it["M"] in (8, 16)) if not prefill else (it["flops"] < 60e9) for it in items]
    w8_streams = args.w8_streams

    def launch_all(st):
        start = torch.cuda.Event()
        start.record(st)
        side.wait_event(start)
        lane2.wait_event(start)
        for it, two in zip(items, second):
            gst = lane2 if (two and w8_streams > 2) else st
            if codes == "int8":
                binding.w8a8_quantize_act(it["X"], out=(it["xq"], it["sx"]), stream=side)
            else:
                binding.w8a8_quantize_act_f16(it["X"], out=(it["xq"], it["sx"]), stream=side)
            ready = torch.cuda.Event()
            ready.record(side)
            gst.wait_event(ready)
            if codes == "int8":
                binding.w8a8_gemm(it["xq"], it["sx"], it["w"], out=it["Y"], tile_m=args.w8_tile_m, stream=gst)
            else:
                binding.w8a8_gemm_f16(it["xq"], it["sx"], it["w"], out=it["Y"], tile_m=args.w8_tile_m, stream=gst)
        for sd in (side, lane2):
            done = torch.cuda.Event()
            done.record(sd)
            st.wait_event(done)

    with torch.cuda.stream(stream):
        launch_all(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch_all(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    t_ms = e0.elapsed_time(e1)
    with torch.cuda.stream(stream):
        while time.time() - t0 < 1.5:
            for _ in range(20):
                graph.replay()
            stream.synchronize()
    clocks = sampler.stop()
    t_max_s = reduce_max(t_ms / 1e3, world)
    step_s = t_ms / 1e3 / args.steps
    if prefill:
        value = aggregate(step_flops * args.steps / 1e12, world, t_max_s)
        achieved = step_flops / step_s / 1e12
        peak, unit, bound = peaks["bf16_tflops"], "TFLOP/s", "tensor"  # a ms-scale step: the burst peak
    else:
        value = aggregate(step_bytes * args.steps / 1e9, world, t_max_s)
        achieved = step_bytes / step_s / 1e9
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        # the oracle (binary32 quantiser, exact int64 product) on the first
        # `cols` output columns of every GEMM of the step, scaled by N / cols
        import oracle.w8a8 as w8_oracle  # the CPU baseline leg only
        cols = 64 if prefill else 2048
        t_sample = t_full = 0.0
        qw = {name: w8_oracle.quantize_weight(Wh) for name, Wh in host.items()}
        for it in items:
            q, sw = qw[it["name"]]
            Xh = it["X"].cpu().numpy()
            ts = time.perf_counter()
            qx, sx = w8_oracle.quantize_act(Xh)
            w8_oracle.gemm(qx, sx, q[:, :cols], sw[:cols])
            dt = time.perf_counter() - ts
            t_sample += dt
            t_full += dt * it["N"] / cols
        units = step_flops / 1e12 if prefill else step_bytes / 1e9
        cpu = {"value": round(units / t_full, 6), "unit": unit, "cores": 1, "kind": "oracle",
               "sample": f"every GEMM of one step on its first {cols} output columns (all rows, full K), "
                         f"{t_sample:.1f} s measured, scaled by N/{cols} per GEMM to a full step ({t_full:.1f} s)"}
    label = "prefill, M in {128,1024,4096}" if prefill else "decode, M in {1,8,16,32}"
    out = {
        "metric": f"W8A8 {unit}, Llama-3-8B linear layers, {label} (per-token quantiser + GEMM)",
        "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max_s * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"w8a8{'_prefill' if prefill else ''}: qkv, o_proj, gate_up, down x M",
                   "activation_codes": codes, "tile_m": args.w8_tile_m or "auto",
                   "launches_per_step": 2 * len(items), "bytes_per_step": step_bytes, "flops_per_step": step_flops,
                   "streams": "the activation quantisers on a second stream, each GEMM waiting for its own "
                              "quantiser (the products are independent)"
                              + ("; the GEMMs of M = 16 and 8 (decode) or under 60 GFLOP (prefill) on a third"
                                 if args.w8_streams > 2 else ""),
                   "l2": f"each GEMM has its own packed weights ({weight_bytes / 1e6:.0f} MB per step > 129 MB L2)"},
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4),
                     "traffic": None if prefill else read_traffic("w8", "llama3_8b_w8a8"),
                     "peak_source": peaks["source"], "kernel": "w8tc_kernel (+ w8_quant_act_kernel), whole step"
                     if prefill else "w8_kernel (+ w8_quant_act_kernel), whole step"},
        "gpu_launches": 2 * len(items) * args.steps, "clocks": clocks, "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_rtn_reference(args, rank):
    """Reference arm of --workload rtn: the binary32 oracle on the host."""
    if rank != 0:
        return
    import oracle.rtn as rtn_oracle
    from w4a16_quantized_gemm_gb300 import synth
    g = 128
    W = {n: synth.fp16_weights(K, N, g) for n, (K, N) in synth.LLAMA3_8B.items()}
    step_bytes = sum(rtn_oracle.bytes_moved(K, N, g) for (K, N) in synth.LLAMA3_8B.values())
    for _ in range(args.warmup if args.warmup < 2 else 1):
        rtn_oracle.quantize(W["o_proj"], g)
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(steps):
        for w in W.values():
            rtn_oracle.quantize(w, g)
    dt = time.perf_counter() - t0
    v = round(step_bytes / 1e9 * steps / dt, 4)
    print(json.dumps({"impl": "reference", "metric": "RTN INT4 quantisation GB/s (fp16 weights in, "
                      "codes/zeros/scales out), Llama-3-8B linears", "value": v, "unit": "GB/s", "n_gpus": 1,
                      "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / steps, 3),
                      "higher_is_better": True, "data": "synthetic",
                      "config": {"workload": "rtn: qkv/o_proj/gate_up/down fp16 weights, g=128"},
                      "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                       "sample": f"{steps} whole steps"},
                      "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
          flush=True)


def run_single(spec_text, path):
    """One GEMM shape, launched 15 times with a 256 MB write between launches
    (cold L2) -- a small, bounded case for ncu captures."""
    import numpy as np
    import torch

    from w4a16_quantized_gemm_gb300 import binding, synth
    M, K, N, g = (int(v) for v in spec_text.split(","))
    q, z, s, _ = synth.weights(K, N, g)
    w = binding.pack(torch.from_numpy(q).cuda(), torch.from_numpy(z).cuda(),
                     torch.from_numpy(s.view(np.uint16)).cuda().view(torch.float16), g)
    X = torch.from_numpy(synth.activations(M, K).view(np.uint16)).cuda().view(torch.float16)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cfg = {"path": path} if path else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ts = []
    for i in range(15):
        flush.fill_(i & 0xFF)
        ev[0].record()
        binding.gemm(X, w, out=Y, config=cfg)
        ev[1].record()
        torch.cuda.synchronize()
        ts.append(ev[0].elapsed_time(ev[1]) * 1e3)
    print(json.dumps({"single": [M, K, N, g], "plan": binding.plan(w, M, cfg),
                      "us_cold_isolated_median": sorted(ts[5:])[5]}))


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--w8-streams", type=int, default=3, choices=(2, 3),
                   help="W8A8 workloads: 2 = quantisers on a second stream; 3 = also the smaller GEMMs on a third")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + ["rtn", "silu", "kv", "w8a8", "w8a8_prefill"],
                   default="decode")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--w8-tile-m", type=int, choices=[0, 64, 128, 256], default=0,
                   help="W8A8 rows of X per CTA of the tensor-memory kernel (0: automatic)")
    p.add_argument("--w8-codes", choices=["auto", "int8", "f16"], default="auto",
                   help="W8A8 activation codes: int8 or fp16 integers (auto: fp16 for prefill, int8 for decode)")
    p.add_argument("--no-detail", action="store_true",
                   help="skip the per-configuration detail (every GEMM of workloads 0-4 in steady state, "
                        "the per-M decode steps and the prefill step)")
    p.add_argument("--single", default=None, help="M,K,N,g: one GEMM 15 times, cold L2 (for ncu captures)")
    p.add_argument("--path", type=int, default=0,
                   help="with --single: 1 decode, 2 prefill (shared-memory W^T), 3 tensor-memory, 0 automatic")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.single:
        run_single(args.single, args.path)
        return
    rank, world, local = dist_env()
    if world != args.gpus and "RANK" in os.environ:
        p.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        if args.workload == "rtn":
            run_rtn_reference(args, rank)
        elif args.workload in ("silu", "kv", "w8a8", "w8a8_prefill"):
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": f"the {args.workload} workload reports its "
                                  "oracle timing as cpu_baseline on its own line"}), flush=True)
        else:
            run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        if args.workload == "rtn":
            run_rtn(args, rank, world, local)
        elif args.workload == "silu":
            run_silu(args, rank, world, local)
        elif args.workload == "kv":
            run_kv(args, rank, world, local)
        elif args.workload in ("w8a8", "w8a8_prefill"):
            run_w8a8(args, rank, world, local, prefill=args.workload == "w8a8_prefill")
        else:
            run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
