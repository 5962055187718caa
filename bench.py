"""Benchmark of the NVFP4 linear-layer path on GB300.

One step = nvfp4_linear at every decode M (1, 2, 4, 8, 16, 32, 48) on the
decode-shaped weight [4096, 4096] (bf16 N(0, 0.02^2) with 0.5% outliers x8,
FourOverSix-quantised once beforehand; activations [M, 4096] bf16 N(0, 1)).
At these M the dispatch takes the W4A16 GEMM, so value = the W4A16 GEMMs'
algorithmic bytes / step time (GB/s).  Each call reads a weight no recent call
touched: quantised copies rotate through buffers totalling several times the
L2.  The step is captured in a CUDA graph; kernels are timed with CUDA events
on the launching stream.

Reported alongside: the whole path per step (FourOverSix quantisation of the
bf16 weight followed by the same linears), the quantiser alone, the W4A4
throughput on the prefill workload (activations [M, 4096] 0.5*Student-t(4),
weight [11008, 4096]) against the FP4 MMA rate measured in the same run, the
W4A16/W4A4 crossover sweep and the other library calls.

--impl reference times the CPU oracle (test infrastructure) on a bounded
sample of the same workload.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

N_DEC = K_DEC = 4096
DECODE_M = synth.DECODE_M
METRIC = "NVFP4 linear: W4A16 GB/s (M<=48), W4A4 TFLOPS (M>48), % of roofline"
WORKLOAD = "decode-shaped NVFP4 linear: W[4096,4096] bf16 N(0,0.02^2) 0.5% outliers x8, " \
           "FourOverSix-quantised once; linear (W4A16) at M in {1,2,4,8,16,32,48}"
ROT_SLOTS = 64           # quantised-weight slots (9.4 MB each)
ROT_W = 12               # bf16 weight copies (32 MB each)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


FP4_PER_BF16 = 13.5 / 2.25   # nominal dense FP4 : bf16 tensor rate


def fp4_peaks():
    """(burst, sustained) dense FP4 TFLOP/s: the measured bf16 peaks times the
    nominal FP4/bf16 ratio (the file holds no FP4 figure), and their source."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["bf16_tflops"]) * FP4_PER_BF16, float(p["bf16_tflops_sustained"]) * FP4_PER_BF16,
                "measured bf16 (MEASURED_PEAKS.json bf16_tflops, bf16_tflops_sustained) x 6")
    except Exception:
        return 1900.0 * FP4_PER_BF16, 1700.0 * FP4_PER_BF16, "fallback bf16 1.9 / 1.7 PFLOP/s x 6"


def q_bytes(N, K):   # quantiser: bf16 read once + codes + MMA scales written
    return N * K * 2 + N * K // 2 + N * K // 16


def w4a16_bytes(M, N, K):   # weights (codes + scales) + X + Y
    return N * K // 2 + N * K // 16 + M * K * 2 + M * N * 2


def actq_bytes(M, K):
    return M * K * 2 + M * K // 2 + M * K // 16


def w4a4_bytes(M, N, K):
    return N * K // 2 + N * K // 16 + M * K // 2 + M * K // 16 + M * N * 2


# ------------------------------------------------------------- clock sampler

class ClockSampler:
    FIELDS = "clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap,power.draw"

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- our arm ---

def traffic_from_profiles(kernel_key: str, src_files: dict):
    """DRAM bytes per launch of `kernel_key` from the committed ncu summary, or
    None when the summary is missing or was taken on a different source: the
    summary holds source_sha_<tag> for every {tag: source file} given."""
    path = os.path.join(ROOT, "profiles", f"{kernel_key}.traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.strip().split("=", 1)
                    kv[k.strip()] = v.strip()
        for tag, src_file in src_files.items():
            with open(src_file, "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()[:16]
            if kv.get(f"source_sha_{tag}") != sha:
                return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def max_over_ranks(x: float, dev) -> float:
    """The largest x over all ranks (the replicas' common clock: the job is as
    slow as its slowest replica); x itself without a process group."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(step_bytes: int, steps: int, world: int, elapsed: float) -> float:
    """Whole-job GB/s of `world` replicas that each ran `steps` steps of
    `step_bytes` in at most `elapsed` seconds."""
    return step_bytes * steps * world / elapsed / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import nvfp4_weight_quantized_gb300 as nv
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()

    hbm_peak, _, peak_src = peaks()
    N, K = N_DEC, K_DEC
    w_bits = synth.decode_weight()
    W0 = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    Ws = [W0] + [W0.clone() for _ in range(ROT_W - 1)]
    q0 = nv.nvfp4_quantize_fos(W0, logical_scales=False, choice=True)
    m4_fraction = float(q0.m4_count.item()) / (N * K // 16)
    slots = [nv.NVFP4Weight(q0.codes.clone(), q0.scales_mma.clone(), q0.tensor_scale.clone(), N, K)
             for _ in range(ROT_SLOTS)]
    qws = torch.empty(nv.nvfp4_workspace_bytes(nv.OP_QUANTIZE_FOS, 0, N, K), dtype=torch.uint8, device=dev)
    Xs = {M: torch.from_numpy(synth.decode_act(M).view(np.int16)).view(torch.bfloat16).to(dev)
          for M in DECODE_M}
    Ys = {M: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in DECODE_M}
    lws = {M: torch.empty(max(nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, N, K), 256), dtype=torch.uint8,
                          device=dev) for M in DECODE_M}
    # weights are quantised once per slot and only read by the GEMMs (the
    # quantiser of the whole-path step writes slots no GEMM of that step
    # reads), so the GEMMs may start streaming them before the previous
    # kernel ends
    nv.nvfp4_set_weight_prefetch(True)
    cross = nv.nvfp4_get_crossover(N, K)
    paths = {M: ("w4a16" if M <= cross else "w4a4") for M in DECODE_M}
    launches_per_step = sum(1 if paths[M] == "w4a16" else 3 for M in DECODE_M)

    stream = torch.cuda.Stream(device=dev)
    nm = len(DECODE_M)
    steps_per_cycle = ROT_SLOTS // nm            # 9: slot rotation period of the step
    full_per_cycle = ROT_SLOTS // (nm + 1)       # 8: the same for the whole-path step

    def quant_into(slot, src):
        d = slot
        st = nv.lib().nvfp4_quantize_fos(src.data_ptr(), N, K, 0.0, d.codes.data_ptr(), None,
                                         d.scales_mma.data_ptr(), d.tensor_scale.data_ptr(), None, None,
                                         qws.data_ptr(), qws.numel(), stream.cuda_stream)
        assert st == 0, nv.nvfp4_status_string(st)

    def linear(M, slot):
        nv.nvfp4_linear(Xs[M], slot, out=Ys[M], workspace=lws[M], stream=stream)

    def step_ops(s):
        """The timed step: every decode M on its own cold quantised weight."""
        base = (s % steps_per_cycle) * nm
        for j, M in enumerate(DECODE_M):
            linear(M, slots[base + j])

    def full_step_ops(s):
        """The whole path: quantise a bf16 weight, then the same linears."""
        base = (s % full_per_cycle) * (nm + 1)
        quant_into(slots[base], Ws[s % ROT_W])
        for j, M in enumerate(DECODE_M):
            linear(M, slots[base + 1 + j])

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    W_steps = max(args.warmup, 3)
    K_steps = args.steps
    with torch.cuda.stream(stream):
        for s in range(full_per_cycle):  # eager warm-up (also sets kernel attributes)
            full_step_ops(s)
        for s in range(steps_per_cycle):
            step_ops(s)
    stream.synchronize()
    # one graph per position in the slot-rotation cycle, and one graph of a
    # whole cycle (steps_per_cycle consecutive steps, every slot read once)
    # starting at the position the timed region starts at: the timed steps
    # replay whole cycles, then single steps for the remainder
    graphs = [capture(lambda s=s: step_ops(s)) for s in range(steps_per_cycle)]
    p0 = W_steps % steps_per_cycle
    cycle_graph = capture(lambda: [step_ops(p0 + j) for j in range(steps_per_cycle)])
    full_graphs = [capture(lambda s=s: full_step_ops(s)) for s in range(full_per_cycle)]
    # per-kernel graphs (for per-kernel durations): 4 graphs of 16 calls over
    # disjoint slot sets, replayed in turn, so every call reads weights no
    # other call of the last ~600 MB touched (cold, larger than L2)
    reps, nsets = 16, ROT_SLOTS // 16
    g_quant = [capture(lambda k=k: [quant_into(slots[16 * k + i], Ws[(16 * k + i) % ROT_W]) for i in range(reps)])
               for k in range(nsets)]
    g_lin = {M: [capture(lambda M=M, k=k: [linear(M, slots[16 * k + i]) for i in range(reps)])
                 for k in range(nsets)] for M in DECODE_M}
    torch.cuda.synchronize()

    def timed(gs):
        """Seconds per call: the graph set replayed once (warm), then timed."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            for g in gs:
                g.replay()
            e0.record(stream)
            for g in gs:
                g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / len(gs)

    with torch.cuda.stream(stream):
        cycle_graph.replay()  # set-up: the first replay of a graph uploads it
        for s in range(W_steps):
            graphs[s % steps_per_cycle].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        s = W_steps
        while s + steps_per_cycle <= W_steps + K_steps:
            cycle_graph.replay()
            s += steps_per_cycle
        for s in range(s, W_steps + K_steps):
            graphs[s % steps_per_cycle].replay()
        t_end.record(stream)
    t_end.synchronize()
    # per-kernel durations and the whole-path step, still inside the sampled window
    q_avg = statistics.median(timed(g_quant) for _ in range(3)) / reps
    full_s = statistics.median(timed(full_graphs) for _ in range(3))
    lin_avg = {M: statistics.median(timed(g_lin[M]) for _ in range(3)) / reps for M in DECODE_M}
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) * 1e-3, dev)

    lin_bytes = {M: w4a16_bytes(M, N, K) if paths[M] == "w4a16" else actq_bytes(M, K) + w4a4_bytes(M, N, K)
                 for M in DECODE_M}
    step_bytes = sum(lin_bytes.values())
    ms_per_step = elapsed / K_steps * 1e3
    value = replica_value(step_bytes, K_steps, world, elapsed)

    # dominant kernel family of the step: the W4A16 GEMM (every M of the step
    # takes it while the crossover is above 48)
    w16_time = sum(lin_avg[M] for M in DECODE_M if paths[M] == "w4a16")
    w16_bytes = sum(w4a16_bytes(M, N, K) for M in DECODE_M if paths[M] == "w4a16")
    csrc = os.path.join(ROOT, "nvfp4_weight_quantized_gb300", "csrc")
    if w16_time > 0:
        dom = "gemm_w4a16 (w4a16_sk_kernel for M <= 8, w4a16_rf_kernel above)"
        achieved = w16_bytes / w16_time / 1e9
        # DRAM bytes per launch, averaged over the decode M sweep
        traffic = traffic_from_profiles("w4a16_decode", {"sk": os.path.join(csrc, "gemm_w4a16_sk.cu"),
                                                         "rf": os.path.join(csrc, "gemm_w4a16_rf.cu"),
                                                         "frag": os.path.join(csrc, "w4a16_frag.cuh")})
        launches = sum(1 for M in DECODE_M if paths[M] == "w4a16")
    else:
        dom = "gemm_w4a4 (activation quantisation + w4a4 kernels)"
        achieved = step_bytes / sum(lin_avg.values()) / 1e9
        traffic = None
        launches = launches_per_step

    full_bytes = q_bytes(N, K) + step_bytes
    detail = {
        # the W4A16 calls on their own: algorithmic bytes over the summed per-call times
        "w4a16_gbs": round(w16_bytes / w16_time / 1e9, 1) if w16_time > 0 else None,
        "w4a16_frac_hbm": round(w16_bytes / w16_time / 1e9 / hbm_peak, 4) if w16_time > 0 else None,
        # the whole path per step: FourOverSix quantisation of the bf16 weight + the same linears
        "full_step": {"ms_per_step": round(full_s * 1e3, 5), "gbs": round(full_bytes / full_s / 1e9, 1),
                      "bytes_per_step": full_bytes, "launches_per_step": launches_per_step + 2,
                      "timing": f"{full_per_cycle} CUDA graphs (one per slot-rotation position), "
                                "replayed once warm then timed, median of 3"},
        "quantize_fos_us": round(q_avg * 1e6, 2),
        "quantize_fos_gbs": round(q_bytes(N, K) / q_avg / 1e9, 1),
        "m4_block_fraction": round(m4_fraction, 4),
        "crossover_m": cross,
        "linear": {str(M): {"path": paths[M], "us": round(lin_avg[M] * 1e6, 2),
                            "gbs": round(lin_bytes[M] / lin_avg[M] / 1e9, 1),
                            "frac_hbm": round(lin_bytes[M] / lin_avg[M] / 1e9 / hbm_peak, 3)}
                   for M in DECODE_M},
    }
    if not args.no_prefill and rank == 0:
        # each detail runs guarded: an exception is reported in the line
        fp4_peak = guarded(lambda nv_, dev_, stream_: fp4_peak_measured(nv_), nv, dev, stream)
        if not isinstance(fp4_peak, dict) or "tflops" not in fp4_peak:
            detail["fp4_peak"], fp4_peak = fp4_peak, None
        detail["w4a4_prefill"] = guarded(lambda nv_, dev_, stream_: prefill_sweep(nv_, dev_, stream_, fp4_peak),
                                         nv, dev, stream)
        for key, fn in (("crossover", crossover_sweep), ("model_quantizer", model_quantizer),
                        ("act_fos", act_fos_compare), ("gate_up_silu_mul", gate_up_bench),
                        ("qat_step", qat_bench), ("gptq_fos", gptq_bench), ("mlp_decode", mlp_decode_bench)):
            detail[key] = guarded(fn, nv, dev, stream)

    e2e = measure_e2e(nv, dev, stream, q0, args, step_bytes) if rank == 0 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(sample_rows=args.cpu_rows)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K_steps,
        "warmup": W_steps, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1)+e4m3 weights, bf16 act, fp32 acc",
        "data": "synthetic (seeded numpy PCG64), stands in for real model weights and prompts",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(DECODE_M),
                   "parallelism": f"replicas x{world} (no collective)",
                   "l2": f"inputs larger than L2: {ROT_SLOTS} quantised weight slots rotate, "
                         f"{nm * steps_per_cycle} of them in the step (about "
                         f"{nm * steps_per_cycle * 9437184 / 1e9:.2f} GB)",
                   "timing": f"CUDA graphs of {steps_per_cycle} steps (then of one step for the remainder), "
                             "CUDA events on the launching stream around the replays; "
                  "per-kernel durations from 4 graphs x 16 calls over disjoint cold weight slots"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "launches_per_step": launches},
        "gpu_launches": launches_per_step * K_steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "detail": detail,
    }
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


def fp4_peak_measured(nv):
    """The block-scaled FP4 MMA rate of this GPU from the library's own MMA
    stream (nvfp4_measure_fp4_mma: one CTA pair per two SMs, operands in
    shared memory, no memory traffic): the best of three runs after a
    warm-up, with the clock it ran at."""
    nv.nvfp4_measure_fp4_mma(2000)
    runs = [nv.nvfp4_measure_fp4_mma(20000) for _ in range(3)]
    best = max(runs, key=lambda r: r["tflops"])
    return {"tflops": round(best["tflops"], 1), "pairs": best["pairs"], "sm_mhz": round(best["sm_mhz"]),
            "runs_tflops": [round(r["tflops"], 1) for r in runs],
            "source": "measured: nvfp4_measure_fp4_mma, 20000 x 4 MMAs of 256x256x64 per CTA pair, "
                      "no memory traffic (best of 3)"}


def prefill_sweep(nv, dev, stream, fp4_peak=None):
    """W4A4 GEMM TFLOPS on the prefill workload (graph of 5 launches each),
    as a fraction of the measured FP4 MMA rate (and, as context, of the
    measured bf16 peaks times the nominal FP4 : bf16 ratio)."""
    import torch
    N, K = 11008, 4096
    wp = torch.from_numpy(synth.prefill_weight().view(np.int16)).view(torch.bfloat16).to(dev)
    qp = nv.nvfp4_quantize_fos(wp, logical_scales=False, choice=False)
    res = {}
    burst, sustained, src = fp4_peaks()
    for M in synth.PREFILL_M:
        X = torch.from_numpy(synth.prefill_act(M).view(np.int16)).view(torch.bfloat16).to(dev)
        a = nv.nvfp4_quantize_act(X)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()  # made on the default stream, used on `stream`
        reps = 5 if M >= 1024 else 20
        with torch.cuda.stream(stream):
            for _ in range(2):
                nv.nvfp4_gemm_w4a4(a, qp, out=Y, stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                nv.nvfp4_gemm_w4a4(a, qp, out=Y, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / reps
        tf = 2 * M * N * K / t / 1e12
        row = {"gemm_us": round(t * 1e6, 1), "tflops": round(tf, 1),
               "frac_fp4_burst_x6": round(tf / burst, 3), "frac_fp4_sustained_x6": round(tf / sustained, 3)}
        if fp4_peak:
            row["frac_fp4_measured"] = round(tf / fp4_peak["tflops"], 3)
        res[str(M)] = row
    res["fp4_peak_tflops"] = {"measured": fp4_peak, "burst_x6": round(burst, 1), "sustained_x6": round(sustained, 1),
                              "x6_source": src}
    return res


def crossover_sweep(nv, dev, stream):
    """The W4A16 / W4A4 crossover of nvfp4_linear on this GPU: both paths
    graph-timed over M = 1 .. 256 on the decode, prefill and MLP weight
    shapes (cold weights, weight prefetch on), the largest M where W4A16 is
    still faster, and the built-in table's entry beside it."""
    from nvfp4_weight_quantized_gb300 import tune
    out = {}
    saved = nv.nvfp4_get_weight_prefetch()
    nv.nvfp4_set_weight_prefetch(True)
    try:
        for N, K in ((4096, 4096), (11008, 4096), (22016, 4096), (4096, 11008)):
            times = tune.measure(N, K)
            out[f"{N}x{K}"] = {
                "measured_crossover_m": tune.crossover_from(times), "table_crossover_m": nv.nvfp4_get_crossover(N, K),
                "us": {str(M): [round(t16 * 1e6, 2), round(t4 * 1e6, 2)] for M, (t16, t4) in sorted(times.items())},
                "us_columns": ["w4a16", "act quant + w4a4"]}
    finally:
        nv.nvfp4_set_weight_prefetch(bool(saved))
    return out


def act_fos_compare(nv, dev, stream, M=1024):
    """FourOverSix for activations against the M=6-only rule on the prefill
    workload (W [11008, 4096], X [M, 4096] 0.5 * Student-t(4)): normwise error
    of the W4A4 output against W4A16 on the unquantised activations (same
    quantised weight, so the difference is the activation quantisation), the
    M=4 block fraction, and the quantiser's cost (graph of 10 calls each)."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    qp = nv.nvfp4_quantize_fos(bf(synth.prefill_weight()), logical_scales=False, choice=False)
    X = bf(synth.prefill_act(M))
    torch.cuda.synchronize()  # inputs were made on the default stream
    with torch.cuda.stream(stream):
        y16 = nv.nvfp4_gemm_w4a16(X, qp, nv.OUT_F32, stream=stream).double()
        a6 = nv.nvfp4_quantize_act(X, stream=stream)
        y6 = nv.nvfp4_gemm_w4a4(a6, qp, nv.OUT_F32, stream=stream).double()
        q4 = nv.nvfp4_quantize_fos(X, logical_scales=False, choice=True, stream=stream)
        a4 = nv.NVFP4Act(codes=q4.codes, scales_mma=q4.scales_mma, tensor_scale=q4.tensor_scale, M=M, K=X.shape[1])
        y4 = nv.nvfp4_gemm_w4a4(a4, qp, nv.OUT_F32, stream=stream).double()
    stream.synchronize()
    ref = torch.linalg.norm(y16)
    err6 = float(torch.linalg.norm(y6 - y16) / ref)
    err4 = float(torch.linalg.norm(y4 - y16) / ref)
    m4 = float(q4.choice.float().mean())

    def timed(fn, reps=10):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    t6 = timed(lambda: nv.nvfp4_quantize_act(X, stream=stream))
    t4 = timed(lambda: nv.nvfp4_quantize_fos(X, logical_scales=False, choice=False, stream=stream))
    # the same two quantisers as one cooperative launch each (read once, grid barrier)
    saved = nv.nvfp4_get_single_launch_quantizer()
    nv.nvfp4_set_single_launch_quantizer(True)
    try:
        t6s = timed(lambda: nv.nvfp4_quantize_act(X, stream=stream))
        t4s = timed(lambda: nv.nvfp4_quantize_fos(X, logical_scales=False, choice=False, stream=stream))
    finally:
        nv.nvfp4_set_single_launch_quantizer(saved)
    return {"M": M, "rel_err_m6": round(err6, 5), "rel_err_fos": round(err4, 5), "m4_block_fraction": round(m4, 4),
            "quant_us_m6": round(t6 * 1e6, 2), "quant_us_fos": round(t4 * 1e6, 2),
            "quant_us_m6_single_launch": round(t6s * 1e6, 2), "quant_us_fos_single_launch": round(t4s * 1e6, 2),
            "error": "||Y_w4a4 - Y_w4a16||_F / ||Y_w4a16||_F, same quantised weight"}


def gate_up_bench(nv, dev, stream):
    """Gated MLP projection silu(X W_gate^T) * (X W_up^T) on the MLP
    gate/up weight [2 x 11008, 4096] (N(0, 0.02^2) x per-row lognormal(0, 0.5)):
    nvfp4_linear_silu_mul against nvfp4_linear on the same weight (Y [M, 2F]),
    4 weight copies rotating so that reads are cold: M <= 8 takes W4A16 and
    the separate silu kernel, M = 32 / 48 single-CTA W4A4 with silu(G) * U in
    its epilogue, prefill M the CTA-pair kernel with it in its epilogue.  At
    prefill M also the separate form (fp32 output: GEMM to fp32 in 1024-row
    chunks, then the silu kernel) and the fused form on single CTAs."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    gate_up, _ = synth.mlp_weights()
    q = nv.nvfp4_quantize_fos(bf(gate_up), logical_scales=False, choice=False)
    N, K = q.N, q.K
    copies = [q] + [nv.NVFP4Weight(q.codes.clone(), q.scales_mma.clone(), q.tensor_scale.clone(), N, K)
                     for _ in range(3)]
    torch.cuda.synchronize()  # made on the default stream, used on `stream`

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            fn(0)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    res = {}
    for M in (1, 8, 32, 48, 4096, 16384):
        X = bf(synth.prefill_act(M) if M > 64 else synth.decode_act(M))
        Y1 = torch.empty((M, N // 2), dtype=torch.bfloat16, device=dev)
        Y2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws1 = torch.empty(nv.nvfp4_workspace_bytes(nv.OP_LINEAR_SILU_MUL, M, N, K), dtype=torch.uint8, device=dev)
        ws2 = torch.empty(max(nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, N, K), 256), dtype=torch.uint8, device=dev)
        reps = 8 if M <= 64 else 3
        t1 = timed(lambda i: nv.nvfp4_linear_silu_mul(X, copies[i % 4], out=Y1, workspace=ws1, stream=stream), reps)
        t2 = timed(lambda i: nv.nvfp4_linear(X, copies[i % 4], out=Y2, workspace=ws2, stream=stream), reps)
        res[str(M)] = {"silu_mul_us": round(t1 * 1e6, 2), "linear_us": round(t2 * 1e6, 2)}
        if M > 64:
            # the separate form, which an fp32 output takes
            Y1f = torch.empty((M, N // 2), dtype=torch.float32, device=dev)
            t3 = timed(lambda i: nv.nvfp4_linear_silu_mul(X, copies[i % 4], nv.OUT_F32, out=Y1f, workspace=ws1,
                                                          stream=stream), reps)
            # the fused form on single CTAs (CTA pairs off)
            saved = nv.nvfp4_get_w4a4_cluster()
            nv.nvfp4_set_w4a4_cluster(1)
            try:
                t4 = timed(lambda i: nv.nvfp4_linear_silu_mul(X, copies[i % 4], out=Y1, workspace=ws1,
                                                              stream=stream), reps)
            finally:
                nv.nvfp4_set_w4a4_cluster(saved)
            res[str(M)]["silu_mul_separate_fp32_us"] = round(t3 * 1e6, 2)
            res[str(M)]["silu_mul_single_cta_us"] = round(t4 * 1e6, 2)
            res[str(M)]["silu_mul_tflops"] = round(2 * M * N * K / t1 / 1e12, 1)
            del Y1f
        del ws1, ws2, Y1, Y2, X
    return res


def mlp_decode_bench(nv, dev, stream):
    """The MLP-shaped linears at decode sizes (gate/up W [2 x 11008, 4096] and
    down W [4096, 11008], N(0, 0.02^2) x per-row lognormal(0, 0.5);
    X [M, K] ~ N(0, 1), M in {1, 8, 32, 48}): nvfp4_linear with enough weight
    copies to rotate over more than 4x L2, so every call reads cold weights
    (one CUDA graph of one call per copy, replayed once warm, then timed), and
    the share of blocks that keep the M=4 scale on these weights."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    hbm_peak = peaks()[0]
    res = {}
    for name, w in zip(("gate_up", "down"), synth.mlp_weights()):
        q = nv.nvfp4_quantize_fos(bf(w), logical_scales=False, choice=True)
        N, K = q.N, q.K
        wbytes = N * K // 2 + nv.nvfp4_scales_mma_bytes(N, K)
        n_copies = max(4, -(-4 * 126 * 2**20 // wbytes))
        copies = [q] + [nv.NVFP4Weight(q.codes.clone(), q.scales_mma.clone(), q.tensor_scale.clone(), N, K)
                        for _ in range(n_copies - 1)]
        cross = nv.nvfp4_get_crossover(N, K)
        torch.cuda.synchronize()  # made on the default stream, used on `stream`
        row = {"N": N, "K": K, "weight_copies": n_copies, "crossover_m": cross,
               "m4_block_fraction": round(float(q.m4_count.item()) / (N * K // 16), 4)}
        for M in synth.MLP_M:
            X = bf(synth.act_normal(M, K, seed=320 + M))
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, N, K), 256), dtype=torch.uint8,
                             device=dev)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                nv.nvfp4_linear(X, copies[0], out=Y, workspace=ws, stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in copies:
                    nv.nvfp4_linear(X, c, out=Y, workspace=ws, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):  # replay() launches on the current stream
                g.replay()
                e0.record(stream)
                g.replay()
                e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e-3 / n_copies
            path = "w4a16" if M <= cross else "w4a4"
            nbytes = w4a16_bytes(M, N, K) if path == "w4a16" else actq_bytes(M, K) + w4a4_bytes(M, N, K)
            row[str(M)] = {"path": path, "us": round(t * 1e6, 2), "gbs": round(nbytes / t / 1e9, 1),
                           "frac_hbm": round(nbytes / t / 1e9 / hbm_peak, 3)}
            del g, X, Y, ws
        res[name] = row
        del copies, q
        torch.cuda.synchronize()
    return res


def guarded(fn, *args):
    """fn(*args), or {"exception": ...} if it raises: a failing detail
    measurement is reported in the JSON line instead of ending the run."""
    try:
        return fn(*args)
    except Exception as e:  # noqa: BLE001
        return {"exception": f"{type(e).__name__}: {e}"}


def qat_bench(nv, dev, stream, M=4096):
    """One quantisation-aware training step of the prefill linear (W [11008,
    4096], X [M, 4096]): the FP4 forward (activation quantisation + W4A4,
    weight quantised once) and the straight-through backward (W_hat^T and
    X_hat^T dequantised, dY^T transposed, dX = dY W_hat and dW = dY^T X_hat on
    the library's bf16 tensor-core GEMM), in CUDA graphs; the backward's
    TFLOP/s (its two GEMMs' flops over the whole call) against the measured
    sustained bf16 peak."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    qp = nv.nvfp4_quantize_fos(bf(synth.prefill_weight()), logical_scales=False, choice=False)
    N, K = qp.N, qp.K
    X = bf(synth.prefill_act(M))
    dY = (torch.randn(M, N, device=dev, generator=torch.Generator(device=dev).manual_seed(7))).to(torch.bfloat16)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    A = nv.nvfp4_quantize_act(X)
    torch.cuda.synchronize()  # made on the default stream, used on `stream`

    def fwd():
        nv.nvfp4_gemm_w4a4(nv.nvfp4_quantize_act(X, stream=stream), qp, out=Y, stream=stream)

    def bwd():
        nv.nvfp4_qat_backward(dY, qp, A, stream=stream)

    def timed(fn, reps=5):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    tf, tb = timed(fwd), timed(bwd)
    fl = 2.0 * M * N * K
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_sus, src = float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        bf16_sus, src = 1700.0, "fallback"
    return {"M": M, "N": N, "K": K, "forward_us": round(tf * 1e6, 1), "forward_tflops": round(fl / tf / 1e12, 1),
            "backward_us": round(tb * 1e6, 1), "backward_tflops": round(2 * fl / tb / 1e12, 1),
            "backward_frac_bf16_sustained": round(2 * fl / tb / 1e12 / bf16_sus, 3),
            "bf16_sustained_tflops": bf16_sus, "peak_source": src,
            "timing": "CUDA graph of 5 calls each, CUDA events"}


def gptq_bench(nv, dev, stream, T=4096):
    """GPTQ inside FourOverSix scales on the decode weight [4096, 4096] with a
    synthetic Hessian H = 2 X^T X / T (X: T tokens of N(0, 1) features, the
    first quarter of the features x3), as an offline step: its time, and the
    layer error tr(dW H dW^T) of its codes relative to FourOverSix
    round-to-nearest with the same scales (dW = W - W_hat, binary64)."""
    import torch
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    W = bf(synth.decode_weight())
    N, K = W.shape
    g = torch.Generator(device=dev).manual_seed(11)
    X = torch.randn(T, K, device=dev, generator=g)
    X[:, : K // 4] *= 3.0
    H = (2.0 / T) * (X.t() @ X)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        q = nv.nvfp4_gptq_fos(W, H, stream=stream)  # warm
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q = nv.nvfp4_gptq_fos(W, H, stream=stream)
        e1.record(stream)
        f = nv.nvfp4_quantize_fos(W, stream=stream)
    e1.synchronize()
    assert nv.nvfp4_get_device_status(stream) == 0

    e2 = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0, -0.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64, device=dev)
    e4 = torch.tensor([((b >> 3) & 15 and (1 + (b & 7) / 8.0) * 2.0 ** (((b >> 3) & 15) - 7)) or (b & 7) / 8.0 * 2 ** -6
                       for b in range(128)], dtype=torch.float64, device=dev)

    def dequant(codes, scales, ts):
        c = codes.long()
        v = e2[torch.stack([c & 15, c >> 4], dim=-1).reshape(N, K)]
        return v * e4[scales.long()].repeat_interleave(16, dim=1) * float(ts.item())

    W64, H64 = W.double(), H.double()

    def layer_err(wq):
        d = W64 - wq
        return float(((d @ H64) * d).sum())
    eg = layer_err(dequant(q.codes, q.scales, q.tensor_scale))
    er = layer_err(dequant(f.codes, f.scales, f.tensor_scale))
    return {"N": N, "K": K, "tokens": T, "ms": round(e0.elapsed_time(e1), 2),
            "layer_err_gptq_over_rtn": round(eg / er, 4),
            "scales_equal_fos": bool(torch.equal(q.scales, f.scales))}


def model_quantizer(nv, dev, stream, layers=32, distinct=2):
    """Whole-model quantiser throughput: a 32-layer stack (qkv 6144x4096, o
    4096x4096, gate/up 22016x4096, down 4096x11008; N(0, 0.02^2), 0.5 %
    outliers x8) quantised one matrix at a time, inputs resident.  `distinct`
    layers are generated on the device from seeded generators (each larger
    than L2) and reused in turn; the timed region is one CUDA graph of all
    4 * layers FourOverSix quantisations.  Reports GB/s of bf16 read, the
    fraction of HBM on the quantiser's algorithmic bytes, and the fraction of
    blocks that chose M=4."""
    import torch
    shapes = [(N, K) for _, N, K in synth.MODEL_LAYER_SHAPES]
    gen = torch.Generator(device=dev)
    ws = []
    for li in range(distinct):
        mats = []
        for wi, (N, K) in enumerate(shapes):
            gen.manual_seed(500 + 4 * li + wi)
            w = torch.randn(N, K, device=dev, generator=gen) * 0.02
            w = torch.where(torch.rand(N, K, device=dev, generator=gen) < 0.005, w * 8, w)
            mats.append(w.to(torch.bfloat16))
            del w
        ws.append(mats)
    outs = []
    for N, K in shapes:
        outs.append((torch.empty(N * K // 2, dtype=torch.uint8, device=dev),
                     torch.empty(nv.nvfp4_scales_mma_bytes(N, K), dtype=torch.uint8, device=dev),
                     torch.empty(1, dtype=torch.float32, device=dev)))
    wsb = max(nv.nvfp4_workspace_bytes(nv.OP_QUANTIZE_FOS, 0, N, K) for N, K in shapes)
    qws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    m4 = torch.zeros(1, dtype=torch.int64, device=dev)

    def quant(w, o, N, K, count):
        st = nv.lib().nvfp4_quantize_fos(w.data_ptr(), N, K, 0.0, o[0].data_ptr(), None, o[1].data_ptr(),
                                         o[2].data_ptr(), None, m4.data_ptr() if count else None, qws.data_ptr(),
                                         qws.numel(), stream.cuda_stream)
        assert st == 0, nv.nvfp4_status_string(st)

    # the layers and the counter were made on the default stream
    torch.cuda.synchronize()
    # fraction of M=4 blocks over the distinct layers (outside the timed region)
    n4, nblk = 0, 0
    with torch.cuda.stream(stream):
        for mats in ws:
            for w, o, (N, K) in zip(mats, outs, shapes):
                quant(w, o, N, K, True)
                stream.synchronize()
                n4 += int(m4.item())
                nblk += N * K // 16
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for li in range(layers):
            for w, o, (N, K) in zip(ws[li % distinct], outs, shapes):
                quant(w, o, N, K, False)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) * 1e-3
    elems = layers * sum(N * K for N, K in shapes)
    qb = layers * sum(q_bytes(N, K) for N, K in shapes)
    hbm_peak = peaks()[0]
    del ws, g
    torch.cuda.empty_cache()
    return {"layers": layers, "params": elems, "ms": round(t * 1e3, 3),
            "gbs_bf16_read": round(2 * elems / t / 1e9, 1), "frac_hbm": round(qb / t / 1e9 / hbm_peak, 3),
            "m4_block_fraction": round(n4 / nblk, 4),
            "inputs": f"{distinct} distinct layers generated on the device (torch, seeded), reused in turn"}


def measure_e2e(nv, dev, stream, q, args, step_bytes):
    """The same step through the public API with host buffers: every step
    copies each linear's quantised weight (codes, MMA-tiled scales, tensor
    scale; one weight per M, as in the device-resident step) and its
    activations from pinned host memory, runs nvfp4_linear, and copies every
    output back, all inside the timed region.  A step's inputs sit in one
    pinned buffer and go over in one host-to-device copy, on a copy stream,
    into one of two device buffers in turn, so the next step's copy overlaps
    this step's calls and its device-to-host read of the outputs."""
    import torch
    N, K = N_DEC, K_DEC
    # the copy of a step writes the weights its GEMMs read: no GEMM may start
    # streaming its weight before the kernel ahead of it has finished
    nv.nvfp4_set_weight_prefetch(False)
    align = lambda n: (n + 1023) // 1024 * 1024  # noqa: E731
    parts = [q.codes, q.scales_mma, q.tensor_scale]
    seg_w = [align(t.numel() * t.element_size()) for t in parts]
    offs, o = {}, 0
    for M in DECODE_M:
        offs[M] = o
        o += sum(seg_w) + align(M * K * 2)
    h_in = torch.empty(o, dtype=torch.uint8).pin_memory()
    d_in = [torch.empty(o, dtype=torch.uint8, device=dev) for _ in range(2)]
    y_off, yo = {}, 0
    for M in DECODE_M:
        y_off[M] = yo
        yo += M * N * 2
    h_out = [torch.empty(yo, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_out = [torch.empty(yo, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, off, t):
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    w = [{}, {}]
    X = [{}, {}]
    Y = [{}, {}]
    for M in DECODE_M:
        xh = torch.from_numpy(synth.decode_act(M).view(np.int16)).view(torch.bfloat16)
        o = offs[M]
        for t, n in zip(parts, seg_w):
            view(h_in, o, t).copy_(t.cpu())
            o += n
        view(h_in, o, xh).copy_(xh)
        for b in range(2):
            o = offs[M]
            views = []
            for t, n in zip(parts, seg_w):
                views.append(view(d_in[b], o, t))
                o += n
            w[b][M] = nv.NVFP4Weight(views[0], views[1], views[2], N, K)
            X[b][M] = view(d_in[b], o, xh)
            Y[b][M] = d_out[b][y_off[M]:y_off[M] + M * N * 2].view(torch.bfloat16).view(M, N)
    lws = {M: torch.empty(max(nv.nvfp4_workspace_bytes(nv.OP_LINEAR, M, N, K), 256), dtype=torch.uint8,
                          device=dev) for M in DECODE_M}
    h2d, d2h = h_in.numel(), h_out[0].numel()
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):
        done[b].record(stream)

    def step(i):
        b = i % 2
        copy_stream.wait_event(done[b])  # the buffer's previous step is over
        with torch.cuda.stream(copy_stream):
            d_in[b].copy_(h_in, non_blocking=True)
            copied[b].record(copy_stream)
        stream.wait_event(copied[b])
        with torch.cuda.stream(stream):
            for M in DECODE_M:
                nv.nvfp4_linear(X[b][M], w[b][M], out=Y[b][M], workspace=lws[M], stream=stream)
            h_out[b].copy_(d_out[b], non_blocking=True)
            done[b].record(stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for b in range(2):
        done[b].record(stream)  # the timed copies start after e0
    for i in range(args.steps):
        step(i)
    e1.record(stream)  # after the last step's outputs are back (its copy came before its calls)
    e1.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / args.steps
    return {"value": round(step_bytes / t / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(t * 1e3, 4),
            "pipelining": "two device input buffers: a step's host-to-device copy overlaps the previous "
                          "step's calls and output read-back"}


# ------------------------------------------------------------ CPU oracle ---

def cpu_prepare(sample_rows: int):
    """The oracle's inputs for a sample of the decode workload: the first
    `sample_rows` weight rows FourOverSix-quantised (tensor scale from the
    whole tensor; done once, like the weight of the timed step) and the
    activations of every M."""
    import oracle
    w = synth.decode_weight()
    ts = oracle.tensor_scale(w)
    q = oracle.quantize_rows(w[:sample_rows], ts, True)
    return {"rows": sample_rows, "ts": ts, "q": q, "xs": {M: synth.decode_act(M) for M in DECODE_M}}


def cpu_step(prep: dict, threads: int = 1):
    """One bounded oracle pass over a prepared sample: those output columns
    of every linear (binary64 reference GEMM), the rows split over `threads`
    threads (independent oracle calls; each releases the GIL).  Returns
    (seconds, algorithmic bytes of the sampled share of the step)."""
    import concurrent.futures as cf
    import oracle
    rows, q, xs, ts = prep["rows"], prep["q"], prep["xs"], prep["ts"]
    bounds = np.linspace(0, rows, threads + 1).astype(int)

    def gemms(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        for M in DECODE_M if a < b else ():
            oracle.gemm_w4a16(xs[M], q["codes"][a:b], q["scales"][a:b], ts)

    t0 = time.perf_counter()
    if threads == 1:
        gemms(0)
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(gemms, range(threads)))
    dt = time.perf_counter() - t0
    frac = rows / N_DEC
    return dt, sum(w4a16_bytes(M, N_DEC, K_DEC) * frac for M in DECODE_M)


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline(sample_rows: int = 1024):
    """The oracle on the host: single thread on a sample of the step (the
    reported figure), and, beside it, the whole step split over every core."""
    dt, nbytes = cpu_step(cpu_prepare(sample_rows))
    out = {"value": round(nbytes / dt / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{sample_rows} of 4096 weight rows (quantised once beforehand): those output "
                     f"columns for every M (binary64 reference GEMM), single thread, {dt:.1f} s"}
    cores = host_cores()
    if cores > 1:
        dt_all, nb_all = cpu_step(cpu_prepare(N_DEC), threads=cores)
        out["all_cores"] = {"value": round(nb_all / dt_all / 1e9, 6), "unit": "GB/s", "cores": cores,
                            "sample": f"the whole step (4096 weight rows) split by weight row over {cores} "
                                      f"threads, {dt_all:.1f} s"}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows = args.cpu_rows_reference
    prep = cpu_prepare(rows)
    for _ in range(args.warmup):
        cpu_step(prep)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, nbytes = cpu_step(prep)
        times.append(dt)
    t = sum(times)
    value = nbytes * args.steps / t / 1e9
    sample = f"{rows} of 4096 weight rows per step (quantised once beforehand; every M of the binary64 GEMM), " \
             "single thread"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "N": N_DEC, "K": K_DEC, "M": list(DECODE_M)},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def profile_case(which: str, m_decode: int):
    """One launch of each hot kernel on a small case, for a profiler capture:
    the FourOverSix quantiser and W4A16 at M = m_decode on the decode weight
    [4096, 4096], activation quantisation + W4A4 at M = 2048 on the prefill
    weight [11008, 4096].  Prints the device status; times nothing."""
    import torch
    import nvfp4_weight_quantized_gb300 as nv
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    dev = torch.device("cuda")
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    if which in ("all", "quant", "w4a16"):
        q = nv.nvfp4_quantize_fos(bf(synth.decode_weight()), logical_scales=False, choice=False)
        if which in ("all", "w4a16"):
            nv.nvfp4_gemm_w4a16(bf(synth.decode_act(m_decode)), q)
    if which in ("all", "w4a4"):
        qp = nv.nvfp4_quantize_fos(bf(synth.prefill_weight()), logical_scales=False, choice=False)
        a = nv.nvfp4_quantize_act(bf(synth.prefill_act(2048)))
        nv.nvfp4_gemm_w4a4(a, qp)
    if which == "w4a4_small":  # single-CTA W4A4 (M <= 128) on the prefill weight
        qp = nv.nvfp4_quantize_fos(bf(synth.prefill_weight()), logical_scales=False, choice=False)
        a = nv.nvfp4_quantize_act(bf(synth.prefill_act(m_decode)))
        nv.nvfp4_gemm_w4a4(a, qp)
    if which == "gate_up":  # the gated MLP projection, fused form, on the gate/up weight [2 x 11008, 4096]
        qg = nv.nvfp4_quantize_fos(bf(synth.mlp_weights()[0]), logical_scales=False, choice=False)
        nv.nvfp4_linear_silu_mul(bf(synth.prefill_act(2048)), qg)
    if which == "qat":  # straight-through backward on the prefill weight [11008, 4096], M = 2048
        qp = nv.nvfp4_quantize_fos(bf(synth.prefill_weight()), logical_scales=False, choice=False)
        a = nv.nvfp4_quantize_act(bf(synth.prefill_act(2048)))
        g = torch.Generator(device=dev).manual_seed(7)
        dY = torch.randn((2048, 11008), device=dev, generator=g).bfloat16()
        nv.nvfp4_qat_backward(dY, qp, a)
    if which == "w4a16_any":  # a K that is a multiple of 16 but not of 64: [4096, 4080], M = m_decode
        qa = nv.nvfp4_quantize_fos(bf(synth.decode_weight()[:, :4080].copy()), logical_scales=False,
                                   choice=False)
        nv.nvfp4_gemm_w4a16(bf(synth.decode_act(m_decode)[:, :4080].copy()), qa)
    if which == "fp4_rate":  # the FP4 MMA rate kernel, 2000 x 4 MMAs per CTA pair
        nv.nvfp4_measure_fp4_mma(2000)
    torch.cuda.synchronize()
    print("profile case", which, "status", nv.nvfp4_status_string(nv.nvfp4_get_device_status()))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--cpu-rows-reference", type=int, default=64)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["all", "quant", "w4a16", "w4a4", "w4a4_small", "gate_up", "qat",
                                                "w4a16_any", "fp4_rate"],
                    help="launch each hot kernel once on a small case (for ncu) and exit")
    ap.add_argument("--profile-m", type=int, default=16, help="decode M of --profile-case (and M of w4a4_small)")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case, args.profile_m)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
