"""Throughput of the RT-Lynx 2:4 activation-sparse linear on the attention QKV
projection of a single-stream DiT at 1024 px: X 4608 x 3072 bf16 (4096 image +
512 text tokens), W 9216 x 3072, rank-64 LoRA.

A step is one lynx_linear call: the fused sparsify + LoRA down-projection pass
over X, and the tcgen05 2:4-sparse GEMM with the LoRA-up accumulation and the
s epilogue.
The metric is effective TFLOP/s = 2 M N K / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
bounded row samples of the same workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = ("qkv", "qkv")
METRIC = "effective TFLOP/s (2MNK) of fused sparse linear; % of sparse BF16 peak; x vs dense"
ROTATE = 4          # device copies of the inputs, cycled so that each step reads cold (L2-evicted) data
PROFILE_EVERY = 8   # timed steps between two that carry the per-stage events
FALLBACK_PEAKS = {"hbm_gbs": 6682.8, "bf16_tflops": 1967.9, "bf16_tflops_sustained": 1755.1,
                  "source": "pool measurement recorded before this run (STREAM copy, cuBLAS bf16 8192^3)"}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d.setdefault("source", "MEASURED_PEAKS.json")
        return d
    return dict(FALLBACK_PEAKS)


def profiled_traffic(profile: str, source: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source is still the one captured."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        src = open(os.path.join(ROOT, "activation_sparse_linear_gb300", "csrc", source), "rb").read()
    except OSError:
        return None
    sha = re.search(r"kernel_source_sha256_prefix:\s*([0-9a-f]+)", text)
    traffic = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    if not sha or not traffic or not hashlib.sha256(src).hexdigest().startswith(sha.group(1)):
        return None
    return int(traffic.group(1))


def peak_value(peaks: dict, *names, default=None):
    for n in names:
        for k, v in peaks.items():
            if k == n and isinstance(v, (int, float)):
                return float(v)
    return default


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 10.0:  # nvidia-smi is up before the timed region starts
            time.sleep(0.02)
        self.skip = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=5)
            self.lines = self.lines[max(0, self.skip - 1):]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_rows_rate(t: dict, rows_per_call: int, budget_s: float, max_calls: int | None = None,
                     threads: int | None = None):
    """Time the plain C++ oracle on consecutive row samples with ``threads`` std::threads (default: every host
    core); returns (TFLOP/s, rows, seconds, calls)."""
    from oracle import cpp
    O = cpp.CppOracle(cpp.build())
    if threads:
        O.threads = threads
    M, N, K = t["M"], t["N"], t["K"]
    done_rows, calls, t0 = 0, 0, time.perf_counter()
    while True:
        r0 = (calls * rows_per_call) % M
        rows = np.arange(r0, min(r0 + rows_per_call, M))
        O.linear(t["X"], t["W"], t["LA"], t["LB"], rows=rows)
        done_rows += len(rows)
        calls += 1
        el = time.perf_counter() - t0
        if (max_calls is not None and calls >= max_calls) or (max_calls is None and el >= budget_s):
            break
    return 2.0 * done_rows * N * K / el / 1e12, done_rows, el, calls


def host_cores() -> int:
    from oracle import cpp
    return cpp.host_threads()


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def cpu_baseline_leg(t: dict) -> dict:
    """The C++ oracle on bounded row samples of the bench workload: every host core (about 10 s), then one
    thread (about 8 s)."""
    cores = host_cores()
    tf, rows, secs, _ = oracle_rows_rate(t, 8 * cores, 10.0, threads=cores)
    tf1, rows1, secs1, _ = oracle_rows_rate(t, 8, 8.0, threads=1)
    return {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} rows of the QKV workload in {secs:.1f} s on {cores} std::threads "
                      f"(plain C++ double oracle; W, LA, LB widened once per call)",
            "cpu_model": cpu_model(),
            "t1": {"value": tf1, "unit": "TFLOP/s", "threads": 1,
                   "sample": f"{rows1} rows in {secs1:.1f} s on one thread"}}


def oracle_config_timings() -> dict:
    """The plain C++ oracle on the host cores over the five workloads:
    tiny, QKV, MLP (up + down) and the CFG batch (four layers) in full on every core; the block stack at
    M = 1024 in full (32 linears) and extrapolated linearly in M to the larger M; one thread on a row sample of
    each layer, extrapolated to all rows (rows are independent)."""
    import synth
    from oracle import cpp
    O = cpp.CppOracle(cpp.build())
    cores = host_cores()

    def run_layer(t, rows=None, threads=cores):
        O.threads = threads
        t0 = time.perf_counter()
        if t["sparse"]:
            O.linear(t["X"], t["W"], t["LA"], t["LB"], rows=rows)
        else:
            O.linear_dense(t["X"], t["W"], rows=rows)
        return time.perf_counter() - t0

    out = {"cores": cores, "cpu_model": cpu_model(), "configs": {}}
    plans = [("tiny", [("tiny", "linear", None, 0)]), ("qkv", [("qkv", "qkv", None, 0)]),
             ("mlp", [("mlp", "up", None, 0), ("mlp", "down", None, 0)]),
             ("cfg2", [("cfg2", ly, None, 0) for ly in ("qkv", "out", "up", "down")]),
             ("stack M=1024", [("stack", ly, 1024, b) for b in range(8) for ly in ("qkv", "out", "up", "down")])]
    for name, layers in plans:
        secs, secs1, flops = 0.0, 0.0, 0.0
        for wl, ly, M, blk in layers:
            t = synth.layer_tensors(wl, ly, M=M, block=blk)
            secs += run_layer(t)
            sample = np.arange(0, t["M"], max(1, t["M"] // 16))  # 16 rows on one thread
            secs1 += run_layer(t, rows=sample, threads=1) * t["M"] / len(sample)
            flops += 2.0 * t["M"] * t["N"] * t["K"]
        out["configs"][name] = {"seconds": secs, "tflops": flops / secs / 1e12, "seconds_t1_extrapolated": secs1,
                                "tflops_t1": flops / secs1 / 1e12}
    st = out["configs"]["stack M=1024"]
    out["configs"]["stack (extrapolated in M)"] = {f"M={m}": st["seconds"] * m / 1024 for m in (4608, 9216, 16384)}
    return out


def run_reference(args) -> int:
    """The oracle as it stands, on the host cores: each step is one C++ oracle call on a bounded row sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import synth
    t = synth.layer_tensors(*WORKLOAD)
    cores = host_cores()
    rows = 4 * cores
    oracle_rows_rate(t, rows, 0, max_calls=max(1, args.warmup), threads=cores)  # warm-up
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_rows_rate(t, rows, 0, max_calls=1, threads=cores)
        times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    value = 2.0 * rows * t["N"] * t["K"] / step_s / 1e12
    sample = (f"{rows} of {t['M']} rows per step (QKV 4608x3072 -> 9216, rank 64), plain C++ double oracle on "
              f"{cores} std::threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(t, "reference"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(t, impl="lynx"):
    return {"workload": "attention QKV projection, single-stream DiT 1024px: X 4608x3072 bf16 "
                        "(4096 image + 512 text tokens, N(0,1), 3% outlier channels x10), W 9216x3072 "
                        "N(0,1/3072), LoRA rank 64 N(0,0.02), seeded",
            "M": t["M"], "N": t["N"], "K": t["K"], "R": t["R"],
            "l2": f"inputs rotated over {ROTATE} device copies (> L2) so every step reads L2-cold data"
            if impl != "reference" else "n/a (host)"}


# ----------------------------------------------------------------------------- GPU arm
def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lynx", choices=["lynx", "reference"])
    ap.add_argument("--profile-case", default=None, choices=["linear", "fused", "dense", "wsparse"],
                    help="run only W + K calls of lynx_linear / lynx_linear_fused / lynx_linear_dense (no LoRA) / "
                         "lynx_linear_wsparse (W pruned and compressed once, before the calls) on the workload and "
                         "print their mean time: a short command for profilers")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the C++ oracle on the host cores over all five workloads and exit (no GPU work)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.oracle_configs:
        print(json.dumps({"oracle_config_timings": oracle_config_timings()}), flush=True)
        return 0

    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import activation_sparse_linear_gb300 as asl
    import synth

    t = synth.layer_tensors(*WORKLOAD, batch=rank)  # each replica its own batch of tokens, shared weights
    M, N, K, R = t["M"], t["N"], t["K"], t["R"]
    dev = torch.device("cuda", local)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    base = {k: to_dev(t[k]) for k in ("X", "W", "LA", "LB")}
    sets = []
    for i in range(ROTATE):
        sets.append({
            "X": base["X"].clone(), "W": base["W"].clone(), "LA": base["LA"].clone(), "LB": base["LB"].clone(),
            "Y": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
            "ws": torch.empty(asl.lynx_workspace_bytes(M, N, K, R), dtype=torch.uint8, device=dev),
        })
    del base
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    L = asl.lib

    def call(s):
        return L.lynx_linear(s["X"].data_ptr(), s["W"].data_ptr(), s["LA"].data_ptr(), s["LB"].data_ptr(),
                             s["Y"].data_ptr(), M, N, K, R, s["ws"].data_ptr(), s["ws"].numel(), sp)

    if args.profile_case:
        ws_d = torch.empty(asl.lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=dev)
        pruned = {}
        if args.profile_case == "wsparse":
            pruned = {id(s): asl.lynx_prune_weight(s["W"]) for s in sets}
            torch.cuda.synchronize()

        def case(s):
            if args.profile_case == "linear":
                return call(s)
            if args.profile_case == "wsparse":
                wv, wm = pruned[id(s)]
                return L.lynx_linear_wsparse(s["X"].data_ptr(), wv.data_ptr(), wm.data_ptr(), s["LA"].data_ptr(),
                                             s["LB"].data_ptr(), s["Y"].data_ptr(), M, N, K, R, ws_d.data_ptr(),
                                             ws_d.numel(), sp)
            if args.profile_case == "fused":
                return L.lynx_linear_fused(s["X"].data_ptr(), s["W"].data_ptr(), s["LA"].data_ptr(),
                                           s["LB"].data_ptr(), s["Y"].data_ptr(), M, N, K, R, ws_d.data_ptr(),
                                           ws_d.numel(), sp)
            return L.lynx_linear_dense(s["X"].data_ptr(), s["W"].data_ptr(), None, None, s["Y"].data_ptr(), M, N,
                                       K, R, None, 0, sp)
        for i in range(args.warmup):
            assert case(sets[i % ROTATE]) == 0
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(args.steps):
            assert case(sets[i % ROTATE]) == 0
        c1.record(stream)
        torch.cuda.synchronize()
        st = asl.lynx_sync_status()
        assert st == 0, asl.lynx_status_string(st)
        if rank == 0:
            print(json.dumps({"profile_case": args.profile_case, "calls": args.steps,
                              "ms_per_call": c0.elapsed_time(c1) / args.steps}), flush=True)
        return 0

    # warm-up
    for i in range(args.warmup):
        assert call(sets[i % ROTATE]) == 0
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)

    # Per-stage events on every PROFILE_EVERY-th timed step (created up front: torch creates events lazily on
    # first record).  An event recorded between two kernels keeps the next launch from overlapping the
    # previous kernel's tail (about 8 us per step with four events), so the other steps run without them.
    nev = 3
    prof_steps = list(range(0, args.steps, PROFILE_EVERY))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in prof_steps]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    import ctypes
    ev_arrays = [(ctypes.c_void_p * nev)(*[e.cuda_event for e in row]) for row in evs]

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            if i % PROFILE_EVERY == 0:
                L.lynx_profile_next(ev_arrays[i // PROFILE_EVERY], nev)
            if call(sets[i % ROTATE]) != 0:
                raise RuntimeError("lynx_linear failed")
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_per_step = elapsed_ms / args.steps
    flops = 2.0 * M * N * K
    value = flops * args.steps * world / (elapsed_ms * 1e-3) / 1e12

    stage_ms = np.array([[row[j].elapsed_time(row[j + 1]) for j in range(nev - 1)] for row in evs])
    stage_avg = stage_ms.mean(axis=0)  # fused sparsify + LoRA-down pass, sparse GEMM

    peaks = load_peaks()
    dense_tf = peak_value(peaks, "bf16_tflops", "bf16_tflops_burst", default=1967.9)
    hbm = peak_value(peaks, "hbm_gbs", "hbm_GBps", default=6682.8)
    sparse_peak = 2.0 * dense_tf
    gemm_flops = 2.0 * M * N * K + 2.0 * M * N * R  # sparse branch (dense-equivalent) + LoRA-up
    gemm_tf = gemm_flops / (stage_avg[1] * 1e-3) / 1e12
    # algorithmic bytes of the fused pass: X and LB read once; compressed values, metadata, s and T' written
    prologue_bytes = M * K * 2 + R * K * 2 + M * K + M * K / 8 + M * 4 + M * R * 2
    prologue_gbs = prologue_bytes / (stage_avg[0] * 1e-3) / 1e9

    # tensor-core rate of smem-resident back-to-back MMAs (dense vs 2:4 sparse)
    mma_dense_tf, mma_dense_mpc = asl.lynx_mma_rate(0, 20000)
    mma_sparse_tf, mma_sparse_mpc = asl.lynx_mma_rate(1, 20000)
    mma_sparse_cp_tf, _ = asl.lynx_mma_rate(2, 20000)
    mma_sparse_c2_tf, _ = asl.lynx_mma_rate(3, 20000)
    mma_sparse_c4_tf, _ = asl.lynx_mma_rate(4, 20000)
    mma_more = {f"mode{m}": asl.lynx_mma_rate(m, 20000)[0] for m in (5, 6, 7, 8)}

    # dense cuBLAS and this library's dense tcgen05 GEMM (a selectively skipped layer, no LoRA) at the same shape,
    # same rotation, same stream, timed in alternating blocks so that both see the same clocks under the power cap
    def cublas_dense(i):
        s = sets[i % ROTATE]
        torch.matmul(s["X"], s["W"].t(), out=s["Y"])

    def lynx_dense(i):
        s = sets[i % ROTATE]
        if L.lynx_linear_dense(s["X"].data_ptr(), s["W"].data_ptr(), None, None, s["Y"].data_ptr(), M, N, K, R, None,
                               0, sp) != 0:
            raise RuntimeError("lynx_linear_dense failed")

    for i in range(args.warmup):
        cublas_dense(i)
        lynx_dense(i)
    nd_block = max(1, min(args.steps, 500) // 5)
    nd = 5 * nd_block
    t_arm = {"cublas": 0.0, "lynx": 0.0}
    torch.cuda.synchronize()
    for blk in range(5):
        for arm, fn in (("cublas", cublas_dense), ("lynx", lynx_dense)):
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for i in range(nd_block):
                fn(blk * nd_block + i)
            b1.record(stream)
            torch.cuda.synchronize()
            t_arm[arm] += b0.elapsed_time(b1)
    dense_ms = t_arm["cublas"] / nd
    lynx_dense_ms = t_arm["lynx"] / nd

    # The weight-2:4 comparator at the same shape (W pruned and compressed once, outside the timed region):
    # the same sparse tensor-core path with W~ as the sparse operand, with the same rank-64 LoRA branch.
    wpruned = [asl.lynx_prune_weight(sets[i]["W"]) for i in range(ROTATE)]
    ws_w = torch.empty(asl.lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=dev)

    def wsparse(i):
        s = sets[i % ROTATE]
        wv, wm = wpruned[i % ROTATE]
        return L.lynx_linear_wsparse(s["X"].data_ptr(), wv.data_ptr(), wm.data_ptr(), s["LA"].data_ptr(),
                                     s["LB"].data_ptr(), s["Y"].data_ptr(), M, N, K, R, ws_w.data_ptr(),
                                     ws_w.numel(), sp)
    for i in range(args.warmup):
        wsparse(i)
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for i in range(nd):
        if wsparse(i) != 0:
            raise RuntimeError("lynx_linear_wsparse failed")
    l1.record(stream)
    torch.cuda.synchronize()
    wsparse_ms = l0.elapsed_time(l1) / nd
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)

    # The library 2:4 path as shipped: torch's semi-structured sparse GEMM (cuSPARSELt) on the same pruned W, with
    # the algorithm cuSPARSELt's own search picks (context for the weight-2:4 comparator; no LoRA branch).
    cslt = {"unavailable": "not measured"}
    try:
        s0 = sets[0]
        dense_w = torch.empty_like(s0["W"])
        wp = s0["W"].view(N, K // 4, 4)
        keep = wp.abs().float().topk(2, dim=-1).indices
        dense_w.copy_((wp * torch.zeros_like(wp, dtype=torch.bool).scatter_(-1, keep, True)).view(N, K))
        comp = torch._cslt_compress(dense_w)
        alg = None
        cs = getattr(getattr(torch._C, "_cusparselt", None), "mm_search", None)
        if cs is not None:
            try:
                alg = int(cs(comp, s0["X"].t()))
            except Exception:
                alg = None
        if alg is None:
            import warnings
            with warnings.catch_warnings():
                warnings.simplefilter("ignore")  # the older entry point warns that it is deprecated
                alg = int(torch._cslt_sparse_mm_search(comp, s0["X"].t()))
        for i in range(2):
            torch._cslt_sparse_mm(comp, sets[i % ROTATE]["X"].t(), alg_id=alg)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(10):
            torch._cslt_sparse_mm(comp, sets[i % ROTATE]["X"].t(), alg_id=alg)
        c1.record(stream)
        torch.cuda.synchronize()
        cms = c0.elapsed_time(c1) / 10
        cslt = {"ms": cms, "tflops": flops / (cms * 1e-3) / 1e12, "x_vs_dense_cublas": dense_ms / cms,
                "algorithm": alg, "note": "torch._cslt_sparse_mm (cuSPARSELt) with W 2:4-pruned (the two largest |w| "
                                          "of every 4), the algorithm from cuSPARSELt's own search; no LoRA"}
        del comp, dense_w
    except Exception as ex:  # a torch build without cuSPARSELt for this GPU
        cslt = {"unavailable": f"{type(ex).__name__}: {str(ex)[:160]}"}
    del wpruned, ws_w

    # The in-GEMM selection variant (lynx_linear_fused) at the same shape: the LoRA down-projection, then one GEMM
    # whose epilogue warps select the 2:4 pattern of every dense X tile themselves (no sparsify pass).
    ws_f = torch.empty(asl.lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=dev)

    def fused(i):
        s = sets[i % ROTATE]
        return L.lynx_linear_fused(s["X"].data_ptr(), s["W"].data_ptr(), s["LA"].data_ptr(), s["LB"].data_ptr(),
                                   s["Y"].data_ptr(), M, N, K, R, ws_f.data_ptr(), ws_f.numel(), sp)
    for i in range(args.warmup):
        fused(i)
    torch.cuda.synchronize()
    nf = max(4, nd // 4)
    l0.record(stream)
    for i in range(nf):
        if fused(i) != 0:
            raise RuntimeError("lynx_linear_fused failed")
    l1.record(stream)
    torch.cuda.synchronize()
    fused_ms = l0.elapsed_time(l1) / nf
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)
    del ws_f

    # The other layer shapes of the DiT workloads (MLP up/down, the CFG batch, the largest stack M): step time
    # of lynx_linear and of the dense cuBLAS GEMM at the same shape, two rotating device copies each.  Inputs
    # are seeded normal draws generated on the device (timing only; the parity tests cover these shapes).
    shapes = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    for name, (Ms, Ns, Ks) in (("mlp_up 4608x3072->12288", (4608, 12288, 3072)),
                               ("mlp_down 4608x12288->3072", (4608, 3072, 12288)),
                               ("cfg2_qkv 9216x3072->9216", (9216, 9216, 3072)),
                               ("stack_qkv 16384x3072->9216", (16384, 9216, 3072)),
                               ("stack_down 1024x12288->3072", (1024, 3072, 12288))):
        cs = []
        for _ in range(2):
            cs.append({"X": torch.randn((Ms, Ks), generator=gen, device=dev).to(torch.bfloat16),
                       "W": (torch.randn((Ns, Ks), generator=gen, device=dev) / Ks ** 0.5).to(torch.bfloat16),
                       "LA": (0.02 * torch.randn((Ns, R), generator=gen, device=dev)).to(torch.bfloat16),
                       "LB": (0.02 * torch.randn((R, Ks), generator=gen, device=dev)).to(torch.bfloat16),
                       "Y": torch.empty((Ms, Ns), dtype=torch.bfloat16, device=dev),
                       "ws": torch.empty(asl.lynx_workspace_bytes(Ms, Ns, Ks, R), dtype=torch.uint8, device=dev)})

        def one(c):
            return L.lynx_linear(c["X"].data_ptr(), c["W"].data_ptr(), c["LA"].data_ptr(), c["LB"].data_ptr(),
                                 c["Y"].data_ptr(), Ms, Ns, Ks, R, c["ws"].data_ptr(), c["ws"].numel(), sp)
        ns = 100
        times = []
        for fn in (lambda c: one(c), lambda c: torch.matmul(c["X"], c["W"].t(), out=c["Y"])):
            for i in range(5):
                fn(cs[i % 2])
            torch.cuda.synchronize()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for i in range(ns):
                fn(cs[i % 2])
            a1.record(stream)
            torch.cuda.synchronize()
            times.append(a0.elapsed_time(a1) / ns)
        st = asl.lynx_sync_status()
        assert st == 0, asl.lynx_status_string(st)
        fl = 2.0 * Ms * Ns * Ks
        shapes[name] = {"lynx_ms": times[0], "tflops": fl / (times[0] * 1e-3) / 1e12,
                        "pct_of_sparse_peak": 100.0 * fl / (times[0] * 1e-3) / 1e12 / (2.0 * dense_tf),
                        "cublas_dense_ms": times[1], "x_vs_dense_cublas": times[1] / times[0]}
        del cs
    torch.cuda.empty_cache()

    # The stream-K schedule (opt-in: lynx_debug_force_ksplit(LYNX_KSPLIT_STREAM)) against the automatic one at
    # the stack's few-tile MLP-down shape (64 tiles of 256 x 192 for the CTA pairs), in alternating blocks of calls.
    Ms, Ns, Ks = 1024, 3072, 12288
    cs = [{"X": torch.randn((Ms, Ks), generator=gen, device=dev).to(torch.bfloat16),
           "W": (torch.randn((Ns, Ks), generator=gen, device=dev) / Ks ** 0.5).to(torch.bfloat16),
           "LA": (0.02 * torch.randn((Ns, R), generator=gen, device=dev)).to(torch.bfloat16),
           "LB": (0.02 * torch.randn((R, Ks), generator=gen, device=dev)).to(torch.bfloat16),
           "Y": torch.empty((Ms, Ns), dtype=torch.bfloat16, device=dev)} for _ in range(2)]
    sched = {}
    for mode in (0, asl.LYNX_KSPLIT_STREAM):
        asl.lynx_debug_force_ksplit(mode)
        sched[mode] = (asl.lynx_debug_linear_ksplit(Ms, Ns, Ks),
                       torch.empty(asl.lynx_workspace_bytes(Ms, Ns, Ks, R), dtype=torch.uint8, device=dev))
    sk_ms = {0: [], asl.LYNX_KSPLIT_STREAM: []}
    try:
        for blk in range(5):
            for mode in (0, asl.LYNX_KSPLIT_STREAM):
                asl.lynx_debug_force_ksplit(mode)
                ws_m = sched[mode][1]

                def one_sk(c):
                    return L.lynx_linear(c["X"].data_ptr(), c["W"].data_ptr(), c["LA"].data_ptr(),
                                         c["LB"].data_ptr(), c["Y"].data_ptr(), Ms, Ns, Ks, R, ws_m.data_ptr(),
                                         ws_m.numel(), sp)
                for i in range(3):
                    one_sk(cs[i % 2])
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for i in range(20):
                    one_sk(cs[i % 2])
                a1.record(stream)
                torch.cuda.synchronize()
                sk_ms[mode].append(a0.elapsed_time(a1) / 20)
    finally:
        asl.lynx_debug_force_ksplit(0)
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)
    stream_k = {"shape": "1024x12288->3072 (256 x 192 tiles)",
                "auto_schedule": sched[0][0], "auto_ms": statistics.median(sk_ms[0]),
                "stream_k_schedule": sched[asl.LYNX_KSPLIT_STREAM][0],
                "stream_k_ms": statistics.median(sk_ms[asl.LYNX_KSPLIT_STREAM]),
                "note": "whole lynx_linear calls, median of 5 alternating blocks of 20; stream-K is opt-in because "
                        "it measured slower"}
    del cs, sched
    torch.cuda.empty_cache()

    # The sparsify pass alone (lynx_sparsify, and lynx_sparsify_lora with the LoRA down-projection), back to back
    # on inputs rotated over copies larger than L2: algorithmic bytes per call / time against the HBM peak, at
    # the QKV input and at the largest activations of the workloads (the CFG batch's MLP-down input and the
    # stack's largest M).
    sparsify_alone = {}
    for Ms, Ks in ((4608, 3072), (9216, 12288), (16384, 3072)):
        nset = int(400e6 // (Ms * Ks * 2)) + 2
        xs = [torch.randn((Ms, Ks), generator=gen, device=dev).to(torch.bfloat16) for _ in range(nset)]
        lb = (0.02 * torch.randn((R, Ks), generator=gen, device=dev)).to(torch.bfloat16)
        vals = torch.empty((Ms, Ks // 2), dtype=torch.bfloat16, device=dev)
        meta = torch.empty(asl.lynx_meta_bytes(Ms, Ks), dtype=torch.uint8, device=dev)
        sv = torch.empty(Ms, dtype=torch.float32, device=dev)
        tv = torch.empty((Ms, R), dtype=torch.bfloat16, device=dev)
        res = {"cluster_ctas": asl.lynx_debug_prologue_split(Ms, Ks)}
        base = Ms * Ks * 2 + Ms * Ks + asl.lynx_meta_bytes(Ms, Ks) + 4 * Ms
        for key, fn, nbytes in (
                ("sparsify", lambda x: L.lynx_sparsify(x.data_ptr(), Ms, Ks, vals.data_ptr(), meta.data_ptr(),
                                                       sv.data_ptr(), sp), base),
                ("sparsify_lora_down", lambda x: L.lynx_sparsify_lora(x.data_ptr(), lb.data_ptr(), Ms, Ks, R,
                                                                      vals.data_ptr(), meta.data_ptr(), sv.data_ptr(),
                                                                      tv.data_ptr(), sp), base + R * Ks * 2 + Ms * R * 2)):
            for i in range(3):
                fn(xs[i % nset])
            torch.cuda.synchronize()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nrep = 60
            a0.record(stream)
            for i in range(nrep):
                if fn(xs[i % nset]) != 0:
                    raise RuntimeError(key + " failed")
            a1.record(stream)
            torch.cuda.synchronize()
            us = a0.elapsed_time(a1) / nrep * 1e3
            res[key] = {"us": us, "GBs": nbytes / us / 1e3, "frac_hbm": nbytes / us / 1e3 / hbm}
        sparsify_alone[f"{Ms}x{Ks}"] = res
        del xs, lb, vals, meta, sv, tv
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)
    torch.cuda.empty_cache()

    # The block stack of the fifth workload: 8 blocks x (QKV sparse 3072->9216, out dense 3072->3072, up dense
    # 3072->12288 followed by the MLP's GELU, down sparse 12288->3072 on that GELU output), rank-64 LoRA on the
    # sparse layers, the seeded weights of every block and the seeded block input from synth.  The up layer's
    # epilogue applies the GELU.  Against it: the same 32 linears dense through cuBLAS with the same GELU (torch)
    # between up and down.  Both sides run eagerly and as one CUDA graph each.
    import torch.nn.functional as F
    stack = {}

    def block_weights(b):
        tq = synth.layer_tensors("stack", "qkv", block=b, with_x=False)
        td = synth.layer_tensors("stack", "down", block=b, with_x=False)
        return {"qkv": tq["W"], "la_qkv": tq["LA"], "lb_qkv": tq["LB"],
                "out": synth.layer_tensors("stack", "out", block=b, with_x=False)["W"],
                "up": synth.layer_tensors("stack", "up", block=b, with_x=False)["W"],
                "down": td["W"], "la_down": td["LA"], "lb_down": td["LB"]}

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(8) as ex:
        wts = [{k: to_dev(v) for k, v in w.items()} for w in ex.map(block_weights, range(8))]
        xs = list(ex.map(lambda Ms: synth.layer_x("stack", "qkv", M=Ms, block=0), synth.STACK_M))
    for i, Ms in enumerate(synth.STACK_M):
        x3 = to_dev(xs[i])
        y = {n: torch.empty((Ms, n), dtype=torch.bfloat16, device=dev) for n in (3072, 9216)}
        h = torch.empty((Ms, 12288), dtype=torch.bfloat16, device=dev)
        y_dn = torch.empty((Ms, 3072), dtype=torch.bfloat16, device=dev)
        layers = []
        for w in wts:
            layers += [asl.lynx_layer(x3, w["qkv"], w["la_qkv"], w["lb_qkv"], y[9216], sparse=True),
                       asl.lynx_layer(x3, w["out"], None, None, y[3072], sparse=False),
                       asl.lynx_layer(x3, w["up"], None, None, h, sparse=False, gelu=True),
                       asl.lynx_layer(h, w["down"], w["la_down"], w["lb_down"], y_dn, sparse=True)]
        ws_s = torch.empty(asl.lynx_layers_workspace_bytes(layers), dtype=torch.uint8, device=dev)

        def lynx_stack():
            asl.lynx_run_layers(layers, ws_s, stream=stream)

        def dense_stack():
            for w in wts:
                torch.matmul(x3, w["qkv"].t(), out=y[9216])
                torch.matmul(x3, w["out"].t(), out=y[3072])
                hd = F.gelu(torch.matmul(x3, w["up"].t()))
                torch.matmul(hd, w["down"].t(), out=y_dn)

        lgraph = asl.LynxGraph(layers, ws_s)
        dense_stack()  # cuBLAS workspace and kernels chosen before capture
        torch.cuda.synchronize()
        dgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(dgraph):
            dense_stack()
        torch.cuda.synchronize()
        tt = []
        for fn in (lynx_stack, dense_stack, lambda: lgraph.launch(stream), dgraph.replay):
            fn()
            torch.cuda.synchronize()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(3):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            tt.append(a0.elapsed_time(a1) / 3)
        st = asl.lynx_sync_status()
        assert st == 0, asl.lynx_status_string(st)
        lgraph.close()
        stack[f"M={Ms}"] = {"lynx_ms": tt[0], "all_dense_cublas_ms": tt[1], "x_vs_dense_cublas": tt[1] / tt[0],
                            "lynx_graph_ms": tt[2], "all_dense_cublas_graph_ms": tt[3],
                            "x_vs_dense_cublas_graph": tt[3] / tt[2]}
        del x3, y, h, y_dn, ws_s, layers, lgraph, dgraph
    del wts, xs
    torch.cuda.empty_cache()

    # The MLP pair of the third workload (4608 tokens: up 3072->12288 sparse with LoRA, GELU, down 12288->3072
    # sparse with LoRA) through the layer sequence, unfused and fused, against cuBLAS up, GELU (torch), cuBLAS down.
    tu = synth.layer_tensors("mlp", "up")
    td = synth.layer_tensors("mlp", "down", with_x=False)
    Mm = tu["M"]
    xu = to_dev(tu["X"])
    hu = torch.empty((Mm, 12288), dtype=torch.bfloat16, device=dev)
    yd = torch.empty((Mm, 3072), dtype=torch.bfloat16, device=dev)
    wu, wd = to_dev(tu["W"]), to_dev(td["W"])
    lau, lbu, lad, lbd = to_dev(tu["LA"]), to_dev(tu["LB"]), to_dev(td["LA"]), to_dev(td["LB"])
    pair = [asl.lynx_layer(xu, wu, lau, lbu, hu, sparse=True, gelu=True),
            asl.lynx_layer(hu, wd, lad, lbd, yd, sparse=True)]
    fused = [asl.lynx_layer(xu, wu, lau, lbu, hu, sparse=True, gelu=True, fuse=True),
             asl.lynx_layer(hu, wd, lad, lbd, yd, sparse=True)]
    ws_p = torch.empty(asl.lynx_layers_workspace_bytes(fused), dtype=torch.uint8, device=dev)
    tt = []
    for fn in (lambda: asl.lynx_run_layers(pair, ws_p, stream=stream),
               lambda: torch.matmul(F.gelu(torch.matmul(xu, wu.t())), wd.t(), out=yd),
               lambda: asl.lynx_run_layers(fused, ws_p, stream=stream)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(20):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        tt.append(a0.elapsed_time(a1) / 20)
    st = asl.lynx_sync_status()
    assert st == 0, asl.lynx_status_string(st)
    fl = 2.0 * Mm * 12288 * 3072 * 2
    mlp_pair = {"lynx_ms": tt[0], "tflops": fl / (tt[0] * 1e-3) / 1e12, "cublas_gelu_ms": tt[1],
                "x_vs_dense_cublas": tt[1] / tt[0], "lynx_fused_sparsify_ms": tt[2],
                "note": "up 4608x3072->12288 sparse+LoRA, GELU in its epilogue, down 12288->3072 sparse+LoRA with "
                        "its own sparsify pass; lynx_fused_sparsify_ms: the down layer's sparsification written by "
                        "the up layer's epilogue instead (LYNX_LAYER_FUSE_SPARSIFY)"}
    del xu, hu, yd, wu, wd, pair, fused, ws_p, lau, lbu, lad, lbd
    torch.cuda.empty_cache()

    # End to end through the C-ABI with host buffers, pipelined as a serving loop runs it: every step copies
    # its X from pinned host memory, calls lynx_linear and copies its Y back to pinned host memory, on three
    # streams so that step i's copies overlap the neighbouring steps' compute.  Events order the reuse of the
    # ROTATE device buffer sets (X is overwritten only after the step that read it has computed, Y only after
    # it has been copied out).
    Xh = torch.empty((M, K), dtype=torch.bfloat16, pin_memory=True)
    Xh.copy_(sets[0]["X"].cpu())
    Yh = [torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n, t0=None, t1=None):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        if t0 is not None:
            t0.record(s_in)
        for i in range(n):
            s = sets[i % ROTATE]
            if i >= ROTATE:
                s_in.wait_event(ev_comp[i - ROTATE])
            with torch.cuda.stream(s_in):
                s["X"].copy_(Xh, non_blocking=True)
            ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= ROTATE:
                s_comp.wait_event(ev_out[i - ROTATE])
            if L.lynx_linear(s["X"].data_ptr(), s["W"].data_ptr(), s["LA"].data_ptr(), s["LB"].data_ptr(),
                             s["Y"].data_ptr(), M, N, K, R, s["ws"].data_ptr(), s["ws"].numel(),
                             s_comp.cuda_stream) != 0:
                raise RuntimeError("lynx_linear failed")
            ev_comp[i].record(s_comp)
            s_out.wait_event(ev_comp[i])
            with torch.cuda.stream(s_out):
                Yh[i % 2].copy_(s["Y"], non_blocking=True)
            ev_out[i].record(s_out)
        if t1 is not None:
            s_in.wait_stream(s_out)
            t1.record(s_in)

    ne = min(args.steps, 200)
    e2e_run(4)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(ne, e0, e1)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / ne
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    # CPU baseline: the C++ oracle on bounded row samples, every host core and one thread (single-GPU runs only)
    cpu_base = cpu_baseline_leg(t) if world == 1 else None
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(t),
        "roofline": {"bound": "tensor", "achieved": gemm_tf, "peak": sparse_peak, "unit": "TFLOP/s",
                     "frac": gemm_tf / sparse_peak,
                     "traffic": profiled_traffic("sparse_gemm_pair_qkv.md", "gemm_pair.cu"),
                     "kernel": "sparse GEMM + LoRA-up + s epilogue (tcgen05.mma.sp)",
                     "peak_source": f"2 x dense bf16 burst {dense_tf} TFLOP/s (nominal 2:4 ratio), {peaks['source']}",
                     "measured_sparse_peak": {
                         "tflops": mma_more["mode6"], "frac": gemm_tf / mma_more["mode6"],
                         "source": "this run's pair tcgen05.mma.sp microbenchmark (M 256, N 256, operands resident "
                                   "in shared memory, one issuing thread per pair; lynx_mma_rate mode 6)"}},
        "cpu_baseline": cpu_base,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": M * K * 2,
                "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms,
                "note": "every step: pinned host X -> device, lynx_linear, Y -> pinned host; weights resident; "
                        "copies and compute pipelined over three streams"},
        "gpu_launches": L.lynx_linear_kernel_count(M, N, K, R) * args.steps,
        "clocks": clocks,
        "detail": {
            "stage_ms": {"sparsify_lora_down": stage_avg[0], "sparse_gemm": stage_avg[1]},
            "stage_ms_p10_p50_p90": {
                "sparsify_lora_down": [float(np.percentile(stage_ms[:, 0], q)) for q in (10, 50, 90)],
                "sparse_gemm": [float(np.percentile(stage_ms[:, 1], q)) for q in (10, 50, 90)]},
            "stage_events": f"on every {PROFILE_EVERY}th timed step ({len(prof_steps)} of {args.steps})",
            "sparse_gemm_pct_of_sparse_peak": 100.0 * gemm_tf / sparse_peak,
            "step_pct_of_sparse_peak": 100.0 * (value / world) / sparse_peak,
            "sparsify_lora_down_GBs": prologue_gbs, "sparsify_lora_down_frac_hbm": prologue_gbs / hbm,
            "dense_cublas_ms": dense_ms, "dense_cublas_tflops": flops / (dense_ms * 1e-3) / 1e12,
            "x_vs_dense_cublas": dense_ms / ms_per_step,
            "lynx_dense_gemm_ms": lynx_dense_ms, "lynx_dense_gemm_tflops": flops / (lynx_dense_ms * 1e-3) / 1e12,
            "hbm_peak_GBs": hbm, "dense_bf16_peak_tflops": dense_tf,
            "weight_2to4_comparator": {"ms": wsparse_ms, "tflops": flops / (wsparse_ms * 1e-3) / 1e12,
                                       "x_vs_dense_cublas": dense_ms / wsparse_ms,
                                       "note": "Y = X W~^T + X (LA LB)^T, W~ = 2:4-pruned W as the sparse operand",
                                       "library_2to4_cusparselt": cslt},
            "in_gemm_selection": {"ms": fused_ms, "tflops": flops / (fused_ms * 1e-3) / 1e12,
                                  "x_vs_two_pass": ms_per_step / fused_ms,
                                  "note": "lynx_linear_fused: LoRA down-projection + one GEMM that selects the 2:4 "
                                          "pattern of each dense X tile in its epilogue warps (256 x 256 tiles); "
                                          "every column tile repeats its rows' selection"},
            "other_shapes": shapes,
            "stream_k": stream_k,
            "sparsify_alone": sparsify_alone,
            "block_stack_32_linears": stack,
            "mlp_pair": mlp_pair,
            "mma_microbench": {"dense_tflops": mma_dense_tf, "sparse_tflops_effective": mma_sparse_tf,
                               "dense_macs_per_clk": mma_dense_mpc, "sparse_macs_per_clk_effective": mma_sparse_mpc,
                               "sparse_over_dense": mma_sparse_tf / mma_dense_tf,
                               "sparse_with_meta_copy_tflops_effective": mma_sparse_cp_tf,
                               "sparse_commit_every_2_tflops_effective": mma_sparse_c2_tf,
                               "sparse_2commits_every_4_tflops_effective": mma_sparse_c4_tf,
                               "sparse_a64swizzle_tflops_effective": mma_more["mode5"],
                               "pair_sparse_a128swizzle_tflops_effective": mma_more["mode6"],
                               "pair_sparse_a64swizzle_tflops_effective": mma_more["mode7"],
                               "pair_dense_tflops": mma_more["mode8"],
                               "sparse_gemm_frac_of_microbench": gemm_tf / mma_sparse_tf},
        },
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
