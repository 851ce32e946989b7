"""Benchmark of the batch-1 decode step on GB300: tokens/s and achieved HBM bandwidth as a fraction
of the bytes-per-token floor.

One step = one decode step (one token through every layer, the LM head and the argmax) of the
Llama-3.2-1B-shaped bf16 workload by default: 16 layers, hidden 2048, 32/8 heads, FFN 8192,
vocab 128256, tied embeddings, bf16 KV cache prefilled with N(0,1) to position 1024, greedy decode
over positions 1024..1151 (positions wrap inside that window when more steps are timed). Weights are
seeded synthetic (N(0, 0.02)), 2.47 GB per token, far larger than L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--mode mega|graph]
  python bench.py --impl reference ...   # the reference arm: the CPU oracle on the host cores

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path has no
exchange step); rank 0 prints the JSON line with the max-over-ranks time.
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

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "batch-1 decode tokens/s and achieved HBM GB/s as % of GB300 weight-read floor"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
MIN_TIMED_S = 0.2  # the timed region covers at least this much time


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Dense bf16 peak for a contraction timed alone: MEASURED_PEAKS.json's burst figure, else the
    earlier single measurement on a GB300."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


KERNEL_SOURCES = ["megakernel.cuh", "step.cuh", "ptx.cuh", "engine.h", "kernels.h", "mega_bf16.cu",
                  "mega_int4.cu"]


def kernel_source_hash() -> str:
    """sha256 over the device-code sources of the step kernels (names and code; comments and
    blank space do not count, so a comment edit keeps a recorded measurement valid)."""
    import hashlib
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "decode_persistent_megakernel_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(d, name)) as f:
            code = f.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        code = " ".join(code.split())
        h.update(name.encode())
        h.update(code.encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for ln in f:
            if "=" in ln and not ln.lstrip().startswith("#"):
                k, v = ln.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return int(kv["dram_bytes_per_launch"])


BLOCK_STEPS = 64  # steps per block of the per-step time distribution


def block_stats(marks: list) -> dict | None:
    """Per-step time over blocks of the timed region: marks = [(step index, ms since the region's
    start)] at the block boundaries, first (0, 0) and last (steps, total). Returns the median, 10th
    and 90th percentile (linear interpolation) of the blocks' ms per step, or None for one block."""
    per = [(t1 - t0) / (i1 - i0) for (i0, t0), (i1, t1) in zip(marks, marks[1:]) if i1 > i0]
    if len(per) < 2:
        return None
    q = np.percentile(np.array(per), [10, 50, 90])
    return {"block_steps": BLOCK_STEPS, "blocks": len(per), "median": float(q[1]), "p10": float(q[0]),
            "p90": float(q[2])}


def algorithmic_bytes(c: dict, pos: int) -> int:
    """Bytes one step must move at position pos: every weight once in its stored format (linears,
    norms, biases, int4 scales), the LM head once, one embedding row, the K/V cache read over
    [0, pos) and one K/V slot written."""
    mb = synth.model_bytes(c)
    w = mb["layers"] + mb["lm_head"] + mb["final_norm"] + c["hidden"] * 2
    kv_per_pos = c["n_layers"] * c["n_kv_heads"] * c["head_dim"] * 2 * 2
    return w + kv_per_pos * (pos + 1)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
        return rank, local, world, dist
    return 0, 0, 1, None


def barrier(dist, torch):
    if dist is not None:
        dist.barrier()
    if torch is not None and torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(dist, torch, value: float) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(c: dict, world: int) -> dict:
    """The workload description both arms print (same keys and values for the same workload)."""
    P = c["prefill"] + c["prompt"]
    return {"workload": c["name"], "prefill": P,
            "decode_positions": f"{P}..{P + c['steps'] - 1} (timed steps cycle through this window)",
            "l2": "inputs larger than L2 (weights streamed once per step)",
            "parallelism": f"replicas x{world}"}


def oracle_baseline(c, w, K, V, budget_s: float):
    """The CPU oracle, as it stands, on a bounded sample of the same workload: consecutive decode
    steps from the first decode position, until about budget_s of work is done."""
    from oracle import Oracle
    orc = Oracle("f64")
    om = orc.model(c, w)
    K = K.copy()
    V = V.copy()
    tok = int(synth.make_tokens(c, 1)[0])
    P = c["prefill"] + c["prompt"]
    n, t0 = 0, time.perf_counter()
    while True:
        _, tok, rc = orc.decode_step(om, tok, P + n, K, V)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= c["steps"]:
            break
    threads = orc.threads()
    # the same oracle on one thread, over a few of the same steps (the benchmark's second figure)
    orc.set_threads(1)
    K1, V1 = K.copy(), V.copy()
    tok1 = int(synth.make_tokens(c, 1)[0])
    n1, t1 = 0, time.perf_counter()
    while True:
        _, tok1, _ = orc.decode_step(om, tok1, P + n1, K1, V1)
        n1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= min(budget_s, 10.0) or n1 >= c["steps"]:
            break
    orc.set_threads(threads)
    return {"value": n / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "value_1thread": n1 / el1,
            "sample": f"{n} greedy decode steps of {c['name']} at positions {P}..{P + n - 1} "
                      f"(fp64 oracle, {threads} OpenMP threads), {el:.1f} s; one thread: {n1} steps, "
                      f"{el1:.1f} s"}


def ops_measurements(T, torch, peak):
    """Device-timed rates of the op-level paths on inputs larger than L2, as GB/s of the weight bytes
    each call must read: the gathered-expert MLP (64 experts, 8 chosen, hidden 2048, expert FFN
    1024; successive calls route to disjoint expert sets, 805 MB of bf16 experts in all) and the
    batched GEMV at m = 1, 2, 4, 8 over four 16384 x 2048 bf16 matrices taken in turn."""
    out = {}
    st = torch.cuda.current_stream()

    def timed(fn, n):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for i in range(n):
            fn(i)
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    for fmt, group in (("bf16", 64), ("int4", 64)):
        E, k, H, F = 64, 8, 2048, 1024
        m = synth.make_moe(E, k, H, F, fmt, group, "fp16", seed=0)
        f = T.TINFER_INT4 if fmt == "int4" else T.TINFER_BF16
        dev = {n: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
               for n, v in m.items() if v is not None and n[0] in "ws" and n != "weights"}
        gu = torch.empty(T.tinfer_moe_packed_bytes(f, group, E, H, F, 0), dtype=torch.uint8, device="cuda")
        dn = torch.empty(T.tinfer_moe_packed_bytes(f, group, E, H, F, 1), dtype=torch.uint8, device="cuda")
        assert T.tinfer_pack_moe(f, group, 0, E, H, F, dev["wg"], dev.get("sg"), dev["wu"], dev.get("su"),
                                 dev["wd"], dev.get("sd"), gu, dn) == 0
        del dev
        ids = [torch.arange(8 * i, 8 * i + 8, dtype=torch.int32, device="cuda") for i in range(E // k)]
        wts = torch.tensor(m["weights"], device="cuda")
        x = torch.tensor(m["x"], device="cuda")
        h = torch.empty(k * F, device="cuda")
        y = torch.empty(H, device="cuda")
        ms = timed(lambda i: T.tinfer_op_moe(f, group, 0, E, k, H, F, gu, dn, ids[i % len(ids)], wts, x, h, y,
                                             0, None, st), 64)
        nbytes = (gu.numel() + dn.numel()) * k // E
        out[f"moe_{fmt}"] = {"shape": f"{E} experts, top {k}, hidden {H}, expert ffn {F}", "us_per_call": ms * 1e3,
                             "weight_bytes": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
                             "frac": nbytes / (ms * 1e-3) / 1e9 / peak}
        del gu, dn
        torch.cuda.empty_cache()
    rows, cols = 16384, 2048
    mats = []
    for i in range(4):
        W = synth.normal_bf16(f"bench.gemvm.{i}", (rows, cols), 0.0, 0.02, 0)
        pk = torch.empty(rows * cols * 2, dtype=torch.uint8, device="cuda")
        assert T.tinfer_pack_matrix(0, 64, 0, rows, cols, torch.from_numpy(W.view(np.int16)).cuda(), None, pk) == 0
        mats.append(pk)
    res = {}
    for mv in (1, 2, 4, 8):
        xs = torch.randn(mv * cols, device="cuda")
        ys = torch.empty(mv * rows, device="cuda")
        ms = timed(lambda i: T.tinfer_op_gemv_batch(0, 64, 0, rows, cols, mv, mats[i % 4], xs, None, 0, ys, st), 64)
        nb = rows * cols * 2
        res[str(mv)] = {"us_per_call": ms * 1e3, "achieved_gbs": nb / (ms * 1e-3) / 1e9,
                        "frac": nb / (ms * 1e-3) / 1e9 / peak}
    out["gemv_batch_bf16_16384x2048"] = res
    del mats
    torch.cuda.empty_cache()
    # the batched-prefill matrix product on the tensor cores (tinfer_op_gemm_bf16, one call includes
    # its device-to-host status read): a 2048-token prompt through the Llama-shaped gate/up matrix and
    # a compute-bound 4096 x 8192 x 8192 product; four weight matrices taken in turn
    bf16_peak = measured_bf16_tflops()
    gres = {}
    for (m, n, k) in ((2048, 16384, 2048), (4096, 8192, 8192)):
        ws = [torch.from_numpy(synth.normal_bf16(f"bench.gemm.{n}.{k}.{i}", (n, k), 0.0, 0.02, 0).view(np.int16)).cuda()
              for i in range(4)]
        xg = torch.from_numpy(synth.normal_bf16(f"bench.gemm.x.{m}.{k}", (m, k), 0.0, 1.0, 0).view(np.int16)).cuda()
        yg = torch.empty(m, n, device="cuda")
        ms = timed(lambda i: T.tinfer_op_gemm_bf16(m, n, k, xg, ws[i % 4], yg, st), 16)
        tf = 2.0 * m * n * k / (ms * 1e-3) / 1e12
        gres[f"{m}x{n}x{k}"] = {"us_per_call": ms * 1e3, "tflops": tf, "frac": tf / bf16_peak[0],
                                "peak_kind": bf16_peak[1]}
        del ws, xg, yg
        torch.cuda.empty_cache()
    out["gemm_bf16_tcgen05"] = gres
    return out


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores, same config and metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    c = synth.config(args.config)
    w = synth.make_model(c, seed=0)
    K, V = synth.make_kv(c, c["prefill"], seed=0)
    per_step_budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    from oracle import Oracle
    orc = Oracle("f64")
    om = orc.model(c, w)
    P = c["prefill"] + c["prompt"]
    tok = int(synth.make_tokens(c, 1)[0])
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _, tok, _ = orc.decode_step(om, tok, P + (s % c["steps"]), K, V)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
        if sum(times) > per_step_budget * args.steps:
            break
    ms = 1e3 * statistics.mean(times)
    val = 1e3 / ms
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(c, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
                             "sample": f"{len(times)} decode steps of {c['name']} from position {P}"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1280)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--config", default="llama1b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--mode", default="mega", choices=["mega", "graph"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-loop", action="store_true", help="skip the in-kernel token loop measurement")
    ap.add_argument("--no-ops", action="store_true", help="skip the op-level measurements (MoE, batched GEMV)")
    ap.add_argument("--sync", default="stamps", choices=["stamps", "barrier"],
                    help="how a phase waits for the one before it (persistent kernel)")
    ap.add_argument("--ffn-split", action="store_true",
                    help="the column-split down projection variant (bf16 workloads, persistent kernel)")
    ap.add_argument("--no-read-probe", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="steps of the e2e run (default: the workload's)")
    ap.add_argument("--only-ops", action="store_true",
                    help="only the op-level measurements (gathered experts, batched GEMV, prefill GEMM)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import decode_persistent_megakernel_gb300 as T

    rank, local, world, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    T.build()
    if args.only_ops:
        if rank == 0:
            print(json.dumps({"ops": ops_measurements(T, torch, measured_peaks()[0])}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    c = synth.config(args.config, **({"ffn_split": True} if args.ffn_split else {}))
    w = synth.make_model(c, seed=0)
    P = c["prefill"] + c["prompt"]
    S = c["steps"]
    K, V = synth.make_kv(c, P, seed=0)
    modes = [("mega", T.TINFER_MEGAKERNEL)] if args.mode == "mega" else [("graph", T.TINFER_GRAPH)]
    if args.mode == "mega" and not args.no_graph:
        modes.append(("graph", T.TINFER_GRAPH))
    results = {}
    st = torch.cuda.current_stream()
    first = int(synth.make_tokens(c, 1)[0])
    for name, mode in modes:
        eng = T.Engine(c, w, mode, kv=(K, V))
        if mode == T.TINFER_MEGAKERNEL and args.sync == "barrier":
            assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_SYNC, T.TINFER_SYNC_GRID_BARRIER) == 0
        # warm-up, then a short calibration: the timed region covers at least MIN_TIMED_S of steps
        # whatever --steps asks for (so that the clock sampler sees the run); the line reports the
        # steps actually timed
        cal = torch.zeros(args.warmup + 9, dtype=torch.int32, device="cuda")
        cal[0] = first
        for i in range(args.warmup):
            eng.step_dev(cal[i:i + 1], P + (i % S), stream=st, logits=False, argmax=cal[i + 1:i + 2])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for i in range(8):
            j = args.warmup + i
            eng.step_dev(cal[j:j + 1], P + (i % S), stream=st, logits=False, argmax=cal[j + 1:j + 2])
        e1.record(st)
        torch.cuda.synchronize()
        per = max(e0.elapsed_time(e1) / 8, 1e-3)
        steps = max(args.steps, int(np.ceil(MIN_TIMED_S * 1e3 / per)))
        steps = int(max_over_ranks(dist, torch, float(steps)))
        toks = torch.zeros(steps + 1, dtype=torch.int32, device="cuda")
        toks[0] = first
        # block boundaries for the per-step time distribution (events made before the region)
        bev = {i: torch.cuda.Event(enable_timing=True) for i in range(BLOCK_STEPS, steps, BLOCK_STEPS)}
        barrier(dist, torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            barrier(dist, torch)
            e0.record(st)
            for i in range(steps):
                if i in bev:
                    bev[i].record(st)
                eng.step_dev(toks[i:i + 1], P + (i % S), stream=st, logits=False, argmax=toks[i + 1:i + 2])
            e1.record(st)
            barrier(dist, torch)
        ms = e0.elapsed_time(e1)
        dist_ms = block_stats([(0, 0.0)] + [(i, e0.elapsed_time(ev)) for i, ev in sorted(bev.items())] +
                              [(steps, ms)])
        assert eng.error() == T.TINFER_OK
        ms_max = max_over_ranks(dist, torch, ms)
        results[name] = dict(ms_total=ms_max, ms_step=ms_max / steps, steps=steps, clocks=clk.summary(),
                             dist=dist_ms,
                             launches=steps * eng.query(T.TINFER_Q_KERNELS_PER_STEP),
                             grid=eng.query(T.TINFER_Q_GRID), smem=eng.query(T.TINFER_Q_SMEM),
                             threads=eng.query(T.TINFER_Q_BLOCK_THREADS),
                             stages=eng.query(T.TINFER_Q_RING_STAGES), slot=eng.query(T.TINFER_Q_SLOT_BYTES))
        if name == "mega" and not args.no_loop:
            # the in-kernel token loop: the workload's S steps in one launch (tinfer_generate_dev),
            # timed on the device; then end to end through the same call with the first token from
            # the host and every chosen token copied back to pinned host memory inside the region
            toks_l = torch.zeros(S, dtype=torch.int32, device="cuda")
            host_l = torch.zeros(S, dtype=torch.int32).pin_memory()
            assert T.tinfer_generate_dev(eng.ctx, first, P, S, -1, st, toks_l, None) == 0
            torch.cuda.synchronize()
            reps = max(1, int(np.ceil(MIN_TIMED_S * 1e3 / (S * results[name]["ms_step"]))))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(dist, torch)
            e0.record(st)
            for _ in range(reps):
                assert T.tinfer_generate_dev(eng.ctx, first, P, S, -1, st, toks_l, None) == 0
            e1.record(st)
            barrier(dist, torch)
            ms_l = max_over_ranks(dist, torch, e0.elapsed_time(e1))
            barrier(dist, torch)
            t0 = time.perf_counter()
            for _ in range(reps):
                assert T.tinfer_generate_dev(eng.ctx, first, P, S, -1, st, toks_l, None) == 0
                host_l.copy_(toks_l, non_blocking=True)
                st.synchronize()
            el_l = max_over_ranks(dist, torch, time.perf_counter() - t0)
            assert eng.error() == T.TINFER_OK
            results["loop"] = dict(ms_token=ms_l / (reps * S), tokens=reps * S, launches=reps,
                                   e2e=world * reps * S / el_l)
        if name == modes[0][0]:
            # end to end through the public call: host-in-the-loop greedy generation, one pinned
            # 4-byte token copied in and one 4-byte choice copied out per step
            n_e2e = min(S, args.e2e_steps) if args.e2e_steps > 0 else S
            out = np.zeros(n_e2e, dtype=np.int32)
            barrier(dist, torch)
            t0 = time.perf_counter()
            rc = T.tinfer_generate(eng.ctx, first, P, n_e2e, st, out)
            el = time.perf_counter() - t0
            assert rc == 0
            el = max_over_ranks(dist, torch, el)
            results["e2e"] = dict(value=world * n_e2e / el, steps=n_e2e)
        eng.close()
        del eng
        torch.cuda.empty_cache()

    ops = None
    if not args.no_ops and rank == 0:
        ops = ops_measurements(T, torch, measured_peaks()[0])

    # a pure streaming-read probe (page 1's yardstick), same process
    read_gbs = None
    try:
        if args.no_read_probe:
            raise RuntimeError("read probe skipped")
        buf = torch.empty(4 << 30, dtype=torch.uint8, device="cuda").view(torch.int32)
        buf.fill_(1)
        for _ in range(3):
            buf.max()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(10):
            buf.max()
        b.record()
        torch.cuda.synchronize()
        read_gbs = 10 * buf.numel() * 4 / (a.elapsed_time(b) * 1e-3) / 1e9
        del buf
    except Exception:
        pass

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    main_mode = modes[0][0]
    r = results[main_mode]
    steps = r["steps"]
    mean_pos = P + (sum(i % S for i in range(steps)) / steps)
    bytes_step = algorithmic_bytes(c, int(round(mean_pos)))
    peak, peak_kind = measured_peaks()
    achieved = bytes_step / (r["ms_step"] * 1e-3) / 1e9
    tps = world * steps / (r["ms_total"] * 1e-3)
    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_baseline(c, w, K, V, args.cpu_budget)
    line = {
        "metric": METRIC,
        "value": tps,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "steps_requested": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["ms_step"],
        "ms_per_step_blocks": r["dist"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if c["weight_format"] == "bf16" else "int4",
        "data": "synthetic",
        "config": workload_config(c, world),
        "exec_mode": ("persistent megakernel" if main_mode == "mega" else "cuda graph") +
                     (", column-split down projection" if args.ffn_split else "") +
                     (", grid barrier before every phase" if args.sync == "barrier" else ""),
        "positions_timed": f"{P}..{P + min(steps, S) - 1}" + (f", cycled {steps / S:.1f} times" if steps > S else ""),
        "bytes_per_step": bytes_step,
        "floor_frac_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": measured_traffic("decode_megakernel", args.config) if main_mode == "mega" else None,
                     "kernel": "decode_megakernel" if main_mode == "mega" else "whole graph",
                     "peak_kind": peak_kind},
        "read_probe_gbs": read_gbs,
        "floor_frac_read_probe": achieved / read_gbs if read_gbs else None,
        "cpu_baseline": cpu,
        "e2e": {"value": results["e2e"]["value"], "unit": "tokens/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "launch": {"grid": r["grid"], "threads": r["threads"], "smem": r["smem"], "ring_stages": r["stages"],
                   "slot_bytes": r["slot"]},
    }
    if ops is not None:
        line["ops"] = ops
    if "loop" in results:
        lp = results["loop"]
        line["token_loop"] = {"tokens/s": world * 1e3 / lp["ms_token"], "ms_per_token": lp["ms_token"],
                              "tokens_per_launch": S, "launches": lp["launches"],
                              "achieved_gbs": bytes_step / (lp["ms_token"] * 1e-3) / 1e9,
                              "e2e": {"value": lp["e2e"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 4},
                              "call": "tinfer_generate_dev (one cooperative launch per window)"}
    if "graph" in results and main_mode == "mega":
        g = results["graph"]
        line["graph_baseline"] = {"tokens/s": world * g["steps"] / (g["ms_total"] * 1e-3),
                                  "ms_per_step": g["ms_step"], "launches_per_step": g["launches"] // g["steps"],
                                  "parity": "oracle-checked at full size (tests/test_gpu_full.py)",
                                  "achieved_gbs": bytes_step / (g["ms_step"] * 1e-3) / 1e9}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
