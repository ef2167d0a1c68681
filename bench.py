"""Decode benchmark: one JSON line for the persistent decode megakernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8b|1b|8b_b8|8b_long|tiny]
                    [--impl mk|reference]

A step is one full greedy decode step of the Llama-style decoder (embedding,
every layer, the lm_head with the final norm fused, and the argmax SAMPLE),
run as one persistent-kernel launch on inputs already resident in HBM.  The
weights (15 GB for the 8B shape) are far larger than L2, so no flush is
needed between steps.  The KV cache grows by one row per step; algorithmic
bytes per step are counted from each step's positions.

Reported next to the device-timed value: the same metric end to end through
the C ABI with host buffers (mk_decode_step_host: the state copied in from
pinned memory and the sampled tokens copied out, every step), the same task
bodies launched one kernel per op and as a CUDA graph of those launches,
the level-synchronous ablation, the roofline of the kernel against measured
(or fallback) HBM bandwidth, SM clocks sampled during the timed region, and
the CPU oracle timed on a bounded sample on this host.

Multi-GPU: the decode step does not shard (one GPU, no collectives); with
--gpus N each rank runs an independent replica and rank 0 reports the sum.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode µs/step & tokens/s at B=1; achieved HBM GB/s vs ~8 TB/s roofline"
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_NAMES = {
    "tiny": "tiny Llama-style decoder (2 layers, hidden 256), B=1, KV 128",
    "1b": "Llama-3.2-1B-shaped decode, B=1, KV 1024, tied lm_head",
    "8b": "Llama-3-8B-shaped decode, B=1, KV 4096",
    "8b_b8": "Llama-3-8B-shaped decode, B=8, ragged KV in [512, 8192]",
    "8b_long": "Llama-3-8B-shaped decode, B=4, KV 32768, split-KV chunk 1024",
}


def dist_env():
    r = int(os.environ.get("RANK", "0"))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return r, ws, lr


def check_whole_step(task_bytes, w, L):
    """The timed graph is the whole decode step: every layer's attention,
    the lm_head tiles and one SAMPLE per sequence (a benchmark of one layer,
    or without the lm_head, is a known way to overstate decode speed)."""
    import numpy as np
    dt = np.dtype({"names": ["op_id", "m", "n"], "formats": ["<u2", "<i4", "<i4"], "offsets": [0, 28, 32],
                   "itemsize": 64})
    t = np.frombuffer(task_bytes, dtype=dt)
    m = w.model
    combines = int(np.count_nonzero(t["op_id"] == L.MK_OP_ATTENTION_COMBINE))
    samples = int(np.count_nonzero(t["op_id"] == L.MK_OP_SAMPLE))
    lm_tiles = int(np.count_nonzero((t["op_id"] == L.MK_OP_GEMV) & (t["n"] == m.V)))
    if combines != m.L * w.B * m.Hkv or samples != w.B or lm_tiles < 1:
        raise RuntimeError(f"timed graph is not a whole step: {combines} combines, {samples} samples, "
                           f"{lm_tiles} lm_head tiles for {m.L} layers, B={w.B}")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "task_graph_interpreter_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(config, algo_bytes):
    """DRAM bytes per launch from the committed ncu summary of a small case
    of the same kernel (a few layers at full width, full LM head), scaled to
    this launch by algorithmic bytes (every layer streams the same weights,
    so traffic grows in proportion); None unless the capture was taken on
    the current kernel sources.  Returns (bytes, note)."""
    p = os.path.join(ROOT, "profiles", f"dram_traffic_{config}.md")
    if not os.path.exists(p):
        return None, None
    fields = {}
    for line in open(p).read().splitlines():
        if ":" in line and not line.startswith(("#", "|", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    try:
        if fields.get("kernel_source_hash") != kernel_source_hash():
            return None, None
        dram = float(fields["dram_bytes_per_launch"])
        captured = float(fields["captured_algorithmic_bytes"])
    except (KeyError, ValueError):
        return None, None
    return dram * algo_bytes / captured, (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of {fields.get('captured_case')}"
                                          f" ({dram:.4g} B), scaled by algorithmic bytes x{algo_bytes / captured:.3f}")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def algorithmic_bytes(model, B, pos_list):
    """Weights streamed once + every cached key/value read + the new K/V rows
    written + logits written, for one step at the given positions."""
    w = model.streamed_params() * 2
    kv = sum((p + 1) * model.Hkv * model.D * 2 * 2 * model.L for p in pos_list)
    new = B * model.Hkv * model.D * 2 * 2 * model.L
    return w + kv + new + B * model.V * 4


def blas_threads_env():
    """Threads the BLAS may use in this process, as its environment sets them
    (the oracle's widening and elementwise numpy work runs on one thread)."""
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count() or 1


def oracle_steps(workload, steps, warmup, budget_s=None, seed=0):
    """Greedy decode steps of the float64 CPU oracle on the whole workload
    (every layer, full width and vocabulary, the workload's KV lengths),
    timed one by one on this host.  Inputs are generated first (untimed).
    Runs ``warmup`` untimed steps, then up to ``steps`` timed ones, stopping
    early once ``budget_s`` seconds of timed work are done.  Returns the
    per-step seconds."""
    import dataclasses
    import synth
    from oracle import forward as of
    m = workload.model
    w = dataclasses.replace(workload, steps=steps + warmup + 1)
    W = {n: synth.normal_bf16_np(n, shape, mu, sig, seed) for (n, shape, mu, sig) in synth.weight_names(m)}
    st = of.initial_state(m, w.B, w.capacity, w.kv_len, synth.prompt_tokens_np(w, seed),
                          lambda l, k: synth.kv_cache_np(synth.kv_name(l, k), w.B, m.Hkv, w.capacity, m.D,
                                                         w.kv_len, seed))
    for _ in range(warmup):
        of.decode_step(m, W, st, keep_hidden=False)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        of.decode_step(m, W, st, keep_hidden=False)
        times.append(time.perf_counter() - t0)
        if budget_s is not None and sum(times) >= budget_s:
            break
    return times


def oracle_child(config, layers, threads):
    """Child process of ``cpu_baseline``: one warm-up and one timed full
    oracle step with the BLAS limited to ``threads`` (set in the environment
    before numpy loads); prints one JSON line."""
    import dataclasses
    import synth
    w = synth.workload(config)
    if layers:
        w = dataclasses.replace(w, model=dataclasses.replace(w.model, L=layers))
    t = oracle_steps(w, 1, 0)
    print(json.dumps({"seconds": t[0], "blas_threads": blas_threads_env(), "cpus": os.cpu_count()}), flush=True)


def cpu_baseline(args, workload):
    """The CPU oracle timed on this host: one full greedy decode step of the
    whole workload (inputs generated first, untimed), with the BLAS on every
    core and on one core, each in a fresh process."""
    runs = {}
    for threads in (os.cpu_count() or 1, 1):
        env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
                   MKL_NUM_THREADS=str(threads))
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", str(threads), "--config", args.config]
        if args.layers:
            cmd += ["--layers", str(args.layers)]
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1200)
        if r.returncode != 0:
            raise RuntimeError(f"oracle timing failed:\n{r.stderr[-2000:]}")
        runs[threads] = json.loads(r.stdout.strip().splitlines()[-1])
    allc = runs[os.cpu_count() or 1]
    one = runs[1]
    m = workload.model
    return {
        "value": workload.B / allc["seconds"], "unit": "tokens/s", "cores": allc["blas_threads"],
        "kind": "oracle",
        "sample": (f"one full greedy decode step of the float64 numpy oracle on the whole {m.name} workload "
                   f"({m.L} layers, B={workload.B}, KV {max(workload.kv_len)}), timed after generating its "
                   f"inputs, {allc['seconds']:.2f} s with the BLAS on {allc['blas_threads']} threads of "
                   f"{allc['cpus']} CPUs (the oracle's bf16 widening runs on one thread)"),
        "seconds_per_step": allc["seconds"],
        "one_core": {"value": workload.B / one["seconds"], "unit": "tokens/s", "cores": 1,
                     "seconds_per_step": one["seconds"]},
    }


def run_reference(args, workload):
    """The reference arm: the CPU oracle, as it stands, on the same workload
    and metric.  One warm-up step, then full greedy steps until K are timed
    or about two minutes of timed work are done; the line reports the steps
    it really timed."""
    rank, ws, _ = dist_env()
    if rank != 0:
        return
    warm = min(args.warmup, 1)
    times = oracle_steps(workload, args.steps, warm, budget_s=120.0)
    t = sum(times) / len(times)
    v = workload.B / t
    m = workload.model
    cb = {"value": v, "unit": "tokens/s", "cores": blas_threads_env(), "kind": "oracle",
          "sample": (f"{len(times)} full greedy decode steps of the float64 numpy oracle on the whole {m.name} "
                     f"workload ({m.L} layers, B={workload.B}, KV {max(workload.kv_len)}) after {warm} warm-up "
                     f"step(s), BLAS on {blas_threads_env()} threads of {os.cpu_count()} CPUs")}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": len(times), "warmup": warm, "ms_per_step": 1000.0 * t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(args, workload),
        "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                    "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reduce_max(x, ws, device=None):
    """Max over ranks of a float (the slowest replica sets the time); the
    value itself at world size 1."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(B, steps, seconds, ws):
    """Whole-job tokens/s: every replica decodes B sequences per step, the
    job takes as long as its slowest replica."""
    return B * steps / seconds * ws


def config_dict(args, w):
    name = WORKLOAD_NAMES[args.config] + (f", truncated to {w.model.L} layers" if args.layers else "")
    return {"workload": name, "B": w.B, "kv_len_start": list(w.kv_len)[:8],
            "layers": w.model.L, "hidden": w.model.H, "ffn": w.model.F, "vocab": w.model.V,
            "heads_q_kv": [w.model.Hq, w.model.Hkv], "head_dim": w.model.D,
            "l2": "inputs larger than L2 (weights streamed every step exceed the 129 MB L2)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="8b", choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-modes", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="truncate the model to this many layers (small cases for profiling)")
    ap.add_argument("--oracle-child", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(args.config, args.layers, args.oracle_child)
        return

    import dataclasses
    import synth
    base = synth.workload(args.config)
    if args.layers:
        base = dataclasses.replace(base, model=dataclasses.replace(base.model, L=args.layers))
    if args.impl == "reference":
        run_reference(args, base)
        return

    import torch
    rank, ws, lr = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(lr)
    dev = torch.device("cuda", lr)
    from task_graph_interpreter_gb300.build import build
    build()
    from task_graph_interpreter_gb300 import _lib as L
    from task_graph_interpreter_gb300.llama import build_llama_decode

    # enough capacity for warm-up, timed steps and the extra timed modes
    extra = 4 * (args.warmup + args.steps) + 8
    w = synth.custom(base.model, base.B, base.kv_len, extra, chunk=base.chunk, name=base.name)
    weights, kc, vc, hist, state = synth.device_inputs(w, 0, dev)
    dec = build_llama_decode(w.model, w.B, w.kv_len, w.capacity, weights, kc, vc, hist, chunk=w.chunk,
                             device=dev)
    g = dec.graph
    g.state.copy_(state)
    g.lower()
    g.upload()
    stream = torch.cuda.current_stream(dev)
    n_tasks = len(g.tasks_bytes()) // 64
    check_whole_step(g.tasks_bytes(), w, L)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def positions():
        return [int(x) for x in g.state[:, 1].cpu()]

    def timed(mode, K, W):
        for _ in range(W):
            g.step(mode)
        barrier()
        pos0 = positions()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            g.step(mode)
        e1.record(stream)
        barrier()
        ms = e0.elapsed_time(e1)
        code, task = g.status()
        if code != 0:
            raise RuntimeError(f"device status {code} at task {task} in mode {mode}")
        # every timed step generated one token per sequence
        if positions() != [p + K for p in pos0]:
            raise RuntimeError(f"mode {mode}: positions {positions()} after {K} steps from {pos0}")
        nbytes = sum(algorithmic_bytes(w.model, w.B, [p + i for p in pos0]) for i in range(K))
        return ms, nbytes

    with ClockSampler(lr) as clk:
        ms, nbytes = timed(L.MK_MODE_MEGA, args.steps, args.warmup)
    clocks = clk.summary()
    ms = reduce_max(ms, ws, dev)
    ms_step = ms / args.steps
    tok_s = job_throughput(w.B, args.steps, ms / 1000.0, ws)
    hbm_peak, peak_kind = measured_peaks()
    achieved = nbytes / args.steps / (ms_step / 1000.0) / 1e9

    # end to end through the C ABI with host buffers, one sync per step
    state_h = torch.empty(w.B, 2, dtype=torch.int32).pin_memory()
    tok_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
    cur = g.state.cpu()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        state_h.copy_(cur)
        g.step_host(state_h, tok_h)
        stream.synchronize()
        cur[:, 0] = tok_h
        cur[:, 1] += 1
    barrier()
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    e2e = {"value": job_throughput(w.B, args.steps, e2e_s, ws), "unit": "tokens/s", "h2d_bytes_per_step": 8 * w.B,
           "d2h_bytes_per_step": 4 * w.B, "ms_per_step": 1000.0 * e2e_s / args.steps}

    modes = {}
    if not args.no_modes:
        for name, mode in (("per_op", L.MK_MODE_PER_OP), ("per_op_graph", L.MK_MODE_PER_OP_GRAPH),
                           ("per_op_pdl", L.MK_MODE_PER_OP_PDL), ("levels", L.MK_MODE_LEVELS)):
            k = max(4, args.steps // 4)
            mms, mb = timed(mode, k, 2)
            modes[name] = {"ms_per_step": mms / k, "tokens_per_s": w.B * k / (mms / 1000.0),
                           "achieved_gbs": mb / k / (mms / k / 1000.0) / 1e9}
        modes["mega"] = {"ms_per_step": ms_step, "tokens_per_s": w.B / (ms_step / 1000.0), "achieved_gbs": achieved}
        n_groups = None
    if rank != 0:
        return

    cpu = None
    if not args.no_cpu_baseline and ws == 1:  # the oracle baseline is timed at N=1 only
        cpu = cpu_baseline(args, base)

    traffic, traffic_note = profiled_traffic(args.config, nbytes / args.steps)
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": 1000.0 * ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded bf16 weights ~N(0,0.02), KV ~N(0,1); no trained weights)",
        "config": config_dict(args, w),
        "achieved_hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_kind,
                     "traffic": traffic, "traffic_source": traffic_note,
                     "algorithmic_bytes_per_launch": nbytes / args.steps},
        "e2e": e2e, "gpu_launches": args.steps, "tasks_per_step": n_tasks,
        "modes": modes, "clocks": clocks, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    g.close()


if __name__ == "__main__":
    main()
