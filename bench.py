"""Benchmark: Falcon-1 chunked forward on GB300 (tokens/s and roofline).

Workload (one step = one chunked forward over one batch of synthetic
inputs): Falcon-1, B=8, T=2048, H=12, d_k=d_v=64, bf16 q/k/v/o, fp32 state,
chunk 64 — the layer shape of the pages' 124-130M-parameter models.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one replica per GPU (weak scaling: each rank
processes its own batch; the path has no exchange step, so there is no
data-path collective).  Timing: W untimed steps, then K steps between a
barrier + synchronize on both sides, CUDA events on the launching stream,
max over ranks.  The inputs of one step (~102 MB) fit in L2 (129 MB), so the
steps rotate through 4 input sets (~410 MB) and each step reads inputs that
the previous steps evicted.  Rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_SETS = 4
VARIANT_NAMES = ("falcon1", "falcon1a", "falcon2", "falcon2a", "falcon3", "falcon3a")
METRIC = "Falcon-1 chunked fwd tokens/s and % of roofline (GB300, T=2048, H=12, d=64)"


# ---- replicas across ranks (the path has no exchange step: each rank runs
# its own batch; only the timing is combined)
def replica_seed(w, rank: int, i: int) -> int:
    """Seed of input set i on rank `rank`: every replica draws its own batch."""
    return w.seed + 100 * rank + i


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (the job's time); world 1 passes it through."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(w, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return w.B * w.T * world / (ms_per_step / 1e3)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="lm124m_f1_8x2048x12_d64")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--mode", choices=["chunk", "decode", "backward", "varlen"], default="chunk",
                    help="decode: the recurrent one-token step (256 sequences x 12 heads); "
                         "backward: the gradient of the chunk forward for the workload; "
                         "varlen: the workload's B sequences packed with a mix of lengths")
    ap.add_argument("--prologue", action="store_true",
                    help="raw q, k and gate logits: the library applies phi and the sigmoids")
    ap.add_argument("--decode-variant", type=int, default=0)
    ap.add_argument("--pairing", choices=["prefix", "same"], default="prefix",
                    help="same: the same-step pairing ablation (x_t = k_t)")
    ap.add_argument("--sets", type=int, default=N_SETS,
                    help="rotating input sets (fewer only for profiler captures)")
    return ap.parse_args()


def get_workload(name):
    from workloads import WORKLOADS
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


def algorithmic_bytes(w) -> int:
    """Bytes the method must move per forward: q, k, v in and o out in the
    input dtype, beta and lambda in fp32, the final state once in fp32."""
    es = 2 if w.dtype == "bf16" else 4
    th = w.B * w.T * w.H
    beta = th * (w.dv if w.per_channel else 1) * 4
    return th * (2 * w.dk + w.dv + w.dv) * es + beta + th * 4 + w.B * w.H * w.dk * w.dv * 4


def kernel_bytes(w, names) -> list:
    """Algorithmic bytes each kernel of the path must move (the method's own
    inputs and outputs that the kernel touches; intermediates are not
    counted).  The per-chunk kernel reads k, v and the gate inputs, the
    sequential one q and k and writes o and the final state."""
    es = 2 if w.dtype == "bf16" else 4
    th = w.B * w.T * w.H
    beta = th * (w.dv if w.per_channel else 1) * 4
    if len(names) == 1:  # one kernel does the whole forward
        return [algorithmic_bytes(w)]
    state = w.B * w.H * w.dk * w.dv * 4
    if names[0] == "window_prep_kernel":  # keys and gate inputs; then the whole forward
        return [th * w.dk * es + beta + th * 4, algorithmic_bytes(w)]
    if names[0] == "f3a_chunk_kernel":  # q, k, v and gate inputs; then q in, o and the state out
        mid = [0] if len(names) == 3 else []  # the group totals read intermediates only
        return [th * (2 * w.dk + w.dv) * es + beta + th * 4] + mid + [th * (w.dk + w.dv) * es + state]
    if names[0] == "f3_chunk_kernel":  # q, k, v and gate inputs; then o and the state out
        return [th * (2 * w.dk + w.dv) * es + beta + th * 4, th * w.dv * es + state]
    return [th * (w.dk + w.dv) * es + beta + th * 4, th * (2 * w.dk + w.dv) * es + state]


def algorithmic_flops(w) -> int:
    th = w.B * w.T * w.H
    if w.variant in (1, 3, 5):
        per = w.chunk * (w.dk + w.dv) + 4 * w.dk * w.dv
    elif w.variant == 4:
        per = (4 * w.window + 2) * w.dk * w.dv
    else:
        per = w.chunk * (2 * w.dk + 2 * w.dv) + 6 * w.dk * w.dv
    return th * per


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def _oracle_task(task):
    """One oracle run (fp64 numpy recurrence) on a slice of the inputs; runs
    in a worker process."""
    x, variant, window, eps, eps_gamma, pairing = task
    import oracle
    oracle.recurrent(**x, variant=variant, window=window, eps=eps, eps_gamma=eps_gamma,
                     pairing=pairing)
    return x["q"].shape[0] * x["q"].shape[1]


def _oracle_import(_):
    """Worker warm-up: import the oracle (and numpy) before anything is timed."""
    import oracle  # noqa: F401
    return os.getpid()


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


class OraclePool:
    """The oracle over all host cores: one single-threaded worker process per
    core (spawned, so no CUDA state is inherited), the workload split by
    sequence and head so every core has work."""

    def __init__(self):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"   # workers inherit it: one thread each
        self.cores = os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.pool.map(_oracle_import, range(4 * self.cores), chunksize=1)

    def tasks(self, w, x):
        """Split [B, T, H, ...] inputs into about `cores` (sequence, head group) slices."""
        B, H = x["q"].shape[0], x["q"].shape[2]
        groups = max(1, min(H, -(-self.cores // B)))
        bounds = [(H * g) // groups for g in range(groups + 1)]
        out = []
        for b in range(B):
            for g in range(groups):
                h0, h1 = bounds[g], bounds[g + 1]
                sl = {k: v[b:b + 1, :, h0:h1] for k, v in x.items()}
                out.append((sl, w.variant, w.window, w.eps, w.eps_gamma, w.pairing))
        return out

    def run(self, tasks) -> float:
        t0 = time.perf_counter()
        self.pool.map(_oracle_task, tasks, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(w, budget_s=20.0) -> dict:
    """The oracle as it stands (fp64 token-by-token recurrence) over every
    host core on the whole workload (all sequences, heads and tokens),
    repeated while the budget lasts."""
    from workloads import make_inputs
    x = {k: v.double().numpy() for k, v in make_inputs(w).items()}
    pool = OraclePool()
    try:
        tasks = pool.tasks(w, x)
        times = [pool.run(tasks)]
        while sum(times) < budget_s / 2 and len(times) < 5:
            times.append(pool.run(tasks))
    finally:
        pool.close()
    dt = statistics.median(times)
    return {"value": w.B * w.T / dt, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"the whole workload ({w.B} sequences x {w.T} tokens x {w.H} heads), fp64 numpy "
                      f"recurrence, {len(tasks)} (sequence, head group) tasks on {pool.cores} "
                      f"single-threaded worker processes, median of {len(times)} run(s)"}


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel and on this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("workload") != workload:
        return None
    import hashlib
    src = os.path.join(ROOT, "chunked_delta_rule_gb300", "csrc", rec["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return rec["bytes_per_launch"] if h == rec["source_sha"] else None


def run_reference(args, w, rank):
    """The reference arm: the oracle, as it stands, over every host core.
    Each step runs a bounded sample of the workload (the first sequences'
    first tokens, all heads), sized so that the whole run stays within about
    two minutes of CPU time; the throughput is the sample's tokens over its
    time."""
    if rank != 0:
        return
    from workloads import make_inputs
    pool = OraclePool()
    try:
        full = {k: v.double().numpy() for k, v in make_inputs(w).items()}
        per_step = 90.0 / max(args.steps + args.warmup, 1)   # seconds of wall time per step
        Tp = min(w.T, 128)
        t_seq = pool.run(pool.tasks(w, {k: v[:1, :Tp] for k, v in full.items()})) / Tp  # s per token
        busy = min(w.H, pool.cores) / pool.cores   # share of the cores one sequence keeps busy
        if t_seq * w.T * w.B * busy <= per_step:   # the whole workload fits in a step
            nb, T = w.B, w.T
        else:
            nb, T = 1, int(max(16, min(w.T, per_step / max(t_seq, 1e-9))))
        x = {k: v[:nb, :T] for k, v in full.items()}
        tasks = pool.tasks(w, x)
        for _ in range(args.warmup):
            pool.run(tasks)
        times = [pool.run(tasks) for _ in range(args.steps)]
    finally:
        pool.close()
    dt = statistics.mean(times)
    value = nb * T / dt
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
                             "cpu": cpu_model(),
                             "sample": f"per step {nb} of {w.B} sequences x the first {T} of {w.T} tokens "
                                       f"x {w.H} heads, fp64 numpy recurrence, {len(tasks)} tasks on "
                                       f"{pool.cores} single-threaded worker processes"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_config(w, world, n_sets=N_SETS, abytes=None, prologue=False) -> dict:
    """The workload description shared by both arms' JSON lines."""
    cfg = {"workload": w.name + ("_prologue" if prologue else ""), "B": w.B, "T": w.T, "H": w.H,
           "dk": w.dk, "dv": w.dv, "chunk": w.chunk, "variant": VARIANT_NAMES[w.variant],
           "global_batch": w.B * world, "seq_len": w.T, "parallelism": f"replicas x{world}"}
    if abytes is not None:
        cfg["l2"] = f"rotating {n_sets} input sets ({n_sets * abytes / 1e6:.0f} MB)"
    return cfg


def run_decode(args):
    """Recurrent decode step: one token for 256 sequences x 12 heads, d = 64,
    fp32 state in HBM.  4 state sets (4 x 50 MB) rotate so every step reads
    a state that is not in L2."""
    import torch

    import chunked_delta_rule_gb300 as F
    from workloads import make_decode_inputs
    torch.cuda.set_device(0)
    sets = []
    for i in range(args.sets):
        x, carry, w = make_decode_inputs(args.decode_variant, window=8, seed=5 + 10 * i,
                                         device="cuda")
        sets.append((x, carry))
    p = F.Params(B=w.B, T=1, H=w.H, dk=w.dk, dv=w.dv, window=w.window, variant=w.variant,
                 dtype=F.FALCON_BF16)
    o = torch.empty((w.B, 1, w.H, w.dv), dtype=torch.bfloat16, device="cuda")

    def step(i):
        x, c = sets[i % len(sets)]
        F.falcon_recurrent_step(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], c, o,
                                torch.cuda.current_stream())

    # the step is a few microseconds of GPU time: replay it from a CUDA graph
    # so the host's per-call overhead does not set the pace
    per_graph = 32
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(per_graph):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // per_graph)
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * per_graph)
    args.steps = reps * per_graph
    bh = w.B * w.H
    Wp = w.window if w.variant in (4, 5) else 1
    nbytes = bh * (2 * w.dk * w.dv * 4 + (w.dk + 2 * w.dk + 2 * w.dv) * 2 + 8 + 8
                   + (Wp - 1) * (w.dk + w.dv) * 2 + (w.dk + w.dv) * 2 * (Wp > 1))
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"metric": "Falcon recurrent decode step tokens/s", "value": w.B / (ms / 1e3),
                      "unit": "tokens/s", "ms_per_step": ms, "steps": args.steps,
                      "config": {"workload": f"decode_{w.B}x{w.H}_d{w.dk}", "variant": w.variant,
                                 "window": Wp, "state_sets": len(sets)},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                   "frac": gbs / peak, "algorithmic_bytes": nbytes,
                                   "kernel": "recurrent_step_kernel"}}), flush=True)


def run_backward(args, w):
    """Backward of the chunk forward (dq, dk, dv, dbeta, dlambda from dO)
    for the workload, 4 rotating input sets; one kernel per call."""
    import torch

    import chunked_delta_rule_gb300 as F
    from workloads import make_cotangents, make_inputs
    torch.cuda.set_device(0)
    p = F.Params(B=w.B, T=w.T, H=w.H, dk=w.dk, dv=w.dv, chunk=w.chunk, window=w.window, eps=w.eps,
                 eps_gamma=w.eps_gamma, variant=w.variant,
                 dtype=F.FALCON_BF16 if w.dtype == "bf16" else F.FALCON_F32,
                 pairing=F.FALCON_PAIR_SAME_STEP if w.pairing == "same" else F.FALCON_PAIR_PREFIX)
    chunked = w.variant in (0, 1) and w.dk == 64 and w.dv == 64
    chunk_k = ("bwdc_prep_tc_kernel + bwdc_chain_tc_kernel (both chains) + bwdc_grad_tc_kernel"
               if w.dtype == "bf16" else
               "bwdc_prep_kernel + bwdc_fwd_chain_kernel + bwdc_bwd_chain_kernel + bwdc_grad_kernel")
    kernel = (f"{chunk_k} (whole call)"
              if chunked else "falcon_bwd_win_kernel" if (w.variant in (4, 5) or w.dk == 128)
              else "falcon_bwd_kernel")
    sets = []
    for i in range(args.sets):
        x = make_inputs(w, seed=w.seed + i, device="cuda")
        x.update(make_cotangents(w, 50 + i, device="cuda", with_dS=False))
        sets.append(x)
    g = {n: torch.empty_like(sets[0][m]) for n, m in
         (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dlam", "lam"))}
    ws_n = F.falcon_backward_workspace_size(p)
    ws = F.alloc_workspace(ws_n)
    stream = torch.cuda.current_stream()

    def step(i):
        x = sets[i % len(sets)]
        F.falcon_backward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, x["dO"], None,
                          g["dq"], g["dk"], g["dv"], g["dbeta"], g["dlam"], None, None, ws, ws_n,
                          stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    es = 2 if w.dtype == "bf16" else 4
    th = w.B * w.T * w.H
    beta = th * (w.dv if w.per_channel else 1) * 4
    # q, k, v, dO in and dq, dk, dv out in the dtype; beta, lambda in and
    # their gradients out in fp32
    nbytes = th * (2 * w.dk + w.dv + w.dv) * es + th * (2 * w.dk + w.dv) * es + 2 * (beta + th * 4)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"metric": "Falcon chunked backward tokens/s", "value": w.B * w.T / (ms / 1e3),
                      "unit": "tokens/s", "ms_per_step": ms, "steps": args.steps,
                      "warmup": args.warmup, "higher_is_better": True,
                      "dtype": "bf16" if w.dtype == "bf16" else "f32",
                      "config": {"workload": w.name + "_backward", "B": w.B, "T": w.T, "H": w.H,
                                 "dk": w.dk, "dv": w.dv, "variant": w.variant, "window": w.window,
                                 "pairing": w.pairing, "l2": f"rotating {len(sets)} input sets"},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                   "frac": gbs / peak, "algorithmic_bytes": nbytes,
                                   "kernel": kernel,
                                   "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
                      "gpu_launches": args.steps * (4 if chunked else 1),
                      "clocks": clk}), flush=True)


VARLEN_FRACTIONS = (1.0, 0.75, 0.5, 0.25, 1.0, 0.125, 0.875, 0.375)


def run_varlen(args, w):
    """Packed sequences: the workload's B sequences with lengths T x (1, 3/4,
    1/2, 1/4, 1, 1/8, 7/8, 3/8) (cycled), one falcon_chunk_fwd_varlen call per
    step; tokens/s counts the real tokens."""
    import torch

    import chunked_delta_rule_gb300 as F
    from workloads import make_inputs, make_raw_inputs, pack_varlen
    torch.cuda.set_device(0)
    lengths = [max(1, int(w.T * VARLEN_FRACTIONS[b % len(VARLEN_FRACTIONS)])) for b in range(w.B)]
    p = F.Params(B=w.B, T=w.T, H=w.H, dk=w.dk, dv=w.dv, chunk=w.chunk, window=w.window, eps=w.eps,
                 eps_gamma=w.eps_gamma, variant=w.variant,
                 dtype=F.FALCON_BF16 if w.dtype == "bf16" else F.FALCON_F32,
                 pairing=F.FALCON_PAIR_SAME_STEP if w.pairing == "same" else F.FALCON_PAIR_PREFIX,
                 prologue=3 if args.prologue else 0)
    gen = make_raw_inputs if args.prologue else make_inputs
    sets = []
    for i in range(args.sets):
        packed, cu = pack_varlen(gen(w, seed=w.seed + i), lengths, device="cuda")
        sets.append((packed, cu))
    total = sum(lengths)
    o = torch.empty((total, w.H, w.dv), dtype=sets[0][0]["q"].dtype, device="cuda")
    carry = F.empty_carry(p)
    ws_n = F.falcon_varlen_workspace_size(p)
    ws = F.alloc_workspace(ws_n)
    stream = torch.cuda.current_stream()

    def step(i):
        x, cu = sets[i % len(sets)]
        F.falcon_chunk_fwd_varlen(p, cu, total, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o,
                                  carry, ws, ws_n, stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    wr = w.with_(B=1, T=total)
    abytes = algorithmic_bytes(wr) + (w.B - 1) * w.H * w.dk * w.dv * 4
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("hbm_gbs", 6800.0)
    gbs = abytes / (ms / 1e3) / 1e9
    print(json.dumps({"metric": "Falcon chunked fwd over packed sequences, tokens/s", "value": total / (ms / 1e3),
                      "unit": "tokens/s", "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
                      "higher_is_better": True, "dtype": "bf16" if w.dtype == "bf16" else "f32",
                      "config": {"workload": w.name + "_varlen" + ("_prologue" if args.prologue else ""),
                                 "lengths": lengths, "tokens": total, "H": w.H, "dk": w.dk,
                                 "padded_fraction": 1 - total / (w.B * w.T)},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                   "frac": gbs / peak, "algorithmic_bytes": abytes,
                                   "note": "whole call (gather, kernels, scatter) against the real tokens' bytes"},
                      "clocks": clk}), flush=True)


def main():
    args = parse()
    if args.mode == "decode":
        run_decode(args)
        return
    w = get_workload(args.workload)
    if args.pairing == "same":
        w = w.with_(name=w.name + "_same_step", pairing="same")
    if args.mode == "backward":
        run_backward(args, w)
        return
    if args.mode == "varlen":
        run_varlen(args, w)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    base = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        base = cpu_baseline(w)      # host work first: nothing forked after CUDA init

    import torch
    import torch.distributed as dist

    import chunked_delta_rule_gb300 as F
    from workloads import make_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    p = F.Params(B=w.B, T=w.T, H=w.H, dk=w.dk, dv=w.dv, chunk=w.chunk, window=w.window,
                 eps=w.eps, eps_gamma=w.eps_gamma, variant=w.variant,
                 dtype=F.FALCON_BF16 if w.dtype == "bf16" else F.FALCON_F32,
                 pairing=F.FALCON_PAIR_SAME_STEP if w.pairing == "same" else F.FALCON_PAIR_PREFIX,
                 prologue=3 if args.prologue else 0)
    from workloads import make_raw_inputs
    gen = make_raw_inputs if args.prologue else make_inputs
    sets = [gen(w, seed=replica_seed(w, rank, i), device=dev) for i in range(args.sets)]
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=sets[0]["q"].dtype, device=dev)
    carry = F.empty_carry(p, dev)
    ws_n = F.falcon_workspace_size(p)
    ws = F.alloc_workspace(ws_n, dev) if ws_n else None
    impl_used, launches = F.falcon_chunk_fwd_plan(p)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        x = sets[i % len(sets)]
        F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, carry, ws,
                           ws_n, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and vis.split(",")[local].strip().isdigit():
        gpu_index = int(vis.split(",")[local])
    clocks = ClockSampler(gpu_index)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    # per-kernel times, in a separate pass: the library records the caller's
    # events around each kernel it launches (which keeps every kernel apart)
    nev = launches + 1
    n_k = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(n_k)]
    for evs in ev:
        for e in evs:
            e.record(stream)   # creates the event handles before they are handed over
    torch.cuda.synchronize()
    for i in range(n_k):
        x = sets[i % len(sets)]
        F.falcon_chunk_fwd_timed(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, carry,
                                 ws, ws_n, stream, ev[i])
    torch.cuda.synchronize()
    kern_ms = [statistics.mean(evs[j].elapsed_time(evs[j + 1]) for evs in ev)
               for j in range(launches)]
    per_call_ms = statistics.mean(evs[0].elapsed_time(evs[-1]) for evs in ev)
    ms_step = ms / args.steps
    tokens = w.B * w.T * world
    value = job_tokens_per_s(w, world, ms_step)

    # end to end through the C ABI with host buffers: every step copies its
    # inputs from pinned host memory to the device, makes the call and reads
    # its output back.  Two buffer sets and three streams let step i's input
    # copy run while step i-1 computes and step i-2's output comes back (the
    # copy engines of both directions work at once); each buffer is reused
    # only after the step that last used it is done with it.
    host = {k: v.cpu().pin_memory() for k, v in sets[0].items()}
    dev_in = [{k: torch.empty_like(v) for k, v in sets[0].items()} for _ in range(2)]
    o_dev = [o, torch.empty_like(o)]
    o_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    carry_dev = [carry, F.empty_carry(p, dev)]
    S_host = [torch.empty(carry["S"].shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o.numel() * o.element_size() + carry["S"].numel() * 4   # outputs and the final state
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set j on the device
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the call on set j is done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output j is back on the host

    def e2e_step(i):
        j = i & 1
        s_h2d.wait_event(ev_used[j])
        with torch.cuda.stream(s_h2d):
            for k2 in host:
                dev_in[j][k2].copy_(host[k2], non_blocking=True)
        ev_in[j].record(s_h2d)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])
        x = dev_in[j]
        F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o_dev[j], carry_dev[j],
                           ws, ws_n, stream)
        ev_used[j].record(stream)
        s_d2h.wait_event(ev_used[j])
        with torch.cuda.stream(s_d2h):
            o_host[j].copy_(o_dev[j], non_blocking=True)
            S_host[j].copy_(carry_dev[j]["S"], non_blocking=True)
        ev_out[j].record(s_d2h)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_h2d.wait_event(e0)
    s_d2h.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_out[0])
    stream.wait_event(ev_out[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)

    if rank == 0:
        peaks = {}
        try:
            peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        except Exception:
            pass
        hbm_peak = peaks.get("hbm_gbs", 6800.0)
        abytes = algorithmic_bytes(w)
        if impl_used == F.FALCON_IMPL_SCAN:
            names = ["window_prep_kernel", "window_scan_kernel"]
        elif impl_used != F.FALCON_IMPL_TC:
            names = ["generic_chunk_kernel"]
        elif w.per_channel:
            names = ["tc_f2_kernel"]
        elif w.variant == 5:  # Falcon-3A (the chain in groups: their totals first)
            names = (["f3a_chunk_kernel", "f3a_group_kernel", "f3a_chain_kernel"] if launches == 3
                     else ["f3a_chunk_kernel", "f3a_chain_kernel"])
        elif w.variant == 4:  # Falcon-3
            names = ["f3_chunk_kernel", "f3_chain_kernel"]
        elif w.dk == 64:
            names = ["tc_wyu_kernel", "tc_fwd_chain_kernel"]
        else:
            names = ["tc_wyu_kernel", "tc_fwd_kernel"]
        kbytes = kernel_bytes(w, names)
        if args.prologue and launches > len(names):  # the gather pass: q, k, v and gates in, the same out
            es = 2 if w.dtype == "bf16" else 4
            th = w.B * w.T * w.H
            pb = 2 * (th * (2 * w.dk + w.dv) * es + th * ((w.dv if w.per_channel else 1) + 1) * 4)
            names = ["prologue_kernel"] + names
            kbytes = [pb] + kbytes
        dom = max(range(launches), key=lambda j: kern_ms[j])
        kernel = names[dom]
        achieved = kbytes[dom] / (kern_ms[dom] / 1e3) / 1e9
        step_achieved = abytes / (ms_step / 1e3) / 1e9  # the whole step, kernels overlapped
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"}
        if impl_used == F.FALCON_IMPL_SCAN:
            # fp32 FMA pipes: 152 SMs x 128 lanes x 2 flop per clock at the
            # sampled SM clock (CUDA cores; no tensor-core work on this path)
            mhz = clk.get("sm_mhz") or 2070.0
            alu_peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
            fl = algorithmic_flops(w) / (kern_ms[dom] / 1e3) / 1e12
            roof = {"bound": "alu", "achieved": fl, "peak": alu_peak, "unit": "TFLOP/s",
                    "frac": fl / alu_peak, "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 "
                    "flop x SM clock", "hbm_achieved_gbs": achieved, "hbm_frac": achieved / hbm_peak}
        line = {
            "metric": METRIC,
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": bench_config(w, world, len(sets), abytes, args.prologue),
            "roofline": dict(roof, traffic=traffic_for(kernel, w.name), kernel=kernel,
                             algorithmic_bytes=abytes, algorithmic_flops=algorithmic_flops(w),
                             kernel_algorithmic_bytes=kbytes[dom], step_achieved=step_achieved,
                             step_frac=step_achieved / hbm_peak),
            "kernels": [{"name": n, "ms": kern_ms[j], "share": kern_ms[j] / sum(kern_ms)}
                        for j, n in enumerate(names)],
            "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "clocks": clk,
        }
        if base is not None:
            line["cpu_baseline"] = base
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
