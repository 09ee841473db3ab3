"""Benchmark of the PTPC-FP8 MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|skewed|tiny|sweep@T]

A step is one full layer forward (routing, permutation, quantisation, gate/up
GEMM with SwiGLU, requantisation, down GEMM, combine) over one batch of
seeded synthetic inputs, already resident in HBM. The default workload is the
largest one, the Qwen3.5-like layer at T=16384 tokens (D=4096, 512 experts
of I=1024, top-10 plus a shared expert): 4.5 TFLOP over 6.5 GB of touched
FP8 weights, close to the ridge between the FP8 tensor roof and HBM. At N=1
the same run then times every other workload (tiny, decode, prefill, skewed,
T in {1, 64, 512, 4096}) the same way and reports them under
`all_workloads`.

Timing: W untimed warm-up steps, then K timed steps; before every step a
256 MiB buffer is written so no weight stays in the 129 MB L2. Each step is
bracketed by CUDA events recorded by the library on the launching stream
(moe_forward_profiled), which also gives every kernel's duration inside the
timed region. Under torchrun each rank runs its own replica (no data-path
collective); the step time is the max over ranks.

One JSON line on rank 0. `--impl reference` times the CPU oracle instead
(rank 0 only).
"""

import argparse
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

METRIC = "fused-MoE layer tokens/s"
L2_FLUSH_BYTES = 256 << 20
# the largest workload (16384 tokens, 512 experts, top-10 + shared): the line's
# headline; every other workload is timed in the same run under all_workloads
DEFAULT_WORKLOAD = "sweep@16384"
ALL_WORKLOADS = ("tiny", "decode", "prefill", "skewed", "sweep@1", "sweep@64",
                 "sweep@512", "sweep@4096", "sweep@16384")
# GB300 dense FP8 tensor throughput as NVIDIA states it (without sparsity)
NOMINAL_FP8_TFLOPS = 4500.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def workload_config(name):
    """A named workload, "sweep@T", or "custom:T=..,D=..,E=..,k=..,I=..
    [,shared=1][,router=normal]" (used for small profiling captures)."""
    from expert_layer_ptpc_gb300 import synthetic as syn
    if name.startswith("sweep@"):
        return syn.sweep_config(int(name.split("@")[1]))
    if name.startswith("custom:"):
        kv = dict(p.split("=") for p in name[len("custom:"):].split(","))
        return syn.LayerConfig(
            "custom", int(kv["T"]), int(kv["D"]), int(kv["E"]), int(kv["k"]),
            int(kv["I"]), bool(int(kv.get("shared", "0"))),
            kv.get("router", "normal"))
    return syn.CONFIGS[name]


def describe(cfg):
    s = (f"{cfg.name}: T={cfg.T} D={cfg.D} E={cfg.E} top-{cfg.k} I={cfg.I}"
         f"{' + shared expert' if cfg.shared else ''}, PTPC FP8 e4m3"
         f"{', bf16 router GEMM' if cfg.router == 'weights' else ''}")
    return s


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured (MEASURED_PEAKS.json)"
    return 6800.0, 1900.0, "fallback (6.8 TB/s, 1.9 PFLOP/s bf16)"


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed region"
        if len(rows) < 3:
            rows = [s for _, s in self.samples]
            window = "whole run (timed region shorter than the sampling period)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "window": window}


def max_over_ranks(x, device):
    """The largest value of x over all ranks (a replica run is as slow as its
    slowest rank); x itself when no process group is running."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tokens_per_s(T, world, max_ms):
    """Whole-job throughput of `world` replicas that each process T tokens per
    step, the step taking max_ms on the slowest rank."""
    return world * T / (max_ms * 1e-3)


def captured_traffic(cfg, algorithmic_bytes):
    """DRAM traffic of the gate/up launch from a committed ncu record of the
    same kernel instantiation on a smaller case (profiles/traffic_*.json),
    scaled to this launch by its algorithmic bytes. Returns (traffic,
    source), or (None, None) when no record covers this launch's kernel or
    the kernel sources changed since the capture."""
    import hashlib
    per_expert = cfg.T * cfg.k / max(1, cfg.E)
    # the instantiation the gate/up dispatch picks from the rows per expert
    if per_expert <= 16:
        name = "traffic_gateup_decode.json"
    elif per_expert >= 256:
        name = "traffic_gateup_pair.json"
    else:
        return None, None
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None, None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != rec["sources_sha256"]:
        return None, None
    return (rec["traffic_per_algorithmic_byte"] * algorithmic_bytes,
            f"ncu capture of {rec['kernel']} scaled by algorithmic bytes "
            f"(profiles/{name})")


def physical_gpu(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    return parts[local_rank] if local_rank < len(parts) else str(local_rank)


def kernel_launches_per_step(cfg):
    R = cfg.T * cfg.k
    permute = 1 if R <= 8192 else 3
    # routing: one kernel (route) from given logits; from router weights the
    # fused router GEMM + top-k where it applies, else router GEMM + route
    fused = (cfg.E <= 512 and cfg.k <= 16 and cfg.D % 64 == 0 and
             cfg.T * cfg.E * cfg.D >= (1 << 20))
    routing = 2 if cfg.router == "weights" and not fused else 1
    # the down weights' scale bound, when y takes the fp16 encoding (its fp32
    # size reaches 32 MiB)
    bound = 1 if cfg.rows * cfg.D * 4 >= (32 << 20) else 0
    # routing, permute, quant, gate/up GEMM, requant, down GEMM, combine
    return bound + routing + permute + 1 + 1 + 1 + 1 + 1


def algorithmic_bytes(cfg, counts):
    """Bytes the layer must move at least once: every touched expert's FP8
    weights and fp32 channel scales, x and out (bf16), the router input."""
    touched = int((counts[:cfg.E] > 0).sum()) + (1 if cfg.shared else 0)
    per_expert = 3 * cfg.I * cfg.D + 4 * (2 * cfg.I + cfg.D)
    router = 4 * cfg.T * cfg.E if cfg.router != "weights" else 2 * cfg.E * cfg.D
    gate = 2 * cfg.D if cfg.shared else 0
    return touched * per_expert + 2 * cfg.T * cfg.D * 2 + router + gate, touched


def gateup_bytes(cfg, touched):
    """Algorithmic bytes of one gate/up GEMM launch: per touched expert its
    2I x D FP8 weights and 2I fp32 scales; per row the D FP8 codes and scale
    in, the I fp32 outputs out."""
    rows = cfg.rows
    return touched * (2 * cfg.I * cfg.D + 8 * cfg.I) + rows * (cfg.D + 4) + \
        rows * cfg.I * 4


def implementation_bytes(cfg, touched, pre=False):
    """Bytes the forward's launches move, intermediates included (reported
    beside the algorithmic bytes for diagnosis): every launch's reads and
    writes counted once, as if nothing stayed in L2 between launches."""
    T, D, E, k, I = cfg.T, cfg.D, cfg.E, cfg.k, cfg.I
    R, rows = T * k, cfg.rows
    y16 = rows * D * 4 >= (32 << 20)      # the forward's fp16 encoding of y
    ybytes = rows * D * 2 + rows * 4 if y16 else rows * D * 4
    b = 0
    # routing: logits in (or x and the router matrix), ids and weights out
    if cfg.router == "weights":
        fused = (E <= 512 and k <= 16 and D % 64 == 0 and T * E * D >= (1 << 20))
        b += 2 * T * D + 2 * E * D + (0 if fused else 2 * 4 * T * E)
    else:
        b += 4 * T * E
    b += 8 * T * k
    # permutation: ids in; counts, offsets and both row maps out
    b += 4 * R + 8 * (cfg.groups + 1) + 8 * R
    # quantiser: x in (and the residual and gamma, the new residual out, for
    # the pre-norm forward), codes and scales of every destination row out,
    # the shared gate's weights in and gate out
    b += 2 * T * D + (2 * T * D * 2 + 2 * D if pre else 0) + rows * (D + 4)
    b += (2 * D + 4 * T) if cfg.shared else 0
    # gate/up GEMM: weights, codes and scales in, fp32 h out
    b += gateup_bytes(cfg, touched)
    # requantisation: h in, codes and scales out
    b += rows * I * 4 + rows * (I + 4)
    # down GEMM: weights, scales and codes in, y out; the fp16 encoding's
    # bound reads every group's down scales first
    b += touched * (D * I + 4 * D) + rows * (I + 4) + ybytes
    b += cfg.groups * D * 4 + 4 * cfg.groups if y16 else 0
    # combine: y, the row map and the weights in, bf16 out
    b += ybytes + 8 * T * k + 2 * T * D + (4 * T if cfg.shared else 0)
    return b


def layer_flops(cfg):
    router = 2.0 * cfg.T * cfg.D * cfg.E if cfg.router == "weights" else 0.0
    return 2.0 * cfg.rows * cfg.D * 2 * cfg.I + 2.0 * cfg.rows * cfg.I * cfg.D + router


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def _limit_threads():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS"):
        os.environ[v] = "1"


def _oracle_quantize(args):
    cfg_name, e, seed = args
    import oracle
    cfg = workload_config(cfg_name)
    from expert_layer_ptpc_gb300 import synthetic as syn
    gu, d = syn.gen_expert_weights(cfg, e, "cpu", seed)
    return e, oracle.quantize_expert_ref(gu.numpy(), d.numpy())


def _oracle_inputs(cfg_name, seed):
    import oracle
    from expert_layer_ptpc_gb300 import synthetic as syn
    cfg = workload_config(cfg_name)
    x = syn.gen_x(cfg, "cpu", seed).float().numpy()
    if cfg.router == "weights":
        wr = syn.gen_router_weights(cfg, "cpu", seed).float().numpy()
        logits = oracle.router_logits_ref(x, wr)
    else:
        wr, logits = None, syn.gen_logits(cfg, "cpu", seed).numpy()
    wg = syn.gen_shared_gate(cfg, "cpu", seed).float().numpy() if cfg.shared else None
    return cfg, x, wr, logits, wg


_W = {}


def _worker_init(cfg_name, inputs):
    """Timing worker: holds the workload's inputs (x, router matrix, logits,
    shared gate) and quantised weights."""
    _limit_threads()
    x, wr, logits, wg = inputs
    _W.update(cfg=workload_config(cfg_name), x=x, wr=wr, logits=logits, wg=wg,
              quant={})


def _worker_add(quant):
    _W["quant"].update(quant)
    return len(_W["quant"])


def _worker_timed(tokens):
    """Seconds for oracle.moe_forward_ref on `tokens` (routing and permutation
    over the whole batch, expert FFNs for the tokens)."""
    import oracle
    c = _W["cfg"]
    q = _W["quant"]
    t0 = time.perf_counter()
    oracle.moe_forward_ref(_W["x"], c.k, lambda e: q[e], c.E,
                           logits=None if _W["wr"] is not None else _W["logits"],
                           router_w=_W["wr"], w_g=_W["wg"],
                           renormalize=c.renormalize, tokens=tokens)
    return time.perf_counter() - t0


_POOL = None


def oracle_pool():
    """One spawn-started process pool for the oracle's weight quantisation
    (started before it is needed; never forked from a process holding a CUDA
    context)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        _limit_threads()
        _POOL = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 2)))
    return _POOL


class OracleRunner:
    """The shared pool quantises expert weights in parallel (untimed); one
    single-threaded worker runs the timed oracle."""

    def __init__(self, cfg_name, seed=0, inputs=None, pool=None):
        import multiprocessing as mp
        _limit_threads()
        ctx = mp.get_context("spawn")
        self.cfg_name, self.seed = cfg_name, seed
        self.cfg = workload_config(cfg_name)
        if inputs is None:
            _, x, wr, logits, wg = _oracle_inputs(cfg_name, seed)
            inputs = (x, wr, logits, wg)
        self.logits = inputs[2]
        self.quant_pool = pool if pool is not None else oracle_pool()
        self.timer = ctx.Pool(1, initializer=_worker_init,
                              initargs=(cfg_name, inputs))
        self.have = set()

    def prepare(self, tokens):
        import oracle
        cfg = self.cfg
        ids, _ = oracle.route_ref(self.logits, cfg.k, cfg.renormalize)
        es = set(int(e) for e in ids[tokens].ravel())
        if cfg.shared:
            es.add(cfg.E)
        todo = sorted(es - self.have)
        if todo:
            q = dict(self.quant_pool.map(
                _oracle_quantize, [(self.cfg_name, e, self.seed) for e in todo]))
            self.timer.apply(_worker_add, (q,))
            self.have |= set(todo)

    def time(self, tokens):
        return self.timer.apply(_worker_timed, (list(tokens),))

    def close(self):
        self.timer.terminate()


def cpu_baseline(cfg_name, seed=0, budget_s=20.0, pool=None):
    """The oracle, as it stands, timed on this host on a bounded sample of the
    workload's tokens. Weight quantisation (done once per model on both
    sides) is outside the timing."""
    cfg = workload_config(cfg_name)
    run = OracleRunner(cfg_name, seed, pool=pool)
    try:
        run.prepare([0])
        dt1 = run.time([0])
        n_tok = int(max(1, min(cfg.T, budget_s // max(dt1, 1e-3))))
        tokens = list(range(n_tok))
        run.prepare(tokens)
        dt = run.time(tokens)
    finally:
        run.close()
    return {"value": n_tok / dt, "unit": "tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": (f"first {n_tok} of {cfg.T} tokens of the {cfg.name} "
                       f"batch (routing and permutation over all tokens, expert "
                       f"FFNs for the sample), fp64 numpy, 1 BLAS thread, "
                       f"{dt:.1f} s; weights quantised outside the timing")}


def bench_config(cfg, touched, world):
    """The `config` object of a JSON line, the same for both arms."""
    return {"workload": describe(cfg), "T": cfg.T, "D": cfg.D, "E": cfg.E,
            "k": cfg.k, "I": cfg.I, "shared": cfg.shared,
            "touched_experts": int(touched),
            "l2": "flushed before every step (256 MiB write)",
            "parallelism": f"replicas x{world}"}


def _reference_inputs(cfg, seed=0):
    """x, router input and shared gate of the workload as the GPU arm draws
    them (on the GPU when there is one, so both arms route the same tokens),
    as numpy arrays."""
    import torch
    import oracle
    from expert_layer_ptpc_gb300 import synthetic as syn
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = syn.gen_x(cfg, dev, seed).float().cpu().numpy()
    if cfg.router == "weights":
        wr = syn.gen_router_weights(cfg, dev, seed).float().cpu().numpy()
        logits = oracle.router_logits_ref(x, wr)
    else:
        wr, logits = None, syn.gen_logits(cfg, dev, seed).cpu().numpy()
    wg = (syn.gen_shared_gate(cfg, dev, seed).float().cpu().numpy()
          if cfg.shared else None)
    return x, wr, logits, wg


def run_reference(args, cfg, world):
    """The reference arm: the CPU oracle, on the GPU arm's tokens. Each step
    evaluates one token of the batch (rotating), routing and permutation over
    the whole batch included. Expert weights come from the same seeded
    recipe, drawn on the host (their values do not change the oracle's
    time)."""
    import numpy as np
    import oracle
    x, wr, logits, wg = _reference_inputs(cfg)
    ids, _ = oracle.route_ref(logits, cfg.k, cfg.renormalize)
    touched = int((np.bincount(ids.ravel(), minlength=cfg.E) > 0).sum())
    run = OracleRunner(args.workload, 0, inputs=(x, wr, logits, wg))
    try:
        steps = [i % cfg.T for i in range(args.warmup + args.steps)]
        run.prepare(sorted(set(steps)))
        for t in steps[:args.warmup]:
            run.time([t])
        times = [run.time([t]) for t in steps[args.warmup:]]
    finally:
        run.close()
    total = sum(times)
    value = args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": bench_config(cfg, touched, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1,
                         "kind": "oracle",
                         "sample": "one token of the batch per step (expert "
                                   "FFNs of its experts; routing and "
                                   "permutation over the batch), fp64 numpy, "
                                   "1 BLAS thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Workload:
    """A layer with its seeded inputs on the device, ready to time."""

    def __init__(self, cfg, dev, layer=None, prenorm=False):
        import torch
        from expert_layer_ptpc_gb300 import synthetic as syn
        from expert_layer_ptpc_gb300.layer import MoELayer
        self.cfg = cfg
        self.layer = layer if layer is not None else MoELayer.synthetic(cfg, dev, seed=0)
        self.x = syn.gen_x(cfg, dev, 0)
        self.logits = None if cfg.router == "weights" else syn.gen_logits(cfg, dev, 0)
        self.out = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device=dev)
        self.ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
        self.tw = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
        self.pre = {}
        if prenorm:   # layer input = RMSNorm(x + residual) * gamma
            if self.logits is None:
                raise SystemExit("--prenorm needs a workload with router logits")
            g = torch.Generator(device="cpu").manual_seed(12345)
            res = (torch.randn(cfg.T, cfg.D, generator=g) * 0.5).to(torch.bfloat16).to(dev)
            gamma = (1.0 + 0.1 * torch.randn(cfg.D, generator=g)).to(torch.bfloat16).to(dev)
            self.pre = {"residual": res, "gamma": gamma, "eps": 1e-6,
                        "residual_out": torch.empty_like(res)}

    def step(self, evs=None):
        self.layer.forward(self.x, self.logits, out=self.out, topk_ids=self.ids,
                           topk_w=self.tw, events=evs, **self.pre)

    def check_status(self, where):
        st, bits = self.layer.status()
        if st != 0:
            raise RuntimeError(f"device status {st} ({bits:#x}) {where}")


def measure(args, w, stream, flush, sampler=None, graph=True):
    """W warm-up steps, K timed graph replays (L2 flushed before each), then
    K steps with the library's per-kernel marks. Returns step times (ms),
    per-kernel times (ms) and the wall-clock window of the timed steps."""
    import torch
    from expert_layer_ptpc_gb300 import binding
    nev = binding.MOE_FORWARD_EVENTS

    def make_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)]
               for _ in range(n)]
        for row in evs:          # create the driver events up front
            for e in row:
                e.record(stream)
        return evs

    warm = make_events(1)[0]
    for _ in range(max(args.warmup, 1)):
        flush.fill_(1)
        w.step(warm)
    torch.cuda.synchronize()
    w.check_status("after warm-up")

    # The step a serving loop runs: one CUDA graph holding the whole forward
    # (kernels chained with programmatic dependent launch).
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            w.step()
        g.replay()
        torch.cuda.synchronize()

    marks = [(torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if sampler is not None:
        sampler.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        marks[i][0].record(stream)
        if g is not None:
            g.replay()
        else:
            w.step()
        marks[i][1].record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.barrier()
    t1 = time.time()
    w.check_status("in the timed region")
    step_ms = [a.elapsed_time(b) for a, b in marks]

    # the same forward with the library's step marks, to time each kernel on
    # its launching stream (the marks serialise the kernels)
    evs = make_events(args.steps)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        w.step(evs[i])
    torch.cuda.synchronize()
    w.check_status("in the profiled run")
    phase_ms = [[e[j].elapsed_time(e[j + 1]) for e in evs] for j in range(nev - 1)]
    profiled_ms = sum(e[0].elapsed_time(e[nev - 1]) for e in evs) / len(evs)
    del g
    return step_ms, phase_ms, profiled_ms, (t0, t1)


def rooflines(cfg, counts, step_ms, phase_ms, pre=False):
    """Roofline of the gate/up GEMM launch and of the whole layer step."""
    B, touched = algorithmic_bytes(cfg, counts)
    if pre:   # the residual read and the new residual written, gamma
        B += 2 * cfg.T * cfg.D * 2 + 2 * cfg.D
    F = layer_flops(cfg)
    hbm, bf16, peak_src = peaks()
    fp8_peak = 2.0 * bf16     # measured bf16 x the nominal fp8/bf16 ratio of 2
    gemm_ms = sum(phase_ms[4]) / len(phase_ms[4])
    gu_bytes = gateup_bytes(cfg, touched)
    # the gate/up GEMM: bound by whichever roof is lower for its bytes/flops
    gu_flops = 2.0 * cfg.rows * cfg.D * 2 * cfg.I
    tensor_bound = gu_flops / (fp8_peak * 1e12) > gu_bytes / (hbm * 1e9)
    if tensor_bound:
        ach = gu_flops / (gemm_ms * 1e-3) / 1e12
        gemm = {"bound": "tensor", "achieved": ach, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": ach / fp8_peak,
                "peak_source": peak_src + ", fp8 = 2 x bf16 burst",
                "frac_of_nominal_fp8": ach / NOMINAL_FP8_TFLOPS}
    else:
        ach = gu_bytes / (gemm_ms * 1e-3) / 1e9
        gemm = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": peak_src}
    traffic, tsrc = captured_traffic(cfg, gu_bytes)
    gemm.update({
        "kernel": "gate/up grouped GEMM (tcgen05, SwiGLU epilogue)",
        "traffic": traffic, "traffic_source": tsrc,
        "algorithmic_bytes_per_launch": gu_bytes,
        "flops_per_launch": gu_flops, "ms_per_launch": gemm_ms})
    ms = statistics.mean(step_ms)
    t_roof = max(F / (fp8_peak * 1e12), B / (hbm * 1e9))
    B_impl = implementation_bytes(cfg, touched, pre)
    layer = {
        "bound": "tensor" if F / (fp8_peak * 1e12) > B / (hbm * 1e9) else "hbm",
        "algorithmic_bytes": B, "flops": F,
        "achieved_gbs": B / (ms * 1e-3) / 1e9,
        "achieved_fp8_tflops": F / (ms * 1e-3) / 1e12,
        "t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms * 1e-3),
        "frac_tensor_of_nominal_fp8": F / (ms * 1e-3) / 1e12 / NOMINAL_FP8_TFLOPS,
        # diagnosis: the bytes the launches move with the intermediates
        "implementation_bytes": B_impl,
        "implementation_gbs": B_impl / (ms * 1e-3) / 1e9}
    return gemm, layer, touched


KERNEL_NAMES = ["router", "route", "permute", "quant_x", "gateup_gemm", "requant",
                "down_gemm", "combine"]


def kernel_times(phase_ms, pre=False):
    names = list(KERNEL_NAMES)
    if pre:
        names[3] = "addnorm_quant_x"
    return {n: round(sum(p) / len(p), 5) for n, p in zip(names, phase_ms)}


def run_all_workloads(args, dev, stream, flush, sweep_layer, pool):
    """Every workload but the headline one, each timed the same way (graph
    replays, L2 flushed before each step) with its roofline fractions and the
    oracle's speed on a few of its tokens."""
    import torch
    from expert_layer_ptpc_gb300 import synthetic as syn
    res = {}
    for name in ALL_WORKLOADS:
        if name == args.workload:
            continue
        cfg = workload_config(name)
        layer = sweep_layer if name.startswith("sweep@") else None
        w = Workload(cfg, dev, layer=layer)
        step_ms, phase_ms, _, _ = measure(args, w, stream, flush)
        counts = torch.bincount(w.ids.view(-1).long(), minlength=cfg.E).cpu().numpy()
        gemm, layer_rf, touched = rooflines(cfg, counts, step_ms, phase_ms)
        ms = statistics.mean(step_ms)
        res[name] = {
            "workload": describe(cfg), "tokens_per_s": cfg.T / (ms * 1e-3),
            "ms_per_step": ms, "touched_experts": touched,
            "layer_roofline": {k: layer_rf[k] for k in (
                "bound", "frac", "t_roof_ms", "achieved_gbs", "achieved_fp8_tflops",
                "implementation_bytes")},
            "gateup_gemm_roofline": {k: gemm[k] for k in (
                "bound", "frac", "achieved", "unit", "ms_per_launch")},
            "kernel_ms": kernel_times(phase_ms),
            "cpu_baseline": (None if args.no_cpu_baseline else
                             cpu_baseline(name, budget_s=3.0, pool=pool)),
        }
        del w
        if layer is None:
            torch.cuda.empty_cache()
    return res


def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from expert_layer_ptpc_gb300 import build
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = Workload(cfg, dev, prenorm=args.prenorm)
    pre = w.pre
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    sampler = ClockSampler(physical_gpu(local_rank))
    sampler.barrier = (lambda: dist.barrier()) if world > 1 else (lambda: None)
    sampler.start()
    time.sleep(0.3)
    step_ms, phase_ms, profiled_ms, (t_wall0, t_wall1) = measure(
        args, w, stream, flush, sampler, graph=not args.no_graph)
    time.sleep(0.3)
    sampler.stop()
    mean_ms = sum(step_ms) / len(step_ms)
    max_ms = max_over_ranks(mean_ms, dev)

    # e2e: the same forward through the public API from pinned host buffers,
    # copies in and out inside the timed region, pipelined the way a serving
    # loop runs it: two slots of device buffers; batch i+1 is copied in (one
    # stream) and batch i-1's output copied out (another) while batch i's
    # forward runs. The time of K steps is taken from the start of the first
    # copy-in to the end of the last copy-out.
    x, logits, out, layer = w.x, w.logits, w.out, w.layer
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    x_h = x.cpu().pin_memory()
    lg_h = logits.cpu().pin_memory() if logits is not None else None
    out_h = [torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    lg_d = [torch.empty_like(logits) if logits is not None else None for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    if pre:   # the residual stream goes in and comes back too
        res_h = pre["residual"].cpu().pin_memory()
        res_out_h = [torch.empty_like(res_h).pin_memory() for _ in range(2)]
        res_d = [torch.empty_like(pre["residual"]) for _ in range(2)]
        res_out_d = [torch.empty_like(pre["residual"]) for _ in range(2)]
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "comp", "out")}
    # weights below 512 MiB could stay in L2 from one step to the next: the
    # L2 is flushed on the compute stream before each of those forwards
    weights_bytes = layer.w_gu.numel() + layer.w_d.numel()
    flush_e2e = weights_bytes < (512 << 20)

    def e2e_steps(n):
        for i in range(n):
            sl = i % 2
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev["comp"][sl])    # forward i-2 read this slot
                x_d[sl].copy_(x_h, non_blocking=True)
                if lg_h is not None:
                    lg_d[sl].copy_(lg_h, non_blocking=True)
                if pre:
                    res_d[sl].copy_(res_h, non_blocking=True)
                ev["in"][sl].record(cin)
            stream.wait_event(ev["in"][sl])
            if i >= 2:
                stream.wait_event(ev["out"][sl])      # output i-2 copied out
            if flush_e2e:
                flush.fill_(i & 0xFF)
            if pre:
                layer.forward(x_d[sl], lg_d[sl], out=out_d[sl], residual=res_d[sl],
                              gamma=pre["gamma"], eps=pre["eps"],
                              residual_out=res_out_d[sl], stream=stream)
            else:
                layer.forward(x_d[sl], lg_d[sl], out=out_d[sl], stream=stream)
            ev["comp"][sl].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev["comp"][sl])
                out_h[sl].copy_(out_d[sl], non_blocking=True)
                if pre:
                    res_out_h[sl].copy_(res_out_d[sl], non_blocking=True)
                ev["out"][sl].record(cout)

    e2e_steps(max(args.warmup, 2))
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(cin)
    e2e_steps(args.steps)
    b.record(cout)          # after the last copy-out
    torch.cuda.synchronize()
    w.check_status("in the end-to-end run")
    e2e_mean = a.elapsed_time(b) / args.steps
    e2e_max = max_over_ranks(e2e_mean, dev)
    h2d = x.numel() * 2 + (logits.numel() * 4 if logits is not None else 0)
    d2h = out.numel() * 2
    if pre:
        h2d += pre["residual"].numel() * 2
        d2h += pre["residual"].numel() * 2

    if rank != 0:
        return
    counts = torch.bincount(w.ids.view(-1).long(), minlength=cfg.E).cpu().numpy()
    gemm_roofline, layer_roofline, touched = rooflines(
        cfg, counts, [max_ms], phase_ms, bool(pre))
    kernel_ms = kernel_times(phase_ms, bool(pre))
    dominant = max(kernel_ms, key=kernel_ms.get)
    clocks = sampler.summary(t_wall0, t_wall1)
    prenorm = None
    if pre:
        # the fused add + RMSNorm + quant launch: x, residual and gamma in;
        # the new residual, the codes of every destination row (k + shared)
        # and their scales (and the gate) out. Unfused, the normalised bf16
        # activations would be written and read once more.
        hbm = peaks()[0]
        q_ms = sum(phase_ms[3]) / len(phase_ms[3])
        qb = 3 * cfg.T * cfg.D * 2 + 2 * cfg.D + cfg.rows * (cfg.D + 4) + \
            (4 * cfg.T + 2 * cfg.D if cfg.shared else 0)
        prenorm = {"kernel": "add + RMSNorm + per-token FP8 quant (fused)",
                   "ms_per_launch": q_ms, "algorithmic_bytes_per_launch": qb,
                   "achieved_gbs": qb / (q_ms * 1e-3) / 1e9,
                   "frac": qb / (q_ms * 1e-3) / 1e9 / hbm, "peak_gbs": hbm,
                   "unfused_extra_bytes": 2 * cfg.T * cfg.D * 2}
    tokens_per_s = replica_tokens_per_s(cfg.T, world, max_ms)
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
        "data": "synthetic",
        "config": bench_config(cfg, touched, world),
        "cuda_graph": not args.no_graph,
        "roofline": gemm_roofline,
        "layer_roofline": layer_roofline,
        "kernel_ms": kernel_ms, "dominant_kernel": dominant,
        "profiled_ms_per_step": profiled_ms,
        "e2e": {"value": replica_tokens_per_s(cfg.T, world, e2e_max),
                "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_max,
                "pipeline": "two buffer slots: copy-in of batch i+1 and copy-out "
                            "of batch i-1 on their own streams during forward i",
                "l2": ("flushed before every forward" if flush_e2e else
                       f"not flushed: {weights_bytes / 2**30:.1f} GiB of expert "
                       "weights, larger than L2")},
        "gpu_launches": kernel_launches_per_step(cfg) * args.steps,
        "clocks": clocks,
    }
    if prenorm is not None:
        line["config"]["prenorm"] = {"eps": pre["eps"], "input": "RMSNorm(x + residual) * gamma"}
        line["prenorm"] = prenorm
    if world == 1:
        pool = None if args.no_cpu_baseline else oracle_pool()
        if pool is not None:
            line["cpu_baseline"] = cpu_baseline(args.workload, pool=pool)
        if not args.no_all_workloads and not args.prenorm:
            sweep_layer = layer if cfg.name.startswith("sweep") else None
            del w
            line["all_workloads"] = run_all_workloads(args, dev, stream, flush,
                                                      sweep_layer, pool)
    print(json.dumps(line), flush=True)


def run_compare_scales(args, cfg, local_rank):
    """The workload's two expert GEMMs (gate/up-shaped N = 2I, K = D and
    down-shaped N = D, K = I, over the T k routed rows) with PTPC,
    512-subchannel and BlockScale-128 scales on the one block-scaled engine,
    and the production PTPC grouped GEMM beside them. Each launch is timed
    with CUDA events on its stream, L2 flushed before every call; the median
    of `steps` calls. One JSON line."""
    import torch
    from expert_layer_ptpc_gb300 import binding, build, scaled
    build.build()
    torch.cuda.set_device(local_rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def median_ms(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ts = sorted(a.elapsed_time(b) for a, b in ev)
        return ts[len(ts) // 2]

    sampler = ClockSampler(physical_gpu(local_rank))
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    result = {}
    for which in ("gateup", "down"):
        row = {}
        for mode in ("ptpc", "sub512", "block128"):
            prob = scaled.make_problem(mode, cfg, which)
            row[mode + "_ms"] = median_ms(lambda: scaled.run(prob))
            if mode == "ptpc":
                # the layer's own kernel for this projection: gate/up with its
                # SwiGLU epilogue (N = 2I weight rows in, I columns out), down
                # as a plain PTPC GEMM
                kind = (binding.MOE_GEMM_GATEUP_SWIGLU if which == "gateup"
                        else binding.MOE_GEMM_DOWN)
                R0 = prob["qa"].shape[0]
                n_out = prob["qw"].shape[1] // (2 if which == "gateup" else 1)
                prod_out = torch.empty((R0, n_out), dtype=torch.float32, device="cuda")
                row["ptpc_production_ms"] = median_ms(lambda: binding.moe_grouped_gemm(
                    kind, prob["qa"], prob["sa"], prob["qw"], prob["sw"],
                    prob["offsets"], out=prod_out))
                row["ptpc_production_kernel"] = (
                    "gate/up with SwiGLU" if which == "gateup" else "down")
                del prod_out
                R, K = prob["qa"].shape
                N = prob["qw"].shape[1]
                row["shape"] = {"rows": R, "N": N, "K": K, "groups": cfg.E}
                row["flops"] = 2.0 * R * N * K
            del prob
            torch.cuda.empty_cache()
        st, bits = binding.moe_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} ({bits:#x})")
        for k in ("ptpc", "sub512", "block128", "ptpc_production"):
            row[k + "_tflops"] = row["flops"] / (row[k + "_ms"] * 1e-3) / 1e12
        row["block128_over_ptpc"] = row["block128_ms"] / row["ptpc_ms"]
        row["sub512_over_ptpc"] = row["sub512_ms"] / row["ptpc_ms"]
        result[which] = row
    t1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    print(json.dumps({
        "metric": "scale_granularity_gemm_ms", "unit": "ms", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "e4m3",
        "data": "synthetic", "config": {"workload": describe(cfg),
                                        "l2": "flushed before every call"},
        "engine": "one tcgen05 engine for all three modes (128 x 128 tiles); "
                  "ptpc_production = moe_grouped_gemm, the layer's own kernel "
                  "(gate/up: with its SwiGLU epilogue)",
        "gemms": result, "clocks": sampler.summary(t0, t1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-workloads", action="store_true",
                    help="time only the named workload (the others are "
                         "otherwise timed after it, N=1 only)")
    ap.add_argument("--router-gemm", action="store_true",
                    help="route every workload from a bf16 router matrix: the "
                         "fused tensor-core router GEMM + top-k is in the step")
    ap.add_argument("--prenorm", action="store_true",
                    help="feed the layer from the residual stream: fused add + "
                         "RMSNorm + quant replaces the quantisation step")
    ap.add_argument("--compare-scales", action="store_true",
                    help="time the workload's expert GEMMs with PTPC, "
                         "512-subchannel and BlockScale-128 scales (one JSON line)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the forward directly instead of replaying a "
                         "CUDA graph of it")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = workload_config(args.workload)
    if args.router_gemm and cfg.router != "weights":
        # route from a bf16 router matrix (N(0, 0.02)) through the layer's
        # fused router GEMM + top-k instead of the workload's given logits
        from dataclasses import replace
        cfg = replace(cfg, router="weights")

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg, world)
        return
    if args.compare_scales:
        if rank == 0:
            run_compare_scales(args, cfg, local_rank)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, cfg, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
