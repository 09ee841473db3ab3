"""Benchmark of the PTPC-FP8 MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|skewed|tiny|sweep@T]

A step is one full layer forward (routing, permutation, quantisation, gate/up
GEMM with SwiGLU, requantisation, down GEMM, combine) over one batch of
seeded synthetic inputs, already resident in HBM. The default workload is the
decode-shaped layer (T=16, D=4096, E=128, top-8, I=1536): it streams the
touched experts' FP8 weights from HBM, so the roofline is HBM bandwidth.

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


def captured_traffic(algorithmic_bytes, bn_decode):
    """DRAM traffic of the gate/up launch from the committed ncu record
    (profiles/traffic_gateup_decode.json), scaled to this launch by its
    algorithmic bytes; None when the record is missing, was taken on another
    tile shape, or the kernel sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_gateup_decode.json")
    if not bn_decode or not os.path.exists(path):
        return None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != rec["sources_sha256"]:
        return None
    return rec["traffic_per_algorithmic_byte"] * algorithmic_bytes


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


def _worker_init(cfg_name, seed):
    """Timing worker: holds the workload's inputs and quantised weights."""
    _limit_threads()
    cfg, x, wr, logits, wg = _oracle_inputs(cfg_name, seed)
    _W.update(cfg=cfg, x=x, wr=wr, logits=logits, wg=wg, quant={})


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


class OracleRunner:
    """A spawn-started pool quantises expert weights in parallel (untimed);
    one single-threaded worker runs the timed oracle."""

    def __init__(self, cfg_name, seed=0):
        import multiprocessing as mp
        _limit_threads()
        ctx = mp.get_context("spawn")
        self.cfg_name, self.seed = cfg_name, seed
        self.cfg, _, _, self.logits, _ = _oracle_inputs(cfg_name, seed)
        self.quant_pool = ctx.Pool(max(1, min(16, os.cpu_count() or 2)))
        self.timer = ctx.Pool(1, initializer=_worker_init,
                              initargs=(cfg_name, seed))
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
        self.quant_pool.terminate()
        self.timer.terminate()


def cpu_baseline(cfg_name, seed=0, budget_s=20.0):
    """The oracle, as it stands, timed on this host on a bounded sample of the
    workload's tokens. Weight quantisation (done once per model on both
    sides) is outside the timing."""
    cfg = workload_config(cfg_name)
    run = OracleRunner(cfg_name, seed)
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


def run_reference(args, cfg):
    """The reference arm: the CPU oracle. Each step evaluates one token of the
    batch (rotating), routing over the whole batch included."""
    run = OracleRunner(args.workload, 0)
    try:
        run.prepare(list(range(cfg.T)))
        for i in range(args.warmup):
            run.time([i % cfg.T])
        times = [run.time([i % cfg.T]) for i in range(args.steps)]
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
        "config": {"workload": describe(cfg), "T": cfg.T, "D": cfg.D,
                   "E": cfg.E, "k": cfg.k, "I": cfg.I, "shared": cfg.shared},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1,
                         "kind": "oracle",
                         "sample": "one token of the batch per step (expert "
                                   "FFNs of its k experts; routing and "
                                   "permutation over the batch), fp64 numpy, "
                                   "1 BLAS thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from expert_layer_ptpc_gb300 import binding, build
    from expert_layer_ptpc_gb300 import synthetic as syn
    from expert_layer_ptpc_gb300.layer import MoELayer

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    layer = MoELayer.synthetic(cfg, dev, seed=0)
    x = syn.gen_x(cfg, dev, 0)
    logits = None if cfg.router == "weights" else syn.gen_logits(cfg, dev, 0)
    out = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device=dev)
    pre = {}
    if args.prenorm:   # layer input = RMSNorm(x + residual) * gamma
        if logits is None:
            raise SystemExit("--prenorm needs a workload with router logits")
        g = torch.Generator(device="cpu").manual_seed(12345)
        res = (torch.randn(cfg.T, cfg.D, generator=g) * 0.5).to(torch.bfloat16).to(dev)
        gamma = (1.0 + 0.1 * torch.randn(cfg.D, generator=g)).to(torch.bfloat16).to(dev)
        pre = {"residual": res, "gamma": gamma, "eps": 1e-6,
               "residual_out": torch.empty_like(res)}
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    tw = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nev = binding.MOE_FORWARD_EVENTS

    def make_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)]
               for _ in range(n)]
        for row in evs:          # create the driver events up front
            for e in row:
                e.record(stream)
        return evs

    def step(evs=None):
        layer.forward(x, logits, out=out, topk_ids=ids, topk_w=tw, events=evs, **pre)

    # warm-up (also validates the run)
    warm = make_events(1)[0]
    for _ in range(max(args.warmup, 1)):
        flush.fill_(1)
        step(warm)
    torch.cuda.synchronize()
    st, bits = binding.moe_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({bits:#x}) after warm-up")

    # The step a serving loop runs: one CUDA graph holding the whole forward
    # (kernels chained with programmatic dependent launch).
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    # timed region 1: whole steps
    sampler = ClockSampler(physical_gpu(local_rank))
    sampler.start()
    time.sleep(0.3)
    marks = [(torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        marks[i][0].record(stream)
        run_step()
        marks[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    st, bits = binding.moe_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({bits:#x}) in the timed region")
    step_ms = [a.elapsed_time(b) for a, b in marks]

    # timed region 2: the same forward with the library's step marks, to time
    # each kernel on its launching stream (the marks serialise the kernels)
    evs = make_events(args.steps)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(evs[i])
    torch.cuda.synchronize()
    st, bits = binding.moe_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({bits:#x}) in the profiled run")
    phase_ms = [[e[j].elapsed_time(e[j + 1]) for e in evs] for j in range(nev - 1)]
    profiled_ms = sum(e[0].elapsed_time(e[nev - 1]) for e in evs) / len(evs)
    mean_ms = sum(step_ms) / len(step_ms)
    max_ms = max_over_ranks(mean_ms, dev)

    # e2e: the same forward through the public API from pinned host buffers,
    # copies in and out inside the timed region
    x_h = x.cpu().pin_memory()
    lg_h = logits.cpu().pin_memory() if logits is not None else None
    out_h = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)
    lg_d = torch.empty_like(logits) if logits is not None else None
    if pre:   # the residual stream goes in and comes back too
        res_h = pre["residual"].cpu().pin_memory()
        res_out_h = torch.empty_like(res_h).pin_memory()
        res_d = torch.empty_like(pre["residual"])

    def e2e_step():
        x_d.copy_(x_h, non_blocking=True)
        if lg_d is not None:
            lg_d.copy_(lg_h, non_blocking=True)
        if pre:
            res_d.copy_(res_h, non_blocking=True)
            layer.forward(x_d, lg_d, out=out, residual=res_d, gamma=pre["gamma"],
                          eps=pre["eps"], residual_out=pre["residual_out"])
            res_out_h.copy_(pre["residual_out"], non_blocking=True)
        else:
            layer.forward(x_d, lg_d, out=out)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(args.warmup, 1)):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        e_ms.append((a, b))
    torch.cuda.synchronize()
    e2e_mean = sum(a.elapsed_time(b) for a, b in e_ms) / len(e_ms)
    e2e_max = max_over_ranks(e2e_mean, dev)
    h2d = x.numel() * 2 + (logits.numel() * 4 if logits is not None else 0)
    d2h = out.numel() * 2
    if pre:
        h2d += pre["residual"].numel() * 2
        d2h += pre["residual"].numel() * 2

    if rank != 0:
        return
    counts = torch.bincount(ids.view(-1).long(), minlength=cfg.E).cpu().numpy()
    B, touched = algorithmic_bytes(cfg, counts)
    if pre:   # the residual read and the new residual written, gamma
        B += 2 * cfg.T * cfg.D * 2 + 2 * cfg.D
    F = layer_flops(cfg)
    hbm, bf16, peak_src = peaks()
    gemm_ms = sum(phase_ms[4]) / len(phase_ms[4])
    gu_bytes = gateup_bytes(cfg, touched)
    names = ["router", "route", "permute",
             "addnorm_quant_x" if pre else "quant_x", "gateup_gemm", "requant",
             "down_gemm", "combine"]
    kernel_ms = {n: round(sum(p) / len(p), 5) for n, p in zip(names, phase_ms)}
    dominant = max(kernel_ms, key=kernel_ms.get)
    layer_gbs = B / (max_ms * 1e-3) / 1e9
    fp8_peak = 2.0 * bf16     # measured bf16 x the nominal fp8/bf16 ratio of 2
    # the gate/up GEMM: bound by whichever roof is lower for its bytes/flops
    gu_flops = 2.0 * cfg.rows * cfg.D * 2 * cfg.I
    tensor_bound = gu_flops / (fp8_peak * 1e12) > gu_bytes / (hbm * 1e9)
    if tensor_bound:
        ach = gu_flops / (gemm_ms * 1e-3) / 1e12
        gemm_roofline = {"bound": "tensor", "achieved": ach, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": ach / fp8_peak,
                         "peak_source": peak_src + ", fp8 = 2 x bf16 burst"}
    else:
        ach = gu_bytes / (gemm_ms * 1e-3) / 1e9
        gemm_roofline = {"bound": "hbm", "achieved": ach, "peak": hbm,
                         "unit": "GB/s", "frac": ach / hbm,
                         "peak_source": peak_src}
    # decode-sized token tiles (<= 16 rows per expert on average) run the
    # instantiation the traffic record was captured on
    decode_tiles = cfg.rows / max(1, cfg.groups) <= 16
    traffic = captured_traffic(gu_bytes, decode_tiles)
    gemm_roofline.update({
        "kernel": "gate/up grouped GEMM (tcgen05, SwiGLU epilogue)",
        "traffic": traffic,
        "traffic_source": ("ncu capture scaled by algorithmic bytes "
                           "(profiles/traffic_gateup_decode.json)"
                           if traffic is not None else None),
        "algorithmic_bytes_per_launch": gu_bytes,
        "flops_per_launch": gu_flops, "ms_per_launch": gemm_ms})
    t_roof = max(F / (fp8_peak * 1e12), B / (hbm * 1e9))
    B_impl = implementation_bytes(cfg, touched, bool(pre))
    layer_roofline = {
        "bound": "tensor" if F / (fp8_peak * 1e12) > B / (hbm * 1e9) else "hbm",
        "algorithmic_bytes": B, "flops": F, "achieved_gbs": layer_gbs,
        "achieved_fp8_tflops": F / (max_ms * 1e-3) / 1e12,
        "t_roof_ms": t_roof * 1e3, "frac": t_roof / (max_ms * 1e-3),
        # diagnosis: the bytes the launches move with the intermediates
        "implementation_bytes": B_impl,
        "implementation_gbs": B_impl / (max_ms * 1e-3) / 1e9}
    clocks = sampler.summary(t_wall0, t_wall1)
    prenorm = None
    if pre:
        # the fused add + RMSNorm + quant launch: x, residual and gamma in;
        # the new residual, the codes of every destination row (k + shared)
        # and their scales (and the gate) out. Unfused, the normalised bf16
        # activations would be written and read once more.
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
        "config": {"workload": describe(cfg), "T": cfg.T, "D": cfg.D,
                   "E": cfg.E, "k": cfg.k, "I": cfg.I, "shared": cfg.shared,
                   "touched_experts": touched,
                   "l2": "flushed before every step (256 MiB write)",
                   "cuda_graph": graph is not None,
                   "parallelism": f"replicas x{world}"},
        "roofline": gemm_roofline,
        "layer_roofline": layer_roofline,
        "kernel_ms": kernel_ms, "dominant_kernel": dominant,
        "profiled_ms_per_step": profiled_ms,
        "e2e": {"value": replica_tokens_per_s(cfg.T, world, e2e_max),
                "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_max},
        "gpu_launches": kernel_launches_per_step(cfg) * args.steps,
        "clocks": clocks,
    }
    if prenorm is not None:
        line["config"]["prenorm"] = {"eps": pre["eps"], "input": "RMSNorm(x + residual) * gamma"}
        line["prenorm"] = prenorm
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
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
                row["ptpc_production_ms"] = median_ms(lambda: binding.moe_grouped_gemm(
                    binding.MOE_GEMM_DOWN, prob["qa"], prob["sa"], prob["qw"], prob["sw"],
                    prob["offsets"], out=prob["out"]))
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
                  "ptpc_production = moe_grouped_gemm (the layer's kernel)",
        "gemms": result, "clocks": sampler.summary(t0, t1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
            run_reference(args, cfg)
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
