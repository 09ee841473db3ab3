"""End-to-end parity of moe_forward (through the C ABI) against the oracle.

Small layers are checked on every token. The five workloads run at their full
sizes, in the launch configuration the benchmark uses; there the routing and
the permutation are compared bit for bit on all tokens, and the outputs on a
sample of at least 256 tokens (every output row depends only on its own token
once the routing is fixed) aimed at the rows where the GEMM tiles change:
every expert's first and last row and the rows on either side of each tile
boundary inside its slice (`parity_tokens`). The GPU-quantised weights of
every expert the sample touches are compared byte for byte with the
oracle's.

Every comparison reads the forward's own intermediates
(moe_forward_intermediates) and goes stage by stage (staged_layer_check):
x codes and scales bit for bit; h within the fp32 GEMM and SwiGLU bound of
the oracle's exact h; the requantisation codes and scales bit for bit with
the oracle taking that integer decision on the GPU's own fp32 h; y within
the fp32 accumulation (and fp16 encoding) bound of the oracle's down GEMM on
those codes; the output under the accuracy contract against the oracle's
combine of that y: max|gpu - oracle| <= 2e-2 * rms(oracle) beyond the half
bf16 ulp that the output's own rounding may cost each element, and
sum|gpu - oracle| / sum|oracle| <= 5e-3 (gpu_helpers.layer_tolerance_ok).
End to end against the plain oracle, whose requantisation decides on its
own fp32 rounding of the exact h, the L1 bound applies too."""

import numpy as np
import pytest
import torch

import oracle
from expert_layer_ptpc_gb300 import synthetic as syn
from tests.gpu_helpers import (U32, ensure_library, gemm_bound,
                               layer_tolerance_ok, parity_tokens,
                               quantize_experts, require_gpu, staged_layer_check)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_gpu()
    ensure_library()


class _Run:
    """A layer on the GPU plus the oracle's view of the same inputs."""

    def __init__(self, cfg, seed=0):
        from expert_layer_ptpc_gb300.layer import MoELayer
        self.cfg = cfg
        self.seed = seed
        self.layer = MoELayer.synthetic(cfg, "cuda", seed)
        self.qcache = {}

    def inputs(self, cfg):
        x = syn.gen_x(cfg, "cuda", self.seed)
        logits = (None if cfg.router == "weights"
                  else syn.gen_logits(cfg, "cuda", self.seed))
        return x, logits

    def expert_weights(self, es, batch=32):
        """The oracle's quantisation of experts `es` (from the same seeded raw
        weights, drawn on the GPU and copied back), each compared byte for
        byte with the GPU's own quantisation. Experts go through the process
        pool in batches, so host memory holds at most `batch` raw experts."""
        missing = [e for e in es if e not in self.qcache]
        L = self.layer
        for i in range(0, len(missing), batch):
            part = missing[i:i + batch]
            raw = []
            for e in part:
                gu, d = syn.gen_expert_weights(self.cfg, e, "cuda", self.seed)
                raw.append((gu.cpu().numpy(), d.cpu().numpy()))
            for e, q in zip(part, quantize_experts(raw)):
                self.qcache[e] = q
                assert np.array_equal(L.w_gu[e].cpu().numpy(), q[0]), e
                assert np.array_equal(L.s_gu[e].cpu().numpy().view(np.uint32),
                                      q[1].view(np.uint32)), e
                assert np.array_equal(L.w_d[e].cpu().numpy(), q[2]), e
                assert np.array_equal(L.s_d[e].cpu().numpy().view(np.uint32),
                                      q[3].view(np.uint32)), e
        return {e: self.qcache[e] for e in es}

    def check(self, cfg, sample=False):
        from expert_layer_ptpc_gb300 import binding
        T, k, E = cfg.T, cfg.k, cfg.E
        x, logits = self.inputs(cfg)
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        out = self.layer.forward(x, logits, topk_ids=ids, topk_w=tw)
        st, bits = self.layer.status()
        assert st == 0, f"device status {st} bits {bits:#x}"

        xn = x.float().cpu().numpy()
        w_rtol = 64 * U32
        amb = np.zeros(T, bool)
        if logits is None:
            wr = self.layer.router_w.float().cpu().numpy()
            ln = oracle.router_logits_ref(xn, wr)
            if T * E * cfg.D >= (1 << 20):
                # the layer routes on tensor-core fp32 logits, within the
                # fp32 accumulation bound of these exact ones. A token whose
                # top k (or its order) has a gap within twice that bound has
                # more than one correct selection: its ids must then be a
                # valid choice, and its output is not compared.
                bound = gemm_bound(np.abs(xn.astype(np.float64)) @
                                   np.abs(wr.astype(np.float64)).T, cfg.D)
                bt = 2 * bound.max(axis=1)
                srt = -np.sort(-ln.astype(np.float64), axis=1)[:, :min(k + 1, E)]
                amb = ((srt[:, :-1] - srt[:, 1:]) <= bt[:, None]).any(axis=1)
                # the bound is the worst case (every partial sum rounding the
                # same way), so a few percent of the seeded tokens fall in it
                assert amb.mean() < 0.15, f"{amb.sum()} of {T} tokens near a tie"
                w_rtol += 4 * float(bound.max())
                exact = xn.astype(np.float64) @ wr.astype(np.float64).T
                gid = ids.cpu().numpy()
                for t in np.flatnonzero(amb):
                    ch = np.zeros(E, bool)
                    ch[gid[t]] = True
                    if not ch.all():
                        assert exact[t, ch].min() >= exact[t, ~ch].max() - bt[t]
        else:
            ln = logits.cpu().numpy()
        rid, rw = oracle.route_ref(ln, k, cfg.renormalize)
        ok_t = ~amb
        assert np.array_equal(ids.cpu().numpy()[ok_t], rid[ok_t])
        np.testing.assert_allclose(tw.cpu().numpy()[ok_t], rw[ok_t], rtol=w_rtol, atol=0)
        if not amb.any():
            # permutation of the same ids, full size, bit-exact
            counts, offs, s2f, f2s = binding.moe_permute(ids, E)
            rc, ro, rs, rf = oracle.permute_ref(rid, E)
            assert np.array_equal(counts.cpu().numpy(), rc)
            assert np.array_equal(offs.cpu().numpy(), ro)
            assert np.array_equal(s2f.cpu().numpy(), rs)
            assert np.array_equal(f2s.cpu().numpy(), rf)

        if sample:
            # the GPU's own ids give the row layout its GEMM tiles saw
            tokens = parity_tokens(ids.cpu().numpy(), E, cfg.shared, seed=T + 17)
        else:
            tokens = np.arange(T)
        tokens = tokens[ok_t[tokens]]     # unique routing only
        return self.compare_outputs(cfg, xn, ln, out, rid, rw, tokens)

    def compare_outputs(self, cfg, xv, ln, out, rid, rw, tokens):
        """The forward's outputs on `tokens` (layer input xv, routing rid/rw
        equal to the GPU's there): stage by stage against the oracle taking
        the requantisation decisions on the GPU's fp32 h, where the accuracy
        contract applies, and end to end against the plain oracle, where the
        L1 bound applies (its max error is reported: a code of h that the
        GPU's fp32 h rounds the other way moves a few tail elements by up to
        about 0.04 rms)."""
        from expert_layer_ptpc_gb300 import binding
        T, k, E = cfg.T, cfg.k, cfg.E
        touched = sorted(set(int(e) for e in rid[tokens].ravel()))
        if cfg.shared:
            touched.append(E)
        qmap = self.expert_weights(touched)
        wg = (self.layer.shared_gate_w.float().cpu().numpy()
              if cfg.shared else None)
        got = out.float().cpu().numpy()[tokens]
        inter = binding.moe_forward_intermediates(self.layer.dims(T), self.layer._ws)
        staged = staged_layer_check(cfg, xv, got, rid, rw, inter, tokens, qmap, wg)
        r = oracle.moe_forward_ref(
            xv, k, lambda e: qmap[e], E, logits=ln, w_g=wg,
            renormalize=cfg.renormalize, tokens=tokens)
        _, max_rel, l1, raw = layer_tolerance_ok(got, r["out64"])
        assert l1 <= 5e-3, f"{cfg.name}: L1 ratio {l1:.3e} against the oracle"
        return {"staged": staged, "oracle_max_excess": max_rel, "oracle_l1": l1,
                "oracle_raw_max": raw}


# ---------------------------------------------------------------------------
# small layers, every token
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [
    syn.LayerConfig("s1", 300, 512, 16, 4, 256, True, "normal"),
    syn.LayerConfig("s2", 97, 256, 8, 8, 128, False, "normal"),
    syn.LayerConfig("s3", 50, 384, 32, 3, 384, False, "normal", False),
    syn.LayerConfig("s4", 1, 256, 64, 6, 128, True, "normal"),
    syn.LayerConfig("s5", 129, 256, 1, 1, 256, False, "normal"),
    syn.LayerConfig("s6", 40, 256, 12, 2, 128, True, "weights"),
    # rows x D x 4 bytes >= 32 MiB: the expert output takes the fp16 encoding
    syn.LayerConfig("s7", 1024, 1024, 16, 8, 256, True, "normal"),
    # T x E x D >= 2^20 with router weights: the fused tensor-core router
    syn.LayerConfig("s8", 256, 1024, 16, 4, 256, True, "weights"),
], ids=lambda c: c.name)
def test_small_layer_all_tokens(cfg):
    _Run(cfg).check(cfg)


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------
def test_tiny_layer():
    cfg = syn.CONFIGS["tiny"]
    _Run(cfg).check(cfg)


def test_decode_layer():
    cfg = syn.CONFIGS["decode"]
    _Run(cfg).check(cfg)


def test_prefill_layer():
    cfg = syn.CONFIGS["prefill"]
    _Run(cfg).check(cfg, sample=True)


def test_skewed_layer():
    cfg = syn.CONFIGS["skewed"]
    _Run(cfg).check(cfg, sample=True)


@pytest.fixture(scope="module")
def sweep_run():
    return _Run(syn.CONFIGS["sweep"])


@pytest.mark.parametrize("T", syn.SWEEP_T)
def test_sweep_layer(sweep_run, T):
    cfg = syn.sweep_config(T)
    sweep_run.check(cfg, sample=T > 256)


@pytest.mark.parametrize("cfg", [
    syn.LayerConfig("p1", 300, 512, 16, 4, 256, True, "normal"),
    syn.LayerConfig("p2", 1024, 1024, 16, 8, 256, False, "normal"),   # fp16 y
], ids=lambda c: c.name)
def test_prenorm_layer_all_tokens(cfg):
    """moe_forward_prenorm: the layer on RMSNorm(x + residual) * gamma. The new
    residual is compared bit for bit with the oracle's; the output against the
    oracle layer evaluated on the oracle's normalised activations v."""
    from expert_layer_ptpc_gb300 import binding
    run = _Run(cfg)
    x, logits = run.inputs(cfg)
    g = torch.Generator().manual_seed(99)
    res = (torch.randn(cfg.T, cfg.D, generator=g) * 0.5).to(torch.bfloat16)
    gamma = (1.0 + 0.2 * torch.randn(cfg.D, generator=g)).to(torch.bfloat16)
    res_d = res.cuda()
    res_out = torch.empty_like(res_d)
    out = run.layer.forward(x, logits, residual=res_d, gamma=gamma.cuda(),
                            eps=1e-6, residual_out=res_out)
    st, bits = run.layer.status()
    assert st == 0, bits
    ref = oracle.add_rmsnorm_ref(x.float().cpu().numpy(), res.float().numpy(),
                                 gamma.float().numpy(), 1e-6)
    assert np.array_equal(res_out.float().cpu().numpy(), ref[0])
    assert torch.equal(res_d.cpu(), res)             # residual itself untouched
    ln = logits.cpu().numpy()
    rid, rw = oracle.route_ref(ln, cfg.k, cfg.renormalize)
    run.compare_outputs(cfg, ref[1], ln, out, rid, rw, np.arange(cfg.T))


def test_prenorm_prefill_sampled():
    """moe_forward_prenorm on the prefill workload at full size, in the
    launch configuration and with the inputs `bench.py --prenorm` times
    (residual N(0, 0.5^2) and gamma 1 + N(0, 0.1^2), bf16, seed 12345): the
    new residual of every token bit for bit, the output of the tile-boundary
    sample of tokens against the oracle layer on the oracle's normalised
    activations."""
    from expert_layer_ptpc_gb300 import binding
    cfg = syn.CONFIGS["prefill"]
    run = _Run(cfg)
    x, logits = run.inputs(cfg)
    g = torch.Generator(device="cpu").manual_seed(12345)
    res = (torch.randn(cfg.T, cfg.D, generator=g) * 0.5).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn(cfg.D, generator=g)).to(torch.bfloat16)
    res_out = torch.empty((cfg.T, cfg.D), dtype=torch.bfloat16, device="cuda")
    out = run.layer.forward(x, logits, residual=res.cuda(), gamma=gamma.cuda(),
                            eps=1e-6, residual_out=res_out)
    st, bits = run.layer.status()
    assert st == 0, bits
    ref = oracle.add_rmsnorm_ref(x.float().cpu().numpy(), res.float().numpy(),
                                 gamma.float().numpy(), 1e-6)
    assert np.array_equal(res_out.float().cpu().numpy(), ref[0])
    ln = logits.cpu().numpy()
    rid, rw = oracle.route_ref(ln, cfg.k, cfg.renormalize)
    tokens = parity_tokens(rid, cfg.E, cfg.shared, seed=cfg.T + 3)
    run.compare_outputs(cfg, ref[1], ln, out, rid, rw, tokens)


def test_forward_on_two_streams_at_once():
    """Two forwards in flight at once on two streams, each with its own
    workspace (the ABI's contract: every call is asynchronous on the caller's
    stream and allocates nothing). Each output equals, bit for bit, the same
    forward run alone."""
    import ctypes
    from expert_layer_ptpc_gb300 import binding
    cfg = syn.LayerConfig("conc", 2048, 1024, 32, 4, 512, True, "normal")
    run = _Run(cfg)
    L = run.layer
    x1, lg1 = run.inputs(cfg)
    x2, lg2 = syn.gen_x(cfg, "cuda", 1), syn.gen_logits(cfg, "cuda", 1)
    ref1 = L.forward(x1, lg1).clone()
    ref2 = L.forward(x2, lg2).clone()
    torch.cuda.synchronize()
    dims = L.dims(cfg.T)
    need = max(binding.load_library().moe_forward_workspace_size(ctypes.byref(dims)), 1)
    ws = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [torch.empty_like(ref1) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for i, (x, lg) in enumerate(((x1, lg1), (x2, lg2))):
            binding.moe_forward(dims, x, L.w_gu, L.s_gu, L.w_d, L.s_d, router_logits=lg,
                                shared_gate_w=L.shared_gate_w, out=outs[i], ws=ws[i],
                                stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        st, bits = binding.moe_workspace_status(ws[i], streams[i])
        assert st == 0, bits
    assert torch.equal(outs[0].view(torch.int16), ref1.view(torch.int16))
    assert torch.equal(outs[1].view(torch.int16), ref2.view(torch.int16))


def test_forward_is_deterministic():
    cfg = syn.LayerConfig("det", 2000, 512, 32, 4, 256, True, "normal")
    run = _Run(cfg)
    x, logits = run.inputs(cfg)
    a = run.layer.forward(x, logits).clone()
    b = run.layer.forward(x, logits).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# a few tokens: the single-launch forward
# ---------------------------------------------------------------------------
SINGLE_LAUNCH = [
    syn.LayerConfig("f1", 2, 512, 64, 8, 256, True, "normal"),
    syn.LayerConfig("f2", 3, 256, 4, 3, 128, False, "normal"),     # experts shared by tokens
    syn.LayerConfig("f3", 4, 1024, 128, 6, 512, True, "normal", False),
    syn.LayerConfig("f4", 1, 4096, 512, 10, 1024, True, "normal"),  # the T=1 sweep shape
    syn.LayerConfig("f5", 3, 2048, 1024, 32, 128, False, "normal"),   # k = 32, E = 1024
    syn.LayerConfig("f6", 1, 128, 8, 1, 128, True, "normal"),      # one row per group
]


@pytest.mark.parametrize("cfg", SINGLE_LAUNCH, ids=lambda c: c.name)
def test_single_launch_layer(cfg):
    """Batches of at most four tokens on given logits: every token, stage by
    stage against the oracle from the intermediates the forward leaves in
    the workspace; chained kernels by default, one cooperative launch with
    MOE_SMALL_FORWARD=1 (the next test)."""
    import os
    from expert_layer_ptpc_gb300 import binding
    run = _Run(cfg)
    expect = os.environ.get("MOE_SMALL_FORWARD", "0") == "1"
    assert binding.moe_forward_single_launch(run.layer.dims(cfg.T)) == expect
    run.check(cfg)


def test_single_launch_variant():
    """The same small layers, the T=1 sweep point and a guard-band case with
    the single-launch forward turned on (MOE_SMALL_FORWARD=1), in a child
    process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MOE_SMALL_FORWARD="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
           os.path.join(root, "tests", "test_gpu_layer.py"), "-k",
           "test_single_launch_layer or test_sweep_layer[1] or g6"]
    r = subprocess.run(cmd, env=env, cwd=root, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_empty_batch_is_noop():
    cfg = syn.LayerConfig("empty", 0, 256, 8, 2, 128, False, "normal")
    run = _Run(syn.LayerConfig("empty", 4, 256, 8, 2, 128, False, "normal"))
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    out = run.layer.forward(x, lg)
    assert out.shape == (0, 256)
    assert cfg.T == 0


@pytest.mark.parametrize("cfg", [
    syn.LayerConfig("g1", 300, 512, 16, 4, 256, True, "normal"),
    syn.LayerConfig("g2", 1024, 1024, 16, 8, 256, True, "normal"),    # fp16 y, CTA pairs
    syn.LayerConfig("g3", 40, 256, 12, 2, 128, True, "weights"),      # exact router GEMM
    syn.LayerConfig("g4", 256, 1024, 16, 4, 256, False, "weights"),   # fused router
    syn.LayerConfig("g5", 9000, 256, 8, 2, 128, False, "normal"),     # multi-block permute
    syn.LayerConfig("g6", 3, 1024, 64, 8, 512, True, "normal"),       # single launch
], ids=lambda c: c.name)
def test_forward_leaves_guard_bands_intact(cfg):
    """Canaries in place of a memory checker: the forward workspace is filled
    with a pattern, the forward runs, and the guard band behind every
    sub-buffer (moe_forward_workspace_layout) still holds the pattern, so no
    kernel wrote past the end of a buffer it owns. The output tensor's
    neighbours are checked the same way."""
    from expert_layer_ptpc_gb300 import binding
    run = _Run(cfg)
    x, logits = run.inputs(cfg)
    L = run.layer
    dims = L.dims(cfg.T)
    ws = L.workspace(cfg.T)
    ws.fill_(0xA5)
    pad = 4096
    big = torch.full((cfg.T * cfg.D + 2 * pad,), 0x5A5A, dtype=torch.int16, device="cuda")
    out = big[pad:pad + cfg.T * cfg.D].view(torch.bfloat16).view(cfg.T, cfg.D)
    L.forward(x, logits, out=out)
    assert L.status() == (0, 0)
    host = ws.cpu().numpy()
    for off, n in binding.moe_forward_workspace_layout(dims):
        band = host[off + n:off + n + 256]
        assert np.all(band == 0xA5), (cfg.name, off, n, np.flatnonzero(band != 0xA5)[:4])
    b = big.cpu().numpy()
    assert np.all(b[:pad] == 0x5A5A) and np.all(b[pad + cfg.T * cfg.D:] == 0x5A5A)
