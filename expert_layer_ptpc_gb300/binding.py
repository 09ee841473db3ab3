"""Thin ctypes binding of libmoe_ptpc.so (declared in include/moe_ptpc.h).

Argument marshalling only: every function here checks torch tensors' device,
dtype and contiguity, allocates outputs with torch when the caller passes
none, and forwards raw device pointers plus the current CUDA stream to the C
entry point of the same name. All arithmetic runs in the library's kernels.
The library is loaded on first use; if it is missing this raises instead of
falling back to anything else.
"""

import ctypes
import os

import torch

from . import build as _build

MOE_DTYPE_BF16 = 0
MOE_DTYPE_F32 = 1
MOE_GEMM_GATEUP_SWIGLU = 0
MOE_GEMM_DOWN = 1


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("D", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("shared", ctypes.c_int32),
                ("renormalize", ctypes.c_int32)]


class moe_prenorm(ctypes.Structure):
    _fields_ = [("residual", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("residual_out", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_router_logits": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_route": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_permute_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_quant_ptpc": (_I, [_P, _I, _I64, _I, _P, _I, _I64, _P, _P, _P]),
    "moe_shared_gate": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_grouped_gemm": (_I, [_I, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _P, _I,
                              _I, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_scale_max": (_I, [_P, _I, _I, _P, _P]),
    "moe_grouped_gemm_down_f16": (_I, [_P, _P, _I64, _P, _P, _P, _P, _I, _I, _I,
                                       _P, _P, _I, _P]),
    "moe_combine_f16": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_forward_workspace_size": (_SZ, [ctypes.POINTER(moe_dims)]),
    "moe_forward": (_I, [ctypes.POINTER(moe_dims), _P, _P, _P, _P, _P, _P, _P,
                         _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_profiled": (_I, [ctypes.POINTER(moe_dims), _P, _P, _P, _P, _P,
                                  _P, _P, _P, _P, _P, _P, _P, _SZ,
                                  ctypes.POINTER(ctypes.c_void_p), _I, _P]),
    "moe_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "moe_workspace_status": (_I, [_P, _SZ, _P, ctypes.POINTER(ctypes.c_uint)]),
    "moe_forward_intermediates": (_I, [_P, _P, _SZ, _P]),
    "moe_forward_workspace_layout": (_I, [_P, _P, _P, _I]),
    "moe_forward_single_launch": (_I, [_P, _I, _I]),
    "moe_debug_expire_wait": (_I, [_I, _P, _SZ, _P]),
    "moe_router_topk": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_add_rmsnorm_quant": (_I, [_P, _P, _P, ctypes.c_float, _I64, _I, _P, _P, _I,
                                   _I64, _P, _P, _P, _P, _P]),
    "moe_forward_prenorm": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _SZ, _P, _I, _P]),
    "moe_quant_blocks": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "moe_quant_weight_blocks": (_I, [_P, _I64, _I, _P, _P, _P]),
    "moe_grouped_gemm_scaled": (_I, [_I, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _P, _P]),
}

MOE_SCALE_PTPC, MOE_SCALE_SUB512, MOE_SCALE_BLOCK128 = 0, 1, 2

MOE_FORWARD_EVENTS = 9

_lib = None


def load_library(path=None):
    """Load (once) and return the ctypes handle of the library: the checked
    variant (libmoe_ptpc_check.so) when MOE_LIBRARY_VARIANT=check."""
    global _lib
    if _lib is None:
        path = path or _build.library_path(os.environ.get("MOE_LIBRARY_VARIANT", ""))
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "expert_layer_ptpc_gb300.build.build() (needs nvcc)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_names():
    return sorted(_SIGNATURES)


def status_string(status):
    return load_library().moe_status_string(status).decode()


def _check(fn, status):
    if status != 0:
        raise MoeError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------------------
def moe_router_logits(x, w_r, logits=None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(w_r, torch.bfloat16, "w_r")
    T, D = x.shape
    E = w_r.shape[0]
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check("moe_router_logits", load_library().moe_router_logits(
        _ptr(x), _ptr(w_r), T, E, D, _ptr(logits), _stream(stream)))
    return logits


def moe_route(logits, k, renormalize=True, ids=None, weights=None, stream=None):
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check("moe_route", load_library().moe_route(
        _ptr(logits), T, E, k, int(bool(renormalize)), _ptr(ids), _ptr(weights),
        _stream(stream)))
    return ids, weights


def moe_permute(ids, E, stream=None):
    _need(ids, torch.int32, "topk_ids")
    T, k = ids.shape
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2f = torch.empty(T * k, dtype=torch.int32, device=dev)
    f2s = torch.empty(T * k, dtype=torch.int32, device=dev)
    lib = load_library()
    nws = lib.moe_permute_workspace_size(T, E, k)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
    _check("moe_permute", lib.moe_permute(
        _ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(s2f), _ptr(f2s),
        _ptr(ws), nws, _stream(stream)))
    return counts, offsets, s2f, f2s


def moe_permute_noalloc(ids, E, counts, offsets, s2f, f2s, stream=None):
    """moe_permute without a workspace: the library's fixed scratch array is
    used (see include/moe_ptpc.h for its limit and sharing rules). All output
    tensors are supplied by the caller; nothing is allocated."""
    _need(ids, torch.int32, "topk_ids")
    for t, n in ((counts, "expert_counts"), (offsets, "expert_offsets"),
                 (s2f, "sorted_to_flat"), (f2s, "flat_to_sorted")):
        _need(t, torch.int32, n)
    T, k = ids.shape
    _check("moe_permute_noalloc", load_library().moe_permute_noalloc(
        _ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(s2f), _ptr(f2s),
        _stream(stream)))
    return counts, offsets, s2f, f2s


def moe_quant_ptpc(inp, dst_rows=None, copies=1, extra_row_base=-1,
                   out_rows=None, out_q=None, out_scale=None, stream=None):
    """Per-row e4m3 quantisation of a [rows, cols] bf16 or fp32 tensor.
    Returns (codes uint8 [out_rows, cols], scales fp32 [out_rows])."""
    if inp.dtype == torch.bfloat16:
        dt = MOE_DTYPE_BF16
    elif inp.dtype == torch.float32:
        dt = MOE_DTYPE_F32
    else:
        raise ValueError("input must be bf16 or fp32")
    _need(inp, inp.dtype, "input")
    rows, cols = inp.shape
    if dst_rows is not None:
        _need(dst_rows, torch.int32, "dst_rows")
    if out_rows is None:
        out_rows = rows if dst_rows is None else rows * copies
        if extra_row_base >= 0:
            out_rows = max(out_rows, extra_row_base + rows)
    if out_q is None:
        out_q = torch.empty((out_rows, cols), dtype=torch.uint8, device=inp.device)
    if out_scale is None:
        out_scale = torch.empty(out_rows, dtype=torch.float32, device=inp.device)
    _check("moe_quant_ptpc", load_library().moe_quant_ptpc(
        _ptr(inp), dt, rows, cols, _ptr(dst_rows), copies, extra_row_base,
        _ptr(out_q), _ptr(out_scale), _stream(stream)))
    return out_q, out_scale


def moe_shared_gate(x, w_g, gate=None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(w_g, torch.bfloat16, "w_g")
    T, D = x.shape
    if gate is None:
        gate = torch.empty(T, dtype=torch.float32, device=x.device)
    _check("moe_shared_gate", load_library().moe_shared_gate(
        _ptr(x), _ptr(w_g), T, D, _ptr(gate), _stream(stream)))
    return gate


def moe_grouped_gemm(kind, A, a_scale, W, w_scale, group_offsets, out=None,
                     rows_hint=0, stream=None):
    """kind MOE_GEMM_GATEUP_SWIGLU: W [G, 2N, K] -> out [rows, N] fp32;
    kind MOE_GEMM_DOWN: W [G, N, K] -> out [rows, N] fp32."""
    _need(A, torch.uint8, "A")
    _need(a_scale, torch.float32, "a_scale")
    _need(W, torch.uint8, "W")
    _need(w_scale, torch.float32, "w_scale")
    _need(group_offsets, torch.int32, "group_offsets")
    a_rows, K = A.shape
    G = W.shape[0]
    N = W.shape[1] // 2 if kind == MOE_GEMM_GATEUP_SWIGLU else W.shape[1]
    if W.shape[2] != K or group_offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((a_rows, N), dtype=torch.float32, device=A.device)
    _check("moe_grouped_gemm", load_library().moe_grouped_gemm(
        kind, _ptr(A), _ptr(a_scale), a_rows, _ptr(W), _ptr(w_scale),
        _ptr(group_offsets), G, N, K, _ptr(out), MOE_DTYPE_F32, rows_hint,
        _stream(stream)))
    return out


def moe_combine(y, flat_to_sorted, topk_w, y_shared=None, shared_gate=None,
                out=None, stream=None):
    _need(y, torch.float32, "y")
    _need(flat_to_sorted, torch.int32, "flat_to_sorted")
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    D = y.shape[1]
    if out is None:
        out = torch.empty((T, D), dtype=torch.bfloat16, device=y.device)
    _check("moe_combine", load_library().moe_combine(
        _ptr(y), _ptr(flat_to_sorted), _ptr(topk_w), T, k, D, _ptr(y_shared),
        _ptr(shared_gate), _ptr(out), _stream(stream)))
    return out


def moe_scale_max(scale, bound=None, stream=None):
    """bound[g] = max_n scale[g, n] for a [G, N] fp32 tensor."""
    _need(scale, torch.float32, "scale")
    G, N = scale.shape
    if bound is None:
        bound = torch.empty(G, dtype=torch.float32, device=scale.device)
    _check("moe_scale_max", load_library().moe_scale_max(
        _ptr(scale), G, N, _ptr(bound), _stream(stream)))
    return bound


def moe_grouped_gemm_down_f16(A, a_scale, W, w_scale, w_bound, group_offsets,
                              y16=None, row_scale=None, rows_hint=0, stream=None):
    """Down projection W [G, N, K] with y = row_scale[:, None] * y16:
    returns (y16 [rows, N] fp16, row_scale [rows] fp32)."""
    _need(A, torch.uint8, "A")
    _need(a_scale, torch.float32, "a_scale")
    _need(W, torch.uint8, "W")
    _need(w_scale, torch.float32, "w_scale")
    _need(w_bound, torch.float32, "w_bound")
    _need(group_offsets, torch.int32, "group_offsets")
    a_rows, K = A.shape
    G, N = W.shape[0], W.shape[1]
    if W.shape[2] != K or group_offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    if y16 is None:
        y16 = torch.empty((a_rows, N), dtype=torch.float16, device=A.device)
    if row_scale is None:
        row_scale = torch.empty(a_rows, dtype=torch.float32, device=A.device)
    _check("moe_grouped_gemm_down_f16", load_library().moe_grouped_gemm_down_f16(
        _ptr(A), _ptr(a_scale), a_rows, _ptr(W), _ptr(w_scale), _ptr(w_bound),
        _ptr(group_offsets), G, N, K, _ptr(y16), _ptr(row_scale), rows_hint,
        _stream(stream)))
    return y16, row_scale


def moe_combine_f16(y16, row_scale, flat_to_sorted, topk_w, y16_shared=None,
                    row_scale_shared=None, shared_gate=None, out=None, stream=None):
    _need(y16, torch.float16, "y16")
    _need(row_scale, torch.float32, "row_scale")
    _need(flat_to_sorted, torch.int32, "flat_to_sorted")
    _need(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    D = y16.shape[1]
    if out is None:
        out = torch.empty((T, D), dtype=torch.bfloat16, device=y16.device)
    _check("moe_combine_f16", load_library().moe_combine_f16(
        _ptr(y16), _ptr(row_scale), _ptr(flat_to_sorted), _ptr(topk_w), T, k, D,
        _ptr(y16_shared), _ptr(row_scale_shared), _ptr(shared_gate), _ptr(out),
        _stream(stream)))
    return out


def make_dims(T, D, E, k, I, shared, renormalize=True):
    return moe_dims(T, D, E, k, I, int(bool(shared)), int(bool(renormalize)))


def moe_forward_workspace_size(dims):
    return load_library().moe_forward_workspace_size(ctypes.byref(dims))


def moe_forward_single_launch(dims, router_weights=False, prenorm=False):
    """Whether moe_forward with these dims runs as one cooperative launch."""
    r = load_library().moe_forward_single_launch(ctypes.byref(dims),
                                                 int(bool(router_weights)),
                                                 int(bool(prenorm)))
    if r < 0:
        raise MoeError("moe_forward_single_launch", r)
    return bool(r)


def moe_forward_workspace_layout(dims):
    """[(offset, size)] of the forward workspace's sub-buffers for dims; each
    is followed by a guard band of at least 256 bytes that no kernel writes."""
    lib = load_library()
    n = lib.moe_forward_workspace_layout(ctypes.byref(dims), None, None, 0)
    if n < 0:
        raise MoeError("moe_forward_workspace_layout", n)
    offs = (ctypes.c_size_t * n)()
    sizes = (ctypes.c_size_t * n)()
    lib.moe_forward_workspace_layout(ctypes.byref(dims), offs, sizes, n)
    return list(zip(offs, sizes))


class Intermediates(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "topk_ids", "topk_w", "expert_offsets", "sorted_to_flat", "flat_to_sorted",
        "xq", "sx", "gate", "h", "hq", "sh", "y", "y_row_scale")] + \
        [("y_fp16", ctypes.c_int32)]


def moe_forward_intermediates(dims, ws):
    """Views (torch tensors sharing the workspace's memory) of the
    intermediates the last forward on `ws` left there: offsets, s2f, f2s,
    xq [rows, D], sx [rows], gate [T], h [rows, I], hq [rows, I], sh [rows], and
    y ([rows, D] fp32, or fp16 codes with y_row_scale [rows])."""
    m = Intermediates()
    _check("moe_forward_intermediates", load_library().moe_forward_intermediates(
        ctypes.byref(dims), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(m)))
    base = ws.data_ptr()
    T, D, E, k, I = dims.T, dims.D, dims.E, dims.k, dims.I
    R = T * k
    rows = R + (T if dims.shared else 0)
    G = E + (1 if dims.shared else 0)

    def view(addr, n, dtype, shape):
        off = addr - base
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).view(shape)

    out = {
        "expert_offsets": view(m.expert_offsets, G + 1, torch.int32, (G + 1,)),
        "sorted_to_flat": view(m.sorted_to_flat, R, torch.int32, (R,)),
        "flat_to_sorted": view(m.flat_to_sorted, R, torch.int32, (R,)),
        "xq": view(m.xq, rows * D, torch.uint8, (rows, D)),
        "sx": view(m.sx, rows, torch.float32, (rows,)),
        "gate": view(m.gate, T, torch.float32, (T,)),
        "h": view(m.h, rows * I, torch.float32, (rows, I)),
        "hq": view(m.hq, rows * I, torch.uint8, (rows, I)),
        "sh": view(m.sh, rows, torch.float32, (rows,)),
        "y_fp16": bool(m.y_fp16),
    }
    if m.y_fp16:
        out["y"] = view(m.y, rows * D, torch.float16, (rows, D))
        out["y_row_scale"] = view(m.y_row_scale, rows, torch.float32, (rows,))
    else:
        out["y"] = view(m.y, rows * D, torch.float32, (rows, D))
    return out


def moe_forward(dims, x, w_gu, s_gu, w_d, s_d, router_logits=None,
                router_w=None, shared_gate_w=None, out=None, ws=None,
                topk_ids=None, topk_w=None, stream=None, events=None,
                residual=None, gamma=None, eps=1e-6, residual_out=None):
    """The whole layer; returns out [T, D] bf16. `events`: optional list of
    MOE_FORWARD_EVENTS torch.cuda.Event(enable_timing=True), recorded at the
    step boundaries (moe_forward_profiled). With `residual` and `gamma` the
    layer input is RMSNorm(x + residual) (moe_forward_prenorm): the new
    residual goes to `residual_out` (default: residual, updated in place)."""
    _need(x, torch.bfloat16, "x")
    for t, n in ((w_gu, "w_gu"), (w_d, "w_d")):
        _need(t, torch.uint8, n)
    for t, n in ((s_gu, "s_gu"), (s_d, "s_d")):
        _need(t, torch.float32, n)
    if router_logits is not None:
        _need(router_logits, torch.float32, "router_logits")
    if router_w is not None:
        _need(router_w, torch.bfloat16, "router_w")
    if shared_gate_w is not None:
        _need(shared_gate_w, torch.bfloat16, "shared_gate_w")
    lib = load_library()
    if out is None:
        out = torch.empty((dims.T, dims.D), dtype=torch.bfloat16, device=x.device)
    need = lib.moe_forward_workspace_size(ctypes.byref(dims))
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    if residual is not None:
        _need(residual, torch.bfloat16, "residual")
        _need(gamma, torch.bfloat16, "gamma")
        if residual_out is None:
            residual_out = residual
        _need(residual_out, torch.bfloat16, "residual_out")
        pre = moe_prenorm(residual.data_ptr(), gamma.data_ptr(), float(eps),
                          residual_out.data_ptr())
        handles = None
        if events is not None:
            if len(events) != MOE_FORWARD_EVENTS:
                raise ValueError(f"need {MOE_FORWARD_EVENTS} events")
            handles = (ctypes.c_void_p * MOE_FORWARD_EVENTS)(
                *[ctypes.c_void_p(e.cuda_event) for e in events])
        _check("moe_forward_prenorm", lib.moe_forward_prenorm(
            ctypes.byref(dims), ctypes.byref(pre), _ptr(x), _ptr(router_logits),
            _ptr(w_gu), _ptr(s_gu), _ptr(w_d), _ptr(s_d), _ptr(shared_gate_w),
            _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel(), handles,
            MOE_FORWARD_EVENTS if handles is not None else 0, _stream(stream)))
        return out
    args = (ctypes.byref(dims), _ptr(x), _ptr(router_logits), _ptr(router_w),
            _ptr(w_gu), _ptr(s_gu), _ptr(w_d), _ptr(s_d), _ptr(shared_gate_w),
            _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(ws), ws.numel())
    if events is None:
        _check("moe_forward", lib.moe_forward(*args, _stream(stream)))
    else:
        if len(events) != MOE_FORWARD_EVENTS:
            raise ValueError(f"need {MOE_FORWARD_EVENTS} events")
        handles = (ctypes.c_void_p * MOE_FORWARD_EVENTS)(
            *[ctypes.c_void_p(e.cuda_event) for e in events])
        _check("moe_forward_profiled", lib.moe_forward_profiled(
            *args, handles, MOE_FORWARD_EVENTS, _stream(stream)))
    return out


def moe_router_topk(x, w_r, k, renormalize=True, ids=None, weights=None,
                    logits=None, stream=None):
    """Router GEMM + top-k + softmax in one kernel; returns (ids, weights).
    `logits`: optional [T, E] fp32 tensor that receives the GEMM result."""
    _need(x, torch.bfloat16, "x")
    _need(w_r, torch.bfloat16, "w_r")
    T, D = x.shape
    E = w_r.shape[0]
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=x.device)
    _check("moe_router_topk", load_library().moe_router_topk(
        _ptr(x), _ptr(w_r), T, D, E, k, int(bool(renormalize)), _ptr(ids),
        _ptr(weights), _ptr(logits), _stream(stream)))
    return ids, weights


def moe_quant_blocks(x, block, q=None, scales=None, stream=None):
    """x [rows, K] bf16 -> (q [rows, K] e4m3, scales [rows, K / block] fp32),
    one scale per 1 x block piece along K (block 128 or 512)."""
    _need(x, torch.bfloat16, "x")
    rows, K = x.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, K // block), dtype=torch.float32, device=x.device)
    _check("moe_quant_blocks", load_library().moe_quant_blocks(
        _ptr(x), rows, K, block, _ptr(q), _ptr(scales), _stream(stream)))
    return q, scales


def moe_quant_weight_blocks(w, q=None, scales=None, stream=None):
    """w [..., K] fp32 (rows a multiple of 128) -> (q same shape e4m3,
    scales [rows / 128, K / 128] fp32), one scale per 128 x 128 block."""
    _need(w, torch.float32, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    if q is None:
        q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows // 128, K // 128), dtype=torch.float32, device=w.device)
    _check("moe_quant_weight_blocks", load_library().moe_quant_weight_blocks(
        _ptr(w), rows, K, _ptr(q), _ptr(scales), _stream(stream)))
    return q, scales


def moe_grouped_gemm_scaled(kind, A, a_scale, W, w_scale, group_offsets, out=None,
                            stream=None):
    """kind MOE_SCALE_PTPC / SUB512 / BLOCK128: W [G, N, K] -> out [rows, N]
    fp32 with the scale layouts of include/moe_ptpc.h."""
    _need(A, torch.uint8, "A")
    _need(a_scale, torch.float32, "a_scale")
    _need(W, torch.uint8, "W")
    _need(w_scale, torch.float32, "w_scale")
    _need(group_offsets, torch.int32, "group_offsets")
    a_rows, K = A.shape
    G, N = W.shape[0], W.shape[1]
    if W.shape[2] != K or group_offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((a_rows, N), dtype=torch.float32, device=A.device)
    _check("moe_grouped_gemm_scaled", load_library().moe_grouped_gemm_scaled(
        kind, _ptr(A), _ptr(a_scale), a_rows, _ptr(W), _ptr(w_scale), _ptr(group_offsets),
        G, N, K, _ptr(out), _stream(stream)))
    return out


def moe_add_rmsnorm_quant(x, residual, gamma, eps=1e-6, dst_rows=None, copies=1,
                          extra_row_base=-1, out_rows=None, residual_out=None,
                          out_q=None, out_scale=None, gate_w=None, gate_out=None,
                          stream=None):
    """residual_out = bf16(x + residual); codes / scales of RMSNorm(.) * gamma
    written like moe_quant_ptpc. Returns (residual_out, out_q, out_scale,
    gate_out)."""
    _need(x, torch.bfloat16, "x")
    _need(residual, torch.bfloat16, "residual")
    _need(gamma, torch.bfloat16, "gamma")
    rows, cols = x.shape
    if out_rows is None:
        out_rows = rows
    if residual_out is None:
        residual_out = torch.empty_like(x)
    if out_q is None:
        out_q = torch.empty((out_rows, cols), dtype=torch.uint8, device=x.device)
    if out_scale is None:
        out_scale = torch.empty(out_rows, dtype=torch.float32, device=x.device)
    if gate_w is not None and gate_out is None:
        gate_out = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("moe_add_rmsnorm_quant", load_library().moe_add_rmsnorm_quant(
        _ptr(x), _ptr(residual), _ptr(gamma), float(eps), rows, cols,
        _ptr(residual_out), _ptr(dst_rows), copies, extra_row_base, _ptr(out_q),
        _ptr(out_scale), _ptr(gate_w), _ptr(gate_out), _stream(stream)))
    return residual_out, out_q, out_scale, gate_out


def moe_debug_expire_wait(limit_us, ws=None, stream=None):
    """Launch a bounded wait that nothing completes (expires after limit_us);
    the next moe_workspace_status(ws) (moe_device_status() without a
    workspace) reports it. Raises MoeError on bad input."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_debug_expire_wait", load_library().moe_debug_expire_wait(
        int(limit_us), _ptr(ws), nbytes, _stream(stream)))


def moe_device_status(stream=None):
    """Errors of the standalone steps: read and clear the device error word
    on the stream, synchronise it, and return (status, error bits)."""
    detail = ctypes.c_uint(0)
    st = load_library().moe_device_status(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def moe_workspace_status(ws, stream=None):
    """Errors of the most recent forward on workspace `ws`: read and clear its
    error word on the stream, synchronise it, return (status, error bits)."""
    detail = ctypes.c_uint(0)
    st = load_library().moe_workspace_status(
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream), ctypes.byref(detail))
    return st, detail.value
