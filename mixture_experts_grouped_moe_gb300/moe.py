"""Thin ctypes binding of libmoe_gb300 (include/moe.h), same names as the C ABI.

Only argument marshalling lives here: tensors become raw pointers, the
current torch CUDA stream becomes the `stream` argument, and a negative
status raises MoEError.  Every step of the layer runs in the CUDA library;
there is no Python or CPU fallback.  If the library is missing the first
call raises (build it with `mixture_experts_grouped_moe_gb300.build`).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5

MOE_BF16 = 0
MOE_FP8_BLOCK128 = 1
MOE_FP8_TOKEN = 2
MOE_MXFP4 = 3
MOE_MODE_GROUPED = 0
MOE_MODE_SWAP = 1

EXPORTED = [
    "moe_status_string", "moe_version", "moe_align_sort_sizes", "moe_block_size_m_heuristic",
    "moe_ksplit_heuristic", "moe_plan", "moe_fused_workspace_size", "moe_workspace_layout",
    "moe_workspace_status", "moe_route_topk", "moe_align_sort_workspace_size", "moe_align_sort",
    "moe_quantize_fp8_act", "moe_quantize_fp8_weights", "moe_quantize_fp8_rows", "moe_fused_forward",
    "moe_host_staging_bytes", "moe_fused_forward_host", "moe_align_sort_noalloc", "moe_quantize_mxfp4",
    "moe_train_workspace_size", "moe_fused_forward_train", "moe_fused_backward", "moe_options_init",
    "moe_fused_forward_ex",
]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class moe_plan_t(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("block_m", ctypes.c_int), ("split_k1", ctypes.c_int),
                ("split_k2", ctypes.c_int), ("max_padded", ctypes.c_int64), ("max_blocks", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t)]


class moe_options_t(ctypes.Structure):
    _fields_ = [("gemm_pair", ctypes.c_int), ("one_stage", ctypes.c_int), ("pdl_mask", ctypes.c_int),
                ("stage_events", ctypes.c_void_p), ("h_wait_limit_us", ctypes.c_uint),
                ("unsatisfiable_h_wait", ctypes.c_int), ("light_tiles", ctypes.c_int), ("tc_router", ctypes.c_int)]


class moe_ws_layout_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "status", "topk_ids", "topk_weights", "sorted_ids", "sorted_weights", "sorted_expert_ids",
        "num_tokens_post_padded", "expert_counts", "x_sorted", "x_scales", "inter", "inter_scales", "inter_h",
        "y", "router_logits", "total")]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {_build.LIB} is missing "
                                   "(run mixture_experts_grouped_moe_gb300.build.build())")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "moe_status_string": (ctypes.c_char_p, [I]),
            "moe_version": (I, []),
            "moe_align_sort_sizes": (I, [I, I, I, I, P, P]),
            "moe_block_size_m_heuristic": (I, [I, I, I, I, I, P, I]),
            "moe_ksplit_heuristic": (I, [I, I, I, I, I, I, I]),
            "moe_plan": (I, [I, I, I, I, I, I, I, I, I, P]),
            "moe_fused_workspace_size": (SZ, [I, I, I, I, I, I, I, I]),
            "moe_workspace_layout": (I, [I, I, I, I, I, I, I, I, P]),
            "moe_workspace_status": (I, [P, P, P]),
            "moe_route_topk": (I, [P, P, P, I, I, I, I, I, P, P, P, P]),
            "moe_align_sort_workspace_size": (SZ, [I, I, I]),
            "moe_align_sort": (I, [P, P, I, I, I, I, P, P, P, P, P, P, SZ, P]),
            "moe_quantize_fp8_act": (I, [P, I64, I, P, P, P]),
            "moe_quantize_fp8_weights": (I, [P, I64, I, P, P, P]),
            "moe_quantize_fp8_rows": (I, [P, I64, I, P, P, P]),
            "moe_fused_forward": (I, [I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, SZ, P]),
            "moe_host_staging_bytes": (SZ, [I, I]),
            "moe_fused_forward_host": (I, [I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, SZ, P]),
            "moe_options_init": (I, [P]),
            "moe_fused_forward_ex": (I, [I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, SZ, P, P]),
            "moe_train_workspace_size": (SZ, [I, I, I, I, I]),
            "moe_fused_forward_train": (I, [P, P, P, P, P, I, I, I, I, I, P, P, SZ, P, P]),
            "moe_fused_backward": (I, [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, SZ, P, P]),
            "moe_quantize_mxfp4": (I, [P, I64, I, P, P, I, P]),
            "moe_align_sort_noalloc": (I, [P, P, I, I, I, I, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _p(t):
    """Raw pointer of a tensor / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoEError(fn, rc)
    return rc


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_version() -> int:
    return load().moe_version()


def moe_align_sort_sizes(T, k, E, block_m):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check("moe_align_sort_sizes", load().moe_align_sort_sizes(T, k, E, block_m, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def moe_block_size_m_heuristic(token, topk, expert, inter_dim, units, candidates=(32, 64, 128)):
    arr = (ctypes.c_int * len(candidates))(*candidates)
    r = load().moe_block_size_m_heuristic(token, topk, expert, inter_dim, units, arr, len(candidates))
    if r < 0:
        raise MoEError("moe_block_size_m_heuristic", r)
    return r


def moe_ksplit_heuristic(token, topk, expert, inter_dim, model_dim, units, block_m):
    r = load().moe_ksplit_heuristic(token, topk, expert, inter_dim, model_dim, units, block_m)
    if r < 0:
        raise MoEError("moe_ksplit_heuristic", r)
    return r


def moe_plan(dtype, T, H, I, E, k, block_m=0, split_k=0, num_sms=0) -> moe_plan_t:
    p = moe_plan_t()
    _check("moe_plan", load().moe_plan(dtype, T, H, I, E, k, block_m, split_k, num_sms, ctypes.byref(p)))
    return p


def moe_fused_workspace_size(dtype, T, H, I, E, k, block_m=0, split_k=0) -> int:
    return load().moe_fused_workspace_size(dtype, T, H, I, E, k, block_m, split_k)


def moe_workspace_layout(dtype, T, H, I, E, k, block_m=0, split_k=0) -> moe_ws_layout_t:
    lay = moe_ws_layout_t()
    _check("moe_workspace_layout",
           load().moe_workspace_layout(dtype, T, H, I, E, k, block_m, split_k, ctypes.byref(lay)))
    return lay


def moe_workspace_status(ws, stream=None) -> int:
    v = ctypes.c_int()
    _check("moe_workspace_status", load().moe_workspace_status(_p(ws), ctypes.byref(v), _stream(stream)))
    return v.value


def moe_route_topk(x, W_router, bias, T, H, E, k, topk_ids, topk_weights, logits=None, stream=None,
                   renormalize=True):
    return _check("moe_route_topk", load().moe_route_topk(
        _p(x), _p(W_router), _p(bias), T, H, E, k, 1 if renormalize else 0, _p(topk_ids), _p(topk_weights),
        _p(logits), _stream(stream)))


def moe_align_sort_workspace_size(T, k, E) -> int:
    return load().moe_align_sort_workspace_size(T, k, E)


def moe_align_sort(topk_ids, topk_weights, T, k, E, block_m, sorted_ids, sorted_weights, sorted_expert_ids,
                   num_tokens_post_padded, expert_counts, ws, ws_bytes, stream=None):
    return _check("moe_align_sort", load().moe_align_sort(
        _p(topk_ids), _p(topk_weights), T, k, E, block_m, _p(sorted_ids), _p(sorted_weights),
        _p(sorted_expert_ids), _p(num_tokens_post_padded), _p(expert_counts), _p(ws), ws_bytes,
        _stream(stream)))


def moe_align_sort_noalloc(topk_ids, topk_weights, T, k, E, block_m, sorted_ids, sorted_weights,
                           sorted_expert_ids, num_tokens_post_padded, expert_counts, stream=None):
    """moe_align_sort with the library's fixed device scratch instead of a caller workspace."""
    return _check("moe_align_sort_noalloc", load().moe_align_sort_noalloc(
        _p(topk_ids), _p(topk_weights), T, k, E, block_m, _p(sorted_ids), _p(sorted_weights),
        _p(sorted_expert_ids), _p(num_tokens_post_padded), _p(expert_counts), _stream(stream)))


def moe_quantize_fp8_act(X, R, C, q, s, stream=None):
    return _check("moe_quantize_fp8_act", load().moe_quantize_fp8_act(_p(X), R, C, _p(q), _p(s), _stream(stream)))


def moe_quantize_fp8_weights(W, R, C, q, s, stream=None):
    return _check("moe_quantize_fp8_weights",
                  load().moe_quantize_fp8_weights(_p(W), R, C, _p(q), _p(s), _stream(stream)))


def moe_quantize_fp8_rows(X, R, C, q, s, stream=None):
    return _check("moe_quantize_fp8_rows", load().moe_quantize_fp8_rows(_p(X), R, C, _p(q), _p(s), _stream(stream)))


def moe_quantize_mxfp4(X, R, C, q, s, tiled=False, stream=None):
    return _check("moe_quantize_mxfp4",
                  load().moe_quantize_mxfp4(_p(X), R, C, _p(q), _p(s), 1 if tiled else 0, _stream(stream)))


def moe_fused_forward(dtype, x, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I, E, k,
                      block_m, split_k, out, ws, ws_bytes, stream=None):
    return _check("moe_fused_forward", load().moe_fused_forward(
        dtype, _p(x), _p(W_router), _p(router_bias), _p(W_gate_up), _p(w1_scale), _p(W_down), _p(w2_scale),
        T, H, I, E, k, block_m, split_k, _p(out), _p(ws), ws_bytes, _stream(stream)))


def moe_host_staging_bytes(T, H) -> int:
    return load().moe_host_staging_bytes(T, H)


def moe_fused_forward_host(dtype, x_host, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I,
                           E, k, block_m, split_k, out_host, ws, ws_bytes, stream=None):
    return _check("moe_fused_forward_host", load().moe_fused_forward_host(
        dtype, _p(x_host), _p(W_router), _p(router_bias), _p(W_gate_up), _p(w1_scale), _p(W_down), _p(w2_scale),
        T, H, I, E, k, block_m, split_k, _p(out_host), _p(ws), ws_bytes, _stream(stream)))


class Options:
    """Per-call choices of moe_fused_forward_ex (see moe_options_t in include/moe.h).

    Keyword arguments override the library's defaults: gemm_pair (-1/0/1), one_stage (0/1),
    pdl_mask (-1 or a mask), stage_events (7 torch.cuda.Event or None), h_wait_limit_us,
    unsatisfiable_h_wait (0/1, for the timeout test only), light_tiles (-1/0/1), tc_router (-1/0/1)."""

    def __init__(self, **kw):
        self.c = moe_options_t()
        _check("moe_options_init", load().moe_options_init(ctypes.byref(self.c)))
        self._events = None
        for key, val in kw.items():
            setattr(self, key, val)

    def __setattr__(self, key, val):
        if key in ("c", "_events"):
            object.__setattr__(self, key, val)
        elif key == "stage_events":
            if val is None:
                self._events = None
                self.c.stage_events = None
            else:
                arr = (ctypes.c_void_p * len(val))(*[e.cuda_event for e in val])
                self._events = (arr, list(val))  # keep both alive while the options are in use
                self.c.stage_events = ctypes.cast(arr, ctypes.c_void_p)
        elif key in dict(moe_options_t._fields_):
            setattr(self.c, key, val)
        else:
            raise AttributeError(key)

    def __getattr__(self, key):
        if key in dict(moe_options_t._fields_):
            return getattr(self.c, key)
        raise AttributeError(key)


def _opt(options):
    if options is None:
        return None
    return ctypes.byref(options.c if isinstance(options, Options) else options)


def moe_fused_forward_ex(dtype, x, W_router, router_bias, W_gate_up, w1_scale, W_down, w2_scale, T, H, I, E, k,
                         block_m, split_k, out, ws, ws_bytes, options=None, stream=None):
    return _check("moe_fused_forward_ex", load().moe_fused_forward_ex(
        dtype, _p(x), _p(W_router), _p(router_bias), _p(W_gate_up), _p(w1_scale), _p(W_down), _p(w2_scale),
        T, H, I, E, k, block_m, split_k, _p(out), _p(ws), ws_bytes, _opt(options), _stream(stream)))


def moe_train_workspace_size(T, H, I, E, k) -> int:
    return load().moe_train_workspace_size(T, H, I, E, k)


def moe_fused_forward_train(x, W_router, router_bias, W_gate_up, W_down, T, H, I, E, k, out, ws, ws_bytes,
                            options=None, stream=None):
    return _check("moe_fused_forward_train", load().moe_fused_forward_train(
        _p(x), _p(W_router), _p(router_bias), _p(W_gate_up), _p(W_down), T, H, I, E, k, _p(out), _p(ws), ws_bytes,
        _opt(options), _stream(stream)))


def moe_fused_backward(x, W_router, router_bias, W_gate_up, W_down, dout, T, H, I, E, k, dx, dW_gate_up, dW_down,
                       dW_router, dbias, ws, ws_bytes, options=None, stream=None):
    return _check("moe_fused_backward", load().moe_fused_backward(
        _p(x), _p(W_router), _p(router_bias), _p(W_gate_up), _p(W_down), _p(dout), T, H, I, E, k, _p(dx),
        _p(dW_gate_up), _p(dW_down), _p(dW_router), _p(dbias), _p(ws), ws_bytes, _opt(options), _stream(stream)))


class MoETrain:
    """Owns the training workspace of one bf16 layer shape: forward(), then backward()."""

    def __init__(self, T, H, I, E, k, device="cuda", options=None):
        import torch
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.options = options
        self.ws_bytes = moe_train_workspace_size(T, H, I, E, k)
        if self.ws_bytes == 0:
            raise MoEError("moe_train_workspace_size", MOE_ERR_INVALID_ARG)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def forward(self, x, w, out, stream=None):
        moe_fused_forward_train(x, w["W_router"], w.get("bias"), w["W_gate_up"], w["W_down"], self.T, self.H, self.I,
                                self.E, self.k, out, self.ws, self.ws_bytes, self.options, stream)
        return out

    def backward(self, x, w, dout, stream=None):
        """Returns dict dx (bf16), dW_gate_up, dW_down, dW_router, dbias (fp32)."""
        import torch
        dev = x.device
        g = {"dx": torch.empty(self.T, self.H, dtype=torch.bfloat16, device=dev),
             "dW_gate_up": torch.empty(self.E, 2 * self.I, self.H, dtype=torch.float32, device=dev),
             "dW_down": torch.empty(self.E, self.H, self.I, dtype=torch.float32, device=dev),
             "dW_router": torch.empty(self.E, self.H, dtype=torch.float32, device=dev),
             "dbias": torch.empty(self.E, dtype=torch.float32, device=dev)}
        moe_fused_backward(x, w["W_router"], w.get("bias"), w["W_gate_up"], w["W_down"], dout, self.T, self.H, self.I,
                           self.E, self.k, g["dx"], g["dW_gate_up"], g["dW_down"], g["dW_router"], g["dbias"], self.ws,
                           self.ws_bytes, self.options, stream)
        return g

    def status(self, stream=None) -> int:
        return moe_workspace_status(self.ws, stream)


# ------------------------------------------------------------- conveniences

class FusedMoE:
    """Owns the workspace for one layer shape and calls moe_fused_forward.

    weights: dict with W_router, bias (or None), W_gate_up, W_down (CUDA
    tensors); for FP8 also w1_scale, w2_scale and e4m3 (uint8) weight stacks.
    """

    def __init__(self, dtype, T, H, I, E, k, block_m=0, split_k=0, device="cuda", host_staging=False, options=None):
        import torch
        self.dtype, self.T, self.H, self.I, self.E, self.k = dtype, T, H, I, E, k
        self.options = options  # None (library defaults) or an Options
        self.block_m, self.split_k = block_m, split_k
        self.plan = moe_plan(dtype, T, H, I, E, k, block_m, split_k)
        self.ws_bytes = moe_fused_workspace_size(dtype, T, H, I, E, k, block_m, split_k)
        if self.ws_bytes == 0:
            raise MoEError("moe_fused_workspace_size", MOE_ERR_INVALID_ARG)
        extra = moe_host_staging_bytes(T, H) if host_staging else 0
        self.ws = torch.empty(self.ws_bytes + extra, dtype=torch.uint8, device=device)
        self.layout = moe_workspace_layout(dtype, T, H, I, E, k, block_m, split_k)

    def __call__(self, x, w, out, stream=None, options=None):
        """One forward; `options` (an Options) overrides the layer's own for this call."""
        opts = options if options is not None else self.options
        if opts is None:
            moe_fused_forward(self.dtype, x, w["W_router"], w.get("bias"), w["W_gate_up"], w.get("w1_scale"),
                              w["W_down"], w.get("w2_scale"), self.T, self.H, self.I, self.E, self.k, self.block_m,
                              self.split_k, out, self.ws, self.ws_bytes, stream)
        else:
            moe_fused_forward_ex(self.dtype, x, w["W_router"], w.get("bias"), w["W_gate_up"], w.get("w1_scale"),
                                 w["W_down"], w.get("w2_scale"), self.T, self.H, self.I, self.E, self.k, self.block_m,
                                 self.split_k, out, self.ws, self.ws_bytes, opts, stream)
        return out

    def capture(self, x, w, out, options=None):
        """A CUDA graph of one forward on these buffers (x, the weights, out and the workspace stay
        bound to it): graph.replay() reruns the whole layer, every kernel of the call, with one
        launch from the host -- for shapes where the host's per-call work would outlast the GPU's.
        The library allocates nothing and never synchronises, so a call is capturable as it is."""
        import torch
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self(x, w, out, options=options)  # outside the capture: the per-device launch limits are read here
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(graph):
            self(x, w, out, options=options)
        return graph

    def forward_host(self, x_host, w, out_host, stream=None):
        moe_fused_forward_host(self.dtype, x_host, w["W_router"], w.get("bias"), w["W_gate_up"], w.get("w1_scale"),
                               w["W_down"], w.get("w2_scale"), self.T, self.H, self.I, self.E, self.k,
                               self.block_m, self.split_k, out_host, self.ws, self.ws.numel(), stream)
        return out_host

    def view(self, name, dtype, shape):
        """A tensor view of one intermediate buffer of the workspace (after a call)."""
        import torch
        off = getattr(self.layout, name)
        if off < 0:
            return None
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty(0, dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def status(self, stream=None) -> int:
        return moe_workspace_status(self.ws, stream)
