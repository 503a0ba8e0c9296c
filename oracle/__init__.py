"""CPU oracle for the fused MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding)
never imports, links or calls anything here, and this package never touches
the CUDA library: the two sides meet only through the seeded inputs.

`moe_oracle.c` is plain C compiled with gcc into `_build/liboracle.so` and
driven through ctypes; the thin functions below only marshal numpy arrays.
Every function cites the part of the fused-MoE pages it follows (see the C
source for the definitions).  The host heuristics of the pages are restated
in `heuristics.py`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (plain C11, IEEE arithmetic, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_quant_1x128.argtypes = [P, i, i, P, P]
        lib.oracle_quant_128x128.argtypes = [P, ctypes.c_long, i, P, P]
        lib.oracle_quant_rows.argtypes = [P, ctypes.c_long, i, P, P]
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_mx_exponent.restype = ctypes.c_int
        lib.oracle_mx_exponent.argtypes = [ctypes.c_float]
        lib.oracle_quant_mx4.argtypes = [P, ctypes.c_long, i, P, P]
        lib.oracle_quant_mx4_mt.argtypes = [P, ctypes.c_long, i, P, P, i]
        lib.oracle_router_logit.restype = ctypes.c_float
        lib.oracle_router_logit.argtypes = [P, P, i, P, i]
        lib.oracle_route.argtypes = [P, P, P, i, i, i, i, i, P, P, P, i]
        lib.oracle_align_sort.argtypes = [P, i, i, i, i, P, P, P, P]
        lib.oracle_moe_forward_bf16.argtypes = [P, P, P, P, P, i, i, i, i, i, P, i, P, i]
        lib.oracle_moe_forward_fp8.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, P, i]
        lib.oracle_moe_forward_fp8_token.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, P, i]
        lib.oracle_moe_forward_mxfp4.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, P, i]
        lib.oracle_moe_forward_expert_major.argtypes = [i, P, P, P, P, P, P, P, i, i, i, i, i, P, i, P, i]
        lib.oracle_moe_backward_bf16.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P, P, P, P, P, i]
        _lib = lib
        return lib


def default_threads() -> int:
    return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------------ e4m3

def e4m3_decode(codes) -> np.ndarray:
    """Value of each OCP E4M3 code (fp64)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    """RNE, saturating E4M3 code of each fp32 value."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def e4m3_table() -> np.ndarray:
    """Decoded value of all 256 codes (fp64), for vectorised dequantisation."""
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def quant_1x128(X_bits) -> tuple[np.ndarray, np.ndarray]:
    """Per-1x128-group quantisation ("per_1x128" on the AITER page): codes [R,C], scales [R,C/128]."""
    X = _u16(X_bits)
    R, C = X.reshape(-1, X.shape[-1]).shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 128), np.float32)
    _load().oracle_quant_1x128(_ptr(X), R, C, _ptr(q), _ptr(s))
    return q.reshape(X.shape), s


def quant_128x128(W_bits) -> tuple[np.ndarray, np.ndarray]:
    """Per-128x128-block weight quantisation; W viewed as [rows, C]: codes, scales [rows/128, C/128]."""
    W = _u16(W_bits)
    C = W.shape[-1]
    R = W.size // C
    q = np.empty(W.shape, np.uint8)
    s = np.empty((R // 128, C // 128), np.float32)
    _load().oracle_quant_128x128(_ptr(W), R, C, _ptr(q), _ptr(s))
    return q, s


def quant_rows(X_bits) -> tuple[np.ndarray, np.ndarray]:
    """One scale per row ("per_Token" on the AITER page): X viewed as [rows, C]; codes, scales [rows]."""
    X = _u16(X_bits)
    C = X.shape[-1]
    R = X.size // C
    q = np.empty(X.shape, np.uint8)
    s = np.empty(R, np.float32)
    _load().oracle_quant_rows(_ptr(X), R, C, _ptr(q), _ptr(s))
    return q, s


# ----------------------------------------------------------------- MXFP4

def e2m1_decode(codes) -> np.ndarray:
    """Value of each E2M1 code (0..15: sign << 3 | magnitude index), fp64."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e2m1_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def e2m1_encode(values) -> np.ndarray:
    """Nearest E2M1 code (ties to the even mantissa), clamped to +-6."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.oracle_e2m1_encode(float(x)) for x in v.ravel()], dtype=np.uint8).reshape(v.shape)


def mx_exponent(amax: float) -> int:
    """Shared (unbiased) exponent of an MX FP4 block: floor(log2 amax) - 2, 0 for amax 0."""
    return int(_load().oracle_mx_exponent(float(amax)))


def quant_mx4(X_bits) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 ("per_1x32") quantisation of X viewed as [rows, C]: codes (one per byte), E8M0 scales [rows, C/32]."""
    X = _u16(X_bits)
    C = X.shape[-1]
    R = X.size // C
    q = np.empty(X.shape, np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    _load().oracle_quant_mx4_mt(_ptr(X), R, C, _ptr(q), _ptr(s), default_threads())
    return q, s


# ---------------------------------------------------------------- router

def router_logit(x_row_bits, w_row_bits, bias=None, e: int = 0) -> np.float32:
    """One fp32 router logit in the fixed summation order."""
    x = _u16(x_row_bits)
    w = _u16(w_row_bits)
    b = _f32(bias)
    return np.float32(_load().oracle_router_logit(_ptr(x), _ptr(w), x.shape[-1], _ptr(b), e))


def route(x_bits, Wr_bits, bias, k: int, nthreads: int | None = None, renormalize: bool = True):
    """Gating + top-k (AITER page, section 3): ids [T,k] int32, weights [T,k] fp64, logits [T,E] fp32.

    renormalize=True: softmax over the k selected (the layer's weights); False: softmax over all E
    evaluated at the selected experts."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    T, H = x.shape
    E = Wr.shape[0]
    b = _f32(bias)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float32)
    _load().oracle_route(_ptr(x), _ptr(Wr), _ptr(b), T, H, E, k, 1 if renormalize else 0, _ptr(ids), _ptr(w),
                         _ptr(logits),
                         nthreads or default_threads())
    return ids, w, logits


def align_sort_sizes(T: int, k: int, E: int, B: int) -> tuple[int, int]:
    """Buffer sizes of the token sort (AITER page, section 3.1): T*k + E*B - k and its block count."""
    p = T * k + E * B - k
    return p, (p + B - 1) // B


def align_sort(ids, E: int, B: int):
    """Token sort by expert with per-expert padding to B (AITER page, section 3.1).

    Returns sorted_ids [P_max], sorted_expert_ids [NB_max], num_tokens_post_padded, counts [E]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    P, NB = align_sort_sizes(T, k, E, B)
    sorted_ids = np.empty(P, np.int32)
    sorted_eids = np.empty(NB, np.int32)
    npp = np.zeros(1, np.int32)
    counts = np.empty(E, np.int32)
    _load().oracle_align_sort(_ptr(ids), T, k, E, B, _ptr(sorted_ids), _ptr(sorted_eids), _ptr(npp),
                              _ptr(counts))
    return sorted_ids, sorted_eids, int(npp[0]), counts


# --------------------------------------------------------------- forward

def _expert_major(mode, x, Wr, bias, Wgu, s1, Wd, s2, k, tok, nthreads):
    """The same layer evaluated expert by expert (bit-identical to the per-token loop)."""
    T, H = x.shape
    E, twoI, _ = Wgu.shape
    I = twoI // 2
    out = np.empty((len(tok), H), np.float64)
    rc = _load().oracle_moe_forward_expert_major(mode, _ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu), _ptr(s1),
                                                 _ptr(Wd), _ptr(s2), T, H, I, E, k, _ptr(tok), len(tok), _ptr(out),
                                                 nthreads or default_threads())
    if rc != 0:
        raise MemoryError("oracle expert-major scratch")
    return out


def moe_forward_bf16(x_bits, Wr_bits, bias, Wgu_bits, Wd_bits, k: int, tokens=None,
                     nthreads: int | None = None, expert_major: bool = False) -> np.ndarray:
    """bf16 fused MoE layer (fp64 accumulation) for `tokens` (all if None): out [n, H] fp64.

    expert_major=True evaluates the same sums in the same order expert by expert (faster for many
    tokens; bit-identical results)."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    Wgu = _u16(Wgu_bits)
    Wd = _u16(Wd_bits)
    T, H = x.shape
    E, twoI, _ = Wgu.shape
    I = twoI // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    if expert_major:
        return _expert_major(0, x, Wr, bias, Wgu, None, Wd, None, k, tok, nthreads)
    out = np.empty((len(tok), H), np.float64)
    _load().oracle_moe_forward_bf16(_ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu), _ptr(Wd), T, H, I, E, k,
                                    _ptr(tok), len(tok), _ptr(out), nthreads or default_threads())
    return out


def moe_forward_fp8(x_bits, Wr_bits, bias, Wgu_q, w1s, Wd_q, w2s, k: int, tokens=None,
                    nthreads: int | None = None, expert_major: bool = False) -> np.ndarray:
    """Block-scaled FP8 fused MoE layer for `tokens`: out [n, H] fp64.

    Wgu_q [E,2I,H] / Wd_q [E,H,I] e4m3 codes with scales w1s [E*2I/128, H/128], w2s [E*H/128, I/128]."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    Wgu_q = np.ascontiguousarray(Wgu_q, np.uint8)
    Wd_q = np.ascontiguousarray(Wd_q, np.uint8)
    T, H = x.shape
    E, twoI, _ = Wgu_q.shape
    I = twoI // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    if expert_major:
        return _expert_major(1, x, Wr, bias, Wgu_q, _f32(w1s), Wd_q, _f32(w2s), k, tok, nthreads)
    out = np.empty((len(tok), H), np.float64)
    _load().oracle_moe_forward_fp8(_ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu_q), _ptr(_f32(w1s)),
                                   _ptr(Wd_q), _ptr(_f32(w2s)), T, H, I, E, k, _ptr(tok), len(tok),
                                   _ptr(out), nthreads or default_threads())
    return out


def moe_forward_fp8_token(x_bits, Wr_bits, bias, Wgu_q, w1s, Wd_q, w2s, k: int, tokens=None,
                          nthreads: int | None = None, expert_major: bool = False) -> np.ndarray:
    """Per-token FP8 fused MoE layer for `tokens`: out [n, H] fp64.

    Wgu_q [E,2I,H] / Wd_q [E,H,I] e4m3 codes with one scale per output channel: w1s [E*2I], w2s [E*H]."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    Wgu_q = np.ascontiguousarray(Wgu_q, np.uint8)
    Wd_q = np.ascontiguousarray(Wd_q, np.uint8)
    T, H = x.shape
    E, twoI, _ = Wgu_q.shape
    I = twoI // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    if expert_major:
        return _expert_major(2, x, Wr, bias, Wgu_q, _f32(w1s), Wd_q, _f32(w2s), k, tok, nthreads)
    out = np.empty((len(tok), H), np.float64)
    _load().oracle_moe_forward_fp8_token(_ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu_q), _ptr(_f32(w1s)),
                                         _ptr(Wd_q), _ptr(_f32(w2s)), T, H, I, E, k, _ptr(tok), len(tok),
                                         _ptr(out), nthreads or default_threads())
    return out


def moe_forward_mxfp4(x_bits, Wr_bits, bias, Wgu_q, w1x, Wd_q, w2x, k: int, tokens=None,
                      nthreads: int | None = None, expert_major: bool = False) -> np.ndarray:
    """MXFP4 fused MoE layer for `tokens`: out [n, H] fp64.

    Wgu_q [E,2I,H] / Wd_q [E,H,I] E2M1 codes (one per byte) with E8M0 scales w1x [E*2I, H/32], w2x [E*H, I/32]."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    Wgu_q = np.ascontiguousarray(Wgu_q, np.uint8)
    Wd_q = np.ascontiguousarray(Wd_q, np.uint8)
    w1x = np.ascontiguousarray(w1x, np.uint8)
    w2x = np.ascontiguousarray(w2x, np.uint8)
    T, H = x.shape
    E, twoI, _ = Wgu_q.shape
    I = twoI // 2
    tok = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    if expert_major:
        return _expert_major(3, x, Wr, bias, Wgu_q, w1x, Wd_q, w2x, k, tok, nthreads)
    out = np.empty((len(tok), H), np.float64)
    _load().oracle_moe_forward_mxfp4(_ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu_q), _ptr(w1x), _ptr(Wd_q),
                                     _ptr(w2x), T, H, I, E, k, _ptr(tok), len(tok), _ptr(out),
                                     nthreads or default_threads())
    return out


def moe_backward_bf16(x_bits, Wr_bits, bias, Wgu_bits, Wd_bits, dout_bits, k: int, nthreads: int | None = None):
    """Gradients of the bf16 layer for loss = sum(dout * out): dict of fp64 arrays
    dx [T,H], dW_gate_up [E,2I,H], dW_down [E,H,I], dW_router [E,H], dbias [E]."""
    x = _u16(x_bits)
    Wr = _u16(Wr_bits)
    Wgu = _u16(Wgu_bits)
    Wd = _u16(Wd_bits)
    dout = _u16(dout_bits)
    T, H = x.shape
    E, twoI, _ = Wgu.shape
    I = twoI // 2
    g = {"dx": np.empty((T, H)), "dW_gate_up": np.empty((E, 2 * I, H)), "dW_down": np.empty((E, H, I)),
         "dW_router": np.empty((E, H)), "dbias": np.empty(E)}
    rc = _load().oracle_moe_backward_bf16(_ptr(x), _ptr(Wr), _ptr(_f32(bias)), _ptr(Wgu), _ptr(Wd), _ptr(dout),
                                          T, H, I, E, k, _ptr(g["dx"]), _ptr(g["dW_gate_up"]), _ptr(g["dW_down"]),
                                          _ptr(g["dW_router"]), _ptr(g["dbias"]), nthreads or default_threads())
    if rc != 0:
        raise MemoryError("oracle backward scratch")
    return g
