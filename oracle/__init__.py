"""CPU oracle of the fused MoE decode layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The product path never does, and this package never
imports the product.  The arithmetic lives in ``oracle.c`` (plain C, doubles, bf16 rounding
at the layer's rounding points); this file only builds that library and marshals numpy
arrays into it.

bf16 arrays travel as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP when available)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-lm"]
    tmp = _LIB + f".tmp{os.getpid()}"
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-o", tmp], capture_output=True,
                       text=True)
    if r.returncode != 0:  # no OpenMP runtime: single-threaded build
        r = subprocess.run(base + ["-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _LIB)
    return _LIB


class Spec(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_q_heads", "head_dim", "kv_dim", "q_rank", "o_rank", "n_experts", "topk",
        "moe_inter", "shared_inter", "window", "swa_width", "causal", "block_size",
        "kv_record_bytes")] + [(n, C.c_float) for n in ("eps", "swiglu_clamp", "routed_scale")]


_WKEYS = ["attn_norm", "q_norm", "kv_norm", "ffn_norm", "wqkv", "wqkv_s", "wq_b", "wq_b_s", "wo_a",
          "wo_a_s", "wo_b", "wo_b_s", "router", "sh_gu", "sh_gu_s", "sh_d", "sh_d_s", "ex_gu",
          "ex_gu_s", "ex_d", "ex_d_s"]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _WKEYS]


class Step(C.Structure):
    _fields_ = [("rows", C.c_int32), ("x", C.c_void_p), ("positions", C.c_void_p),
                ("row_req", C.c_void_p), ("block_table", C.c_void_p), ("max_blocks", C.c_int32),
                ("cache", C.c_void_p), ("stride_block", C.c_int64), ("stride_tok", C.c_int64),
                ("num_blocks", C.c_int64), ("force_idx", C.c_void_p)]


_TKEYS = ["xn", "qkv", "q_latn", "kvn", "q", "o", "oa", "h", "u", "logits", "probs", "topk_idx",
          "topk_w", "t_s", "y_s", "t_r", "y_r", "out"]


class Trace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _TKEYS]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            L = _lib
            L.orc_e8m0.restype = C.c_double
            L.orc_e8m0.argtypes = [C.c_uint8]
            L.orc_e4m3.restype = C.c_double
            L.orc_e4m3.argtypes = [C.c_uint8]
            L.orc_e2m1.restype = C.c_double
            L.orc_e2m1.argtypes = [C.c_uint8]
            L.orc_encode_e4m3.restype = C.c_uint8
            L.orc_encode_e4m3.argtypes = [C.c_float]
            L.orc_round_bf16.restype = C.c_double
            L.orc_round_bf16.argtypes = [C.c_double]
            L.orc_bf16_bits.restype = C.c_uint16
            L.orc_bf16_bits.argtypes = [C.c_double]
            L.orc_swiglu.restype = C.c_double
            L.orc_swiglu.argtypes = [C.c_double, C.c_double, C.c_double]
            L.orc_layer.restype = C.c_int
            L.orc_layer.argtypes = [C.POINTER(Spec), C.POINTER(Weights), C.POINTER(Step),
                                    C.POINTER(Trace)]
            L.orc_ffn_layer.restype = None
            L.orc_ffn_layer.argtypes = [C.POINTER(Spec), C.POINTER(Weights), C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                        C.POINTER(Trace)]
            L.orc_kv_insert.restype = C.c_int
            L.orc_attention.restype = C.c_int
            L.orc_key_range.restype = C.c_int
            L.orc_get_threads.restype = C.c_int
        return _lib


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ----------------------------------------------------------------------------- helpers
def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return C.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def make_spec(spec: dict) -> Spec:
    return Spec(**{k: spec[k] for k, _ in Spec._fields_})


# ------------------------------------------------------------------- number formats
def e8m0(code: int) -> float:
    return lib().orc_e8m0(code)


def e4m3(code: int) -> float:
    return lib().orc_e4m3(code)


def e2m1(nibble: int) -> float:
    return lib().orc_e2m1(nibble)


def encode_e4m3(v: float) -> int:
    return int(lib().orc_encode_e4m3(v))


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(v)


def bf16_bits(v: float) -> int:
    return int(lib().orc_bf16_bits(v))


def bf16_round_array(v) -> np.ndarray:
    """float64 array -> bf16 bit patterns, round to nearest even (orc_bf16_bits per element)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_bits_array(_p(v), C.c_size_t(v.size), _p(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def swiglu(g: float, u: float, clamp: float) -> float:
    return lib().orc_swiglu(g, u, clamp)


# ---------------------------------------------------------------------------- stages
def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    x = _c(x, np.uint16)
    rows, dim = x.shape
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(_c(gamma, np.uint16)), rows, dim, C.c_float(eps), _p(out))
    return out


def gemv_mxfp8(x: np.ndarray, w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x bf16 bits [rows, K]; w e4m3 [N, K]; s E8M0 [N/32, K/32] -> float64 [rows, N]."""
    x, w, s = _c(x, np.uint16), _c(w, np.uint8), _c(s, np.uint8)
    rows, k = x.shape
    n = w.shape[0]
    y = np.empty((rows, n), np.float64)
    lib().orc_gemv_mxfp8(_p(x), rows, _p(w), _p(s), n, k, _p(y))
    return y


def gemv_mxfp4(x: np.ndarray, w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x bf16 bits [rows, K]; w packed e2m1 [N, K/2]; s E8M0 [N, K/32] -> float64 [rows, N]."""
    x, w, s = _c(x, np.uint16), _c(w, np.uint8), _c(s, np.uint8)
    rows, k = x.shape
    n = w.shape[0]
    y = np.empty((rows, n), np.float64)
    lib().orc_gemv_mxfp4(_p(x), rows, _p(w), _p(s), n, k, _p(y))
    return y


def kv_quant(kv: np.ndarray):
    """One token's kv (bf16 bits [dim]) -> (codes u8 [dim], scale f32)."""
    kv = _c(kv, np.uint16)
    codes = np.empty(kv.shape[0], np.uint8)
    sc = C.c_float()
    lib().orc_kv_quant(_p(kv), kv.shape[0], _p(codes), C.byref(sc))
    return codes, np.float32(sc.value)


def attend(q, keys, vals, scale):
    q, keys, vals = (_c(a, np.float64) for a in (q, keys, vals))
    out = np.empty(q.shape[0], np.float64)
    lib().orc_attend(_p(q), _p(keys), _p(vals), keys.shape[0], q.shape[0], C.c_double(scale),
                     _p(out))
    return out


def router(u, wr, topk, routed_scale=1.0, positions=None, force_idx=None):
    u, wr = _c(u, np.uint16), _c(wr, np.float32)
    rows, hidden = u.shape
    E = wr.shape[0]
    logits = np.empty((rows, E), np.float32)
    probs = np.empty((rows, E), np.float64)
    idx = np.empty((rows, topk), np.int32)
    w = np.empty((rows, topk), np.float64)
    pos = _c(positions, np.int32) if positions is not None else None
    fi = _c(force_idx, np.int32) if force_idx is not None else None
    lib().orc_router(_p(u), _p(wr), rows, E, hidden, topk, C.c_float(routed_scale),
                     _p(pos) if pos is not None else None, _p(fi) if fi is not None else None,
                     _p(logits), _p(probs), _p(idx), _p(w))
    return dict(logits=logits, probs=probs, idx=idx, w=w)


def ffn(x, gu, gu_s, d, d_s, inter, clamp, fmt4):
    x = _c(x, np.uint16)
    rows, hidden = x.shape
    t = np.empty((rows, inter), np.uint16)
    y = np.empty((rows, hidden), np.float64)
    gu, gu_s, d, d_s = (_c(a, np.uint8) for a in (gu, gu_s, d, d_s))
    lib().orc_ffn(_p(x), rows, int(fmt4), _p(gu), _p(gu_s), _p(d), _p(d_s), inter, hidden,
                  C.c_double(clamp), _p(t), _p(y))
    return t, y


class _StepArrays:
    """Keeps the numpy arrays behind an orc_step alive."""

    def __init__(self, spec, step, cache, force_idx):
        self.x = _c(step["x"], np.uint16)
        self.pos = _c(step["positions"], np.int32)
        self.req = _c(step["row_req"], np.int32)
        self.tab = _c(step["block_table"], np.int32)
        self.cache = cache
        self.fi = _c(force_idx, np.int32) if force_idx is not None else None
        nb = cache.shape[0]
        self.st = Step(rows=self.x.shape[0], x=_p(self.x), positions=_p(self.pos),
                       row_req=_p(self.req), block_table=_p(self.tab),
                       max_blocks=self.tab.shape[1], cache=_p(cache),
                       stride_block=cache.strides[0], stride_tok=cache.strides[1],
                       num_blocks=nb, force_idx=_p(self.fi) if self.fi is not None else None)


def key_range(spec, step, row):
    cache = _c(step["kv_cache"], np.uint8)
    sa = _StepArrays(spec, step, cache, None)
    lo, hi = C.c_int(), C.c_int()
    ok = lib().orc_key_range(C.byref(make_spec(spec)), C.byref(sa.st), row, C.byref(lo),
                             C.byref(hi))
    return (lo.value, hi.value) if ok else None


def kv_insert(spec, step, kvn):
    """Inserts kvn (bf16 bits [rows, kv_dim]) into a copy of the step's cache; returns
    (rc, new cache)."""
    cache = np.array(step["kv_cache"], dtype=np.uint8, copy=True, order="C")
    sa = _StepArrays(spec, step, cache, None)
    kvn = _c(kvn, np.uint16)
    rc = lib().orc_kv_insert(C.byref(make_spec(spec)), C.byref(sa.st), _p(kvn))
    return rc, cache


def attention(spec, step, q, cache=None):
    """q bf16 bits [rows, n_q*head_dim] -> (rc, o bf16 bits)."""
    cache = _c(step["kv_cache"] if cache is None else cache, np.uint8)
    sa = _StepArrays(spec, step, cache, None)
    q = _c(q, np.uint16)
    o = np.empty_like(q)
    rc = lib().orc_attention(C.byref(make_spec(spec)), C.byref(sa.st), _p(q), _p(o))
    return rc, o


def layer(spec: dict, weights: dict, step: dict, force_idx=None):
    """Runs the whole layer step.  Inputs are numpy arrays (bf16 as uint16 bits); the
    step's cache is copied, so the caller's arrays are not modified.  Returns a dict with
    every stage's output plus ``cache`` (after the insert) and ``rc``."""
    E, K, R = spec["n_experts"], spec["topk"], np.asarray(step["x"]).shape[0]
    H, I, Is = spec["hidden"], spec["moe_inter"], spec["shared_inter"]
    QW = spec["n_q_heads"] * spec["head_dim"]
    A = spec["q_rank"] + spec["kv_dim"]
    dt = {"logits": np.float32, "probs": np.float64, "topk_idx": np.int32, "topk_w": np.float64,
          "y_s": np.float64, "y_r": np.float64}
    shapes = dict(xn=(R, H), qkv=(R, A), q_latn=(R, spec["q_rank"]), kvn=(R, spec["kv_dim"]),
                  q=(R, QW), o=(R, QW), oa=(R, spec["o_rank"]), h=(R, H), u=(R, H),
                  logits=(R, E), probs=(R, E), topk_idx=(R, K), topk_w=(R, K), t_s=(R, Is),
                  y_s=(R, H), t_r=(R, K, I), y_r=(R, H), out=(R, H))
    out = {k: np.zeros(shapes[k], dt.get(k, np.uint16)) for k in _TKEYS}
    tr = Trace(**{k: _p(out[k]) for k in _TKEYS})
    wa = {k: _c(weights[k], np.float32 if k == "router" else
                (np.uint16 if k.endswith("norm") else np.uint8)) for k in _WKEYS}
    w = Weights(**{k: _p(wa[k]) for k in _WKEYS})
    cache = np.array(step["kv_cache"], dtype=np.uint8, copy=True, order="C")
    sa = _StepArrays(spec, step, cache, force_idx)
    rc = lib().orc_layer(C.byref(make_spec(spec)), C.byref(w), C.byref(sa.st), C.byref(tr))
    out["cache"] = cache
    out["rc"] = rc
    return out


_FFN_TKEYS = ["h", "u", "logits", "probs", "topk_idx", "topk_w", "t_s", "y_s", "t_r", "y_r",
              "out"]


def ffn_layer(spec: dict, weights: dict, x, attn, positions, force_idx=None):
    """The FFN launch: the residual h = bf16(x + attn) of one step's rows, then the FFN seam
    and the MoE (orc_ffn_layer).  x and attn are bf16 bits [rows, H]; only the FFN entries
    of ``weights`` are read (the attention ones may be absent).  Returns a dict with h, u,
    the routing, the expert outputs and ``out``."""
    x, attn = _c(x, np.uint16), _c(attn, np.uint16)
    pos = _c(positions, np.int32)
    R = x.shape[0]
    E, K, H = spec["n_experts"], spec["topk"], spec["hidden"]
    I, Is = spec["moe_inter"], spec["shared_inter"]
    dt = {"logits": np.float32, "probs": np.float64, "topk_idx": np.int32, "topk_w": np.float64,
          "y_s": np.float64, "y_r": np.float64}
    shapes = dict(h=(R, H), u=(R, H), logits=(R, E), probs=(R, E), topk_idx=(R, K),
                  topk_w=(R, K), t_s=(R, Is), y_s=(R, H), t_r=(R, K, I), y_r=(R, H), out=(R, H))
    out = {k: np.zeros(shapes[k], dt.get(k, np.uint16)) for k in _FFN_TKEYS}
    tr = Trace(**{k: _p(out[k]) for k in _FFN_TKEYS})
    keys = [k for k in _WKEYS if k in weights]
    wa = {k: _c(weights[k], np.float32 if k == "router" else
                (np.uint16 if k.endswith("norm") else np.uint8)) for k in keys}
    w = Weights(**{k: _p(wa[k]) for k in keys})
    fi = _c(force_idx, np.int32) if force_idx is not None else None
    lib().orc_ffn_layer(C.byref(make_spec(spec)), C.byref(w), _p(x), _p(attn), _p(pos),
                        _p(fi) if fi is not None else None, R, C.byref(tr))
    return out


__all__ = ["build", "lib", "set_threads", "get_threads", "e8m0", "e4m3", "e2m1", "encode_e4m3",
           "round_bf16", "bf16_bits", "bf16_round_array", "bf16_to_f64", "swiglu", "rmsnorm", "gemv_mxfp8",
           "gemv_mxfp4", "kv_quant", "attend", "router", "ffn", "key_range", "kv_insert",
           "attention", "layer", "ffn_layer"]
