"""Plain CPU oracle of the MoE layer step (fp64 C code, loaded with ctypes).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  It shares no code with the
CUDA path.  Each function cites the passage it follows in ``moe_oracle.c``.

Parity status per function (pins live in ``tests/test_oracle_pins.py``):
quantise/dequantise, router logits, top-k and weights, GELU, the pre-norm,
the layer, bucketing and the LFU step are all pinned.  The layer is pinned
through its single-expert and invariance cases, and through a k = 2
decomposition: every token's output against the weighted sum of its
experts' FFNs plus the shared FFN, each computed by an independent numpy
path from the canonical bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attn_oracle.c")]
_LIB = os.path.join(_HERE, "_moe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over independent rows)."""
    if force or not os.path.exists(_LIB) or any(
            os.path.getmtime(_LIB) < os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, *_SRCS, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class QT(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class Layer(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_experts", ctypes.c_int), ("d_expert", ctypes.c_int),
                ("top_k", ctypes.c_int), ("d_shared", ctypes.c_int), ("group", ctypes.c_int),
                ("router", QT), ("logit_bias", ctypes.c_void_p),
                ("shared_gate", QT), ("shared_up", QT), ("shared_down", QT),
                ("gate", QT), ("up", QT), ("down", QT)]


class AttnLayer(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("group", ctypes.c_int),
                ("wq", QT), ("wk", QT), ("wv", QT), ("wo", QT)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            L.orc_set_threads.restype = i32
            L.orc_set_threads.argtypes = [i32]
            L.orc_half_to_double.restype = ctypes.c_double
            L.orc_half_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = ctypes.c_double
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_gelu_tanh.restype = ctypes.c_double
            L.orc_gelu_tanh.argtypes = [ctypes.c_double]
            L.orc_quantise.restype = i32
            L.orc_quantise.argtypes = [P, i64, i64, i32, i32, P, P, P]
            L.orc_dequant.restype = None
            L.orc_dequant.argtypes = [ctypes.POINTER(QT), i64, i64, i32, i32, P]
            L.orc_router_logits.restype = None
            L.orc_router_logits.argtypes = [ctypes.POINTER(Layer), P, P]
            L.orc_topk.restype = None
            L.orc_topk.argtypes = [P, i32, i32, P]
            L.orc_routing_weights.restype = None
            L.orc_routing_weights.argtypes = [P, P, i32, P]
            L.orc_ffn.restype = None
            L.orc_ffn.argtypes = [ctypes.POINTER(QT)] * 3 + [i32, i32, i32, P, P]
            L.orc_moe_layer.restype = i32
            L.orc_moe_layer.argtypes = [ctypes.POINTER(Layer), P, i32, P, i32, P, P, P, P]
            L.orc_rms_normalise.restype = None
            L.orc_rms_normalise.argtypes = [P, i32, ctypes.c_double, P]
            L.orc_bucket.restype = i32
            L.orc_bucket.argtypes = [P, i32, i32, i32, P, P, P]
            L.orc_lfu_step.restype = i32
            L.orc_lfu_step.argtypes = [i32, P, P, P, i64, P, i32, i32, P, P, P]
            L.ora_rms.restype = None
            L.ora_rms.argtypes = [P, i32, ctypes.c_double]
            L.ora_rope.restype = None
            L.ora_rope.argtypes = [P, i32, i64, ctypes.c_double]
            L.ora_attn_step.restype = i32
            L.ora_attn_step.argtypes = [ctypes.POINTER(AttnLayer), P, i64, i32, ctypes.c_double,
                                        P, P, i64, P]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(x, dtype=None):
    """numpy view of a numpy array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if x.element_size() == 2 and x.is_floating_point():
            import torch
            x = x.view(torch.int16)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    return a.view(dtype) if dtype is not None else a


# ------------------------------------------------------------------ scalars

def set_threads(n: int = 0) -> int:
    """OpenMP threads of the oracle's loops from now on (n <= 0: leave as is);
    returns the count in effect.  Results do not depend on it."""
    return int(lib().orc_set_threads(int(n)))


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(int(h) & 0xFFFF)


def gelu_tanh(x: float) -> float:
    return lib().orc_gelu_tanh(float(x))


# ---------------------------------------------------------- quantised data

def quantise(w: np.ndarray, bits: int, group: int):
    """fp32 [rows, cols] -> (q uint8, scale uint16, bias uint16) canonical."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    q = np.zeros((rows, cols * bits // 8), dtype=np.uint8)
    s = np.zeros((rows, cols // group), dtype=np.uint16)
    b = np.zeros((rows, cols // group), dtype=np.uint16)
    rc = lib().orc_quantise(_p(w), rows, cols, bits, group, _p(q), _p(s), _p(b))
    if rc != 0:
        raise ValueError("orc_quantise: bad arguments")
    return q, s, b


def _qt(q, s, b, keep):
    q, s, b = _np(q, np.uint8), _np(s, np.uint16), _np(b, np.uint16)
    keep.extend([q, s, b])
    return QT(q.ctypes.data, s.ctypes.data, b.ctypes.data)


def dequant(q, s, b, rows: int, cols: int, bits: int, group: int) -> np.ndarray:
    keep = []
    t = _qt(q, s, b, keep)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_dequant(ctypes.byref(t), rows, cols, bits, group, _p(out))
    return out


# ------------------------------------------------------------------ routing

def topk(logits: np.ndarray, k: int) -> np.ndarray:
    l = np.ascontiguousarray(logits, dtype=np.float32)
    ids = np.empty(k, dtype=np.int32)
    lib().orc_topk(_p(l), l.shape[0], k, _p(ids))
    return ids


def routing_weights(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    l = np.ascontiguousarray(logits, dtype=np.float32)
    i = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.empty(i.shape[0], dtype=np.float64)
    lib().orc_routing_weights(_p(l), _p(i), i.shape[0], _p(w))
    return w


# -------------------------------------------------------------------- layer

class LayerView:
    """ctypes view of one layer's canonical weights (keeps the arrays alive)."""

    def __init__(self, shape, layer: Dict[str, object]):
        self.keep = []

        def qt(name):
            t = layer[name]
            if hasattr(t, "q"):
                return _qt(t.q, t.scale, t.bias, self.keep)
            return _qt(*t, self.keep)

        lb = layer.get("logit_bias")
        lb_ptr = None
        if lb is not None:
            lb = _np(lb, np.float32)
            self.keep.append(lb)
            lb_ptr = lb.ctypes.data
        self.s = Layer(shape.d_model, shape.n_experts, shape.d_expert, shape.top_k,
                       shape.d_shared, shape.group, qt("router"), lb_ptr,
                       qt("shared_gate"), qt("shared_up"), qt("shared_down"),
                       qt("gate"), qt("up"), qt("down"))
        self.shape = shape


def router_logits(view: LayerView, x_bf16: np.ndarray) -> np.ndarray:
    x = np.array([lib().orc_bf16_to_double(int(v)) for v in _np(x_bf16, np.uint16).ravel()])
    out = np.empty(view.shape.n_experts, dtype=np.float32)
    lib().orc_router_logits(ctypes.byref(view.s), _p(x), _p(out))
    return out


RMS_EPS = 1e-6


def rms_normalise(x: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    xx = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(xx)
    lib().orc_rms_normalise(_p(xx), xx.shape[0], eps, _p(out))
    return out


def moe_layer(view: LayerView, x_bf16, forced_ids: Optional[np.ndarray] = None,
              prenorm: bool = False):
    """Returns dict(ids [T,k] int32, w [T,k] f64, logits [T,E] f32, y [T,D] f64).

    prenorm: the layer reads the RMS-normalised input (unit gain, eps 1e-6)."""
    sh = view.shape
    x = _np(x_bf16, np.uint16)
    T = x.shape[0]
    ids = np.empty((T, sh.top_k), dtype=np.int32)
    w = np.empty((T, sh.top_k), dtype=np.float64)
    logits = np.empty((T, sh.n_experts), dtype=np.float32)
    y = np.empty((T, sh.d_model), dtype=np.float64)
    fptr = None
    if forced_ids is not None:
        forced_ids = np.ascontiguousarray(forced_ids, dtype=np.int32).reshape(T, sh.top_k)
        fptr = forced_ids.ctypes.data
    rc = lib().orc_moe_layer(ctypes.byref(view.s), _p(x), T, fptr, 1 if prenorm else 0,
                             _p(ids), _p(w),
                             _p(logits), _p(y))
    if rc != 0:
        raise ValueError("orc_moe_layer: bad arguments")
    return dict(ids=ids, w=w, logits=logits, y=y)


def ffn(wg, wu, wd, D: int, F: int, group: int, x: np.ndarray) -> np.ndarray:
    keep = []
    g, u, d = _qt(*wg, keep), _qt(*wu, keep), _qt(*wd, keep)
    xx = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(D, dtype=np.float64)
    lib().orc_ffn(ctypes.byref(g), ctypes.byref(u), ctypes.byref(d), D, F, group, _p(xx), _p(out))
    return out


# ------------------------------------------------------------ bucketing

def bucket(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    if lib().orc_bucket(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm)) != 0:
        raise ValueError("orc_bucket: id out of range")
    return counts, offsets, perm


# ------------------------------------------------------------ LFU cache

class LFUCache:
    """State of one layer's slot cache driven by the oracle's LFU step."""

    def __init__(self, n_slots: int, n_experts: int):
        self.n_slots, self.n_experts = n_slots, n_experts
        self.expert = np.full(n_slots, -1, dtype=np.int32)
        self.count = np.zeros(n_slots, dtype=np.int64)
        self.last = np.zeros(n_slots, dtype=np.int64)
        self.step_no = 0

    def step(self, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        k = ids.shape[0]
        hit = np.empty(k, dtype=np.int32)
        slot = np.empty(k, dtype=np.int32)
        ev = np.empty(k, dtype=np.int32)
        m = lib().orc_lfu_step(self.n_slots, _p(self.expert), _p(self.count), _p(self.last),
                               self.step_no, _p(ids), k, self.n_experts, _p(hit), _p(slot), _p(ev))
        if m < 0:
            raise ValueError("orc_lfu_step: bad ids")
        self.step_no += 1
        return hit, slot, ev


# ------------------------------------------------------- decode attention

def head_rms(v: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) (unit-gain RMS normalisation of one head)."""
    vv = np.ascontiguousarray(v, dtype=np.float64).copy()
    lib().ora_rms(_p(vv), vv.shape[0], eps)
    return vv


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary embedding of one head vector at position pos (rotate-half pairs)."""
    vv = np.ascontiguousarray(v, dtype=np.float64).copy()
    lib().ora_rope(_p(vv), vv.shape[0], int(pos), float(theta))
    return vv


class AttnState:
    """One attention layer of the oracle: its canonical 4-bit weights and its
    own fp16 KV cache ([Hkv][cap][d], position p in slot p % cap)."""

    def __init__(self, shape, weights: Dict[str, object], cap: int, window: int, theta: float):
        self.keep = []

        def qt(name):
            t = weights[name]
            if hasattr(t, "q"):
                return _qt(t.q, t.scale, t.bias, self.keep)
            return _qt(*t, self.keep)

        self.s = AttnLayer(shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                           shape.group, qt("wq"), qt("wk"), qt("wv"), qt("wo"))
        self.shape, self.cap, self.window, self.theta = shape, cap, window, theta
        n = shape.n_kv_heads * cap * shape.head_dim
        self.k = np.zeros(n, np.uint16)
        self.v = np.zeros(n, np.uint16)

    def step(self, x_bf16, pos: int) -> np.ndarray:
        """The attention block's output (fp64 [D], before the residual) for the
        token x at position pos; stores the token's k, v in the cache."""
        x = _np(x_bf16, np.uint16).reshape(-1)
        y = np.empty(self.shape.d_model, np.float64)
        rc = lib().ora_attn_step(ctypes.byref(self.s), _p(x), int(pos), int(self.window),
                                 float(self.theta), _p(self.k), _p(self.v), int(self.cap), _p(y))
        if rc != 0:
            raise ValueError("ora_attn_step: bad arguments")
        return y
