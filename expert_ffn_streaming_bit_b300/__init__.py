"""Python binding of libmoe_b300 (the C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C entry points' names.  Importing this package
loads the in-tree ``libmoe_b300.so``, rebuilding it first when a source is
newer; if it cannot be built or loaded the import fails (there is no fallback
path).  Build it with ``python -m expert_ffn_streaming_bit_b300.build``
or ``__graft_entry__.build()``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB

# Rebuild in-tree when a source is newer than the library (a no-op otherwise).
# A failed build or a missing library makes this import fail: there is no
# fallback path.
if _build.stale():
    _build.build()
if not os.path.exists(LIB_PATH):
    raise ImportError("libmoe_b300.so is not built (python -m expert_ffn_streaming_bit_b300.build)")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
MOE_FWD_RESIDUAL = 1
MOE_FWD_PRENORM = 2
MOE_PLAN_ONLY = 1
MOE_INJECT_NONE, MOE_INJECT_H2D_FAIL, MOE_INJECT_SLOW_COPY, MOE_INJECT_PINNED_ALLOC_FAIL = 0, 1, 2, 3
MOE_INJECT_DEVICE_STALL = 4
MOE_INJECT_READ_FAIL = 5
MOE_INJECT_GEMM_STALL = 6
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_OOM", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_TIMEOUT", -5: "MOE_ERR_INJECTED", -6: "MOE_ERR_STATE",
          -7: "MOE_ERR_DEVICE", -8: "MOE_ERR_IO"}


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("d_expert", ctypes.c_int), ("top_k", ctypes.c_int), ("d_shared", ctypes.c_int),
                ("group", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_slots", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("expert_store", ctypes.c_char_p),
                ("io_threads", ctypes.c_int)]


class moe_qtensor(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [("router", moe_qtensor), ("router_logit_bias", ctypes.c_void_p),
                ("shared_gate", moe_qtensor), ("shared_up", moe_qtensor),
                ("shared_down", moe_qtensor), ("exp_gate", ctypes.POINTER(moe_qtensor)),
                ("exp_up", ctypes.POINTER(moe_qtensor)), ("exp_down", ctypes.POINTER(moe_qtensor))]


class moe_cache_result(ctypes.Structure):
    _fields_ = [("hit", ctypes.c_int32 * 64), ("slot", ctypes.c_int32 * 64),
                ("evicted", ctypes.c_int32 * 64), ("misses", ctypes.c_int)]


class moe_layer_stats(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("weights", ctypes.c_void_p), ("hits", ctypes.c_int),
                ("misses", ctypes.c_int), ("bytes_h2d", ctypes.c_int64),
                ("cache", ctypes.POINTER(moe_cache_result))]


class moe_info(ctypes.Structure):
    _fields_ = [("device_weight_bytes", ctypes.c_int64), ("pinned_pool_bytes", ctypes.c_int64),
                ("device_scratch_bytes", ctypes.c_int64), ("expert_blob_bytes", ctypes.c_int64),
                ("num_sms", ctypes.c_int), ("store_direct_io", ctypes.c_int),
                ("io_threads", ctypes.c_int)]


class moe_attn_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("group", ctypes.c_int), ("n_layers", ctypes.c_int),
                ("window", ctypes.c_int), ("max_seq", ctypes.c_int),
                ("sliding", ctypes.c_void_p), ("rope_theta", ctypes.c_void_p)]


class moe_attn_weights(ctypes.Structure):
    _fields_ = [("wq", moe_qtensor), ("wk", moe_qtensor), ("wv", moe_qtensor), ("wo", moe_qtensor)]


_P, _I = ctypes.c_void_p, ctypes.c_int
_sig = {
    "moe_create": (_I, [ctypes.POINTER(moe_config), ctypes.POINTER(moe_layer_weights),
                        ctypes.POINTER(ctypes.c_void_p)]),
    "moe_destroy": (None, [_P]),
    "moe_store_write": (_I, [ctypes.POINTER(moe_config), ctypes.POINTER(moe_layer_weights),
                             ctypes.c_char_p]),
    "moe_layer_forward": (_I, [_P, _I, _P, _I, _P, _I, _P, _P, ctypes.POINTER(moe_layer_stats)]),
    "moe_forward_stack": (_I, [_P, _P, _I, _P, _I, _P]),
    "moe_forward_stack_host": (_I, [_P, _P, _I, _P, _I, _P]),
    "moe_forward_stack_noalloc": (_I, [_P, _P, _P, _I, _P, _P]),
    "moe_stack_ids": (_I, [_P, _I, _I, _P, _P]),
    "moe_cache_step": (_I, [_P, _I, _P, _I, _I, ctypes.POINTER(moe_cache_result)]),
    "moe_cache_reset": (_I, [_P]),
    "moe_trace_enable": (_I, [_P, _I]),
    "moe_trace_read": (_I, [_P, _P, _I]),
    "moe_prefill_phase_ms": (_I, [_P, _P, _P]),
    "moe_last_buckets": (_I, [_P, _P, _P, _P]),
    "moe_slot_plan_create": (_I, [_I, _I, ctypes.POINTER(ctypes.c_void_p)]),
    "moe_slot_plan_step": (_I, [_P, _P, _I, ctypes.POINTER(moe_cache_result)]),
    "moe_slot_plan_destroy": (None, [_P]),
    "moe_get_info": (_I, [_P, ctypes.POINTER(moe_info)]),
    "moe_debug_inject": (_I, [_P, _I, _I]),
    "moe_set_timeout_ms": (_I, [_P, _I]),
    "moe_attn_create": (_I, [ctypes.POINTER(moe_attn_config), ctypes.POINTER(moe_attn_weights),
                             ctypes.POINTER(ctypes.c_void_p)]),
    "moe_attn_destroy": (None, [_P]),
    "moe_attn_last_error": (ctypes.c_char_p, [_P]),
    "moe_attn_forward": (_I, [_P, _I, _P, ctypes.c_longlong, _P, _I, _P]),
    "moe_attn_reset": (_I, [_P]),
    "moe_decode_step": (_I, [_P, _P, _P, ctypes.c_longlong, _P, _I, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_error": (ctypes.c_char_p, [_P]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def moe_last_error(handle=None) -> str:
    h = handle.ptr if isinstance(handle, Handle) else handle
    return _lib.moe_last_error(h).decode()


def _check(status: int, handle=None):
    if status != MOE_OK:
        raise MoEError(status, moe_last_error(handle))


class Handle:
    """Owns a moe_handle*; destroyed with the object or by moe_destroy."""

    def __init__(self, ptr: int, cfg: moe_config):
        self.ptr = ptr
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib.moe_destroy(self.ptr)
            self.ptr = None


def _host(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous()
        if a.is_floating_point() and a.element_size() == 2:
            import torch
            a = a.view(torch.int16)
        a = a.numpy()
    return np.ascontiguousarray(a)


def _qt(t, keep: list) -> moe_qtensor:
    q, s, b = (_host(v) for v in ((t.q, t.scale, t.bias) if hasattr(t, "q") else t))
    keep.extend([q, s, b])
    return moe_qtensor(q.ctypes.data, s.ctypes.data, b.ctypes.data)


def _layer_struct(layer: Dict[str, object], keep: list, experts: bool = True) -> moe_layer_weights:
    w = moe_layer_weights()
    w.router = _qt(layer["router"], keep)
    lb = layer.get("logit_bias")
    if lb is not None:
        lb = _host(lb).astype(np.float32)
        keep.append(lb)
        w.router_logit_bias = lb.ctypes.data
    w.shared_gate = _qt(layer["shared_gate"], keep)
    w.shared_up = _qt(layer["shared_up"], keep)
    w.shared_down = _qt(layer["shared_down"], keep)
    for name, field in (("gate", "exp_gate"), ("up", "exp_up"), ("down", "exp_down")):
        if not experts:
            continue
        t = layer[name]
        q, s, b = _host(t.q), _host(t.scale), _host(t.bias)
        keep.extend([q, s, b])
        E = q.shape[0]
        arr = (moe_qtensor * E)()
        for e in range(E):
            arr[e] = moe_qtensor(q[e].ctypes.data, s[e].ctypes.data, b[e].ctypes.data)
        keep.append(arr)
        setattr(w, field, ctypes.cast(arr, ctypes.POINTER(moe_qtensor)))
    return w


def moe_create(shape, layers: Sequence[Dict[str, object]], n_slots: int = 0,
               max_tokens: int = 1, expert_store: Optional[str] = None,
               io_threads: int = 8) -> Handle:
    """shape: a synth.MoEShape-like object; layers: per-layer canonical weights.
    expert_store: path of a file written by moe_store_write (streaming mode
    then reads the routed experts from it; only the router and shared
    tensors of `layers` are passed)."""
    cfg = moe_config(shape.d_model, shape.n_experts, shape.d_expert, shape.top_k,
                     shape.d_shared, shape.group, len(layers), n_slots, max_tokens,
                     expert_store.encode() if expert_store else None,
                     io_threads if expert_store else 0)
    keep: List[object] = []
    arr = (moe_layer_weights * len(layers))(
        *[_layer_struct(l, keep, experts=expert_store is None) for l in layers])
    out = ctypes.c_void_p()
    _check(_lib.moe_create(ctypes.byref(cfg), arr, ctypes.byref(out)))
    return Handle(out.value, cfg)


def moe_store_write(shape, layers: Sequence[Dict[str, object]], path: str):
    """Write the expert store file of `layers` (routed experts only) to path."""
    cfg = moe_config(shape.d_model, shape.n_experts, shape.d_expert, shape.top_k,
                     shape.d_shared, shape.group, len(layers), 0, 1, None, 0)
    keep: List[object] = []
    arr = (moe_layer_weights * len(layers))(*[_layer_struct(l, keep) for l in layers])
    _check(_lib.moe_store_write(ctypes.byref(cfg), arr, path.encode()))


def moe_destroy(handle: Handle):
    if handle.ptr:
        _lib.moe_destroy(handle.ptr)
        handle.ptr = None


def _dev_ptr(t) -> int:
    assert t.is_cuda and t.is_contiguous()
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def moe_layer_forward(handle: Handle, layer: int, x, y, flags: int = 0, forced_ids=None,
                      stream=None, want_ids: bool = False):
    """x, y: CUDA bf16 tensors [T, D].  Returns a dict of stats (ids/weights on
    request; in streaming mode also the cache step: hit, slot and evicted per id)."""
    T = x.shape[0]
    K = handle.cfg.top_k
    st = moe_layer_stats()
    cr = moe_cache_result()
    st.cache = ctypes.pointer(cr)
    ids = w = None
    if want_ids:
        ids = np.empty((T, K), np.int32)
        w = np.empty((T, K), np.float32)
        st.ids, st.weights = ids.ctypes.data, w.ctypes.data
    fptr = None
    if forced_ids is not None:
        forced_ids = np.ascontiguousarray(forced_ids, dtype=np.int32).reshape(T, K)
        fptr = forced_ids.ctypes.data
    _check(_lib.moe_layer_forward(handle.ptr, layer, _dev_ptr(x), T, _dev_ptr(y), flags, fptr,
                                  _stream_ptr(stream), ctypes.byref(st)), handle)
    out = dict(ids=ids, weights=w, hits=st.hits, misses=st.misses, bytes_h2d=st.bytes_h2d)
    if handle.cfg.n_slots > 0:
        out.update(hit=np.array(cr.hit[:K], np.int32), slot=np.array(cr.slot[:K], np.int32),
                   evicted=np.array(cr.evicted[:K], np.int32))
    return out


def moe_forward_stack(handle: Handle, x, y, n_layers: int, stream=None):
    _check(_lib.moe_forward_stack(handle.ptr, _dev_ptr(x), x.shape[0], _dev_ptr(y), n_layers,
                                  _stream_ptr(stream)), handle)


def moe_forward_stack_host(handle: Handle, x: np.ndarray, y: np.ndarray, n_layers: int,
                           stream=None):
    """x, y: host uint16 (bf16 bits) arrays [T, D]; y is written."""
    assert x.dtype == np.uint16 and y.dtype == np.uint16 and y.flags["C_CONTIGUOUS"]
    x = np.ascontiguousarray(x)
    _check(_lib.moe_forward_stack_host(handle.ptr, x.ctypes.data, x.shape[0], y.ctypes.data,
                                       n_layers, _stream_ptr(stream)), handle)


def moe_forward_stack_noalloc(handle: Handle, x, y, n_layers: int, stream=None,
                              want_status: bool = False):
    """One token through the stack with the library's fixed scratch array
    (no allocation of any kind).  x, y: CUDA bf16 tensors [1, D].  With
    want_status, returns the kernel's device status word (0 ok, 1 a device
    wait ran out, 2 an expert id out of range); the call then waits for it."""
    assert x.shape[0] == 1 and y.shape[0] == 1
    status = np.zeros(1, np.int32) if want_status else None
    _check(_lib.moe_forward_stack_noalloc(handle.ptr, _dev_ptr(x), _dev_ptr(y), n_layers,
                                          _stream_ptr(stream),
                                          status.ctypes.data if want_status else None), handle)
    return int(status[0]) if want_status else None


def moe_stack_ids(handle: Handle, n_layers: int, T: int):
    K = handle.cfg.top_k
    ids = np.empty((n_layers, T, K), np.int32)
    w = np.empty((n_layers, T, K), np.float32)
    _check(_lib.moe_stack_ids(handle.ptr, n_layers, T, ids.ctypes.data, w.ctypes.data), handle)
    return ids, w


def moe_cache_step(handle: Handle, layer: int, ids, flags: int = 0):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    r = moe_cache_result()
    _check(_lib.moe_cache_step(handle.ptr, layer, ids.ctypes.data, ids.shape[0], flags,
                               ctypes.byref(r)), handle)
    k = ids.shape[0]
    return (np.array(r.hit[:k], np.int32), np.array(r.slot[:k], np.int32),
            np.array(r.evicted[:k], np.int32), r.misses)


def moe_last_buckets(handle: Handle, T: int):
    """(counts [E], offsets [E+1], perm [T*k]) of the last multi-token call."""
    E, K = handle.cfg.n_experts, handle.cfg.top_k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * K, np.int32)
    _check(_lib.moe_last_buckets(handle.ptr, counts.ctypes.data, offsets.ctypes.data,
                                 perm.ctypes.data), handle)
    return counts, offsets, perm


MOE_TRACE_EVENTS = 13


def moe_trace_enable(handle: Handle, on: bool = True):
    _check(_lib.moe_trace_enable(handle.ptr, 1 if on else 0), handle)


def moe_trace_read(handle: Handle, n_layers: int) -> np.ndarray:
    """int64 [num_sms][n_layers][MOE_TRACE_EVENTS] %globaltimer stamps (ns)."""
    G = moe_get_info(handle)["num_sms"]
    out = np.zeros((G, n_layers, MOE_TRACE_EVENTS), np.int64)
    _check(_lib.moe_trace_read(handle.ptr, out.ctypes.data, n_layers), handle)
    return out


def moe_prefill_phase_ms(handle: Handle):
    """Summed CUDA-event times (ms) of the recorded multi-token calls:
    (router, bucketing, gate/up GEMM, down GEMM, combine), and the call count."""
    ms = (ctypes.c_float * 5)()
    calls = ctypes.c_int()
    _check(_lib.moe_prefill_phase_ms(handle.ptr, ms, ctypes.byref(calls)), handle)
    return list(ms), calls.value


def moe_cache_reset(handle: Handle):
    _check(_lib.moe_cache_reset(handle.ptr), handle)


class SlotPlan:
    """Host-only LFU slot planner (moe_slot_plan_*)."""

    def __init__(self, n_slots: int, n_experts: int):
        out = ctypes.c_void_p()
        _check(_lib.moe_slot_plan_create(n_slots, n_experts, ctypes.byref(out)))
        self.ptr = out.value

    def step(self, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        r = moe_cache_result()
        _check(_lib.moe_slot_plan_step(self.ptr, ids.ctypes.data, ids.shape[0], ctypes.byref(r)))
        k = ids.shape[0]
        return (np.array(r.hit[:k], np.int32), np.array(r.slot[:k], np.int32),
                np.array(r.evicted[:k], np.int32))

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib.moe_slot_plan_destroy(self.ptr)
            self.ptr = None


def moe_slot_plan_create(n_slots: int, n_experts: int) -> SlotPlan:
    return SlotPlan(n_slots, n_experts)


def moe_slot_plan_step(plan: SlotPlan, ids):
    return plan.step(ids)


def moe_slot_plan_destroy(plan: SlotPlan):
    plan.__del__()


def moe_get_info(handle: Handle) -> Dict[str, int]:
    i = moe_info()
    _check(_lib.moe_get_info(handle.ptr, ctypes.byref(i)), handle)
    return {f: getattr(i, f) for f, _ in moe_info._fields_}


def moe_debug_inject(handle: Optional[Handle], what: int, arg: int = 0):
    _check(_lib.moe_debug_inject(handle.ptr if handle else None, what, arg), handle)


def moe_set_timeout_ms(handle: Handle, ms: int):
    _check(_lib.moe_set_timeout_ms(handle.ptr, ms), handle)


# ------------------------------------------------------- decode attention

class AttnHandle:
    """Owns a moe_attn*; destroyed with the object or by moe_attn_destroy."""

    def __init__(self, ptr: int, cfg: moe_attn_config):
        self.ptr = ptr
        self.cfg = cfg

    def __del__(self):
        if getattr(self, "ptr", None):
            _lib.moe_attn_destroy(self.ptr)
            self.ptr = None


def _attn_check(status: int, handle: Optional[AttnHandle] = None):
    if status != MOE_OK:
        msg = _lib.moe_attn_last_error(handle.ptr if handle else None).decode()
        raise MoEError(status, msg)


def moe_attn_create(shape, layers: Sequence[Dict[str, object]]) -> AttnHandle:
    """shape: a synth.AttnShape-like object (sliding flags and RoPE bases per
    layer); layers: per-layer canonical weights wq, wk, wv, wo."""
    L = len(layers)
    sliding = np.ascontiguousarray([int(shape.sliding[l]) for l in range(L)], np.int32)
    theta = np.ascontiguousarray([shape.theta(l) for l in range(L)], np.float32)
    cfg = moe_attn_config(shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                          shape.group, L, shape.window, shape.max_seq, sliding.ctypes.data,
                          theta.ctypes.data)
    keep: List[object] = [sliding, theta]
    arr = (moe_attn_weights * L)(*[moe_attn_weights(_qt(l["wq"], keep), _qt(l["wk"], keep),
                                                    _qt(l["wv"], keep), _qt(l["wo"], keep))
                                   for l in layers])
    out = ctypes.c_void_p()
    _attn_check(_lib.moe_attn_create(ctypes.byref(cfg), arr, ctypes.byref(out)))
    return AttnHandle(out.value, cfg)


def moe_attn_destroy(handle: AttnHandle):
    if handle.ptr:
        _lib.moe_attn_destroy(handle.ptr)
        handle.ptr = None


def moe_attn_forward(handle: AttnHandle, layer: int, x, pos: int, y, flags: int = 0, stream=None):
    """x, y: CUDA bf16 tensors [1, D] (or [D])."""
    _attn_check(_lib.moe_attn_forward(handle.ptr, layer, _dev_ptr(x), int(pos), _dev_ptr(y), flags,
                                      _stream_ptr(stream)), handle)


def moe_attn_reset(handle: AttnHandle):
    _attn_check(_lib.moe_attn_reset(handle.ptr), handle)


def moe_decode_step(attn: AttnHandle, moe: Handle, x, pos: int, y, n_layers: int, stream=None):
    """One decode token through n_layers (attention, then the MoE layer)."""
    _attn_check(_lib.moe_decode_step(attn.ptr, moe.ptr, _dev_ptr(x), int(pos), _dev_ptr(y),
                                     n_layers, _stream_ptr(stream)), attn)
