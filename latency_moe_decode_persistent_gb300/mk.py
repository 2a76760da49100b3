"""ctypes binding of the C ABI in include/mk.h (argument marshalling only).

Every entry point keeps the C name.  Pointers are passed as integers (device or
host addresses); PyTorch tensors are accepted where a pointer is expected and
their ``data_ptr()`` is used.  All compute happens in ``libmk.so``: importing
this module never falls back to anything else, and calling an entry point
raises if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

MK_OK, MK_ERR_INVALID, MK_ERR_UNSUPPORTED, MK_ERR_NOMEM = 0, -1, -2, -3
MK_ERR_TIMEOUT, MK_ERR_CUDA, MK_ERR_BAD_STATE, MK_ERR_BAD_INPUT, MK_ERR_RANGE = -4, -5, -6, -7, -8
MK_DT_F32, MK_DT_BF16, MK_DT_FP8E4M3_B128, MK_DT_MXFP4_B32, MK_DT_FP8E4M3 = 0, 1, 2, 3, 4
MK_DESC_VERSION = 3

#: every symbol include/mk.h declares
EXPORTS = ["mk_create", "mk_decode_step", "mk_decode_step_sample", "mk_decode_batch", "mk_decode_step_host",
           "mk_layer_forward", "mk_get_status", "mk_get_stats", "mk_debug_skip_barrier", "mk_set_routing_trace",
           "mk_set_stage_trace", "mk_reset", "mk_layer_forward_noalloc", "mk_destroy", "mk_status_string",
           "mk_last_error"]

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class mk_model_desc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_int), ("n_layers", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("n_shared", ctypes.c_int),
                ("expert_inter", ctypes.c_int), ("vocab", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_T", ctypes.c_int),
                ("max_pages_per_stream", ctypes.c_int), ("weight_dtype", ctypes.c_int),
                ("router_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
                ("timeout_ms", ctypes.c_int), ("expert_dtype", ctypes.c_int),
                ("lm_head_dtype", ctypes.c_int)]


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in (
        "attn_norm", "w_qkv", "w_qkv_scale", "w_o", "w_o_scale", "moe_norm", "w_router",
        "router_bias", "w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale", "ws1", "ws1_scale",
        "ws3", "ws3_scale", "ws2", "ws2_scale")]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp),
                ("layers", ctypes.POINTER(mk_layer_weights)), ("lm_head_scale", _vp)]


class mk_kv_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.POINTER(_vp)), ("v_pool", ctypes.POINTER(_vp)),
                ("page_table", _vp), ("n_pages", ctypes.c_int),
                ("k_scale", ctypes.POINTER(ctypes.c_float)), ("v_scale", ctypes.POINTER(ctypes.c_float))]


class mk_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("accepted_sum", ctypes.c_uint64),
                ("distinct_experts_sum", ctypes.c_uint64), ("last_accepted", _i32),
                ("last_distinct_experts", _i32), ("fused", _i32), ("grid_ctas", _i32),
                ("launches_per_step", _i32), ("barriers_per_step", _i32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmk.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libmk.so not found at %s: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    S = ctypes.c_int
    L.mk_create.argtypes = [ctypes.POINTER(mk_model_desc), ctypes.POINTER(mk_weights),
                            ctypes.POINTER(_vp)]
    L.mk_create.restype = S
    L.mk_decode_step.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.POINTER(mk_kv_cache), _vp,
                                 _vp, _vp, _vp]
    L.mk_decode_step.restype = S
    L.mk_decode_step_sample.argtypes = [_vp, _vp, ctypes.c_int, _vp, ctypes.POINTER(mk_kv_cache),
                                        ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
    L.mk_decode_step_sample.restype = S
    L.mk_decode_batch.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                  ctypes.POINTER(mk_kv_cache), _vp, _vp, _vp, _vp]
    L.mk_decode_batch.restype = S
    L.mk_decode_step_host.argtypes = L.mk_decode_step.argtypes
    L.mk_decode_step_host.restype = S
    L.mk_layer_forward.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                   ctypes.POINTER(mk_kv_cache), _vp, _vp, _vp, _vp]
    L.mk_layer_forward.restype = S
    L.mk_layer_forward_noalloc.argtypes = [ctypes.POINTER(mk_model_desc),
                                           ctypes.POINTER(mk_layer_weights), _vp, _vp, _vp,
                                           ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                           _vp, _vp, _vp, _vp]
    L.mk_layer_forward_noalloc.restype = S
    L.mk_set_routing_trace.argtypes = [_vp, _vp, _vp]
    L.mk_set_routing_trace.restype = S
    L.mk_set_stage_trace.argtypes = [_vp, _vp, ctypes.c_int, _vp]
    L.mk_set_stage_trace.restype = S
    L.mk_debug_skip_barrier.argtypes = [_vp, ctypes.c_int]
    L.mk_debug_skip_barrier.restype = S
    L.mk_get_status.argtypes = [_vp]
    L.mk_get_status.restype = S
    L.mk_get_stats.argtypes = [_vp, ctypes.POINTER(mk_stats)]
    L.mk_get_stats.restype = S
    L.mk_reset.argtypes = [_vp]
    L.mk_reset.restype = S
    L.mk_destroy.argtypes = [_vp]
    L.mk_destroy.restype = None
    L.mk_status_string.argtypes = [S]
    L.mk_status_string.restype = ctypes.c_char_p
    L.mk_last_error.argtypes = [_vp]
    L.mk_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


class MKError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s (%d): %s" % (mk_status_string(status), status, msg))
        self.status = status


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(st, status):
    if status != MK_OK:
        raise MKError(status, mk_last_error(st))
    return status


# ---------------------------------------------------------------- entry points
def mk_status_string(s: int) -> str:
    return lib().mk_status_string(s).decode()


def mk_last_error(st) -> str:
    r = lib().mk_last_error(st)
    return r.decode() if r else ""


def mk_create(desc: mk_model_desc, weights: mk_weights) -> int:
    h = _vp()
    s = lib().mk_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h))
    _check(None, s)
    return h.value


def mk_decode_step(st, draft_tokens, T, positions, kv: mk_kv_cache, out_logits, out_accepted,
                   out_argmax=None, stream=None, check=True) -> int:
    s = lib().mk_decode_step(st, _ptr(draft_tokens), T, _ptr(positions), ctypes.byref(kv),
                             _ptr(out_logits), _ptr(out_accepted), _ptr(out_argmax), _ptr(stream))
    return _check(st, s) if check else s


def mk_decode_step_sample(st, draft_tokens, T, positions, kv: mk_kv_cache, temperature, uniforms,
                          out_logits, out_accepted, out_token, stream=None, check=True) -> int:
    s = lib().mk_decode_step_sample(st, _ptr(draft_tokens), T, _ptr(positions), ctypes.byref(kv),
                                    float(temperature), _ptr(uniforms), _ptr(out_logits),
                                    _ptr(out_accepted), _ptr(out_token), _ptr(stream))
    return _check(st, s) if check else s


def mk_debug_skip_barrier(st, barrier: int) -> int:
    return lib().mk_debug_skip_barrier(st, barrier)


def mk_decode_batch(st, n_streams, draft_tokens, T, positions, kv: mk_kv_cache, out_logits,
                    out_accepted, out_argmax=None, stream=None, check=True) -> int:
    s = lib().mk_decode_batch(st, n_streams, _ptr(draft_tokens), T, _ptr(positions),
                              ctypes.byref(kv), _ptr(out_logits), _ptr(out_accepted),
                              _ptr(out_argmax), _ptr(stream))
    return _check(st, s) if check else s


def mk_decode_step_host(st, h_tokens, T, h_positions, kv: mk_kv_cache, h_logits, h_accepted,
                        h_argmax=None, stream=None, check=True) -> int:
    s = lib().mk_decode_step_host(st, _ptr(h_tokens), T, _ptr(h_positions), ctypes.byref(kv),
                                  _ptr(h_logits), _ptr(h_accepted), _ptr(h_argmax), _ptr(stream))
    return _check(st, s) if check else s


def mk_layer_forward(st, layer, hidden_in, T, positions, kv: mk_kv_cache, hidden_out,
                     out_topk_idx=None, out_topk_w=None, stream=None, check=True) -> int:
    s = lib().mk_layer_forward(st, layer, _ptr(hidden_in), T, _ptr(positions), ctypes.byref(kv),
                               _ptr(hidden_out), _ptr(out_topk_idx), _ptr(out_topk_w),
                               _ptr(stream))
    return _check(st, s) if check else s


def mk_layer_forward_noalloc(desc: mk_model_desc, lw: mk_layer_weights, k_pool, v_pool, page_table,
                             n_pages, hidden_in, T, ctx, positions, hidden_out, out_topk_idx=None,
                             out_topk_w=None, out_status=None, stream=None, check=True) -> int:
    s = lib().mk_layer_forward_noalloc(ctypes.byref(desc), ctypes.byref(lw), _ptr(k_pool),
                                       _ptr(v_pool), _ptr(page_table), n_pages, _ptr(hidden_in), T,
                                       ctx, _ptr(positions), _ptr(hidden_out), _ptr(out_topk_idx),
                                       _ptr(out_topk_w), _ptr(out_status), _ptr(stream))
    return _check(None, s) if check else s


def mk_set_routing_trace(st, idx_trace, w_trace=None) -> int:
    return _check(st, lib().mk_set_routing_trace(st, _ptr(idx_trace), _ptr(w_trace)))


def mk_set_stage_trace(st, times, capacity=0, events=None) -> int:
    return _check(st, lib().mk_set_stage_trace(st, _ptr(times), capacity, _ptr(events)))


def mk_get_status(st) -> int:
    return lib().mk_get_status(st)


def mk_get_stats(st) -> mk_stats:
    out = mk_stats()
    _check(st, lib().mk_get_stats(st, ctypes.byref(out)))
    return out


def mk_reset(st) -> int:
    return _check(st, lib().mk_reset(st))


def mk_destroy(st) -> None:
    if st:
        lib().mk_destroy(st)


# ---------------------------------------------------------------- marshalling helpers
class ModelArgs:
    """ctypes structs for a model whose tensors live on the device.

    ``model`` needs ``cfg`` (dimensions and dtypes), ``layers`` (each with
    attn_norm, w_qkv, w_o, moe_norm, w_router, router_bias, w1, w3, w2, ws1, ws3,
    ws2; matrices as objects with ``data`` and ``scale`` tensors) and, for a
    stack with an LM head, ``embed``, ``final_norm`` and ``lm_head``.  The
    object keeps the structs alive for as long as the state uses them.
    """

    def __init__(self, model, max_T: int, max_pages: int, timeout_ms: int = 0):
        cfg = model.cfg
        self.desc = mk_model_desc(
            MK_DESC_VERSION, cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads,
            cfg.head_dim, cfg.rope_base, cfg.rms_eps, cfg.n_experts, cfg.top_k, cfg.n_shared,
            cfg.expert_inter, cfg.vocab, cfg.page_size, max_T, max_pages, cfg.weight_dtype,
            cfg.router_dtype, MK_DT_FP8E4M3 if cfg.kv_dtype == MK_DT_FP8E4M3_B128 else cfg.kv_dtype,
            timeout_ms,
            getattr(cfg, "routed_dtype", cfg.weight_dtype), getattr(cfg, "lm_dtype", MK_DT_BF16))
        n = cfg.n_layers
        self.layers = (mk_layer_weights * n)()
        for i, L in enumerate(model.layers):
            lw = self.layers[i]

            def mat(name, m):
                setattr(lw, name, _ptr(m.data) if m is not None else 0)
                setattr(lw, name + "_scale", _ptr(m.scale) if m is not None else 0)
            lw.attn_norm = _ptr(L.attn_norm)
            lw.moe_norm = _ptr(L.moe_norm)
            lw.router_bias = _ptr(L.router_bias)
            lw.w_router = _ptr(L.w_router.data)
            mat("w_qkv", L.w_qkv)
            mat("w_o", L.w_o)
            mat("w1", L.w1)
            mat("w3", L.w3)
            mat("w2", L.w2)
            mat("ws1", L.ws1)
            mat("ws3", L.ws3)
            mat("ws2", L.ws2)
        self.weights = mk_weights(_ptr(getattr(model, "embed", None)),
                                  _ptr(getattr(model, "final_norm", None)),
                                  _ptr(getattr(model, "lm_head", None)), self.layers,
                                  _ptr(getattr(model, "lm_head_scale", None)))


class KVArgs:
    """mk_kv_cache for pools and a page table held as device tensors."""

    def __init__(self, k_pools: Sequence, v_pools: Sequence, page_table, n_pages: int,
                 scales: Optional[Sequence] = None):
        n = len(k_pools)
        self._k = (_vp * n)(*[_ptr(t) for t in k_pools])
        self._v = (_vp * n)(*[_ptr(t) for t in v_pools])
        self.page_table = page_table
        ks = vs = None
        if scales is not None:
            self._ks = (ctypes.c_float * n)(*[float(a) for a, _ in scales])
            self._vs = (ctypes.c_float * n)(*[float(b) for _, b in scales])
            ks = ctypes.cast(self._ks, ctypes.POINTER(ctypes.c_float))
            vs = ctypes.cast(self._vs, ctypes.POINTER(ctypes.c_float))
        self.kv = mk_kv_cache(ctypes.cast(self._k, ctypes.POINTER(_vp)),
                              ctypes.cast(self._v, ctypes.POINTER(_vp)), _ptr(page_table), n_pages,
                              ks, vs)
