"""Glue between the seeded generators and the oracle (data movement only)."""
import numpy as np

import oracle
from latency_moe_decode_persistent_gb300 import synth


def oracle_dims(cfg: synth.Config) -> oracle.Dims:
    kvk = {synth.WDT_F32: "f32", synth.WDT_BF16: "bf16", synth.WDT_FP8: "fp8"}[cfg.kv_dtype]
    return oracle.Dims(cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_experts,
                       cfg.top_k, cfg.expert_inter, cfg.rms_eps, cfg.rope_base, kvk)


def lin(m, e=None):
    kind, q, s = synth.oracle_linear(m, e)
    return oracle.Linear(kind, q, s)


def layer_view(model: synth.Model, l: int, expert_cache=None) -> oracle.LayerView:
    L = model.layers[l]
    cache = {} if expert_cache is None else expert_cache

    def expert(e):
        key = (l, e)
        if key not in cache:
            cache[key] = (lin(L.w1, e), lin(L.w3, e), lin(L.w2, e))
        return cache[key]

    shared = None
    if L.ws1 is not None:
        shared = (lin(L.ws1), lin(L.ws3), lin(L.ws2))
    return oracle.LayerView(
        attn_norm=L.attn_norm.cpu().numpy().astype(np.float64),
        w_qkv=lin(L.w_qkv), w_o=lin(L.w_o),
        moe_norm=L.moe_norm.cpu().numpy().astype(np.float64),
        w_router=lin(L.w_router),
        router_bias=L.router_bias.cpu().numpy().astype(np.float64),
        expert=expert, shared=shared)


def kv_view(kv: synth.KVCache, l: int, stream: int = 0):
    kind, kp, vp, pt, ctx = synth.oracle_kv(kv, l, stream)
    return oracle.kv_from_pool(kind, kp, vp, pt, ctx, kv.scales[l] if kv.scales else (1.0, 1.0))


def kv_scales(kv: synth.KVCache):
    """Per-layer (K, V) scales for the oracle's stack or layer calls."""
    return kv.scales if kv.scales else [(1.0, 1.0)] * len(kv.k_pools)


def embed_fn(model):
    def f(tok):
        rows = model.embed[np.asarray(tok, dtype=np.int64)]
        return oracle.bf16_decode(synth._np(rows))
    return f


def lm_head_lin(model):
    if model.lm_head_scale is not None:
        return oracle.Linear("fp8", synth._np(model.lm_head), synth._np(model.lm_head_scale))
    return oracle.Linear("bf16", synth._np(model.lm_head))


def rel_err(a, b):
    """max |a - b| / RMS(b)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / np.sqrt(np.mean(b * b)))
