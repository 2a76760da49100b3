"""Seeded synthetic inputs for the verify-step workloads.

This module only draws random numbers and encodes them in the stored weight
formats (bf16 bits, FP8 E4M3 bytes with 1x128 fp32 block scales, fp32).  It holds
none of the method's arithmetic; both the CUDA path (through the C-ABI) and the
fp64 oracle consume what it makes, which is why it sits in a module of its own.

Recipes (the workloads of the single-stream decode study, with synthetic values
standing in for the real checkpoint and prompts):
  * matrices            N(0, 1/fan_in)
  * RMSNorm weights     1 (``gamma_jitter`` > 0 gives 1 + jitter*U(-1,1))
  * router bias         U(-0.1, 0.1) (0 for the tiny fp32 layer)
  * cached K/V entries  N(0, 1), stored in the cache dtype
  * embedding rows      N(0, 1) (bf16); LM head N(0, 1/H) (bf16, or FP8 1x128 as the matrices)
  * page table          a seeded permutation of physical pages
  * FP8 weights         per 1x128 block: scale = amax/448, code = RNE(w/scale)
  * MXFP4 expert weights per 1x32 block: E8M0 scale 2^(floor(log2 amax) - 2),
                        E2M1 code = RNE(w/scale) saturated at +-6, two codes per
                        byte (element 2j in the low nibble)
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

WDT_F32, WDT_BF16, WDT_FP8, WDT_MXFP4 = 0, 1, 2, 3
_KIND = {WDT_F32: "f32", WDT_BF16: "bf16", WDT_FP8: "fp8", WDT_MXFP4: "mxfp4"}


@dataclass
class Config:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    expert_inter: int
    n_layers: int = 1
    vocab: int = 0                 # 0: single-layer workload (no embedding / LM head)
    page_size: int = 64
    weight_dtype: int = WDT_FP8
    router_dtype: int = WDT_BF16
    kv_dtype: int = WDT_BF16
    n_shared: int = 1
    T: int = 6
    ctx: int = 2048
    seed: int = 0
    bias_range: float = 0.1
    rms_eps: float = 1e-6
    rope_base: float = 10000.0
    gamma_jitter: float = 0.0
    expert_dtype: int = -1         # routed-expert storage; -1: the same as weight_dtype
    lm_dtype: int = WDT_BF16       # LM head storage: bf16 or FP8 (1x128 scales)
    kv_scales: tuple = (1.0, 1.0)  # FP8 KV cache: (K, V) scale of every layer (value = code * scale),
                                   # or a list of per-layer (K, V) pairs

    @property
    def qkv_rows(self):
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def routed_dtype(self):
        return self.weight_dtype if self.expert_dtype < 0 else self.expert_dtype


def tiny_config(**kw) -> Config:
    """Tiny fp32 MoE layer: H 512, 8/2 heads of 64, 16 experts top-2 + shared, I 256,
    ctx 128 fp32, T 1, seed 0, router bias 0."""
    c = Config("tiny_fp32_layer", 512, 8, 2, 64, 16, 2, 256, weight_dtype=WDT_F32,
               router_dtype=WDT_F32, kv_dtype=WDT_F32, T=1, ctx=128, seed=0, bias_range=0.0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def bf16_layer_config(**kw) -> Config:
    """One full-width MoE layer with bf16 weights, T 6, ctx 2048 bf16, seed 1."""
    c = Config("bf16_layer", 4096, 32, 4, 128, 384, 8, 512, weight_dtype=WDT_BF16,
               router_dtype=WDT_BF16, kv_dtype=WDT_BF16, T=6, ctx=2048, seed=1)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def fp8_layer_config(**kw) -> Config:
    """Same layer with FP8 E4M3 expert/attention weights (1x128 fp32 scales),
    bf16 router, T 8, ctx 65536, seed 2."""
    c = Config("fp8_layer_ctx64k", 4096, 32, 4, 128, 384, 8, 512, weight_dtype=WDT_FP8,
               router_dtype=WDT_BF16, kv_dtype=WDT_BF16, T=8, ctx=65536, seed=2)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def stack_config(**kw) -> Config:
    """43 FP8 layers + bf16 embedding / LM head over vocab 129280, T 6, ctx 2048, seed 3."""
    c = Config("fp8_stack_43L", 4096, 32, 4, 128, 384, 8, 512, n_layers=43, vocab=129280,
               weight_dtype=WDT_FP8, router_dtype=WDT_BF16, kv_dtype=WDT_BF16, T=6,
               ctx=2048, seed=3)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


# ---------------------------------------------------------------------------
# deterministic generators
# ---------------------------------------------------------------------------

def _seed_of(seed: int, *names) -> int:
    h = hashlib.sha256(("%d|" % seed + "|".join(str(n) for n in names)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed, *names) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed_of(seed, *names))
    return g


def randn(shape, std, device, seed, *names, dtype=torch.float32):
    g = _gen(device, seed, *names)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, lo, hi, device, seed, *names):
    g = _gen(device, seed, *names)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def quantize_fp8_blocks(w: torch.Tensor):
    """Encode w[..., N, K] (fp32) as FP8 E4M3 codes with 1x128 block scales.

    Returns (codes uint8 [..., N, K], scale fp32 [..., K/128, N]); the decoded
    weight is fp8(code[n][k]) * scale[k//128][n].
    """
    *lead, N, K = w.shape
    assert K % 128 == 0
    blocks = w.reshape(*lead, N, K // 128, 128)
    amax = blocks.abs().amax(dim=-1).clamp_min(1e-30)
    scale = (amax / 448.0).to(torch.float32)
    q = (blocks / scale.unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(*lead, N, K)
    return codes, scale.transpose(-1, -2).contiguous()


# E2M1 rounding: the midpoints between the representable magnitudes
# 0, 0.5, 1, 1.5, 2, 3, 4, 6; a magnitude exactly at a midpoint takes the code
# with an even mantissa bit (the upper one at 0.75, 1.75 and 3.5)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_E2M1_TIE_UP = (0.75, 1.75, 3.5)


def quantize_mxfp4_blocks(w: torch.Tensor):
    """Encode w[..., N, K] (fp32) as MXFP4: per 32 consecutive inputs one E8M0
    scale 2^X with X = floor(log2(amax)) - 2 (so the block's largest magnitude
    lands in [4, 8) before rounding), elements rounded to E2M1 (nearest, ties
    to even, saturating at 6).  Returns (packed uint8 [..., N, K/2] with element
    2j in the low nibble of byte j, scale codes uint8 [..., K/32, N])."""
    *lead, N, K = w.shape
    assert K % 32 == 0
    blocks = w.reshape(*lead, N, K // 32, 32).to(torch.float64)
    amax = blocks.abs().amax(dim=-1)
    x = torch.where(amax > 0, torch.floor(torch.log2(amax.clamp_min(1e-300))) - 2, torch.full_like(amax, -127))
    x = x.clamp(-127, 127)
    v = blocks / torch.exp2(x).unsqueeze(-1)
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.int64)
    for m in _E2M1_MID:
        code += (a > m).to(torch.int64)
    for m in _E2M1_TIE_UP:
        code += (a == m).to(torch.int64)
    code = code.clamp(max=7) + 8 * (v < 0).to(torch.int64)
    code = code.reshape(*lead, N, K).to(torch.uint8)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    scale = (x + 127).to(torch.uint8).transpose(-1, -2).contiguous()
    return packed.contiguous(), scale


@dataclass
class Mat:
    """A stored matrix: ``data`` in the weight dtype (fp32 / bf16 / uint8 FP8 codes),
    ``scale`` fp32 [.., in/128, out] for FP8, else None."""
    dtype: int
    data: torch.Tensor
    scale: Optional[torch.Tensor] = None


def make_matrix(shape, fan_in, wdt, device, seed, *names, chunk=32) -> Mat:
    """Draw N(0, 1/fan_in) weights of ``shape`` ([N][K] or [E][N][K]) and encode them."""
    std = fan_in ** -0.5
    if len(shape) == 2:
        lead, parts = (), [None]
    else:
        lead, parts = (shape[0],), list(range(0, shape[0], chunk))
    if wdt == WDT_F32:
        if not lead:
            return Mat(wdt, randn(shape, std, device, seed, *names))
        out = torch.empty(shape, dtype=torch.float32, device=device)
        for p in parts:
            e1 = min(shape[0], p + chunk)
            out[p:e1] = randn((e1 - p,) + tuple(shape[1:]), std, device, seed, *names, p)
        return Mat(wdt, out)
    if wdt == WDT_BF16:
        if not lead:
            return Mat(wdt, randn(shape, std, device, seed, *names, dtype=torch.bfloat16))
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for p in parts:
            e1 = min(shape[0], p + chunk)
            out[p:e1] = randn((e1 - p,) + tuple(shape[1:]), std, device, seed, *names, p,
                              dtype=torch.bfloat16)
        return Mat(wdt, out)
    if wdt == WDT_MXFP4:
        quant = quantize_mxfp4_blocks
    else:
        quant = quantize_fp8_blocks
    if not lead:
        q, s = quant(randn(shape, std, device, seed, *names))
        return Mat(wdt, q, s)
    E, N, K = shape
    if wdt == WDT_MXFP4:
        q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
        s = torch.empty((E, K // 32, N), dtype=torch.uint8, device=device)
    else:
        q = torch.empty(shape, dtype=torch.uint8, device=device)
        s = torch.empty((E, K // 128, N), dtype=torch.float32, device=device)
    for p in parts:
        e1 = min(E, p + chunk)
        qq, ss = quant(randn((e1 - p, N, K), std, device, seed, *names, p))
        q[p:e1] = qq
        s[p:e1] = ss
        del qq, ss
    return Mat(wdt, q, s)


@dataclass
class Layer:
    attn_norm: torch.Tensor
    w_qkv: Mat
    w_o: Mat
    moe_norm: torch.Tensor
    w_router: Mat
    router_bias: torch.Tensor
    w1: Mat
    w3: Mat
    w2: Mat
    ws1: Optional[Mat] = None
    ws3: Optional[Mat] = None
    ws2: Optional[Mat] = None


@dataclass
class Model:
    cfg: Config
    layers: List[Layer]
    embed: Optional[torch.Tensor] = None      # bf16 [V][H]
    final_norm: Optional[torch.Tensor] = None
    lm_head: Optional[torch.Tensor] = None    # bf16 [V][H], or uint8 FP8 codes
    lm_head_scale: Optional[torch.Tensor] = None  # FP8 LM head: fp32 [H/128][V]


def _gamma(cfg, device, *names):
    if cfg.gamma_jitter > 0:
        return 1.0 + uniform((cfg.hidden,), -cfg.gamma_jitter, cfg.gamma_jitter, device,
                             cfg.seed, *names)
    return torch.ones(cfg.hidden, dtype=torch.float32, device=device)


def make_layer(cfg: Config, l: int, device) -> Layer:
    H, I, E, d = cfg.hidden, cfg.expert_inter, cfg.n_experts, cfg.head_dim
    wd, s = cfg.weight_dtype, cfg.seed
    lay = Layer(
        attn_norm=_gamma(cfg, device, l, "attn_norm"),
        w_qkv=make_matrix((cfg.qkv_rows, H), H, wd, device, s, l, "w_qkv"),
        w_o=make_matrix((H, cfg.n_q_heads * d), cfg.n_q_heads * d, wd, device, s, l, "w_o"),
        moe_norm=_gamma(cfg, device, l, "moe_norm"),
        w_router=make_matrix((E, H), H, cfg.router_dtype, device, s, l, "w_router"),
        router_bias=(uniform((E,), -cfg.bias_range, cfg.bias_range, device, s, l, "bias")
                     if cfg.bias_range > 0 else torch.zeros(E, device=device)),
        w1=make_matrix((E, I, H), H, cfg.routed_dtype, device, s, l, "w1"),
        w3=make_matrix((E, I, H), H, cfg.routed_dtype, device, s, l, "w3"),
        w2=make_matrix((E, H, I), I, cfg.routed_dtype, device, s, l, "w2"),
    )
    if cfg.n_shared:
        lay.ws1 = make_matrix((I, H), H, wd, device, s, l, "ws1")
        lay.ws3 = make_matrix((I, H), H, wd, device, s, l, "ws3")
        lay.ws2 = make_matrix((H, I), I, wd, device, s, l, "ws2")
    return lay


def make_model(cfg: Config, device) -> Model:
    layers = [make_layer(cfg, l, device) for l in range(cfg.n_layers)]
    m = Model(cfg, layers)
    if cfg.vocab:
        m.embed = randn((cfg.vocab, cfg.hidden), 1.0, device, cfg.seed, "embed",
                        dtype=torch.bfloat16)
        m.final_norm = _gamma(cfg, device, "final_norm")
        if cfg.lm_dtype == WDT_FP8:
            m.lm_head, m.lm_head_scale = quantize_fp8_blocks(
                randn((cfg.vocab, cfg.hidden), cfg.hidden ** -0.5, device, cfg.seed, "lm_head"))
        else:
            m.lm_head = randn((cfg.vocab, cfg.hidden), cfg.hidden ** -0.5, device, cfg.seed,
                              "lm_head", dtype=torch.bfloat16)
    return m


# ---------------------------------------------------------------------------
# KV cache
# ---------------------------------------------------------------------------

@dataclass
class KVCache:
    """Per layer K and V pools [n_pages][Hkv][P][d] plus page tables
    [n_streams][max_pages]; ``ctx[s]`` cached positions per stream.  An FP8
    cache holds uint8 E4M3 codes and ``scales[l]`` = (K scale, V scale)."""
    k_pools: List[torch.Tensor]
    v_pools: List[torch.Tensor]
    page_table: torch.Tensor
    ctx: List[int]
    page_size: int
    max_pages: int
    scales: Optional[List[tuple]] = None

    @property
    def n_pages(self):
        return self.k_pools[0].shape[0]


def make_kv(cfg: Config, device, ctxs=None, T=None, extra_pages=0, seed_tag="kv") -> KVCache:
    """Paged K/V cache holding ``ctxs[s]`` N(0,1) entries per stream, with room for
    T more positions; physical pages are a seeded permutation."""
    ctxs = [cfg.ctx] if ctxs is None else list(ctxs)
    T = cfg.T if T is None else T
    P = cfg.page_size
    need = [(c + T + P - 1) // P for c in ctxs]
    max_pages = max(need)
    n_pages = sum(need) + extra_pages
    perm = torch.randperm(n_pages, generator=_gen("cpu", cfg.seed, seed_tag, "perm"))
    pt = torch.full((len(ctxs), max_pages), -1, dtype=torch.int32)
    o = 0
    for s_, n in enumerate(need):
        pt[s_, :n] = perm[o:o + n].to(torch.int32)
        o += n
    shape = (n_pages, cfg.n_kv_heads, P, cfg.head_dim)
    kp, vp = [], []
    if cfg.kv_dtype == WDT_FP8:
        # N(0,1) entries stored as E4M3 codes of value / scale (saturating)
        per = cfg.kv_scales
        scales = ([tuple(map(float, per[l])) for l in range(cfg.n_layers)]
                  if isinstance(per[0], (tuple, list)) else [tuple(map(float, per))] * cfg.n_layers)
        for l in range(cfg.n_layers):
            ks, vs = scales[l]
            for pools, tag, sc in ((kp, "k", ks), (vp, "v", vs)):
                x = randn(shape, 1.0, device, cfg.seed, seed_tag, l, tag) / sc
                pools.append(x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
        return KVCache(kp, vp, pt.to(device), ctxs, P, max_pages, scales)
    kvt = torch.float32 if cfg.kv_dtype == WDT_F32 else torch.bfloat16
    for l in range(cfg.n_layers):
        kp.append(randn(shape, 1.0, device, cfg.seed, seed_tag, l, "k", dtype=kvt))
        vp.append(randn(shape, 1.0, device, cfg.seed, seed_tag, l, "v", dtype=kvt))
    return KVCache(kp, vp, pt.to(device), ctxs, P, max_pages)


# ---------------------------------------------------------------------------
# numpy views for the oracle (data movement only)
# ---------------------------------------------------------------------------

def _np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    return t.cpu().numpy().copy()


def oracle_linear(m: Mat, e: Optional[int] = None):
    """The matrix (or expert e of it) as an ``oracle.Linear``-shaped tuple
    (kind, q, scale) of host numpy arrays."""
    data = m.data if e is None else m.data[e]
    sc = None
    if m.scale is not None:
        sc = _np(m.scale if e is None else m.scale[e])
    return _KIND[m.dtype], _np(data), sc


def oracle_kv(kv: KVCache, l: int, stream: int = 0):
    """Raw host copies for the oracle: (kind, k_pool, v_pool, page_table_row, ctx).

    Pools are the stored bits ([n_pages][Hkv][P][d], float32 or uint16 bf16
    bits); the oracle decodes them and follows the page table itself.
    """
    dt = kv.k_pools[l].dtype
    kind = "f32" if dt == torch.float32 else "fp8" if dt == torch.uint8 else "bf16"
    return (kind, _np(kv.k_pools[l]), _np(kv.v_pools[l]),
            kv.page_table[stream].cpu().numpy().astype(np.int64), kv.ctx[stream])
