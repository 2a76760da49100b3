"""Plain fp64 CPU oracle for one speculative-verify decode step of a MoE stack.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
call it.  It shares no code with the CUDA path (``latency_moe_decode_persistent_gb300``)
and never imports it; its only inputs are the arrays the seeded generators make.

What is computed, and where it comes from.
The pages ("DeepSeek-V4.1-Flash breaks 1,000 tokens per second for one user",
ezolabs; "Why one GB300 doesn't beat 4x RTX PRO 6000 at single-stream decode",
al-engr) fix the *problem*: one verify step checks a block of drafted tokens
(block verification, ezolabs "How we got here" and "Serving stack"), tokens per
second = tokens per verify step x verify steps per second (al-engr "The
decomposition"), and the step is a 43-layer, 384-expert MoE stack ending in an
lm_head and an accept kernel (al-engr "Where the 11.2 ms goes", kernel table).
They never print the layer equations.  The layer math below is the plainest
reading of the workload description that goes with them: pre-norm residual
blocks, GQA attention with rotate-half RoPE over a paged KV cache, a sigmoid
router whose bias only steers selection, top-K with weights normalised to 1,
SwiGLU experts plus one shared expert, RMSNorm + LM head + greedy argmax, and
the longest-accepted-prefix rule.  Each of these readings is the plainest one
the pages and the workload description support; none is printed on the pages.

Arithmetic: every floating-point value is widened to fp64 and computed in fp64.
The only deliberate roundings are the ones the method itself performs: the new
K/V entries are stored in the cache dtype (bf16 or fp32) before attention reads
them back.

Parity status of each function is stated in its docstring; the pins live in
``tests/test_oracle_pins.py``.  ``stack_forward`` composes pinned parts; the
pages print no worked example for this model, so it is pinned through special
cases: with every O and down projection zero the stack reduces to final RMSNorm
+ LM head on the embeddings (checked against torch), an appended identity layer
changes nothing, and block verification equals sequential decode.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np

__all__ = [
    "FP8_E4M3_TABLE", "fp8_e4m3_decode", "bf16_decode", "round_to_bf16", "round_to_f32",
    "E2M1_TABLE", "e2m1_unpack", "e8m0_decode", "round_to_e4m3",
    "Linear", "dequant", "linear", "rmsnorm", "rope", "sigmoid", "silu",
    "attention_gqa", "route", "swiglu", "LayerView", "layer_forward", "stack_forward",
    "accept_count", "tokens_per_second", "step_seconds_from", "argmax_lowest",
    "softmax_t", "sample_index", "sample_verify",
]


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def _e4m3fn_value(code: int) -> float:
    """Value of one OCP FP8 E4M3 ("fn": finite, NaN only) byte.

    Format definition (OCP 8-bit floating point specification, E4M3): 1 sign bit,
    4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
    (value = m/8 * 2^-6); S.1111.111 is NaN; there is no infinity, so exponent
    field 15 with mantissa 0..6 is an ordinary normal number (max 448).
    """
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        v = (m / 8.0) * 2.0 ** (-6)
    else:
        v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


#: fp64 value of every FP8 E4M3 code, built from the format definition above.
FP8_E4M3_TABLE = np.array([_e4m3fn_value(c) for c in range(256)], dtype=np.float64)


def fp8_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 FP8 E4M3 codes -> fp64 values (table lookup). Pinned."""
    return FP8_E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> fp64 values.

    bfloat16 is the upper half of an IEEE binary32: widen by appending 16 zero
    bits, then reinterpret.  Pinned.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (ties to even), as fp64.

    bfloat16 keeps 8 significant bits (7 stored) and binary32's exponent range.
    Rounding is done directly from fp64 with ``np.ldexp``/``np.frexp`` so no
    double rounding through binary32 happens.  Subnormal bfloat16 results
    (|x| < 2^-126) are rounded on the 2^-133 grid.  Pinned.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])            # x = m * 2^e, 0.5 <= |m| < 1
    # significand grid: 8 bits => unit = 2^(e-8); below 2^-126 the grid is fixed
    unit_exp = np.maximum(e - 8, -133)
    scaled = np.ldexp(x[nz], -unit_exp)
    out[nz] = np.ldexp(np.round(scaled), unit_exp)   # np.round: ties to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest OCP FP8 E4M3 ("fn") value, ties to even,
    saturating at +-448 (the format has no infinity), returned as fp64.

    E4M3 keeps 4 significant bits (3 stored); normal numbers reach down to 2^-6
    and subnormals are multiples of 2^-9.  Pinned (torch's float8 cast, hand
    ties, saturation)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])
    unit_exp = np.maximum(e - 4, -9)
    out[nz] = np.ldexp(np.round(np.ldexp(x[nz], -unit_exp)), unit_exp)
    return np.clip(out, -448.0, 448.0)


def _e2m1_value(code: int) -> float:
    """Value of one FP4 E2M1 element (OCP Microscaling Formats v1.0): 1 sign bit,
    2 exponent bits with bias 1, 1 mantissa bit; exponent field 0 is subnormal
    (value m/2); there are no infinities or NaN (largest magnitude 6)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    v = m / 2.0 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -v if s else v


#: fp64 value of every FP4 E2M1 code (4 bits), from the format definition above.
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    """E8M0 scale bytes -> fp64: 2^(code - 127); 0xFF is NaN (OCP Microscaling
    Formats v1.0).  Pinned."""
    c = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, out)


def e2m1_unpack(packed: np.ndarray) -> np.ndarray:
    """uint8 bytes holding two E2M1 codes each -> fp64 element values along the
    last axis, doubled in length.  Reading of the storage layout: element 2j
    is the low nibble of byte j and element 2j+1 its high nibble.  Pinned."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.float64)
    out[..., 0::2] = E2M1_TABLE[b & 0xF]
    out[..., 1::2] = E2M1_TABLE[b >> 4]
    return out


def round_to_f32(x: np.ndarray) -> np.ndarray:
    """Round fp64 to the nearest binary32 value (ties to even), returned as fp64.

    Used for the fp32 KV cache of the all-fp32 layer.  Pinned (hand-chosen
    halfway values, normal and subnormal)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Linear layers with the weight encodings of the workload
# ---------------------------------------------------------------------------

@dataclass
class Linear:
    """A weight matrix W[out][in] in one of the stored encodings.

    kind "f32":  q is float32 [out][in].
    kind "bf16": q is uint16 bfloat16 bits [out][in].
    kind "fp8":  q is uint8 FP8 E4M3 codes [out][in]; scale is float32
                 [in/128][out]; the real weight is
                 W[n][k] = fp8(q[n][k]) * scale[k // 128][n]
                 (1 x 128 blocks along the input dimension).
    kind "mxfp4": q is uint8 [out][in/2], two FP4 E2M1 codes per byte (element
                 2j in the low nibble of byte j); scale is uint8 E8M0 [in/32][out];
                 W[n][k] = e2m1(code[n][k]) * 2^(scale[k // 32][n] - 127)
                 (MXFP4: 1 x 32 blocks along the input dimension).
    """
    kind: str
    q: np.ndarray
    scale: Optional[np.ndarray] = None

    @property
    def shape(self):
        return self.q.shape


def dequant(lin: Linear, rows: Optional[slice] = None) -> np.ndarray:
    """Exact fp64 value of W (or of a row range of it).  Pinned."""
    q = lin.q if rows is None else lin.q[rows]
    if lin.kind == "f32":
        return q.astype(np.float64)
    if lin.kind == "bf16":
        return bf16_decode(q)
    if lin.kind == "fp8":
        s = lin.scale if rows is None else lin.scale[:, rows]
        w = fp8_e4m3_decode(q)                        # [n][in]
        blk = np.repeat(s.T.astype(np.float64), 128, axis=1)   # [n][in]
        return w * blk[:, : w.shape[1]]
    if lin.kind == "mxfp4":
        s = lin.scale if rows is None else lin.scale[:, rows]
        w = e2m1_unpack(q)                            # [n][in]
        blk = np.repeat(e8m0_decode(s.T), 32, axis=1)   # [n][in]
        return w * blk[:, : w.shape[1]]
    raise ValueError(f"unknown weight kind {lin.kind}")


def linear(lin: Linear, x: np.ndarray, row_block: int = 16384) -> np.ndarray:
    """y[..., n] = sum_k W[n][k] x[..., k] in fp64 (W dequantised exactly).

    Rows are dequantised in blocks only to bound memory; each output is the
    plain dot product of one dequantised row with x.  Pinned.
    """
    x = np.asarray(x, dtype=np.float64)
    n_out = lin.q.shape[0]
    out = np.empty(x.shape[:-1] + (n_out,), dtype=np.float64)
    for r0 in range(0, n_out, row_block):
        r1 = min(n_out, r0 + row_block)
        w = dequant(lin, slice(r0, r1))
        out[..., r0:r1] = x @ w.T
    return out


# ---------------------------------------------------------------------------
# Elementwise pieces
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma.  Pinned."""
    x = np.asarray(x, dtype=np.float64)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / r * np.asarray(gamma, dtype=np.float64)


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half rotary embedding over the whole head dimension.

    x[..., d] at integer positions pos (broadcast over the leading axes of x
    except the head axis): for i < d/2 the pair (x_i, x_{i+d/2}) is rotated by
    the angle pos * base^(-2i/d).  Pinned (identity at 0, norm, relative-position
    property, 2-D closed form).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv      # [..., half]
    while ang.ndim < x.ndim:
        ang = ang[..., None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def sigmoid(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x: np.ndarray) -> np.ndarray:
    """silu(a) = a * sigmoid(a).  Pinned."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def argmax_lowest(v: np.ndarray) -> np.ndarray:
    """Argmax over the last axis; equal maxima resolve to the lowest index
    (np.argmax returns the first occurrence)."""
    return np.argmax(np.asarray(v), axis=-1)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def attention_gqa(q: np.ndarray, k_ctx: np.ndarray, v_ctx: np.ndarray,
                  k_new: np.ndarray, v_new: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention of a verify block over cache + block.

    q      [T][Hq][d]     queries of the block (already rotated)
    k_ctx  [Hkv][ctx][d]  cached keys at positions 0..ctx-1 (already rotated)
    v_ctx  [Hkv][ctx][d]
    k_new  [T][Hkv][d]    keys of the block, as stored in the cache
    v_new  [T][Hkv][d]
    Query t of head h sees every cached key and block keys 0..t; its KV head is
    g = floor(h * Hkv / Hq); scores are scaled by 1/sqrt(d).  Returns o[T][Hq][d].
    Pinned (one key, equal keys, causality, split-merge, brute force).
    """
    T, Hq, d = q.shape
    Hkv = k_new.shape[1]
    ctx = k_ctx.shape[1]
    scale = 1.0 / math.sqrt(d)
    o = np.zeros((T, Hq, d), dtype=np.float64)
    for h in range(Hq):
        g = (h * Hkv) // Hq
        kc, vc = k_ctx[g], v_ctx[g]                      # [ctx][d]
        for t in range(T):
            keys = np.concatenate([kc, k_new[: t + 1, g, :]], axis=0)
            vals = np.concatenate([vc, v_new[: t + 1, g, :]], axis=0)
            s = keys @ q[t, h] * scale
            m = s.max()
            p = np.exp(s - m)
            o[t, h] = (p @ vals) / p.sum()
    return o


def gather_paged(pool: np.ndarray, page_table: np.ndarray, ctx: int) -> np.ndarray:
    """Positions 0..ctx-1 of one stream from a paged pool.

    pool [n_pages][Hkv][P][d]; page_table[j] is the physical page holding
    logical positions j*P .. j*P+P-1.  Returns [Hkv][ctx][d] (fp64).
    """
    P = pool.shape[2]
    n_log = (ctx + P - 1) // P
    pages = pool[np.asarray(page_table[:n_log], dtype=np.int64)]     # [n_log][Hkv][P][d]
    seq = np.transpose(pages, (1, 0, 2, 3)).reshape(pool.shape[1], n_log * P, pool.shape[3])
    return seq[:, :ctx, :]


# ---------------------------------------------------------------------------
# Router and experts
# ---------------------------------------------------------------------------

def route(logits: np.ndarray, bias: np.ndarray, top_k: int):
    """Sigmoid router with a selection-only bias.

    s = sigmoid(logits); the K experts with the largest s + bias are selected
    (equal keys: lower expert index first); their weights are s / sum(s) over
    the selected set.  Returns (idx [T][K] sorted by key desc, w [T][K], s, key).
    Pinned (brute force on 16 experts, weights sum to 1, bias = 0 case).
    """
    s = sigmoid(logits)
    key = s + np.asarray(bias, dtype=np.float64)
    T, E = key.shape
    idx = np.empty((T, top_k), dtype=np.int64)
    w = np.empty((T, top_k), dtype=np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-key[t, e], e))
        sel = np.array(order[:top_k], dtype=np.int64)
        idx[t] = sel
        w[t] = s[t, sel] / s[t, sel].sum()
    return idx, w, s, key


def swiglu(w1: Linear, w3: Linear, w2: Linear, z: np.ndarray) -> np.ndarray:
    """W2 (silu(W1 z) * (W3 z)) for rows of z [n][H] -> [n][H]: W1 is the gate
    (through silu), W3 the up projection.  Pinned (a hand-computed case with
    W1 != W3, in which swapping the two roles changes the result)."""
    return linear(w2, silu(linear(w1, z)) * linear(w3, z))


# ---------------------------------------------------------------------------
# One layer and the stack
# ---------------------------------------------------------------------------

@dataclass
class LayerView:
    """Accessors for one layer's weights (arrays, or callables fetching them).

    expert(e) must return (w1, w3, w2) Linear objects for routed expert e.  The
    oracle only asks for the experts that the router selects: computing only the
    selected experts *is* the definition of a sparse MoE.
    """
    attn_norm: np.ndarray
    w_qkv: Linear
    w_o: Linear
    moe_norm: np.ndarray
    w_router: Linear
    router_bias: np.ndarray
    expert: Callable[[int], Sequence[Linear]]
    shared: Optional[Sequence[Linear]] = None


@dataclass
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    expert_inter: int
    rms_eps: float = 1e-6
    rope_base: float = 10000.0
    kv_dtype: str = "bf16"          # "bf16" | "f32" | "fp8" (e4m3 codes times a per-layer scale)


def layer_forward(x: np.ndarray, lw: LayerView, dims: Dims, k_ctx: np.ndarray,
                  v_ctx: np.ndarray, ctx: int,
                  route_hook: Optional[Callable] = None, kv_scale=(1.0, 1.0)):
    """One pre-norm decoder layer for a verify block of T tokens.

    x [T][H] residual input; k_ctx, v_ctx [Hkv][ctx][d] cached entries.
    Token t sits at position ctx + t.  Steps (reading of the workload, see the
    module docstring):
      u = RMSNorm(x; attn_norm); q,k,v = W_qkv u (rows: Hq heads of q, then Hkv
      of k, then Hkv of v); rotate q and k at their positions; store k and v in
      the cache dtype; o = causal GQA attention; h = x + W_o o;
      z = RMSNorm(h; moe_norm); s = sigmoid(W_router z); select top-K of
      s + bias; x' = h + sum_j w_j SwiGLU_{e_j}(z) + SwiGLU_shared(z).
    ``route_hook(t, key_row, idx_row)`` may replace a token's selection when the
    oracle's own K-th/(K+1)-th key gap is a near tie (see ``stack_forward``).
    Returns (x', info) with info holding k_new, v_new (as stored), idx, w, key,
    and the attention output.
    """
    T, H = x.shape
    Hq, Hkv, d = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    pos = ctx + np.arange(T)
    u = rmsnorm(x, lw.attn_norm, dims.rms_eps)
    qkv = linear(lw.w_qkv, u)                                   # [T][(Hq+2Hkv)d]
    q = qkv[:, : Hq * d].reshape(T, Hq, d)
    k = qkv[:, Hq * d: (Hq + Hkv) * d].reshape(T, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d:].reshape(T, Hkv, d)
    q = rope(q, pos[:, None], dims.rope_base)
    k = rope(k, pos[:, None], dims.rope_base)
    if dims.kv_dtype == "fp8":
        # stored as e4m3 codes of value / scale, read back as code * scale
        k_new = round_to_e4m3(k / kv_scale[0]) * kv_scale[0]
        v_new = round_to_e4m3(v / kv_scale[1]) * kv_scale[1]
    else:
        rnd = round_to_bf16 if dims.kv_dtype == "bf16" else round_to_f32
        k_new, v_new = rnd(k), rnd(v)
    o = attention_gqa(q, k_ctx, v_ctx, k_new, v_new)            # [T][Hq][d]
    h = x + linear(lw.w_o, o.reshape(T, Hq * d))
    z = rmsnorm(h, lw.moe_norm, dims.rms_eps)
    logits = linear(lw.w_router, z)                             # [T][E]
    idx, w, s, key = route(logits, lw.router_bias, dims.top_k)
    overridden = []
    if route_hook is not None:
        for t in range(T):
            new = route_hook(t, key[t], idx[t])
            if new is not None:
                new = np.asarray(new, dtype=np.int64)
                idx[t] = new
                w[t] = s[t, new] / s[t, new].sum()
                overridden.append(t)
    moe = np.zeros_like(h)
    for e in sorted(set(int(v_) for v_ in idx.ravel())):
        toks = [t for t in range(T) if e in idx[t]]
        w1, w3, w2 = lw.expert(e)
        y = swiglu(w1, w3, w2, z[toks])
        for i, t in enumerate(toks):
            j = int(np.nonzero(idx[t] == e)[0][0])
            moe[t] += w[t, j] * y[i]
    if lw.shared is not None:
        moe += swiglu(lw.shared[0], lw.shared[1], lw.shared[2], z)
    x_out = h + moe
    info = dict(k_new=k_new, v_new=v_new, k_rot=k, v_raw=v, idx=idx, w=w, key=key, s=s, attn=o, h=h,
                z=z, logits_router=logits, overridden=overridden,
                distinct=len(set(int(v_) for v_ in idx.ravel())))
    return x_out, info


def accept_count(tokens: Sequence[int], argmax: Sequence[int]) -> int:
    """Longest accepted draft prefix.

    tokens = [d_0, d_1, ..., d_k]: d_0 is the last accepted token, d_1..d_k are
    drafts; argmax[i] is the model's choice after seeing d_0..d_i.  Draft d_i
    is accepted while every earlier draft was and d_i == argmax[i-1].  Returns
    n = max j <= k with d_i == argmax[i-1] for all 1 <= i <= j; the step then
    emits n + 1 tokens (d_1..d_n and argmax[n]), so tokens per verify step =
    accepted + 1 (al-engr "The decomposition": 5.94 = 4.94 accepted + 1).
    Pinned (exhaustive on small vocabularies).
    """
    n = 0
    for i in range(1, len(tokens)):
        if int(tokens[i]) == int(argmax[i - 1]):
            n = i
        else:
            break
    return n


def softmax_t(logits_row: np.ndarray, temperature: float) -> np.ndarray:
    """Sampling distribution at temperature t > 0: p = exp(l / t) / sum exp(l / t),
    in fp64 with the maximum subtracted first (top-p 1: no truncation).  Pinned."""
    z = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    e = np.exp(z - np.max(z))
    return e / e.sum()


def sample_index(weights: np.ndarray, v: float) -> int:
    """Inverse-CDF draw in index order from non-negative weights: the smallest x
    with w_0 + ... + w_x > v * sum(w), for a uniform v in [0, 1).  A zero weight
    is never drawn.  Pinned (boundaries by hand)."""
    w = np.asarray(weights, dtype=np.float64)
    cum = np.cumsum(w)
    target = float(v) * cum[-1]
    x = int(np.searchsorted(cum, target, side="right"))
    if x >= len(w):                       # v * sum at the very top: the last nonzero weight
        x = int(np.nonzero(w > 0)[0][-1])
    return x


def sample_verify(logits: np.ndarray, tokens: Sequence[int], temperature: float,
                  uniforms: Sequence[float]):
    """Verification of a draft block by sampling at temperature t (top-p 1).

    tokens = [d_0, d_1, ..., d_k]; row i of logits is the model's distribution
    p_i = softmax_t(logits[i], t) after d_0..d_i.  The drafts are proposed
    greedily, so the draft distribution at each position is a point mass on
    d_i.  Speculative sampling then accepts d_i with probability
    min(1, p_{i-1}(d_i) / 1) = p_{i-1}(d_i): draft i is accepted while every
    earlier draft was and uniforms[i-1] < p_{i-1}(d_i).  With n drafts accepted,
    the step emits d_1..d_n and one token drawn with uniforms[k]:
      - after a rejection (n < k) from the residual max(0, p_n - q) normalised,
        which for the point mass q on d_{n+1} is p_n with d_{n+1} removed;
      - after k acceptances from p_k.
    The emitted tokens are then distributed as sampling from the model one
    token at a time.  Returns (n, drawn token).
    (ezolabs "Appendix: method", Decode speed: temperature 1.0, top-p 1.0;
    block verification, section "How we got here".)  Pinned.
    """
    lg = np.asarray(logits, dtype=np.float64)
    k = len(tokens) - 1
    n = 0
    for i in range(1, k + 1):
        p = softmax_t(lg[i - 1], temperature)
        if float(uniforms[i - 1]) < p[int(tokens[i])]:
            n = i
        else:
            break
    p = softmax_t(lg[n], temperature)
    if n < k:
        p = p.copy()
        p[int(tokens[n + 1])] = 0.0
    return n, sample_index(p, float(uniforms[k]))


def tokens_per_second(tokens_per_step: float, step_seconds: float) -> float:
    """tokens/s = tokens per verify step x verify steps per second
    (al-engr "The decomposition")."""
    return tokens_per_step / step_seconds


def step_seconds_from(tokens_per_step: float, tok_per_s: float) -> float:
    """Step time implied by tokens per step and tokens per second."""
    return tokens_per_step / tok_per_s


def stack_forward(tokens: Sequence[int], embed: np.ndarray, layers: Sequence[LayerView],
                  final_norm: np.ndarray, lm_head: Linear, dims: Dims,
                  kv_ctx: Sequence, ctx: int, route_hook_factory=None,
                  on_layer: Optional[Callable] = None, kv_scales: Optional[Sequence] = None):
    """Full verify step: embedding, L layers, final norm, LM head, argmax, accept.

    tokens [T] int (d_0..d_k); embed: callable(token ids) -> fp64 rows [T][H]
    or a [V][H] fp64 array; kv_ctx[l] = (k_ctx, v_ctx) for layer l.
    Returns dict(logits [T][V], argmax [T], accepted, layers=[info...]).
    ``route_hook_factory(l)`` gives the per-layer hook (see ``layer_forward``).
    Pinned through the special cases named in the module docstring.
    """
    T = len(tokens)
    x = embed(np.asarray(tokens)) if callable(embed) else np.asarray(embed)[np.asarray(tokens)]
    x = np.asarray(x, dtype=np.float64)
    infos = []
    for l, lw in enumerate(layers):
        hook = route_hook_factory(l) if route_hook_factory is not None else None
        x, info = layer_forward(x, lw, dims, kv_ctx[l][0], kv_ctx[l][1], ctx, hook,
                                kv_scale=kv_scales[l] if kv_scales is not None else (1.0, 1.0))
        infos.append(info)
        if on_layer is not None:
            on_layer(l, x, info)
    xf = rmsnorm(x, final_norm, dims.rms_eps)
    logits = linear(lm_head, xf)
    am = argmax_lowest(logits)
    acc = accept_count(tokens, am)
    return dict(logits=logits, argmax=am, accepted=acc, layers=infos, x_final=x)


def kv_from_pool(kind: str, k_pool: np.ndarray, v_pool: np.ndarray,
                 page_table: np.ndarray, ctx: int, scales=(1.0, 1.0)):
    """Decode a stream's cached K/V (stored bits) and follow its page table.

    kind "bf16": pools hold uint16 bfloat16 bits; "f32": float32 values; "fp8":
    uint8 E4M3 codes, read as code * scale (scales = (K scale, V scale)).
    Returns (k_ctx, v_ctx), each fp64 [Hkv][ctx][d].  Pinned (a hand-built pool
    whose entries name their page, head and slot, read through a permuted
    page table).
    """
    if kind == "fp8":
        dec = fp8_e4m3_decode
    else:
        dec = bf16_decode if kind == "bf16" else (lambda a: np.asarray(a, dtype=np.float64))
    P = k_pool.shape[2]
    n_log = (ctx + P - 1) // P
    pt = np.asarray(page_table[:n_log], dtype=np.int64)
    return (gather_paged(dec(k_pool[pt]), np.arange(n_log), ctx) * scales[0],
            gather_paged(dec(v_pool[pt]), np.arange(n_log), ctx) * scales[1])


def linear_from(kind: str, q: np.ndarray, scale=None) -> Linear:
    """Build a Linear from (kind, stored array, scale) as the generators hand it over."""
    return Linear(kind, q, scale)
