"""Pins of the fp64 oracle against facts fixed outside it: format definitions,
closed forms, library routines, brute force, the pages' printed arithmetic and
the method's own invariants.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_persistent_gb300 import synth
from tests import helpers

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# --------------------------------------------------------------------- formats
def test_fp8_points_from_spec():
    g = json.load(open(os.path.join(GOLD, "fp8_e4m3_points.json")))
    for code, val in g["points"]:
        got = oracle.fp8_e4m3_decode(np.array([int(code, 16)]))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in g["nan"]:
        assert np.isnan(oracle.fp8_e4m3_decode(np.array([int(code, 16)]))[0])


def test_fp8_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    ours = oracle.FP8_E4M3_TABLE
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~fin)
    assert np.array_equal(ours[fin], ref[fin])


def test_bf16_decode_and_round_match_torch():
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))
    x32 = x.astype(np.float32)
    t = torch.from_numpy(x32).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_decode(bits), t.float().double().numpy())
    # rounding an fp32-representable value: torch's RNE fp32->bf16 is the library reference
    assert np.array_equal(oracle.round_to_bf16(x32.astype(np.float64)), t.float().double().numpy())


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even significand (1)
    assert oracle.round_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: even is 1 + 2^-6
    assert oracle.round_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert oracle.round_to_bf16(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 1 + 2 ** -7


def test_f32_round_ties_to_even():
    # binary32 keeps 24 significant bits: 1 + 2^-24 lies halfway between 1 and
    # 1 + 2^-23, and the tie goes to the even significand (1)
    assert oracle.round_to_f32(np.array([1 + 2 ** -24]))[0] == 1.0
    # 1 + 3*2^-24 lies halfway between 1 + 2^-23 and 1 + 2^-22: even is 1 + 2^-22
    assert oracle.round_to_f32(np.array([1 + 3 * 2 ** -24]))[0] == 1 + 2 ** -22
    # just above a halfway point rounds up
    assert oracle.round_to_f32(np.array([1 + 2 ** -24 + 2 ** -40]))[0] == 1 + 2 ** -23
    # subnormal grid 2^-149: 3*2^-150 is halfway between 2^-149 and 2^-148 -> 2^-148
    assert oracle.round_to_f32(np.array([3 * 2.0 ** -150]))[0] == 2.0 ** -148
    # 2^-150 is halfway between 0 and 2^-149 -> 0 (even)
    assert oracle.round_to_f32(np.array([2.0 ** -150]))[0] == 0.0
    # a value binary32 holds exactly is unchanged
    assert oracle.round_to_f32(np.array([0.1875]))[0] == 0.1875


def test_mxfp4_points_from_spec():
    g = json.load(open(os.path.join(GOLD, "mxfp4_points.json")))
    assert g["block"] == 32
    for code, val in g["e2m1"]:
        got = oracle.E2M1_TABLE[int(code, 16)]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code, val in g["e8m0"]:
        assert oracle.e8m0_decode(np.array([int(code, 16)]))[0] == val, code
    for code in g["e8m0_nan"]:
        assert np.isnan(oracle.e8m0_decode(np.array([int(code, 16)]))[0])


def test_e8m0_matches_torch():
    codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).float().double().numpy()
    assert np.array_equal(oracle.e8m0_decode(np.arange(255)), ref)


def test_e2m1_nibble_order():
    # byte 0x21: element 0 is the low nibble (0x1 = 0.5), element 1 the high
    # nibble (0x2 = 1.0); byte 0xF7: 6.0 then -6.0
    got = oracle.e2m1_unpack(np.array([[0x21, 0xF7]], dtype=np.uint8))
    assert got.tolist() == [[0.5, 1.0, 6.0, -6.0]]


def test_mxfp4_linear_exact_on_small_values():
    # every E2M1 value times 2 is an integer and E8M0 scales are powers of two,
    # so a 1 x 32 block-scaled product is exact in fp64 and must equal an
    # integer computation scaled per block
    N, K = 12, 96
    codes = rng.integers(0, 16, size=(N, K))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = rng.integers(120, 131, size=(K // 32, N)).astype(np.uint8)
    x = rng.integers(-4, 5, size=(3, K)).astype(np.float64)
    got = oracle.linear(oracle.Linear("mxfp4", packed, sc), x)
    twice = np.array([int(round(2 * oracle.E2M1_TABLE[c])) for c in range(16)], dtype=np.int64)
    w2 = twice[codes]                                     # 2 * element value, integer
    want = np.zeros((3, N))
    for kb in range(K // 32):
        part = x[:, kb * 32:(kb + 1) * 32].astype(np.int64) @ w2[:, kb * 32:(kb + 1) * 32].T
        want += part * np.ldexp(1.0, sc[kb].astype(np.int64) - 127 - 1)[None, :]
    assert np.array_equal(got, want)


def test_e4m3_rounding_matches_torch_and_ties():
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))
    x = x[np.abs(x) <= 448.0].astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(oracle.round_to_e4m3(x), ref)
    # 1 + 2^-4 lies halfway between 1 and 1.125: the even significand (1) wins;
    # 1 + 3 * 2^-4 lies halfway between 1.125 and 1.25: 1.25 wins
    assert oracle.round_to_e4m3(np.array([1 + 2 ** -4, 1 + 3 * 2 ** -4])).tolist() == [1.0, 1.25]
    # subnormal grid 2^-9; 2^-10 is halfway between 0 and 2^-9 -> 0
    assert oracle.round_to_e4m3(np.array([2.0 ** -10, 3 * 2.0 ** -10])).tolist() == [0.0, 2 * 2.0 ** -9]
    # no infinity: beyond 448 the result saturates
    assert oracle.round_to_e4m3(np.array([1000.0, -1e9])).tolist() == [448.0, -448.0]


def test_kv_from_pool_fp8_scales():
    codes = np.array([[[[0x38, 0x40]]]], dtype=np.uint8)   # e4m3 1.0 and 2.0
    k, v = oracle.kv_from_pool("fp8", codes, codes, np.array([0]), 1, scales=(0.5, 4.0))
    assert k[0, 0].tolist() == [0.5, 1.0] and v[0, 0].tolist() == [4.0, 8.0]


# ---------------------------------------------------------------- linear/dequant
def test_fp8_linear_exact_on_integer_weights():
    # codes for the integers 1..8 and their negatives, power-of-two block scales:
    # every product and sum is exact in fp64, so an integer computation must agree bit for bit
    int_codes = {v: c for c in range(256) for v in [oracle.FP8_E4M3_TABLE[c]]
                 if not np.isnan(v) and v == int(v) and abs(v) <= 8}
    vals = np.array(sorted(int_codes))
    N, K = 24, 384
    wv = rng.choice(vals, size=(N, K))
    q = np.vectorize(lambda v: int_codes[v])(wv).astype(np.uint8)
    scale = (2.0 ** rng.integers(-6, 4, size=(K // 128, N))).astype(np.float32)
    x = rng.integers(-5, 6, size=(3, K)).astype(np.float64)
    got = oracle.linear(oracle.Linear("fp8", q, scale), x)
    want = np.zeros((3, N))
    wi = wv.astype(np.int64)
    xi = x.astype(np.int64)
    for kb in range(K // 128):
        part = xi[:, kb * 128:(kb + 1) * 128] @ wi[:, kb * 128:(kb + 1) * 128].T   # int64
        want += part * scale[kb][None, :].astype(np.float64)
    assert np.array_equal(got, want)


def test_linear_identity_and_bf16():
    eye = np.eye(64, dtype=np.float32)
    x = rng.standard_normal((2, 64))
    assert np.array_equal(oracle.linear(oracle.Linear("f32", eye), x), x)
    bits = torch.from_numpy(eye).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.linear(oracle.Linear("bf16", bits), x), x)


# ------------------------------------------------------------------ elementwise
def test_rmsnorm_constant_vector():
    for c in (0.0, 1e-4, 0.5, 3.0, -7.0):
        g = rng.uniform(0.5, 1.5, 96)
        got = oracle.rmsnorm(np.full((1, 96), c), g, 1e-6)
        assert np.allclose(got, g * c / math.sqrt(c * c + 1e-6), rtol=1e-14, atol=0)


def test_silu_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(oracle.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_rope_closed_forms():
    x = rng.standard_normal((3, 128))
    assert np.array_equal(oracle.rope(x, np.zeros(3), 10000.0), x)          # identity at 0
    p = np.array([1, 100, 65535])
    r = oracle.rope(x, p, 10000.0)
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # d = 2: rotation of (x0, x1) by the angle p
    v = np.array([[0.3, -1.2]])
    for pp in (0.5, 3.0, 17.0):
        got = oracle.rope(v, np.array([pp]), 10000.0)[0]
        want = [0.3 * math.cos(pp) + 1.2 * math.sin(pp), -1.2 * math.cos(pp) + 0.3 * math.sin(pp)]
        assert np.allclose(got, want, rtol=0, atol=1e-15)
    # d = 4: pairs are (0, 2) and (1, 3), pair i rotates at base^(-2i/d)
    v4 = np.array([[1.0, 0.0, 0.0, 0.0]])
    got = oracle.rope(v4, np.array([2.0]), 100.0)[0]
    assert np.allclose(got, [math.cos(2.0), 0, math.sin(2.0), 0], atol=1e-15)
    v4 = np.array([[0.0, 1.0, 0.0, 0.0]])
    got = oracle.rope(v4, np.array([2.0]), 100.0)[0]
    a = 2.0 * 100.0 ** (-0.5)
    assert np.allclose(got, [0, math.cos(a), 0, math.sin(a)], atol=1e-15)


def test_rope_relative_position():
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    vals = []
    for p in (5, 105, 1005, 60005):
        vals.append(oracle.rope(q[None], np.array([p + 7]), 10000.0)[0] @
                    oracle.rope(k[None], np.array([p]), 10000.0)[0])
    assert np.allclose(vals, vals[0], rtol=1e-9)


# -------------------------------------------------------------------- attention
def _brute_attention(q, kc, vc, kn, vn):
    T, Hq, d = q.shape
    Hkv = kn.shape[1]
    out = np.zeros_like(q)
    for t in range(T):
        for h in range(Hq):
            g = h * Hkv // Hq
            keys = [kc[g, j] for j in range(kc.shape[1])] + [kn[j, g] for j in range(t + 1)]
            vals = [vc[g, j] for j in range(vc.shape[1])] + [vn[j, g] for j in range(t + 1)]
            sc = [sum(q[t, h, i] * kk[i] for i in range(d)) / math.sqrt(d) for kk in keys]
            mx = max(sc)
            ws = [math.exp(s - mx) for s in sc]
            tot = sum(ws)
            for i in range(d):
                out[t, h, i] = sum(w * vv[i] for w, vv in zip(ws, vals)) / tot
    return out


def _rand_attn(T=3, Hq=4, Hkv=2, d=8, ctx=5):
    return (rng.standard_normal((T, Hq, d)), rng.standard_normal((Hkv, ctx, d)),
            rng.standard_normal((Hkv, ctx, d)), rng.standard_normal((T, Hkv, d)),
            rng.standard_normal((T, Hkv, d)))


def test_attention_brute_force():
    args = _rand_attn()
    assert np.allclose(oracle.attention_gqa(*args), _brute_attention(*args), rtol=1e-12, atol=1e-13)


def test_attention_single_key_and_equal_keys():
    q, kc, vc, kn, vn = _rand_attn(T=1, ctx=0)
    o = oracle.attention_gqa(q, kc, vc, kn, vn)
    for h in range(4):
        assert np.allclose(o[0, h], vn[0, h * 2 // 4], rtol=1e-15)
    q, kc, vc, kn, vn = _rand_attn(T=1, ctx=9)
    kc[:] = 0.7
    kn[:] = 0.7
    o = oracle.attention_gqa(q, kc, vc, kn, vn)
    for h in range(4):
        g = h * 2 // 4
        mean = (vc[g].sum(0) + vn[0, g]) / 10
        assert np.allclose(o[0, h], mean, rtol=1e-12)


def test_attention_causal_in_block():
    q, kc, vc, kn, vn = _rand_attn(T=4)
    o = oracle.attention_gqa(q, kc, vc, kn, vn)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[3] += 5.0
    vn2[3] -= 3.0
    o2 = oracle.attention_gqa(q, kc, vc, kn2, vn2)
    assert np.array_equal(o[:3], o2[:3])
    assert not np.allclose(o[3], o2[3])


def test_attention_split_merge_equals_direct():
    """Log-sum-exp merge of two halves of the key set equals one softmax."""
    q, kc, vc, kn, vn = _rand_attn(T=1, Hq=1, Hkv=1, d=16, ctx=40)
    o = oracle.attention_gqa(q, kc, vc, kn, vn)[0, 0]
    keys = np.concatenate([kc[0], kn[:1, 0]])
    vals = np.concatenate([vc[0], vn[:1, 0]])
    parts = []
    for sl in (slice(0, 17), slice(17, None)):
        s = keys[sl] @ q[0, 0] / 4.0
        m = s.max()
        p = np.exp(s - m)
        parts.append((m, p.sum(), p @ vals[sl]))
    M = max(p[0] for p in parts)
    num = sum(math.exp(m - M) * a for m, _, a in parts)
    den = sum(math.exp(m - M) * l for m, l, _ in parts)
    assert np.allclose(o, num / den, rtol=1e-12)


def test_gqa_head_mapping():
    q, kc, vc, kn, vn = _rand_attn(T=1, Hq=8, Hkv=2, ctx=3)
    vc[0], vn[:, 0] = 1.0, 1.0
    vc[1], vn[:, 1] = -2.0, -2.0
    o = oracle.attention_gqa(q, kc, vc, kn, vn)
    assert np.allclose(o[0, :4], 1.0) and np.allclose(o[0, 4:], -2.0)


def test_paged_gather_follows_table():
    pool = rng.standard_normal((5, 2, 4, 3))
    pt = np.array([3, 0, 4])
    seq = oracle.gather_paged(pool, pt, 10)
    for p in range(10):
        assert np.array_equal(seq[:, p], pool[pt[p // 4], :, p % 4])


def test_kv_from_pool_hand_built_table():
    # 3 physical pages of 2 positions, 2 kv heads, head dim 2; entry
    # (page p, head h, slot i) holds (100h + 10p + i, -(100h + 10p + i)).
    P, Hkv, d = 2, 2, 2
    pool = np.zeros((3, Hkv, P, d), dtype=np.float32)
    for p in range(3):
        for h in range(Hkv):
            for i in range(P):
                pool[p, h, i] = (100 * h + 10 * p + i, -(100 * h + 10 * p + i))
    vpool = pool + 0.5
    # logical page 0 -> physical 2, 1 -> 0, 2 -> 1; five cached positions
    pt = np.array([2, 0, 1])
    k, v = oracle.kv_from_pool("f32", pool, vpool, pt, 5)
    want_h0 = [20, 21, 0, 1, 10]
    want_h1 = [120, 121, 100, 101, 110]
    assert k.shape == (2, 5, 2)
    assert k[0, :, 0].tolist() == want_h0 and k[1, :, 0].tolist() == want_h1
    assert k[0, :, 1].tolist() == [-x for x in want_h0]
    assert v[1, :, 0].tolist() == [x + 0.5 for x in want_h1]
    # the same pool stored as bf16 bits (small integers are exact in bf16)
    bits = torch.from_numpy(pool).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kb, _ = oracle.kv_from_pool("bf16", bits, bits, pt, 3)
    assert kb[0, :, 0].tolist() == [20, 21, 0] and kb[1, :, 1].tolist() == [-120, -121, -100]


# ----------------------------------------------------------------------- router
def test_router_brute_force_16_choose_2():
    for trial in range(20):
        logits = rng.standard_normal((1, 16)) * 2
        bias = rng.uniform(-0.1, 0.1, 16) if trial % 2 else np.zeros(16)
        idx, w, s, key = oracle.route(logits, bias, 2)
        best = None
        for pair in itertools.combinations(range(16), 2):
            rest = [e for e in range(16) if e not in pair]
            if min(key[0, list(pair)]) > max(key[0, rest]):
                assert best is None
                best = set(pair)
        assert best == set(idx[0].tolist())
        assert abs(w.sum() - 1.0) < 1e-15
        sig = 1 / (1 + np.exp(-logits[0, list(idx[0])]))
        assert np.allclose(w[0], sig / sig.sum(), rtol=1e-15)      # weights from unbiased s


def test_router_top8_properties_and_ties():
    logits = rng.standard_normal((6, 384))
    idx, w, s, key = oracle.route(logits, rng.uniform(-0.1, 0.1, 384), 8)
    for t in range(6):
        assert len(set(idx[t].tolist())) == 8
        assert abs(w[t].sum() - 1) < 1e-14
    # zero bias reduces to the plain top-K of s
    idx0, *_ = oracle.route(logits, np.zeros(384), 8)
    for t in range(6):
        assert set(idx0[t].tolist()) == set(np.argsort(-logits[t])[:8].tolist())
    # exact ties: lower index first
    lg = np.zeros((1, 10))
    idx, *_ = oracle.route(lg, np.zeros(10), 3)
    assert idx[0].tolist() == [0, 1, 2]


# ----------------------------------------------------------------------- accept
def _accept_brute(tokens, am):
    k = len(tokens) - 1
    for n in range(k, -1, -1):
        if all(tokens[i] == am[i - 1] for i in range(1, n + 1)):
            return n
    return 0


def test_accept_exhaustive_small():
    for T in range(1, 5):
        for toks in itertools.product(range(3), repeat=T):
            for am in itertools.product(range(3), repeat=T):
                assert oracle.accept_count(toks, am) == _accept_brute(toks, am)


def test_accept_special_cases():
    am = [5, 6, 7, 8, 9, 10]
    assert oracle.accept_count([1] + am[:5], am) == 5
    assert oracle.accept_count([1, 4, 6, 7, 8, 9], am) == 0
    assert oracle.accept_count([1, 5, 6, 0, 8, 9], am) == 2


def test_decomposition_golden():
    g = json.load(open(os.path.join(GOLD, "decomposition.json")))
    c = g["cases"]
    assert abs(oracle.tokens_per_second(c[0]["tokens_per_step"], c[0]["step_ms"] / 1e3)
               - c[0]["tok_s"]) <= c[0]["tol"]
    assert abs(oracle.tokens_per_second(c[1]["tokens_per_step"], c[1]["step_ms"] / 1e3)
               - c[1]["tok_s"]) <= c[1]["tol"]
    assert abs(oracle.step_seconds_from(c[2]["tokens_per_step"], c[2]["tok_s"]) * 1e3
               - c[2]["step_ms"]) <= c[2]["tol_ms"]
    assert abs(c[3]["accepted"] + 1 - c[3]["tokens_per_step"]) < 1e-12
    r = c[4]
    assert abs(r["tok_s_a"] / r["tok_s_b"] - r["ratio"]) <= r["tol"]
    assert abs(r["factors"][0] * r["factors"][1] - r["ratio"]) <= r["tol"]


# ------------------------------------------------------------------ whole layer
def _tiny(**kw):
    cfg = synth.tiny_config(**kw)
    model = synth.make_model(cfg, "cpu")
    return cfg, model


def test_block_verification_equals_sequential_decode():
    """Verifying T tokens in one pass = T single-token steps with KV appends."""
    cfg, model = _tiny(T=4, ctx=70, gamma_jitter=0.1, bias_range=0.1)
    kv = synth.make_kv(cfg, "cpu")
    dims = helpers.oracle_dims(cfg)
    lv = helpers.layer_view(model, 0)
    kc, vc = helpers.kv_view(kv, 0)
    x = np.random.default_rng(7).standard_normal((4, cfg.hidden))
    blk, info = oracle.layer_forward(x, lv, dims, kc, vc, cfg.ctx)
    kcs, vcs = kc, vc
    for t in range(4):
        y, inf1 = oracle.layer_forward(x[t:t + 1], lv, dims, kcs, vcs, cfg.ctx + t)
        assert np.allclose(y[0], blk[t], rtol=0, atol=1e-11)
        kcs = np.concatenate([kcs, np.transpose(inf1["k_new"], (1, 0, 2))], axis=1)
        vcs = np.concatenate([vcs, np.transpose(inf1["v_new"], (1, 0, 2))], axis=1)


def test_moe_identical_experts_reduce_to_dense_swiglu():
    cfg, model = _tiny(T=2)
    L = model.layers[0]
    L.w1.data[:] = L.w1.data[0:1]
    L.w3.data[:] = L.w3.data[0:1]
    L.w2.data[:] = L.w2.data[0:1]
    L.ws2.data.zero_()
    kv = synth.make_kv(cfg, "cpu")
    dims = helpers.oracle_dims(cfg)
    lv = helpers.layer_view(model, 0)
    kc, vc = helpers.kv_view(kv, 0)
    x = np.random.default_rng(3).standard_normal((2, cfg.hidden))
    out, info = oracle.layer_forward(x, lv, dims, kc, vc, cfg.ctx)
    dense = oracle.swiglu(*lv.expert(0), info["z"])
    assert np.allclose(out - info["h"], dense, rtol=1e-12, atol=1e-13)


def test_swiglu_gate_and_up_roles_hand_case():
    # H = 2, I = 1: W1 (gate) reads z_0 with weight 2, W3 (up) reads z_1 with
    # weight 3, W2 writes the intermediate to the two outputs with weights 1
    # and -0.5.  For z = (1, 1): gate 2, up 3, intermediate silu(2) * 3 =
    # 6 / (1 + e^-2) = 5.284782467867294.  Swapping gate and up would give
    # silu(3) * 2 = 5.7154447609345995.  For z = (-1, 2): gate -2, up 6,
    # intermediate -12 / (1 + e^2) = -1.4304350642654104.
    w1 = oracle.Linear("f32", np.array([[2.0, 0.0]], dtype=np.float32))
    w3 = oracle.Linear("f32", np.array([[0.0, 3.0]], dtype=np.float32))
    w2 = oracle.Linear("f32", np.array([[1.0], [-0.5]], dtype=np.float32))
    y = oracle.swiglu(w1, w3, w2, np.array([[1.0, 1.0], [-1.0, 2.0]]))
    want = np.array([[5.284782467867294, -2.642391233933647],
                     [-1.4304350642654104, 0.7152175321327052]])
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    assert not np.allclose(y[0, 0], 5.7154447609345995, rtol=1e-3)


def test_moe_linear_in_weights():
    """Scaling one routed expert's W2 by c scales its contribution by c (c = 4, exact in fp32)."""
    cfg, model = _tiny(T=1)
    kv = synth.make_kv(cfg, "cpu")
    dims = helpers.oracle_dims(cfg)
    kc, vc = helpers.kv_view(kv, 0)
    x = np.random.default_rng(5).standard_normal((1, cfg.hidden))
    lv = helpers.layer_view(model, 0)
    out, info = oracle.layer_forward(x, lv, dims, kc, vc, cfg.ctx)
    e0 = int(info["idx"][0, 0])
    model.layers[0].w2.data[e0] *= 4.0
    lv2 = helpers.layer_view(model, 0)
    out2, info2 = oracle.layer_forward(x, lv2, dims, kc, vc, cfg.ctx)
    contrib = info["w"][0, 0] * oracle.swiglu(*lv.expert(e0), info["z"])
    assert np.allclose(out2 - out, 3.0 * contrib, rtol=1e-10, atol=1e-12)


def test_stack_accept_and_argmax_consistency():
    cfg = synth.tiny_config(n_layers=2, vocab=300, T=4, ctx=64)
    model = synth.make_model(cfg, "cpu")
    kv = synth.make_kv(cfg, "cpu")
    dims = helpers.oracle_dims(cfg)
    layers = [helpers.layer_view(model, l) for l in range(2)]
    kvs = [helpers.kv_view(kv, l) for l in range(2)]
    toks = [3, 10, 20, 30]
    r = oracle.stack_forward(toks, helpers.embed_fn(model), layers,
                             model.final_norm.numpy().astype(np.float64),
                             helpers.lm_head_lin(model), dims, kvs, cfg.ctx)
    assert r["logits"].shape == (4, 300)
    assert np.array_equal(r["argmax"], np.argmax(r["logits"], -1))
    # drafts equal to the model's own argmax are all accepted (causality makes this
    # self-consistent: argmax[i] depends only on tokens 0..i)
    toks2 = [3] + [int(a) for a in r["argmax"][:3]]
    r2 = oracle.stack_forward(toks2, helpers.embed_fn(model), layers,
                              model.final_norm.numpy().astype(np.float64),
                              helpers.lm_head_lin(model), dims, kvs, cfg.ctx)
    assert np.array_equal(r2["argmax"][0], r["argmax"][0])
    # greedy chain: build drafts left to right from the model's own choices
    chain = [3]
    for i in range(3):
        rr = oracle.stack_forward(chain + [0] * (3 - i), helpers.embed_fn(model), layers,
                                  model.final_norm.numpy().astype(np.float64),
                                  helpers.lm_head_lin(model), dims, kvs, cfg.ctx)
        chain.append(int(rr["argmax"][i]))
    rf = oracle.stack_forward(chain, helpers.embed_fn(model), layers,
                              model.final_norm.numpy().astype(np.float64),
                              helpers.lm_head_lin(model), dims, kvs, cfg.ctx)
    assert rf["accepted"] == 3


def _zero_layer_outputs(layer):
    """Zero the O projection and every down projection: the layer becomes the identity."""
    layer.w_o.data.zero_()
    layer.w2.data.zero_()
    if layer.ws2 is not None:
        layer.ws2.data.zero_()


def _stack(model, cfg, toks, n_layers=None):
    n = cfg.n_layers if n_layers is None else n_layers
    kv = synth.make_kv(cfg, "cpu")
    return oracle.stack_forward(toks, helpers.embed_fn(model),
                                [helpers.layer_view(model, l) for l in range(n)],
                                model.final_norm.numpy().astype(np.float64),
                                helpers.lm_head_lin(model), helpers.oracle_dims(cfg),
                                [helpers.kv_view(kv, l) for l in range(n)], cfg.ctx)


def test_stack_identity_layers_reduce_to_final_norm_and_lm_head():
    # With every O projection and every down projection zero, both residual
    # branches add nothing and the stack's logits are the LM head applied to the
    # RMS-normalised embeddings: computed here with torch's own bf16 decoding
    # and a plain matrix product.  A dropped residual, a second norm or a wrong
    # gamma changes the result.
    cfg = synth.tiny_config(n_layers=2, vocab=300, T=4, ctx=64, gamma_jitter=0.1)
    model = synth.make_model(cfg, "cpu")
    for lay in model.layers:
        _zero_layer_outputs(lay)
    toks = [7, 123, 5, 299]
    r = _stack(model, cfg, toks)
    e = model.embed[torch.tensor(toks)].to(torch.float64)
    g = model.final_norm.to(torch.float64)
    xn = e / torch.sqrt((e * e).mean(dim=1, keepdim=True) + cfg.rms_eps) * g
    want = (xn @ model.lm_head.to(torch.float64).T).numpy()
    assert np.allclose(r["logits"], want, rtol=1e-12, atol=1e-12)
    assert np.allclose(r["x_final"], e.numpy(), rtol=0, atol=0)
    assert np.array_equal(r["argmax"], np.argmax(want, axis=1))


def test_stack_appended_identity_layer_changes_nothing():
    # Layer l of the stack is applied once and in order: a two-layer stack
    # whose second layer is the identity gives the one-layer stack's result,
    # while a second live layer moves it.
    cfg = synth.tiny_config(n_layers=2, vocab=300, T=3, ctx=64)
    model = synth.make_model(cfg, "cpu")
    toks = [11, 42, 250]
    one = _stack(model, cfg, toks, n_layers=1)
    two_live = _stack(model, cfg, toks)
    _zero_layer_outputs(model.layers[1])
    two_ident = _stack(model, cfg, toks)
    assert np.allclose(two_ident["logits"], one["logits"], rtol=1e-13, atol=1e-13)
    assert not np.allclose(two_live["logits"], one["logits"], rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------------------
# Temperature-sampling verification

def test_softmax_t_closed_form():
    # logits ln 1, ln 2, ln 3 at t = 1 give 1/6, 2/6, 3/6; at t = 1/2 the squares 1, 4, 9
    l = np.log([1.0, 2.0, 3.0])
    assert np.allclose(oracle.softmax_t(l, 1.0), [1 / 6, 2 / 6, 3 / 6], rtol=0, atol=1e-15)
    assert np.allclose(oracle.softmax_t(l, 0.5), [1 / 14, 4 / 14, 9 / 14], rtol=0, atol=1e-15)
    # a shift of every logit changes nothing (up to the rounding of l + 1000, an
    # ulp of 1.1e-13); huge logits do not overflow
    assert np.allclose(oracle.softmax_t(l + 1000.0, 1.0), [1 / 6, 2 / 6, 3 / 6], rtol=0, atol=1e-12)


def test_sample_index_boundaries():
    w = [1.0, 2.0, 3.0, 0.0]          # cumulative 1, 3, 6, 6 of 6
    assert oracle.sample_index(w, 0.0) == 0
    assert oracle.sample_index(w, 1 / 6 - 1e-9) == 0
    assert oracle.sample_index(w, 1 / 6) == 1          # strictly above the cumulative 1
    assert oracle.sample_index(w, 0.5 - 1e-9) == 1
    assert oracle.sample_index(w, 0.5) == 2
    assert oracle.sample_index(w, 1 - 1e-12) == 2      # the zero weight is never drawn
    assert oracle.sample_index([0.0, 0.0, 5.0], 0.0) == 2


def test_sample_verify_hand_case():
    # t = 1, rows over 3 tokens with p = (1/6, 2/6, 3/6), (1/2, 1/4, 1/4), (0.1, 0.1, 0.8)
    lg = np.log(np.array([[1, 2, 3], [2, 1, 1], [1, 1, 8]], dtype=np.float64))
    # d_1 = 2: p_0(2) = 0.5 > 0.4 accepted; d_2 = 1: p_1(1) = 0.25 <= 0.3 rejected.
    # Residual of row 1 without token 1: (1/2, 0, 1/4) / (3/4) = (2/3, 0, 1/3); v = 0.7 -> token 2
    assert oracle.sample_verify(lg, [0, 2, 1], 1.0, [0.4, 0.3, 0.7]) == (1, 2)
    # v = 0.6 -> token 0 (cumulative 2/3 > 0.6)
    assert oracle.sample_verify(lg, [0, 2, 1], 1.0, [0.4, 0.3, 0.6]) == (1, 0)
    # both accepted (0.4 < 0.5, 0.2 < 0.25): the bonus comes from row 2, v = 0.15 -> token 1
    assert oracle.sample_verify(lg, [0, 2, 1], 1.0, [0.4, 0.2, 0.15]) == (2, 1)
    # first draft rejected (0.5 is not < 0.5): residual of row 0 without token 2 is (1/3, 2/3, 0)
    assert oracle.sample_verify(lg, [0, 2, 1], 1.0, [0.5, 0.0, 0.5]) == (0, 1)


def test_sample_verify_emits_the_model_distribution():
    # Speculative sampling's guarantee: the first emitted token (the draft if
    # accepted, else the residual draw) is distributed as p_0, whatever the
    # draft.  Integrate over a midpoint grid of (accept, draw) uniforms; the
    # grid is exact to 1/N in each coordinate.
    rng = np.random.default_rng(9)
    V, N = 5, 300
    lg = rng.normal(size=(2, V))
    p0 = oracle.softmax_t(lg[0], 0.8)
    grid = (np.arange(N) + 0.5) / N
    for d in (0, 3):
        counts = np.zeros(V)
        for u in grid:
            for v in grid:
                n, tok = oracle.sample_verify(lg, [4, d], 0.8, [u, v])
                counts[d if n == 1 else tok] += 1
        assert np.max(np.abs(counts / N ** 2 - p0)) < 2.0 / N


def test_sample_verify_low_temperature_is_greedy():
    rng = np.random.default_rng(10)
    V, T = 50, 6
    for trial in range(20):
        lg = rng.normal(size=(T, V))
        am = oracle.argmax_lowest(lg)
        toks = [int(rng.integers(V))]
        for i in range(T - 1):
            toks.append(int(am[i]) if rng.random() < 0.7 else int(rng.integers(V)))
        u = rng.uniform(0.01, 0.99, size=T)
        n, tok = oracle.sample_verify(lg, toks, 1e-4, u)
        assert n == oracle.accept_count(toks, am)
        if n < T - 1:
            # the rejected draft differs from the argmax, which the residual then draws
            assert tok == int(am[n])
        else:
            assert tok == int(am[T - 1])
