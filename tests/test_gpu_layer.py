"""Single-layer parity of the CUDA path (mk_layer_forward) against the fp64 oracle
on the three single-layer workloads and on edge shapes."""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_persistent_gb300 import mk, synth
from tests import gpu_common as gc
from tests import helpers

pytestmark = pytest.mark.gpu


def _run(cfg, ctxs=None, T=None, x_seed=11, l=0):
    T = cfg.T if T is None else T
    b = gc.Built(cfg, ctxs=ctxs, T=T)
    try:
        g = torch.Generator(device="cpu").manual_seed(x_seed)
        x = torch.randn((T, cfg.hidden), generator=g).cuda()
        # oracle inputs are read before the GPU appends K/V (positions >= ctx only)
        kc_before = helpers.kv_view(b.kv, l)
        out, idx, w = b.layer(x, l, T)
        log = []
        ref, info = gc.oracle_layer(b, x.cpu().numpy(), l, gpu_idx=idx.cpu().numpy(), log=log)
        gc.check_routing(info, idx.cpu().numpy(), cfg.top_k)
        err = helpers.rel_err(out.cpu().numpy(), ref)
        # routing weights of the GPU's selection, where it equals the oracle's
        gc.check_weights(info, idx.cpu().numpy(), w.cpu().numpy(), gc.WTOL[cfg.weight_dtype])
        # K/V appended at positions ctx..ctx+T-1 (stored in the cache dtype)
        kv_err = _appended_err(b, info, l, T)
        return err, kv_err, log, info
    finally:
        b.close()


def _appended_fp8_err(b, info, l, T):
    """FP8 cache: the block's K/V are stored as E4M3 codes of value / scale.  A
    code must be the nearest code to the oracle's value / scale, allowing the
    GPU's own rounding of the value (up to 2e-3 of the RMS of the values) to
    move it across a midpoint.  Returns the worst excess in code units relative
    to half a code step (0 when every code is a nearest code)."""
    kv = b.kv
    P = kv.page_size
    ctx = kv.ctx[0]
    pt = kv.page_table[0].cpu().numpy()
    ks, vs = kv.scales[l]
    worst = 0.0
    for t in range(T):
        pos = ctx + t
        ph = int(pt[pos // P])
        for pool, ref, sc in ((kv.k_pools[l], info["k_rot"][t], ks), (kv.v_pools[l], info["v_raw"][t], vs)):
            got = oracle.fp8_e4m3_decode(pool[ph, :, pos % P, :].cpu().numpy())
            want = np.clip(np.asarray(ref, dtype=np.float64) / sc, -448.0, 448.0)
            slack = 2e-3 * np.sqrt(np.mean(ref ** 2)) / sc
            # half the spacing of E4M3 codes around want (subnormal spacing 2^-9)
            e = np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -6)))
            half = 0.5 * np.exp2(e - 3)
            excess = np.abs(got - want) - (half + slack)
            worst = max(worst, float(np.max(excess / half)))
    return worst


def _appended_err(b, info, l, T):
    kv = b.kv
    if kv.scales:
        return _appended_fp8_err(b, info, l, T)
    P = kv.page_size
    ctx = kv.ctx[0]
    pt = kv.page_table[0].cpu().numpy()
    errs = []
    for t in range(T):
        pos = ctx + t
        ph = int(pt[pos // P])
        kg = kv.k_pools[l][ph, :, pos % P, :].float().cpu().numpy()
        vg = kv.v_pools[l][ph, :, pos % P, :].float().cpu().numpy()
        errs.append(np.max(np.abs(kg - info["k_new"][t])) / (np.sqrt(np.mean(info["k_new"] ** 2)) + 1e-30))
        errs.append(np.max(np.abs(vg - info["v_new"][t])) / (np.sqrt(np.mean(info["v_new"] ** 2)) + 1e-30))
    return max(errs)


def test_tiny_fp32_layer():
    cfg = synth.tiny_config()
    err, kv_err, log, _ = _run(cfg)
    assert err < gc.TOL[synth.WDT_F32], err
    assert kv_err < 1e-4, kv_err


@pytest.mark.parametrize("T,ctx", [(1, 0), (1, 1), (2, 63), (3, 64), (1, 65), (4, 130)])
def test_tiny_fp32_layer_edges(T, ctx):
    cfg = synth.tiny_config(T=T, ctx=ctx, gamma_jitter=0.1, bias_range=0.1)
    err, kv_err, log, _ = _run(cfg, T=T)
    assert err < gc.TOL[synth.WDT_F32], err
    assert kv_err < 1e-4


def test_bf16_layer():
    cfg = synth.bf16_layer_config()
    err, kv_err, log, info = _run(cfg)
    assert err < gc.TOL[synth.WDT_BF16], err
    assert kv_err < 2e-2, kv_err


def test_fp8_layer_64k():
    cfg = synth.fp8_layer_config()
    err, kv_err, log, info = _run(cfg)
    assert err < gc.TOL[synth.WDT_FP8], err
    assert kv_err < 2e-2, kv_err


@pytest.mark.parametrize("T,ctx", [(1, 0), (8, 1), (2, 63), (5, 64), (6, 65), (7, 700)])
def test_fp8_layer_edges(T, ctx):
    cfg = synth.fp8_layer_config(T=T, ctx=ctx, gamma_jitter=0.1)
    err, kv_err, log, info = _run(cfg, T=T)
    assert err < gc.TOL[synth.WDT_FP8], err
    assert kv_err < 2e-2


def test_fp8_layer_is_deterministic():
    cfg = synth.fp8_layer_config(ctx=300)
    b = gc.Built(cfg)
    try:
        x = torch.randn((cfg.T, cfg.hidden), generator=torch.Generator().manual_seed(3)).cuda()
        outs = [b.layer(x)[0].clone() for _ in range(2)]
        assert torch.equal(outs[0], outs[1])
    finally:
        b.close()


def test_out_of_range_input_is_reported():
    """A residual entry of 1e5 cannot be an f16 GEMV input (largest finite value
    65504): the layer must stop with MK_ERR_RANGE rather than return infinities;
    after mk_reset the same state computes normal inputs again."""
    cfg = synth.fp8_layer_config(ctx=100, T=2)
    b = gc.Built(cfg)
    try:
        x = torch.randn((cfg.T, cfg.hidden), generator=torch.Generator().manual_seed(4)).cuda()
        good, _, _ = b.layer(x)
        good = good.clone()
        y = x.clone()
        y[1, 77] = 1e5
        out = torch.empty_like(y)
        mk.mk_layer_forward(b.st, 0, y, cfg.T, b.positions(cfg.T), b.kvargs.kv, out)
        assert mk.mk_get_status(b.st) == mk.MK_ERR_RANGE
        assert mk.mk_reset(b.st) == mk.MK_OK
        again, _, _ = b.layer(x)
        assert torch.equal(again, good)
    finally:
        b.close()


@pytest.mark.parametrize("T,ctx", [(6, 300), (8, 65536), (1, 0), (3, 65)])
def test_mxfp4_expert_layer(T, ctx):
    """FP8 attention and shared expert with MXFP4 routed experts (E2M1 codes,
    E8M0 1 x 32 scales), against the oracle's exact decoding of the same bytes."""
    cfg = synth.fp8_layer_config(T=T, ctx=ctx, expert_dtype=synth.WDT_MXFP4, gamma_jitter=0.1)
    err, kv_err, log, info = _run(cfg, T=T)
    assert err < gc.TOL[synth.WDT_FP8], err
    assert kv_err < 2e-2


@pytest.mark.parametrize("T,ctx", [(6, 300), (8, 65536), (1, 0), (3, 65), (2, 127)])
def test_fp8_kv_layer(T, ctx):
    """FP8 E4M3 KV cache with per-layer K and V scales: attention over the codes
    against the oracle's decoding of the same bytes, and the block's appended
    entries stored as nearest codes of value / scale."""
    cfg = synth.fp8_layer_config(T=T, ctx=ctx, kv_dtype=synth.WDT_FP8, kv_scales=(0.0125, 0.02),
                                 gamma_jitter=0.1)
    err, kv_err, log, info = _run(cfg, T=T)
    assert err < gc.TOL[synth.WDT_FP8], err
    assert kv_err <= 0.0, kv_err


def test_fp8_kv_scale_checks_and_noalloc_refusal():
    """A non-positive FP8 KV scale is refused before launch (MK_ERR_INVALID), and
    the allocation-free entry point, which takes no scales, refuses FP8 caches."""
    cfg = synth.fp8_layer_config(T=2, ctx=100, kv_dtype=synth.WDT_FP8, kv_scales=(0.0125, 0.02))
    b = gc.Built(cfg)
    try:
        x = torch.randn((2, cfg.hidden), generator=torch.Generator().manual_seed(5)).cuda()
        out = torch.empty_like(x)
        bad = mk.KVArgs(b.kv.k_pools, b.kv.v_pools, b.kv.page_table, b.kv.n_pages, [(0.0, 0.02)])
        r = mk.mk_layer_forward(b.st, 0, x, 2, b.positions(2), bad.kv, out, check=False)
        assert r == mk.MK_ERR_INVALID
        b.layer(x)     # the state is still usable with valid scales
        # refused before the entry point touches its device array
        r = mk.mk_layer_forward_noalloc(b.args.desc, b.args.layers[0], b.kv.k_pools[0], b.kv.v_pools[0],
                                        b.kv.page_table, b.kv.n_pages, x, 2, b.kv.ctx[0],
                                        b.positions(2), out, check=False)
        assert r == mk.MK_ERR_UNSUPPORTED
    finally:
        b.close()
