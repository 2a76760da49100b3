"""Single-layer parity of the CUDA path (mk_layer_forward) against the fp64 oracle
on the three single-layer workloads and on edge shapes."""
import numpy as np
import pytest
import torch

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


def _appended_err(b, info, l, T):
    kv = b.kv
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
