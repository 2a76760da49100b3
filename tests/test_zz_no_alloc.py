"""mk_layer_forward_noalloc: the allocation-free layer entry point, for callers
that cannot call cudaMalloc, must give the same result as mk_layer_forward.

It runs the same kernel with all of its state in one static device array, so the
test calls it twice in a row (the array keeps the previous call's contents) and
compares each result with the state-based entry point's.  This file is
collected last; it must pass alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from latency_moe_decode_persistent_gb300 import mk, synth
from tests import gpu_common as gc
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make_cfg", [lambda: synth.fp8_layer_config(ctx=300, T=6),
                                      lambda: synth.tiny_config(T=1)])
def test_noalloc_matches_layer_forward_twice(make_cfg):
    cfg = make_cfg()
    b = gc.Built(cfg)
    try:
        T = cfg.T
        x = torch.randn((T, cfg.hidden), generator=torch.Generator().manual_seed(17)).cuda()
        ref_out, ref_idx, ref_w = b.layer(x)
        kv = b.kv
        pos = b.positions(T)
        for call in range(2):
            out = torch.full_like(x, float("nan"))
            idx = torch.full((T, cfg.top_k), -1, dtype=torch.int32, device="cuda")
            w = torch.zeros((T, cfg.top_k), dtype=torch.float32, device="cuda")
            status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
            mk.mk_layer_forward_noalloc(b.args.desc, b.args.layers[0], kv.k_pools[0], kv.v_pools[0],
                                        kv.page_table, kv.n_pages, x, T, kv.ctx[0], pos, out, idx, w,
                                        status)
            torch.cuda.synchronize()
            assert int(status.item()) == mk.MK_OK, "call %d: device status %d" % (call, int(status.item()))
            # the same kernel on the same inputs, and its reductions are
            # order-independent integer sums: the results are bit for bit equal
            assert torch.equal(out, ref_out)
            assert torch.equal(idx, ref_idx)
            assert torch.equal(w, ref_w)
    finally:
        b.close()


def test_noalloc_refuses_a_ctx_that_differs_from_the_positions():
    # the host stages RoPE rows for positions ctx .. ctx+T-1 only; a launch whose
    # positions start elsewhere is refused on the device before any stage runs
    cfg = synth.fp8_layer_config(ctx=300, T=4)
    b = gc.Built(cfg)
    try:
        T = cfg.T
        x = torch.randn((T, cfg.hidden), generator=torch.Generator().manual_seed(19)).cuda()
        kv = b.kv
        out = torch.full_like(x, float("nan"))
        status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        mk.mk_layer_forward_noalloc(b.args.desc, b.args.layers[0], kv.k_pools[0], kv.v_pools[0],
                                    kv.page_table, kv.n_pages, x, T, kv.ctx[0] - 5, b.positions(T),
                                    out, None, None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == mk.MK_ERR_BAD_INPUT
        assert torch.isnan(out).all()
        # a matching call right after works on the same array
        mk.mk_layer_forward_noalloc(b.args.desc, b.args.layers[0], kv.k_pools[0], kv.v_pools[0],
                                    kv.page_table, kv.n_pages, x, T, kv.ctx[0], b.positions(T),
                                    out, None, None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == mk.MK_OK
        assert not torch.isnan(out).any()
    finally:
        b.close()


def test_noalloc_rejects_bad_arguments():
    cfg = synth.tiny_config()
    d = mk.ModelArgs(synth.make_model(cfg, "cpu"), 1, 4).desc
    x = torch.zeros((1, cfg.hidden), device="cuda")
    # T above max_T is refused on the host, before anything is launched
    s = mk.mk_layer_forward_noalloc(d, mk.mk_layer_weights(), 1, 1, 1, 1, x, 9, 0, 1, 1, check=False)
    assert s in (mk.MK_ERR_INVALID, mk.MK_ERR_UNSUPPORTED)
    assert mk.mk_last_error(None)
