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
        tol = gc.TOL[cfg.weight_dtype]
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
            assert helpers.rel_err(out.cpu().numpy(), ref_out.cpu().numpy()) <= tol
            assert torch.equal(idx, ref_idx)
            assert torch.allclose(w, ref_w, rtol=0, atol=tol)
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
