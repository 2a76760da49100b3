"""Exact ties on the GPU path: equal router keys go to the lower expert index,
equal logits go to the lowest token id, as the oracle's rules state.

Ties are built so that both sides see exactly equal values: a zero router
matrix makes every sigmoid score exactly 0.5 (the keys are then 0.5 + bias), and
two identical LM-head rows give two bitwise-equal logits on the GPU, where
every output row goes through the same arithmetic."""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_persistent_gb300 import mk, synth
from tests import gpu_common as gc
from tests import helpers

pytestmark = pytest.mark.gpu


def _mini_layer(**kw):
    c = synth.Config("mini_fp8_layer", 1024, 8, 2, 128, 64, 4, 256, weight_dtype=synth.WDT_FP8,
                     router_dtype=synth.WDT_BF16, kv_dtype=synth.WDT_BF16, T=4, ctx=200, seed=81)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _tied_bias(E, seed):
    """Distinct biases 0.2/E apart (more than the 1e-3 near-tie band), then the
    two largest made equal and the 4th and 5th largest made equal."""
    b = np.linspace(-0.1, 0.1, E)[np.random.default_rng(seed).permutation(E)]
    order = np.argsort(-b, kind="stable")
    b[order[1]] = b[order[0]]
    b[order[4]] = b[order[3]]
    return b.astype(np.float32), order


@pytest.mark.parametrize("make_cfg", [_mini_layer,
                                      lambda: synth.tiny_config(T=3, ctx=70, top_k=4, bias_range=0.1)])
def test_equal_router_keys_go_to_the_lower_index(make_cfg):
    cfg = make_cfg()
    b = gc.Built(cfg)
    try:
        L = b.model.layers[0]
        L.w_router.data.zero_()
        bias, order = _tied_bias(cfg.n_experts, 5)
        L.router_bias.copy_(torch.from_numpy(bias))
        x = torch.randn((cfg.T, cfg.hidden), generator=torch.Generator().manual_seed(2)).cuda()
        out, idx, w = b.layer(x)
        K = cfg.top_k
        # every token: the two tied leaders in index order, then the 3rd, then
        # the lower index of the pair tied at the K-th place
        r = [int(e) for e in order[:5]]
        want = [min(r[0], r[1]), max(r[0], r[1]), r[2], min(r[3], r[4])][:K]
        ref, info = gc.oracle_layer(b, x.cpu().numpy())
        for t in range(cfg.T):
            assert idx[t].tolist() == want, (t, idx[t].tolist(), want)
            assert info["idx"][t].tolist() == want          # the oracle's rule agrees
            assert torch.equal(w[t], torch.full((K,), 1.0 / K, device="cuda"))
        assert helpers.rel_err(out.cpu().numpy(), ref) < gc.TOL[cfg.weight_dtype]
    finally:
        b.close()


def test_equal_logits_go_to_the_lowest_token_id():
    cfg = synth.Config("mini_fp8_stack", 1024, 8, 2, 128, 64, 4, 256, n_layers=1, vocab=4096,
                       weight_dtype=synth.WDT_FP8, router_dtype=synth.WDT_BF16,
                       kv_dtype=synth.WDT_BF16, T=3, ctx=130, seed=83)
    b = gc.Built(cfg)
    try:
        toks = [11, 22, 33]
        dims = helpers.oracle_dims(cfg)
        layers = [helpers.layer_view(b.model, 0)]
        kvs = [helpers.kv_view(b.kv, 0)]
        fn = b.model.final_norm.cpu().numpy().astype(np.float64)
        r0 = oracle.stack_forward(toks, helpers.embed_fn(b.model), layers, fn,
                                  helpers.lm_head_lin(b.model), dims, kvs, cfg.ctx)
        # rows 1000 and 3000 both become token 1's normalised final hidden
        # direction: its logit there is |xf| (about 32) against O(1) elsewhere
        xf = oracle.rmsnorm(r0["x_final"], fn, cfg.rms_eps)[1]
        row = torch.from_numpy(xf / np.linalg.norm(xf)).to(torch.bfloat16)
        lo, hi = 1000, 3000
        b.model.lm_head[lo] = row.cuda()
        b.model.lm_head[hi] = row.cuda()
        logits, acc, am, _ = b.step(toks, trace=False)
        assert int(am[1]) == lo
        assert logits[1, lo].item() == logits[1, hi].item()
        for t in range(cfg.T):
            mx = logits[t].max()
            assert int(am[t]) == int(torch.nonzero(logits[t] == mx)[0])
        r = oracle.stack_forward(toks, helpers.embed_fn(b.model), layers, fn,
                                 helpers.lm_head_lin(b.model), dims, kvs, cfg.ctx)
        assert helpers.rel_err(logits.cpu().numpy(), r["logits"]) < gc.TOL[cfg.weight_dtype]
        if r["logits"][1, lo] == r["logits"][1, hi]:
            assert int(r["argmax"][1]) == lo
    finally:
        b.close()
