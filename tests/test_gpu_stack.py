"""Full verify-step parity (mk_decode_step): logits, argmax, accepted count and
per-layer routing against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_persistent_gb300 import mk, synth
from tests import gpu_common as gc
from tests import helpers

pytestmark = pytest.mark.gpu


def mini_stack(**kw):
    c = synth.Config("mini_fp8_stack", 1024, 8, 2, 128, 64, 4, 256, n_layers=3, vocab=4096,
                     weight_dtype=synth.WDT_FP8, router_dtype=synth.WDT_BF16,
                     kv_dtype=synth.WDT_BF16, T=6, ctx=200, seed=21)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def make_drafts(b: gc.Built, d0: int, k: int, p_accept: float, seed: int):
    """Drafts d_1..d_k built left to right: the stack's own argmax with probability
    p_accept, else a uniform token (prefix passes run on the GPU path)."""
    rng = np.random.default_rng(seed)
    toks = [d0]
    for i in range(k):
        _, _, am, _ = b.step(toks, trace=False)
        a = int(am[i].item())
        toks.append(a if rng.random() < p_accept else int(rng.integers(0, b.cfg.vocab)))
    return toks


def compare_step(b: gc.Built, toks):
    logits, acc, am, trace = b.step(toks)
    cfg = b.cfg
    tr = trace.cpu().numpy()
    log = []
    dims = helpers.oracle_dims(cfg)
    layers = [helpers.layer_view(b.model, l) for l in range(cfg.n_layers)]
    kvs = [helpers.kv_view(b.kv, l) for l in range(cfg.n_layers)]
    r = oracle.stack_forward(toks, helpers.embed_fn(b.model), layers,
                             b.model.final_norm.cpu().numpy().astype(np.float64),
                             helpers.lm_head_lin(b.model), dims, kvs, b.kv.ctx[0],
                             route_hook_factory=lambda l: gc.tie_hook(tr[l], cfg.top_k, log),
                             kv_scales=helpers.kv_scales(b.kv))
    wt = b.wtrace.cpu().numpy()
    for l, info in enumerate(r["layers"]):
        gc.check_routing(info, tr[l], cfg.top_k, where="layer %d" % l)
        gc.check_weights(info, tr[l], wt[l], gc.WTOL[cfg.weight_dtype], where="layer %d" % l)
    lg = logits.cpu().numpy()
    err = helpers.rel_err(lg, r["logits"])
    ref = r["logits"]
    rms = np.sqrt(np.mean(ref ** 2))
    decisive = []
    for t in range(len(toks)):
        s = np.sort(ref[t])[::-1]
        dec = (s[0] - s[1]) > gc.GAP * rms
        decisive.append(dec)
        if dec:
            assert int(am[t]) == int(r["argmax"][t]), (t, int(am[t]), int(r["argmax"][t]))
    if all(decisive):
        assert acc == r["accepted"]
    return err, acc, r, log


def test_mini_stack_step():
    cfg = mini_stack()
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 17, cfg.T - 1, 0.83, seed=5)
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


@pytest.mark.parametrize("T,ctx", [(1, 0), (2, 64), (8, 129)])
def test_mini_stack_edges(T, ctx):
    cfg = mini_stack(T=T, ctx=ctx, gamma_jitter=0.1, seed=22 + T)
    b = gc.Built(cfg)
    try:
        toks = [int(v) for v in np.random.default_rng(T).integers(0, cfg.vocab, T)]
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


def test_mini_stack_mxfp4_experts():
    cfg = mini_stack(expert_dtype=synth.WDT_MXFP4, seed=24, hidden=1024, expert_inter=256)
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 33, cfg.T - 1, 0.83, seed=6)
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


def test_mini_stack_fp8_kv_cache():
    """FP8 E4M3 KV cache with a different (K, V) scale in every layer, through the
    whole verify step."""
    cfg = mini_stack(kv_dtype=synth.WDT_FP8, seed=25, ctx=700,
                     kv_scales=[(0.0125, 0.02), (0.03, 0.01), (0.02, 0.0125)])
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 35, cfg.T - 1, 0.83, seed=7)
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


def test_mini_stack_fp8_lm_head():
    """FP8 E4M3 LM head with 1x128 scales: logits, argmax and accept count against
    the oracle's exact decoding of the same codes."""
    cfg = mini_stack(lm_dtype=synth.WDT_FP8, seed=26)
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 36, cfg.T - 1, 0.83, seed=8)
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


def _sampling_near_boundary(lg, toks, temp, u, n_ref, tok_ref, eps=1e-5):
    """True when an accept test or the draw lies within eps of its decision
    boundary (in the fp64 reading of the same logits), where float32 may decide
    the other way."""
    for i in range(1, min(n_ref + 2, len(toks))):
        p = oracle.softmax_t(lg[i - 1], temp)
        if abs(float(u[i - 1]) - p[int(toks[i])]) < eps:
            return True
    p = oracle.softmax_t(lg[n_ref], temp)
    if n_ref < len(toks) - 1:
        p[int(toks[n_ref + 1])] = 0.0
    cum = np.cumsum(p) / p.sum()
    v = float(u[-1])
    lo = cum[tok_ref - 1] if tok_ref > 0 else 0.0
    return abs(v - lo) < eps or abs(cum[tok_ref] - v) < eps


@pytest.mark.parametrize("temp", [1.0, 0.6])
def test_mini_stack_sampling_verify(temp):
    """mk_decode_step_sample against the oracle's sampling rule applied to the
    GPU's own logits (the logits themselves are compared with the oracle by the
    argmax-path tests); decisions within 1e-5 of a boundary are skipped.  Then a
    temperature of 1e-3 must reproduce argmax verification."""
    cfg = mini_stack(seed=27)
    b = gc.Built(cfg)
    try:
        rng = np.random.default_rng(12)
        compared = 0
        for trial in range(10):
            toks = make_drafts(b, int(rng.integers(cfg.vocab)), cfg.T - 1, 0.83, seed=100 + trial)
            u = rng.uniform(size=cfg.T).astype(np.float32)
            n, tok, lg = b.step_sample(toks, temp, u)
            lg64 = lg.astype(np.float64)
            n_ref, tok_ref = oracle.sample_verify(lg64, toks, temp, u.astype(np.float64))
            if _sampling_near_boundary(lg64, toks, temp, u, n_ref, tok_ref):
                continue
            assert (n, tok) == (n_ref, tok_ref), (trial, n, tok, n_ref, tok_ref)
            compared += 1
        assert compared >= 8
        toks = make_drafts(b, 7, cfg.T - 1, 0.83, seed=5)
        _, acc, am, _ = b.step(toks, trace=False)
        n, tok, _ = b.step_sample(toks, 1e-3, np.full(cfg.T, 0.5, dtype=np.float32))
        assert n == acc and tok == int(am[acc].item())
    finally:
        b.close()


def test_mini_stack_all_drafts_accepted_and_deterministic():
    cfg = mini_stack(seed=31)
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 5, cfg.T - 1, 1.0, seed=1)
        l1, a1, am1, _ = b.step(toks, trace=False)
        l2, a2, am2, _ = b.step(toks, trace=False)
        assert torch.equal(l1, l2) and a1 == a2 and torch.equal(am1, am2)
        assert a1 == cfg.T - 1
        st = mk.mk_get_stats(b.st)
        assert st.fused == 1 and st.launches_per_step == 1 and st.steps >= 2
    finally:
        b.close()


def test_host_buffer_entry_matches_device_entry():
    cfg = mini_stack(seed=41)
    b = gc.Built(cfg)
    try:
        toks = [3, 9, 27, 81, 243, 729]
        lg, acc, am, _ = b.step(toks, trace=False)
        h_tok = torch.tensor(toks, dtype=torch.int32).pin_memory()
        h_pos = torch.arange(b.kv.ctx[0], b.kv.ctx[0] + len(toks), dtype=torch.int32).pin_memory()
        h_lg = torch.empty((len(toks), cfg.vocab), dtype=torch.float32).pin_memory()
        h_acc = torch.zeros(1, dtype=torch.int32).pin_memory()
        h_am = torch.zeros(len(toks), dtype=torch.int32).pin_memory()
        mk.mk_decode_step_host(b.st, h_tok, len(toks), h_pos, b.kvargs.kv, h_lg, h_acc, h_am)
        assert torch.equal(h_lg, lg.cpu()) and int(h_acc) == acc and torch.equal(h_am, am.cpu())
    finally:
        b.close()


@pytest.mark.slow
def test_full_43_layer_stack():
    """The 43-layer FP8 stack, vocab 129280, T 6, ctx 2048, drafts at 0.83."""
    cfg = synth.stack_config()
    b = gc.Built(cfg)
    try:
        toks = make_drafts(b, 1000, cfg.T - 1, 0.83, seed=3)
        err, acc, r, log = compare_step(b, toks)
        assert err < gc.TOL[synth.WDT_FP8], err
    finally:
        b.close()


def _full_width_stack(**kw):
    """3 layers of the 43-layer stack's full layer shape (H 4096, 384 experts
    top-8, I 512), vocab 4096: the routed stages then hold several hundred
    items per input chunk, more than the CTAs of a chunk.  At ctx 8192 each
    attention split holds several KV pages, which the warps of a split share."""
    c = synth.Config("full_width_3layer", 4096, 32, 4, 128, 384, 8, 512, n_layers=3, vocab=4096,
                     weight_dtype=synth.WDT_FP8, router_dtype=synth.WDT_BF16,
                     kv_dtype=synth.WDT_BF16, T=8, ctx=300, seed=52)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("make_cfg", [lambda: mini_stack(seed=51), _full_width_stack,
                                      lambda: _full_width_stack(ctx=8192, seed=53)])
def test_block_verification_is_batch_invariant(make_cfg):
    """Block verification = sequential decode, bit for bit on the GPU: the logits
    of position i from a step over the first i+1 tokens equal row i of the full
    step (the work split of the routed-expert stages changes with the set of
    distinct experts, so this pins that a token's result does not depend on the
    other tokens of the block).  The pages' greedy byte-for-byte gate, adapted."""
    cfg = make_cfg()
    b = gc.Built(cfg)
    try:
        toks = [int(v) for v in np.random.default_rng(9).integers(0, cfg.vocab, cfg.T)]
        full, _, am_full, _ = b.step(toks, trace=False)
        for n in range(1, cfg.T):
            part, _, am, _ = b.step(toks[:n], trace=False)
            assert torch.equal(part, full[:n]), "prefix of %d tokens differs" % n
            assert torch.equal(am, am_full[:n])
    finally:
        b.close()


def test_decode_batch_matches_single_streams():
    """mk_decode_batch over two streams with different contexts gives each stream
    exactly the result of mk_decode_step on that stream alone."""
    cfg = mini_stack(seed=61)
    ctxs = [200, 131]
    b = gc.Built(cfg, ctxs=ctxs)
    try:
        S, T, V = len(ctxs), cfg.T, cfg.vocab
        rng = np.random.default_rng(4)
        toks = torch.tensor(rng.integers(0, V, (S, T)), dtype=torch.int32, device="cuda")
        pos = torch.stack([torch.arange(c, c + T, dtype=torch.int32) for c in ctxs]).cuda()
        logits = torch.empty((S, T, V), dtype=torch.float32, device="cuda")
        acc = torch.zeros(S, dtype=torch.int32, device="cuda")
        am = torch.zeros((S, T), dtype=torch.int32, device="cuda")
        mk.mk_decode_batch(b.st, S, toks, T, pos, b.kvargs.kv, logits, acc, am)
        assert mk.mk_get_status(b.st) == mk.MK_OK
        for s in range(S):
            kv1 = mk.KVArgs(b.kv.k_pools, b.kv.v_pools, b.kv.page_table[s], b.kv.n_pages)
            lg = torch.empty((T, V), dtype=torch.float32, device="cuda")
            a1 = torch.zeros(1, dtype=torch.int32, device="cuda")
            m1 = torch.zeros(T, dtype=torch.int32, device="cuda")
            mk.mk_decode_step(b.st, toks[s].contiguous(), T, pos[s].contiguous(), kv1.kv, lg, a1, m1)
            assert mk.mk_get_status(b.st) == mk.MK_OK
            assert torch.equal(lg, logits[s]) and int(a1) == int(acc[s]) and torch.equal(m1, am[s])
        # stream 1 against the oracle as well (its own page-table row and context)
        dims = helpers.oracle_dims(cfg)
        layers = [helpers.layer_view(b.model, l) for l in range(cfg.n_layers)]
        kvs = [helpers.kv_view(b.kv, l, stream=1) for l in range(cfg.n_layers)]
        r = oracle.stack_forward(toks[1].tolist(), helpers.embed_fn(b.model), layers,
                                 b.model.final_norm.cpu().numpy().astype(np.float64),
                                 helpers.lm_head_lin(b.model), dims, kvs, ctxs[1])
        assert helpers.rel_err(logits[1].cpu().numpy(), r["logits"]) < gc.TOL[synth.WDT_FP8]
    finally:
        b.close()


def test_timeout_is_reported_and_reset_recovers():
    """Failure path without a GPU fault: CTA 0 withholds one grid-barrier arrival
    (a test hook), every other CTA's bounded wait runs out after timeout_ms, the
    step reports MK_ERR_TIMEOUT, later steps refuse to run until mk_reset, and
    after mk_reset the state computes the same logits as before."""
    cfg = mini_stack(seed=71)
    b = gc.Built(cfg, timeout_ms=50)
    try:
        toks = [7, 8, 9, 10, 11, 12]
        ref, acc_ref, _, _ = b.step(toks, trace=False)
        ref = ref.clone()
        mk.mk_debug_skip_barrier(b.st, 2)
        tok = torch.tensor(toks, dtype=torch.int32, device="cuda")
        logits = torch.empty_like(ref)
        acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        pos = b.positions(len(toks))
        mk.mk_decode_step(b.st, tok, len(toks), pos, b.kvargs.kv, logits, acc, None)
        assert mk.mk_get_status(b.st) == mk.MK_ERR_TIMEOUT
        mk.mk_debug_skip_barrier(b.st, 0)
        mk.mk_decode_step(b.st, tok, len(toks), pos, b.kvargs.kv, logits, acc, None)
        assert mk.mk_get_status(b.st) == mk.MK_ERR_TIMEOUT   # sticky until reset
        assert mk.mk_reset(b.st) == mk.MK_OK
        again, acc2, _, _ = b.step(toks, trace=False)
        assert torch.equal(again, ref) and acc2 == acc_ref
    finally:
        b.close()


def test_concurrency_streams_match_their_own_oracle_runs():
    """The concurrency workload's shape at reduced depth: 4 streams, each with its
    own context drawn from U[1024, 8192] (seed 4) and T = 6, over a 3-layer stack
    of the full-width FP8 layer (hidden 4096, 384 experts top-8 + shared, vocab
    129280), verified in one mk_decode_batch call.  Each stream is then run alone
    with the routing trace on (its logits must equal the batch's bit for bit) and
    compared with its own oracle run: routing and weights per layer, logits,
    decisive argmax and the accept count."""
    cfg = synth.stack_config(n_layers=3, seed=4)
    ctxs = [int(c) for c in np.random.default_rng(4).integers(1024, 8193, 4)]
    b = gc.Built(cfg, ctxs=ctxs)
    try:
        S, T, V, K = len(ctxs), cfg.T, cfg.vocab, cfg.top_k
        toks = np.random.default_rng(44).integers(0, V, (S, T))
        dims = helpers.oracle_dims(cfg)
        layers = [helpers.layer_view(b.model, l) for l in range(cfg.n_layers)]
        fn = b.model.final_norm.cpu().numpy().astype(np.float64)
        lm = helpers.lm_head_lin(b.model)
        # oracle inputs before the step appends K/V (positions >= ctx only)
        kvs = [[helpers.kv_view(b.kv, l, stream=s) for l in range(cfg.n_layers)] for s in range(S)]
        tok = torch.tensor(toks, dtype=torch.int32, device="cuda")
        pos = torch.stack([torch.arange(c, c + T, dtype=torch.int32) for c in ctxs]).cuda()
        logits = torch.empty((S, T, V), dtype=torch.float32, device="cuda")
        acc = torch.zeros(S, dtype=torch.int32, device="cuda")
        am = torch.zeros((S, T), dtype=torch.int32, device="cuda")
        mk.mk_decode_batch(b.st, S, tok, T, pos, b.kvargs.kv, logits, acc, am)
        assert mk.mk_get_status(b.st) == mk.MK_OK, mk.mk_last_error(b.st)
        for s in range(S):
            kv1 = mk.KVArgs(b.kv.k_pools, b.kv.v_pools, b.kv.page_table[s], b.kv.n_pages)
            tr = torch.full((cfg.n_layers, T, K), -1, dtype=torch.int32, device="cuda")
            wt = torch.zeros((cfg.n_layers, T, K), dtype=torch.float32, device="cuda")
            lg1 = torch.empty((T, V), dtype=torch.float32, device="cuda")
            a1 = torch.zeros(1, dtype=torch.int32, device="cuda")
            m1 = torch.zeros(T, dtype=torch.int32, device="cuda")
            mk.mk_set_routing_trace(b.st, tr, wt)
            mk.mk_decode_step(b.st, tok[s].contiguous(), T, pos[s].contiguous(), kv1.kv, lg1, a1, m1)
            assert mk.mk_get_status(b.st) == mk.MK_OK, mk.mk_last_error(b.st)
            mk.mk_set_routing_trace(b.st, None, None)
            assert torch.equal(lg1, logits[s]) and int(a1) == int(acc[s]) and torch.equal(m1, am[s])
            trn, wtn = tr.cpu().numpy(), wt.cpu().numpy()
            log = []
            r = oracle.stack_forward(toks[s].tolist(), helpers.embed_fn(b.model), layers, fn, lm,
                                     dims, kvs[s], ctxs[s],
                                     route_hook_factory=lambda l: gc.tie_hook(trn[l], K, log))
            for l, info in enumerate(r["layers"]):
                gc.check_routing(info, trn[l], K, where="stream %d layer %d" % (s, l))
                gc.check_weights(info, trn[l], wtn[l], gc.WTOL[synth.WDT_FP8],
                                 where="stream %d layer %d" % (s, l))
            ref = r["logits"]
            assert helpers.rel_err(logits[s].cpu().numpy(), ref) < gc.TOL[synth.WDT_FP8], s
            rms = np.sqrt(np.mean(ref ** 2))
            dec = []
            for t in range(T):
                srt = np.sort(ref[t])[::-1]
                dec.append(srt[0] - srt[1] > gc.GAP * rms)
                if dec[-1]:
                    assert int(am[s, t]) == int(r["argmax"][t]), (s, t)
            if all(dec):
                assert int(acc[s]) == r["accepted"], s
    finally:
        b.close()
