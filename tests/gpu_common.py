"""Shared pieces of the GPU parity tests: run the C-ABI path, run the oracle on
the same seeded inputs, compare by the rules of the verify-step contract."""
import numpy as np
import torch

import oracle
from latency_moe_decode_persistent_gb300 import mk, synth
from tests import helpers

GAP = 1e-3            # decisive routing / argmax gap
TOL = {synth.WDT_F32: 1e-4, synth.WDT_BF16: 2e-2, synth.WDT_FP8: 6e-2}
# routing weights where the selection is decisive: the kernel forms them in
# fp32 from the same sigmoid scores, so they follow the oracle far more closely
# than the hidden state does (a router normalising the biased keys s + b
# instead of s would move each weight by about 1e-2)
WTOL = {synth.WDT_F32: 1e-5, synth.WDT_BF16: 1e-3, synth.WDT_FP8: 1e-3}


class Built:
    """A model + KV cache on the GPU and a library state bound to them."""

    def __init__(self, cfg, ctxs=None, T=None, max_T=None, device="cuda", timeout_ms=0):
        self.cfg = cfg
        self.model = synth.make_model(cfg, device)
        self.kv = synth.make_kv(cfg, device, ctxs=ctxs, T=T if T is not None else cfg.T)
        self.max_T = max_T or max(cfg.T, T or 0)
        self.args = mk.ModelArgs(self.model, self.max_T, self.kv.max_pages, timeout_ms)
        self.st = mk.mk_create(self.args.desc, self.args.weights)
        self.kvargs = mk.KVArgs(self.kv.k_pools, self.kv.v_pools, self.kv.page_table,
                                self.kv.n_pages, self.kv.scales)

    def close(self):
        mk.mk_destroy(self.st)
        self.st = None

    def positions(self, T, stream=0):
        c = self.kv.ctx[stream]
        return torch.arange(c, c + T, dtype=torch.int32, device="cuda")

    def layer(self, x, l=0, T=None):
        T = x.shape[0] if T is None else T
        out = torch.empty_like(x)
        K = self.cfg.top_k
        idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, K), dtype=torch.float32, device="cuda")
        mk.mk_layer_forward(self.st, l, x, T, self.positions(T), self.kvargs.kv, out, idx, w)
        st = mk.mk_get_status(self.st)
        assert st == mk.MK_OK, mk.mk_last_error(self.st)
        return out, idx, w

    def step(self, tokens, trace=True):
        T = len(tokens)
        tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
        logits = torch.empty((T, self.cfg.vocab), dtype=torch.float32, device="cuda")
        acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        am = torch.empty(T, dtype=torch.int32, device="cuda")
        tr = None
        if trace:
            tr = torch.full((self.cfg.n_layers, T, self.cfg.top_k), -1, dtype=torch.int32,
                            device="cuda")
            self.wtrace = torch.full((self.cfg.n_layers, T, self.cfg.top_k), float("nan"),
                                     dtype=torch.float32, device="cuda")
            mk.mk_set_routing_trace(self.st, tr, self.wtrace)
        mk.mk_decode_step(self.st, tok, T, self.positions(T), self.kvargs.kv, logits, acc, am)
        st = mk.mk_get_status(self.st)
        assert st == mk.MK_OK, mk.mk_last_error(self.st)
        if trace:
            mk.mk_set_routing_trace(self.st, None, None)
        return logits, int(acc.item()), am, tr


    def step_sample(self, tokens, temperature, uniforms):
        """mk_decode_step_sample: (accepted, drawn token, logits as numpy)."""
        T = len(tokens)
        tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
        u = torch.tensor(np.asarray(uniforms, dtype=np.float32), device="cuda")
        logits = torch.empty((T, self.cfg.vocab), dtype=torch.float32, device="cuda")
        acc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        mk.mk_decode_step_sample(self.st, tok, T, self.positions(T), self.kvargs.kv, temperature, u,
                                 logits, acc, out)
        st = mk.mk_get_status(self.st)
        assert st == mk.MK_OK, mk.mk_last_error(self.st)
        return int(acc.item()), int(out.item()), logits.cpu().numpy()


def kth_gap(key_row, K):
    s = np.sort(key_row)[::-1]
    return s[K - 1] - s[K] if len(s) > K else np.inf


def valid_choice(key_row, chosen, K):
    """A selection is valid if it holds every expert whose key beats the K-th key by
    more than GAP and no expert whose key falls short of it by more than GAP."""
    s = np.sort(key_row)[::-1]
    kth = s[K - 1]
    ch = set(int(e) for e in chosen)
    if len(ch) != K:
        return False
    must = set(np.nonzero(key_row > kth + GAP)[0].tolist())
    cant = set(np.nonzero(key_row < kth - GAP)[0].tolist())
    return must <= ch and not (ch & cant)


def tie_hook(gpu_idx_layer, K, log):
    """Oracle route hook: on a near tie (K-th/(K+1)-th key gap <= GAP) where the
    GPU's selection is a valid choice, continue with the GPU's selection so that
    later computation compares like with like.  Each use is logged."""
    def hook(t, key_row, idx_row):
        g = np.asarray(gpu_idx_layer[t])
        if set(g.tolist()) == set(int(v) for v in idx_row):
            return None
        if kth_gap(key_row, K) <= GAP and valid_choice(key_row, g, K):
            log.append((t, sorted(g.tolist()), sorted(int(v) for v in idx_row)))
            return g
        return None
    return hook


def oracle_layer(b: Built, x, l=0, gpu_idx=None, log=None):
    cfg = b.cfg
    dims = helpers.oracle_dims(cfg)
    lv = helpers.layer_view(b.model, l)
    kc, vc = helpers.kv_view(b.kv, l)
    hook = tie_hook(gpu_idx, cfg.top_k, log if log is not None else []) if gpu_idx is not None else None
    return oracle.layer_forward(np.asarray(x, dtype=np.float64), lv, dims, kc, vc, b.kv.ctx[0], hook,
                                kv_scale=helpers.kv_scales(b.kv)[l])


def check_routing(info, gpu_idx, K, where=""):
    """Exact match where the oracle's selection is decisive, validity elsewhere."""
    T = gpu_idx.shape[0]
    for t in range(T):
        g = set(int(v) for v in gpu_idx[t])
        o = set(int(v) for v in info["idx"][t])
        if kth_gap(info["key"][t], K) > GAP:
            assert g == o, "%s token %d: gpu %s oracle %s" % (where, t, sorted(g), sorted(o))
        else:
            assert valid_choice(info["key"][t], list(g), K), "%s token %d invalid tie choice" % (where, t)


def check_weights(info, gpu_idx, gpu_w, wtol, where=""):
    """Routing weights of every token whose GPU selection equals the oracle's (all
    decisive tokens, and near ties where the oracle took the GPU's choice): each
    expert's weight within wtol of the oracle's.  Returns the largest difference."""
    worst = 0.0
    for t in range(gpu_idx.shape[0]):
        o = {int(e): float(info["w"][t, j]) for j, e in enumerate(info["idx"][t])}
        g = [int(e) for e in gpu_idx[t]]
        if set(g) != set(o):
            continue
        for j, e in enumerate(g):
            d = abs(float(gpu_w[t, j]) - o[e])
            worst = max(worst, d)
            assert d <= wtol, "%s token %d expert %d: gpu w %.6f oracle %.6f" % (
                where, t, e, float(gpu_w[t, j]), o[e])
    return worst
