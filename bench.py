#!/usr/bin/env python3
"""Verify-step benchmark of the persistent megakernel (one JSON line on stdout).

Workload: the 43-layer FP8 MoE stack (hidden 4096, 32/4 heads of 128, 384
experts top-8 + 1 shared, expert width 512, vocab 129280, bf16 embedding and LM
head), one stream, T = 6 (d_0 + 5 drafts built at 0.83 per-position agreement),
2048 cached positions in 64-token bf16 pages; synthetic seeded weights (seed 3).

A step is one mk_decode_step: every stage of the hot path in one launch.  The
per-step weight stream (~16 GB) is far larger than the 129 MB L2, so no flush is
needed between timed iterations.  `value` is tokens/s = (mean accepted + 1) x
steps/s with the inputs resident in HBM; `e2e` is the same metric through
mk_decode_step_host with pinned host buffers (token/position upload and
logits/argmax/accept download inside the timed region).

`--impl reference` times the fp64 oracle (oracle/) on the host cores instead.
With N > 1 GPUs (torchrun) every rank runs an independent replica of the step
for its own stream ("replicas only": the step has no data-parallel split); value
is the sum of tokens over ranks divided by the slowest rank's time.
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-step µs & 1-stream tok/s (43-layer FP8, T=6); HBM GB/s vs roofline"
WORKLOAD = ("43-layer FP8 (e4m3, 1x128 scales) MoE stack: H 4096, 32 q / 4 kv heads x 128, "
            "384 experts top-8 + 1 shared, I 512, vocab 129280 (bf16 embed/LM head); "
            "1 stream, T=6 (k=5 drafts, 0.83 agreement), ctx 2048 bf16 KV in 64-token pages; seed 3")


def workload_of(cfg):
    """The workload string of a run: the default one, or the same stack with the
    layer count, block size or routed-expert format the run overrode."""
    w = WORKLOAD
    if getattr(cfg, "routed_dtype", cfg.weight_dtype) == 3:
        w = w.replace("384 experts top-8", "384 MXFP4 experts (e2m1, 1x32 e8m0 scales) top-8")
    if cfg.kv_dtype == 2:
        w = w.replace("bf16 KV", "FP8 e4m3 KV (per-layer K/V scales %g/%g)" % tuple(cfg.kv_scales))
    if cfg.ctx != 2048:
        w = w.replace("ctx 2048", "ctx %d" % cfg.ctx)
    if cfg.lm_dtype == 2:
        w = w.replace("(bf16 embed/LM head)", "(bf16 embed, FP8 e4m3 1x128 LM head)")
    if cfg.n_layers == 43 and cfg.T == 6:
        return w
    return w.replace("43-layer", "%d-layer" % cfg.n_layers).replace(
        "T=6 (k=5 drafts", "T=%d (k=%d drafts" % (cfg.T, cfg.T - 1))


def variant_kw(args, synth):
    """Config overrides of the routed-expert format, KV format and context."""
    kw = {}
    if args.experts == "mxfp4":
        kw["expert_dtype"] = synth.WDT_MXFP4
    if args.kv == "fp8":
        kw["kv_dtype"] = synth.WDT_FP8
        kw["kv_scales"] = FP8_KV_SCALES
    if args.ctx:
        kw["ctx"] = args.ctx
    if args.lm == "fp8":
        kw["lm_dtype"] = synth.WDT_FP8
    return kw


FP8_KV_SCALES = (0.0125, 0.0125)   # value = code x scale: N(0, 1) entries span about +-400 codes


def rank_info():
    r = int(os.environ.get("RANK", "0"))
    w = int(os.environ.get("WORLD_SIZE", "1"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return r, w, lr


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def _code_only(text):
    """C++ source without its comments and with whitespace collapsed: what the
    compiled kernel depends on, so that editing a comment keeps a stored figure."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("mk_kernel.cu", "mk_internal.h", "mk_api.cu"):
        with open(os.path.join(ROOT, "latency_moe_decode_persistent_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic():
    """Per-launch DRAM bytes of the step kernel from the committed ncu summary,
    only if it was captured on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "mk_step_kernel_traffic.txt")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("traffic_bytes_per_launch_full_workload")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [l.strip().split(",") for l in open(self.f.name) if l.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except Exception:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def algorithmic_bytes(cfg, distinct_per_step, ctx):
    """HBM bytes a step must move at minimum: every weight byte it uses once (the
    distinct routed experts counted on the device), the KV cache read and the
    block's K/V write, the embedding rows, and the logits written."""
    H, I, E, d = cfg.hidden, cfg.expert_inter, cfg.n_experts, cfg.head_dim
    nqkv = cfg.qkv_rows
    fp8 = lambda rows, cols: rows * cols + (cols // 128) * rows * 4
    mxfp4 = lambda rows, cols: rows * cols // 2 + (cols // 32) * rows
    shared = fp8(I, H) * 2 + fp8(H, I)
    routed = shared if getattr(cfg, "routed_dtype", cfg.weight_dtype) != 3 else mxfp4(I, H) * 2 + mxfp4(H, I)
    expert = routed
    kv_es = 1 if cfg.kv_dtype == 2 else 2
    per_layer = (fp8(nqkv, H) + fp8(H, cfg.n_q_heads * d) + E * H * 2 + E * 4 + 2 * H * 4
                 + (shared if cfg.n_shared else 0)
                 + ctx * cfg.n_kv_heads * d * 2 * kv_es + cfg.T * cfg.n_kv_heads * d * 2 * kv_es)
    total = cfg.n_layers * per_layer + distinct_per_step * expert
    lm = fp8(cfg.vocab, H) if cfg.lm_dtype == 2 else cfg.vocab * H * 2
    total += cfg.T * H * 2 + H * 4 + lm + cfg.T * cfg.vocab * 4
    return total


def oracle_sample(model, kv, cfg, toks, layers_to_time, ref_lm=True):
    """Time the oracle on `layers_to_time` layers (+ optionally the LM head) with
    the weights staged in host memory beforehand.  Returns (per-layer seconds,
    lm seconds)."""
    import numpy as np
    import oracle
    from tests import helpers
    dims = helpers.oracle_dims(cfg)
    x = helpers.embed_fn(model)(np.asarray(toks))
    cache = {}
    per = []
    for l in layers_to_time:
        lv = helpers.layer_view(model, l, expert_cache=cache)
        kc, vc = helpers.kv_view(kv, l)
        ksc = helpers.kv_scales(kv)[l]
        oracle.layer_forward(x, lv, dims, kc, vc, kv.ctx[0], kv_scale=ksc)   # staging pass (untimed)
        t0 = time.perf_counter()
        y, _ = oracle.layer_forward(x, lv, dims, kc, vc, kv.ctx[0], kv_scale=ksc)
        per.append(time.perf_counter() - t0)
        x = y
    lm_s = 0.0
    if ref_lm:
        lm = helpers.lm_head_lin(model)
        fn = model.final_norm.cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        lg = oracle.linear(lm, oracle.rmsnorm(x, fn, cfg.rms_eps))
        oracle.argmax_lowest(lg)
        lm_s = time.perf_counter() - t0
    return per, lm_s


P_AGREE = 0.83       # per-position probability that a draft is the stack's own argmax
DRAFT_BLOCKS = 256   # independent draft blocks; timed step i verifies block i % DRAFT_BLOCKS


def draft_plan(n_blocks, k, vocab, seed):
    """The seeded draws behind the draft blocks: per block the last accepted
    token d_0 and, for each of the k draft positions, whether the draft copies
    the stack's argmax (probability P_AGREE) and the uniform token used if not."""
    import numpy as np
    rng = np.random.default_rng(seed)
    plan = []
    for _ in range(n_blocks):
        d0 = int(rng.integers(0, vocab))
        agree = rng.random(k) < P_AGREE
        rnd = rng.integers(0, vocab, k)
        plan.append((d0, [bool(a) for a in agree], [int(r) for r in rnd]))
    return plan


def planned_accepts(plan):
    """Accepted drafts of each block as its draws fix them: a draft that copies
    the argmax is accepted, and a uniform token matches the argmax only with
    probability 1/vocab, so the count is the run of leading agreements."""
    out = []
    for _, agree, _ in plan:
        n = 0
        while n < len(agree) and agree[n]:
            n += 1
        out.append(n)
    return out


def tokens_per_step_of(plan, steps=None):
    """Mean tokens per verify step (accepted + 1) over `steps` steps that cycle
    through the plan's blocks in order (default: every block once)."""
    acc = planned_accepts(plan)
    steps = len(acc) if steps is None else steps
    return sum(acc[i % len(acc)] for i in range(steps)) / float(steps) + 1.0


def build_drafts(step_fn, plan_block):
    """Drafts d_1..d_k left to right: d_i is the argmax after d_0..d_{i-1} (from
    an untimed prefix pass) when the block's draw says so, else its uniform token."""
    d0, agree, rnd = plan_block
    toks = [d0]
    for i in range(len(agree)):
        am = step_fn(toks)
        toks.append(int(am[i]) if agree[i] else rnd[i])
    return toks


def reduce_over_ranks(mean_ms, tok_per_step, e2e_s, e2e_tok, distributed):
    """Whole-job figures of the replicas: the slowest rank's step time, and tokens
    summed over ranks divided by that time (device-timed and end to end).  Rank
    timings meet through the process group's CPU backend; no data-path
    collective is involved.  Returns (slowest ms, tok/s, e2e tok/s)."""
    if not distributed:
        return mean_ms, tok_per_step / (mean_ms / 1e3), e2e_tok
    import torch
    import torch.distributed as dist
    t = torch.tensor([mean_ms, tok_per_step, e2e_s, e2e_tok], dtype=torch.float64)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    slow_ms = float(mx[0])
    return slow_ms, float(sm[1]) / (slow_ms / 1e3), float(sm[1]) / float(mx[2])


def run_mk(args):
    import torch
    from latency_moe_decode_persistent_gb300 import mk, synth
    rank, world, lrank = rank_info()
    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    kw = {}
    if args.layers:
        kw["n_layers"] = args.layers
    if args.T:
        kw["T"] = args.T
    kw.update(variant_kw(args, synth))
    cfg = synth.stack_config(**kw)
    t_gen = time.perf_counter()
    model = synth.make_model(cfg, dev)
    kv = synth.make_kv(cfg, dev)
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen
    margs = mk.ModelArgs(model, cfg.T, kv.max_pages)
    st = mk.mk_create(margs.desc, margs.weights)
    kva = mk.KVArgs(kv.k_pools, kv.v_pools, kv.page_table, kv.n_pages, kv.scales)
    T, V = cfg.T, cfg.vocab
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    pos = torch.arange(cfg.ctx, cfg.ctx + T, dtype=torch.int32, device=dev)
    logits = torch.empty((T, V), dtype=torch.float32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    am = torch.zeros(T, dtype=torch.int32, device=dev)

    def step_prefix(toks):
        n = len(toks)
        tk = torch.tensor(toks, dtype=torch.int32, device=dev)
        mk.mk_decode_step(st, tk, n, pos[:n], kva.kv, logits, acc, am, sh)
        stream.synchronize()
        return am[:n].cpu().tolist()

    # draft blocks: the stack's own argmax with probability 0.83 per position,
    # else a uniform token; every block has its own d_0 and draws (seed 3 + rank)
    plan = draft_plan(DRAFT_BLOCKS, T - 1, V, seed=3 + rank)
    blocks = [build_drafts(step_prefix, b) for b in plan]
    tok_all = torch.tensor(blocks, dtype=torch.int32, device=dev)     # [blocks][T]
    nb = len(blocks)

    def one(i=0):
        mk.mk_decode_step(st, tok_all[i % nb], T, pos, kva.kv, logits, acc, am, sh)

    # one verify step of every block (untimed): the tokens per step of the
    # workload, as the device counts accepted drafts
    v0 = mk.mk_get_stats(st)
    for i in range(nb):
        one(i)
    stream.synchronize()
    v1 = mk.mk_get_stats(st)
    acc_all = (v1.accepted_sum - v0.accepted_sum) / float(v1.steps - v0.steps)
    for i in range(max(args.warmup, 3)):
        one(i)
    stream.synchronize()
    if mk.mk_get_status(st) != mk.MK_OK:
        raise RuntimeError("device status: " + mk.mk_last_error(st))
    s0 = mk.mk_get_stats(st)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    accs = []
    clocks = ClockSampler(lrank)
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        one(i)
        ev[i][1].record(stream)
    g1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    total_ms = g0.elapsed_time(g1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if mk.mk_get_status(st) != mk.MK_OK:
        raise RuntimeError("device status: " + mk.mk_last_error(st))
    s1 = mk.mk_get_stats(st)
    nsteps = s1.steps - s0.steps
    acc_timed = (s1.accepted_sum - s0.accepted_sum) / max(nsteps, 1)
    distinct = (s1.distinct_experts_sum - s0.distinct_experts_sum) / max(nsteps, 1)
    acc_mean = acc_all
    tok_per_step = acc_mean + 1.0

    if args.stage_trace:
        stage_breakdown(mk, st, cfg, one, stream, dev)

    # end to end through the host-buffer entry point, over the same blocks
    h_tok = torch.tensor(blocks, dtype=torch.int32).pin_memory()
    h_pos = pos.cpu().pin_memory()
    h_lg = torch.empty((T, V), dtype=torch.float32).pin_memory()
    h_acc = torch.zeros(1, dtype=torch.int32).pin_memory()
    h_am = torch.zeros(T, dtype=torch.int32).pin_memory()
    for i in range(2):
        mk.mk_decode_step_host(st, h_tok[i % nb], T, h_pos, kva.kv, h_lg, h_acc, h_am, sh)
    e2e_steps = max(3, args.steps // 2)
    if pg:
        pg.barrier()
    e2e_accepted = 0
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        mk.mk_decode_step_host(st, h_tok[i % nb], T, h_pos, kva.kv, h_lg, h_acc, h_am, sh)
        e2e_accepted += int(h_acc[0])
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    # the same tokens per step as `value` (every block's count); the e2e steps
    # above cycle through the first blocks, whose counts were read back too
    e2e_tok = tok_per_step / e2e_s

    mean_ms = total_ms / args.steps
    slow_ms, value, e2e_value = reduce_over_ranks(mean_ms, tok_per_step, e2e_s, e2e_tok,
                                                  pg is not None)
    if rank != 0:
        mk.mk_destroy(st)
        return

    peaks = measured_peaks()
    peak, peak_src = (peaks["hbm_gbs"], "measured") if peaks else (6800.0, "fallback")
    bytes_step = algorithmic_bytes(cfg, distinct, cfg.ctx)
    achieved = bytes_step / (mean_ms / 1e3) / 1e9
    cpu = None
    planned = tokens_per_step_of(plan)
    if world == 1 and not args.no_cpu_baseline:
        per, lm_s = oracle_sample(model, kv, cfg, blocks[0], [0])
        est = cfg.n_layers * per[0] + lm_s
        cpu = {"value": planned / est, "unit": "tok/s", "cores": os.cpu_count(),
               "kind": "oracle",
               "sample": "fp64 numpy oracle on layer 0 of the first draft block's step (%.2f s) + "
                         "final norm/LM head/argmax (%.2f s), extrapolated to %d layers = %.1f "
                         "s/step; %.4f tokens/step, the same draws as the GPU arm; weights staged "
                         "to host memory beforehand (untimed); numpy BLAS on all host cores"
                         % (per[0], lm_s, cfg.n_layers, est, planned)}
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(slow_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (("fp8e4m3 weights x f16 activations -> fp32 (bf16 LM head), int64 fixed-point reductions"
                   if args.experts == "fp8" else
                   "mxfp4 routed experts, fp8e4m3 attention/shared weights x f16 activations -> fp32 "
                   "(bf16 LM head), int64 fixed-point reductions")
                  + ("; fp8e4m3 KV codes x f16 queries / probabilities" if args.kv == "fp8" else "")
                  + ("; fp8e4m3 1x128 LM head" if args.lm == "fp8" else "")),
        "data": "synthetic (seeded random weights of the named architecture)",
        "config": {"workload": workload_of(cfg), "global_batch": world, "seq_len": T,
                   "parallelism": "replicas (1 stream per GPU)" if world > 1 else "single GPU",
                   "l2": "no flush: each step streams ~%.1f GB, far above the 129 MB L2" % (bytes_step / 1e9)},
        "step_us": {"mean": round(mean_ms * 1e3, 2), "median": round(statistics.median(step_ms) * 1e3, 2),
                    "p10": round(sorted(step_ms)[len(step_ms) // 10] * 1e3, 2),
                    "p90": round(sorted(step_ms)[(9 * len(step_ms)) // 10] * 1e3, 2)},
        "tokens_per_step": round(tok_per_step, 4), "accepted_mean": round(acc_mean, 4),
        "draft_blocks": {"n": nb, "p_agree": P_AGREE, "seed": 3 + rank,
                         "planned_tokens_per_step": round(planned, 4),
                         "expected_tokens_per_step": round(sum(P_AGREE ** j for j in range(T)), 4),
                         "accepted_mean_timed_steps": round(acc_timed, 4),
                         "e2e_accepted_mean": round(e2e_accepted / e2e_steps, 4),
                         "note": "tokens_per_step = 1 + the device's accepted count averaged over one "
                                 "verify step of every block; timed step i verifies block i % n"},
        "distinct_experts_per_layer": round(distinct / cfg.n_layers, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     # the stored figure belongs to the default workload only
                     "traffic": ncu_traffic() if workload_of(cfg) == WORKLOAD else None,
                     "kernel": "mk_step_kernel", "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": int(bytes_step)},
        "e2e": {"value": round(e2e_value, 3), "unit": "tok/s",
                "h2d_bytes_per_step": 2 * T * 4, "d2h_bytes_per_step": T * V * 4 + 4 + T * 4},
        "gpu_launches": args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "setup_s": {"generate_weights": round(t_gen, 1)},
    }
    print(json.dumps(out), flush=True)
    mk.mk_destroy(st)


def run_streams(args):
    """Concurrency workload: S independent streams, each a T=6 block at its own
    context (U[1024, 8192], seed 4) over the 43-layer FP8 stack, verified by
    mk_decode_batch.  Drafts per stream as in the single-stream workload."""
    import numpy as np
    import torch
    from latency_moe_decode_persistent_gb300 import mk, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    S = args.streams
    rng = np.random.default_rng(4)
    ctxs = [int(c) for c in rng.integers(1024, 8193, S)]
    cfg = synth.stack_config(seed=4, **({"n_layers": args.layers} if args.layers else {}))
    model = synth.make_model(cfg, dev)
    kv = synth.make_kv(cfg, dev, ctxs=ctxs)
    margs = mk.ModelArgs(model, cfg.T, kv.max_pages)
    st = mk.mk_create(margs.desc, margs.weights)
    kva = mk.KVArgs(kv.k_pools, kv.v_pools, kv.page_table, kv.n_pages)
    T, V = cfg.T, cfg.vocab
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    logits = torch.empty((S, T, V), dtype=torch.float32, device=dev)
    acc = torch.zeros(S, dtype=torch.int32, device=dev)
    am = torch.zeros((S, T), dtype=torch.int32, device=dev)
    pos = torch.stack([torch.arange(c, c + T, dtype=torch.int32) for c in ctxs]).to(dev)
    toks = []
    plan = draft_plan(S, T - 1, V, seed=40)
    for s in range(S):
        row = mk.KVArgs(kv.k_pools, kv.v_pools, kv.page_table[s], kv.n_pages)

        def step_prefix(tk, s=s, row=row):
            n = len(tk)
            t = torch.tensor(tk, dtype=torch.int32, device=dev)
            mk.mk_decode_step(st, t, n, pos[s, :n].contiguous(), row.kv, logits[s], acc[s:], am[s], sh)
            stream.synchronize()
            return am[s, :n].cpu().tolist()
        toks.append(build_drafts(step_prefix, plan[s]))
    tok = torch.tensor(toks, dtype=torch.int32, device=dev)

    def one():
        mk.mk_decode_batch(st, S, tok, T, pos, kva.kv, logits, acc, am, sh)

    for _ in range(max(args.warmup, 3)):
        one()
    stream.synchronize()
    s0 = mk.mk_get_stats(st)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(args.steps):
        one()
    g1.record(stream)
    torch.cuda.synchronize()
    if mk.mk_get_status(st) != mk.MK_OK:
        raise RuntimeError("device status: " + mk.mk_last_error(st))
    s1 = mk.mk_get_stats(st)
    ms = g0.elapsed_time(g1) / args.steps
    n = s1.steps - s0.steps
    acc_mean = (s1.accepted_sum - s0.accepted_sum) / max(n, 1)
    distinct = (s1.distinct_experts_sum - s0.distinct_experts_sum) / max(n, 1) / cfg.n_layers
    per_stream = (acc_mean + 1.0) / (ms / 1e3)
    print(json.dumps({
        "metric": "verify-step us and tok/s, %d concurrent streams (43-layer FP8, T=6)" % S,
        "value": round(per_stream * S, 3), "unit": "tok/s (all streams)", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 5),
        "higher_is_better": True, "per_stream_tok_s": round(per_stream, 3),
        "tokens_per_stream_step": round(acc_mean + 1.0, 4),
        "distinct_experts_per_layer_per_stream": round(distinct, 2),
        "launches_per_step": S, "dtype": "fp8e4m3 weights x f16 activations -> fp32",
        "data": "synthetic", "config": {"workload": "%d streams x T=6, contexts %s, seed 4; streams run one "
                                                    "after another (one launch each)" % (S, ctxs)}}), flush=True)
    mk.mk_destroy(st)


STAGES = ["qkv", "attention", "o_proj", "router+shared_gate_up", "routed_gate_up", "routed_down"]


def stage_breakdown(mk, st, cfg, one, stream, dev):
    """One more step with the in-kernel barrier timeline on; prints, per stage
    kind, the wall time between barrier releases summed over layers and the
    mean/max per-CTA work time (stderr)."""
    import torch
    G = mk.mk_get_stats(st).grid_ctas
    cap = 6 * cfg.n_layers + 3
    buf = torch.zeros((G, cap, 2), dtype=torch.int64, device=dev)
    ev = torch.zeros((G, 1024, 2), dtype=torch.int64, device=dev)
    mk.mk_set_stage_trace(st, buf, cap, ev)
    one()
    stream.synchronize()
    mk.mk_set_stage_trace(st, None, 0, None)
    if os.environ.get("MK_TRACE_DUMP"):
        import numpy as np
        np.savez_compressed(os.environ["MK_TRACE_DUMP"], barriers=buf.cpu().numpy(), events=ev.cpu().numpy())
    t = buf.cpu().numpy().astype("float64")
    arr, rel = t[:, :, 0], t[:, :, 1]
    names = ["init"] + [STAGES[i % 6] for i in range(6 * cfg.n_layers)] + ["lm_head", "logits_argmax"]
    agg = {}
    for b in range(cap):
        prev_rel = rel[:, b - 1] if b else arr[:, 0] - 0.0
        wall = rel[:, b].max() - (rel[:, b - 1].max() if b else arr[:, 0].min())
        work = arr[:, b] - (rel[:, b - 1] if b else arr[:, 0])
        lat = rel[:, b].min() - arr[:, b].max()
        a = agg.setdefault(names[b], [0.0, 0.0, 0.0, 0.0, 0])
        a[0] += wall
        a[1] += work.mean()
        a[2] += work.max()
        a[3] += lat
        a[4] += 1
    total = rel[:, cap - 1].max() - arr[:, 0].min()
    sys.stderr.write("stage breakdown (us, summed over layers) total %.1f\n" % (total / 1e3))
    sys.stderr.write("%-24s %5s %10s %10s %10s %10s\n" % ("stage", "n", "wall", "work_mean", "work_max", "bar_lat"))
    for k, a in agg.items():
        sys.stderr.write("%-24s %5d %10.1f %10.1f %10.1f %10.1f\n" % (k, a[4], a[0] / 1e3, a[1] / 1e3, a[2] / 1e3, a[3] / 1e3))
    # intra-stage events: mean offset (us) from the start of the stage they fall in
    e = ev.cpu().numpy()
    import collections
    offs = collections.defaultdict(list)
    import numpy as np
    for cta in range(G):
        starts = np.sort(rel[cta])
        for k in list(range(1024 - 72)) + [1024 - 72]:
            eid, tm = int(e[cta, k, 0]), float(e[cta, k, 1])
            if tm == 0:
                if k < 1024 - 72:
                    continue
                break
            i = int(np.searchsorted(starts, tm, "right")) - 1
            if i >= 0:
                offs[eid].append((tm - starts[i]) / 1e3)
    # cycle accounting of the GEMV loops (ids >= 900)
    cyc = collections.defaultdict(list)
    for cta in range(G):
        for k in range(1024 - 64, 1024):
            eid, val = int(e[cta, k, 0]), float(e[cta, k, 1])
            if eid >= 900:
                cyc[eid].append(val)
    names = {0: "wait", 1: "compute", 2: "other"}
    for eid in sorted(cyc):
        if eid >= 1990:
            v = cyc[eid]
            sys.stderr.write("  probe %d mean %10.1f\n" % (eid, sum(v) / len(v)))
    cyc = {k: v for k, v in cyc.items() if k < 1990}
    for eid in sorted(cyc):
        v = cyc[eid]
        if eid < 950:
            st_, k_ = (eid - 900) // 4, (eid - 900) % 4
            sys.stderr.write("  consumer st%d %-8s mean %10.0f cycles/step\n" % (st_, names.get(k_, k_), sum(v) / len(v)))
        elif eid < 980:
            st_, k_ = (eid - 950) // 2, (eid - 950) % 2
            sys.stderr.write("  producer st%d %-8s mean %10.0f cycles/step\n" % (st_, "slotwait" if k_ == 0 else "total", sum(v) / len(v)))
        else:
            st_, k_ = (eid - 980) // 2, (eid - 980) % 2
            sys.stderr.write("  producer st%d %-8s mean %10.0f cycles/step\n" % (st_, "tma" if k_ == 0 else "bulk", sum(v) / len(v)))
    offs = {k: v for k, v in offs.items() if k < 900}
    sys.stderr.write("events (mean us after the stage's barrier release; id = stage*16+k)\n")
    for eid in sorted(offs):
        v = offs[eid]
        sys.stderr.write("  %4d  st%-2d k%-2d  n=%6d  mean %8.2f  max %8.2f\n" % (eid, eid // 16, eid % 16, len(v), sum(v) / len(v), max(v)))


def run_reference(args):
    """The fp64 oracle on the host cores, on a bounded sample of the same step.

    Each timed step runs one decoder layer of the verify step in the oracle
    (the sample's layers cycled); the full step's time is that layer's time x
    the layer count + the LM head (timed once).  Tokens per step come from the
    same seeded draft draws as the GPU arm, cycled over the same number of
    steps, so both arms divide by the same tokens."""
    rank, world, lrank = rank_info()
    if rank != 0:
        return
    import numpy as np
    import torch
    from latency_moe_decode_persistent_gb300 import synth
    vkw = variant_kw(args, synth)
    cfg = synth.stack_config(**vkw)
    dev = torch.device("cuda", lrank) if torch.cuda.is_available() else torch.device("cpu")
    # only the layers the sample uses are generated (per-layer seeds make them
    # identical to the full model's)
    nl = min(cfg.n_layers, max(1, args.ref_layers))
    sub = synth.stack_config(n_layers=nl, **vkw)
    model = synth.make_model(sub, dev)
    kv = synth.make_kv(sub, dev)
    plan = draft_plan(DRAFT_BLOCKS, cfg.T - 1, cfg.vocab, seed=3)
    tok_step = tokens_per_step_of(plan)
    # the oracle does not build the drafts (that takes prefix passes of the whole
    # stack); a layer's cost does not depend on which tokens it verifies
    toks = [plan[0][0]] + plan[0][2]
    # warm-up: stage weights, measure the LM head once
    per, lm_s = oracle_sample(model, kv, sub, toks, [0], ref_lm=True)
    for i in range(args.warmup):
        oracle_sample(model, kv, sub, toks, [i % nl], ref_lm=False)
    samples, fulls = [], []
    for i in range(args.steps):
        p, _ = oracle_sample(model, kv, sub, toks, [i % nl], ref_lm=False)
        samples.append(p[0])
        fulls.append(cfg.n_layers * p[0] + lm_s)
    step_s = statistics.mean(fulls)
    value = tok_step / step_s
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(samples) * 1e3, 1),
        "full_step_ms_extrapolated": round(step_s * 1e3, 1),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_of(cfg), "global_batch": 1, "seq_len": cfg.T},
        "tokens_per_step": round(tok_step, 4),
        "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": round(value, 6),
                         "sample": "each timed step (ms_per_step): one decoder layer of the verify "
                                   "step in the fp64 numpy oracle (layers %s cycled); value = "
                                   "tokens/step / (layer time x 43 + LM head %.2f s, timed once); "
                                   "weights staged to host memory beforehand; %.4f tokens/step from "
                                   "the GPU arm's seeded draft draws (%d blocks, 0.83 agreement)"
                                   % (list(range(nl)), lm_s, tok_step, DRAFT_BLOCKS)},
        "e2e": {"value": round(value, 6), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (debug)")
    ap.add_argument("--ref-layers", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-trace", action="store_true", help="print an in-kernel stage breakdown to stderr")
    ap.add_argument("--T", type=int, default=0, help="verify block size (T sweep; default 6)")
    ap.add_argument("--experts", default="fp8", choices=["fp8", "mxfp4"],
                    help="routed-expert storage of the stack (the default workload is FP8)")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="KV cache format (the default workload is bf16)")
    ap.add_argument("--ctx", type=int, default=0, help="cached context of the stream (default 2048)")
    ap.add_argument("--lm", default="bf16", choices=["bf16", "fp8"],
                    help="LM head storage (the default workload is bf16)")
    ap.add_argument("--streams", type=int, default=0,
                    help="concurrency workload: S streams of T=6 tokens, contexts U[1024, 8192], seed 4 "
                         "(mk_decode_batch); prints its own line")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.streams:
        run_streams(args)
    else:
        run_mk(args)


if __name__ == "__main__":
    main()
