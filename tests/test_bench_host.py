"""Host-side pieces of the bench that need no GPU: the key that ties a stored
ncu traffic figure to the kernel code it was measured on, and the algorithmic
byte count the roofline divides by."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_code_key_ignores_comments_and_layout_only():
    a = "int f(int x) {\n    // twice\n    return 2 * x; /* doubled */\n}\n"
    b = "int f(int x) { return 2 * x; }  // a different comment\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_stored_traffic_matches_current_code_or_is_dropped():
    # the committed figure is reported only while the kernel code matches the
    # hash stored beside it
    t = bench.ncu_traffic()
    assert t is None or 0.9e10 < t < 2.0e10


def test_algorithmic_bytes_of_the_43_layer_workload():
    # The roofline's numerator, written out from the layer shapes (FP8 codes plus
    # one fp32 scale per 128 inputs and output row; bf16 router, embedding and LM
    # head; bf16 KV at ctx 2048; T = 6):
    qkv = 5120 * 4096 + 32 * 5120 * 4
    o = 4096 * 4096 + 32 * 4096 * 4
    router = 384 * 4096 * 2 + 384 * 4
    norms = 2 * 4096 * 4
    expert = 2 * (512 * 4096 + 32 * 512 * 4) + (4096 * 512 + 4 * 4096 * 4)
    kv = 2048 * 4 * 128 * 2 * 2 + 6 * 4 * 128 * 2 * 2
    per_layer = qkv + o + router + norms + expert + kv
    once = 6 * 4096 * 2 + 4096 * 4 + 129280 * 4096 * 2 + 6 * 129280 * 4
    distinct = 1874  # routed experts over the 43 layers of the bench's step
    want = 43 * per_layer + distinct * expert + once
    from latency_moe_decode_persistent_gb300 import synth
    cfg = synth.stack_config(T=6, ctx=2048)
    assert bench.algorithmic_bytes(cfg, distinct, 2048) == want == 15491394048


def test_workload_string_follows_the_run():
    # the default run is described by the default workload string (the one the
    # stored traffic figure belongs to); a run with fewer layers or another block
    # size says so
    from latency_moe_decode_persistent_gb300 import synth
    assert bench.workload_of(synth.stack_config()) == bench.WORKLOAD
    w = bench.workload_of(synth.stack_config(n_layers=2, T=4))
    assert w.startswith("2-layer") and "T=4 (k=3 drafts" in w and w != bench.WORKLOAD


def test_planned_tokens_per_step_follow_the_draws():
    # a block accepts the run of leading agreements of its draws; at 0.83 the
    # mean approaches the expectation sum_j 0.83^j = 3.96 tokens per step
    plan = bench.draft_plan(32, 5, 129280, seed=3)
    acc = bench.planned_accepts(plan)
    for (_, agree, _), n in zip(plan, acc):
        assert all(agree[:n]) and (n == 5 or not agree[n])
    tps = bench.tokens_per_step_of(plan, 32)
    assert abs(tps - (sum(acc) / 32 + 1)) < 1e-12
    assert 3.0 < tps < 5.0
    # cycling: 40 steps over 32 blocks count the first 8 twice
    assert abs(bench.tokens_per_step_of(plan, 40) - ((sum(acc) + sum(acc[:8])) / 40 + 1)) < 1e-12
    # the same seed gives the same plan in both arms
    assert bench.draft_plan(32, 5, 129280, seed=3) == plan
    big = bench.draft_plan(bench.DRAFT_BLOCKS, 5, 129280, seed=3)
    assert abs(bench.tokens_per_step_of(big) - 3.96) < 0.15


def test_algorithmic_bytes_with_mxfp4_experts():
    # MXFP4 routed experts: half a byte per weight plus one E8M0 byte per 32
    # inputs and output row; attention, router and shared expert stay FP8
    from latency_moe_decode_persistent_gb300 import synth
    fp8 = synth.stack_config(T=6, ctx=2048)
    fp4 = synth.stack_config(T=6, ctx=2048, expert_dtype=synth.WDT_MXFP4)
    routed_fp8 = 2 * (512 * 4096 + 32 * 512 * 4) + (4096 * 512 + 4 * 4096 * 4)
    routed_fp4 = 2 * (512 * 4096 // 2 + 128 * 512) + (4096 * 512 // 2 + 16 * 4096)
    assert routed_fp4 == 3342336
    d = 1874
    assert bench.algorithmic_bytes(fp8, d, 2048) - bench.algorithmic_bytes(fp4, d, 2048) == d * (routed_fp8 - routed_fp4)


def test_fp8_kv_workload_bytes_and_name():
    # an FP8 KV cache moves one byte per cached element instead of two: 43 layers
    # x ctx x 4 kv heads x 128 dims x (K, V), plus the block's own entries
    from latency_moe_decode_persistent_gb300 import synth
    b16 = synth.stack_config(T=6, ctx=65536)
    f8 = synth.stack_config(T=6, ctx=65536, kv_dtype=synth.WDT_FP8, kv_scales=bench.FP8_KV_SCALES)
    d = 1874
    diff = bench.algorithmic_bytes(b16, d, 65536) - bench.algorithmic_bytes(f8, d, 65536)
    assert diff == 43 * (65536 + 6) * 4 * 128 * 2
    w = bench.workload_of(f8)
    assert "ctx 65536" in w and "FP8 e4m3 KV (per-layer K/V scales 0.0125/0.0125)" in w
    assert bench.workload_of(synth.stack_config()) == bench.WORKLOAD


def test_fp8_lm_head_bytes_and_name():
    # FP8 LM head: one byte per weight plus a float32 scale per 128 inputs of a row
    from latency_moe_decode_persistent_gb300 import synth
    b16 = synth.stack_config()
    f8 = synth.stack_config(lm_dtype=synth.WDT_FP8)
    d = 1874
    V, H = 129280, 4096
    assert bench.algorithmic_bytes(b16, d, 2048) - bench.algorithmic_bytes(f8, d, 2048) == V * H * 2 - (V * H + 32 * V * 4)
    assert "FP8 e4m3 1x128 LM head" in bench.workload_of(f8)
