"""The bench's CPU-baseline legs run the fp64 oracle on small samples (CPU only)."""
import bench
from synth import MLA_GLM_QUEST_32K, QWEN3_30B_A3B_QUEST_128K, SNAPKV_AIME_32K, make_quest_decode_inputs, \
    make_snapkv_inputs


def test_quest_cpu_baseline_with_append_and_windows():
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=2, context_min=300, context_max=500, topk_pages=4)
    x = make_quest_decode_inputs(wl, poison_tail=False)
    r = bench.cpu_oracle_throughput(x, n_requests=2, cores=2, sink=16, recent=32)
    assert r["value"] > 0 and r["cores"] == 2 and r["kind"] == "oracle" and "append" in r["sample"]


def test_latent_cpu_baseline():
    wl = MLA_GLM_QUEST_32K.scaled(batch=2, num_q_heads=16, context_min=200, context_max=200, topk_pages=3)
    x = make_quest_decode_inputs(wl, poison_tail=False)
    r = bench.cpu_oracle_throughput(x, n_requests=1, cores=1)
    assert r["value"] > 0 and r["cores"] == 1


def test_snapkv_cpu_baseline():
    wl = SNAPKV_AIME_32K.scaled(batch=1, num_q_heads=8, num_kv_heads=2, prompt_min=400, prompt_max=400,
                                keep_topk=50)
    x = make_snapkv_inputs(wl, poison_tail=False)
    r = bench.snapkv_cpu_baseline(x, cores=2)
    assert r["value"] > 0 and r["unit"] == "requests/s" and r["cores"] == 2
