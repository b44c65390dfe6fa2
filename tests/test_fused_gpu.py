"""The one-launch Quest step (se_quest_fused_step) on the GPU against the fp64 oracle.

Same comparison rules as the four-call path (selection exact outside the 1e-3
band around the k-th score, output within 2e-2, lse within 1e-3): the tiny
workload, ragged appends with and without keep windows, every group-size
class, edge lengths, the appended token bit-exact against the append entry
point, and the full 32K and 128K workloads on sampled requests.
"""
import math

import pytest
import torch

import sparse_decode_attention_quest_gb300 as se
from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
from synth import QWEN3_30B_A3B_QUEST_128K, QWEN3_4B_QUEST_32K, TINY_QUEST_4K, make_quest_decode_inputs
from tests.parity import compare_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors(se_lib, cuda_device):
    se.se_read_device_error(clear=True)
    yield
    assert se.se_read_device_error(clear=True) == 0


def _prepare(wl, dev, device_gen=False, sink=0, recent=0):
    x = make_quest_decode_inputs(wl, device=dev if device_gen else "cpu", poison_tail=True)
    k = x.k_cache.to(dev)
    v = x.v_cache.to(dev)
    step = QuestDecodeStep(k, v, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(max(x.seq_lens_after), 1), sink_tokens=sink, recent_tokens=recent)
    before = torch.tensor(x.seq_lens, dtype=torch.int32, device=dev)
    after = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    step.build_summaries(before)
    return x, step, after


def _run_fused(x, step, after, dev):
    if x.workload.append:
        step.run_fused(x.q.to(dev), after, x.k_new.to(dev), x.v_new.to(dev))
    else:
        step.run_fused(x.q.to(dev), after)
    torch.cuda.synchronize()


def _scale(wl):
    return 1.0 / math.sqrt(wl.head_dim)


def test_fused_tiny_workload(cuda_device):
    wl = TINY_QUEST_4K
    x, step, a = _prepare(wl, cuda_device)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, [0], _scale(wl), "fused tiny")


@pytest.mark.parametrize("sink,recent", [(0, 0), (64, 512), (16, 64)])
def test_fused_ragged_append(cuda_device, sink, recent):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=5, context_min=900, context_max=4100, topk_pages=24, seed=81)
    x, step, a = _prepare(wl, cuda_device, sink=sink, recent=recent)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"fused ragged {sink}/{recent}", sink, recent)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (16, 2), (32, 2), (12, 4)])
def test_fused_group_sizes(cuda_device, hq, hkv):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, num_q_heads=hq, num_kv_heads=hkv, context_min=500,
                                         context_max=2500, topk_pages=16, seed=83 + hq)
    x, step, a = _prepare(wl, cuda_device)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"fused g={hq // hkv}")


def test_fused_edge_lengths(cuda_device):
    lens = (0, 1, 15, 16, 17, 31, 33, 160, 161, 700)
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=len(lens), lengths=lens, topk_pages=6, seed=87)
    x, step, a = _prepare(wl, cuda_device)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "fused edges")


def test_fused_append_equals_the_append_entry_point(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=6, lengths=(15, 16, 17, 31, 32, 400), topk_pages=4, seed=89)
    x, s1, a = _prepare(wl, cuda_device)
    x2, s2, a2 = _prepare(wl, cuda_device)
    _run_fused(x, s1, a, cuda_device)
    before = torch.tensor(x2.seq_lens, dtype=torch.int32, device=cuda_device)
    s2.append(x2.k_new.to(cuda_device), x2.v_new.to(cuda_device), before)
    torch.cuda.synchronize()
    assert torch.equal(s1.k_cache.view(torch.int16), s2.k_cache.view(torch.int16))
    assert torch.equal(s1.v_cache.view(torch.int16), s2.v_cache.view(torch.int16))
    assert torch.equal(s1.summary.view(torch.int16), s2.summary.view(torch.int16))


def test_fused_full_qwen3_4b_32k_sampled(cuda_device):
    wl = QWEN3_4B_QUEST_32K
    x, step, a = _prepare(wl, cuda_device, device_gen=True)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, [0, wl.batch - 1], _scale(wl), "fused qwen3-4b full")


def test_fused_full_qwen3_30b_a3b_128k_sampled(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K
    x, step, a = _prepare(wl, cuda_device, device_gen=True)
    _run_fused(x, step, a, cuda_device)
    compare_decode(x, step, [0, 13, wl.batch - 1], _scale(wl), "fused qwen3-30b full")


def test_fused_step_is_repeatable(cuda_device):
    # the one-launch step (cluster-wide scores, selection and split merge over distributed
    # shared memory) run again on the same inputs gives bit-identical selections, outputs and
    # log-sum-exps; without an append, every run sees the same cache
    wl = QWEN3_4B_QUEST_32K.scaled(batch=4, context_min=6000, context_max=12000, topk_pages=64, append=False,
                                   seed=81)
    x, step, a = _prepare(wl, cuda_device)
    _run_fused(x, step, a, cuda_device)
    sel0, cnt0, out0, lse0 = step.sel.clone(), step.counts.clone(), step.out.clone(), step.lse.clone()
    for _ in range(8):
        _run_fused(x, step, a, cuda_device)
        assert torch.equal(step.counts, cnt0)
        for b in range(wl.batch):
            for h in range(wl.num_kv_heads):
                n = int(cnt0[b, h])
                assert torch.equal(step.sel[b, h, :n], sel0[b, h, :n])
        assert torch.equal(step.out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(step.lse, lse0)


@pytest.mark.parametrize("context,topk,period", [(4096, 32, 5), (131072, 256, 20)])
def test_fused_selection_with_tied_pages(cuda_device, context, topk, period):
    # Every page of a request repeats the keys of one of its first `period`
    # pages, so the page scores take `period` values, each on many pages, and the
    # k-th largest sits inside a tied level. The selection must take the tied
    # pages with the lowest ids, in the one-launch step (bucket select over the
    # cluster's scores; 8 candidates per thread at 4K, 32 at 128K) and in the
    # four-call path alike; both read their scores off equal keys, so equal
    # pages score equally on each side.
    wl = QWEN3_4B_QUEST_32K.scaled(batch=1, num_q_heads=16, num_kv_heads=4, context_min=context,
                                   context_max=context, topk_pages=topk, append=False, seed=95)
    x, fused, a = _prepare(wl, cuda_device, device_gen=context > 8192)
    n = context // wl.page_size
    bt = x.block_table[0].long().to(cuda_device)
    src = bt[torch.arange(n, device=cuda_device) % period]
    fused.k_cache[bt[:n]] = fused.k_cache[src]
    fused.build_summaries(a)
    sep = QuestDecodeStep(fused.k_cache, fused.v_cache, new_summary(fused.k_cache), x.block_table.to(cuda_device),
                          wl.num_q_heads, wl.topk_pages, context)
    sep.build_summaries(a)
    q = x.q.to(cuda_device)
    fused.run_fused(q, a)
    sep.run(q, a)
    torch.cuda.synchronize()
    scores = sep.scores[0].cpu()
    for h in range(wl.num_kv_heads):
        s = scores[h, :n - 1]
        order = sorted(range(n - 1), key=lambda p: (-float(s[p]), p))
        want = sorted(order[:topk]) + [n - 1]
        level = float(s[order[topk - 1]])
        assert sum(1 for p in range(n - 1) if float(s[p]) == level) > 1, "the k-th score must be tied"
        assert int(sep.counts[0, h]) == topk + 1 and int(fused.counts[0, h]) == topk + 1
        assert sep.sel[0, h, :topk + 1].tolist() == want, h
        assert fused.sel[0, h, :topk + 1].tolist() == want, h
