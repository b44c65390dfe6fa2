"""Recorded steps (se_capture_begin / se_capture_end / se_graph_launch) on the GPU.

A step recorded once and replayed must compute what the live calls compute on
the values its buffers hold at each launch: new queries, new K/V rows and
lengths that grow by one token per step, all written into the recorded
buffers between launches.
"""
import pytest
import torch

import sparse_decode_attention_quest_gb300 as se
from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
from synth import QWEN3_30B_A3B_QUEST_128K, make_quest_decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors(se_lib, cuda_device):
    se.se_read_device_error(clear=True)
    yield
    assert se.se_read_device_error(clear=True) == 0


def _make(x, wl, dev):
    k = x.k_cache.to(dev).clone()
    v = x.v_cache.to(dev).clone()
    step = QuestDecodeStep(k, v, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(x.seq_lens_after))
    step.build_summaries(torch.tensor(x.seq_lens, dtype=torch.int32, device=dev))
    return step


def test_replayed_step_follows_its_buffers(cuda_device):
    dev = cuda_device
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=4, context_min=2000, context_max=5000, topk_pages=24, seed=97)
    x = make_quest_decode_inputs(wl, device="cpu", poison_tail=True)
    live, rec = _make(x, wl, dev), _make(x, wl, dev)
    B, Hq, H, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    # The requests start two tokens short and grow by one token per step; the
    # last step ends at the lengths the block table was built for.
    start = torch.tensor(x.seq_lens, dtype=torch.int32) - 2
    assert int(start.min()) >= 0
    bq = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device=dev)
    bkn = torch.zeros(B, H, D, dtype=torch.bfloat16, device=dev)
    bvn = torch.zeros(B, H, D, dtype=torch.bfloat16, device=dev)
    bbefore = torch.zeros(B, dtype=torch.int32, device=dev)
    bafter = torch.zeros(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    se.se_capture_begin(stream)
    rec.run(bq, bafter, bkn, bvn, bbefore, stream=stream)
    graph = se.se_capture_end(stream)
    g = torch.Generator().manual_seed(5)
    try:
        for t in range(3):
            q = torch.randn(B, Hq, D, generator=g).bfloat16().to(dev)
            kn = torch.randn(B, H, D, generator=g).bfloat16().to(dev)
            vn = torch.randn(B, H, D, generator=g).bfloat16().to(dev)
            before = (start + t).to(dev)
            after = before + 1
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                bq.copy_(q)
                bkn.copy_(kn)
                bvn.copy_(vn)
                bbefore.copy_(before)
                bafter.copy_(after)
                graph.launch(stream)
            live.run(q, after, kn, vn, before)
            torch.cuda.synchronize()
            assert torch.equal(rec.counts, live.counts), t
            for b in range(B):
                for h in range(H):
                    n = int(live.counts[b, h])
                    assert torch.equal(rec.sel[b, h, :n], live.sel[b, h, :n]), (t, b, h)
            assert torch.equal(rec.out.view(torch.int16), live.out.view(torch.int16)), t
            assert torch.equal(rec.lse, live.lse), t
        assert torch.equal(rec.k_cache.view(torch.int16), live.k_cache.view(torch.int16))
        assert torch.equal(rec.v_cache.view(torch.int16), live.v_cache.view(torch.int16))
        assert torch.equal(rec.summary.view(torch.int16), live.summary.view(torch.int16))
    finally:
        graph.destroy()
