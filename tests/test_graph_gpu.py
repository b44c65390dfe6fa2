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


def test_replayed_step_with_its_copies(cuda_device):
    """The input upload (pinned host -> device), the four calls and the result
    download recorded in one step: each replay computes what the live calls do
    on the values the host buffer holds at that launch."""
    dev = cuda_device
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=1500, context_max=4000, topk_pages=16, seed=41)
    x = make_quest_decode_inputs(wl, device="cpu", poison_tail=True)
    live, rec = _make(x, wl, dev), _make(x, wl, dev)
    B, Hq, H, D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    start = torch.tensor(x.seq_lens, dtype=torch.int32) - 2
    assert int(start.min()) >= 0
    shapes = [((B, Hq, D), torch.bfloat16), ((B, H, D), torch.bfloat16), ((B, H, D), torch.bfloat16),
              ((B,), torch.int32), ((B,), torch.int32)]
    offs, size = [], 0
    for shp, dt in shapes:
        offs.append(size)
        n = 1
        for v in shp:
            n *= v
        size += (n * torch.empty((), dtype=dt).element_size() + 15) // 16 * 16
    h_in = torch.zeros(size, dtype=torch.uint8).pin_memory()
    d_in = torch.zeros(size, dtype=torch.uint8, device=dev)

    def views(buf):
        out = []
        for (shp, dt), o in zip(shapes, offs):
            n = 1
            for v in shp:
                n *= v
            nb = n * torch.empty((), dtype=dt).element_size()
            out.append(buf[o:o + nb].view(dt).view(shp))
        return out

    hq, hkn, hvn, hbefore, hafter = views(h_in)
    dq, dkn, dvn, dbefore, dafter = views(d_in)
    h_out = torch.zeros(rec.out.shape, dtype=rec.out.dtype).pin_memory()
    stream = torch.cuda.Stream(device=dev)
    se.se_capture_begin(stream)
    se.se_copy_async(d_in, h_in, stream)
    rec.run(dq, dafter, dkn, dvn, dbefore, stream=stream)
    se.se_copy_async(h_out, rec.out, stream)
    graph = se.se_capture_end(stream)
    g = torch.Generator().manual_seed(6)
    try:
        for t in range(3):
            q = torch.randn(B, Hq, D, generator=g).bfloat16()
            kn = torch.randn(B, H, D, generator=g).bfloat16()
            vn = torch.randn(B, H, D, generator=g).bfloat16()
            before = start + t
            after = before + 1
            stream.synchronize()
            hq.copy_(q)
            hkn.copy_(kn)
            hvn.copy_(vn)
            hbefore.copy_(before)
            hafter.copy_(after)
            graph.launch(stream)
            stream.synchronize()
            live.run(q.to(dev), after.to(dev), kn.to(dev), vn.to(dev), before.to(dev))
            torch.cuda.synchronize()
            assert torch.equal(rec.counts, live.counts), t
            assert torch.equal(h_out.view(torch.int16), live.out.cpu().view(torch.int16)), t
            assert torch.equal(rec.lse, live.lse), t
    finally:
        graph.destroy()


@pytest.mark.parametrize("nbytes, offset", [(16, 0), (4096, 0), (328_000, 0), (1000, 0), (777, 3),
                                            (9 << 20, 0), ((9 << 20) + 5, 1)])
def test_copy_async_every_path(cuda_device, nbytes, offset):
    """se_copy_async host -> device -> device -> host on one stream: the kernel
    (16-byte pieces, or bytes for unaligned sizes and offsets) up to 8 MiB, the
    copy engine above, and device to device; the bytes come back unchanged."""
    dev = cuda_device
    g = torch.Generator().manual_seed(nbytes + offset)
    src = torch.randint(0, 256, (nbytes + offset,), dtype=torch.uint8, generator=g).pin_memory()
    d1 = torch.zeros(nbytes + offset, dtype=torch.uint8, device=dev)
    d2 = torch.zeros(nbytes + offset, dtype=torch.uint8, device=dev)
    back = torch.zeros(nbytes + offset, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.Stream(device=dev)
    se.se_copy_async(d1[offset:], src[offset:], stream)
    se.se_copy_async(d2[offset:], d1[offset:], stream)
    se.se_copy_async(back[offset:], d2[offset:], stream)
    stream.synchronize()
    assert torch.equal(back[offset:], src[offset:])
    assert int(back[:offset].sum()) == 0
