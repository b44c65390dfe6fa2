"""se_sparse_paged_decode_noalloc, the decode for callers that cannot allocate.

Some callers have no way to hand the library a workspace: plugins that only
receive inputs and outputs, processes whose device memory belongs to another
framework's allocator, loops that forbid cudaMalloc after start-up. For them
the decode keeps its split partials in a fixed array inside the library. This
file checks, through the C ABI, that two calls in a row (the second on other
queries, so stale array contents would show) give the same output as
se_sparse_paged_decode with a caller workspace and agree with the fp64 oracle,
that the case really spreads items over several CTAs (so the array's partials
and counters are used), that a latent cache and sizes beyond the array are
refused. It is collected last so that a failure here comes after every other
test has run.
"""
import math

import pytest
import torch

import sparse_decode_attention_quest_gb300 as se
from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
from synth import QWEN3_30B_A3B_QUEST_128K, make_quest_decode_inputs
from tests.parity import LSE_ATOL, OUT_ATOL, compare_decode

pytestmark = pytest.mark.gpu


def _case(dev):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=4, context_min=2000, context_max=5000, topk_pages=40,
                                         append=False, seed=41)
    x = make_quest_decode_inputs(wl, device="cpu")
    k, v = x.k_cache.to(dev), x.v_cache.to(dev)
    step = QuestDecodeStep(k, v, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(x.seq_lens_after))
    lens = torch.tensor(x.seq_lens, dtype=torch.int32, device=dev)
    step.build_summaries(lens)
    return wl, x, step, lens


def test_noalloc_decode_matches_the_workspace_decode(se_lib, cuda_device):
    wl, x, step, lens = _case(cuda_device)
    _, per_split, _ = se.se_sparse_decode_plan(wl.batch, wl.num_q_heads, wl.num_kv_heads, 128, 128,
                                               step.sel_stride)
    gen = torch.Generator().manual_seed(5)
    for call in range(2):
        q = x.q if call == 0 else torch.randn(x.q.shape, generator=gen).to(torch.bfloat16)
        q = q.to(cuda_device)
        step.select(q, lens)
        # A CTA slice holds max(per_split, ceil(pages / CTAs)) selected pages, with at
        # least one CTA per SM; an item with more pages than that spans two or more
        # slices, so its partials go through the array and are merged there.
        counts = step.counts.flatten().tolist()
        sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
        per_cta_max = max(per_split, -(-sum(counts) // sms))
        assert max(counts) > per_cta_max, (counts, per_cta_max)
        se.se_sparse_paged_decode(step.kv, q, step.block_table, lens, step.sel, step.counts, step.sm_scale,
                                  step.out, step.lse, step.workspace)
        out = torch.full_like(step.out, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        se.se_sparse_paged_decode_noalloc(step.kv, q, step.block_table, lens, step.sel, step.counts,
                                          step.sm_scale, out, lse)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out.float()).all())
        assert (out.float() - step.out.float()).abs().max().item() <= OUT_ATOL, call
        assert (lse - step.lse).abs().max().item() <= LSE_ATOL, call
        # and against the fp64 oracle on the same queries and selection
        step.out.copy_(out)
        step.lse.copy_(lse)
        x.q = q.cpu()
        compare_decode(x, step, list(range(wl.batch)), step.sm_scale, f"noalloc call {call}")
    assert se.se_read_device_error(clear=True) == 0


def test_noalloc_decode_refuses_a_latent_cache(se_lib, cuda_device):
    dev = cuda_device
    cache = torch.zeros(4, 1, 16, 576, dtype=torch.bfloat16, device=dev)
    kv = se.paged_kv(cache, None, None, 512)
    q = torch.zeros(2, 64, 576, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(2, 4, dtype=torch.int32, device=dev)
    lens = torch.zeros(2, dtype=torch.int32, device=dev)
    sel = torch.zeros(2, 1, 8, dtype=torch.int32, device=dev)
    cnt = torch.zeros(2, 1, dtype=torch.int32, device=dev)
    out = torch.empty(2, 64, 512, dtype=torch.bfloat16, device=dev)
    with pytest.raises(se.SparseEngineError) as e:
        se.se_sparse_paged_decode_noalloc(kv, q, bt, lens, sel, cnt, 1 / math.sqrt(576), out)
    assert e.value.status == 2 and "workspace" in str(e.value)


def test_noalloc_decode_refuses_sizes_beyond_its_array(se_lib, cuda_device):
    # 256 requests x 32 query heads need more than 8 MiB of split partials.
    B, Hq, H, k = 256, 32, 4, 40
    nsplit, _, _ = se.se_sparse_decode_plan(B, Hq, H, 128, 128, k + 1)
    assert B * Hq * nsplit * 129 * 4 > (8 << 20)
    dev = cuda_device
    cache = torch.zeros(4, H, 16, 128, dtype=torch.bfloat16, device=dev)
    kv = se.paged_kv(cache, cache.clone(), None)
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(B, 4, dtype=torch.int32, device=dev)
    lens = torch.zeros(B, dtype=torch.int32, device=dev)
    sel = torch.zeros(B, H, k + 1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, H, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(se.SparseEngineError) as e:
        se.se_sparse_paged_decode_noalloc(kv, q, bt, lens, sel, cnt, 1 / math.sqrt(128), out)
    assert e.value.status == 3 and "8 MiB" in str(e.value)
