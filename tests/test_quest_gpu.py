"""Quest decode path on the GPU against the fp64 oracle (through the C ABI).

Cases: the tiny 4K workload in full; oracle-sized cases with the 32K Qwen3-4B
and ragged Qwen3-30B-A3B recipes that span several score chunks, top-k
passes and decode splits, with ragged tails; every group size the GQA kernel
takes; edge lengths (0, 1, 15, 16, 17 tokens, budget above the page count);
invariants (summaries bit-exact, bound >= true logit, select-all = dense,
block-table permutation, split count, append idempotence); device-side
range checks; and the full-size workloads checked on sampled requests.
"""
import math

import numpy as np
import pytest
import torch

import oracle.quest as oq
import sparse_decode_attention_quest_gb300 as se
from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
from synth import (MLA_GLM_QUEST_32K, QWEN3_30B_A3B_QUEST_128K, QWEN3_4B_QUEST_32K, TINY_QUEST_4K,
                   make_quest_decode_inputs)
from tests.parity import OUT_ATOL, compare_decode, oracle_inputs

pytestmark = pytest.mark.gpu


def _prepare(wl, dev, device_gen=False, sel_stride=None, poison=True, sink=0, recent=0):
    x = make_quest_decode_inputs(wl, device=dev if device_gen else "cpu", poison_tail=poison)
    k = x.k_cache.to(dev)
    v = None if x.v_cache is None else x.v_cache.to(dev)
    step = QuestDecodeStep(k, v, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(max(x.seq_lens_after), 1), head_dim_v=wl.head_dim_v, sel_stride=sel_stride,
                           sink_tokens=sink, recent_tokens=recent)
    before = torch.tensor(x.seq_lens, dtype=torch.int32, device=dev)
    after = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    step.build_summaries(before)
    return x, step, before, after


def _run(x, step, before, after, dev):
    q = x.q.to(dev)
    if x.workload.append:
        step.run(q, after, x.k_new.to(dev), x.v_new.to(dev), before)
    else:
        step.run(q, after)
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _no_device_errors(se_lib, cuda_device):
    se.se_read_device_error(clear=True)
    yield
    assert se.se_read_device_error(clear=True) == 0


def _scale(wl):
    return 1.0 / math.sqrt(wl.head_dim)


def test_tiny_workload_full(cuda_device):
    wl = TINY_QUEST_4K
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, [0], _scale(wl), "tiny")


def test_ragged_append_oracle_sized(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=5, context_min=900, context_max=4100, topk_pages=24)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "ragged")


def test_qwen3_4b_recipe_oracle_sized(cuda_device):
    wl = QWEN3_4B_QUEST_32K.scaled(batch=2, context_min=4096, context_max=4096, topk_pages=32)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "qwen3-4b")


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (16, 2), (32, 2), (12, 4)])
def test_group_sizes(cuda_device, hq, hkv):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, num_q_heads=hq, num_kv_heads=hkv, context_min=500,
                                         context_max=1300, topk_pages=12, seed=11)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"G={hq // hkv}")


@pytest.mark.parametrize("append", [False, True])
@pytest.mark.parametrize("sel_stride", [None, 64])  # one decode split per request, or several + merge
def test_edge_lengths(cuda_device, append, sel_stride):
    lens = (0, 1, 15, 16, 17, 31, 33, 160, 161, 700) if not append else (1, 15, 16, 17, 31, 33, 160, 161, 700, 0)
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=len(lens), lengths=lens, topk_pages=6, append=append, seed=5)
    x, step, b, a = _prepare(wl, cuda_device, sel_stride=sel_stride)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "edges")
    counts = step.counts.cpu()
    for i, L in enumerate(x.seq_lens_after):
        n = math.ceil(L / 16)
        assert int(counts[i, 0]) == min(n, wl.topk_pages + 1)
    if not append:
        out = step.out.float().cpu()
        assert torch.equal(out[0], torch.zeros_like(out[0]))            # empty request
        assert bool(torch.isneginf(step.lse[0].cpu()).all())


def test_summaries_bit_exact(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=100, context_max=900, append=False, seed=7)
    x, step, b, a = _prepare(wl, cuda_device)
    torch.cuda.synchronize()
    inp = oracle_inputs(x)
    summ = step.summary.float().cpu().numpy()
    bt = x.block_table.cpu().numpy()
    for r in range(wl.batch):
        req = oq.QuestRequest(inp["k_cache"], None, inp["block_table"][r], x.seq_lens[r], wl.num_kv_heads,
                              wl.head_dim, wl.head_dim, 16)
        for h in range(wl.num_kv_heads):
            m, M = req.summaries[h]
            for p in range(m.shape[0]):
                np.testing.assert_array_equal(summ[bt[r, p], h, 0], m[p])
                np.testing.assert_array_equal(summ[bt[r, p], h, 1], M[p])


def test_append_matches_rebuild_and_is_idempotent(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=6, lengths=(15, 16, 17, 31, 32, 400), topk_pages=4, seed=9)
    x, step, b, a = _prepare(wl, cuda_device)
    step.append(x.k_new.to(cuda_device), x.v_new.to(cuda_device), b)
    once = step.summary.clone()
    step.append(x.k_new.to(cuda_device), x.v_new.to(cuda_device), b)
    torch.cuda.synchronize()
    assert torch.equal(once.view(torch.int16), step.summary.view(torch.int16))
    fresh = new_summary(step.k_cache)
    se.se_quest_build_summaries(se.paged_kv(step.k_cache, step.v_cache, fresh), step.block_table, a,
                                step.max_seq_len)
    torch.cuda.synchronize()
    bt = x.block_table
    for r in range(wl.batch):
        n = x.pages_per_request[r]
        idx = bt[r, :n].long().to(cuda_device)
        assert torch.equal(fresh[idx].view(torch.int16), once[idx].view(torch.int16)), r


def test_score_is_an_upper_bound_of_the_group_logit(cuda_device):
    wl = QWEN3_4B_QUEST_32K.scaled(batch=2, context_min=1000, context_max=1000, seed=13)
    x, step, b, a = _prepare(wl, cuda_device)
    se.se_quest_score_pages(step.kv, x.q.to(cuda_device), step.block_table, a, step.max_seq_len, step.scores)
    torch.cuda.synchronize()
    scores = step.scores.double().cpu()
    G = wl.group
    for r in range(wl.batch):
        n = x.pages_per_request[r]
        for h in range(wl.num_kv_heads):
            qg = x.q[r, h * G:(h + 1) * G].double().sum(0)
            for p in range(n - 1):
                keys = x.k_cache[int(x.block_table[r, p]), h].double()
                true_max = float((keys @ qg).max())
                # fp32 accumulation of ~256 products of magnitude <= ~50: allow 1e-3 relative slack
                assert float(scores[r, h, p]) >= true_max - 1e-3 * max(1.0, abs(true_max)), (r, h, p)


def _scores_both_ways(wl, dev):
    """Scores of one workload through se_quest_score_pages and se_quest_score_pages_ws."""
    x, step, b, a = _prepare(wl, dev)
    q = x.q.to(dev)
    plain = torch.full_like(step.scores, float("nan"))
    pre = torch.full_like(step.scores, float("nan"))
    se.se_quest_score_pages(step.kv, q, step.block_table, a, step.max_seq_len, plain)
    ws = torch.empty(se.se_quest_score_workspace_size(wl.batch, wl.num_kv_heads, wl.head_dim), dtype=torch.uint8,
                     device=dev)
    se.se_quest_score_pages_ws(step.kv, q, step.block_table, a, step.max_seq_len, pre, ws)
    torch.cuda.synchronize()
    return x, plain.cpu(), pre.cpu()


def _check_same_scores(x, plain, pre):
    for r, n in enumerate(x.pages_per_request):
        got, ref = pre[r, :, :max(n - 1, 0)], plain[r, :, :max(n - 1, 0)]
        assert torch.isfinite(ref).all(), r
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), r


@pytest.mark.parametrize("kv_heads,group", [(1, 4), (2, 8), (3, 2), (4, 8), (5, 1), (6, 3), (7, 16), (8, 4)])
def test_score_workspace_gives_the_same_scores(cuda_device, kv_heads, group):
    # every KV-head count of the d-128 kernel; ragged lengths over several CTA slices
    wl = QWEN3_4B_QUEST_32K.scaled(batch=5, num_kv_heads=kv_heads, num_q_heads=kv_heads * group,
                                   context_min=700, context_max=5000, seed=60 + kv_heads)
    _check_same_scores(*_scores_both_ways(wl, cuda_device))


def test_score_workspace_latent_and_many_requests_per_slice(cuda_device):
    # the latent cache (64 query heads of 576 channels); then 1,200 short requests, so that
    # every CTA slice crosses several requests and reads several requests' sums
    wl = MLA_GLM_QUEST_32K.scaled(batch=6, context_min=900, context_max=9000, topk_pages=12, seed=71)
    _check_same_scores(*_scores_both_ways(wl, cuda_device))
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=1200, context_min=17, context_max=120, topk_pages=2,
                                         append=False, seed=72)
    _check_same_scores(*_scores_both_ways(wl, cuda_device))


def test_select_all_equals_dense(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=300, context_max=1000, topk_pages=80,
                                         append=False, seed=17)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    inp = oracle_inputs(x)
    dense = {}
    for r in range(wl.batch):
        n = x.pages_per_request[r]
        assert step.counts[r].tolist() == [n] * wl.num_kv_heads
        dense[r] = [list(range(n))] * wl.num_kv_heads
    ref = oq.decode_step(inp, wl.topk_pages, _scale(wl), pages_override=dense)
    out = step.out.float().cpu().numpy()
    for r in range(wl.batch):
        assert np.abs(out[r] - ref[r].out).max() <= OUT_ATOL


def test_decode_on_the_oracle_selection(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=1500, context_max=3000, topk_pages=20,
                                         append=False, seed=19)
    x, step, b, a = _prepare(wl, cuda_device)
    inp = oracle_inputs(x)
    ref = oq.decode_step(inp, wl.topk_pages, _scale(wl))
    sel = torch.zeros(wl.batch, wl.num_kv_heads, wl.topk_pages + 1, dtype=torch.int32)
    cnt = torch.zeros(wl.batch, wl.num_kv_heads, dtype=torch.int32)
    for r in range(wl.batch):
        for h in range(wl.num_kv_heads):
            pg = ref[r].heads[h].pages
            sel[r, h, :len(pg)] = torch.tensor(pg)
            cnt[r, h] = len(pg)
    step.attend(x.q.to(cuda_device), a, sel.to(cuda_device), cnt.to(cuda_device))
    torch.cuda.synchronize()
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    for r in range(wl.batch):
        assert np.abs(out[r] - ref[r].out).max() <= OUT_ATOL
        assert np.abs(lse[r] - ref[r].lse).max() <= 1e-3


def test_block_table_permutation_is_invisible(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=600, context_max=2000, topk_pages=10, seed=23)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    out1, sel1 = step.out.clone(), step.sel.clone()
    # Same logical content at other physical pages.
    P = x.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)
    k2 = x.k_cache[perm].to(cuda_device)
    v2 = x.v_cache[perm].to(cuda_device)
    bt2 = inv[x.block_table.long()].to(torch.int32)
    step2 = QuestDecodeStep(k2, v2, new_summary(k2), bt2.to(cuda_device), wl.num_q_heads, wl.topk_pages,
                            step.max_seq_len)
    step2.build_summaries(b)
    _run(x, step2, b, a, cuda_device)
    assert torch.equal(sel1, step2.sel)
    assert torch.equal(out1.view(torch.int16), step2.out.view(torch.int16))


def test_split_count_does_not_change_the_result(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=2, context_min=3000, context_max=3000, topk_pages=40,
                                         append=False, seed=29)
    x, s1, b, a = _prepare(wl, cuda_device)
    _run(x, s1, b, a, cuda_device)
    x2, s2, b2, a2 = _prepare(wl, cuda_device, sel_stride=wl.topk_pages + 1 + 200)
    _run(x2, s2, b2, a2, cuda_device)
    assert torch.equal(s1.counts, s2.counts)
    assert torch.equal(s1.sel, s2.sel[:, :, :wl.topk_pages + 1])
    assert (s1.out.float() - s2.out.float()).abs().max().item() <= 1e-2
    assert (s1.lse - s2.lse).abs().max().item() <= 1e-4


def test_decode_twice_on_one_workspace_leaves_its_counters_zero(cuda_device):
    # Items span several CTAs (41 pages each, at least 16 per CTA slice): the CTA that
    # publishes an item's last partial merges them and resets the item's arrival
    # counter. Two calls back to back on one workspace give the same output, and the
    # counters are zero after each.
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=2500, context_max=4000, topk_pages=40,
                                         append=False, seed=33)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    out1, lse1 = step.out.clone(), step.lse.clone()
    nsplit, _, launches = se.se_sparse_decode_plan(wl.batch, wl.num_q_heads, wl.num_kv_heads, 128, 128,
                                                   step.sel_stride)
    assert launches == 1
    rows = wl.batch * wl.num_q_heads
    off = (rows * nsplit * 129 * 4 + 15) // 16 * 16
    counters = step.workspace[off:off + 4 * wl.batch * wl.num_kv_heads]
    assert int(counters.count_nonzero()) == 0
    for _ in range(2):
        step.out.fill_(float("nan"))
        step.attend(x.q.to(cuda_device), a)
        torch.cuda.synchronize()
        assert torch.equal(step.out.view(torch.int16), out1.view(torch.int16))
        assert torch.equal(step.lse, lse1)
        assert int(counters.count_nonzero()) == 0
    compare_decode(x, step, list(range(wl.batch)), _scale(wl), "twice")


def test_select_pages_entry_point_matches_the_two_calls(cuda_device):
    wl = QWEN3_4B_QUEST_32K.scaled(batch=2, context_min=2000, context_max=2400, topk_pages=16, seed=31)
    x, step, b, a = _prepare(wl, cuda_device)
    q = x.q.to(cuda_device)
    step.select(q, a)
    ws = torch.empty(se.se_quest_select_workspace_size(wl.batch, wl.num_kv_heads, step.max_seq_len),
                     dtype=torch.uint8, device=cuda_device)
    sel = torch.empty_like(step.sel)
    cnt = torch.empty_like(step.counts)
    se.se_quest_select_pages(step.kv, q, step.block_table, a, step.max_seq_len, wl.topk_pages, sel, cnt, ws)
    torch.cuda.synchronize()
    assert torch.equal(cnt, step.counts) and torch.equal(sel, step.sel)


def test_out_of_range_page_id_sets_the_error_word(cuda_device):
    wl = TINY_QUEST_4K.scaled(context_min=160, context_max=160, topk_pages=4)
    x, step, b, a = _prepare(wl, cuda_device)
    bad = step.block_table.clone()
    bad[0, 3] = x.num_pages + 5          # outside the pool: every kernel checks and skips it
    step.block_table = bad
    step.kv = se.paged_kv(step.k_cache, step.v_cache, step.summary)
    se.se_quest_score_pages(step.kv, x.q.to(cuda_device), bad, a, step.max_seq_len, step.scores)
    torch.cuda.synchronize()
    assert se.se_read_device_error(clear=True) & se.DEVERR_PAGE_RANGE
    assert float(step.scores[0, 0, 3]) == float("-inf")


def test_short_workspace_is_rejected(cuda_device):
    wl = TINY_QUEST_4K
    x, step, b, a = _prepare(wl, cuda_device)
    with pytest.raises(se.SparseEngineError) as e:
        se.se_sparse_paged_decode(step.kv, x.q.to(cuda_device), step.block_table, a, step.sel, step.counts, 0.1,
                                  step.out, None, step.workspace[:16])
    assert e.value.status == 3


# ---------------------------------------------------------------- full size, sampled requests
@pytest.mark.parametrize("kind", ["h4", "h8", "latent"])
def test_score_unit_pool_gives_the_same_scores(cuda_device, kind):
    # At least 128 candidate pages per CTA: with the workspace the scoring kernel
    # puts a quarter of the pages in a pool of 8-page units that free warps take,
    # so which warp scores a page depends on timing. Every score must still equal,
    # bit for bit, the one of the call without the workspace (equal slices only).
    if kind == "latent":
        wl = MLA_GLM_QUEST_32K.scaled(batch=22, seed=81)
    else:
        hkv = 4 if kind == "h4" else 8
        wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=6, num_kv_heads=hkv, num_q_heads=4 * hkv,
                                             context_min=120000, context_max=131072, append=False,
                                             seed=80 + hkv)
    x, plain, pre = _scores_both_ways_dev(wl, cuda_device)
    total = sum(max(n - 1, 0) for n in x.pages_per_request)
    assert total >= 128 * 2 * torch.cuda.get_device_properties(cuda_device).multi_processor_count
    _check_same_scores(x, plain, pre)


def _scores_both_ways_dev(wl, dev):
    """_scores_both_ways with the inputs generated on the device (large workloads)."""
    x, step, b, a = _prepare(wl, dev, device_gen=True)
    q = x.q.to(dev)
    plain = torch.full_like(step.scores, float("nan"))
    pre = torch.full_like(step.scores, float("nan"))
    se.se_quest_score_pages(step.kv, q, step.block_table, a, step.max_seq_len, plain)
    ws = torch.empty(se.se_quest_score_workspace_size(wl.batch, wl.num_kv_heads, wl.head_dim), dtype=torch.uint8,
                     device=dev)
    for _ in range(2):  # the second call finds the pool counter as the first left it
        pre.fill_(float("nan"))
        se.se_quest_score_pages_ws(step.kv, q, step.block_table, a, step.max_seq_len, pre, ws)
    torch.cuda.synchronize()
    return x, plain.cpu(), pre.cpu()


@pytest.mark.parametrize("hq,hkv,topk", [(32, 2, 600), (32, 4, 400)])
def test_decode_items_over_many_slices(cuda_device, hq, hkv, topk):
    # One request whose items (KV heads) hold hundreds of selected pages: at 16
    # pages per CTA slice each item spans 25-40 CTAs, so the CTA that completes an
    # item's count merges its partials in many batches of four, and every CTA's
    # slice ends mid-item. Groups of 16 (the two-row MMA states) and 8 query heads.
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=1, num_q_heads=hq, num_kv_heads=hkv, context_min=40000,
                                         context_max=40000, topk_pages=topk, append=False, seed=90 + hkv)
    x, step, b, a = _prepare(wl, cuda_device)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, [0], _scale(wl), f"many slices G={hq // hkv}")


def test_full_qwen3_4b_32k_sampled(cuda_device):
    wl = QWEN3_4B_QUEST_32K
    x, step, b, a = _prepare(wl, cuda_device, device_gen=True)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, [0, wl.batch - 1], _scale(wl), "qwen3-4b full")


def test_full_qwen3_30b_a3b_128k_sampled(cuda_device):
    wl = QWEN3_30B_A3B_QUEST_128K
    x, step, b, a = _prepare(wl, cuda_device, device_gen=True)
    _run(x, step, b, a, cuda_device)
    longest = int(np.argmax(x.seq_lens))
    shortest = int(np.argmin(x.seq_lens))
    compare_decode(x, step, sorted({longest, shortest, 7}), _scale(wl), "qwen3-30b full")


# ---------------------------------------------------------------- scores of a large batch, sampled pages
@pytest.mark.parametrize("hkv,head_dim", [(1, 128), (2, 128), (3, 128), (4, 128), (5, 128), (6, 128), (7, 128),
                                          (8, 128), (1, 576)])
def test_scores_on_sampled_pages_of_a_large_batch(cuda_device, hkv, head_dim):
    """About 100K candidate pages, so that every CTA's slice holds more than 256
    pages of one request and each scoring warp walks past its first 32-page
    block-table window; scores of sampled pages (the window edges included)
    against the oracle bound recomputed from those pages' keys."""
    if head_dim == 576:
        wl = MLA_GLM_QUEST_32K.scaled(batch=50, seed=61)
    else:
        wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=25, num_kv_heads=hkv, num_q_heads=4 * hkv,
                                             context_min=64000, context_max=64000, append=False, seed=60 + hkv)
    x, step, b, a = _prepare(wl, cuda_device, device_gen=True)
    step.select(x.q, a)
    torch.cuda.synchronize()
    scores = step.scores.cpu().numpy()
    G = wl.num_q_heads // wl.num_kv_heads
    rng = np.random.default_rng(0)
    q = x.q.float().cpu().numpy().astype(np.float64)
    for r in range(wl.batch):
        n = math.ceil(x.seq_lens_after[r] / wl.page_size)
        pages = {0, 255, 256, 257, 263, 264, 511, 512, n - 2} | set(rng.integers(0, n - 1, 12).tolist())
        for p in sorted(pg for pg in pages if 0 <= pg < n - 1):
            phys = int(x.block_table[r, p])
            blk = x.k_cache[phys].double().cpu().numpy()          # [Hkv][16][D], a full page
            for h in range(wl.num_kv_heads):
                m, M = oq.page_summary(blk[h])
                qg = q[r, h * G:(h + 1) * G]
                want = oq.group_page_scores(qg, m[None, :], M[None, :])[0]
                scale = np.maximum(np.abs(qg * m), np.abs(qg * M)).sum()
                got = float(scores[r, h, p])
                assert abs(got - want) <= 2e-5 * scale + 1e-6, (r, h, p, got, want)


# ---------------------------------------------------------------- sink / recent keep windows
@pytest.mark.parametrize("sink,recent", [(64, 512), (16, 64), (64, 256), (0, 512), (64, 0), (100, 37)])
def test_windowed_selection_oracle_sized(cuda_device, sink, recent):
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=4, context_min=900, context_max=4100, topk_pages=24, seed=71)
    x, step, b, a = _prepare(wl, cuda_device, sink=sink, recent=recent)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"windows {sink}/{recent}", sink, recent)


@pytest.mark.parametrize("sel_stride", [None, 80])
def test_windowed_edge_lengths(cuda_device, sel_stride):
    # windows that overlap each other or cover the whole request, unaligned lengths
    lens = (0, 1, 15, 16, 17, 63, 64, 65, 130, 600)
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=len(lens), lengths=lens, topk_pages=2, append=False, seed=73)
    x, step, b, a = _prepare(wl, cuda_device, sel_stride=sel_stride, sink=64, recent=64)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "windowed edges", 64, 64)


def test_windowed_full_qwen3_30b_a3b_128k_sampled(cuda_device):
    # The decode-time keep settings of the throughput runs: sink 64, recent 512, 1,472 selected.
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(topk_pages=92)
    x, step, b, a = _prepare(wl, cuda_device, device_gen=True, sink=64, recent=512)
    _run(x, step, b, a, cuda_device)
    compare_decode(x, step, [0, 9, wl.batch - 1], _scale(wl), "windowed 128k", 64, 512)


# ---------------------------------------------------------------- top-k on crafted scores
def _topk_case(scores_rows, lens, k, dev, sink=0, recent=0):
    """Run the top-k entry point on given fp32 scores [B][1][stride]; compare with the oracle exactly."""
    B = len(lens)
    stride = scores_rows.shape[-1]
    max_len = max(lens)
    sc = scores_rows.to(dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    sel = torch.full((B, 1, se.se_quest_kept_pages_max(k, sink, recent)), -7, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, 1, dtype=torch.int32, device=dev)
    if sink == 0 and recent == 0:
        se.se_quest_topk_pages(sc, lens_t, 1, max_len, k, sel, cnt)
    else:
        se.se_quest_topk_pages_windowed(sc, lens_t, 1, max_len, k, sink, recent, sel, cnt)
    torch.cuda.synchronize()
    for b, L in enumerate(lens):
        n = math.ceil(L / 16)
        s = scores_rows[b, 0].double().numpy()
        ref = oq.select_pages(s, n, k) if sink == 0 and recent == 0 else \
            oq.select_pages_windowed(s, L, 16, k, sink, recent)
        got = sel[b, 0, :int(cnt[b, 0])].tolist()
        assert got == ref, (b, L, got[:8], ref[:8])


@pytest.mark.parametrize("kind", ["distinct", "all_equal", "few_values", "with_neg_inf", "near_ties"])
def test_topk_exact_on_crafted_scores(cuda_device, kind):
    g = torch.Generator().manual_seed(3)
    lens = [16 * 300, 16 * 2000 + 5, 16 * 6145, 16 * 8193, 16 * 40 + 1]
    stride = max(math.ceil(L / 16) for L in lens)
    B = len(lens)
    if kind == "distinct":
        s = torch.randn(B, 1, stride, generator=g)
    elif kind == "all_equal":
        s = torch.full((B, 1, stride), 1.25)
    elif kind == "few_values":
        s = torch.randint(0, 5, (B, 1, stride), generator=g).float()
    elif kind == "with_neg_inf":
        s = torch.randn(B, 1, stride, generator=g)
        s[torch.rand(B, 1, stride, generator=g) < 0.3] = float("-inf")
    else:  # many scores within a few ulps of each other: crowded buckets, exact order still defined
        s = 100.0 + torch.randint(0, 3000, (B, 1, stride), generator=g).float() * 1e-5
    for k in (1, 37, 256):
        _topk_case(s, lens, k, cuda_device)
        _topk_case(s, lens, k, cuda_device, sink=64, recent=512)


def test_topk_beyond_8192_candidates_uses_the_shared_memory_kernel(cuda_device):
    g = torch.Generator().manual_seed(4)
    lens = [16 * 10000, 16 * 9000 + 3]
    stride = 10000
    s = torch.randn(2, 1, stride, generator=g)
    s[0, 0, ::7] = 0.5  # ties
    _topk_case(s, lens, 300, cuda_device)
    _topk_case(s, lens, 300, cuda_device, sink=100, recent=700)


def test_overlapped_append_serial_order_and_graph_replay_agree(cuda_device):
    """The step without events runs score, top-k, append (alongside the top-k), decode; with
    events it runs append, score, top-k, decode; captured in a CUDA graph it runs the first
    order under programmatic dependent launch. All three give the same selection, output
    and lse, bit for bit (the append is idempotent, so they share one cache)."""
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(batch=6, context_min=3000, context_max=9000, topk_pages=24, seed=83)
    x, step, before, after = _prepare(wl, cuda_device)
    dev = cuda_device
    q, kn, vn = x.q.to(dev), x.k_new.to(dev), x.v_new.to(dev)
    s = torch.cuda.Stream(dev)
    results = []
    with torch.cuda.stream(s):
        step.run(q, after, kn, vn, before, stream=s)                      # overlapped
    s.synchronize()
    results.append((step.sel.clone(), step.counts.clone(), step.out.clone(), step.lse.clone()))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(s):
        step.run(q, after, kn, vn, before, stream=s, events=ev)           # serial
    s.synchronize()
    results.append((step.sel.clone(), step.counts.clone(), step.out.clone(), step.lse.clone()))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
        step.run(q, after, kn, vn, before, stream=s)
    for _ in range(3):
        step.out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    results.append((step.sel.clone(), step.counts.clone(), step.out.clone(), step.lse.clone()))
    for r in results[1:]:
        assert torch.equal(r[1], results[0][1])
        for bh in range(wl.batch * wl.num_kv_heads):
            n = int(r[1].view(-1)[bh])
            assert torch.equal(r[0].view(wl.batch * wl.num_kv_heads, -1)[bh, :n],
                               results[0][0].view(wl.batch * wl.num_kv_heads, -1)[bh, :n])
        assert torch.equal(r[2], results[0][2])
        assert torch.equal(r[3], results[0][3])
    compare_decode(x, step, range(wl.batch), _scale(wl), "graph-replayed overlapped step")
