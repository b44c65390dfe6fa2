"""SnapKV eviction on the GPU against the fp64 oracle (through the C ABI).

Window row log-sum-exps and candidate scores against the oracle's softmax
definition; kept positions under the selection rule (exempt within 1e-3
relative of the keep-th pooled score); compaction byte-exact; the selection
kernel alone on crafted scores (ties, crowded buckets) bit-exact; the full
32K workload on sampled (request, KV head) pairs.
"""
import math

import numpy as np
import pytest
import torch

import oracle.snapkv as osk
import sparse_decode_attention_quest_gb300 as se
from synth import SNAPKV_AGENT_32K, SNAPKV_AIME_32K, SNAPKV_PREFILL_32K, make_snapkv_inputs
from tests.parity import exempt

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_errors(se_lib, cuda_device):
    se.se_read_device_error(clear=True)
    yield
    assert se.se_read_device_error(clear=True) == 0


def _run(x, dev, keep=None, pool=None):
    wl = x.workload
    keep = wl.keep_topk if keep is None else keep
    pool = wl.pool_kernel if pool is None else pool
    k, v = x.k_cache.to(dev), x.v_cache.to(dev)
    src = se.paged_kv(k, v, None)
    bt = x.src_block_table.to(dev)
    lens = torch.tensor(x.prompt_lens, dtype=torch.int32, device=dev)
    max_len = max(x.prompt_lens)
    W, G, H, B = wl.window, wl.group, wl.num_kv_heads, wl.batch
    stride = max(max_len - W, 1)
    scores = torch.full((B, H, stride), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, H, W * G), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(se.se_snapkv_workspace_size(B, H, W, max_len), dtype=torch.uint8, device=dev)
    qw = x.q_window.to(dev)
    scale = 1.0 / math.sqrt(wl.head_dim)
    se.se_snapkv_window_scores(src, qw, bt, lens, max_len, scale, scores, lse, ws)
    S, R = wl.keep_sink, wl.recent
    kept = torch.full((B, H, S + keep + R), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, H, dtype=torch.int32, device=dev)
    if S == 0 and R == W:
        se.se_snapkv_select(scores, lens, H, W, max_len, pool, keep, kept, cnt)
    else:
        se.se_snapkv_select_windowed(scores, lens, H, W, max_len, pool, keep, S, R, kept, cnt)
    dk = torch.full((x.dst_num_pages, H, 16, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    dv = torch.full_like(dk, float("nan"))
    dst = se.paged_kv(dk, dv, None)
    dbt = x.dst_block_table.to(dev)
    se.se_snapkv_compact(src, bt, lens, dst, dbt, kept, cnt)
    torch.cuda.synchronize()
    return dict(scores=scores.cpu(), lse=lse.cpu(), kept=kept.cpu(), cnt=cnt.cpu(), dk=dk.cpu(), dv=dv.cpu(),
                ws=ws, src=src, qw=qw, bt=bt, lens=lens, dst=dst, dbt=dbt, scale=scale, keep=keep, pool=pool,
                sink=S, recent=R)


def _check_pair(x, res, b, h):
    wl = x.workload
    W, G = wl.window, wl.group
    n = x.prompt_lens[b]
    ref = osk.snapkv_head(x.q_window[b, :, h * G:(h + 1) * G, :], x.k_cache, x.src_block_table[b], h, n, W,
                          res["pool"], res["keep"], res["scale"], sink=res["sink"], recent=res["recent"])
    # row log-sum-exp (fp32 sums of exact bf16 products)
    np.testing.assert_allclose(res["lse"][b, h].numpy(), ref["lse"].reshape(-1), rtol=0, atol=2e-3)
    # candidate scores (probability sums, fp32)
    got = res["scores"][b, h, :n - W].double().numpy()
    np.testing.assert_allclose(got, ref["scores"], rtol=2e-3, atol=1e-6)
    # kept positions: exact except candidates within 1e-3 of the keep-th pooled score
    cnt = int(res["cnt"][b, h])
    assert cnt == len(ref["kept"]), (cnt, len(ref["kept"]))
    kept = res["kept"][b, h, :cnt].tolist()
    assert kept == sorted(set(kept))
    assert set(range(max(0, n - res["recent"]), n)) <= set(kept) and set(range(min(res["sink"], n))) <= set(kept)
    gs, rs = set(kept), set(ref["kept"])
    for j in range(n - W):
        if (j in gs) != (j in rs):
            assert exempt(ref["pooled"][j], ref["threshold"]), (b, h, j, ref["pooled"][j], ref["threshold"])
    # compaction: kept token t is byte-identical at (dst page t // 16, slot t % 16)
    src_rows_k = torch.stack([x.k_cache[int(x.src_block_table[b, j // 16]), h, j % 16] for j in kept])
    src_rows_v = torch.stack([x.v_cache[int(x.src_block_table[b, j // 16]), h, j % 16] for j in kept])
    dst_k = torch.stack([res["dk"][int(x.dst_block_table[b, t // 16]), h, t % 16] for t in range(cnt)])
    dst_v = torch.stack([res["dv"][int(x.dst_block_table[b, t // 16]), h, t % 16] for t in range(cnt)])
    assert torch.equal(src_rows_k.view(torch.int16), dst_k.view(torch.int16))
    assert torch.equal(src_rows_v.view(torch.int16), dst_v.view(torch.int16))


def test_snapkv_oracle_sized_ragged(cuda_device):
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=700, prompt_max=2600, keep_topk=96)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device)
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            _check_pair(x, res, b, h)


@pytest.mark.parametrize("pool", [1, 3, 17, 21])  # 17: the widest window pooled by shuffles; 21: the loop
def test_snapkv_pool_sizes_and_small_windows(cuda_device, pool):
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, num_q_heads=16, num_kv_heads=4, window=16, prompt_min=300,
                                   prompt_max=1000, keep_topk=40, seed=8)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device, pool=pool)
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            _check_pair(x, res, b, h)


@pytest.mark.parametrize("n", [2048, 32])
def test_snapkv_short_prompts_keep_everything(cuda_device, n):
    # n - W == keep: every position is kept; n == W: only the window (no candidate).
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=n, prompt_max=n, keep_topk=2016, seed=9)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device)
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            assert int(res["cnt"][b, h]) == n
            assert res["kept"][b, h, :n].tolist() == list(range(n))
            _check_pair(x, res, b, h)


def test_snapkv_score_and_compact_matches_the_steps(cuda_device):
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=1500, prompt_max=3000, keep_topk=128, seed=10)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device)
    B, H, W = wl.batch, wl.num_kv_heads, wl.window
    max_len = max(x.prompt_lens)
    ws = torch.empty(se.se_snapkv_workspace_size(B, H, W, max_len), dtype=torch.uint8, device=cuda_device)
    kept = torch.full((B, H, 128 + W), -1, dtype=torch.int32, device=cuda_device)
    cnt = torch.zeros(B, H, dtype=torch.int32, device=cuda_device)
    dk = torch.zeros((x.dst_num_pages, H, 16, 128), dtype=torch.bfloat16, device=cuda_device)
    dv = torch.zeros_like(dk)
    se.se_snapkv_score_and_compact(res["src"], res["qw"], res["bt"], res["lens"], max_len, wl.pool_kernel, 128,
                                   res["scale"], se.paged_kv(dk, dv, None), res["dbt"], kept, cnt, ws)
    torch.cuda.synchronize()
    assert torch.equal(kept.cpu(), res["kept"]) and torch.equal(cnt.cpu(), res["cnt"])
    for b in range(B):
        n_pages = x.dst_pages_per_request[b]
        idx = x.dst_block_table[b, :n_pages].long()
        assert torch.equal(dk.cpu()[idx].view(torch.int16), res["dk"][idx].view(torch.int16))


@pytest.mark.parametrize("kind", ["distinct", "ties", "flat"])
def test_snapkv_select_exact_on_crafted_scores(cuda_device, kind):
    g = torch.Generator().manual_seed(11)
    W, H = 32, 2
    lens = [5000, 30000]
    stride = max(lens) - W
    if kind == "distinct":
        s = torch.rand(2, H, stride, generator=g)
    elif kind == "ties":
        s = torch.randint(0, 4, (2, H, stride), generator=g).float() * 0.25
    else:
        s = torch.full((2, H, stride), 0.125)
    keep = 2016
    dev = cuda_device
    kept = torch.full((2, H, keep + W), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(2, H, dtype=torch.int32, device=dev)
    se.se_snapkv_select(s.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev), H, W, max(lens), 7, keep,
                        kept, cnt)
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        for h in range(H):
            pooled = osk.max_pool_clipped(s[b, h, :n - W].double().numpy(), 7)
            ref = osk.keep_positions(pooled, n, W, keep)
            assert kept[b, h, :int(cnt[b, h])].tolist() == ref, (kind, b, h)


def test_snapkv_full_32k_sampled(cuda_device):
    wl = SNAPKV_PREFILL_32K
    x = make_snapkv_inputs(wl, device=cuda_device)
    res = _run(x, cuda_device)
    xc = x  # inputs stay on the device; copy the sampled pairs' data for the oracle
    xc.k_cache = x.k_cache.cpu()
    xc.v_cache = x.v_cache.cpu()
    xc.q_window = x.q_window.cpu()
    xc.src_block_table = x.src_block_table.cpu()
    xc.dst_block_table = x.dst_block_table.cpu()
    for b, h in ((0, 0), (wl.batch - 1, wl.num_kv_heads - 1), (1, 3)):
        _check_pair(xc, res, b, h)


def test_snapkv_is_repeatable(cuda_device):
    # the full 4 x 32K eviction (tcgen05 score passes, selection, gather) run again gives
    # bit-identical scores, row log-sum-exps, kept positions and compacted rows
    x = make_snapkv_inputs(SNAPKV_PREFILL_32K, device=cuda_device)
    first = _run(x, cuda_device)
    for _ in range(4):
        again = _run(x, cuda_device)
        for key in ("scores", "lse", "kept", "cnt"):
            assert torch.equal(first[key].view(torch.int32), again[key].view(torch.int32)), key
        for key in ("dk", "dv"):
            assert torch.equal(first[key].view(torch.int16), again[key].view(torch.int16)), key


# ---------------------------------------------------------------- keep windows (sink / recent)
@pytest.mark.parametrize("W,S,R,keep", [(16, 16, 64, 96), (32, 64, 512, 300), (32, 0, 256, 200), (32, 64, 32, 100)])
def test_snapkv_windows_oracle_sized(cuda_device, W, S, R, keep):
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=700, prompt_max=2600, window=W, keep_topk=keep, keep_sink=S,
                                   keep_recent=R, seed=12)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device)
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            _check_pair(x, res, b, h)


@pytest.mark.parametrize("kind", ["distinct", "ties"])
def test_snapkv_windowed_select_exact_on_crafted_scores(cuda_device, kind):
    g = torch.Generator().manual_seed(13)
    W, H, S, R, keep = 16, 2, 64, 512, 4096
    lens = [5000, 30000, 600]
    stride = max(lens) - W
    s = torch.rand(3, H, stride, generator=g) if kind == "distinct" else \
        torch.randint(0, 4, (3, H, stride), generator=g).float() * 0.25
    dev = cuda_device
    kept = torch.full((3, H, S + keep + R), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(3, H, dtype=torch.int32, device=dev)
    se.se_snapkv_select_windowed(s.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev), H, W, max(lens), 7,
                                 keep, S, R, kept, cnt)
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        for h in range(H):
            pooled = osk.max_pool_clipped(s[b, h, :n - W].double().numpy(), 7)
            ref = osk.keep_positions_windowed(pooled, n, W, keep, S, R)
            assert kept[b, h, :int(cnt[b, h])].tolist() == ref, (kind, b, h)


def _full_sampled(wl, dev, pairs):
    x = make_snapkv_inputs(wl, device=dev)
    res = _run(x, dev)
    x.k_cache, x.v_cache, x.q_window = x.k_cache.cpu(), x.v_cache.cpu(), x.q_window.cpu()
    x.src_block_table, x.dst_block_table = x.src_block_table.cpu(), x.dst_block_table.cpu()
    for b, h in pairs:
        _check_pair(x, res, b, h)


def test_snapkv_many_chunks_sampled(cuda_device):
    # 160 (request, KV head) pairs of 1.5K-6K tokens: the score kernel cuts them into
    # chunks of about 21 pairs (pass 2 of a chunk runs one phase after its pass 1),
    # so pairs on both sides of several chunk boundaries are checked.
    wl = SNAPKV_PREFILL_32K.scaled(batch=40, num_q_heads=16, num_kv_heads=4, prompt_min=1500, prompt_max=6000,
                                   keep_topk=300, seed=16)
    _full_sampled(wl, cuda_device, ((0, 0), (5, 0), (5, 1), (10, 3), (21, 2), (39, 3)))


def test_snapkv_more_pairs_than_one_launch(cuda_device):
    # 2,056 pairs of short prompts (33-200 tokens, some of them only the window plus one
    # candidate) take two launches of the score kernel; pairs of both are checked.
    wl = SNAPKV_PREFILL_32K.scaled(batch=257, prompt_min=33, prompt_max=200, keep_topk=20, seed=17)
    _full_sampled(wl, cuda_device, ((0, 0), (100, 5), (255, 7), (256, 0), (256, 7)))


def test_snapkv_aime_budget_full_32k_sampled(cuda_device):
    # 16-query window, sink 16, recent 64, 4,096 selected
    _full_sampled(SNAPKV_AIME_32K, cuda_device, ((0, 0), (3, 7)))


def test_snapkv_agent_budget_full_32k_sampled(cuda_device):
    # sink 64, recent 512, 15,808 selected: half of each 32K prompt kept
    _full_sampled(SNAPKV_AGENT_32K, cuda_device, ((1, 2), (2, 5)))


# ---------------------------------------------------------------- periodic eviction during decode
def test_periodic_decode_eviction_over_compacted_pages(cuda_device):
    """Prefill eviction (3,000-token prompts, window 16, sink 16, recent 64, 400 selected), then
    one period of 64 decode steps appended to the compacted pages, then the periodic eviction
    over them; the second eviction is checked against the oracle on the logical sequence
    (prefill-kept rows, then the appended rows) with the last 16 decode queries as window."""
    from sparse_decode_attention_quest_gb300.pipeline import SnapKVDecodeCache
    dev = cuda_device
    wl = SNAPKV_AIME_32K.scaled(batch=2, prompt_min=3000, prompt_max=3000, keep_topk=400, seed=14)
    x = make_snapkv_inputs(wl)
    B, H, Hq, D, W = wl.batch, wl.num_kv_heads, wl.num_q_heads, wl.head_dim, wl.window
    S, R, K, pool, period = wl.keep_sink, wl.recent, wl.keep_topk, wl.pool_kernel, 64
    scale = 1.0 / math.sqrt(D)
    cache = SnapKVDecodeCache(B, H, Hq, D, W, pool, K, S, R, period, dev)
    lens = torch.tensor(x.prompt_lens, dtype=torch.int32, device=dev)
    cache.evict_from(se.paged_kv(x.k_cache.to(dev), x.v_cache.to(dev), None), x.src_block_table.to(dev), lens,
                     x.q_window.to(dev), max(x.prompt_lens))
    torch.cuda.synchronize()
    G = wl.group
    n0 = x.prompt_lens[0]
    kept0 = {}
    for b in range(B):
        for h in range(H):
            ref = osk.snapkv_head(x.q_window[b, :, h * G:(h + 1) * G, :], x.k_cache, x.src_block_table[b], h, n0, W,
                                  pool, K, scale, sink=S, recent=R)
            got = cache.kept[b, h, :int(cache.counts[b, h])].tolist()
            assert got == ref["kept"], (b, h)  # no ties at the threshold for this seed
            kept0[(b, h)] = ref["kept"]
    g = torch.Generator().manual_seed(15)
    k_app = torch.randn(period, B, H, D, generator=g).to(torch.bfloat16)
    v_app = torch.randn(period, B, H, D, generator=g).to(torch.bfloat16)
    q_dec = torch.randn(period, B, Hq, D, generator=g).to(torch.bfloat16)
    for t in range(period):
        cache.append(k_app[t].to(dev), v_app[t].to(dev), q_dec[t].to(dev))
    torch.cuda.synchronize()
    assert cache.evictions == 2 and cache.steps == 0
    kk, kv_ = cache.k[cache.live].cpu(), cache.v[cache.live].cpu()
    for b in range(B):
        for h in range(H):
            rows_k = [x.k_cache[int(x.src_block_table[b, j // 16]), h, j % 16] for j in kept0[(b, h)]]
            rows_k += [k_app[t, b, h] for t in range(period)]
            rows_v = [x.v_cache[int(x.src_block_table[b, j // 16]), h, j % 16] for j in kept0[(b, h)]]
            rows_v += [v_app[t, b, h] for t in range(period)]
            n1 = len(rows_k)
            npg = -(-n1 // 16)
            logical = torch.zeros(npg, H, 16, D, dtype=torch.bfloat16)
            padded = torch.zeros(npg * 16, D, dtype=torch.bfloat16)
            padded[:n1] = torch.stack(rows_k)
            logical[:, h] = padded.view(npg, 16, D)
            qw = q_dec[period - W:, b, h * G:(h + 1) * G, :]          # [W][G][D], oldest first
            ref = osk.snapkv_head(qw, logical, torch.arange(npg), h, n1, W, pool, K, scale, sink=S, recent=R)
            cnt = int(cache.counts[b, h])
            got = cache.kept[b, h, :cnt].tolist()
            assert cnt == len(ref["kept"])
            gs, rs = set(got), set(ref["kept"])
            for j in range(n1 - W):
                if (j in gs) != (j in rs):
                    assert exempt(ref["pooled"][j], ref["threshold"]), (b, h, j)
            # the compacted rows are the logical rows at the kept positions, bit for bit
            for t, j in enumerate(got):
                page = int(cache.block_table[b, t // 16])
                assert torch.equal(kk[page, h, t % 16].view(torch.int16), rows_k[j].view(torch.int16))
                assert torch.equal(kv_[page, h, t % 16].view(torch.int16), rows_v[j].view(torch.int16))


def test_a_wait_that_runs_out_sets_the_error_word_and_the_next_call_is_correct(cuda_device):
    """The score kernel's mbarrier waits are bounded. With the wait probe, the MMA issuer
    of every CTA waits on a barrier phase that nothing completes; after 200 us it gives
    up, sets SE_DEVERR_WAIT_TIMEOUT and the kernel finishes (copies drained, tensor
    memory freed). The next call in the same process is correct."""
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=1500, prompt_max=3000, keep_topk=100, seed=18)
    x = make_snapkv_inputs(wl)
    res = _run(x, cuda_device)
    se.se_read_device_error(clear=True)
    se.se_debug_snapkv_wait_probe(200)
    scores = torch.zeros_like(res["scores"]).to(cuda_device)
    max_len = max(x.prompt_lens)
    se.se_snapkv_window_scores(res["src"], res["qw"], res["bt"], res["lens"], max_len, res["scale"], scores, None,
                               res["ws"])
    torch.cuda.synchronize()
    assert se.se_read_device_error(clear=True) & se.DEVERR_WAIT_TIMEOUT
    again = _run(x, cuda_device)
    assert torch.equal(again["scores"].view(torch.int32), res["scores"].view(torch.int32))
    for b, h in ((0, 0), (1, 5)):
        _check_pair(x, again, b, h)
