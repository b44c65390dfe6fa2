"""The seeded input generators: determinism, valid block tables, poison placement."""
import math

import torch

from synth import (TINY_QUEST_4K, QWEN3_30B_A3B_QUEST_128K, SNAPKV_PREFILL_32K, MLA_GLM_QUEST_32K,
                   make_quest_decode_inputs, make_snapkv_inputs)


def _small_ragged():
    return QWEN3_30B_A3B_QUEST_128K.scaled(batch=3, context_min=40, context_max=90)


def test_quest_inputs_deterministic():
    a = make_quest_decode_inputs(_small_ragged())
    b = make_quest_decode_inputs(_small_ragged())
    assert a.seq_lens == b.seq_lens
    assert torch.equal(a.block_table, b.block_table)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.q, b.q)


def test_block_table_is_a_partition_of_the_pool():
    x = make_quest_decode_inputs(_small_ragged())
    used = []
    for b, n in enumerate(x.pages_per_request):
        used += x.block_table[b, :n].tolist()
        assert n == math.ceil((x.seq_lens[b] + 1) / 16)
    assert sorted(used) == list(range(x.num_pages))


def test_poison_only_past_the_length():
    x = make_quest_decode_inputs(_small_ragged())
    for b, L in enumerate(x.seq_lens):
        for pos in range(x.pages_per_request[b] * 16):
            phys = int(x.block_table[b, pos // 16])
            row = x.k_cache[phys, :, pos % 16, :].float()
            assert bool(torch.isnan(row).all()) == (pos >= L), (b, pos)


def test_outlier_channels_scaled():
    x = make_quest_decode_inputs(TINY_QUEST_4K.scaled(context_min=1024, context_max=1024))
    k = x.k_cache.float()[:, 0].reshape(-1, 128)
    std = k.std(dim=0)
    ch = x.outlier_channels[0]
    assert len(ch) == 4
    assert bool((std[ch] > 6).all()) and float(std[[c for c in range(128) if c not in ch]].max()) < 1.2


def test_latent_outliers_outside_the_value():
    wl = MLA_GLM_QUEST_32K.scaled(batch=2, context_min=64, context_max=64)
    x = make_quest_decode_inputs(wl)
    assert x.v_cache is None and x.k_cache.shape[-1] == 576
    assert all(512 <= c < 576 for c in x.outlier_channels[0])


def test_latent_outliers_over_the_whole_row():
    # outliers_in_value draws the outlier channels over all 576 dims, the value's
    # too, and scales them by outlier_scale
    wl = MLA_GLM_QUEST_32K.scaled(batch=2, context_min=512, context_max=512, outliers_in_value=True,
                                  outlier_channels=12, outlier_scale=3.0, seed=73)
    x = make_quest_decode_inputs(wl)
    ch = x.outlier_channels[0]
    assert len(ch) == 12 and any(c < 512 for c in ch) and all(0 <= c < 576 for c in ch)
    std = x.k_cache.float()[:, 0].reshape(-1, 576).std(dim=0)
    assert bool((std[ch] > 2.5).all()) and float(std[[c for c in range(576) if c not in ch]].max()) < 1.2


def test_snapkv_inputs():
    wl = SNAPKV_PREFILL_32K.scaled(batch=2, prompt_min=100, prompt_max=300)
    x = make_snapkv_inputs(wl)
    assert x.q_window.shape == (2, 32, 32, 128)
    for b, n in enumerate(x.prompt_lens):
        assert x.dst_pages_per_request[b] == math.ceil(min(n, 2048) / 16)
        for h in range(8):
            assert len(x.sink_positions[b][h]) == round(0.05 * n)
