"""Budget accounting against the rows the settings tables print (tests/golden/table_budgets.json)."""
import json
import os

import pytest

import numpy as np

from oracle import budgets
from oracle import quest
from oracle import snapkv
from synth import SNAPKV_PREFILL_32K, QWEN3_30B_A3B_QUEST_128K, QWEN3_4B_QUEST_32K

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "table_budgets.json")))


@pytest.mark.parametrize("row", GOLD["rows"], ids=lambda r: r["cite"])
def test_total_is_selected_plus_sink_plus_recent(row):
    assert budgets.total_kept_tokens(row["selected"], row["sink"], row["recent"]) == row["total"]
    if "pages" in row:
        assert budgets.selected_pages(row["selected"]) == row["pages"]


def test_workload_budgets_follow_the_tables():
    # 2,048 and 4,096 selected tokens are 128 and 256 sixteen-token pages.
    assert QWEN3_4B_QUEST_32K.topk_pages == budgets.selected_pages(2048)
    assert QWEN3_30B_A3B_QUEST_128K.topk_pages == budgets.selected_pages(4096)
    s = GOLD["snapkv_longbench"]
    wl = SNAPKV_PREFILL_32K
    assert (wl.keep_topk, wl.window, wl.pool_kernel) == (s["selected"], s["recent"], s["pooling_kernel"])
    assert s["scoring_window"] == wl.window
    assert budgets.total_kept_tokens(wl.keep_topk, s["sink"], wl.window) == 2048


def test_partial_page_budget_rejected():
    with pytest.raises(ValueError):
        budgets.selected_pages(2008)


@pytest.mark.parametrize("row", [r for r in GOLD["rows"] if r["method"] == "Quest"], ids=lambda r: r["cite"])
def test_windowed_selection_keeps_the_printed_total(row):
    # At a page-aligned 128K length the sink, the selected pages and the recent window add up
    # to the total the table prints (16-token pages).
    L, ps = 131072, 16
    n = L // ps
    scores = np.random.default_rng(0).standard_normal(n - 1)
    pages = quest.select_pages_windowed(scores, L, ps, budgets.selected_pages(row["selected"]), row["sink"],
                                        row["recent"])
    assert len(pages) * ps == row["total"]


@pytest.mark.parametrize("row", [r for r in GOLD["rows"] if r["method"] == "SnapKV"], ids=lambda r: r["cite"])
def test_snapkv_windows_keep_the_printed_total(row):
    # A 32K prompt, the 16-query observation window of that run: sink + selected + recent.
    n, W = 32768, 16
    pooled = np.random.default_rng(1).standard_normal(n - W)
    kept = snapkv.keep_positions_windowed(pooled, n, W, row["selected"], row["sink"], row["recent"])
    assert len(kept) == row["total"]


def test_snapkv_workloads_follow_the_tables():
    from synth import SNAPKV_AGENT_32K, SNAPKV_AIME_32K
    aime = [r for r in GOLD["rows"] if r["method"] == "SnapKV"][0]
    wl = SNAPKV_AIME_32K
    assert (wl.keep_sink, wl.keep_recent, wl.keep_topk, wl.window) == (aime["sink"], aime["recent"],
                                                                       aime["selected"], 16)
    wl = SNAPKV_AGENT_32K
    assert (wl.keep_sink, wl.keep_recent, wl.keep_topk) == (64, 512, 15808)
