"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Every mutant replaces one oracle function for the duration of one test; the
pins must then fail. This shows the pins are strong enough to notice a
dropped term, a swapped operand, a wrong index or tie rule.
"""
import numpy as np
import pytest

import oracle.quest as quest
import oracle.snapkv as snapkv
from tests import oracle_pins as pins


def _run_all(checks, mod):
    for c in checks:
        c(mod)


def _q_summary_swapped(rows):
    return rows.max(axis=0), rows.min(axis=0)


def _q_append_never_resets(m, M, k, offset):
    k = np.asarray(k, dtype=np.float64)
    return np.minimum(m, k), np.maximum(M, k)


def _q_bound_min(q, m, M):
    return np.minimum(q[None] * m, q[None] * M).sum(axis=1)


def _q_bound_drops_min_term(q, m, M):
    return (q[None] * M).sum(axis=1)


def _q_group_mean(qg, m, M):
    return sum(quest.head_page_bounds(qg[h], m, M) for h in range(qg.shape[0])) / qg.shape[0]


def _q_select_ties_high(scores, n, k):
    if n <= 0:
        return []
    ranked = sorted(range(n - 1), key=lambda p: (-scores[p], -p))
    return sorted(ranked[:k]) + [n - 1]


def _q_select_no_last(scores, n, k):
    if n <= 0:
        return []
    return sorted(sorted(range(n - 1), key=lambda p: (-scores[p], p))[:k])


def _q_select_last_in_budget(scores, n, k):
    if n <= 0:
        return []
    return sorted(sorted(range(n - 1), key=lambda p: (-scores[p], p))[:max(k - 1, 0)]) + [n - 1]


def _q_attention_no_scale(qg, K, V, scale):
    z = qg @ K.T
    e = np.exp(z - z.max(axis=1, keepdims=True))
    d = e.sum(axis=1, keepdims=True)
    return (e / d) @ V, z.max(axis=1) + np.log(d[:, 0])


def _s_mask_off_by_one(q, K, scale):
    W, n = q.shape[0], K.shape[0]
    z = scale * np.einsum("wgd,jd->wgj", q, K)
    hidden = np.arange(n)[None, :] >= (n - W + np.arange(W))[:, None]
    hidden[:, 0] = False
    z = np.where(hidden[:, None, :], -np.inf, z)
    e = np.exp(z - z.max(axis=2, keepdims=True))
    return e / e.sum(axis=2, keepdims=True)


def _s_scores_include_window(a):
    return a.sum(axis=(0, 1))[: a.shape[2] - a.shape[0]] + a[:, :, -1].sum()


def _s_pool_right_only(s, k):
    return np.array([s[j: j + k].max() for j in range(len(s))])


def _s_keep_ties_high(pooled, n, W, keep):
    c = n - W
    if c <= keep:
        chosen = list(range(c))
    else:
        chosen = sorted(sorted(range(c), key=lambda j: (-pooled[j], -j))[:keep])
    return chosen + list(range(c, n))


def _q_windows_recent_whole_pages(n_tokens, page_size, sink_tokens, recent_tokens):
    # recent window counted as whole pages from the end (misses the partial page at its start)
    n = -(-n_tokens // page_size)
    rp = recent_tokens // page_size
    sp = -(-min(sink_tokens, n_tokens) // page_size)
    kept = sorted(set(range(min(sp, n))) | set(range(max(n - max(rp, 1), 0), n)))
    return kept, [p for p in range(n) if p not in kept]


def _q_windowed_sink_in_budget(scores, n_tokens, page_size, topk, sink_tokens, recent_tokens):
    kept, cands = quest.keep_windows(n_tokens, page_size, sink_tokens, recent_tokens)
    k = max(topk - -(-sink_tokens // page_size), 0)
    return sorted(set(kept) | set(sorted(cands, key=lambda p: (-scores[p], p))[:k]))


def _s_windowed_recent_is_window(pooled, n, window, keep, sink, recent):
    # recent window taken as the observation window (the larger recent window ignored)
    return snapkv.keep_positions(pooled, n, window, keep) if sink == 0 else \
        sorted(set(range(min(sink, n))) | set(snapkv.keep_positions(pooled, n, window, keep)))


def _q_kth_off_by_one(scores, n_pages, topk):
    cands = [scores[p] for p in range(n_pages - 1)]
    if len(cands) <= topk:
        return None
    return sorted(cands, reverse=True)[min(topk, len(cands) - 1)]


def _q_kth_ascending(scores, n_pages, topk):
    cands = [scores[p] for p in range(n_pages - 1)]
    if len(cands) <= topk:
        return None
    return sorted(cands)[topk - 1]


def _q_kth_last_page_a_candidate(scores, n_pages, topk):
    cands = [scores[p] for p in range(min(n_pages, len(scores)))] + ([float("inf")] if n_pages > 0 else [])
    if len(cands) <= topk:
        return None
    return sorted(cands, reverse=True)[topk - 1]


def _q_kth_all_kept_when_equal(scores, n_pages, topk):
    cands = [scores[p] for p in range(n_pages - 1)]
    if len(cands) < topk:
        return None
    return sorted(cands, reverse=True)[topk - 1]


def _q_kth_windowed_counts_kept(scores, n_tokens, page_size, topk, sink_tokens, recent_tokens):
    # the kept windows ranked with the candidates
    n = -(-n_tokens // page_size)
    cands = list(range(max(n - 1, 0)))
    if len(cands) <= topk:
        return None
    return sorted((scores[p] for p in cands), reverse=True)[topk - 1]


def _q_kth_windowed_off_by_one(scores, n_tokens, page_size, topk, sink_tokens, recent_tokens):
    _, cands = quest.keep_windows(n_tokens, page_size, sink_tokens, recent_tokens)
    if len(cands) <= topk:
        return None
    return sorted((scores[p] for p in cands), reverse=True)[topk - 2 if topk > 1 else 0]


def _s_kth_off_by_one(pooled, keep):
    if len(pooled) <= keep:
        return None
    return sorted(pooled.tolist(), reverse=True)[keep]


def _s_kth_ascending(pooled, keep):
    if len(pooled) <= keep:
        return None
    return sorted(pooled.tolist())[keep - 1]


def _s_kth_windowed_counts_sink(pooled, n, window, keep, sink, recent):
    # the sink and recent positions ranked with the candidates
    cands = [pooled[j] for j in range(n - window)]
    if len(cands) <= keep:
        return None
    return sorted(cands, reverse=True)[keep - 1]


def _s_kth_windowed_off_by_one(pooled, n, window, keep, sink, recent):
    always = set(range(min(sink, n))) | set(range(max(0, n - recent), n))
    cands = [pooled[j] for j in range(n - window) if j not in always]
    if len(cands) <= keep:
        return None
    return sorted(cands, reverse=True)[min(keep, len(cands) - 1)]


MUTANTS = [
    (quest, "page_summary", _q_summary_swapped, pins.QUEST_CHECKS),
    (quest, "append_to_summary", _q_append_never_resets, pins.QUEST_CHECKS),
    (quest, "head_page_bounds", _q_bound_min, pins.QUEST_CHECKS),
    (quest, "head_page_bounds", _q_bound_drops_min_term, pins.QUEST_CHECKS),
    (quest, "group_page_scores", _q_group_mean, pins.QUEST_CHECKS),
    (quest, "select_pages", _q_select_ties_high, pins.QUEST_CHECKS),
    (quest, "select_pages", _q_select_no_last, pins.QUEST_CHECKS),
    (quest, "select_pages", _q_select_last_in_budget, pins.QUEST_CHECKS),
    (quest, "softmax_attention", _q_attention_no_scale, pins.QUEST_CHECKS),
    (quest, "keep_windows", _q_windows_recent_whole_pages, pins.QUEST_CHECKS),
    (quest, "select_pages_windowed", _q_windowed_sink_in_budget, pins.QUEST_CHECKS),
    (quest, "kth_score", _q_kth_off_by_one, pins.QUEST_CHECKS),
    (quest, "kth_score", _q_kth_ascending, pins.QUEST_CHECKS),
    (quest, "kth_score", _q_kth_last_page_a_candidate, pins.QUEST_CHECKS),
    (quest, "kth_score", _q_kth_all_kept_when_equal, pins.QUEST_CHECKS),
    (quest, "kth_score_windowed", _q_kth_windowed_counts_kept, pins.QUEST_CHECKS),
    (quest, "kth_score_windowed", _q_kth_windowed_off_by_one, pins.QUEST_CHECKS),
    (snapkv, "window_probabilities", _s_mask_off_by_one, pins.SNAPKV_CHECKS),
    (snapkv, "candidate_scores", _s_scores_include_window, pins.SNAPKV_CHECKS),
    (snapkv, "max_pool_clipped", _s_pool_right_only, pins.SNAPKV_CHECKS),
    (snapkv, "keep_positions", _s_keep_ties_high, pins.SNAPKV_CHECKS),
    (snapkv, "keep_positions_windowed", _s_windowed_recent_is_window, pins.SNAPKV_CHECKS),
    (snapkv, "kth_pooled", _s_kth_off_by_one, pins.SNAPKV_CHECKS),
    (snapkv, "kth_pooled", _s_kth_ascending, pins.SNAPKV_CHECKS),
    (snapkv, "kth_pooled_windowed", _s_kth_windowed_counts_sink, pins.SNAPKV_CHECKS),
    (snapkv, "kth_pooled_windowed", _s_kth_windowed_off_by_one, pins.SNAPKV_CHECKS),
]


@pytest.mark.parametrize("mod,name,bad,checks", MUTANTS, ids=lambda x: getattr(x, "__name__", ""))
def test_pins_catch_planted_mistake(monkeypatch, mod, name, bad, checks):
    monkeypatch.setattr(mod, name, bad)
    with pytest.raises(AssertionError):
        _run_all(checks, mod)
