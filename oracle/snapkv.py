"""fp64 oracle for SnapKV-style KV eviction at the end of prefill.

TEST INFRASTRUCTURE (see the package docstring): never imported by the
product path.

Sources
-------
[SparseEngine: Sparse-First Inference Engine] names SnapKV as a physical KV
eviction method (Table 14; Figure 2 caption shows it as a representative
implementation) and gives its settings: a 32-query scoring window, pooling
kernel 7, 2,016 selected tokens plus 32 recent ones (Table 8), and
probability-based prefill scores (Table 10). Physical eviction must release KV
storage rather than mask reads (Table 15 note), so the kept tokens are
gathered into compacted pages, which is the state Chain Cache later resumes
from (Figure 3 caption).

The pages do not print SnapKV's equations; the steps are the published SnapKV
method written from its definition, with these readings:

1. the window is the last W prompt positions n-W .. n-1; row w attends causally
   to keys j <= n-W+w (the history includes the current token, Table 7);
2. alpha_{w,h,j} = softmax_j(sm_scale * q_{w,h} . k_j) for each query head h of
   the KV head's GQA group;
3. the score of a candidate position j < n-W is the sum of the probabilities
   alpha_{w,h,j} over the window rows and the group's query heads;
4. the scores are max-pooled with an odd kernel, stride 1, the window clipped to
   the candidate range [0, n-W);
5. the ``keep`` best candidates by pooled score (ties to the lower position) are
   kept in ascending order, followed by the W window positions; with no more
   than ``keep`` candidates every position is kept;
6. the kept rows are copied unchanged into compacted pages, kept token t landing
   in logical page t // page_size, slot t % page_size.

Keep windows (Tables 9-12: SnapKV with sink 0/16/64 and recent 64/256/512
tokens beside 4,096 or 15,808 selected, a 16-query observation window in
Table 10; the budget excludes them, Table 10 caption). Reading: the first S
positions and the last R positions (R >= W) are always kept; the ``keep``
best pooled candidates among the positions between them are added; the scores
and their pooling are those of steps 3-4 (every position before the window).
S = 0, R = W is step 5.
"""
from __future__ import annotations

import numpy as np

from .quest import f64


def window_probabilities(q_win: np.ndarray, K: np.ndarray, sm_scale: float) -> np.ndarray:
    """alpha [W][G][n]: causal softmax of the window queries q_win [W][G][D] over keys K [n][D]."""
    W = q_win.shape[0]
    n = K.shape[0]
    z = sm_scale * np.einsum("wgd,jd->wgj", q_win, K)
    last_visible = n - W + np.arange(W)                     # position of window row w
    hidden = np.arange(n)[None, :] > last_visible[:, None]  # [W][n]
    z = np.where(hidden[:, None, :], -np.inf, z)
    zmax = z.max(axis=2, keepdims=True)
    e = np.exp(z - zmax)
    return e / e.sum(axis=2, keepdims=True)


def window_lse(q_win: np.ndarray, K: np.ndarray, sm_scale: float) -> np.ndarray:
    """LSE [W][G]: log sum_j exp(sm_scale * q_{w,g} . k_j) over the keys row w sees (j <= n-W+w)."""
    W = q_win.shape[0]
    n = K.shape[0]
    z = sm_scale * np.einsum("wgd,jd->wgj", q_win, K)
    hidden = np.arange(n)[None, :] > (n - W + np.arange(W))[:, None]
    z = np.where(hidden[:, None, :], -np.inf, z)
    zmax = z.max(axis=2, keepdims=True)
    return zmax[:, :, 0] + np.log(np.exp(z - zmax).sum(axis=2))


def candidate_scores(alpha: np.ndarray) -> np.ndarray:
    """s_j = sum_w sum_h alpha_{w,h,j} over the candidates j < n-W."""
    W, _, n = alpha.shape
    return alpha[:, :, :n - W].sum(axis=(0, 1))


def max_pool_clipped(s: np.ndarray, kernel: int) -> np.ndarray:
    """Stride-1 max over the window [j - kernel//2, j + kernel//2] clipped to the array."""
    half = kernel // 2
    return np.array([s[max(0, j - half): j + half + 1].max() for j in range(len(s))])


def keep_positions(pooled: np.ndarray, n: int, window: int, keep: int) -> list:
    """Ascending top-``keep`` candidates by pooled score (ties: lower j), then the window."""
    cands = n - window
    if cands <= keep:
        chosen = list(range(cands))
    else:
        chosen = sorted(sorted(range(cands), key=lambda j: (-pooled[j], j))[:keep])
    return chosen + list(range(cands, n))


def keep_positions_windowed(pooled: np.ndarray, n: int, window: int, keep: int, sink: int, recent: int) -> list:
    """Ascending: the first ``sink`` and last ``recent`` positions, plus the ``keep`` best pooled
    candidates between them (ties: lower j); every position when no more than ``keep`` remain."""
    always = set(range(min(sink, n))) | set(range(max(0, n - recent), n))
    cands = [j for j in range(n - window) if j not in always]
    if len(cands) <= keep:
        return list(range(n))
    chosen = sorted(cands, key=lambda j: (-pooled[j], j))[:keep]
    return sorted(always | set(chosen))


def kth_pooled_windowed(pooled: np.ndarray, n: int, window: int, keep: int, sink: int, recent: int):
    """The keep-th largest pooled candidate score, or None when every position is kept."""
    always = set(range(min(sink, n))) | set(range(max(0, n - recent), n))
    cands = [pooled[j] for j in range(n - window) if j not in always]
    if len(cands) <= keep:
        return None
    return sorted(cands, reverse=True)[keep - 1]


def kth_pooled(pooled: np.ndarray, keep: int):
    """The keep-th largest pooled score (selection threshold), or None when all are kept."""
    if len(pooled) <= keep:
        return None
    return sorted(pooled.tolist(), reverse=True)[keep - 1]


def request_keys(cache, block_table_row, h: int, n: int, page_size: int) -> np.ndarray:
    """Logical key (or value) rows 0..n-1 of one KV head, gathered through the block table."""
    rows = []
    for p in range((n + page_size - 1) // page_size):
        valid = min(page_size, n - p * page_size)
        rows.append(f64(cache[int(block_table_row[p]), h, :valid, :]))
    return np.vstack(rows)


def snapkv_head(q_win_group, k_cache, block_table_row, h: int, n: int, window: int,
                pool_kernel: int, keep: int, sm_scale: float, page_size: int = 16, sink: int = 0,
                recent: int = None) -> dict:
    """Scores, pooled scores, threshold and kept positions of one (request, KV head)
    (keep windows ``sink`` / ``recent``; recent None is the observation window)."""
    K = request_keys(k_cache, block_table_row, h, n, page_size)
    alpha = window_probabilities(f64(q_win_group), K, sm_scale)
    s = candidate_scores(alpha)
    pooled = max_pool_clipped(s, pool_kernel)
    if sink == 0 and recent in (None, window):
        kept, tau = keep_positions(pooled, n, window, keep), kth_pooled(pooled, keep)
    else:
        kept = keep_positions_windowed(pooled, n, window, keep, sink, recent)
        tau = kth_pooled_windowed(pooled, n, window, keep, sink, recent)
    return {"scores": s, "pooled": pooled, "threshold": tau, "kept": kept, "alpha_total": alpha.sum(),
            "lse": window_lse(f64(q_win_group), K, sm_scale)}


def compact_rows(cache, block_table_row, h: int, kept: list, page_size: int = 16):
    """The kept rows, in kept order, copied unchanged (same dtype, no arithmetic)."""
    return [cache[int(block_table_row[j // page_size]), h, j % page_size, :] for j in kept]


def snapkv_step(inputs, requests=None, heads=None) -> dict:
    """Oracle eviction over a batch. ``inputs``: CPU k_cache, block_table, prompt_lens,
    q_window [B][W][Hq][D], window, pool_kernel, keep_topk, sm_scale, num_kv_heads.
    Returns {(b, h): snapkv_head(...)}."""
    out = {}
    B = len(inputs["prompt_lens"])
    Hkv = inputs["num_kv_heads"]
    G = inputs["q_window"].shape[2] // Hkv
    for b in (range(B) if requests is None else requests):
        for h in (range(Hkv) if heads is None else heads):
            qg = inputs["q_window"][b, :, h * G:(h + 1) * G, :]
            out[(b, h)] = snapkv_head(qg, inputs["k_cache"], inputs["block_table"][b], h,
                                      int(inputs["prompt_lens"][b]), inputs["window"],
                                      inputs["pool_kernel"], inputs["keep_topk"], inputs["sm_scale"],
                                      inputs.get("page_size", 16), inputs.get("sink", 0), inputs.get("recent"))
    return out
