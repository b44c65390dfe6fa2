"""Pins of the fp64 oracle against facts other than the oracle itself.

Each ``check_*`` takes the oracle modules as arguments and raises
AssertionError when the oracle disagrees with brute force, a closed form, a
library routine or an invariant. ``test_oracle_*.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` plants plausible mistakes in copies of
oracle functions and asserts that some check catches each one.
"""
import math

import numpy as np
import torch

PS = 4  # small page size keeps brute force cheap; the oracle takes it as a parameter


def _rng(seed):
    return np.random.default_rng(seed)


def _paged(rng, n_tokens, H, D, page_size=PS, permute=True, poison=True, dv=None):
    """A paged cache [P][H][ps][D] (+ value cache) holding logical rows, and its table."""
    n = (n_tokens + page_size - 1) // page_size
    dv = D if dv is None else dv
    Kl = rng.standard_normal((H, n * page_size, D))
    Vl = rng.standard_normal((H, n * page_size, dv))
    phys = rng.permutation(n + 3)[:n] if permute else np.arange(n)
    P = n + 3
    kc = rng.standard_normal((P, H, page_size, D))
    vc = rng.standard_normal((P, H, page_size, dv))
    for p in range(n):
        kc[phys[p]] = Kl[:, p * page_size:(p + 1) * page_size]
        vc[phys[p]] = Vl[:, p * page_size:(p + 1) * page_size]
    if poison:
        for pos in range(n_tokens, n * page_size):
            kc[phys[pos // page_size], :, pos % page_size] = np.nan
            vc[phys[pos // page_size], :, pos % page_size] = np.nan
    return kc, vc, phys, Kl[:, :n_tokens], Vl[:, :n_tokens]


# ------------------------------------------------------------------ summaries
def check_summary_bruteforce(quest):
    rng = _rng(1)
    for L in (1, 3, 4, 9, 13):
        kc, vc, bt, Kl, _ = _paged(rng, L, 2, 5)
        req = quest.QuestRequest(kc, vc, bt, L, 2, 5, 5, PS)
        for h in range(2):
            m, M = req.summaries[h]
            assert m.shape[0] == (L + PS - 1) // PS
            for p in range(m.shape[0]):
                toks = range(p * PS, min(L, (p + 1) * PS))
                for c in range(5):
                    vals = [float(Kl[h, j, c]) for j in toks]
                    assert m[p, c] == min(vals) and M[p, c] == max(vals), (L, h, p, c)


def check_append_matches_rebuild(quest):
    rng = _rng(2)
    H, D = 2, 6
    for L0 in (1, 4, 7, 8):
        n_add = 6
        kc, vc, bt, Kl, Vl = _paged(rng, L0 + n_add, H, D, poison=False)
        req = quest.QuestRequest(kc, vc, bt, L0, H, D, D, PS)
        for t in range(n_add):
            pos = L0 + t
            req.append(Kl[:, pos], Vl[:, pos])
        fresh = quest.QuestRequest(kc, vc, bt, L0 + n_add, H, D, D, PS)
        for h in range(H):
            np.testing.assert_array_equal(req.summaries[h][0], fresh.summaries[h][0])
            np.testing.assert_array_equal(req.summaries[h][1], fresh.summaries[h][1])


# ------------------------------------------------------------------ bounds
def check_bound_dominates_logits(quest):
    rng = _rng(3)
    for trial in range(20):
        D = int(rng.integers(1, 9))
        rows = rng.standard_normal((int(rng.integers(1, 6)), D)) * rng.choice([1.0, 8.0], size=D)
        m, M = quest.page_summary(rows)
        q = rng.standard_normal(D)
        U = quest.head_page_bounds(q, m[None], M[None])[0]
        assert U >= max(float(q @ r) for r in rows) - 1e-12 * (1 + abs(U)), trial


def check_bound_single_token_exact(quest):
    rng = _rng(4)
    for _ in range(10):
        k = rng.standard_normal(7)
        q = rng.standard_normal(7)
        m, M = quest.page_summary(k[None])
        U = quest.head_page_bounds(q, m[None], M[None])[0]
        assert math.isclose(U, float(q @ k), rel_tol=1e-12, abs_tol=1e-12)


def check_bound_sign_cases(quest):
    rng = _rng(5)
    rows = rng.standard_normal((4, 6))
    m, M = quest.page_summary(rows)
    qp = np.abs(rng.standard_normal(6))
    assert math.isclose(quest.head_page_bounds(qp, m[None], M[None])[0], float(qp @ M), rel_tol=1e-12)
    qn = -np.abs(rng.standard_normal(6))
    assert math.isclose(quest.head_page_bounds(qn, m[None], M[None])[0], float(qn @ m), rel_tol=1e-12)


def check_group_score_bounds_group_logit(quest):
    rng = _rng(6)
    for _ in range(20):
        G, D, t = int(rng.integers(1, 5)), 5, int(rng.integers(1, 5))
        rows = rng.standard_normal((t, D))
        qg = rng.standard_normal((G, D))
        m, M = quest.page_summary(rows)
        U = quest.group_page_scores(qg, m[None], M[None])[0]
        assert U >= max(float(qg.sum(0) @ r) for r in rows) - 1e-12 * (1 + abs(U))
        # a group of one query head is the per-head bound
        U1 = quest.group_page_scores(qg[:1], m[None], M[None])[0]
        assert math.isclose(U1, quest.head_page_bounds(qg[0], m[None], M[None])[0], rel_tol=1e-12)


# ------------------------------------------------------------------ selection
def _rank_select(scores, n, k):
    """Brute force by rank counting: p is kept iff fewer than k candidates beat it."""
    keep = []
    for p in range(n - 1):
        better = sum(1 for r in range(n - 1)
                     if scores[r] > scores[p] or (scores[r] == scores[p] and r < p))
        if better < k:
            keep.append(p)
    return keep + [n - 1]


def check_select_bruteforce(quest):
    rng = _rng(7)
    for _ in range(50):
        n = int(rng.integers(1, 20))
        k = int(rng.integers(1, 8))
        scores = rng.integers(-3, 4, size=max(n - 1, 0)).astype(float)  # many ties
        assert quest.select_pages(scores, n, k) == _rank_select(scores, n, k), (n, k, scores)
    assert quest.select_pages(np.array([]), 1, 4) == [0]
    assert quest.select_pages(np.arange(5.0), 6, 10) == list(range(6))


# ------------------------------------------------------------------ keep windows
def _window_rank_select(scores, n_tokens, ps, k, S, R):
    """Brute force from the token-level definition: page p is kept when it holds one of the
    first S tokens, one of the last R tokens, or is the last page; among the other pages, p
    is selected when fewer than k of them beat it (higher score, or equal and lower index)."""
    n = -(-n_tokens // ps)

    def kept(p):
        first, last = p * ps, min((p + 1) * ps, n_tokens) - 1
        return p == n - 1 or first < S or last >= n_tokens - R

    cands = [p for p in range(n) if not kept(p)]
    sel = [p for p in cands
           if sum(1 for r in cands if scores[r] > scores[p] or (scores[r] == scores[p] and r < p)) < k]
    return sorted([p for p in range(n) if kept(p)] + sel)


def check_select_windowed_bruteforce(quest):
    rng = _rng(17)
    for _ in range(200):
        L = int(rng.integers(0, 90))
        S, R, k = int(rng.integers(0, 20)), int(rng.integers(0, 30)), int(rng.integers(1, 6))
        n = -(-L // PS)
        scores = rng.integers(-2, 3, size=max(n - 1, 0)).astype(float)  # many ties
        assert quest.select_pages_windowed(scores, L, PS, k, S, R) == _window_rank_select(scores, L, PS, k, S, R), \
            (L, S, R, k, scores)
    # Windows that cover every page keep every page.
    assert quest.select_pages_windowed(np.zeros(9), 40, PS, 1, 20, 20) == list(range(10))


def check_select_windowed_reduces_to_plain(quest):
    rng = _rng(19)
    for _ in range(50):
        L = int(rng.integers(1, 90))
        n = -(-L // PS)
        k = int(rng.integers(1, 8))
        scores = rng.standard_normal(max(n - 1, 0))
        assert quest.select_pages_windowed(scores, L, PS, k, 0, 0) == quest.select_pages(scores, n, k)
        assert quest.kth_score_windowed(scores, L, PS, k, 0, 0) == quest.kth_score(scores, n, k)


# ------------------------------------------------------------------ selection thresholds
# tau, the k-th largest candidate score, centres the exemption band of the parity
# rule. Pinned by rank counting from its definition: tau is the score of the one
# candidate that exactly k - 1 candidates rank before (higher score, or equal score
# and lower index); with no more candidates than k every candidate is kept and there
# is no threshold.
def _rank_k_score(scores, cands, k):
    cands = list(cands)
    if len(cands) <= k:
        return None
    hits = [scores[p] for p in cands
            if sum(1 for r in cands if scores[r] > scores[p] or (scores[r] == scores[p] and r < p)) == k - 1]
    assert len(hits) == 1
    return hits[0]


def _window_candidates(n_tokens, ps, S, R):
    """Pages in neither keep window (token-level definition), the last page excluded."""
    n = -(-n_tokens // ps)
    return [p for p in range(n) if not (p == n - 1 or p * ps < S or min((p + 1) * ps, n_tokens) - 1 >= n_tokens - R)]


def check_kth_score_rank_counting(quest):
    rng = _rng(27)
    for _ in range(150):
        n = int(rng.integers(0, 24))
        k = int(rng.integers(1, 9))
        scores = rng.integers(-3, 4, size=max(n - 1, 0)).astype(float)  # many ties
        assert quest.kth_score(scores, n, k) == _rank_k_score(scores, range(n - 1), k), (n, k, scores)
    # distinct scores: tau is the k-th value counted from the top
    assert quest.kth_score(np.array([5.0, 1.0, 4.0, 2.0, 3.0]), 6, 2) == 4.0
    assert quest.kth_score(np.array([5.0, 1.0, 4.0]), 4, 3) is None       # 3 candidates, k = 3: all kept
    assert quest.kth_score(np.array([5.0, 1.0, 4.0, 2.0]), 5, 4) is None


def check_kth_score_windowed_rank_counting(quest):
    rng = _rng(29)
    for _ in range(200):
        L = int(rng.integers(0, 90))
        S, R, k = int(rng.integers(0, 20)), int(rng.integers(0, 30)), int(rng.integers(1, 6))
        n = -(-L // PS)
        scores = rng.integers(-2, 3, size=max(n - 1, 0)).astype(float)
        ref = _rank_k_score(scores, _window_candidates(L, PS, S, R), k)
        assert quest.kth_score_windowed(scores, L, PS, k, S, R) == ref, (L, S, R, k, scores)


def check_decode_threshold_is_lowest_selected_score(quest):
    """The threshold a decode reports is the lowest score among its selected candidates
    (the top k by score hold the k-th largest as their minimum)."""
    rng = _rng(31)
    H, G, D = 2, 2, 4
    for L, k, S, R in ((37, 3, 0, 0), (41, 2, 0, 0), (61, 4, 5, 9), (64, 3, 4, 8), (9, 4, 0, 0)):
        kc, vc, bt, _, _ = _paged(rng, L, H, D)
        q = rng.standard_normal((H * G, D))
        res = quest.QuestRequest(kc, vc, bt, L, H, D, D, PS).decode(q, k, 0.5, sink_tokens=S, recent_tokens=R)
        cands = _window_candidates(L, PS, S, R)
        for hr in res.heads:
            chosen = [p for p in hr.pages if p in cands]
            if len(cands) <= k:
                assert hr.threshold is None
            else:
                assert len(chosen) == k and hr.threshold == min(hr.scores[p] for p in chosen), (L, k, S, R)


# ------------------------------------------------------------------ attention
def _sdpa(qg, K, V, scale):
    q = torch.from_numpy(qg)[None, :, None, :]          # [1][G][1][D]
    k = torch.from_numpy(K)[None, None].expand(1, qg.shape[0], -1, -1)
    v = torch.from_numpy(V)[None, None].expand(1, qg.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    lse = torch.logsumexp(scale * (q @ k.transpose(-1, -2)), dim=-1)
    return o[0, :, 0].numpy(), lse[0, :, 0].numpy()


def check_select_all_equals_dense(quest):
    rng = _rng(8)
    for L in (1, 5, 8, 13):
        H, G, D = 2, 3, 8
        kc, vc, bt, Kl, Vl = _paged(rng, L, H, D)
        q = rng.standard_normal((H * G, D))
        scale = 1 / math.sqrt(D)
        req = quest.QuestRequest(kc, vc, bt, L, H, D, D, PS)
        n = (L + PS - 1) // PS
        res = req.decode(q, topk_pages=n, sm_scale=scale)
        for h in range(H):
            assert res.heads[h].pages == list(range(n))
            o, lse = _sdpa(q[h * G:(h + 1) * G], Kl[h], Vl[h], scale)
            np.testing.assert_allclose(res.out[h * G:(h + 1) * G], o, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(res.lse[h * G:(h + 1) * G], lse, rtol=1e-10, atol=1e-12)


def check_single_token_attention(quest):
    rng = _rng(9)
    kc, vc, bt, Kl, Vl = _paged(rng, 1, 1, 4)
    q = rng.standard_normal((2, 4))
    res = quest.QuestRequest(kc, vc, bt, 1, 1, 4, 4, PS).decode(q, 3, 0.7)
    np.testing.assert_allclose(res.out, np.vstack([Vl[0, 0], Vl[0, 0]]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(res.lse, 0.7 * (q @ Kl[0, 0]), rtol=1e-14)


def check_empty_request(quest):
    """A request with no token selects nothing and attends to nothing (empty sum)."""
    kc = np.zeros((2, 1, PS, 4))
    res = quest.QuestRequest(kc, kc.copy(), np.array([0]), 0, 1, 4, 4, PS).decode(np.ones((2, 4)), 3, 1.0)
    assert res.heads[0].pages == [] and res.heads[0].threshold is None
    np.testing.assert_array_equal(res.out, np.zeros((2, 4)))
    assert np.all(np.isneginf(res.lse))


def check_permutation_invariance(quest):
    rng = _rng(10)
    L, H, D = 11, 2, 4
    kc, vc, bt, Kl, Vl = _paged(rng, L, H, D, permute=False)
    q = rng.standard_normal((2 * H, D))
    base = quest.QuestRequest(kc, vc, bt, L, H, D, D, PS).decode(q, 1, 0.5)
    perm = rng.permutation(kc.shape[0])
    inv = np.argsort(perm)
    kc2, vc2 = kc[perm], vc[perm]           # physical page p moves to slot inv[p]
    bt2 = inv[bt]
    other = quest.QuestRequest(kc2, vc2, bt2, L, H, D, D, PS).decode(q, 1, 0.5)
    np.testing.assert_array_equal(base.out, other.out)
    assert [h.pages for h in base.heads] == [h.pages for h in other.heads]


def check_latent_value_is_key_prefix(quest):
    rng = _rng(11)
    L, D, Dv = 9, 10, 6
    kc, _, bt, Kl, _ = _paged(rng, L, 1, D)
    q = rng.standard_normal((3, D))
    lat = quest.QuestRequest(kc, None, bt, L, 1, D, Dv, PS).decode(q, 2, 0.3)
    sep = quest.QuestRequest(kc, np.ascontiguousarray(kc[..., :Dv]), bt, L, 1, D, Dv, PS).decode(q, 2, 0.3)
    np.testing.assert_array_equal(lat.out, sep.out)


def check_selection_uses_the_bound(quest):
    """A page whose keys align with the query wins; the last page is always present."""
    D, L = 4, 5 * PS
    kc = np.zeros((5, 1, PS, D))
    kc[2, 0, 1] = [5.0, 0, 0, 0]      # page 2 holds the only key aligned with q
    kc[0, 0, 0] = [-5.0, 0, 0, 0]
    bt = np.arange(5)
    q = np.array([[1.0, 0, 0, 0]])
    res = quest.QuestRequest(kc, kc.copy(), bt, L, 1, D, D, PS).decode(q, 1, 1.0)
    assert res.heads[0].pages == [2, 4]
    # Closed form: page 2 bound = 1*5 = 5, page 0 bound = max(1*-5, 1*0) = 0, others 0.
    np.testing.assert_array_equal(res.heads[0].scores, [0.0, 0.0, 5.0, 0.0])


# ------------------------------------------------------------------ SnapKV
def _torch_window_probs(q_win, K, scale):
    W = q_win.shape[0]
    n = K.shape[0]
    z = scale * torch.einsum("wgd,jd->wgj", torch.from_numpy(q_win), torch.from_numpy(K))
    mask = torch.ones(n, n, dtype=torch.bool).tril()[n - W:]      # causal rows of the window
    z = z.masked_fill(~mask[:, None, :], float("-inf"))
    return torch.softmax(z, dim=-1).numpy()


def check_window_probabilities(snapkv):
    rng = _rng(12)
    for n, W in ((5, 1), (9, 4), (16, 16), (23, 8)):
        q = rng.standard_normal((W, 3, 6))
        K = rng.standard_normal((n, 6))
        a = snapkv.window_probabilities(q, K, 0.4)
        np.testing.assert_allclose(a, _torch_window_probs(q, K, 0.4), rtol=1e-12, atol=1e-15)
        # every row is a distribution over its causal history
        np.testing.assert_allclose(a.sum(axis=2), np.ones((W, 3)), rtol=1e-13)


def check_window_lse(snapkv):
    rng = _rng(18)
    for n, W in ((6, 2), (20, 8), (9, 9)):
        q = rng.standard_normal((W, 2, 5))
        K = rng.standard_normal((n, 5))
        z = 0.3 * torch.einsum("wgd,jd->wgj", torch.from_numpy(q), torch.from_numpy(K))
        mask = torch.ones(n, n, dtype=torch.bool).tril()[n - W:]
        ref = torch.logsumexp(z.masked_fill(~mask[:, None, :], float("-inf")), dim=-1).numpy()
        np.testing.assert_allclose(snapkv.window_lse(q, K, 0.3), ref, rtol=1e-12)


def check_candidate_scores(snapkv):
    rng = _rng(13)
    n, W, G = 11, 3, 2
    a = rng.random((W, G, n))
    s = snapkv.candidate_scores(a)
    assert s.shape == (n - W,)
    for j in range(n - W):
        assert math.isclose(s[j], sum(a[w, g, j] for w in range(W) for g in range(G)), rel_tol=1e-14)


def check_max_pool(snapkv):
    rng = _rng(14)
    for n, k in ((1, 7), (5, 7), (30, 7), (30, 3), (12, 1)):
        s = rng.standard_normal(n)
        ref = torch.nn.functional.max_pool1d(torch.from_numpy(s)[None, None], k, stride=1,
                                             padding=k // 2)[0, 0].numpy()
        np.testing.assert_array_equal(snapkv.max_pool_clipped(s, k), ref)
    s = rng.standard_normal(9)
    np.testing.assert_array_equal(snapkv.max_pool_clipped(s, 1), s)


def check_keep_positions(snapkv):
    rng = _rng(15)
    for _ in range(40):
        n = int(rng.integers(2, 25))
        W = int(rng.integers(1, n + 1))
        keep = int(rng.integers(1, 10))
        pooled = rng.integers(0, 4, size=n - W).astype(float)
        got = snapkv.keep_positions(pooled, n, W, keep)
        ref = _rank_select(pooled, n - W + 1, keep)[:-1] if n - W > 0 else []
        assert got == ref + list(range(n - W, n)), (n, W, keep)
        assert len(got) == min(n, keep + W)


def check_keep_positions_windowed(snapkv):
    """Rank counting from the definition: j is kept when j < S, j >= n - R, or (j < n - W and
    fewer than keep other candidates beat it); every position when keep covers the candidates."""
    rng = _rng(23)
    for _ in range(200):
        n = int(rng.integers(2, 40))
        W = int(rng.integers(1, n + 1))
        R = int(rng.integers(W, n + 3))
        S = int(rng.integers(0, 12))
        keep = int(rng.integers(1, 8))
        pooled = rng.integers(0, 4, size=n - W).astype(float)
        cands = [j for j in range(n - W) if j >= S and j < n - R]
        if len(cands) <= keep:
            ref = list(range(n))
        else:
            ref = [j for j in range(n) if j < S or j >= n - R or (j in cands and sum(
                1 for r in cands if pooled[r] > pooled[j] or (pooled[r] == pooled[j] and r < j)) < keep)]
        assert snapkv.keep_positions_windowed(pooled, n, W, keep, S, R) == ref, (n, W, R, S, keep)
        if S == 0 and R == W:
            assert ref == snapkv.keep_positions(pooled, n, W, keep)


def check_kth_pooled_rank_counting(snapkv):
    rng = _rng(33)
    for _ in range(150):
        c = int(rng.integers(0, 24))
        keep = int(rng.integers(1, 9))
        pooled = rng.integers(0, 4, size=c).astype(float)
        assert snapkv.kth_pooled(pooled, keep) == _rank_k_score(pooled, range(c), keep), (c, keep, pooled)
    assert snapkv.kth_pooled(np.array([0.1, 0.7, 0.3, 0.5]), 3) == 0.3
    assert snapkv.kth_pooled(np.array([0.1, 0.7, 0.3]), 3) is None


def check_kth_pooled_windowed_rank_counting(snapkv):
    rng = _rng(35)
    for _ in range(200):
        n = int(rng.integers(2, 40))
        W = int(rng.integers(1, n + 1))
        R = int(rng.integers(W, n + 3))
        S = int(rng.integers(0, 12))
        keep = int(rng.integers(1, 8))
        pooled = rng.integers(0, 4, size=n - W).astype(float)
        cands = [j for j in range(n - W) if S <= j < n - R]
        assert snapkv.kth_pooled_windowed(pooled, n, W, keep, S, R) == _rank_k_score(pooled, cands, keep), \
            (n, W, R, S, keep)


def check_snapkv_threshold_is_lowest_kept_score(snapkv):
    """The threshold of a head is the lowest pooled score among its chosen candidates."""
    rng = _rng(37)
    D, G = 6, 2
    for n, W, keep, S, R in ((40, 4, 5, 0, None), (45, 3, 6, 4, 9), (12, 4, 9, 0, None), (30, 2, 3, 3, 2)):
        kc, _, bt, _, _ = _paged(rng, n, 1, D)
        q = rng.standard_normal((W, G, D))
        res = snapkv.snapkv_head(q, kc, bt, 0, n, W, 3, keep, 0.4, PS, sink=S, recent=R)
        RR = W if R is None else R
        cands = [j for j in range(n - W) if S <= j < n - RR]
        chosen = [j for j in res["kept"] if j in cands]
        if len(cands) <= keep:
            assert res["threshold"] is None
        else:
            assert len(chosen) == keep and res["threshold"] == min(res["pooled"][j] for j in chosen), (n, W, keep)


def check_snapkv_head_end_to_end(snapkv):
    """Whole head against torch routines: softmax, max_pool1d and a stable sort."""
    rng = _rng(16)
    n, W, G, D, keep = 37, 5, 2, 8, 6
    kc, _, bt, Kl, _ = _paged(rng, n, 1, D)
    q = rng.standard_normal((W, G, D))
    res = snapkv.snapkv_head(q, kc, bt, 0, n, W, 3, keep, 0.35, PS)
    a = torch.from_numpy(_torch_window_probs(q, Kl[0], 0.35))
    s = a[:, :, :n - W].sum(dim=(0, 1))
    pooled = torch.nn.functional.max_pool1d(s[None, None], 3, 1, 1)[0, 0]
    order = torch.sort(-pooled, stable=True).indices[:keep].sort().values.tolist()
    assert res["kept"] == order + list(range(n - W, n))
    np.testing.assert_allclose(res["scores"], s.numpy(), rtol=1e-12)
    # invariant: the probabilities of all W*G window rows add up to W*G
    assert math.isclose(res["alpha_total"], W * G, rel_tol=1e-12)


def check_compaction_exact(snapkv):
    rng = _rng(17)
    kc, _, bt, Kl, _ = _paged(rng, 14, 2, 3, poison=False)
    kept = [0, 5, 6, 13]
    rows = snapkv.compact_rows(kc, bt, 1, kept, PS)
    for r, j in zip(rows, kept):
        np.testing.assert_array_equal(r, Kl[1, j])


QUEST_CHECKS = [check_summary_bruteforce, check_append_matches_rebuild, check_bound_dominates_logits,
                check_bound_single_token_exact, check_bound_sign_cases,
                check_group_score_bounds_group_logit, check_select_bruteforce,
                check_select_all_equals_dense, check_single_token_attention, check_empty_request,
                check_permutation_invariance, check_latent_value_is_key_prefix,
                check_selection_uses_the_bound, check_select_windowed_bruteforce,
                check_select_windowed_reduces_to_plain, check_kth_score_rank_counting,
                check_kth_score_windowed_rank_counting, check_decode_threshold_is_lowest_selected_score]
SNAPKV_CHECKS = [check_window_probabilities, check_window_lse, check_candidate_scores, check_max_pool,
                 check_keep_positions, check_keep_positions_windowed, check_kth_pooled_rank_counting,
                 check_kth_pooled_windowed_rank_counting, check_snapkv_threshold_is_lowest_kept_score,
                 check_snapkv_head_end_to_end, check_compaction_exact]
