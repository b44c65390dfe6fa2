"""fp64 oracle for Quest-style query-aware sparse decode over a paged KV cache.

TEST INFRASTRUCTURE (see the package docstring): never imported by the
product path.

Sources
-------
The SparseEngine pages [SparseEngine: Sparse-First Inference Engine] name
Quest as the engine's query-dependent retrieval method (Figure 2 caption:
representative implementations of SnapKV and Quest; Tables 14 and 15) and say
that prefix caching keeps, next to each KV block, the summaries Quest needs
(Figure 3 caption). They give its settings: 16-token pages (Tables 8, 9, 11),
budgets of 2,048 / 4,096 / 1,472 selected tokens (Tables 8-12), and that
selected budgets exclude separately listed sink and recent tokens (Table 10
caption). The notation table (Table 7) fixes that the causal history [i] of
the current position includes the current token, and names the query-key
logit z and the normalised weight alpha.

The pages do not print Quest's equations. The steps here are the published
Quest method, written from its definition:

1. page summary: per channel c, the minimum m_{p,c} and maximum M_{p,c} of the
   keys of page p, over the page's valid tokens only;
2. per-head bound: U_h(p) = sum_c max(q_{h,c} m_{p,c}, q_{h,c} M_{p,c}), an upper
   bound of q_h . k_j for every token j of page p;
3. group score (reading: one page selection per KV head serves all query heads
   of its GQA group, scored by the sum of their bounds, which bounds the
   group-summed logit from above): U(p) = sum_{h in group} U_h(p);
4. selection: the ``topk`` best-scoring pages among 0..n-2 (reading: ties go
   to the lower page index), plus the last page n-1, which holds the newest
   tokens and is always kept outside the budget; ascending page ids;
4b. keep windows (Tables 9-12: Quest with sink and recent tokens beside the
   selected budget, e.g. sink 64, recent 512, 1,472 selected = 2,048 total;
   reading: page-granular): the pages holding any of the first S tokens and
   the pages holding any of the last R tokens are always kept, as is the last
   page; the ``topk`` best pages are chosen among the pages that are in neither
   window (ties to the lower page index). S = R = 0 is step 4;
5. attention over the selected pages: z_j = sm_scale * q_h . k_j for the
   tokens j < L of those pages, alpha = softmax(z), o_h = sum_j alpha_j v_j and
   lse_h = log sum_j exp(z_j).

A latent (MLA-style) cache stores one row per token whose first
``head_dim_v`` dims are the value (reading: the value shares the row with the
key, which is the full row).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f64(x) -> np.ndarray:
    """Exact upcast of a block (numpy array or CPU torch tensor of any float dtype) to fp64."""
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def num_pages(n_tokens: int, page_size: int) -> int:
    return (n_tokens + page_size - 1) // page_size


# ---------------------------------------------------------------- step 1
def page_summary(rows: np.ndarray):
    """Per-channel (min, max) of the valid key rows [t][D] of one page (t >= 1)."""
    return rows.min(axis=0), rows.max(axis=0)


def append_to_summary(m_page, M_page, k_new, offset: int):
    """Summary of a page after a new key lands in slot ``offset``.

    A token that opens a page (slot 0) is the page's only valid row, so the summary
    is that row; otherwise the new row joins the old minimum and maximum.
    """
    k_new = np.asarray(k_new, dtype=np.float64)
    if offset == 0:
        return k_new.copy(), k_new.copy()
    return np.minimum(m_page, k_new), np.maximum(M_page, k_new)


# ---------------------------------------------------------------- steps 2, 3
def head_page_bounds(q_h: np.ndarray, m: np.ndarray, M: np.ndarray) -> np.ndarray:
    """U_h(p) = sum_c max(q_c * m_{p,c}, q_c * M_{p,c}) for every page p (rows of m, M)."""
    return np.maximum(q_h[None, :] * m, q_h[None, :] * M).sum(axis=1)


def group_page_scores(q_group: np.ndarray, m: np.ndarray, M: np.ndarray) -> np.ndarray:
    """U(p) = sum over the group's query heads of U_h(p)."""
    total = np.zeros(m.shape[0])
    for h in range(q_group.shape[0]):
        total += head_page_bounds(q_group[h], m, M)
    return total


# ---------------------------------------------------------------- step 4
def select_pages(scores, n_pages: int, topk: int) -> list:
    """Ascending logical page ids: the ``topk`` best candidates 0..n-2, plus page n-1."""
    if n_pages <= 0:
        return []
    ranked = sorted(range(n_pages - 1), key=lambda p: (-scores[p], p))
    return sorted(ranked[:topk]) + [n_pages - 1]


def kth_score(scores, n_pages: int, topk: int):
    """The k-th largest candidate score (the selection threshold), or None if all are kept."""
    cands = [scores[p] for p in range(n_pages - 1)]
    if len(cands) <= topk:
        return None
    return sorted(cands, reverse=True)[topk - 1]


def keep_windows(n_tokens: int, page_size: int, sink_tokens: int, recent_tokens: int):
    """(always-kept pages, candidate pages), both ascending: a page is always kept if it
    holds one of the first ``sink_tokens`` tokens, one of the last ``recent_tokens`` tokens,
    or is the last page."""
    n = num_pages(n_tokens, page_size)
    sink = set(range(min(sink_tokens, n_tokens)))
    recent = set(range(max(0, n_tokens - recent_tokens), n_tokens))
    kept, cands = [], []
    for p in range(n):
        tokens = range(p * page_size, min((p + 1) * page_size, n_tokens))
        if p == n - 1 or any(t in sink or t in recent for t in tokens):
            kept.append(p)
        else:
            cands.append(p)
    return kept, cands


def select_pages_windowed(scores, n_tokens: int, page_size: int, topk: int, sink_tokens: int,
                          recent_tokens: int) -> list:
    """Ascending page ids: the kept windows plus the ``topk`` best candidates between them."""
    kept, cands = keep_windows(n_tokens, page_size, sink_tokens, recent_tokens)
    ranked = sorted(cands, key=lambda p: (-scores[p], p))
    return sorted(set(kept) | set(ranked[:topk]))


def kth_score_windowed(scores, n_tokens: int, page_size: int, topk: int, sink_tokens: int, recent_tokens: int):
    """The k-th largest candidate score, or None when every candidate is kept."""
    _, cands = keep_windows(n_tokens, page_size, sink_tokens, recent_tokens)
    if len(cands) <= topk:
        return None
    return sorted((scores[p] for p in cands), reverse=True)[topk - 1]


# ---------------------------------------------------------------- step 5
def softmax_attention(q_group: np.ndarray, K: np.ndarray, V: np.ndarray, sm_scale: float):
    """o = softmax(sm_scale * q K^T) V and lse = log sum exp(sm_scale * q K^T), row-wise."""
    z = sm_scale * (q_group @ K.T)
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    denom = e.sum(axis=1, keepdims=True)
    return (e / denom) @ V, zmax[:, 0] + np.log(denom[:, 0])


# ---------------------------------------------------------------- one request
@dataclass
class HeadResult:
    scores: np.ndarray       # group score of each candidate page 0..n-2
    pages: list              # selected logical pages, ascending, last page included
    threshold: object        # k-th largest candidate score, or None when every page is kept


@dataclass
class RequestResult:
    heads: list              # HeadResult per KV head
    out: np.ndarray          # [Hq][Dv]
    lse: np.ndarray          # [Hq]


@dataclass
class QuestRequest:
    """One request's paged KV view plus its Quest page summaries (the method's state).

    ``k_cache``/``v_cache`` are indexed [physical page][kv head][slot][dim] (numpy or CPU
    torch); ``v_cache`` is None for a latent cache, whose value is the first
    ``head_dim_v`` dims of the key row. Appended tokens are held here, not written into
    the caller's cache.
    """
    k_cache: object
    v_cache: object
    block_table_row: object
    n_tokens: int
    num_kv_heads: int
    head_dim: int
    head_dim_v: int
    page_size: int = 16
    summaries: list = field(default=None)     # per KV head: (m [n][D], M [n][D])
    appended: dict = field(default_factory=dict)  # position -> (k [Hkv][D], v [Hkv][Dv])

    def __post_init__(self):
        if self.summaries is None:
            self.summaries = [self._build_summaries(h) for h in range(self.num_kv_heads)]

    # -- rows of the paged view, with appended tokens overriding their slots
    def page_rows(self, h: int, page: int, value: bool) -> np.ndarray:
        valid = min(self.page_size, self.n_tokens - page * self.page_size)
        phys = int(self.block_table_row[page])
        width = self.head_dim_v if value else self.head_dim
        cache = self.v_cache if (value and self.v_cache is not None) else self.k_cache
        rows = f64(cache[phys, h, :valid, :width]).copy()
        for pos, (kn, vn) in self.appended.items():
            if pos // self.page_size == page and pos % self.page_size < valid:
                src = (vn if (value and vn is not None) else kn)[h]
                rows[pos % self.page_size] = f64(src)[:width]
        return rows

    def _build_summaries(self, h: int):
        n = num_pages(self.n_tokens, self.page_size)
        m = np.empty((n, self.head_dim))
        M = np.empty((n, self.head_dim))
        for p in range(n):
            m[p], M[p] = page_summary(self.page_rows(h, p, value=False))
        return m, M

    def append(self, k_new, v_new=None):
        """Append one token (k_new [Hkv][D], v_new [Hkv][Dv] or None for a latent cache)."""
        pos = self.n_tokens
        page, off = divmod(pos, self.page_size)
        kn = f64(k_new)
        self.appended[pos] = (kn, None if v_new is None else f64(v_new))
        self.n_tokens += 1
        for h in range(self.num_kv_heads):
            m, M = self.summaries[h]
            if page == m.shape[0]:
                m = np.vstack([m, np.zeros((1, self.head_dim))])
                M = np.vstack([M, np.zeros((1, self.head_dim))])
            m[page], M[page] = append_to_summary(m[page], M[page], kn[h], off)
            self.summaries[h] = (m, M)

    def decode(self, q, topk_pages: int, sm_scale: float, pages_override=None, sink_tokens: int = 0,
               recent_tokens: int = 0) -> RequestResult:
        """Select pages per KV head (with the keep windows of step 4b) and attend.
        ``pages_override[h]`` replaces the selection."""
        q = f64(q)
        G = q.shape[0] // self.num_kv_heads
        n = num_pages(self.n_tokens, self.page_size)
        heads, outs, lses = [], [], []
        for h in range(self.num_kv_heads):
            qg = q[h * G:(h + 1) * G]
            m, M = self.summaries[h]
            scores = group_page_scores(qg, m[:max(n - 1, 0)], M[:max(n - 1, 0)])
            if sink_tokens == 0 and recent_tokens == 0:
                pages = select_pages(scores, n, topk_pages)
                tau = kth_score(scores, n, topk_pages)
            else:
                ps = self.page_size
                pages = select_pages_windowed(scores, self.n_tokens, ps, topk_pages, sink_tokens, recent_tokens)
                tau = kth_score_windowed(scores, self.n_tokens, ps, topk_pages, sink_tokens, recent_tokens)
            heads.append(HeadResult(scores, pages, tau))
            use = pages if pages_override is None else list(pages_override[h])
            if not use:  # no token to attend to: the empty sum (zero output, lse = -inf)
                o, lse = np.zeros((G, self.head_dim_v)), np.full(G, -np.inf)
            else:
                K = np.vstack([self.page_rows(h, p, value=False) for p in use])
                V = np.vstack([self.page_rows(h, p, value=True) for p in use])
                o, lse = softmax_attention(qg, K, V, sm_scale)
            outs.append(o)
            lses.append(lse)
        return RequestResult(heads, np.vstack(outs), np.concatenate(lses))


def decode_step(inputs, topk_pages: int, sm_scale: float, requests=None, pages_override=None, sink_tokens: int = 0,
                recent_tokens: int = 0):
    """Oracle decode step over the requests of a batch (all by default).

    ``inputs`` carries CPU copies of: k_cache, v_cache (or None), block_table [B][w],
    seq_lens (tokens before the step), q [B][Hq][D], and for an appending step k_new,
    v_new. Returns {b: RequestResult}.
    """
    out = {}
    B = len(inputs["seq_lens"])
    for b in (range(B) if requests is None else requests):
        req = QuestRequest(inputs["k_cache"], inputs["v_cache"], inputs["block_table"][b],
                           int(inputs["seq_lens"][b]), inputs["num_kv_heads"], inputs["head_dim"],
                           inputs["head_dim_v"], inputs.get("page_size", 16))
        if inputs.get("k_new") is not None:
            vn = inputs["v_new"][b] if inputs.get("v_new") is not None else None
            req.append(inputs["k_new"][b], vn)
        po = None if pages_override is None else pages_override[b]
        out[b] = req.decode(inputs["q"][b], topk_pages, sm_scale, po, sink_tokens, recent_tokens)
    return out
