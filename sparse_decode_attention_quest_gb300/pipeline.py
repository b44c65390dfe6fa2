"""One Quest decode step over a paged cache: buffers plus the C-ABI calls in order.

Host orchestration only (allocation and call order); the work runs in the
library's kernels:
    se_quest_update_summaries   (optional KV append fused with the summary update)
    se_quest_score_pages_ws     (upper-bound score of every candidate page; the group's query
                                 sums computed once per request into a workspace)
    se_quest_topk_pages_windowed (top-k pages + the sink/recent windows + the last page, ascending)
    se_sparse_paged_decode      (split-K flash-decode over the selected pages, partials merged in the same launch)
or all four in one launch (se_quest_fused_step, run_fused).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

from . import (APPEND_OVERLAP_PREVIOUS, paged_kv, se_quest_build_summaries, se_quest_fused_step, se_quest_kept_pages_max,
               se_quest_score_pages, se_quest_score_pages_ws, se_quest_score_workspace_size,
               se_quest_topk_pages_windowed, se_quest_update_summaries,
               se_quest_update_summaries_ex, se_snapkv_score_and_compact_windowed,
               se_snapkv_workspace_size, se_sparse_decode_plan, se_sparse_decode_workspace_size,
               se_sparse_paged_decode)

PAGE = 16


def new_summary(k_cache: torch.Tensor) -> torch.Tensor:
    """Summary storage beside a cache [P][Hkv][16][D]: bf16 [P][Hkv][2][D]."""
    P, H, _, D = k_cache.shape
    return torch.empty(P, H, 2, D, dtype=torch.bfloat16, device=k_cache.device)


class QuestDecodeStep:
    def __init__(self, k_cache: torch.Tensor, v_cache: Optional[torch.Tensor], summary: torch.Tensor,
                 block_table: torch.Tensor, num_q_heads: int, topk_pages: int, max_seq_len: int,
                 head_dim_v: Optional[int] = None, sm_scale: Optional[float] = None, sel_stride: Optional[int] = None,
                 sink_tokens: int = 0, recent_tokens: int = 0, score_workspace: bool = True):
        """score_workspace: score through se_quest_score_pages_ws (the query sums of every
        request computed once, in a workspace of batch x KV heads x 2 x head_dim floats)
        rather than se_quest_score_pages; both give the same scores."""
        self.k_cache, self.v_cache, self.summary = k_cache, v_cache, summary
        self.block_table = block_table
        self.kv = paged_kv(k_cache, v_cache, summary, head_dim_v)
        dev = k_cache.device
        self.B = block_table.shape[0]
        self.H = k_cache.shape[1]
        self.Hq = num_q_heads
        self.D = k_cache.shape[-1]
        self.Dv = self.kv.head_dim_v
        self.topk = topk_pages
        self.max_seq_len = max_seq_len
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(self.D)
        stride = max(1, (max_seq_len + PAGE - 1) // PAGE)
        self.scores = torch.empty(self.B, self.H, stride, dtype=torch.float32, device=dev)
        self.sink, self.recent = sink_tokens, recent_tokens
        kept_max = se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens)
        self.sel_stride = sel_stride if sel_stride is not None else kept_max
        self.sel = torch.empty(self.B, self.H, self.sel_stride, dtype=torch.int32, device=dev)
        self.counts = torch.empty(self.B, self.H, dtype=torch.int32, device=dev)
        self.out = torch.empty(self.B, self.Hq, self.Dv, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(self.B, self.Hq, dtype=torch.float32, device=dev)
        ws = se_sparse_decode_workspace_size(self.B, self.Hq, self.H, self.Dv, self.sel_stride)
        # zero-filled once: the decode's split-merge counters start at zero and every call leaves them so
        self.workspace = torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev)
        self.score_ws = None
        if score_workspace:
            sws = se_quest_score_workspace_size(self.B, self.H, self.D)
            self.score_ws = torch.empty(max(sws, 16), dtype=torch.uint8, device=dev)

    def launches_per_step(self, append: bool = True) -> int:
        """Kernels one run() launches: append, (query sums,) score, top-k, decode (+ the latent split merge)."""
        _, _, dec = se_sparse_decode_plan(self.B, self.Hq, self.H, self.D, self.Dv, self.sel_stride)
        return (1 if append else 0) + (3 if self.score_ws is not None else 2) + dec

    def build_summaries(self, seq_lens: torch.Tensor, stream=None):
        se_quest_build_summaries(self.kv, self.block_table, seq_lens, self.max_seq_len, stream)

    def append(self, k_new, v_new, seq_lens_before, stream=None, overlap_previous=False):
        se_quest_update_summaries_ex(self.kv, k_new, v_new, self.block_table, seq_lens_before,
                                     APPEND_OVERLAP_PREVIOUS if overlap_previous else 0, stream)

    def score(self, q, seq_lens, stream=None):
        if self.score_ws is not None:
            se_quest_score_pages_ws(self.kv, q, self.block_table, seq_lens, self.max_seq_len, self.scores,
                                    self.score_ws, stream)
        else:
            se_quest_score_pages(self.kv, q, self.block_table, seq_lens, self.max_seq_len, self.scores, stream)

    def select(self, q, seq_lens, stream=None):
        self.score(q, seq_lens, stream)
        se_quest_topk_pages_windowed(self.scores, seq_lens, self.H, self.max_seq_len, self.topk, self.sink,
                                     self.recent, self.sel, self.counts, stream)

    def attend(self, q, seq_lens, sel=None, counts=None, stream=None):
        se_sparse_paged_decode(self.kv, q, self.block_table, seq_lens, self.sel if sel is None else sel,
                               self.counts if counts is None else counts, self.sm_scale, self.out, self.lse,
                               self.workspace, stream)

    def run_fused(self, q, seq_lens, k_new=None, v_new=None, stream=None):
        """The whole step in one launch (se_quest_fused_step): ``seq_lens`` are the lengths
        after the append; with k_new/v_new the token at seq_lens - 1 is appended first."""
        se_quest_fused_step(self.kv, k_new, v_new, q, self.block_table, seq_lens, self.max_seq_len, self.topk,
                            self.sink, self.recent, self.sm_scale, self.out, self.lse, self.sel, self.counts, stream)
        return self.out

    def run(self, q, seq_lens, k_new=None, v_new=None, seq_lens_before=None, stream=None,
            events: Optional[Sequence] = None):
        """Full step. ``seq_lens``: lengths including the new token; with k_new/v_new the token
        at ``seq_lens_before`` is appended.

        Without ``events`` the kernels run score, top-k, append, decode: the token lands in its
        request's last page, which is never scored (it is always kept), so the append may run
        alongside the top-k (se_quest_update_summaries_ex, SE_APPEND_OVERLAP_PREVIOUS) and only
        the decode waits for it. With ``events`` (4 CUDA events) they run append, score, top-k,
        decode one after another, with the events recorded on ``stream`` before each, for
        per-kernel timing."""
        s = stream if stream is not None else torch.cuda.current_stream()
        if events is None:
            self.score(q, seq_lens, s)
            se_quest_topk_pages_windowed(self.scores, seq_lens, self.H, self.max_seq_len, self.topk, self.sink,
                                         self.recent, self.sel, self.counts, s)
            if k_new is not None:
                self.append(k_new, v_new, seq_lens_before, s, overlap_previous=True)
            self.attend(q, seq_lens, stream=s)
            return self.out
        events[0].record(s)
        if k_new is not None:
            self.append(k_new, v_new, seq_lens_before, s)
        events[1].record(s)
        self.score(q, seq_lens, s)
        events[2].record(s)
        se_quest_topk_pages_windowed(self.scores, seq_lens, self.H, self.max_seq_len, self.topk, self.sink,
                                     self.recent, self.sel, self.counts, s)
        events[3].record(s)
        self.attend(q, seq_lens, stream=s)
        return self.out


class SnapKVDecodeCache:
    """A SnapKV-compacted paged cache through decode: the prefill eviction, then every
    ``period`` decode steps another eviction over the compacted pages (SparseEngine, Table 10:
    SnapKV with a 16-query observation window, sink 16, recent 64, 4,096 selected, eviction
    every 1,024 decode steps).

    Two page pools of the same size, the live one and the one the next eviction compacts
    into; request b owns pages b * P .. b * P + P - 1 of each (P = pages for sink + keep +
    recent + period tokens). A decode step appends its token's K/V rows to the live pool and
    keeps its query if it is among the last ``window`` of the period, in order: the
    observation window of the next eviction. Host orchestration only; appends and
    evictions run in the library's kernels.
    """

    def __init__(self, batch: int, num_kv_heads: int, num_q_heads: int, head_dim: int, window: int,
                 pool_kernel: int, keep_topk: int, sink_tokens: int, recent_tokens: int, period: int, device,
                 sm_scale: Optional[float] = None):
        if period < window:
            raise ValueError("period must cover the observation window")
        self.B, self.H, self.Hq, self.D = batch, num_kv_heads, num_q_heads, head_dim
        self.W, self.pool, self.keep = window, pool_kernel, keep_topk
        self.sink, self.recent, self.period = sink_tokens, recent_tokens, period
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)
        self.kept_max = sink_tokens + keep_topk + recent_tokens
        self.max_len = self.kept_max + period
        self.P = (self.max_len + PAGE - 1) // PAGE
        shape = (batch * self.P, num_kv_heads, PAGE, head_dim)
        self.k = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.v = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.block_table = torch.arange(batch * self.P, dtype=torch.int32, device=device).view(batch, self.P)
        self.live = 0
        self.lens = torch.zeros(batch, dtype=torch.int32, device=device)
        self.q_window = torch.zeros(batch, window, num_q_heads, head_dim, dtype=torch.bfloat16, device=device)
        self.kept = torch.empty(batch, num_kv_heads, self.kept_max, dtype=torch.int32, device=device)
        self.counts = torch.empty(batch, num_kv_heads, dtype=torch.int32, device=device)
        self.steps = 0
        self.evictions = 0

    def kv(self, pool: Optional[int] = None):
        i = self.live if pool is None else pool
        return paged_kv(self.k[i], self.v[i], None)

    def evict_from(self, src_kv, src_block_table, lens, q_window, max_len: int, stream=None):
        """Compacts (cache, lengths, the window's queries) into the pool that is not live and
        makes it live: the prefill eviction (the prompt's cache) and every periodic one."""
        dst = 1 - self.live
        ws = torch.empty(max(se_snapkv_workspace_size(self.B, self.H, self.W, max_len), 16), dtype=torch.uint8,
                         device=self.lens.device)
        se_snapkv_score_and_compact_windowed(src_kv, q_window, src_block_table, lens, max_len, self.pool, self.keep,
                                             self.sink, self.recent, self.sm_scale, self.kv(dst), self.block_table,
                                             self.kept, self.counts, ws, stream)
        self.lens = self.counts[:, 0].contiguous()  # every KV head of a request keeps as many positions
        self.live = dst
        self.steps = 0
        self.evictions += 1

    def append(self, k_new, v_new, q, stream=None):
        """One decode step: K/V rows of the new token (k_new, v_new [B][Hkv][D]) and its query
        q [B][Hq][D]; evicts when the period is complete."""
        se_quest_update_summaries(self.kv(), k_new, v_new, self.block_table, self.lens, stream)
        first = self.period - self.W
        if self.steps >= first:
            self.q_window[:, self.steps - first].copy_(q)
        self.lens = self.lens + 1
        self.steps += 1
        if self.steps == self.period:
            self.evict_from(self.kv(), self.block_table, self.lens, self.q_window, self.max_len, stream)
