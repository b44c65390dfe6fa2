"""Comparison of the CUDA path's results with the fp64 oracle.

Selection rule: let tau be the oracle's k-th largest candidate score. A page
whose oracle score lies within 1e-3 * |tau| of tau (1e-6 absolute when tau is
0) is exempt; every other candidate's membership must match exactly, the
count must match exactly, and the last page must be present. The same rule
applies to SnapKV kept positions on the pooled scores.

Attention rule: outputs within 2e-2 max-abs of the oracle's attention over
the GPU's own selected pages (so that an exempt swap does not count as an
error); log-sum-exp within 1e-3 absolute (fp32 sums of exact bf16 products).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.quest as oq

OUT_ATOL = 2e-2
LSE_ATOL = 1e-3
SEL_REL = 1e-3


def exempt(score: float, tau, rel: float = SEL_REL) -> bool:
    if tau is None:
        return False
    tol = rel * abs(tau) if tau != 0 else 1e-6
    return abs(score - tau) <= tol


def check_page_selection(gpu_pages, gpu_count: int, head: "oq.HeadResult", n_pages: int, what: str = ""):
    """Raise AssertionError if the GPU selection breaks the rule above."""
    ref = head.pages
    assert gpu_count == len(ref), f"{what}: count {gpu_count} != {len(ref)}"
    got = [int(x) for x in gpu_pages[:gpu_count]]
    assert got == sorted(set(got)), f"{what}: not ascending/unique: {got[:10]}"
    if n_pages > 0:
        assert got[-1] == n_pages - 1, f"{what}: last page missing"
    gs, rs = set(got), set(ref)
    for p in range(max(n_pages - 1, 0)):
        if (p in gs) != (p in rs) and not exempt(head.scores[p], head.threshold):
            raise AssertionError(f"{what}: page {p} membership differs (score {head.scores[p]!r}, "
                                 f"tau {head.threshold!r})")


def oracle_inputs(x, requests=None):
    """CPU copies of a QuestDecodeInputs for oracle.quest.decode_step.

    Only the pages of ``requests`` are copied: they are gathered through the block table
    into a compact cache whose table is the identity, which leaves every logical row the same.
    """
    wl = x.workload
    reqs = list(range(wl.batch)) if requests is None else list(requests)
    bt = x.block_table
    pages, rows, offs = [], [], {}
    at = 0
    for b in reqs:
        n = x.pages_per_request[b]
        pages.append(bt[b, :n].long())
        offs[b] = at
        at += n
    idx = torch.cat(pages)
    k = x.k_cache[idx].cpu()
    v = None if x.v_cache is None else x.v_cache[idx].cpu()
    width = max(x.pages_per_request[b] for b in reqs)
    table = np.zeros((wl.batch, width), dtype=np.int64)
    for b in reqs:
        table[b, :x.pages_per_request[b]] = offs[b] + np.arange(x.pages_per_request[b])
    return {
        "k_cache": k, "v_cache": v, "block_table": table, "seq_lens": list(x.seq_lens),
        "q": x.q.cpu(), "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
        "head_dim_v": wl.head_dim_v, "page_size": wl.page_size,
        "k_new": None if x.k_new is None else x.k_new.cpu(),
        "v_new": None if x.v_new is None else x.v_new.cpu(),
    }


def compare_decode(x, step, requests, sm_scale: float, what: str = "", sink_tokens: int = 0,
                   recent_tokens: int = 0):
    """Selection and output of ``step`` (after run) against the oracle on ``requests``
    (with the keep windows ``sink_tokens`` / ``recent_tokens``).

    Returns the maximum absolute output error seen.
    """
    wl = x.workload
    inp = oracle_inputs(x, requests)
    ref = oq.decode_step(inp, wl.topk_pages, sm_scale, requests=requests, sink_tokens=sink_tokens,
                         recent_tokens=recent_tokens)
    sel = step.sel.cpu().numpy()
    cnt = step.counts.cpu().numpy()
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    worst = 0.0
    lens_after = x.seq_lens_after
    override = {}
    for b in requests:
        n = math.ceil(lens_after[b] / wl.page_size)
        for h in range(wl.num_kv_heads):
            check_page_selection(sel[b, h], int(cnt[b, h]), ref[b].heads[h], n, f"{what} b={b} h={h}")
        override[b] = [list(sel[b, h, :cnt[b, h]]) for h in range(wl.num_kv_heads)]
    again = oq.decode_step(inp, wl.topk_pages, sm_scale, requests=requests, pages_override=override)
    for b in requests:
        err = np.abs(out[b] - again[b].out)
        assert np.isfinite(out[b]).all(), f"{what} b={b}: non-finite output"
        worst = max(worst, float(err.max()))
        assert err.max() <= OUT_ATOL, f"{what} b={b}: max |out - oracle| = {err.max():.4g}"
        both_empty = np.isneginf(lse[b]) & np.isneginf(again[b].lse)  # empty request: -inf on both sides
        lerr = np.where(both_empty, 0.0, np.abs(lse[b] - np.where(both_empty, 0.0, again[b].lse))).max()
        assert lerr <= LSE_ATOL, f"{what} b={b}: max |lse - oracle| = {lerr:.4g}"
    return worst
