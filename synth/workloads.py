"""Seeded synthetic workloads shaped like the SparseEngine evaluation settings.

The SparseEngine pages evaluate Quest and SnapKV on long-context models
(Qwen3-4B, Qwen3-30B-A3B, GLM-4.7-Flash with MLA) at 32K- and 128K-token
inputs with 16-token pages [SparseEngine: Sparse-First Inference Engine,
Figure 5 caption; Tables 8-12]. No dataset or weight is available, so every
tensor here is drawn from seeded generators with the shapes of those models:

* keys, values and queries are N(0, 1) in fp32, cast once to bf16;
* Quest workloads scale a few key channels per KV head by a fixed factor
  (outlier channels, as real keys have);
* the SnapKV workload gives 5% of key positions a shared direction that the
  window queries also carry, which raises those logits by a fixed amount
  (attention sinks);
* physical pages are handed out through a block table, either contiguous or
  randomly permuted;
* slots of a request's last page beyond its length hold NaN ("poison"), so a
  kernel that reads past the valid tokens shows up as a NaN.

Structural draws (lengths, permutations, outlier channels, sink positions)
come from a CPU generator and are identical on every device; bulk values come
from a generator on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace, field
from typing import Optional

import torch

PAGE_SIZE = 16


def pages_for_tokens(n_tokens: int, page_size: int = PAGE_SIZE) -> int:
    """Number of fixed-size pages that hold ``n_tokens`` tokens."""
    return (n_tokens + page_size - 1) // page_size


# --------------------------------------------------------------------------
# Quest decode workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class QuestDecodeWorkload:
    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int            # query / key width
    head_dim_v: int          # value width (== head_dim except for a latent cache)
    context_min: int         # tokens in the cache before the step, per request
    context_max: int         # (uniform integer in [min, max]; equal -> fixed)
    topk_pages: int          # pages chosen by the bound, besides the last page
    append: bool             # the step first appends one token per request
    permuted_table: bool     # random physical page order
    outlier_channels: int = 4
    outlier_scale: float = 8.0
    latent: bool = False     # one cache row holds the key; the value is its first head_dim_v dims
    outliers_in_value: bool = False  # latent cache: outlier channels drawn over all dims, the value's too
    page_size: int = PAGE_SIZE
    lengths: tuple = ()      # explicit per-request lengths (override the uniform draw)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "QuestDecodeWorkload":
        """Same recipe, other sizes (used for oracle-sized parity cases)."""
        return replace(self, **kw)


# 1 request, 1 KV head, 4 query heads, 4096 tokens (256 pages), 32 pages + last.
TINY_QUEST_4K = QuestDecodeWorkload(
    name="tiny_quest_b1_g4_4k", seed=0, batch=1, num_q_heads=4, num_kv_heads=1,
    head_dim=128, head_dim_v=128, context_min=4096, context_max=4096,
    topk_pages=32, append=False, permuted_table=False)

# Qwen3-4B attention shape: 32 query / 8 KV heads, d 128, 32K context, 2048-token budget.
QWEN3_4B_QUEST_32K = QuestDecodeWorkload(
    name="qwen3_4b_quest_b8_32k", seed=1, batch=8, num_q_heads=32, num_kv_heads=8,
    head_dim=128, head_dim_v=128, context_min=32768, context_max=32768,
    topk_pages=128, append=False, permuted_table=True)

# Qwen3-30B-A3B attention shape: 32 query / 4 KV heads, ragged 64K-128K, 4096-token budget,
# one decode step per request including the KV append.
QWEN3_30B_A3B_QUEST_128K = QuestDecodeWorkload(
    name="qwen3_30b_a3b_quest_b32_64k_128k", seed=2, batch=32, num_q_heads=32, num_kv_heads=4,
    head_dim=128, head_dim_v=128, context_min=65536, context_max=131072,
    topk_pages=256, append=True, permuted_table=True)

# GLM-4.7-Flash-like MLA: 64 heads share one latent cache row of 512 latent + 64 RoPE dims.
MLA_GLM_QUEST_32K = QuestDecodeWorkload(
    name="mla_glm_quest_b64_32k", seed=4, batch=64, num_q_heads=64, num_kv_heads=1,
    head_dim=576, head_dim_v=512, context_min=32768, context_max=32768,
    topk_pages=128, append=False, permuted_table=True, latent=True)

QUEST_WORKLOADS = {w.name: w for w in (TINY_QUEST_4K, QWEN3_4B_QUEST_32K,
                                        QWEN3_30B_A3B_QUEST_128K, MLA_GLM_QUEST_32K)}


@dataclass
class QuestDecodeInputs:
    workload: QuestDecodeWorkload
    seq_lens: list            # tokens before the step (python ints)
    pages_per_request: list   # pages allocated to each request (after any append)
    num_pages: int            # physical pages in the pool
    block_table: torch.Tensor  # int32 [B][width], unused entries 0
    k_cache: torch.Tensor      # bf16 [P][Hkv][page][head_dim]
    v_cache: Optional[torch.Tensor]  # bf16 [P][Hkv][page][head_dim_v]; None for a latent cache
    q: torch.Tensor            # bf16 [B][Hq][head_dim]
    k_new: Optional[torch.Tensor]  # bf16 [B][Hkv][head_dim] (append only)
    v_new: Optional[torch.Tensor]  # bf16 [B][Hkv][head_dim_v] (append only, not latent)
    outlier_channels: list = field(default_factory=list)  # per KV head

    @property
    def seq_lens_after(self) -> list:
        return [L + (1 if self.workload.append else 0) for L in self.seq_lens]


def _draw_lengths(wl, g):
    if wl.lengths:
        assert len(wl.lengths) == wl.batch
        return list(wl.lengths)
    if wl.context_min == wl.context_max:
        return [wl.context_min] * wl.batch
    return torch.randint(wl.context_min, wl.context_max + 1, (wl.batch,), generator=g).tolist()


def _block_table(pages_per_request, permuted, g):
    total = sum(pages_per_request)
    phys = torch.randperm(total, generator=g) if permuted else torch.arange(total)
    width = max(pages_per_request) if pages_per_request else 1
    bt = torch.zeros(len(pages_per_request), max(width, 1), dtype=torch.int32)
    at = 0
    for b, n in enumerate(pages_per_request):
        bt[b, :n] = phys[at:at + n].to(torch.int32)
        at += n
    return bt, total


def _randn_bf16(shape, gen, device, chunk_rows=4096, col_scale=None):
    """N(0,1) fp32 draws cast to bf16, generated in chunks along dim 0 to bound memory.

    ``col_scale`` (broadcastable to shape[1:]) multiplies the fp32 draws before the cast.
    """
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device, dtype=torch.float32)
        if col_scale is not None:
            x.mul_(col_scale)
        out[s:e] = x.to(torch.bfloat16)
    return out


def make_quest_decode_inputs(wl: QuestDecodeWorkload, device="cpu", poison_tail=True) -> QuestDecodeInputs:
    device = torch.device(device)
    cpu_g = torch.Generator("cpu").manual_seed(wl.seed)
    lens = _draw_lengths(wl, cpu_g)
    extra = 1 if wl.append else 0
    ppr = [pages_for_tokens(L + extra, wl.page_size) for L in lens]
    bt, num_pages = _block_table(ppr, wl.permuted_table, cpu_g)

    # Outlier key channels, per KV head. For a latent cache the outliers sit in the
    # RoPE part of the row (dims head_dim_v .. head_dim-1), which is not part of the
    # value, unless outliers_in_value draws them over the whole row.
    lo = wl.head_dim_v if wl.latent and not wl.outliers_in_value else 0
    width = wl.head_dim - lo
    outliers = []
    scale = torch.ones(wl.num_kv_heads, 1, wl.head_dim)
    for h in range(wl.num_kv_heads):
        ch = (torch.randperm(width, generator=cpu_g)[:wl.outlier_channels] + lo).tolist()
        outliers.append(sorted(ch))
        scale[h, 0, ch] = wl.outlier_scale
    scale = scale.to(device)

    dev_g = torch.Generator(device).manual_seed(wl.seed)
    kshape = (num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim)
    k_cache = _randn_bf16(kshape, dev_g, device, col_scale=scale)
    v_cache = None
    if not wl.latent:
        v_cache = _randn_bf16((num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim_v), dev_g, device)
    q = _randn_bf16((wl.batch, wl.num_q_heads, wl.head_dim), dev_g, device)
    k_new = v_new = None
    if wl.append:
        k_new = _randn_bf16((wl.batch, wl.num_kv_heads, wl.head_dim), dev_g, device,
                            col_scale=scale[:, 0, :])
        if not wl.latent:
            v_new = _randn_bf16((wl.batch, wl.num_kv_heads, wl.head_dim_v), dev_g, device)

    bt_dev = bt.to(device)
    if poison_tail:
        nan = float("nan")
        for b, L in enumerate(lens):
            for pos in range(L, ppr[b] * wl.page_size):
                phys = int(bt[b, pos // wl.page_size])
                k_cache[phys, :, pos % wl.page_size, :] = nan
                if v_cache is not None:
                    v_cache[phys, :, pos % wl.page_size, :] = nan
    return QuestDecodeInputs(workload=wl, seq_lens=lens, pages_per_request=ppr, num_pages=num_pages,
                             block_table=bt_dev, k_cache=k_cache, v_cache=v_cache, q=q,
                             k_new=k_new, v_new=v_new, outlier_channels=outliers)


# --------------------------------------------------------------------------
# SnapKV prefill-end eviction workload
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class SnapKVWorkload:
    name: str
    seed: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prompt_min: int
    prompt_max: int
    window: int = 32             # observation window (last queries of the prompt)
    pool_kernel: int = 7
    keep_topk: int = 2016        # positions selected besides the kept windows
    keep_sink: int = 0           # first positions always kept
    keep_recent: int = 0         # last positions always kept (0: the observation window)
    sink_fraction: float = 0.05  # share of key positions given the sink direction
    sink_logit_shift: float = 3.0
    permuted_table: bool = True
    page_size: int = PAGE_SIZE

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def recent(self) -> int:
        return self.keep_recent or self.window

    def scaled(self, **kw) -> "SnapKVWorkload":
        return replace(self, **kw)


# Qwen3-4B attention shape at the end of a 32K-token prefill; SnapKV settings of the
# LongBench runs (32-query window, pooling kernel 7, 2016 selected + 32 recent).
SNAPKV_PREFILL_32K = SnapKVWorkload(
    name="snapkv_prefill_b4_32k", seed=3, batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
    prompt_min=32768, prompt_max=32768)


# The same shape with the AIME-run SnapKV settings: 16-query observation window, sink 16,
# recent 64, 4,096 selected (4,176 kept).
SNAPKV_AIME_32K = SnapKVWorkload(
    name="snapkv_aime_b4_32k", seed=5, batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
    prompt_min=32768, prompt_max=32768, window=16, keep_topk=4096, keep_sink=16, keep_recent=64)

# ... and with the agent-run settings: 32-query window, sink 64, recent 512, 15,808 selected.
SNAPKV_AGENT_32K = SnapKVWorkload(
    name="snapkv_agent_b4_32k", seed=6, batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
    prompt_min=32768, prompt_max=32768, window=32, keep_topk=15808, keep_sink=64, keep_recent=512)


@dataclass
class SnapKVInputs:
    workload: SnapKVWorkload
    prompt_lens: list
    src_pages_per_request: list
    dst_pages_per_request: list
    src_block_table: torch.Tensor   # int32 [B][w]
    dst_block_table: torch.Tensor   # int32 [B][w']
    k_cache: torch.Tensor           # bf16 [P][Hkv][page][D]
    v_cache: torch.Tensor
    q_window: torch.Tensor          # bf16 [B][W][Hq][D]: queries of the last W prompt positions
    dst_num_pages: int
    sink_positions: list            # [b][h] -> sorted list of positions


def make_snapkv_inputs(wl: SnapKVWorkload, device="cpu", poison_tail=True) -> SnapKVInputs:
    device = torch.device(device)
    cpu_g = torch.Generator("cpu").manual_seed(wl.seed)
    if wl.prompt_min == wl.prompt_max:
        lens = [wl.prompt_min] * wl.batch
    else:
        lens = torch.randint(wl.prompt_min, wl.prompt_max + 1, (wl.batch,), generator=cpu_g).tolist()
    ppr = [pages_for_tokens(n, wl.page_size) for n in lens]
    bt, num_pages = _block_table(ppr, wl.permuted_table, cpu_g)
    kept = [min(n, wl.keep_sink + wl.keep_topk + wl.recent) for n in lens]
    dppr = [pages_for_tokens(k, wl.page_size) for k in kept]
    dbt, dst_pages = _block_table(dppr, wl.permuted_table, cpu_g)

    dev_g = torch.Generator(device).manual_seed(wl.seed)
    shape = (num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim)
    k_cache = _randn_bf16(shape, dev_g, device)
    v_cache = _randn_bf16(shape, dev_g, device)
    q_window = _randn_bf16((wl.batch, wl.window, wl.num_q_heads, wl.head_dim), dev_g, device)

    # Attention sinks: a shared unit direction u, with amplitude a so that the scaled
    # logit of a window query with a sink key rises by sink_logit_shift
    # (a^2 / sqrt(D) = shift under the 1/sqrt(D) softmax scale).
    amp = math.sqrt(wl.sink_logit_shift * math.sqrt(wl.head_dim))
    sinks = []
    G = wl.group
    for b, n in enumerate(lens):
        row = []
        for h in range(wl.num_kv_heads):
            cnt = int(round(wl.sink_fraction * n))
            pos = torch.randperm(n, generator=cpu_g)[:cnt].sort().values
            u = torch.randn(wl.head_dim, generator=cpu_g)
            u = (u / u.norm()).to(device)
            row.append(pos.tolist())
            if cnt:
                phys = bt[b, pos // wl.page_size].long().to(device)
                slot = (pos % wl.page_size).long().to(device)
                kk = k_cache[phys, h, slot, :].float() + amp * u
                k_cache[phys, h, slot, :] = kk.to(torch.bfloat16)
            qq = q_window[b, :, h * G:(h + 1) * G, :].float() + amp * u
            q_window[b, :, h * G:(h + 1) * G, :] = qq.to(torch.bfloat16)
        sinks.append(row)

    if poison_tail:
        nan = float("nan")
        for b, n in enumerate(lens):
            for pos in range(n, ppr[b] * wl.page_size):
                phys = int(bt[b, pos // wl.page_size])
                k_cache[phys, :, pos % wl.page_size, :] = nan
                v_cache[phys, :, pos % wl.page_size, :] = nan
    return SnapKVInputs(workload=wl, prompt_lens=lens, src_pages_per_request=ppr,
                        dst_pages_per_request=dppr, src_block_table=bt.to(device),
                        dst_block_table=dbt.to(device), k_cache=k_cache, v_cache=v_cache,
                        q_window=q_window, dst_num_pages=dst_pages, sink_positions=sinks)
