"""Quest decode over a latent (MLA-style) cache on the GPU against the fp64 oracle.

The latent recipe: one KV head whose 576-dim row (512 latent + 64 RoPE dims,
outlier channels in the RoPE part) is the key and whose first 512 dims are the
value, shared by 16..64 query heads. Cases: ragged oracle-sized batches with
several decode splits per request and ragged tails, every supported head
count, edge lengths, the decode on the oracle's own selection (output and
log-sum-exp), split-count invariance, and the full 64 x 32K workload checked
on sampled requests.
"""
import math

import numpy as np
import pytest
import torch

import oracle.quest as oq
import sparse_decode_attention_quest_gb300 as se
from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
from synth import MLA_GLM_QUEST_32K, make_quest_decode_inputs
from tests.parity import LSE_ATOL, OUT_ATOL, compare_decode, oracle_inputs

pytestmark = pytest.mark.gpu


def _prepare(wl, dev, device_gen=False, sel_stride=None):
    x = make_quest_decode_inputs(wl, device=dev if device_gen else "cpu", poison_tail=True)
    k = x.k_cache.to(dev)
    step = QuestDecodeStep(k, None, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(max(x.seq_lens_after), 1), head_dim_v=wl.head_dim_v, sel_stride=sel_stride)
    lens = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    step.build_summaries(lens)
    return x, step, lens


def _run(x, step, lens, dev):
    step.run(x.q.to(dev), lens)
    torch.cuda.synchronize()


def _scale(wl):
    return 1.0 / math.sqrt(wl.head_dim)


@pytest.fixture(autouse=True)
def _no_device_errors(se_lib, cuda_device):
    se.se_read_device_error(clear=True)
    yield
    assert se.se_read_device_error(clear=True) == 0


def test_latent_ragged_oracle_sized(cuda_device):
    wl = MLA_GLM_QUEST_32K.scaled(batch=4, context_min=700, context_max=3300, topk_pages=40, seed=41)
    x, step, lens = _prepare(wl, cuda_device)
    _run(x, step, lens, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "latent ragged")


@pytest.mark.parametrize("hq", [16, 32, 48])
def test_latent_head_counts(cuda_device, hq):
    wl = MLA_GLM_QUEST_32K.scaled(batch=3, num_q_heads=hq, context_min=400, context_max=1500, topk_pages=12,
                                  seed=43 + hq)
    x, step, lens = _prepare(wl, cuda_device)
    _run(x, step, lens, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"latent hq={hq}")


@pytest.mark.parametrize("sel_stride", [None, 64])  # one decode slice per request, or several + merge
def test_latent_edge_lengths(cuda_device, sel_stride):
    lens = (0, 1, 15, 16, 17, 33, 250, 1000)
    wl = MLA_GLM_QUEST_32K.scaled(batch=len(lens), lengths=lens, topk_pages=6, seed=47)
    x, step, lens_t = _prepare(wl, cuda_device, sel_stride=sel_stride)
    _run(x, step, lens_t, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), f"latent edges stride={sel_stride}")
    assert float(step.out[0].float().abs().max()) == 0.0       # empty request: zero output
    assert torch.isneginf(step.lse[0]).all()


def test_latent_many_pages_per_slice(cuda_device):
    """About 11,000 selected pages in all, so a CTA slice on a 152-SM GPU holds
    more than 64 pages of one request and walks past two 32-page metadata
    windows."""
    wl = MLA_GLM_QUEST_32K.scaled(batch=10, num_q_heads=16, context_min=18000, context_max=19000,
                                  topk_pages=1100, seed=67)
    x, step, lens = _prepare(wl, cuda_device)
    _run(x, step, lens, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "latent long slices")


def test_latent_one_request_over_many_splits(cuda_device):
    """One request's 1,101 selected pages over 16-page slices: about 70 decode
    splits, so the combine takes their log-sum-exps in several chunks of 32."""
    wl = MLA_GLM_QUEST_32K.scaled(batch=1, num_q_heads=16, context_min=18000, context_max=18000,
                                  topk_pages=1100, seed=71)
    x, step, lens = _prepare(wl, cuda_device)
    _run(x, step, lens, cuda_device)
    compare_decode(x, step, range(wl.batch), _scale(wl), "latent many splits")


def test_latent_value_outlier_channels(cuda_device):
    """Outlier channels (x3) drawn over the whole 576-dim row, so that some fall
    in the value part: the output stays below 4 in magnitude, where bf16
    rounding is well inside the absolute tolerance."""
    wl = MLA_GLM_QUEST_32K.scaled(batch=3, context_min=1800, context_max=3000, topk_pages=30, seed=73,
                                  outliers_in_value=True, outlier_channels=12, outlier_scale=3.0)
    x, step, lens = _prepare(wl, cuda_device)
    assert any(c < wl.head_dim_v for c in x.outlier_channels[0])  # some outliers are value dims
    _run(x, step, lens, cuda_device)
    assert float(step.out.float().abs().max()) < 4.0
    compare_decode(x, step, range(wl.batch), _scale(wl), "latent value outliers")


def test_latent_decode_on_the_oracle_selection(cuda_device):
    wl = MLA_GLM_QUEST_32K.scaled(batch=3, context_min=2000, context_max=2600, topk_pages=30, seed=53)
    x, step, lens = _prepare(wl, cuda_device)
    inp = oracle_inputs(x)
    ref = oq.decode_step(inp, wl.topk_pages, _scale(wl))
    sel = torch.zeros(wl.batch, 1, wl.topk_pages + 1, dtype=torch.int32)
    cnt = torch.zeros(wl.batch, 1, dtype=torch.int32)
    for r in range(wl.batch):
        pg = ref[r].heads[0].pages
        sel[r, 0, :len(pg)] = torch.tensor(pg)
        cnt[r, 0] = len(pg)
    step.attend(x.q.to(cuda_device), lens, sel.to(cuda_device), cnt.to(cuda_device))
    torch.cuda.synchronize()
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    for r in range(wl.batch):
        assert np.abs(out[r] - ref[r].out).max() <= OUT_ATOL
        assert np.abs(lse[r] - ref[r].lse).max() <= LSE_ATOL


def test_latent_split_count_does_not_change_the_result(cuda_device):
    wl = MLA_GLM_QUEST_32K.scaled(batch=2, context_min=3000, context_max=3000, topk_pages=60, seed=59)
    x, s1, lens = _prepare(wl, cuda_device)
    _run(x, s1, lens, cuda_device)
    x2, s2, lens2 = _prepare(wl, cuda_device, sel_stride=wl.topk_pages + 1 + 100)
    _run(x2, s2, lens2, cuda_device)
    assert torch.equal(s1.counts, s2.counts)
    assert torch.equal(s1.sel, s2.sel[:, :, :wl.topk_pages + 1])
    assert (s1.out.float() - s2.out.float()).abs().max().item() <= 1e-2
    assert (s1.lse - s2.lse).abs().max().item() <= 1e-4


def test_full_mla_glm_32k_sampled(cuda_device):
    wl = MLA_GLM_QUEST_32K
    x, step, lens = _prepare(wl, cuda_device, device_gen=True)
    _run(x, step, lens, cuda_device)
    compare_decode(x, step, [0, 31, wl.batch - 1], _scale(wl), "mla-glm full")


def test_latent_decode_is_repeatable(cuda_device):
    """The full 64 x 32K decode run again and again gives bit-identical outputs and
    log-sum-exps. A decode pipeline whose epilogue read the output accumulators before
    the last tiles' PV MMAs had landed gave a request output that changed from one run
    to the next (with the exact log-sum-exp, and within the output tolerance)."""
    wl = MLA_GLM_QUEST_32K
    x, step, lens = _prepare(wl, cuda_device, device_gen=True)
    q = x.q.to(cuda_device)
    step.select(q, lens)
    step.attend(q, lens)
    torch.cuda.synchronize()
    out0, lse0 = step.out.clone(), step.lse.clone()
    for _ in range(12):
        step.attend(q, lens)
        torch.cuda.synchronize()
        assert torch.equal(step.out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(step.lse, lse0)


def test_latent_growing_scores_rescale_every_tile(cuda_device):
    """Scores that grow by more than 2^8 (log2 units) from one 4-page tile to the
    next, so that the decode's running maxima move on every tile and the output
    accumulators are rescaled each time. The RoPE dims of page p carry p times a
    direction shared by every query head; the value dims (the latent part) are
    left as generated. The decode attends over every page in order (an explicit
    selection), against the oracle on the same pages; the last page is ragged."""
    wl = MLA_GLM_QUEST_32K.scaled(batch=2, context_min=2040, context_max=2040, topk_pages=8, seed=71)
    x = make_quest_decode_inputs(wl, device="cpu", poison_tail=True)
    gen = torch.Generator().manual_seed(72)
    u = torch.randn(64, generator=gen)
    n = x.pages_per_request[0]
    for b in range(wl.batch):
        for p in range(n):
            phys = int(x.block_table[b, p])
            rows = x.k_cache[phys, 0, :, 512:].float() + 0.6 * p * u
            x.k_cache[phys, 0, :, 512:] = rows.to(torch.bfloat16)
    x.q[..., 512:] = (u + 0.05 * torch.randn(x.q[..., 512:].shape, generator=gen)).to(x.q.dtype)
    dev = cuda_device
    k = x.k_cache.to(dev)
    step = QuestDecodeStep(k, None, new_summary(k), x.block_table.to(dev), wl.num_q_heads, wl.topk_pages,
                           max(x.seq_lens_after), head_dim_v=wl.head_dim_v, sel_stride=n)
    lens = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    sel = torch.arange(n, dtype=torch.int32).repeat(wl.batch, 1, 1)
    cnt = torch.full((wl.batch, 1), n, dtype=torch.int32)
    step.attend(x.q.to(dev), lens, sel.to(dev), cnt.to(dev))
    torch.cuda.synchronize()
    inp = oracle_inputs(x)
    ref = oq.decode_step(inp, wl.topk_pages, _scale(wl), pages_override=[[list(range(n))]] * wl.batch)
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    # the shared component alone raises the logits by more than 8 (log2 units) per tile
    assert 4 * 0.6 * float(u.square().sum()) * _scale(wl) / math.log(2) > 8
    for r in range(wl.batch):
        assert np.abs(out[r] - ref[r].out).max() <= OUT_ATOL
        assert np.abs(lse[r] - ref[r].lse).max() <= LSE_ATOL
