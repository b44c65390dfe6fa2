"""Sparse decode attention bench: Quest select + sparse paged decode at 64K-128K context.

Workload: the Qwen3-30B-A3B attention shape (32 query / 4 KV heads, head dim
128), 32 requests with ragged contexts uniform in [65536, 131072] tokens,
16-token pages on a randomly permuted block table, a 4096-token budget (256
pages + the last page), one decode step per request that first appends the
new token (KV write + summary update). bf16 cache, fp32 accumulation.

One step = se_quest_score_pages_ws (a kernel summing each request's queries, then the
page scoring) + se_quest_topk_pages + se_quest_update_summaries_ex
(the append, overlapping the top-k: the token lands in the always-kept last page) +
se_sparse_paged_decode over the whole batch (one layer).
Inputs are resident in HBM; L2 is flushed (a 2x L2-sized write, then a 2x L2 read) between
steps, outside the timed spans; every step is timed with CUDA events on the
launching stream.

Output: one JSON line (rank 0). ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode attn tokens/sec & achieved HBM GB/s (frac of 8 TB/s) at 128K, 1 GB300"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
PAGE = 16


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


_BATCH_OVERRIDE = None


def _workload():
    """The 128K workload; ``--batch`` shrinks it only for profiler captures (never reported as the metric)."""
    from synth import QWEN3_30B_A3B_QUEST_128K
    wl = QWEN3_30B_A3B_QUEST_128K
    return wl if _BATCH_OVERRIDE is None else wl.scaled(batch=_BATCH_OVERRIDE)


def _config(wl, extra=None):
    c = {"workload": wl.name, "model_shape": "Qwen3-30B-A3B attention (32 q / 4 kv heads, d 128)",
         "batch": wl.batch, "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
         "head_dim": wl.head_dim, "context": [wl.context_min, wl.context_max], "page_size": wl.page_size,
         "topk_pages": wl.topk_pages, "kept_pages_per_kv_head": wl.topk_pages + 1,
         "append_per_step": wl.append, "block_table": "random permutation",
         "l2": "flushed between timed steps, outside the events: a write of 2x L2 size, then a read of "
               "another 2x L2 buffer (no dirty flush lines left behind)"}
    if extra:
        c.update(extra)
    return c


# --------------------------------------------------------------------------- ranks
def rank_workload(wl, rank):
    """Replica ``rank`` decodes its own batch: the same recipe, seed offset by 1000 x rank."""
    return wl if rank == 0 else wl.scaled(seed=wl.seed + 1000 * rank)


def max_over_ranks(value, world, device="cpu"):
    """The largest ``value`` over all ranks (every rank gets it); the identity at world 1."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch, world, ms_per_step):
    """Whole-job tokens/s: every rank decodes ``batch`` requests per step of ``ms_per_step``."""
    return batch * world / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------- bytes
def algorithmic_bytes(wl, lens_after, counts):
    """Bytes each kernel must move (inputs read once, outputs written once)."""
    B, Hq, H, D, Dv = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.head_dim_v
    n = [math.ceil(L / PAGE) for L in lens_after]
    cand = sum(max(x - 1, 0) for x in n)
    summary_row = 2 * D * 2  # min + max, bf16
    b = {}
    # append: read k_new/v_new, write the K/V rows, read+write the summary rows
    b["append"] = B * H * ((D + Dv) * 2 * 2 + summary_row * 2) if wl.append else 0
    # score: candidate summaries + their block-table entries + q + scores out
    b["score"] = cand * H * summary_row + cand * 4 + B * Hq * D * 2 + cand * H * 4
    # top-k: scores in, selection out
    b["topk"] = cand * H * 4 + B * H * (wl.topk_pages + 1) * 4
    # decode: the selected K and V page blocks + q + bf16 output (a latent row is key and value at once)
    sel_pages = int(sum(counts))
    row = D if wl.latent else D + Dv
    b["decode"] = sel_pages * PAGE * row * 2 + B * Hq * D * 2 + B * Hq * Dv * 2
    return b


# --------------------------------------------------------------------------- L2
class L2Flush:
    """Between timed steps: write a buffer of twice the L2 size (evicts the step's
    data), then read a second one of the same size, so that no dirty line of the
    written buffer is left for the next step's first kernel to write back."""

    def __init__(self, dev):
        import torch
        n = 2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)

    def __call__(self, value):
        self.w.fill_(value)
        self.r.sum()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle
def _oracle_worker(args):
    """One request through the fp64 oracle: state (page summaries) untimed, then the
    decode step (append + score + select + attend) timed."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle.quest as oq
    (k, v, n_tokens, H, D, Dv, q, k_new, v_new, topk, scale, sink, recent) = args
    import numpy as np
    req = oq.QuestRequest(k, v, np.arange(k.shape[0]), n_tokens, H, D, Dv, PAGE)
    t0 = time.perf_counter()
    if k_new is not None:
        req.append(k_new, v_new)
    req.decode(q, topk, scale, sink_tokens=sink, recent_tokens=recent)
    return time.perf_counter() - t0


def _sample_for_oracle(x, requests, sink=0, recent=0):
    items = []
    wl = x.workload
    for b in requests:
        n = x.pages_per_request[b]
        idx = x.block_table[b, :n].long()
        k = x.k_cache[idx].cpu().share_memory_()
        v = None if x.v_cache is None else x.v_cache[idx].cpu().share_memory_()
        items.append((k, v, x.seq_lens[b], wl.num_kv_heads, wl.head_dim, wl.head_dim_v, x.q[b].cpu(),
                      None if x.k_new is None else x.k_new[b].cpu(),
                      None if x.v_new is None else x.v_new[b].cpu(), wl.topk_pages, 1.0 / math.sqrt(wl.head_dim),
                      sink, recent))
    return items


def _pool_times(worker, items, cores):
    """Per-item single-core seconds of ``worker`` over ``items``, one process per core (spawn)."""
    import torch.multiprocessing as mp
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    workers = min(cores, len(items))
    with mp.get_context("spawn").Pool(workers) as pool:
        return pool.map(worker, items), workers


def cpu_oracle_throughput(x, n_requests=None, cores=None, sink=0, recent=0):
    """tokens/s of the oracle over a sample of requests, one process per core (spawn)."""
    cores = cores or len(os.sched_getaffinity(0))
    wl = x.workload
    n_requests = n_requests or min(wl.batch, max(2, 2 * cores))
    reqs = list(range(n_requests))
    items = _sample_for_oracle(x, reqs, sink, recent)
    times, workers = _pool_times(_oracle_worker, items, cores)
    busy = sum(times)  # seconds of single-core oracle work
    value = len(items) / (busy / workers)  # requests (= tokens) per second on `workers` cores
    what = "append + score + select + attend" if x.k_new is not None else "score + select + attend"
    return {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle",
            "sample": f"{len(items)} of the {wl.batch} requests (one decode token each; contexts "
                      f"{[x.seq_lens[b] for b in reqs]}), {what} timed per request, "
                      f"page summaries prebuilt untimed; {busy:.1f} s of single-core work"}


def _snapkv_oracle_worker(args):
    """One (request, KV head) pair of a SnapKV eviction through the fp64 oracle, timed:
    window probabilities and row log-sum-exps, column scores, pooling, the kept positions,
    then the kept K and V rows gathered."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    import oracle.snapkv as osk
    (k, v, n, qg, W, pool, keep, scale, sink, recent) = args
    t0 = time.perf_counter()
    res = osk.snapkv_head(qg, k, np.arange(k.shape[0]), 0, n, W, pool, keep, scale, PAGE, sink=sink, recent=recent)
    osk.compact_rows(k, np.arange(k.shape[0]), 0, res["kept"], PAGE)
    osk.compact_rows(v, np.arange(k.shape[0]), 0, res["kept"], PAGE)
    return time.perf_counter() - t0


def snapkv_cpu_baseline(x, cores=None, n_pairs=None):
    """Evictions (requests) per second of the oracle over a sample of (request, KV head) pairs."""
    cores = cores or len(os.sched_getaffinity(0))
    wl = x.workload
    H, G = wl.num_kv_heads, wl.group
    pairs = [(b, h) for b in range(wl.batch) for h in range(H)][:n_pairs or min(wl.batch * H, cores)]
    items = []
    for b, h in pairs:
        n = x.prompt_lens[b]
        idx = x.src_block_table[b, :x.src_pages_per_request[b]].long()
        k = x.k_cache[idx][:, h:h + 1].cpu().share_memory_()
        v = x.v_cache[idx][:, h:h + 1].cpu().share_memory_()
        items.append((k, v, n, x.q_window[b, :, h * G:(h + 1) * G, :].cpu(), wl.window, wl.pool_kernel,
                      wl.keep_topk, 1.0 / math.sqrt(wl.head_dim), wl.keep_sink, wl.recent))
    times, workers = _pool_times(_snapkv_oracle_worker, items, cores)
    busy = sum(times)
    pairs_per_s = len(items) / (busy / workers)
    return {"value": pairs_per_s / H, "unit": "requests/s", "cores": workers, "kind": "oracle",
            "sample": f"{len(items)} of the {wl.batch * H} (request, KV head) pairs ({wl.batch} prompts of "
                      f"{x.prompt_lens[0]} tokens): scores, pooling, selection and the gather of the kept rows "
                      f"timed per pair, requests/s = pairs/s / {H} KV heads; {busy:.1f} s of single-core work"}


# --------------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    import sparse_decode_attention_quest_gb300 as se
    from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
    from synth import make_quest_decode_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = rank_workload(_workload(), rank)
    x = make_quest_decode_inputs(wl, device=dev, poison_tail=False)
    max_len = max(x.seq_lens_after)
    step = QuestDecodeStep(x.k_cache, x.v_cache, new_summary(x.k_cache), x.block_table, wl.num_q_heads,
                           wl.topk_pages, max_len)
    before = torch.tensor(x.seq_lens, dtype=torch.int32, device=dev)
    after = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    step.build_summaries(before)
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)

    def one_step(ev=None):
        step.run(x.q, after, x.k_new, x.v_new, before, stream=stream, events=ev)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush(1.0)
            one_step()
    torch.cuda.synchronize()
    assert se.se_read_device_error() == 0

    K = args.steps
    sampler = ClockSampler(local_rank)
    sampler.start()
    # (1) Eager steps with an event between every kernel: the per-kernel spans.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush(float(i))
            one_step(evs[i][:4])
            evs[i][4].record(stream)
    torch.cuda.synchronize()
    spans = {"append": [], "score": [], "topk": [], "decode": []}
    eager_ms = []
    for e in evs:
        spans["append"].append(e[0].elapsed_time(e[1]))
        spans["score"].append(e[1].elapsed_time(e[2]))
        spans["topk"].append(e[2].elapsed_time(e[3]))
        spans["decode"].append(e[3].elapsed_time(e[4]))
        eager_ms.append(e[0].elapsed_time(e[4]))

    # (2) The headline: the same step captured once in a CUDA graph and replayed,
    # as a serving loop runs it; L2 flushed between replays, outside the events.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        step.run(x.q, after, x.k_new, x.v_new, before, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush(1.0)
            graph.replay()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush(float(i))
            pairs[i][0].record(stream)
            graph.replay()
            pairs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in pairs), world, dev)
    ms_per_step = total_ms / K
    assert se.se_read_device_error() == 0
    counts = step.counts.cpu().flatten().tolist()
    abytes = algorithmic_bytes(wl, x.seq_lens_after, counts)
    step_bytes = sum(abytes.values())
    peak, peak_kind = _peaks()
    kernels = {}
    for name, v in spans.items():
        ms = statistics.mean(v)
        gbs = abytes[name] / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
        kernels[name] = {"ms": round(ms, 5), "algorithmic_bytes": abytes[name], "gbs": round(gbs, 1),
                         "frac_of_measured_hbm": round(gbs / peak, 4)}
    dom = max(("score", "decode"), key=lambda k: kernels[k]["ms"])
    traffic = _profile_traffic(dom)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, step, x, before, after, stream, flush, dev)

    result = {
        "metric": METRIC, "value": job_throughput(wl.batch, world, ms_per_step), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "data": "synthetic (seeded N(0,1) bf16 keys/values/queries, 4 outlier key channels x8 per KV head)",
        "config": _config(wl, {"parallelism": f"replicas x{world} (each GPU decodes its own batch)",
                               "timing": "step captured in a CUDA graph, replayed; per-kernel spans from an "
                                         "eager pass with events between the kernels"}),
        "eager_ms_per_step": statistics.mean(eager_ms),
        "hbm": {"step_algorithmic_bytes": step_bytes, "step_gbs": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                "frac_of_8tbs": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                "frac_of_measured": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["gbs"], "peak": peak, "unit": "GB/s",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)" if peak_kind ==
                     "measured" else "fallback 6.8 TB/s",
                     "frac": round(kernels[dom]["gbs"] / peak, 4), "traffic": traffic},
        "kernels": kernels,
        "gpu_launches": K * step.launches_per_step(),
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_extra:
        result["extra_workloads"] = {
            "qwen3_30b_a3b_quest_b32_128k_fixed": _fixed_128k_extra(args, dev, flush, stream),
            "snapkv_prefill_b4_32k": _snapkv_extra(args, dev, flush, stream),
            "snapkv_aime_b4_32k": _snapkv_extra(args, dev, flush, stream, _snapkv_wl("SNAPKV_AIME_32K")),
            "snapkv_agent_b4_32k": _snapkv_extra(args, dev, flush, stream, _snapkv_wl("SNAPKV_AGENT_32K")),
            "snapkv_periodic_evict_aime_b4": _periodic_evict_extra(args, dev, flush, stream),
            "tiny_quest_b1_g4_4k": _quest_extra(args, dev, flush, stream, _snapkv_wl("TINY_QUEST_4K"),
                                                cpu_requests=1),
            "qwen3_4b_quest_b8_32k": _quest_extra(args, dev, flush, stream, _snapkv_wl("QWEN3_4B_QUEST_32K"),
                                                  cpu_requests=8),
            "tiny_quest_b1_g4_4k_fused": _quest_extra(args, dev, flush, stream, _snapkv_wl("TINY_QUEST_4K"),
                                                      fused=True),
            "qwen3_4b_quest_b8_32k_fused": _quest_extra(args, dev, flush, stream, _snapkv_wl("QWEN3_4B_QUEST_32K"),
                                                        fused=True),
            "qwen3_30b_a3b_quest_b32_128k_fused": _quest_extra(args, dev, flush, stream, wl, fused=True),
            "mla_glm_quest_b64_32k": _mla_extra(args, dev, flush, stream),
            "qwen3_30b_a3b_quest_sink64_recent512_b32_128k": _windows_extra(args, dev, flush, stream)}
    if rank == 0 and not args.no_cpu_baseline:
        try:
            result["cpu_baseline"] = cpu_oracle_throughput(x, cores=args.cpu_cores)
        except Exception as exc:  # reported, never silently replaced
            result["cpu_baseline"] = {"error": repr(exc)}
    return result


def _profile_traffic(kernel):
    """DRAM traffic per launch from the committed ncu summary, if it matches the current source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        src = os.path.join(ROOT, "sparse_decode_attention_quest_gb300", "csrc", rec["source"])
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if digest != rec["source_sha256_16"]:
            return None
        return rec["bytes_per_launch_full_size"]
    except Exception:
        return None


def _snapkv_extra(args, dev, flush, stream, wl=None, cpu_baseline=True):
    """SnapKV eviction at the end of a 32K prefill (4 requests, 32 q / 8 kv heads): one
    se_snapkv_score_and_compact_windowed call per step (window scores on the tensor cores,
    pool + top-k with the workload's keep windows, compaction), timed with events; L2
    flushed between steps."""
    import torch
    import sparse_decode_attention_quest_gb300 as se
    from synth import SNAPKV_PREFILL_32K, make_snapkv_inputs
    wl = SNAPKV_PREFILL_32K if wl is None else wl
    x = make_snapkv_inputs(wl, device=dev, poison_tail=False)
    B, H, W, G = wl.batch, wl.num_kv_heads, wl.window, wl.group
    max_len = max(x.prompt_lens)
    src = se.paged_kv(x.k_cache, x.v_cache, None)
    lens = torch.tensor(x.prompt_lens, dtype=torch.int32, device=dev)
    dk = torch.empty((x.dst_num_pages, H, 16, 128), dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dst = se.paged_kv(dk, dv, None)
    kept = torch.empty((B, H, wl.keep_sink + wl.keep_topk + wl.recent), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H), dtype=torch.int32, device=dev)
    ws = torch.empty(se.se_snapkv_workspace_size(B, H, W, max_len), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(wl.head_dim)

    def call():
        se.se_snapkv_score_and_compact_windowed(src, x.q_window, x.src_block_table, lens, max_len, wl.pool_kernel,
                                                wl.keep_topk, wl.keep_sink, wl.recent, scale, dst,
                                                x.dst_block_table, kept, cnt, ws, stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            flush(1.0)
            call()
    n = max(5, args.steps // 20)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            flush(float(i))
            pairs[i][0].record(stream)
            call()
            pairs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    kbytes = sum(x.prompt_lens) * H * 128 * 2                  # the prompt keys
    kept_rows = int(cnt.sum().item())
    gather = kept_rows * 256 * 2 * 2                           # K and V rows read and written
    flops = 2 * sum(x.prompt_lens) * H * (W * G) * 128 * 2     # two passes of the window x prompt QK^T
    peak_hbm, _ = _peaks()
    try:
        peak_tf = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        peak_tf = 1900.0
    cpu = None
    if cpu_baseline and not args.no_cpu_baseline:
        try:
            cpu = snapkv_cpu_baseline(x, cores=args.cpu_cores)
        except Exception as exc:  # reported, never silently replaced
            cpu = {"error": repr(exc)}
    return {"ms_per_call": ms, "steps": n, "requests_per_s": B / (ms * 1e-3), "cpu_baseline": cpu,
            "settings": {"window": W, "pool_kernel": wl.pool_kernel, "sink": wl.keep_sink, "recent": wl.recent,
                         "selected": wl.keep_topk, "kept_per_pair": int(cnt[0, 0].item())},
            "keys_read_bytes_per_pass": kbytes, "gather_bytes": gather,
            "hbm_gbs_two_key_passes": round((2 * kbytes + gather) / (ms * 1e-3) / 1e9, 1),
            "tensor_tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "tensor_frac_of_measured_bf16": round(flops / (ms * 1e-3) / 1e12 / peak_tf, 4)}


def _quest_extra(args, dev, flush, stream, wl, sink=0, recent=0, fused=False, cpu_requests=None):
    """One Quest decode step of workload ``wl`` (append if the workload appends, score, top-k
    with the keep windows ``sink``/``recent``, decode), captured in a CUDA graph and replayed
    (L2 flushed between replays); per-kernel spans from an eager pass. ``fused``: the step as
    one se_quest_fused_step launch (its span is the whole step)."""
    import torch
    import sparse_decode_attention_quest_gb300 as se
    from sparse_decode_attention_quest_gb300.pipeline import QuestDecodeStep, new_summary
    from synth import make_quest_decode_inputs
    x = make_quest_decode_inputs(wl, device=dev, poison_tail=False)
    max_len = max(x.seq_lens_after)
    step = QuestDecodeStep(x.k_cache, x.v_cache, new_summary(x.k_cache), x.block_table, wl.num_q_heads,
                           wl.topk_pages, max_len, head_dim_v=wl.head_dim_v, sink_tokens=sink, recent_tokens=recent)
    before = torch.tensor(x.seq_lens, dtype=torch.int32, device=dev)
    after = torch.tensor(x.seq_lens_after, dtype=torch.int32, device=dev)
    step.build_summaries(before)
    if fused:
        def run(ev=None):
            if ev is not None:
                for e in ev[:3]:
                    e.record(stream)
            if wl.append:
                step.run_fused(x.q, after, x.k_new, x.v_new, stream=stream)
            else:
                step.run_fused(x.q, after, stream=stream)
            if ev is not None:
                ev[3].record(stream)
    elif wl.append:
        run = lambda ev=None: step.run(x.q, after, x.k_new, x.v_new, before, stream=stream, events=ev)
    else:
        run = lambda ev=None: step.run(x.q, after, stream=stream, events=ev)
    n = max(5, args.steps // 10)
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush(1.0)
            run()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            flush(float(i))
            run(evs[i][:4])
            evs[i][4].record(stream)
    torch.cuda.synchronize()
    spans = {k: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
             for j, k in ((0, "append"), (1, "score"), (2, "topk"), (3, "decode"))}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        run()
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush(1.0)
            graph.replay()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            flush(float(i))
            pairs[i][0].record(stream)
            graph.replay()
            pairs[i][1].record(stream)
    torch.cuda.synchronize()
    assert se.se_read_device_error() == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    abytes = algorithmic_bytes(wl, x.seq_lens_after, step.counts.cpu().flatten().tolist())
    peak, _ = _peaks()
    step_bytes = sum(abytes.values())
    if fused:
        # events 0-2 are recorded before the one launch and event 3 after it: its span is
        # the third interval (the one the four-kernel step names "topk")
        spans = {"fused_step": spans["topk"]}
        abytes = {"fused_step": step_bytes}
    kern = {k: {"ms": round(v, 5), "algorithmic_bytes": abytes[k],
                "gbs": round(abytes[k] / (v * 1e-3) / 1e9, 1) if v > 0 else 0.0,
                "frac_of_measured_hbm": round(abytes[k] / (v * 1e-3) / 1e9 / peak, 4) if v > 0 else 0.0}
            for k, v in spans.items() if abytes[k] > 0}
    # QK^T over head_dim and PV over head_dim_v for every selected token and query head
    G = wl.num_q_heads // wl.num_kv_heads
    flops = 2 * int(step.counts.sum().item()) * PAGE * G * (wl.head_dim + wl.head_dim_v)
    dk = "fused_step" if fused else "decode"
    kern[dk]["tflops"] = round(flops / (spans[dk] * 1e-3) / 1e12, 1)
    cpu = None
    if cpu_requests and not args.no_cpu_baseline:
        try:
            cpu = cpu_oracle_throughput(x, n_requests=min(wl.batch, cpu_requests), cores=args.cpu_cores, sink=sink,
                                        recent=recent)
        except Exception as exc:  # reported, never silently replaced
            cpu = {"error": repr(exc)}
    return {"ms_per_step": ms, "steps": n, "tokens_per_s": wl.batch / (ms * 1e-3), "cpu_baseline": cpu,
            "step_gbs": round(step_bytes / (ms * 1e-3) / 1e9, 1),
            "step_frac_of_measured_hbm": round(step_bytes / (ms * 1e-3) / 1e9 / peak, 4), "kernels": kern,
            "kept_pages_per_kv_head": round(float(step.counts.float().mean().item()), 2),
            "shape": {"workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
                      "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "head_dim_v": wl.head_dim_v,
                      "context": [wl.context_min, wl.context_max], "topk_pages": wl.topk_pages,
                      "sink_tokens": sink, "recent_tokens": recent, "append": wl.append},
            "launches_per_step": 1 if fused else step.launches_per_step(wl.append)}


def _mla_extra(args, dev, flush, stream):
    """Quest decode over a latent cache: GLM-4.7-Flash-like MLA shape (64 query heads sharing
    one 576-dim latent row, value = its first 512 dims), 64 requests at 32K, a 2,048-token
    budget."""
    from synth import MLA_GLM_QUEST_32K
    wl = MLA_GLM_QUEST_32K if _BATCH_OVERRIDE is None else MLA_GLM_QUEST_32K.scaled(batch=_BATCH_OVERRIDE)
    return _quest_extra(args, dev, flush, stream, wl, cpu_requests=16)


def _windows_extra(args, dev, flush, stream):
    """The 128K workload with the decode-time keep windows of the throughput runs: sink 64,
    recent 512, 1,472 selected tokens (92 pages), 2,048 kept in total."""
    from synth import QWEN3_30B_A3B_QUEST_128K
    return _quest_extra(args, dev, flush, stream, QWEN3_30B_A3B_QUEST_128K.scaled(topk_pages=92), 64, 512,
                        cpu_requests=16)


def _fixed_128k_extra(args, dev, flush, stream):
    """The 128K workload with every request at exactly 131,072 tokens after the append
    (131,071 before it): 8,192 pages per request, 8,191 candidates per KV head."""
    from synth import QWEN3_30B_A3B_QUEST_128K
    wl = QWEN3_30B_A3B_QUEST_128K.scaled(name="qwen3_30b_a3b_quest_b32_128k_fixed", context_min=131071,
                                         context_max=131071)
    return _quest_extra(args, dev, flush, stream, wl, cpu_requests=16)


def _periodic_evict_extra(args, dev, flush, stream):
    """Decode-time SnapKV eviction with the AIME-run settings (Table 10: window 16, sink 16,
    recent 64, 4,096 selected, every 1,024 decode steps): one eviction over the compacted
    4,176 positions plus the 1,024 appended since the last one, and its cost spread over the
    1,024 decode steps of a period."""
    from synth import SNAPKV_AIME_32K
    period = 1024
    n = SNAPKV_AIME_32K.keep_sink + SNAPKV_AIME_32K.keep_topk + SNAPKV_AIME_32K.recent + period
    r = _snapkv_extra(args, dev, flush, stream,
                      SNAPKV_AIME_32K.scaled(name="snapkv_periodic_aime_b4", prompt_min=n, prompt_max=n),
                      cpu_baseline=False)
    r["period_decode_steps"] = period
    r["positions_before_eviction"] = n
    r["amortized_us_per_decode_step"] = round(r["ms_per_call"] * 1e3 / period, 4)
    return r


def _snapkv_wl(name):
    """A workload of the synth package by name."""
    import synth
    return getattr(synth, name)


def _e2e(args, step, x, before, after, stream, flush, dev):
    """The step as a server runs it: the step's inputs (q, k_new, v_new and both lengths)
    packed in one pinned host buffer and copied to the device in one transfer, the step
    through the library, the output copied back to pinned host memory. The upload
    (se_copy_async), the four C-ABI calls and the download (se_copy_async) are recorded
    once with se_capture_begin / se_capture_end and replayed with one se_graph_launch per
    step. Timed too: the copies made by torch around a replay of the four recorded calls
    (``split_ms_per_step``), and the four calls made live every step
    (``calls_ms_per_step``)."""
    import torch

    import sparse_decode_attention_quest_gb300 as se
    wl = x.workload
    parts = [x.q, x.k_new, x.v_new, before, after]
    offs, size = [], 0
    for t in parts:  # each part 16-byte aligned inside the buffer
        offs.append(size)
        size += (t.numel() * t.element_size() + 15) // 16 * 16
    h_buf = torch.empty(size, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(size, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        h_buf[o:o + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        views.append(d_buf[o:o + nb].view(t.dtype).view(t.shape))
    d_q, d_kn, d_vn, d_before, d_after = views
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = size
    d2h = h_out.numel() * h_out.element_size()

    def live(s):
        step.run(d_q, d_after, d_kn, d_vn, d_before, stream=s)

    se.se_capture_begin(stream)
    se.se_copy_async(d_buf, h_buf, stream)
    live(stream)
    se.se_copy_async(h_out, step.out, stream)
    graph_io = se.se_capture_end(stream)
    se.se_capture_begin(stream)
    live(stream)
    graph = se.se_capture_end(stream)

    def e2e_step(mode, ev0=None, ev1=None):
        if mode == "one" and ev0 is None:
            graph_io.launch(stream)  # the whole step: one call
            return
        with torch.cuda.stream(stream):
            if ev0 is not None:
                ev0.record(stream)
            if mode == "one":
                graph_io.launch(stream)
            else:
                d_buf.copy_(h_buf, non_blocking=True)
                if mode == "split":
                    graph.launch(stream)
                else:
                    live(stream)
                h_out.copy_(step.out, non_blocking=True)
            if ev1 is not None:
                ev1.record(stream)

    def timed(mode):
        """Host wall clock per step (no events in the clocked region), then the
        same steps again with events around each for the stream time."""
        for _ in range(args.warmup):
            flush(1.0)
            e2e_step(mode)
        torch.cuda.synchronize()
        n = max(10, args.steps // 4)
        host_ms = []
        for i in range(n):
            with torch.cuda.stream(stream):
                flush(float(i))
            stream.synchronize()  # the flush is done before the clock starts
            t0 = time.perf_counter()
            e2e_step(mode)
            stream.synchronize()  # the output is in host memory
            host_ms.append((time.perf_counter() - t0) * 1e3)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            with torch.cuda.stream(stream):
                flush(float(i))
            e2e_step(mode, *pairs[i])
        torch.cuda.synchronize()
        return n, statistics.mean(host_ms), statistics.mean(a.elapsed_time(b) for a, b in pairs)

    n, ms, stream_ms = timed("one")
    _, split_ms, split_stream_ms = timed("split")
    _, calls_ms, calls_stream_ms = timed("calls")
    graph_io.destroy()
    graph.destroy()
    return {"value": wl.batch / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "host wall clock per step: from before the step's launch (the upload first) to the return of "
                      "a stream synchronize after the download of the output (launches, copies and kernels "
                      "included; the L2 flush before it excluded); stream_ms_per_step: CUDA events around the "
                      "same steps in a second pass",
            "stream_ms_per_step": stream_ms,
            "split_ms_per_step": split_ms, "split_stream_ms_per_step": split_stream_ms,
            "calls_ms_per_step": calls_ms, "calls_stream_ms_per_step": calls_stream_ms,
            "path": "pinned host q/k_new/v_new/lengths (one packed buffer) -> device with se_copy_async, the step's "
                    "four C-ABI calls, output -> pinned host with se_copy_async, all recorded once "
                    "(se_capture_begin / se_capture_end) and replayed with one se_graph_launch per step; "
                    "split_ms_per_step: torch copies around a replay of the four recorded calls; "
                    "calls_ms_per_step: torch copies around the four calls made live"}


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 CPU oracle as the reference arm: each step decodes a bounded sample of
    the same workload's requests on the host cores."""
    import torch
    from synth import make_quest_decode_inputs
    wl = _workload()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = make_quest_decode_inputs(wl, device=dev, poison_tail=False)
    cores = args.cpu_cores or len(os.sched_getaffinity(0))
    per_step = []
    for i in range(args.warmup + args.steps):
        r = cpu_oracle_throughput(x, n_requests=min(wl.batch, cores), cores=cores)
        if i >= args.warmup:
            per_step.append(r)
    value = statistics.mean(r["value"] for r in per_step)
    ms = wl.batch / value * 1e3
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(wl, {"parallelism": "host cores"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": per_step[0]["cores"], "kind": "oracle",
                             "sample": per_step[0]["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary SnapKV measurement")
    ap.add_argument("--snapkv-only", action="store_true", help="only the SnapKV measurement (for profiler captures)")
    ap.add_argument("--mla-only", action="store_true", help="only the latent-cache measurement (for profiler captures)")
    ap.add_argument("--cpu-cores", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller batch (the 128K or, with --mla-only / --snapkv-only, the latent or SnapKV workload) "
                         "for profiler captures only")
    args = ap.parse_args()
    global _BATCH_OVERRIDE
    _BATCH_OVERRIDE = args.batch
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.snapkv_only or args.mla_only:
        args.no_cpu_baseline = True
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.snapkv_only:  # profiler captures of the SnapKV kernels alone (never the reported metric)
        import torch
        dev = torch.device("cuda", local_rank)
        flush = L2Flush(dev)
        from synth import SNAPKV_PREFILL_32K
        wl = SNAPKV_PREFILL_32K if args.batch is None else SNAPKV_PREFILL_32K.scaled(batch=args.batch)
        print(json.dumps({wl.name: _snapkv_extra(args, dev, flush, torch.cuda.Stream(dev), wl, cpu_baseline=False)}))
        return
    if args.mla_only:  # profiler captures of the latent-cache kernels alone (never the reported metric)
        import torch
        dev = torch.device("cuda", local_rank)
        flush = L2Flush(dev)
        print(json.dumps({"mla_glm_quest_b64_32k": _mla_extra(args, dev, flush, torch.cuda.Stream(dev))}))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
