"""Python binding of libsparse_engine.so, the sm_103a sparse decode attention library.

The functions below carry the C ABI's names (include/sparse_engine.h) and do
argument marshalling only: they check dtypes, devices and contiguity of the
torch tensors that own the device memory, pass raw pointers and the current
CUDA stream to the library, and raise ``SparseEngineError`` on any non-OK
status. Every step of the computation runs in the library's CUDA kernels;
there is no CPU path. If the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "SparseEngineError", "SEPagedKV", "paged_kv", "load_library", "se_read_device_error",
    "se_quest_build_summaries", "se_quest_update_summaries", "se_quest_update_summaries_ex",
    "APPEND_OVERLAP_PREVIOUS", "se_quest_score_pages", "se_quest_score_workspace_size", "se_quest_score_pages_ws",
    "se_quest_topk_pages", "se_quest_topk_pages_windowed", "se_quest_kept_pages_max",
    "se_quest_select_workspace_size", "se_quest_select_pages", "se_quest_select_pages_windowed",
    "se_quest_fused_step",
    "se_sparse_decode_workspace_size", "se_sparse_decode_plan", "se_sparse_paged_decode",
    "se_sparse_paged_decode_noalloc", "se_snapkv_workspace_size", "se_snapkv_window_scores", "se_snapkv_select",
    "se_snapkv_compact", "se_snapkv_score_and_compact", "se_snapkv_select_windowed",
    "se_snapkv_score_and_compact_windowed", "se_debug_snapkv_wait_probe", "SEGraph", "se_capture_begin",
    "se_capture_end", "exported_symbols",
]

SE_OK = 0
DEVERR_PAGE_RANGE = 0x1
DEVERR_LENGTH = 0x2
DEVERR_WAIT_TIMEOUT = 0x4
APPEND_OVERLAP_PREVIOUS = 0x1  # se_quest_update_summaries_ex: may run alongside the previous kernel


class SparseEngineError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{detail} [status {status}]")
        self.status = status


class SEPagedKV(ctypes.Structure):
    """Mirror of se_paged_kv_t."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("summary", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32), ("row_stride_k", ctypes.c_int32),
                ("row_stride_v", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_F = ctypes.c_float
_Z = ctypes.c_size_t
_KV = ctypes.POINTER(SEPagedKV)

_SIGNATURES = {
    "se_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "se_last_error_detail": (ctypes.c_char_p, []),
    "se_read_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "se_quest_build_summaries": (ctypes.c_int, [_KV, _P, _I, _P, _I, _I, _P]),
    "se_quest_update_summaries": (ctypes.c_int, [_KV, _P, _P, _P, _I, _P, _I, _P]),
    "se_quest_update_summaries_ex": (ctypes.c_int, [_KV, _P, _P, _P, _I, _P, _I, ctypes.c_uint32, _P]),
    "se_quest_score_pages": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _I, _P, _I, _P]),
    "se_quest_score_workspace_size": (_Z, [_I, _I, _I]),
    "se_quest_score_pages_ws": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _I, _P, _I, _P, _Z, _P]),
    "se_quest_topk_pages": (ctypes.c_int, [_P, _I, _P, _I, _I, _I, _I, _P, _P, _I, _P]),
    "se_quest_topk_pages_windowed": (ctypes.c_int, [_P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P]),
    "se_quest_kept_pages_max": (ctypes.c_longlong, [_I, _I, _I]),
    "se_quest_select_workspace_size": (_Z, [_I, _I, _I]),
    "se_quest_select_pages": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _I, _I, _P, _P, _I, _P, _Z, _P]),
    "se_quest_select_pages_windowed": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P,
                                                      _Z, _P]),
    "se_quest_fused_step": (ctypes.c_int, [_KV, _P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P,
                                           _I, _P]),
    "se_sparse_decode_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "se_sparse_decode_plan": (ctypes.c_int, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I),
                                             ctypes.POINTER(_I)]),
    "se_sparse_paged_decode": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _P, _P, _I, _F, _P, _P, _P, _Z, _P]),
    "se_sparse_paged_decode_noalloc": (ctypes.c_int, [_KV, _P, _I, _P, _I, _P, _I, _P, _P, _I, _F, _P, _P, _P]),
    "se_snapkv_workspace_size": (_Z, [_I, _I, _I, _I]),
    "se_snapkv_window_scores": (ctypes.c_int, [_KV, _P, _I, _I, _P, _I, _P, _I, _I, _F, _P, _I, _P, _P, _Z, _P]),
    "se_snapkv_select": (ctypes.c_int, [_P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P]),
    "se_debug_snapkv_wait_probe": (ctypes.c_int, [ctypes.c_uint32]),
    "se_capture_begin": (ctypes.c_int, [_P]),
    "se_capture_end": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    "se_graph_launch": (ctypes.c_int, [_P, _P]),
    "se_graph_destroy": (None, [_P]),
    "se_copy_async": (ctypes.c_int, [_P, _P, _Z, _P]),
    "se_snapkv_select_windowed": (ctypes.c_int, [_P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P]),
    "se_snapkv_compact": (ctypes.c_int, [_KV, _P, _I, _P, _I, _KV, _P, _I, _P, _I, _P, _P]),
    "se_snapkv_score_and_compact": (ctypes.c_int, [_KV, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I, _F, _KV, _P, _I, _P,
                                                   _I, _P, _P, _Z, _P]),
    "se_snapkv_score_and_compact_windowed": (ctypes.c_int, [_KV, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F,
                                                            _KV, _P, _I, _P, _I, _P, _P, _Z, _P]),
}

_lib = None


def exported_symbols():
    return list(_SIGNATURES)


def load_library():
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with sparse_decode_attention_quest_gb300.build.build() "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int):
    if status != SE_OK:
        lib = load_library()
        raise SparseEngineError(status, lib.se_last_error_detail().decode())


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def paged_kv(k_cache: torch.Tensor, v_cache: Optional[torch.Tensor], summary: Optional[torch.Tensor],
             head_dim_v: Optional[int] = None) -> SEPagedKV:
    """se_paged_kv_t for bf16 caches [P][Hkv][16][row]. ``v_cache`` None = latent cache (v aliases k)."""
    _ptr(k_cache, torch.bfloat16, "k_cache")
    P, H, ps, row_k = k_cache.shape
    if v_cache is None:
        if head_dim_v is None:
            raise ValueError("a latent cache needs head_dim_v")
        v_ptr, row_v, dv = k_cache.data_ptr(), row_k, head_dim_v
    else:
        _ptr(v_cache, torch.bfloat16, "v_cache")
        v_ptr, row_v, dv = v_cache.data_ptr(), v_cache.shape[-1], v_cache.shape[-1]
    if summary is not None:
        _ptr(summary, torch.bfloat16, "summary")
    return SEPagedKV(k_cache.data_ptr(), v_ptr, None if summary is None else summary.data_ptr(),
                     P, H, ps, row_k, dv, row_k, row_v)


class SEGraph:
    """A recorded step (se_capture_begin ... se_capture_end): launch() replays it
    with se_graph_launch; the handle is freed with se_graph_destroy."""

    def __init__(self, handle: int):
        self._h = handle

    def launch(self, stream=None):
        if not self._h:
            raise ValueError("the recorded step has been destroyed")
        _check(load_library().se_graph_launch(self._h, _stream(stream)))

    def destroy(self):
        if self._h:
            load_library().se_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def se_capture_begin(stream=None):
    """Start recording the library calls made on ``stream`` (not the legacy default stream)."""
    _check(load_library().se_capture_begin(_stream(stream)))


def se_capture_end(stream=None) -> SEGraph:
    """End the recording on ``stream``; returns the recorded step."""
    h = ctypes.c_void_p(None)
    _check(load_library().se_capture_end(_stream(stream), ctypes.byref(h)))
    return SEGraph(h.value)


def _copy_ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name}: a host tensor must be in page-locked memory (pin_memory())")
    return t.data_ptr()


def se_copy_async(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """Copy ``src`` into ``dst`` (same number of bytes; device or pinned host memory)
    asynchronously on ``stream``; recordable between se_capture_begin and se_capture_end."""
    nb = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError("se_copy_async: dst and src differ in size")
    _check(load_library().se_copy_async(_copy_ptr(dst, "dst"), _copy_ptr(src, "src"), nb, _stream(stream)))


def se_read_device_error(clear: bool = True) -> int:
    lib = load_library()
    v = ctypes.c_uint32(0)
    _check(lib.se_read_device_error(ctypes.byref(v), int(clear)))
    return v.value


def se_quest_build_summaries(kv: SEPagedKV, block_table, seq_lens, max_seq_len: int, stream=None):
    lib = load_library()
    _check(lib.se_quest_build_summaries(ctypes.byref(kv), _ptr(block_table, torch.int32, "block_table"),
                                        block_table.shape[1], _ptr(seq_lens, torch.int32, "seq_lens"),
                                        seq_lens.shape[0], int(max_seq_len), _stream(stream)))


def se_quest_update_summaries(kv: SEPagedKV, k_new, v_new, block_table, seq_lens_before, stream=None):
    lib = load_library()
    _check(lib.se_quest_update_summaries(ctypes.byref(kv), _ptr(k_new, torch.bfloat16, "k_new"),
                                         _ptr(v_new, torch.bfloat16, "v_new"),
                                         _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                         _ptr(seq_lens_before, torch.int32, "seq_lens_before"),
                                         seq_lens_before.shape[0], _stream(stream)))


def se_quest_update_summaries_ex(kv: SEPagedKV, k_new, v_new, block_table, seq_lens_before, flags: int = 0,
                                 stream=None):
    lib = load_library()
    _check(lib.se_quest_update_summaries_ex(ctypes.byref(kv), _ptr(k_new, torch.bfloat16, "k_new"),
                                            _ptr(v_new, torch.bfloat16, "v_new"),
                                            _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                            _ptr(seq_lens_before, torch.int32, "seq_lens_before"),
                                            seq_lens_before.shape[0], int(flags), _stream(stream)))


def se_quest_score_pages(kv: SEPagedKV, q, block_table, seq_lens, max_seq_len: int, scores, stream=None):
    lib = load_library()
    _check(lib.se_quest_score_pages(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                    _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                    _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], int(max_seq_len),
                                    _ptr(scores, torch.float32, "scores"), scores.shape[-1], _stream(stream)))


def se_quest_score_workspace_size(batch: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load_library().se_quest_score_workspace_size(batch, num_kv_heads, head_dim))


def se_quest_score_pages_ws(kv: SEPagedKV, q, block_table, seq_lens, max_seq_len: int, scores, workspace,
                            stream=None):
    lib = load_library()
    _check(lib.se_quest_score_pages_ws(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                       _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                       _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], int(max_seq_len),
                                       _ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                       _ptr(workspace, torch.uint8, "workspace"),
                                       0 if workspace is None else workspace.numel(), _stream(stream)))


def se_quest_topk_pages(scores, seq_lens, num_kv_heads: int, max_seq_len: int, topk_pages: int, out_pages,
                        out_counts, stream=None):
    lib = load_library()
    _check(lib.se_quest_topk_pages(_ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                   _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], int(num_kv_heads),
                                   int(max_seq_len), int(topk_pages), _ptr(out_pages, torch.int32, "out_pages"),
                                   _ptr(out_counts, torch.int32, "out_counts"), out_pages.shape[-1],
                                   _stream(stream)))


def se_quest_topk_pages_windowed(scores, seq_lens, num_kv_heads: int, max_seq_len: int, topk_pages: int,
                                 sink_tokens: int, recent_tokens: int, out_pages, out_counts, stream=None):
    lib = load_library()
    _check(lib.se_quest_topk_pages_windowed(_ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                            _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0],
                                            int(num_kv_heads), int(max_seq_len), int(topk_pages), int(sink_tokens),
                                            int(recent_tokens), _ptr(out_pages, torch.int32, "out_pages"),
                                            _ptr(out_counts, torch.int32, "out_counts"), out_pages.shape[-1],
                                            _stream(stream)))


def se_quest_kept_pages_max(topk_pages: int, sink_tokens: int, recent_tokens: int) -> int:
    return int(load_library().se_quest_kept_pages_max(topk_pages, sink_tokens, recent_tokens))


def se_quest_select_workspace_size(batch: int, num_kv_heads: int, max_seq_len: int) -> int:
    return int(load_library().se_quest_select_workspace_size(batch, num_kv_heads, max_seq_len))


def se_quest_select_pages(kv: SEPagedKV, q, block_table, seq_lens, max_seq_len: int, topk_pages: int, out_pages,
                          out_counts, workspace, stream=None):
    lib = load_library()
    _check(lib.se_quest_select_pages(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                     _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                     _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], int(max_seq_len),
                                     int(topk_pages), _ptr(out_pages, torch.int32, "out_pages"),
                                     _ptr(out_counts, torch.int32, "out_counts"), out_pages.shape[-1],
                                     _ptr(workspace, torch.uint8, "workspace"),
                                     0 if workspace is None else workspace.numel(), _stream(stream)))


def se_quest_select_pages_windowed(kv: SEPagedKV, q, block_table, seq_lens, max_seq_len: int, topk_pages: int,
                                   sink_tokens: int, recent_tokens: int, out_pages, out_counts, workspace,
                                   stream=None):
    lib = load_library()
    _check(lib.se_quest_select_pages_windowed(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                              _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                              _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0],
                                              int(max_seq_len), int(topk_pages), int(sink_tokens),
                                              int(recent_tokens), _ptr(out_pages, torch.int32, "out_pages"),
                                              _ptr(out_counts, torch.int32, "out_counts"), out_pages.shape[-1],
                                              _ptr(workspace, torch.uint8, "workspace"),
                                              0 if workspace is None else workspace.numel(), _stream(stream)))


def se_quest_fused_step(kv: SEPagedKV, k_new, v_new, q, block_table, seq_lens, max_seq_len: int, topk_pages: int,
                        sink_tokens: int, recent_tokens: int, sm_scale: float, out, out_lse, sel_pages, sel_counts,
                        stream=None):
    lib = load_library()
    _check(lib.se_quest_fused_step(ctypes.byref(kv), _ptr(k_new, torch.bfloat16, "k_new"),
                                   _ptr(v_new, torch.bfloat16, "v_new"), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                   _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                   _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0], int(max_seq_len),
                                   int(topk_pages), int(sink_tokens), int(recent_tokens), float(sm_scale),
                                   _ptr(out, torch.bfloat16, "out"), _ptr(out_lse, torch.float32, "out_lse"),
                                   _ptr(sel_pages, torch.int32, "sel_pages"), _ptr(sel_counts, torch.int32, "sel_counts"),
                                   sel_pages.shape[-1], _stream(stream)))


def se_sparse_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim_v: int,
                                    sel_stride: int) -> int:
    return int(load_library().se_sparse_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim_v,
                                                              sel_stride))


def se_sparse_decode_plan(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, head_dim_v: int,
                          sel_stride: int):
    """(nsplit, pages_per_split, launches) of se_sparse_paged_decode on the current device."""
    lib = load_library()
    a, b, c = _I(0), _I(0), _I(0)
    _check(lib.se_sparse_decode_plan(batch, num_q_heads, num_kv_heads, head_dim, head_dim_v, sel_stride,
                                     ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def se_sparse_paged_decode(kv: SEPagedKV, q, block_table, seq_lens, sel_pages, sel_counts, sm_scale: float, out,
                           out_lse=None, workspace=None, stream=None):
    lib = load_library()
    _check(lib.se_sparse_paged_decode(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                      _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                      _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0],
                                      _ptr(sel_pages, torch.int32, "sel_pages"),
                                      _ptr(sel_counts, torch.int32, "sel_counts"), sel_pages.shape[-1],
                                      float(sm_scale), _ptr(out, torch.bfloat16, "out"),
                                      _ptr(out_lse, torch.float32, "out_lse"),
                                      _ptr(workspace, torch.uint8, "workspace"),
                                      0 if workspace is None else workspace.numel(), _stream(stream)))


def se_sparse_paged_decode_noalloc(kv: SEPagedKV, q, block_table, seq_lens, sel_pages, sel_counts, sm_scale: float,
                                   out, out_lse=None, stream=None):
    """se_sparse_paged_decode without a workspace, for callers that cannot allocate device memory:
    the split partials live in a fixed 8 MiB array inside the library (see the C header)."""
    lib = load_library()
    _check(lib.se_sparse_paged_decode_noalloc(ctypes.byref(kv), _ptr(q, torch.bfloat16, "q"), q.shape[1],
                                              _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                              _ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.shape[0],
                                              _ptr(sel_pages, torch.int32, "sel_pages"),
                                              _ptr(sel_counts, torch.int32, "sel_counts"), sel_pages.shape[-1],
                                              float(sm_scale), _ptr(out, torch.bfloat16, "out"),
                                              _ptr(out_lse, torch.float32, "out_lse"), _stream(stream)))


# ---------------------------------------------------------------- SnapKV
def se_snapkv_workspace_size(batch: int, num_kv_heads: int, window: int, max_prompt_len: int) -> int:
    return int(load_library().se_snapkv_workspace_size(batch, num_kv_heads, window, max_prompt_len))


def se_debug_snapkv_wait_probe(limit_us: int):
    """Test hook: the next SnapKV window-score launch of this thread waits for a count that
    no CTA reaches and gives up after ``limit_us`` (see the C header)."""
    _check(load_library().se_debug_snapkv_wait_probe(int(limit_us)))


def se_snapkv_window_scores(src: SEPagedKV, q_window, block_table, prompt_lens, max_prompt_len: int, sm_scale: float,
                            scores, row_lse=None, workspace=None, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_window_scores(ctypes.byref(src), _ptr(q_window, torch.bfloat16, "q_window"),
                                       q_window.shape[2], q_window.shape[1],
                                       _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
                                       _ptr(prompt_lens, torch.int32, "prompt_lens"), prompt_lens.shape[0],
                                       int(max_prompt_len), float(sm_scale), _ptr(scores, torch.float32, "scores"),
                                       scores.shape[-1], _ptr(row_lse, torch.float32, "row_lse"),
                                       _ptr(workspace, torch.uint8, "workspace"),
                                       0 if workspace is None else workspace.numel(), _stream(stream)))


def se_snapkv_select(scores, prompt_lens, num_kv_heads: int, window: int, max_prompt_len: int, pool_kernel: int,
                     keep_topk: int, kept_pos, kept_counts, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_select(_ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                _ptr(prompt_lens, torch.int32, "prompt_lens"), prompt_lens.shape[0], int(num_kv_heads),
                                int(window), int(max_prompt_len), int(pool_kernel), int(keep_topk),
                                _ptr(kept_pos, torch.int32, "kept_pos"), kept_pos.shape[-1],
                                _ptr(kept_counts, torch.int32, "kept_counts"), _stream(stream)))


def se_snapkv_select_windowed(scores, prompt_lens, num_kv_heads: int, window: int, max_prompt_len: int,
                              pool_kernel: int, keep_topk: int, sink_tokens: int, recent_tokens: int, kept_pos,
                              kept_counts, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_select_windowed(_ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                         _ptr(prompt_lens, torch.int32, "prompt_lens"), prompt_lens.shape[0],
                                         int(num_kv_heads), int(window), int(max_prompt_len), int(pool_kernel),
                                         int(keep_topk), int(sink_tokens), int(recent_tokens),
                                         _ptr(kept_pos, torch.int32, "kept_pos"), kept_pos.shape[-1],
                                         _ptr(kept_counts, torch.int32, "kept_counts"), _stream(stream)))


def se_snapkv_compact(src: SEPagedKV, src_block_table, prompt_lens, dst: SEPagedKV, dst_block_table, kept_pos,
                      kept_counts, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_compact(ctypes.byref(src), _ptr(src_block_table, torch.int32, "src_block_table"),
                                 src_block_table.shape[1], _ptr(prompt_lens, torch.int32, "prompt_lens"),
                                 prompt_lens.shape[0], ctypes.byref(dst),
                                 _ptr(dst_block_table, torch.int32, "dst_block_table"), dst_block_table.shape[1],
                                 _ptr(kept_pos, torch.int32, "kept_pos"), kept_pos.shape[-1],
                                 _ptr(kept_counts, torch.int32, "kept_counts"), _stream(stream)))


def se_snapkv_score_and_compact(src: SEPagedKV, q_window, src_block_table, prompt_lens, max_prompt_len: int,
                                pool_kernel: int, keep_topk: int, sm_scale: float, dst: SEPagedKV, dst_block_table,
                                kept_pos, kept_counts, workspace, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_score_and_compact(ctypes.byref(src), _ptr(q_window, torch.bfloat16, "q_window"),
                                           q_window.shape[2], q_window.shape[1],
                                           _ptr(src_block_table, torch.int32, "src_block_table"),
                                           src_block_table.shape[1], _ptr(prompt_lens, torch.int32, "prompt_lens"),
                                           prompt_lens.shape[0], int(max_prompt_len), int(pool_kernel),
                                           int(keep_topk), float(sm_scale), ctypes.byref(dst),
                                           _ptr(dst_block_table, torch.int32, "dst_block_table"),
                                           dst_block_table.shape[1], _ptr(kept_pos, torch.int32, "kept_pos"),
                                           kept_pos.shape[-1], _ptr(kept_counts, torch.int32, "kept_counts"),
                                           _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                           _stream(stream)))


def se_snapkv_score_and_compact_windowed(src: SEPagedKV, q_window, src_block_table, prompt_lens, max_prompt_len: int,
                                         pool_kernel: int, keep_topk: int, sink_tokens: int, recent_tokens: int,
                                         sm_scale: float, dst: SEPagedKV, dst_block_table, kept_pos, kept_counts,
                                         workspace, stream=None):
    lib = load_library()
    _check(lib.se_snapkv_score_and_compact_windowed(
        ctypes.byref(src), _ptr(q_window, torch.bfloat16, "q_window"), q_window.shape[2], q_window.shape[1],
        _ptr(src_block_table, torch.int32, "src_block_table"), src_block_table.shape[1],
        _ptr(prompt_lens, torch.int32, "prompt_lens"), prompt_lens.shape[0], int(max_prompt_len), int(pool_kernel),
        int(keep_topk), int(sink_tokens), int(recent_tokens), float(sm_scale), ctypes.byref(dst),
        _ptr(dst_block_table, torch.int32, "dst_block_table"), dst_block_table.shape[1],
        _ptr(kept_pos, torch.int32, "kept_pos"), kept_pos.shape[-1], _ptr(kept_counts, torch.int32, "kept_counts"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
