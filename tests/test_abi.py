"""The C-ABI library without a GPU: it loads, exports every symbol include/*.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

import sparse_decode_attention_quest_gb300 as se

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3
FAKE = 0x7f0000000000  # 16-byte aligned, never dereferenced on the host


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names |= set(re.findall(r"^SE_API\s+[\w\s\*]+?\b(se_\w+)\s*\(", open(h).read(), flags=re.M))
    return names


def test_every_declared_symbol_is_exported(se_lib):
    declared = _declared()
    assert len(declared) >= 11
    for name in declared:
        assert hasattr(se_lib, name), name
    assert declared == set(se.exported_symbols())


def test_status_strings(se_lib):
    assert se_lib.se_status_string(0) == b"SE_OK"
    assert se_lib.se_status_string(3) == b"SE_ERR_WORKSPACE"
    assert se_lib.se_status_string(99) == b"SE_ERR_UNKNOWN"


def _kv(**over):
    f = dict(k=FAKE, v=FAKE + 4096, summary=FAKE + 8192, num_pages=64, num_kv_heads=4, page_size=16,
             head_dim=128, head_dim_v=128, row_stride_k=128, row_stride_v=128)
    f.update(over)
    return se.SEPagedKV(**f)


def _build(kv, bt=FAKE, bt_stride=64, lens=FAKE, batch=2, max_len=1000):
    return se_lib_global.se_quest_build_summaries(ctypes.byref(kv) if kv is not None else None, bt, bt_stride,
                                                  lens, batch, max_len, None)


se_lib_global = None


@pytest.fixture(autouse=True)
def _bind(se_lib):
    global se_lib_global
    se_lib_global = se_lib


@pytest.mark.parametrize("kv,expect", [
    (None, INVALID),
    (_kv(k=None), INVALID),
    (_kv(summary=None), INVALID),
    (_kv(page_size=8), INVALID),
    (_kv(k=FAKE + 8), INVALID),            # misaligned
    (_kv(num_kv_heads=0), INVALID),
    (_kv(row_stride_k=64), INVALID),       # row shorter than head_dim
    (_kv(head_dim=64, head_dim_v=64, row_stride_k=64, row_stride_v=64), UNSUPPORTED),
    (_kv(num_pages=1 << 27), UNSUPPORTED),  # 2^31 token rows
])
def test_cache_view_validation(kv, expect):
    assert _build(kv) == expect


def test_batch_validation():
    assert _build(_kv(), batch=-1) == INVALID
    assert _build(_kv(), max_len=-5) == INVALID
    assert _build(_kv(), bt_stride=10, max_len=1000) == INVALID  # needs ceil(1000/16) = 63
    assert _build(_kv(), bt=None) == INVALID


def test_score_validation(se_lib):
    f = se_lib.se_quest_score_pages
    kv = _kv()
    assert f(ctypes.byref(kv), FAKE, 30, FAKE, 64, FAKE, 2, 1000, FAKE, 63, None) == INVALID  # 30 % 4
    assert f(ctypes.byref(kv), FAKE, 32, FAKE, 64, FAKE, 2, 1000, FAKE, 10, None) == INVALID  # score stride
    assert f(ctypes.byref(kv), FAKE + 2, 32, FAKE, 64, FAKE, 2, 1000, FAKE, 63, None) == INVALID
    big = _kv(num_kv_heads=16)  # scoring keeps 1..8 KV heads of d 128 in registers
    assert f(ctypes.byref(big), FAKE, 32, FAKE, 64, FAKE, 2, 1000, FAKE, 63, None) == UNSUPPORTED


def test_score_workspace_validation(se_lib):
    # the group sums P and N: batch x KV heads x 2 x head_dim floats
    assert se_lib.se_quest_score_workspace_size(2, 4, 128) == 2 * 4 * 2 * 128 * 4 + 16
    assert se_lib.se_quest_score_workspace_size(64, 1, 576) == 64 * 2 * 576 * 4 + 16
    assert se_lib.se_quest_score_workspace_size(-1, 4, 128) == 0
    f = se_lib.se_quest_score_pages_ws
    kv = _kv()
    need = se_lib.se_quest_score_workspace_size(2, 4, 128)
    args = lambda ws=FAKE, n=need, hq=32: (ctypes.byref(kv), FAKE, hq, FAKE, 64, FAKE, 2, 1000, FAKE, 63, ws, n,
                                           None)
    assert f(*args(n=need - 1)) == WORKSPACE
    assert f(*args(ws=None)) == INVALID
    assert f(*args(ws=FAKE + 4)) == INVALID                 # misaligned
    assert f(*args(hq=30)) == INVALID                       # the checks of se_quest_score_pages follow
    assert f(None, FAKE, 32, FAKE, 64, FAKE, 2, 1000, FAKE, 63, FAKE, need, None) == INVALID


def test_topk_validation(se_lib):
    f = se_lib.se_quest_topk_pages
    assert f(FAKE, 63, FAKE, 2, 4, 1000, 0, FAKE, FAKE, 8, None) == INVALID        # k = 0
    assert f(FAKE, 63, FAKE, 2, 4, 1000, 8, FAKE, FAKE, 8, None) == INVALID        # stride < k + 1
    assert f(FAKE, 10, FAKE, 2, 4, 1000, 8, FAKE, FAKE, 9, None) == INVALID        # score stride
    assert f(FAKE, 70000, FAKE, 2, 4, 16 * 60000, 8, FAKE, FAKE, 9, None) == UNSUPPORTED


def test_select_workspace(se_lib):
    need = se_lib.se_quest_select_workspace_size(2, 4, 1000)
    assert need == 2 * 4 * 63 * 4
    kv = _kv()
    st = se_lib.se_quest_select_pages(ctypes.byref(kv), FAKE, 32, FAKE, 64, FAKE, 2, 1000, 8, FAKE, FAKE, 9,
                                      FAKE, need - 1, None)
    assert st == WORKSPACE


def test_decode_validation(se_lib):
    f = se_lib.se_sparse_paged_decode
    kv = _kv()
    args = lambda hq=32, scale=0.1, q=FAKE: (ctypes.byref(kv), q, hq, FAKE, 64, FAKE, 2, FAKE, FAKE, 9, scale,
                                             FAKE, None, FAKE, 1 << 20, None)
    assert f(*args(hq=30)) == INVALID
    assert f(*args(q=FAKE + 4)) == INVALID
    assert f(*args(scale=float("nan"))) == INVALID
    assert f(*args(hq=4 * 32)) == UNSUPPORTED  # 32 query heads per KV head
    wide = _kv(head_dim=576, head_dim_v=512, row_stride_k=576, row_stride_v=576, num_kv_heads=1)
    assert f(ctypes.byref(wide), FAKE, 8, FAKE, 64, FAKE, 2, FAKE, FAKE, 9, 0.1, FAKE, None, FAKE, 1 << 20,
             None) == UNSUPPORTED  # latent cache with 8 query heads
    assert f(ctypes.byref(wide), FAKE, 128, FAKE, 64, FAKE, 2, FAKE, FAKE, 9, 0.1, FAKE, None, FAKE, 1 << 30,
             None) == UNSUPPORTED  # latent cache with 128 query heads
    split = _kv(head_dim=576, head_dim_v=512, row_stride_k=576, row_stride_v=576, num_kv_heads=1)
    split.v = FAKE + 4096
    assert f(ctypes.byref(split), FAKE, 64, FAKE, 64, FAKE, 2, FAKE, FAKE, 9, 0.1, FAKE, None, FAKE, 1 << 30,
             None) == INVALID  # a latent cache reads the value from the key row: v must be k


def test_decode_workspace_size(se_lib):
    # slices of >= 16 pages: an item of 257 pages spans at most 18; (Dv + 1) floats per (row, slice)
    # plus one int per row for the per-item slice counts
    assert se_lib.se_sparse_decode_workspace_size(32, 32, 4, 128, 257) == 32 * 32 * 18 * 129 * 4 + 32 * 32 * 4
    # latent cache (one KV head, 512-wide value): 129 selected pages span at most 10 slices; one int per request
    assert se_lib.se_sparse_decode_workspace_size(64, 64, 1, 512, 129) == 64 * 64 * 10 * 513 * 4 + 64 * 4
    assert se_lib.se_sparse_decode_workspace_size(-1, 32, 4, 128, 257) == 0


def test_update_validation(se_lib):
    f = se_lib.se_quest_update_summaries
    kv = _kv()
    assert f(ctypes.byref(kv), FAKE, None, FAKE, 64, FAKE, 2, None) == INVALID   # v_new missing
    lat = _kv(v=FAKE)
    assert f(ctypes.byref(lat), FAKE, FAKE, FAKE, 64, FAKE, 2, None) == INVALID  # latent takes no v_new
    assert f(ctypes.byref(kv), FAKE + 2, FAKE, FAKE, 64, FAKE, 2, None) == INVALID


def test_failure_detail(se_lib):
    assert _build(_kv(page_size=8)) == INVALID
    assert b"page_size" in se_lib.se_last_error_detail()


def test_update_ex_validation(se_lib):
    f = se_lib.se_quest_update_summaries_ex
    kv = _kv()
    assert f(ctypes.byref(kv), FAKE, FAKE, FAKE, 64, FAKE, 2, 0x2, None) == INVALID   # unknown flag
    assert b"flags" in se_lib.se_last_error_detail()
    assert f(ctypes.byref(kv), FAKE, None, FAKE, 64, FAKE, 2, se.APPEND_OVERLAP_PREVIOUS, None) == INVALID  # v_new


def test_a_c_caller_compiles_against_the_header_and_links(se_lib, tmp_path):
    """A plain C program (tests/c_abi_check.c) includes include/sparse_engine.h,
    links the library and checks host-only paths: status strings, rejection
    before any launch, workspace sizes."""
    import os
    import shutil
    import subprocess
    from sparse_decode_attention_quest_gb300 import build as b
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib_dir = os.path.dirname(b.lib_path())
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "c_abi_check.c"), "-o", exe, "-L", lib_dir, "-lsparse_engine",
                    "-Wl,-rpath," + lib_dir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_replayable_step_calls_reject_missing_handles(se_lib):
    # host checks only: a NULL stream (the legacy default stream cannot be
    # recorded), a NULL graph handle; destroying NULL is a no-op
    assert se_lib.se_capture_begin(None) == INVALID
    h = ctypes.c_void_p(None)
    assert se_lib.se_capture_end(None, ctypes.byref(h)) == INVALID
    assert se_lib.se_capture_end(ctypes.c_void_p(FAKE), None) == INVALID
    assert se_lib.se_graph_launch(None, None) == INVALID
    se_lib.se_graph_destroy(None)


def test_copy_async_host_checks(se_lib):
    # an empty copy is a no-op (no CUDA call); a NULL buffer with bytes to copy is refused
    assert se_lib.se_copy_async(None, None, 0, None) == 0
    assert se_lib.se_copy_async(None, ctypes.c_void_p(FAKE), 16, None) == INVALID
    assert se_lib.se_copy_async(ctypes.c_void_p(FAKE), None, 16, None) == INVALID
