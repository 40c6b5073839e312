"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every entry point include/wide.h declares; host-side helpers behave."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wide.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wide_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def libwide():
    from group_masked_gemm_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for fn in ("wide_reorder_masks", "wide_gemm_mn_gate_up", "wide_gemm_k_down",
               "wide_proj_mn", "wide_proj_k"):
        assert fn in names


def test_library_exports_every_declared_symbol(libwide):
    for name in _declared():
        assert hasattr(libwide, name), name


def test_host_only_entry_points(libwide):
    libwide.wide_status_string.restype = ctypes.c_char_p
    libwide.wide_status_string.argtypes = [ctypes.c_int]
    assert libwide.wide_status_string(0) == b"WIDE_OK"
    assert libwide.wide_status_string(5) == b"WIDE_ERR_TIMEOUT"
    assert libwide.wide_status_string(99) == b"WIDE_ERR_UNKNOWN"
    assert libwide.wide_version() >= 10000
    libwide.wide_gemm_k_workspace_size.restype = ctypes.c_size_t
    # prefill reduces in TMEM; the optional workspace splits the tiles of a last
    # wave that is at most half full: 2048 tiles on 152 SMs leave 72, cut in 2
    assert libwide.wide_gemm_k_workspace_size(16384, 14336, 4096, 128) == 72 * 2 * 128 * 256 * 4
    assert libwide.wide_gemm_k_workspace_size(2048, 1024, 4096, 128) == 0  # last wave 104 of 152
    tile = 128 * 256 * 4  # one fp32 share of a 128-token x 256-column tile
    # 10 token tiles x 16 = 160 tiles: a last wave of 8, cut into min(4, 152 // 8) = 4 shares
    assert libwide.wide_gemm_k_workspace_size(1200, 2048, 4096, 128) == 8 * 4 * tile
    assert libwide.wide_gemm_k_workspace_size(1280, 4096, 4096, 512) == 8 * 4 * tile
    # 192 tiles: a last wave of 40, 152 // 40 = 3 shares
    assert libwide.wide_gemm_k_workspace_size(1536, 1024, 4096, 128) == 40 * 3 * tile
    # a single group cannot be shared out
    assert libwide.wide_gemm_k_workspace_size(1200, 128, 4096, 128) == 0
    # fewer tiles than SMs: the required split workspace [splits, T, N], as before
    ws_short = libwide.wide_gemm_k_workspace_size(1000, 1024, 768, 128)
    assert ws_short > 0 and ws_short % (1000 * 768 * 4) == 0
    # decode: fp32 partial sums of the split reduction dimension, [splits, T, N]
    ws16 = libwide.wide_gemm_k_workspace_size(16, 14336, 4096, 128)
    assert ws16 > 0 and ws16 % (16 * 4096 * 4) == 0
    libwide.wide_reorder_workspace_size.restype = ctypes.c_size_t
    # the cooperative reorder (barrier word, ballots and tile offsets per (tile,
    # group)) is requested where it measured faster: few groups or long columns
    assert libwide.wide_reorder_workspace_size(16384, 112) == 0
    assert libwide.wide_reorder_workspace_size(16384, 8) == 16 + 128 * 8 * 20
    assert libwide.wide_reorder_workspace_size(4096, 8) == 0
    assert libwide.wide_reorder_workspace_size(65536, 112) == 16 + 512 * 112 * 20
    # one-launch router + reorder: barrier word, then per (128-token tile, group)
    # four 32-bit ballots and one tile offset; none for decode (T <= 16)
    libwide.wide_route_and_reorder_workspace_size.restype = ctypes.c_size_t
    assert libwide.wide_route_and_reorder_workspace_size(16384, 112) == 16 + 128 * 112 * 20
    assert libwide.wide_route_and_reorder_workspace_size(300, 13) == 16 + 3 * 13 * 20
    assert libwide.wide_route_and_reorder_workspace_size(16, 112) == 0


def test_argument_errors_are_reported_before_any_launch(libwide):
    """Null / misaligned pointers and bad shapes return status codes on the
    host; these calls never reach the GPU (none is present here)."""
    L = libwide
    p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.wide_reorder_masks.argtypes = [p, i, i, p, p, p, sz, p]
    L.wide_gemm_mn_gate_up.argtypes = [p, p, p, p, p, p, i, i, i, i, p, p]
    L.wide_gemm_k_down.argtypes = [p, p, p, p, p, i, i, i, i, p, p, sz, p]
    L.wide_proj_mn.argtypes = [p, p, p, p, p, i, i, i, i, p, p]
    good = p(4096 * 16)
    odd = p(4096 * 16 + 2)
    assert L.wide_reorder_masks(None, 64, 8, good, good, None, 0, None) == 1
    assert L.wide_reorder_masks(good, 0, 8, good, good, None, 0, None) == 1
    assert L.wide_reorder_masks(odd, 64, 8, good, good, None, 0, None) == 1
    # G not in {64,128,256,512}: 32 is a legal tile size but not implemented
    assert L.wide_gemm_mn_gate_up(good, good, good, good, good, good, 64, 256, 1024, 32,
                                  good, None) == 2
    assert L.wide_gemm_mn_gate_up(good, good, good, good, good, good, 64, 256, 1000, 128,
                                  good, None) == 1          # d_ffn not a multiple of 64
    assert L.wide_gemm_mn_gate_up(good, good, good, good, None, None, 64, 256, 1024, 128,
                                  good, None) == 1          # prefill needs perm/counts
    assert L.wide_gemm_mn_gate_up(good, odd, good, good, good, good, 64, 256, 1024, 128,
                                  good, None) == 1          # misaligned weight
    assert L.wide_gemm_k_down(good, good, good, good, good, 64, 1024, 250, 128, good,
                              None, 0, None) == 1            # d_model not a multiple of 64
    assert L.wide_proj_mn(good, good, good, good, good, 64, 4096, 4096, 96, good, None) == 1
    # one group spanning the whole grouped dimension (N_G = 1) passes validation
    # when it is a multiple of 256; with no GPU here the call then fails at launch
    assert L.wide_proj_mn(good, good, good, good, good, 64, 4096, 1536, 1536, good, None) == 4
    assert L.wide_proj_mn(good, good, good, good, good, 64, 4096, 640, 640, good, None) == 1
    assert L.wide_gemm_k_down(good, good, good, good, good, 64, 2048, 256, 2048, good,
                              None, 0, None) == 4
    assert L.wide_gemm_k_down(good, good, good, good, good, 64, 2048, 256, 1024, good,
                              None, 0, None) == 2            # G = 1024 < K = 2048: tile size, not implemented


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from group_masked_gemm_gb300 import ops
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()
