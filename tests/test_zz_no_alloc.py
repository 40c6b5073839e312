"""The allocation-free decode GEMM-K entry point (wide_gemm_k_decode_noalloc).

Some callers cannot call cudaMalloc at all -- a memory planner owns every
device allocation, or a plugin host hands the kernel no workspace.  For them
the library keeps the decode GEMM-K's fp32 partial sums in a fixed device
array of its own.  This test calls that entry point through the C ABI twice
in a row (the array keeps the previous call's contents, which must not leak
into the next result) and checks both outputs against the regular entry
point, which takes a caller-allocated workspace, within the parity tolerance
of the other GPU tests.  It lives in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import TOL, excess_err, mask_dev, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


@pytest.mark.parametrize("T,K,N,G", [(16, 14336, 4096, 128), (4, 4096, 4096, 512),
                                     (1, 2048, 512, 64), (7, 1024, 320, 256)])
def test_noalloc_matches_workspace_entry_point(T, K, N, G):
    rng = np.random.default_rng(T * 1000 + G)
    A = to_dev(syn.bf16_bits(rng.standard_normal((T, K), dtype=np.float32)))
    W = to_dev(syn.bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)))
    m1 = mask_dev((rng.random((T, K // G)) < 0.5).astype(np.uint8))
    m2 = mask_dev((rng.random((T, K // G)) < 0.3).astype(np.uint8))

    ref1 = ops.gemm_k_down(A, W, m1, None, None, G)   # caller workspace
    ref2 = ops.gemm_k_down(A, W, m2, None, None, G)
    y1 = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.gemm_k_decode_noalloc(A, W, m1, G, out=y1)    # two calls in a row,
    ops.gemm_k_decode_noalloc(A, W, m2, G, out=y2)    # different masks
    ops.device_status()

    for y, ref in ((y1, ref1), (y2, ref2)):
        yv, rv = to_f64(y), to_f64(ref)
        assert not np.isnan(yv).any()
        assert excess_err(yv, rv) <= TOL


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ops.lib()
    A = torch.zeros((16, 65536), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((4096, 65536), dtype=torch.bfloat16, device="cuda")
    mask = torch.zeros((16, 65536 // 128), dtype=torch.uint8, device="cuda")
    Y = torch.empty((16, 4096), dtype=torch.bfloat16, device="cuda")
    st = lib.wide_gemm_k_decode_noalloc(ops._ptr(A), ops._ptr(W), ops._ptr(mask), 16, 65536,
                                        4096, 128, ops._ptr(Y), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_WORKSPACE"
    st = lib.wide_gemm_k_decode_noalloc(ops._ptr(A), ops._ptr(W), ops._ptr(mask), 17, 65536,
                                        4096, 128, ops._ptr(Y), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_INVALID_ARG"
