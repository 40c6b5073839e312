"""GPU parity: the CUDA path (through the C ABI, via the ctypes binding)
against the CPU oracle on the same seeded inputs.

Reorder outputs are compared bit-exactly; GEMM outputs within
max|y - y_ref| <= 2e-2 * RMS(y_ref); inactive MN blocks must be exact zeros
and every output element must be written (outputs start as NaN garbage).
"""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import assert_close, inactive_columns, mask_dev, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()
    torch.cuda.init()


def _nan_like(shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def _bits_dev(rng, shape, scale=1.0):
    return syn.bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


# ----------------------------------------------------------------- reorder ---

@pytest.mark.parametrize("coop", [True, False])  # one cooperative launch / one block per column
@pytest.mark.parametrize("T,ng,keep,seed", [
    (1, 1, 0.5, 0), (7, 3, 0.5, 1), (64, 8, 0.5, 2), (300, 28, 0.3, 3),
    (4096, 64, 0.5, 4), (16384, 112, 0.5, 5), (40000, 5, 0.5, 6), (129, 224, 0.1, 7),
    (1000, 3, 0.0, 8), (1000, 3, 1.0, 9), (65537, 2, 0.7, 10), (200000, 3, 0.5, 11)])
def test_reorder_bit_exact(T, ng, keep, seed, coop):
    mask = syn.random_mask(T, ng, keep, seed)
    mask[::7] *= 255  # any nonzero byte is active
    perm, counts = ops.reorder_masks(mask_dev(mask), coop=coop)
    torch.cuda.synchronize()
    p_ref, c_ref = oracle.reorder(mask)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(perm.cpu().numpy(), p_ref)


# ------------------------------------------------------------------ GEMM-MN ---

@pytest.mark.parametrize("T,D,F,G,keep", [
    (64, 256, 1024, 128, 0.5), (300, 512, 1024, 64, 0.5), (300, 512, 1024, 128, 0.5),
    (517, 256, 2048, 256, 0.4), (517, 256, 2048, 512, 0.6), (200, 320, 1024, 128, 1.0),
    (200, 320, 1024, 128, 0.0), (1000, 448, 1536, 128, 0.08), (129, 1024, 512, 128, 0.5)])
def test_gate_up_parity(T, D, F, G, keep):
    inp = syn.ffn_inputs(T, D, F, G, seed=T + G, keep=keep)
    m = mask_dev(inp.mask)
    perm, counts = ops.reorder_masks(m)
    H = _nan_like((T, F))
    ops.gemm_mn_gate_up(to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), m, perm, counts, G, out=H)
    ops.device_status()
    Hg = to_f64(H)
    assert not np.isnan(Hg).any(), "every element of H must be written"
    assert (Hg[inactive_columns(inp.mask, G)] == 0).all()
    assert_close(Hg, oracle.gate_up(inp.X, inp.Wg, inp.Wu, inp.mask, G), "gate_up")


@pytest.mark.parametrize("T,K,N,G,keep", [
    (300, 384, 1024, 64, 0.5), (300, 384, 1024, 128, 0.5), (257, 256, 2048, 256, 0.5),
    (257, 256, 2048, 512, 0.34), (100, 512, 512, 512, 1.0), (640, 192, 4096, 512, 0.66)])
def test_proj_mn_parity(T, K, N, G, keep):
    rng = np.random.default_rng(T * 7 + G)
    X = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, N // G)) < keep).astype(np.uint8)
    m = mask_dev(mask)
    perm, counts = ops.reorder_masks(m)
    Y = _nan_like((T, N))
    ops.proj_mn(to_dev(X), to_dev(W), m, perm, counts, G, out=Y)
    ops.device_status()
    Yg = to_f64(Y)
    assert not np.isnan(Yg).any()
    assert (Yg[inactive_columns(mask, G)] == 0).all()
    assert_close(Yg, oracle.proj_mn(X, W, mask, G), "proj_mn")


# ------------------------------------------------------------------- GEMM-K ---

@pytest.mark.parametrize("T,K,N,G,keep", [
    (64, 1024, 256, 128, 0.5), (300, 1024, 256, 64, 0.5), (300, 2048, 320, 128, 0.5),
    (517, 2048, 384, 256, 0.4), (517, 2048, 256, 512, 0.6), (200, 1024, 512, 128, 1.0),
    (200, 1024, 512, 128, 0.0), (1000, 1536, 256, 128, 0.08),
    # G = 512 (o_proj-sized groups), ragged T, all-active and all-inactive
    (300, 2048, 512, 512, 1.0), (300, 2048, 512, 512, 0.0), (1029, 4096, 768, 512, 0.34),
    # short batches: the groups are split over CTAs with fp32 partials
    (33, 14336, 4096, 128, 0.5), (200, 2048, 1024, 128, 0.05),
    # wide outputs (256-column tiles over grids that fill the SMs), ragged T
    (2048, 1024, 4096, 128, 0.5), (2000, 2048, 4096, 128, 0.3), (1900, 1024, 4096, 256, 0.5),
    (1280, 4096, 4096, 512, 0.34), (1536, 1024, 4096, 128, 1.0), (1536, 1024, 4096, 128, 0.0),
    (2304, 512, 8192, 64, 0.02)])
def test_gemm_k_parity(T, K, N, G, keep):
    rng = np.random.default_rng(T * 3 + G)
    A = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, K // G)) < keep).astype(np.uint8)
    # values inside inactive groups must be ignored: make them huge garbage
    garbage = _bits_dev(rng, (T, K), 1e4)
    A_dirty = np.where(inactive_columns(mask, G), garbage, A)
    m = mask_dev(mask)
    perm, counts = ops.reorder_masks(m)
    Y = _nan_like((T, N))
    ops.gemm_k_down(to_dev(A_dirty), to_dev(W), m, perm, counts, G, out=Y)
    ops.device_status()
    Yg = to_f64(Y)
    assert not np.isnan(Yg).any()
    ref = oracle.proj_k(A, W, mask, G)
    assert_close(Yg, ref, "gemm_k")
    assert (Yg[mask.sum(1) == 0] == 0).all()


@pytest.mark.parametrize("T,K,N,G,keep", [
    # last waves of 8 (ragged last token tile), 40 and 8 tiles: shares of 4, 3, 4
    (1200, 2048, 4096, 128, 0.5), (1536, 1024, 4096, 128, 0.3), (1280, 4096, 4096, 512, 0.34)])
def test_gemm_k_tail_split(T, K, N, G, keep):
    """Tiles of a mostly idle last wave split into shares of their live groups
    (with the optional workspace) and reduced whole (without it): both match
    the oracle."""
    rng = np.random.default_rng(T + K + G)
    A = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, K // G)) < keep).astype(np.uint8)
    m = mask_dev(mask)
    perm, counts = ops.reorder_masks(m)
    assert ops.gemm_k_workspace_size(T, K, N, G) > 0  # the split applies on this device
    ref = oracle.proj_k(A, W, mask, G)
    for ws in (None, torch.empty((16,), dtype=torch.uint8, device="cuda")):
        Y = _nan_like((T, N))
        ops.gemm_k_down(to_dev(A), to_dev(W), m, perm, counts, G, out=Y, ws=ws)
        ops.device_status()
        Yg = to_f64(Y)
        assert not np.isnan(Yg).any()
        assert_close(Yg, ref, "gemm_k tail" if ws is None else "gemm_k whole")


def test_proj_k_matches_gemm_k_down():
    rng = np.random.default_rng(42)
    T, K, N, G = 333, 4096, 512, 512
    A = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, K // G)) < 0.34).astype(np.uint8)
    m = mask_dev(mask)
    Y = ops.proj_k(to_dev(A), to_dev(W), m, None, None, G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.proj_k(A, W, mask, G), "proj_k")


# ---------------------------------------------------------------- whole FFN ---

@pytest.mark.parametrize("T,D,F,G,keep", [(64, 256, 1024, 128, 0.5), (700, 512, 2048, 128, 0.5),
                                          (300, 256, 1024, 64, 0.3), (300, 256, 2048, 256, 0.7)])
def test_ffn_parity(T, D, F, G, keep):
    inp = syn.ffn_inputs(T, D, F, G, seed=11, keep=keep)
    Y = ops.ffn_forward(to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), to_dev(inp.Wd),
                        mask_dev(inp.mask), G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, G), "ffn")


def test_tiny_config_ffn():
    inp = syn.tiny_ffn()
    Y = ops.ffn_forward(to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), to_dev(inp.Wd),
                        mask_dev(inp.mask), inp.G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, inp.G), "tiny")


# ------------------------------------------- M-axis depth (n_groups = 1) ---

@pytest.mark.parametrize("T,K,N,keep", [(300, 512, 768, 0.5), (129, 256, 1024, 0.7), (7, 1024, 512, 0.5),
                                        (2, 768, 256, 1.0), (40, 512, 1536, 0.0)])
def test_whole_width_group_mn(T, K, N, keep):
    """G = N: each token runs the whole projection or nothing (App. B, N_G = 1)."""
    rng = np.random.default_rng(T + N)
    X = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    W2 = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, 1)) < keep).astype(np.uint8)
    m = mask_dev(mask)
    perm, counts = ops.reorder_masks(m)
    Y = _nan_like((T, N))
    ops.proj_mn(to_dev(X), to_dev(W), m, perm, counts, N, out=Y)
    H = _nan_like((T, N))
    ops.gemm_mn_gate_up(to_dev(X), to_dev(W), to_dev(W2), m, perm, counts, N, out=H)
    ops.device_status()
    Yg, Hg = to_f64(Y), to_f64(H)
    assert not np.isnan(Yg).any() and not np.isnan(Hg).any()
    assert (Yg[mask[:, 0] == 0] == 0).all() and (Hg[mask[:, 0] == 0] == 0).all()
    assert_close(Yg, oracle.proj_mn(X, W, mask, N), "proj_mn G=N")
    assert_close(Hg, oracle.gate_up(X, W, W2, mask, N), "gate_up G=N")


@pytest.mark.parametrize("T,K,N,keep", [(300, 768, 384, 0.5), (1029, 1024, 256, 0.3), (5, 1536, 512, 0.6),
                                        (16, 512, 320, 0.5)])
def test_whole_width_group_k(T, K, N, keep):
    """G = K: each token's whole reduction is kept or dropped."""
    rng = np.random.default_rng(T + K)
    A = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, 1)) < keep).astype(np.uint8)
    m = mask_dev(mask)
    perm, counts = ops.reorder_masks(m)
    Y = _nan_like((T, N))
    ops.proj_k(to_dev(A), to_dev(W), m, perm, counts, K, out=Y)
    ops.device_status()
    Yg = to_f64(Y)
    assert not np.isnan(Yg).any()
    assert (Yg[mask[:, 0] == 0] == 0).all()
    assert_close(Yg, oracle.proj_k(A, W, mask, K), "proj_k G=K")


def test_whole_width_group_ffn():
    """The whole FFN with one group per token (dynamic depth on the FFN)."""
    inp = syn.ffn_inputs(500, 256, 1024, 1024, seed=11, keep=0.5)
    Y = ops.ffn_forward(to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), to_dev(inp.Wd),
                        mask_dev(inp.mask), inp.G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, inp.G), "ffn G=F")


# ------------------------------------------------------------------- decode ---

@pytest.mark.parametrize("T", [1, 4, 16])
@pytest.mark.parametrize("G", [64, 128, 256, 512])
def test_decode_parity(T, G):
    inp = syn.llama8b_decode(T, G)
    m = mask_dev(inp.mask)
    H = _nan_like((T, inp.F))
    ops.gemm_mn_gate_up(to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), m, None, None, G, out=H)
    Y = _nan_like((T, inp.D))
    Hin = syn.bf16_bits(np.random.default_rng(T).standard_normal((T, inp.F), dtype=np.float32))
    ops.gemm_k_down(to_dev(Hin), to_dev(inp.Wd), m, None, None, G, out=Y)
    ops.device_status()
    Hg = to_f64(H)
    assert (Hg[inactive_columns(inp.mask, G)] == 0).all()
    assert_close(Hg, oracle.gate_up(inp.X, inp.Wg, inp.Wu, inp.mask, G), "decode gate_up")
    assert_close(to_f64(Y), oracle.proj_k(Hin, inp.Wd, inp.mask, G), "decode down")


def test_decode_ragged_and_empty():
    rng = np.random.default_rng(3)
    T, K, N, G = 5, 320, 640, 64
    X = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, N // G)) < 0.5).astype(np.uint8)
    mask[2] = 0  # a token with no active group
    m = mask_dev(mask)
    Y = ops.proj_mn(to_dev(X), to_dev(W), m, None, None, G)
    Z = ops.proj_k(to_dev(_bits_dev(rng, (T, N))), to_dev(_bits_dev(rng, (K, N), 0.02)), m, None,
                   None, G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.proj_mn(X, W, mask, G), "decode proj_mn")
    assert (to_f64(Z)[2] == 0).all()


@pytest.mark.parametrize("T,K,N,G,keep", [
    (2, 2560, 384, 64, 0.5),      # 40 groups (not a multiple of 32), 3 output tiles
    (7, 4096, 1024, 512, 0.3),    # ragged token box, o_proj-sized groups
    (13, 1536, 256, 128, 1.0),    # every group live
    (16, 2048, 512, 256, 0.0),    # no group live: every split writes zeros
    (1, 14336, 4096, 128, 0.05),  # fewer live groups than splits
])
def test_decode_k_split_edges(T, K, N, G, keep):
    """Decode GEMM-K: live groups dealt in equal shares over the splits, fp32
    partials summed in split order."""
    rng = np.random.default_rng(T * 7 + K)
    A = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, K // G)) < keep).astype(np.uint8)
    Y = _nan_like((T, N))
    ops.proj_k(to_dev(A), to_dev(W), mask_dev(mask), None, None, G, out=Y)
    Y2 = _nan_like((T, N))
    ops.proj_k(to_dev(A), to_dev(W), mask_dev(mask), None, None, G, out=Y2)
    ops.device_status()
    assert torch.equal(Y, Y2)  # deterministic
    assert_close(to_f64(Y), oracle.proj_k(A, W, mask, G), "decode proj_k")


@pytest.mark.parametrize("T,K,N,G", [(5, 4096, 1024, 128), (8, 2048, 768, 256)])
def test_decode_mn_tensor_core_sizes(T, K, N, G):
    """Decode GEMM-MN above 4 tokens (tensor-core kernel), plain and gate/up."""
    rng = np.random.default_rng(T + N)
    X = _bits_dev(rng, (T, K))
    W = _bits_dev(rng, (N, K), 0.02)
    W2 = _bits_dev(rng, (N, K), 0.02)
    mask = (rng.random((T, N // G)) < 0.5).astype(np.uint8)
    Y = ops.proj_mn(to_dev(X), to_dev(W), mask_dev(mask), None, None, G)
    H = ops.gemm_mn_gate_up(to_dev(X), to_dev(W), to_dev(W2), mask_dev(mask), None, None, G)
    ops.device_status()
    assert_close(to_f64(Y), oracle.proj_mn(X, W, mask, G), "decode proj_mn")
    assert_close(to_f64(H), oracle.gate_up(X, W, W2, mask, G), "decode gate_up")


# ------------------------------------------------ determinism and CUDA graphs ---

def test_deterministic_and_graph_capturable():
    inp = syn.ffn_inputs(1000, 512, 2048, 128, seed=5, keep=0.5)
    X, Wg, Wu, Wd = (to_dev(a) for a in (inp.X, inp.Wg, inp.Wu, inp.Wd))
    m = mask_dev(inp.mask)
    H = torch.empty((inp.T, inp.F), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((inp.T, inp.D), dtype=torch.bfloat16, device="cuda")
    perm = torch.empty((inp.n_groups, inp.T), dtype=torch.int32, device="cuda")
    counts = torch.empty((inp.n_groups,), dtype=torch.int32, device="cuda")
    ops.ffn_forward(X, Wg, Wu, Wd, m, inp.G, H=H, Y=Y, perm=perm, counts=counts)
    torch.cuda.synchronize()
    y_eager = Y.clone()
    Y.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ops.ffn_forward(X, Wg, Wu, Wd, m, inp.G, H=H, Y=Y, perm=perm, counts=counts)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), y_eager.view(torch.int16))
    ops.device_status()
