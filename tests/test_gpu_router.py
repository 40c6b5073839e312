"""GPU parity of the router (Sec. 3.1 "Routing Components", Eq. 4-5) and of
router + mask reordering, against the fp64 C oracle.

The decision argmax_c R[t,g,c] is an integer decided by floating point.  The
kernel decides on its own fp32 logits, so:
  - its logits must match the oracle's within the fp32 accumulation error;
  - its mask must equal the decision on its own logits, bit for bit;
  - it may differ from the oracle's mask only where the oracle's two logits
    are closer than the logit error just measured (a near-tie, where either
    class is a correct argmax).
perm/counts after routing are integer work and must be bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import mask_dev, to_dev

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-4  # max |R_gpu - R_ref| / RMS(R_ref): fp32 accumulation over d_model


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


def _router_case(T, D, r, ng, seed):
    rng = np.random.default_rng(seed)
    X = syn.bf16_bits(rng.standard_normal((T, D), dtype=np.float32))
    W1 = syn.bf16_bits(rng.standard_normal((r, D), dtype=np.float32) * np.float32(D ** -0.5))
    W2 = syn.bf16_bits(rng.standard_normal((2 * ng, r), dtype=np.float32) * np.float32(r ** -0.5))
    return X, W1, W2


def _check_router(mask_g, logits_g, logits_ref, mask_ref):
    rms = float(np.sqrt(np.mean(logits_ref ** 2)))
    err = float(np.max(np.abs(logits_g - logits_ref)))
    assert err <= LOGIT_TOL * rms, f"logit error {err / rms:.3g} x RMS"
    own = (logits_g[:, 0::2] >= logits_g[:, 1::2]).astype(np.uint8)
    np.testing.assert_array_equal(mask_g, own)  # decided on its own fp32 logits
    diff = mask_g != mask_ref
    margin = np.abs(logits_ref[:, 0::2] - logits_ref[:, 1::2])
    assert (margin[diff] <= 2 * err).all(), "a decision differs away from a near-tie"
    assert diff.mean() <= 1e-3
    return int(diff.sum())


@pytest.mark.parametrize("T,D,r,ng", [(64, 256, 16, 8), (300, 512, 32, 112), (1000, 4096, 32, 112),
                                      (129, 3072, 16, 64), (17, 1024, 64, 56), (50, 256, 32, 13),
                                      (1, 4096, 32, 112),
                                      # T <= 16: the decode path (one CUDA-core block per token)
                                      (4, 4096, 32, 8), (16, 4096, 32, 112), (7, 256, 16, 13),
                                      (3, 512, 64, 56)])
def test_router_parity(T, D, r, ng):
    X, W1, W2 = _router_case(T, D, r, ng, seed=T + D + r)
    mask_g, logits_g = ops.router_masks(to_dev(X), to_dev(W1), to_dev(W2), logits=True)
    ops.device_status()
    logits_ref, mask_ref = oracle.router(X, W1, W2)
    _check_router(mask_g.cpu().numpy(), logits_g.cpu().numpy().astype(np.float64), logits_ref, mask_ref)
    assert 0.2 < mask_ref.mean() < 0.8


@pytest.mark.parametrize("T,D,r,ng", [(2000, 1024, 32, 56), (16384, 4096, 32, 112), (300, 512, 16, 13),
                                      (129, 256, 64, 8), (40000, 512, 32, 112), (17, 1024, 32, 1024)])
def test_route_and_reorder_fused_matches_two_launches(T, D, r, ng):
    """The one-launch router + reorder (cooperative kernel, grid barriers) gives
    the mask of the router alone and the oracle's reorder of it, bit for bit.
    T = 40000 gives CTAs several tiles; ng = 13 and 1024 are not multiples of
    4; T = 129 and 17 leave a partial tile."""
    if 2 * ng * r * 2 > 64 * 1024:
        r = 16
    X, W1, W2 = _router_case(T, D, r, ng, seed=T + ng)
    Xd, W1d, W2d = to_dev(X), to_dev(W1), to_dev(W2)
    assert ops.route_and_reorder_workspace_size(T, ng) > 0
    mask_f, perm_f, counts_f = ops.route_and_reorder(Xd, W1d, W2d)
    mask_2, perm_2, counts_2 = ops.route_and_reorder(Xd, W1d, W2d, fused=False)
    ops.device_status()
    m = mask_f.cpu().numpy()
    np.testing.assert_array_equal(m, mask_2.cpu().numpy())
    perm_ref, counts_ref = oracle.reorder(m)
    np.testing.assert_array_equal(counts_f.cpu().numpy(), counts_ref)
    np.testing.assert_array_equal(perm_f.cpu().numpy(), perm_ref)
    np.testing.assert_array_equal(perm_2.cpu().numpy(), perm_ref)


def test_route_and_reorder_bit_exact():
    X, W1, W2 = _router_case(2000, 1024, 32, 56, seed=7)
    mask, perm, counts = ops.route_and_reorder(to_dev(X), to_dev(W1), to_dev(W2))
    mask_only = ops.router_masks(to_dev(X), to_dev(W1), to_dev(W2))
    ops.device_status()
    m = mask.cpu().numpy()
    np.testing.assert_array_equal(m, mask_only.cpu().numpy())
    perm_ref, counts_ref = oracle.reorder(m)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_ref)
    np.testing.assert_array_equal(counts.cpu().numpy(), counts_ref)
    logits_ref, mask_ref = oracle.router(X, W1, W2)
    assert (m != mask_ref).mean() <= 1e-3


@pytest.mark.parametrize("T", [200, 5])
def test_router_ties_execute(T):
    """Identical class rows give exactly equal logits: every group executes
    (tensor-core path and decode path)."""
    X, W1, W2 = _router_case(T, 512, 32, 24, seed=3)
    W2[1::2] = W2[0::2]
    mask_g, logits_g = ops.router_masks(to_dev(X), to_dev(W1), to_dev(W2), logits=True)
    ops.device_status()
    lg = logits_g.cpu().numpy()
    np.testing.assert_array_equal(lg[:, 0::2], lg[:, 1::2])
    assert mask_g.cpu().numpy().all()


def test_router_full_size_sampled_rows():
    """The 8B router shape (T = 16384, d_model 4096, r = 32, 112 FFN groups):
    every row on the GPU, 512 sampled rows against the oracle (rows are
    independent), and the routed mask drives the reorder bit-exactly."""
    T, D, r, ng = 16384, 4096, 32, 112
    X, W1, W2 = _router_case(T, D, r, ng, seed=44)
    mask, perm, counts = ops.route_and_reorder(to_dev(X), to_dev(W1), to_dev(W2))
    mask_g, logits_g = ops.router_masks(to_dev(X), to_dev(W1), to_dev(W2), logits=True)
    ops.device_status()
    m = mask.cpu().numpy()
    np.testing.assert_array_equal(m, mask_g.cpu().numpy())
    rows = syn.sample_rows(T, 512, 9)
    logits_ref, mask_ref = oracle.router(X[rows].copy(), W1, W2)
    _check_router(m[rows], logits_g.cpu().numpy()[rows].astype(np.float64), logits_ref, mask_ref)
    perm_ref, counts_ref = oracle.reorder(m)
    np.testing.assert_array_equal(counts.cpu().numpy(), counts_ref)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_ref)


def test_router_argument_errors():
    lib = ops.lib()
    X = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    W1 = torch.zeros((24, 256), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((16, 24), dtype=torch.bfloat16, device="cuda")
    mask = torch.zeros((8, 8), dtype=torch.uint8, device="cuda")
    st = lib.wide_router_masks(ops._ptr(X), ops._ptr(W1), ops._ptr(W2), 8, 256, 24, 8,
                               ops._ptr(mask), None, ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_INVALID_ARG"  # r must be a multiple of 16
    st = lib.wide_router_masks(ops._ptr(X), ops._ptr(W1), ops._ptr(W2), 8, 256, 128, 8,
                               ops._ptr(mask), None, ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_UNSUPPORTED"  # r = 128 is not implemented
