"""GPU parity of routed decode attention (App. B "Implementation of
Attention", decoding; GQA-aligned groups of Sec. 3.1 Eq. 2) against the fp64
C oracle, within the floating-point tolerance of the other GPU tests."""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import assert_close, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


def _dev_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _case(B, Hq, Hk, d, L_max, lens, keep, seed):
    rng = np.random.default_rng(seed)
    Q = syn.bf16_bits(rng.standard_normal((B, Hq, d), dtype=np.float32))
    K = syn.bf16_bits(rng.standard_normal((B, Hk, L_max, d), dtype=np.float32))
    V = syn.bf16_bits(rng.standard_normal((B, Hk, L_max, d), dtype=np.float32))
    lens = np.asarray(lens, np.int32)
    mask = (rng.random((B, Hk)) < keep).astype(np.uint8)
    # nothing past lens[b], and nothing of an inactive group, may be read:
    # fill those parts of the cache with NaN bit patterns
    for b in range(B):
        K[b, :, lens[b]:] = 0x7FC0
        V[b, :, lens[b]:] = 0x7FC0
        for g in range(Hk):
            if mask[b, g] == 0:
                K[b, g] = 0x7FC0
                V[b, g] = 0x7FC0
    return Q, K, V, lens, mask


@pytest.mark.parametrize("B,Hq,Hk,d,L_max,lens,keep", [
    (1, 32, 8, 128, 1, [1], 1.0),
    (3, 32, 8, 128, 700, [700, 129, 128], 0.5),
    (6, 32, 8, 128, 2048, [2048, 0, 1, 255, 256, 1500], 0.5),
    (5, 8, 8, 64, 300, [300, 17, 64, 1, 299], 0.5),
    (4, 16, 2, 128, 513, [513, 512, 100, 3], 1.0),
    (2, 32, 8, 128, 4097, [4097, 130], 0.0),
    (16, 32, 8, 128, 1024, list(range(1024, 0, -64)), 0.34),
])
def test_attn_decode_parity(B, Hq, Hk, d, L_max, lens, keep):
    Q, K, V, lens, mask = _case(B, Hq, Hk, d, L_max, lens, keep, seed=B + L_max)
    O = ops.attn_decode(_dev_bits(Q), _dev_bits(K), _dev_bits(V), torch.from_numpy(lens).cuda(),
                        torch.from_numpy(mask).cuda())
    ops.device_status()
    Og = to_f64(O)
    assert not np.isnan(Og).any()
    qpk = Hq // Hk
    for b in range(B):
        for g in range(Hk):
            if mask[b, g] == 0 or lens[b] == 0:
                assert (Og[b, g * qpk:(g + 1) * qpk] == 0).all()
    ref = oracle.attn_decode(Q, K, V, lens, mask)
    assert_close(Og.reshape(B * Hq, d), ref.reshape(B * Hq, d), "attn_decode")


def test_attn_decode_lens_are_clamped():
    """A length beyond L_max reads only L_max keys (it is clamped), a
    negative one gives zeros."""
    Q, K, V, _, mask = _case(2, 8, 2, 64, 100, [100, 100], 1.0, seed=5)
    lens_bad = np.array([1000, -5], np.int32)
    O = ops.attn_decode(_dev_bits(Q), _dev_bits(K), _dev_bits(V), torch.from_numpy(lens_bad).cuda(),
                        torch.from_numpy(mask).cuda())
    ops.device_status()
    Og = to_f64(O)
    ref = oracle.attn_decode(Q, K, V, np.array([100, 0], np.int32), mask)
    assert (Og[1] == 0).all()
    assert_close(Og.reshape(-1, 64), ref.reshape(-1, 64), "attn_decode clamp")


def test_attn_decode_argument_errors():
    lib = ops.lib()
    Q = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((2, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((2,), 16, dtype=torch.int32, device="cuda")
    mask = torch.ones((2, 4), dtype=torch.uint8, device="cuda")
    ws = torch.empty((1 << 20,), dtype=torch.uint8, device="cuda")
    p = ops._ptr
    st = lib.wide_attn_decode(p(Q), p(K), p(K), p(lens), p(mask), 2, 12, 5, 128, 16, p(Q), p(ws),
                              ws.numel(), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_INVALID_ARG"   # Hq not a multiple of Hk
    st = lib.wide_attn_decode(p(Q), p(K), p(K), p(lens), p(mask), 2, 12, 4, 96, 16, p(Q), p(ws),
                              ws.numel(), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_UNSUPPORTED"   # d = 96
    st = lib.wide_attn_decode(p(Q), p(K), p(K), p(lens), p(mask), 2, 12, 4, 128, 16, p(Q), p(ws),
                              ws.numel(), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_UNSUPPORTED"   # 3 query heads per KV head
    st = lib.wide_attn_decode(p(Q), p(K), p(K), p(lens), p(mask), 2, 16, 4, 128, 16, p(Q), p(ws),
                              16, ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_WORKSPACE"
