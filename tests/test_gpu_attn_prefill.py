"""GPU parity of routed causal prefill attention (App. B "Implementation of
Attention", prefill, Algorithm 4; GQA-aligned groups of Sec. 3.1 Eq. 2)
against the fp64 C oracle.

Tolerance, derived from the kernel's arithmetic: the softmax weights p are
rounded to bf16 (relative error <= 2^-9 each) before the P V product while
the normaliser l sums the unrounded p, so |O - O_ref| <= 2^-9 sum_j p_j |v_j|
/ l, which is the oracle's attention with |V| in place of V (ref_abs); the
bf16 output adds half an ulp, 2^-9 |O_ref|.  The test allows twice both,
plus 1e-4 RMS(O_ref) for the fp32 sums.  A row-level mistake (a wrong token,
a missed key, an unmasked future key) moves O by about |O| and fails it.  The
GEMMs' 2e-2 RMS rule does not fit attention: causal outputs range from |v|
(first tokens) to |v| / sqrt(t), and inactive rows are zero."""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _assert_attn_close(y, ref, ref_abs, what):
    rms = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    excess = np.abs(y - ref) - 2.0 ** -8 * (np.abs(ref) + ref_abs)
    worst = float(excess.max())
    assert worst <= 1e-4 * rms, (f"{what}: max(|y-ref| - 2^-8(|ref| + ref_abs)) = {worst:.3e} "
                                 f"> 1e-4 RMS (plain max|y-ref| = {float(np.abs(y - ref).max()):.3e})")


def _abs_bits(V):
    return (V & np.uint16(0x7FFF)).astype(np.uint16)  # |v| of bf16 bit patterns


def _case(B, T, Hq, Hk, d, keep, seed):
    rng = np.random.default_rng(seed)
    Q = syn.bf16_bits(rng.standard_normal((B, T, Hq, d), dtype=np.float32))
    K = syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32))
    V = syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32))
    mask = (rng.random((B, T, Hk)) < keep).astype(np.uint8)
    return Q, K, V, mask


@pytest.mark.parametrize("B,T,Hq,Hk,d,keep,causal", [
    (1, 64, 4, 1, 128, 1.0, True),
    (2, 300, 8, 2, 128, 0.5, True),     # ragged T, several query and key tiles
    (1, 517, 32, 8, 128, 0.34, True),   # 8B head layout
    (3, 129, 4, 4, 64, 0.6, False),     # non-causal, d = 64, one query head per KV head
    (1, 200, 8, 2, 128, 0.0, True),     # nothing active: every row zero
    (1, 1000, 8, 8, 128, 0.05, True),   # sparse: few admitted rows per group
    (2, 130, 16, 2, 64, 0.5, True),     # 8 query heads per KV head
    (2, 333, 8, 2, 128, 0.7, False),    # non-causal, d = 128: a key tile past T
    (1, 2048, 4, 1, 128, 1.0, True),    # 16 key tiles, every row active
])
def test_attn_prefill_parity(B, T, Hq, Hk, d, keep, causal):
    Q, K, V, mask = _case(B, T, Hq, Hk, d, keep, seed=T + Hq)
    O = ops.attn_prefill(_dev(Q), _dev(K), _dev(V), torch.from_numpy(mask).cuda(), causal=causal)
    ops.device_status()
    Og = to_f64(O)
    assert not np.isnan(Og).any()
    qpk = Hq // Hk
    inactive = np.repeat(mask == 0, qpk, axis=2)  # [B, T, Hq]
    assert (Og[inactive] == 0).all()
    ref = oracle.attn_prefill(Q, K, V, mask, causal=causal)
    ref_abs = oracle.attn_prefill(Q, K, _abs_bits(V), mask, causal=causal)
    _assert_attn_close(Og, ref, ref_abs, "attn_prefill")


def test_attn_prefill_large_logits():
    """Queries scaled by 8 spread the logits over tens of log2 units, so the
    running maximum of a row keeps growing across key tiles and the kernel's
    rescaling of the accumulated output is exercised."""
    B, T, Hq, Hk, d = 1, 700, 8, 2, 128
    Q, K, V, mask = _case(B, T, Hq, Hk, d, 0.6, seed=77)
    Q = syn.bf16_bits(syn.bf16_to_f32(Q) * np.float32(8.0))
    O = ops.attn_prefill(_dev(Q), _dev(K), _dev(V), torch.from_numpy(mask).cuda())
    ops.device_status()
    Og = to_f64(O)
    assert not np.isnan(Og).any()
    ref = oracle.attn_prefill(Q, K, V, mask)
    ref_abs = oracle.attn_prefill(Q, K, _abs_bits(V), mask)
    _assert_attn_close(Og, ref, ref_abs, "attn_prefill large logits")


def test_attn_prefill_full_size_sampled_rows():
    """The full prunable-layer attention: T = 16384, Hq = 32, Hk = 8, d = 128,
    causal, attention keep 0.34; every row on the GPU, 48 sampled positions
    (all heads) against the oracle, including the first and the last."""
    B, T, Hq, Hk, d = 1, 16384, 32, 8, 128
    Q, K, V, mask = _case(B, T, Hq, Hk, d, 0.34, seed=16)
    O = ops.attn_prefill(_dev(Q), _dev(K), _dev(V), torch.from_numpy(mask).cuda())
    ops.device_status()
    rows = np.unique(np.concatenate([[0, T - 1], syn.sample_rows(T, 46, 5)])).astype(np.int32)
    Og = to_f64(O)[:, rows]
    ref = oracle.attn_prefill(Q, K, V, mask, rows=rows)
    ref_abs = oracle.attn_prefill(Q, K, _abs_bits(V), mask, rows=rows)
    _assert_attn_close(Og, ref, ref_abs, "attn_prefill full size")


def test_attn_prefill_argument_errors():
    lib = ops.lib()
    Q = torch.zeros((1, 8, 4, 96), dtype=torch.bfloat16, device="cuda")
    perm = torch.zeros((1, 2, 8), dtype=torch.int32, device="cuda")
    counts = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    p = ops._ptr
    st = lib.wide_attn_prefill(p(Q), p(Q), p(Q), p(perm), p(counts), 1, 8, 4, 2, 96, 1, p(Q), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_UNSUPPORTED"  # d = 96
    st = lib.wide_attn_prefill(p(Q), p(Q), p(Q), p(perm), p(counts), 1, 8, 4, 3, 128, 1, p(Q), ops._stream())
    assert ops.STATUS[st] == "WIDE_ERR_INVALID_ARG"  # Hq not a multiple of Hk
