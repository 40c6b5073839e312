"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times.  The whole output is produced on the GPU; the oracle then
recomputes a seeded subset of token rows (tokens are independent, so a row of
the full problem is exactly the row the oracle computes alone).  Reordering
is compared bit-exactly in full.
"""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import assert_close, inactive_columns, mask_dev, to_dev, to_f64

pytestmark = pytest.mark.gpu

N_ROWS = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


@pytest.fixture(scope="module")
def llama8b():
    return syn.llama8b_prefill(0.5)


def _run_ffn(inp):
    X, Wg, Wu, Wd = (to_dev(a) for a in (inp.X, inp.Wg, inp.Wu, inp.Wd))
    m = mask_dev(inp.mask)
    perm, counts = ops.reorder_masks(m)
    H = ops.gemm_mn_gate_up(X, Wg, Wu, m, perm, counts, inp.G)
    Y = ops.gemm_k_down(H, Wd, m, perm, counts, inp.G)
    ops.device_status()
    return perm, counts, H, Y


def _check_ffn(inp, seed):
    perm, counts, H, Y = _run_ffn(inp)
    p_ref, c_ref = oracle.reorder(inp.mask)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    rows = syn.sample_rows(inp.T, N_ROWS, seed)
    # boundary rows of the reordered tiles of group 0 (first/last active token)
    act0 = p_ref[0][: c_ref[0]]
    if act0.size:
        rows = np.unique(np.concatenate([rows, act0[[0, -1]]]).astype(np.int32))
    Hr = to_f64(H)[rows]
    assert (Hr[inactive_columns(inp.mask[rows], inp.G)] == 0).all()
    assert_close(Hr, oracle.gate_up(inp.X, inp.Wg, inp.Wu, inp.mask, inp.G, rows=rows), "H rows")
    Yr = to_f64(Y)[rows]
    assert_close(Yr, oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, inp.G, rows=rows), "Y rows")
    # whole-output property: tokens with no active group give exact zeros
    none = inp.mask.sum(1) == 0
    if none.any():
        assert (to_f64(Y)[none] == 0).all()


def test_llama8b_prefill_p50(llama8b):
    _check_ffn(llama8b, seed=21)


@pytest.mark.parametrize("keep", [0.75, 0.25, 1.0])
def test_llama8b_prefill_other_sparsities(llama8b, keep):
    rng = np.random.default_rng(2)
    mask = (rng.random(llama8b.mask.shape) < keep).astype(np.uint8)
    _check_ffn(syn.with_mask(llama8b, mask), seed=22)


def test_llama3b_prefill_per_group():
    _check_ffn(syn.llama3b_prefill(), seed=23)


def test_llama8b_layer_projections():
    lay = syn.llama8b_layer()
    Ga = lay.G_attn
    X = to_dev(lay.X)
    ma = mask_dev(lay.mask_attn)
    perm, counts = ops.reorder_masks(ma)
    Q = ops.proj_mn(X, to_dev(lay.Wq), ma, perm, counts, Ga)
    O = ops.proj_k(to_dev(lay.A), to_dev(lay.Wo), ma, perm, counts, Ga)
    ops.device_status()
    rows = syn.sample_rows(lay.T, N_ROWS, 24)
    Qr = to_f64(Q)[rows]
    assert (Qr[inactive_columns(lay.mask_attn[rows], Ga)] == 0).all()
    assert_close(Qr, oracle.proj_mn(lay.X, lay.Wq, lay.mask_attn, Ga, rows=rows), "q_proj rows")
    assert_close(to_f64(O)[rows], oracle.proj_k(lay.A, lay.Wo, lay.mask_attn, Ga, rows=rows),
                 "o_proj rows")
    _check_ffn(lay.ffn, seed=25)
