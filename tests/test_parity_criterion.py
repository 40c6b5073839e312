"""The parity criterion used by the GPU tests, checked on the CPU.

The exact oracle result rounded to bf16 (what a correct kernel returns) must
pass; results with a planted mistake (made here on the CPU from the oracle)
must fail: a dropped group, swapped token rows, a wrong activation sign, a
group mask applied to the wrong group, a transposed weight slice.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from group_masked_gemm_gb300 import synthetic as syn
from parity import TOL, excess_err


def _bf16(x):
    return syn.bf16_to_f32(syn.bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


@pytest.fixture(scope="module")
def case():
    inp = syn.ffn_inputs(96, 256, 1024, 128, seed=3, keep=0.5)
    H = oracle.gate_up(inp.X, inp.Wg, inp.Wu, inp.mask, inp.G)
    Y = oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, inp.G)
    return inp, H, Y


def test_correct_rounding_passes(case):
    inp, H, Y = case
    assert excess_err(_bf16(H), H) <= TOL
    assert excess_err(_bf16(Y), Y) <= TOL
    # the bf16 intermediate of the GPU FFN (H rounded before the down GEMM)
    Hb = syn.bf16_bits(H.astype(np.float32))
    Yb = oracle.proj_k(Hb, inp.Wd, inp.mask, inp.G)
    assert excess_err(_bf16(Yb), Y) <= TOL


def test_planted_mistakes_fail(case):
    inp, H, Y = case
    G = inp.G
    # 1. a dropped group in the down projection
    m = inp.mask.copy()
    t = int(np.argmax(m[:, 2]))
    m[t, 2] = 0
    Y1 = oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, m, G)
    assert excess_err(_bf16(Y1), Y) > TOL
    # 2. two token rows swapped in the scatter
    Y2 = Y.copy()
    Y2[[5, 9]] = Y2[[9, 5]]
    assert excess_err(_bf16(Y2), Y) > TOL
    # 3. silu with the wrong sign, a / (1 + exp(a))
    X, Wg, Wu = (syn.bf16_to_f32(a).astype(np.float64) for a in (inp.X, inp.Wg, inp.Wu))
    a = X @ Wg.T
    h_bad = a * expit(-a) * (X @ Wu.T) * np.repeat(inp.mask, G, axis=1)
    assert excess_err(_bf16(h_bad), H) > TOL
    # 4. the mask of group g applied to group g+1's channels
    H4 = oracle.gate_up(inp.X, inp.Wg, inp.Wu, np.roll(inp.mask, 1, axis=1), G)
    assert excess_err(_bf16(H4), H) > TOL
    # 5. one weight slice transposed within its group
    Wg5 = inp.Wg.copy()
    Wg5[:G, :G] = Wg5[:G, :G].T.copy()
    H5 = oracle.gate_up(inp.X, Wg5, inp.Wu, inp.mask, G)
    assert excess_err(_bf16(H5), H) > TOL
