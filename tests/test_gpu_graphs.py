"""The decode FFN step and routed prefill attention inside CUDA graphs.

The decode GEMM-K and its split finalize are launched as programmatic
dependents of the kernel before them (their set-up overlaps that kernel; a
grid-dependency wait guards every input).  Captured into a graph, the launch
order becomes graph edges; a replay must give exactly the eager result (the
kernels are deterministic), and the eager result must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import assert_close, mask_dev, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


def _replay_equals_eager(fn, outs):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    for o in outs:
        o.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ops.device_status()
    for e, o in zip(eager, outs):
        assert torch.equal(e, o)
    return eager


@pytest.mark.parametrize("T", [1, 4, 16])
def test_decode_ffn_step_in_a_graph(T):
    inp = syn.llama8b_decode(T, 128)
    X, Wg, Wu, Wd, m = to_dev(inp.X), to_dev(inp.Wg), to_dev(inp.Wu), to_dev(inp.Wd), mask_dev(inp.mask)
    H = torch.empty((T, inp.F), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((T, inp.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty((max(16, ops.gemm_k_workspace_size(T, inp.F, inp.D, 128)),), dtype=torch.uint8,
                     device="cuda")

    def step():
        ops.gemm_mn_gate_up(X, Wg, Wu, m, None, None, 128, out=H)
        ops.gemm_k_down(H, Wd, m, None, None, 128, out=Y, ws=ws)
    (y,) = _replay_equals_eager(step, [Y])
    assert_close(to_f64(y), oracle.ffn(inp.X, inp.Wg, inp.Wu, inp.Wd, inp.mask, 128), "decode graph")


def test_attn_prefill_in_a_graph():
    rng = np.random.default_rng(12)
    B, T, Hq, Hk, d = 2, 700, 8, 2, 128
    Q = torch.from_numpy(syn.bf16_bits(rng.standard_normal((B, T, Hq, d), dtype=np.float32)).view(np.int16))
    K = torch.from_numpy(syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32)).view(np.int16))
    V = torch.from_numpy(syn.bf16_bits(rng.standard_normal((B, Hk, T, d), dtype=np.float32)).view(np.int16))
    Q, K, V = (t.view(torch.bfloat16).cuda() for t in (Q, K, V))
    mask = torch.from_numpy((rng.random((B, T, Hk)) < 0.4).astype(np.uint8)).cuda()
    perm = torch.empty((B, Hk, T), dtype=torch.int32, device="cuda")
    counts = torch.empty((B, Hk), dtype=torch.int32, device="cuda")
    for b in range(B):  # the per-sequence reorder, into 16-byte-aligned buffers
        pb, cb = ops.reorder_masks(mask[b].clone())
        perm[b].copy_(pb)
        counts[b].copy_(cb)
    O = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    lib, p = ops.lib(), ops._ptr

    def attn():
        st = lib.wide_attn_prefill(p(Q), p(K), p(V), p(perm), p(counts), B, T, Hq, Hk, d, 1, p(O),
                                   ops._stream())
        assert ops.STATUS[st] == "WIDE_OK"
    _replay_equals_eager(attn, [O])
