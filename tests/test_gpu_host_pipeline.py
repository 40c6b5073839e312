"""The pipelined host API (ops.HostFfnPipeline) returns, for every batch, the
same Y as the device call on that batch, although its copies and kernels of
neighbouring batches overlap on three streams."""
import numpy as np
import pytest
import torch

import oracle
from group_masked_gemm_gb300 import build, ops
from group_masked_gemm_gb300 import synthetic as syn
from parity import assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.lib()


def _pinned_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def test_host_pipeline_matches_device_call_per_batch():
    T, D, F, G, n = 300, 512, 1024, 128, 5
    base = syn.ffn_inputs(T, D, F, G, seed=21, keep=0.5)
    Wg, Wu, Wd = to_dev(base.Wg), to_dev(base.Wu), to_dev(base.Wd)
    pipe = ops.HostFfnPipeline(Wg, Wu, Wd, G, T)
    batches, outs = [], []
    for i in range(n):
        inp = syn.ffn_inputs(T, D, F, G, seed=100 + i, keep=0.3 + 0.1 * i)
        Xh, mh = _pinned_bits(inp.X), torch.from_numpy(inp.mask).pin_memory()
        Yh = torch.empty((T, D), dtype=torch.bfloat16).pin_memory()
        batches.append((inp, Xh, mh))
        outs.append(pipe.submit(Xh, mh, Yh))
    pipe.synchronize()
    ops.device_status()
    for (inp, Xh, mh), Yh in zip(batches, outs):
        Yd = ops.ffn_forward(Xh.cuda(), Wg, Wu, Wd, mh.cuda(), G)
        torch.cuda.synchronize()
        assert torch.equal(Yh, Yd.cpu())  # same kernels, deterministic
        assert_close(to_f64(Yd), oracle.ffn(inp.X, base.Wg, base.Wu, base.Wd, inp.mask, G),
                     "host pipeline")
