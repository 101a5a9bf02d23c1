"""The allocation-free entry point, splitk_gemm_bf16_noalloc.

Some callers cannot allocate device memory (a framework allocator owns the
budget, or a latency-critical path cannot afford cudaMalloc's
synchronisation).  This entry point keeps the kernel's only scratch -- the
tensor map of the weights -- in a static device array inside the library and
allocates nothing.  The test calls it through the C ABI twice in a row, with
different weights and activations, and checks each output against the
regular entry point's within the parity tolerance.  The file is named so
that pytest collects it last.
"""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import synthetic  # noqa: E402
from tests._gpu import assert_parity, to_dev, to_host  # noqa: E402


def _case(seed, L, M, N, K):
    a = synthetic.normal_bf16((L, N, K), seed, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0)
    return a, b


def test_two_calls_in_a_row_match_the_regular_entry_point():
    cases = [(71, 1, 1, 7168, 2048, 4), (72, 2, 16, 300, 1024, 8)]
    inputs = []
    for seed, L, M, N, K, split in cases:
        a, b = _case(seed, L, M, N, K)
        ta, tb = to_dev(a), to_dev(b)
        ref = sk.splitk_gemm_bf16(ta, tb, split_k=split)
        out = torch.empty_like(ref)
        inputs.append((a, b, ta, tb, ref, out, K, split))
    torch.cuda.synchronize()
    # two allocation-free calls back to back on one stream
    for a, b, ta, tb, ref, out, K, split in inputs:
        sk.splitk_gemm_bf16_noalloc(ta, tb, out, split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    for a, b, ta, tb, ref, out, K, split in inputs:
        assert_parity(to_host(out), to_host(ref), a, b, K)


def test_a_capturing_stream_is_refused_with_nothing_enqueued():
    a, b = _case(73, 1, 4, 256, 1024)
    ta, tb = to_dev(a), to_dev(b)
    out = torch.full((1, 4, 256), 7.0, dtype=torch.bfloat16, device=ta.device)
    sk.splitk_gemm_bf16_noalloc(ta, tb, out, split_k=4)          # the device's set-up, outside capture
    torch.cuda.synchronize()
    out.fill_(7.0)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(sk.SplitKError) as e:
            sk.splitk_gemm_bf16_noalloc(ta, tb, out, split_k=4)
        out.mul_(1)                                              # the graph's one node
    assert e.value.code == -13
    g.replay()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    assert sk.splitk_get_status() == 0
