"""The allocation-free entry point, splitk_gemm_bf16_noalloc.

Who needs it: code that may not call cudaMalloc -- a framework whose caching
allocator owns the whole device budget, a latency-critical decode loop that
cannot take cudaMalloc's device-wide synchronisation, or a process that
reserves all GPU memory up front and treats any later allocation as a
failure.  The regular entry point allocates its tensor-map pool on its first
call; this one keeps the kernel's only scratch (the tensor map of the
weights) in a static device array inside the library and allocates nothing.

The tests call it through the C ABI: twice in a row with different weights
and shapes, each output bit for bit equal to the regular entry point's and
within the parity tolerance of the CPU oracle; and, in a fresh process that
calls nothing else of the library first, with the library's pool still
unallocated and the device's free memory unchanged across the calls.  The
file is named so that pytest collects it last.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import synthetic  # noqa: E402
from tests._gpu import assert_parity, oracle_full, to_dev, to_host  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [(71, 1, 1, 7168, 2048, 4), (72, 2, 16, 300, 1024, 8)]   # seed, L, M, N, K, split_k


def _case(seed, L, M, N, K):
    a = synthetic.normal_bf16((L, N, K), seed, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0)
    return a, b


def test_two_calls_in_a_row_equal_the_regular_entry_point_and_the_oracle():
    inputs = []
    for seed, L, M, N, K, split in CASES:
        a, b = _case(seed, L, M, N, K)
        ta, tb = to_dev(a), to_dev(b)
        ref = sk.splitk_gemm_bf16(ta, tb, split_k=split)
        out = torch.full_like(ref, 3.0)
        inputs.append((a, b, ta, tb, ref, out, K, split))
    torch.cuda.synchronize()
    # two allocation-free calls back to back on one stream
    for a, b, ta, tb, ref, out, K, split in inputs:
        sk.splitk_gemm_bf16_noalloc(ta, tb, out, split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    for a, b, ta, tb, ref, out, K, split in inputs:
        got = to_host(out)
        assert np.array_equal(got, to_host(ref))          # same kernel, same plan: same bits
        assert_parity(got, oracle_full(a, b), a, b, K)


# Run in a fresh interpreter: the library's first call of all is an
# allocation-free one, so its pool must still be unallocated afterwards.
_FRESH = r"""
import json, sys
sys.path.insert(0, ROOT)
import numpy as np
import torch
import split_bf16_gemm_swapped_gb300 as sk
from split_bf16_gemm_swapped_gb300 import synthetic
import oracle
from tests import _tol

dev = torch.device("cuda:0")
torch.cuda.set_device(dev)

def bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

# every buffer of both rounds is allocated (by torch) before the first call
rounds = []
for r in range(2):
    calls = []
    for seed, L, M, N, K, split in CASES:
        a = synthetic.normal_bf16((L, N, K), seed + 100 * r, synthetic.STREAM_A, 0.02)
        b = synthetic.normal_bf16((L, M, K), seed + 100 * r, synthetic.STREAM_B, 1.0)
        out = torch.full((L, M, N), 3.0, dtype=torch.bfloat16, device=dev)
        calls.append((a, b, bf16(a), bf16(b), out, K, split))
    rounds.append(calls)
torch.cuda.synchronize()

def run(calls):
    for a, b, ta, tb, out, K, split in calls:
        sk.splitk_gemm_bf16_noalloc(ta, tb, out, split_k=split)
    torch.cuda.synchronize()

report = {"info_before": sk.splitk_cache_info()}
run(rounds[0])                   # loads the kernels, looks up the scratch array
report["info_warm"] = sk.splitk_cache_info()
report["free_warm"] = torch.cuda.mem_get_info()[0]
run(rounds[1])
report["free_after"] = torch.cuda.mem_get_info()[0]
report["info_after"] = sk.splitk_cache_info()
report["status"] = sk.splitk_get_status()
report["parity"] = []
for calls in rounds:
    for a, b, ta, tb, out, K, split in calls:
        got = out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        ok, rep = _tol.check(got, oracle.gemm(a, b, threads=8), K, _tol.max_abs_bf16(a), _tol.max_abs_bf16(b))
        report["parity"].append([bool(ok), rep])
# the diagnostic does see an allocation: the regular entry point creates its pool
a, b, ta, tb, out, K, split = rounds[1][0]
sk.splitk_gemm_bf16(ta, tb, out, split_k=split)
torch.cuda.synchronize()
report["info_regular"] = sk.splitk_cache_info()
print("REPORT " + json.dumps(report))
"""


def test_a_fresh_process_calling_only_the_allocation_free_entry_allocates_nothing():
    script = f"ROOT = {ROOT!r}\nCASES = {CASES!r}\n" + _FRESH
    res = subprocess.run([sys.executable, "-c", script], cwd=ROOT, capture_output=True, text=True,
                         timeout=900)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-3000:]
    line = [x for x in res.stdout.splitlines() if x.startswith("REPORT ")][-1]
    rep = json.loads(line[len("REPORT "):])
    empty = {"device_bytes": 0, "host_bytes": 0, "maps": 0}
    assert rep["info_before"] == empty
    assert rep["info_warm"] == empty                 # the library owns no memory after its calls
    assert rep["info_after"] == empty
    assert rep["free_after"] == rep["free_warm"]     # nor did anything else allocate device memory
    assert rep["status"] == 0
    assert all(ok for ok, _ in rep["parity"]), rep["parity"]
    assert rep["info_regular"]["device_bytes"] > 0 and rep["info_regular"]["maps"] == 1


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
