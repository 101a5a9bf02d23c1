"""Failure detection without a GPU fault.

Every mbarrier wait inside the kernel is bounded by %globaltimer (the Muse
Spark AMD dev page's _spin_bounded model).  The test makes one wait run out
on purpose -- cluster ranks other than 0 are told to skip publishing their
partials, so rank 0 waits on a barrier phase that nothing completes -- and
checks that the launch ends, the fault record names the rank-0 reduction
wait, and the context stays usable for a normal call afterwards.  Nothing
is stored remotely and every other wait stays bounded, so no hang or memory
fault is involved.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import synthetic  # noqa: E402
from tests._gpu import assert_parity, to_dev, to_host  # noqa: E402

ROLE_EPI_REDUCE = 5


def _inputs(M=4, N=256, K=1024):
    a = synthetic.normal_bf16((1, N, K), 900, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((1, M, K), 900, synthetic.STREAM_B, 1.0)
    return a, b


@pytest.mark.parametrize("dedicated", [1, 0])
def test_skipped_publish_times_out_and_the_context_survives(dedicated):
    a, b = _inputs()
    ta, tb = to_dev(a), to_dev(b)
    assert sk.splitk_get_status() == 0
    plan = sk.splitk_plan(4, 256, 1024, 1, 4)
    if not dedicated and plan.mailbox_dedicated:
        # the mailbox moves onto the drained weight ring; with the smaller
        # shared memory 3 CTAs fit an SM, so no weight tiles stay in tensor
        # memory (3 x 256 columns would not fit its 512)
        plan.mailbox_dedicated = 0
        plan.smem_bytes -= 3 * 4 * 512
        plan.a_tmem_tiles = 0
        plan.tmem_cols = max(32, plan.mma_n) * plan.mma_issuers
    try:
        sk.splitk_set_wait_limit_ns(50_000_000)          # 50 ms
        sk.splitk_debug_inject(sk.INJECT_SKIP_PUBLISH)
        sk.splitk_gemm_bf16_planned(ta, tb, None, plan)
        torch.cuda.synchronize()
    finally:
        sk.splitk_debug_inject(0)
        sk.splitk_set_wait_limit_ns(0)
    fault = sk.splitk_get_fault()
    assert fault["code"] == -6, fault
    assert fault["role"] == ROLE_EPI_REDUCE and fault["cluster_rank"] == 0, fault
    # the record is cleared by the read
    assert sk.splitk_get_status() == 0
    # and the device still computes correctly
    c = to_host(sk.splitk_gemm_bf16(ta, tb, split_k=4))
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert_parity(c, oracle.gemm(a, b), a, b, 1024)


def test_no_fault_recorded_in_normal_operation():
    a, b = _inputs(M=16, N=512, K=2048)
    ta, tb = to_dev(a), to_dev(b)
    for split in (1, 2, 4, 8):
        sk.splitk_gemm_bf16(ta, tb, split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_fault()["code"] == 0


@pytest.mark.parametrize("stages,b_stages", [(2, 0), (3, 2)])
def test_persistent_plan_skipped_publish_times_out_and_the_context_survives(stages, b_stages):
    """The persistent kernel's bounded waits (the activations on the weight
    ring, or on a ring of their own): with the peers' partials withheld
    every rank's reduction wait runs out, the launch ends, and a normal call
    afterwards is correct."""
    M, N, K, L, split = 64, 1000, 4096, 1, 4
    a = synthetic.normal_bf16((L, N, K), 901, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), 901, synthetic.STREAM_B, 1.0)
    ta, tb = to_dev(a), to_dev(b)
    props = torch.cuda.get_device_properties(0)
    plan = next(p for p in sk.splitk_plan_candidates_for(M, N, K, L, split, props.multi_processor_count,
                                                          props.shared_memory_per_multiprocessor,
                                                          props.shared_memory_per_block_optin)
                if p.persistent and (p.stages, p.b_stages) == (stages, b_stages))
    plan.grid[1] = 2                                     # each cluster walks several tiles
    try:
        sk.splitk_set_wait_limit_ns(50_000_000)          # 50 ms
        sk.splitk_debug_inject(sk.INJECT_SKIP_PUBLISH)
        sk.splitk_gemm_bf16_planned(ta, tb, None, plan)
        torch.cuda.synchronize()
    finally:
        sk.splitk_debug_inject(0)
        sk.splitk_set_wait_limit_ns(0)
    fault = sk.splitk_get_fault()
    assert fault["code"] == -6, fault
    assert fault["role"] == ROLE_EPI_REDUCE, fault
    assert sk.splitk_get_status() == 0
    c = to_host(sk.splitk_gemm_bf16_planned(ta, tb, None, plan))
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert_parity(c, oracle.gemm(a, b), a, b, K)
