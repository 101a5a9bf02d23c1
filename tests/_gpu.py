"""Helpers of the GPU parity tests: moving bf16 bit patterns between numpy
and torch, and comparing a GPU result with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import split_bf16_gemm_swapped_gb300 as sk
from tests import _tol

DEV = torch.device("cuda:0")


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gemm_gpu(a: np.ndarray, b: np.ndarray, split_k: int = 0, plan=None, flags: int = 0):
    ta, tb = to_dev(a), to_dev(b)
    torch.cuda.synchronize()
    if plan is None:
        tc = sk.splitk_gemm_bf16(ta, tb, split_k=split_k)
    else:
        tc = sk.splitk_gemm_bf16_planned(ta, tb, None, plan, flags)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    return to_host(tc)


def assert_parity(gpu_bits, ref_bits, a, b, K):
    ok, report = _tol.check(gpu_bits, ref_bits, K, _tol.max_abs_bf16(a), _tol.max_abs_bf16(b))
    assert ok, report
    return report


def oracle_full(a, b):
    return oracle.gemm(a, b, threads=8)
