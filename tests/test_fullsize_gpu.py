"""Parity at the full workload sizes, in the launch configuration the
benchmark times (the workload's split_k, the library's plan, PDL on).

The tiny and the two decode workloads (bf16, and with A16W4 and A16W8
weights) are compared with the oracle on every
output element (the threaded oracle takes seconds there).  The wide
projection and the sweep points are checked on sampled outputs one by one
(every element of the first and last token row of the first and last weight
tile, plus random ones); two closed forms check every output exactly at full
size: all-ones inputs give C = K, and weights with one 1.0 per row at column
n mod K give C[l, m, n] = B[l, m, n mod K] bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import os  # noqa: E402

import oracle  # noqa: E402
import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import workloads  # noqa: E402
from tests import _tol  # noqa: E402
from tests._gpu import DEV, to_dev, to_host  # noqa: E402

ONE = 0x3F80
FIXED = [workloads.DECODE_M1, workloads.DECODE_M16, workloads.WIDE_S2, workloads.WIDE_S4]
SWEEP = workloads.all_sweep()


def _sample_indices(w, n_random=3000, seed=0):
    rng = np.random.default_rng(seed)
    L, M, N = w.L, w.M, w.N
    idx = [l * M * N + m * N + n for l in (0, L - 1) for m in (0, M - 1)
           for n in list(range(0, min(N, 128))) + list(range(max(0, N - 128), N))]
    idx += rng.integers(0, L * M * N, size=n_random).tolist()
    return np.unique(np.array(idx, dtype=np.int64))


_A_CACHE = {}


def _weights(w):
    key = (w.N, w.K, w.L, w.seed)
    if key not in _A_CACHE:
        _A_CACHE.clear()
        a = w.make_a()
        _A_CACHE[key] = (a, to_dev(a))
    return _A_CACHE[key]


def _check_sampled(w):
    a, ta = _weights(w)
    b = w.make_b()
    tb = to_dev(b)
    tc = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    c = to_host(tc).reshape(-1)
    idx = _sample_indices(w)
    ref = oracle.elements(a, b, idx)
    ok, rep = _tol.check(c[idx], ref, w.K, _tol.max_abs_bf16(a), _tol.max_abs_bf16(b))
    assert ok, f"{w.name} M={w.M} split={w.split_k}: {rep}"
    # run to run: identical bits
    tc2 = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert torch.equal(tc.view(torch.int16), tc2.view(torch.int16))


@pytest.mark.parametrize("w", [workloads.TINY, workloads.DECODE_M1, workloads.DECODE_M16],
                         ids=lambda w: f"{w.name.split()[0]}-M{w.M}-s{w.split_k}")
def test_decode_workloads_every_output_against_oracle(w):
    a, ta = _weights(w)
    b = w.make_b()
    tc = sk.splitk_gemm_bf16(ta, to_dev(b), split_k=w.split_k)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    ref = oracle.gemm(a, b, threads=max(1, min(32, os.cpu_count() or 1)))
    ok, rep = _tol.check(to_host(tc), ref, w.K, _tol.max_abs_bf16(a), _tol.max_abs_bf16(b))
    assert ok, f"{w.name}: {rep}"


@pytest.mark.parametrize("w", FIXED[2:], ids=lambda w: f"{w.name.split()[0]}-M{w.M}-s{w.split_k}")
def test_wide_workloads_sampled_against_oracle(w):
    _check_sampled(w)


@pytest.mark.parametrize("w", SWEEP, ids=lambda w: f"sweep-M{w.M}-s{w.split_k}")
def test_sweep_points_sampled_against_oracle(w):
    _check_sampled(w)


@pytest.mark.parametrize("w", FIXED + [workloads.sweep(128, 8), workloads.sweep(1, 1)],
                         ids=lambda w: f"{w.name.split()[0]}-M{w.M}-s{w.split_k}")
def test_full_size_closed_forms(w):
    L, M, N, K = w.L, w.M, w.N, w.K
    # all ones: C = K exactly
    ta = torch.full((L, N, K), 1.0, dtype=torch.bfloat16, device=DEV)
    tb = torch.full((L, M, K), 1.0, dtype=torch.bfloat16, device=DEV)
    tc = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert bool((tc == float(K)).all())
    # one 1.0 per weight row at column n mod K: C[l, m, n] = B[l, m, n mod K]
    ta.zero_()
    n = torch.arange(N, device=DEV)
    ta[:, n, n % K] = 1.0
    tb = to_dev(w.make_b())
    tc = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    expect = tb[:, :, (n % K)]
    # exact equality of values (+0 and -0 compare equal: the sign of an exact
    # zero sum depends on the order of the zero products)
    assert torch.equal(tc.float(), expect.float())
    assert sk.splitk_get_status() == 0


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("w", [workloads.DECODE_M1, workloads.DECODE_M16],
                         ids=lambda w: f"{w.name.split()[0]}-M{w.M}-s{w.split_k}")
def test_quantized_decode_workloads_every_output_against_oracle(w, bits):
    """A16W4 and A16W8 weights (seeded codes and scales) at the decode
    workloads' full size, in the plan the library picks: every output
    against the oracle, and run to run the same bits."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    gen, run, ref_fn, deq = ((synthetic.w4_weights, sk.splitk_gemm_w4a16, oracle.gemm_w4a16, oracle.w4_dequant)
                             if bits == 4 else
                             (synthetic.w8_weights, sk.splitk_gemm_w8a16, oracle.gemm_w8a16, oracle.w8_dequant))
    aq, a_s = gen(w.L, w.N, w.K, w.seed)
    b = w.make_b()
    tq, ts, tb = (torch.from_numpy(np.ascontiguousarray(aq)).to(DEV),
                  torch.from_numpy(np.ascontiguousarray(a_s)).to(DEV), to_dev(b))
    tc = run(tq, ts, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    ok, rep = _tol.check(to_host(tc), ref_fn(aq, a_s, b), w.K, float(np.abs(deq(aq, a_s)).max()),
                         _tol.max_abs_bf16(b))
    assert ok, f"A16W{bits} {w.name}: {rep}"
    tc2 = run(tq, ts, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert torch.equal(tc.view(torch.int16), tc2.view(torch.int16))
