"""Pins of the CPU oracle against facts fixed outside it.

Each test would fail on a plausible mistake in ``oracle/splitk_oracle.c``:
a wrong shift in the bf16 widening, truncation or round-half-up instead of
ties-to-even, rounding twice (f64 -> f32 -> bf16), flushed subnormals, a
transposed operand (A row m / B row n), a dropped or repeated k term, a wrong
L stride.  References: exact rational arithmetic (tests/_exact.py), closed
forms, library conversions (numpy bit views, torch's fp32 -> bf16), and the
hand-derived table tests/golden/bf16_rounding.txt.
"""
from __future__ import annotations

import math
import random
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from tests import _exact

GOLDEN = Path(__file__).parent / "golden"


# --------------------------------------------------------------------------
# bf16 -> float64 widening
# --------------------------------------------------------------------------
def test_widen_every_bf16_pattern_matches_numpy_bit_view():
    pats = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (pats << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_f64(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # and the sign of zeros
    assert math.copysign(1.0, oracle.bf16_to_f64(0x8000)) == -1.0


def test_widen_matches_ieee_field_definition_on_samples():
    rng = random.Random(7)
    for h in [0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7F, 0xC2F7] + \
             [rng.randrange(65536) for _ in range(2000)]:
        v = _exact.value(h)
        got = oracle.bf16_to_f64(h)
        if isinstance(v, float):
            assert (math.isnan(v) and math.isnan(got)) or v == got
        else:
            assert Fraction(got) == v, hex(h)


# --------------------------------------------------------------------------
# float64 -> bf16 rounding
# --------------------------------------------------------------------------
def _golden_rounding_cases():
    cases = []
    for line in (GOLDEN / "bf16_rounding.txt").read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok, bits, *_ = line.split()
        x = {"zero": 0.0, "negzero": -0.0, "inf": math.inf, "-inf": -math.inf,
             "nan": math.nan}.get(tok)
        if x is None:
            x = float.fromhex(tok)
        cases.append((tok, x, int(bits, 16)))
    return cases


@pytest.mark.parametrize("tok,x,bits", _golden_rounding_cases())
def test_rounding_golden_table(tok, x, bits):
    assert oracle.f64_to_bf16(x) == bits, tok
    if math.isfinite(x) and x != 0.0:
        # the table itself agrees with exact rational rounding
        assert _exact.round_bf16(Fraction(x)) == bits, tok


def test_rounding_binary32_inputs_match_torch():
    """For binary32 inputs one rounding to bf16 is torch's fp32->bf16 (RNE)."""
    rng = np.random.default_rng(11)
    pats = rng.integers(0, 2 ** 32, size=60000, dtype=np.uint64).astype(np.uint32)
    # plus exact ties and near-ties around random bf16 values
    base = rng.integers(0, 2 ** 16, size=4000, dtype=np.uint32) << 16
    extra = np.concatenate([base | 0x8000, base | 0x7FFF, base | 0x8001, base])
    pats = np.concatenate([pats, extra])
    f32 = pats.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.astype(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in f32], dtype=np.uint16)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} mismatches, first {f32[bad[0]]!r}"


def test_rounding_float64_inputs_match_exact_rationals():
    """Values with bits below binary32 precision: a single rounding decides."""
    rng = random.Random(3)
    xs = []
    for _ in range(3000):
        h = rng.randrange(0x0001, 0x7F7F)       # a finite positive bf16
        lo = _exact.value(h)
        hi = _exact.value(h + 1)
        mid = (lo + hi) / 2
        # just above / below the midpoint by an amount binary32 cannot hold
        eps = (hi - lo) * Fraction(1, 2 ** rng.randrange(20, 40))
        for v in (mid + eps, mid - eps, mid):
            f = float(v)
            if rng.random() < 0.5:
                f = -f
            xs.append(f)
    for f in xs:
        assert oracle.f64_to_bf16(f) == _exact.round_bf16(Fraction(f)), f.hex()


def test_rounding_is_monotone_and_idempotent_on_bf16_values():
    for h in range(0, 0x7F80, 7):
        v = oracle.bf16_to_f64(h)
        assert oracle.f64_to_bf16(v) == h
        assert oracle.f64_to_bf16(-v) == (h | 0x8000)


# --------------------------------------------------------------------------
# The GEMM
# --------------------------------------------------------------------------
ONE = 0x3F80


def _bf16_of_int(v: int) -> int:
    return _exact.round_bf16(v)


@pytest.mark.parametrize("K", [1, 7, 128, 1024, 2048, 7168])
def test_all_ones_gives_K(K):
    M, N, L = 3, 5, 2
    A = np.full((L, N, K), ONE, np.uint16)
    B = np.full((L, M, K), ONE, np.uint16)
    C = oracle.gemm(A, B)
    assert C.shape == (L, M, N)
    assert np.all(C == _bf16_of_int(K))


def test_identity_weights_pass_activations_through_bit_exactly():
    rng = np.random.default_rng(5)
    L, M, N, K = 2, 6, 40, 64
    A = np.zeros((L, N, K), np.uint16)
    for n in range(N):
        A[:, n, n] = ONE
    B = rng.integers(0, 2 ** 16, size=(L, M, K), dtype=np.uint16)
    B[(B & 0x7F80) == 0x7F80] = ONE            # keep inputs finite
    C = oracle.gemm(A, B)
    expect = B[:, :, :N].copy()
    expect[(expect & 0x7FFF) == 0] = 0          # -0 * 1 + 0 sums to +0
    assert np.array_equal(C, expect)


def test_single_nonzero_per_row_gives_rounded_scaled_copy():
    rng = np.random.default_rng(9)
    L, M, N, K = 1, 4, 33, 48
    A = np.zeros((L, N, K), np.uint16)
    perm = rng.integers(0, K, size=N)
    scale = rng.integers(0x3C00, 0x4400, size=N).astype(np.uint16)
    for n in range(N):
        A[0, n, perm[n]] = scale[n]
    B = rng.integers(0x3800, 0x4800, size=(L, M, K)).astype(np.uint16)
    B[rng.random(B.shape) < 0.5] |= 0x8000
    C = oracle.gemm(A, B)
    for m in range(M):
        for n in range(N):
            exact = _exact.value(int(scale[n])) * _exact.value(int(B[0, m, perm[n]]))
            assert C[0, m, n] == _exact.round_bf16(exact), (m, n)


@pytest.mark.parametrize("L,M,N,K", [(1, 1, 1, 1), (1, 2, 3, 5), (2, 3, 4, 8),
                                     (3, 5, 2, 16), (2, 4, 7, 9)])
def test_brute_force_exact_rationals(L, M, N, K):
    from split_bf16_gemm_swapped_gb300 import synthetic
    A = synthetic.normal_bf16((L, N, K), seed=100 + K, stream=0, sigma=0.02)
    B = synthetic.normal_bf16((L, M, K), seed=100 + K, stream=1, sigma=1.0)
    C = oracle.gemm(A, B)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                s = sum(_exact.value(int(A[l, n, k])) * _exact.value(int(B[l, m, k]))
                        for k in range(K))
                assert C[l, m, n] == _exact.round_bf16(s), (l, m, n)
                assert Fraction(oracle.dot_f64(A, B, l, m, n)) == s


def test_orientation_and_batch_index_on_a_structured_case():
    """C[l, m, n] = sum_k A[l, n, k] * B[l, m, k] with distinct small ints."""
    L, M, N, K = 2, 4, 4, 5
    rng = np.random.default_rng(13)
    Ai = rng.integers(-6, 7, size=(L, N, K))
    Bi = rng.integers(-6, 7, size=(L, M, K))
    enc = np.vectorize(lambda v: _exact.round_bf16(int(v)))
    A = enc(Ai).astype(np.uint16)
    B = enc(Bi).astype(np.uint16)
    C = oracle.gemm(A, B)
    ref = np.einsum("lnk,lmk->lmn", Ai, Bi)      # exact small integers
    assert np.array_equal(C, enc(ref).astype(np.uint16))
    # a transposed output or a mixed-up batch index would not match
    assert not np.array_equal(ref, ref.transpose(0, 2, 1))
    assert not np.array_equal(ref, ref[::-1])


def test_float64_sum_matches_numpy_matmul_then_exact_rounding():
    """Larger K: the f64 sum equals numpy's f64 matmul to within f64 rounding,
    and rounding that sum once reproduces the oracle's output."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 1, 3, 64, 2048
    A = synthetic.normal_bf16((L, N, K), seed=21, stream=0, sigma=0.02)
    B = synthetic.normal_bf16((L, M, K), seed=21, stream=1, sigma=1.0)
    af = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bf = (B.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.einsum("lmk,lnk->lmn", bf, af)
    C = oracle.gemm(A, B)
    for m in range(M):
        for n in range(N):
            s = oracle.dot_f64(A, B, 0, m, n)
            assert abs(s - ref[0, m, n]) <= 1e-12 * np.sum(np.abs(bf[0, m] * af[0, n]))
            assert C[0, m, n] == _exact.round_bf16(Fraction(s))


def test_threaded_and_element_paths_agree_with_the_plain_gemm():
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 5, 96, 256
    A = synthetic.normal_bf16((L, N, K), seed=31, stream=0, sigma=0.02)
    B = synthetic.normal_bf16((L, M, K), seed=31, stream=1, sigma=1.0)
    C = oracle.gemm(A, B)
    C4, used = oracle.gemm_threaded(A, B, 4)
    assert used >= 1
    assert np.array_equal(C, C4)
    idx = np.array([0, 17, L * M * N - 1, M * N + 3])
    assert np.array_equal(oracle.elements(A, B, idx), C.reshape(-1)[idx])


def test_pins_catch_planted_mistakes():
    """Mistakes planted on the CPU, by feeding the oracle altered operands,
    must change the output that the exact brute force pins: a dropped last k
    term, a swapped pair of weight rows, a wrong batch slice."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 3, 5, 16
    A = synthetic.normal_bf16((L, N, K), seed=41, stream=0, sigma=0.02)
    B = synthetic.normal_bf16((L, M, K), seed=41, stream=1, sigma=1.0)
    exact = np.array([[[_exact.round_bf16(sum(
        _exact.value(int(A[l, n, k])) * _exact.value(int(B[l, m, k]))
        for k in range(K))) for n in range(N)] for m in range(M)]
        for l in range(L)], dtype=np.uint16)
    assert np.array_equal(oracle.gemm(A, B), exact)
    planted = {
        "dropped k": oracle.gemm(A[:, :, :-1], B[:, :, :-1]),
        "rows swapped": oracle.gemm(A[:, [1, 0, 2, 3, 4]], B),
        "batch mixed": oracle.gemm(A[::-1].copy(), B),
    }
    for name, out in planted.items():
        assert not np.array_equal(out, exact), name


# --------------------------------------------------------------------------
# The GEMM with a bias
# --------------------------------------------------------------------------
def test_bias_alone_passes_through_bit_exactly():
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 3, 37, 16
    A = np.zeros((L, N, K), np.uint16)
    B = synthetic.normal_bf16((L, M, K), 51, 1, 1.0)
    bias = synthetic.normal_bf16((L, N), 51, 0, 0.5)
    C = oracle.gemm_bias(A, B, bias)
    expect = np.broadcast_to(bias[:, None, :], (L, M, N)).copy()
    expect[(expect & 0x7FFF) == 0] = 0
    assert np.array_equal(C, expect)


def test_bias_adds_before_the_single_rounding():
    """All-ones A and B with K=3 and a bias of 1/4 give exactly 3.25 (a bf16
    value); random small cases match the exact rational sum plus bias,
    rounded once."""
    rng = np.random.default_rng(3)
    L, M, N, K = 1, 2, 5, 3
    A = np.full((L, N, K), ONE, np.uint16)
    B = np.full((L, M, K), ONE, np.uint16)
    bias = np.full((L, N), _exact.round_bf16(Fraction(1, 4)), np.uint16)
    C = oracle.gemm_bias(A, B, bias)
    assert np.all(C == _exact.round_bf16(Fraction(13, 4)))          # 3.25 is a bf16
    from split_bf16_gemm_swapped_gb300 import synthetic
    for trial in range(4):
        L, M, N, K = 2, 3, 4, 6
        A = synthetic.normal_bf16((L, N, K), 60 + trial, 0, 0.02)
        B = synthetic.normal_bf16((L, M, K), 60 + trial, 1, 1.0)
        bias = synthetic.normal_bf16((L, N), 60 + trial, 2, 0.1)
        C = oracle.gemm_bias(A, B, bias)
        for l in range(L):
            for m in range(M):
                for n in range(N):
                    s = sum(_exact.value(int(A[l, n, k])) * _exact.value(int(B[l, m, k]))
                            for k in range(K)) + _exact.value(int(bias[l, n]))
                    assert C[l, m, n] == _exact.round_bf16(s)


def test_zero_bias_is_the_plain_gemm():
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 1, 4, 33, 64
    A = synthetic.normal_bf16((L, N, K), 70, 0, 0.02)
    B = synthetic.normal_bf16((L, M, K), 70, 1, 1.0)
    assert np.array_equal(oracle.gemm_bias(A, B, np.zeros((L, N), np.uint16)), oracle.gemm(A, B))


# --------------------------------------------------------------------------
# A16W4: E2M1 weight codes with E8M0 scales per 32 k (the Muse Spark AMD dev
# page, e8m0_f32 and fp4x8_bf16)
# --------------------------------------------------------------------------
def _golden_e2m1():
    rows = []
    for line in (GOLDEN / "e2m1_values.txt").read_text().splitlines():
        if line.strip() and not line.startswith("#"):
            code, value = line.split()[:2]
            rows.append((int(code, 16), float(value)))
    return rows


def test_e2m1_decoding_matches_the_hand_derived_table():
    rows = _golden_e2m1()
    assert [c for c, _ in rows] == list(range(16))
    for code, value in rows:
        got = oracle.e2m1_to_f64(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), code


def test_e8m0_is_the_binary32_with_that_exponent_field():
    """The page: code << 23, read as an f32, is the scale (codes 1..254)."""
    codes = np.arange(1, 255, dtype=np.uint32)
    ref = (codes << 23).view(np.float32).astype(np.float64)
    got = np.array([oracle.e8m0_to_f64(int(c)) for c in codes])
    assert np.array_equal(got, ref)
    assert math.isnan(oracle.e8m0_to_f64(255))


def _exact_w4(Aq, As, l, n, k):
    byte = int(Aq[l, n, k // 2])
    code = byte & 0xF if k % 2 == 0 else byte >> 4
    value = Fraction(_golden_e2m1()[code][1])
    return value * Fraction(2) ** (int(As[l, n, k // 32]) - 127)


def test_nibble_order_and_scale_blocks_on_a_hand_made_row():
    """Low nibble is the even k; the scale of k is byte k // 32 of its row.
    One-hot activations pick single weights out of the product."""
    K, N = 64, 2
    Aq = np.zeros((1, N, K // 2), np.uint8)
    As = np.full((1, N, K // 32), 127, np.uint8)
    Aq[0, 0, 0] = 0x72          # k=0: code 2 (1.0), k=1: code 7 (6.0)
    Aq[0, 0, 16] = 0xB5         # k=32: code 5 (3.0), k=33: code 0xB (-1.5)
    As[0, 0, 1] = 130           # k = 32..63 of row 0 scaled by 2^3
    Aq[0, 1, 31] = 0x10         # row 1, k=62: code 0, k=63: code 1 (0.5)
    As[0, 1, 1] = 125           # ... scaled by 2^-2
    W = oracle.w4_dequant(Aq, As)
    assert (W[0, 0, 0], W[0, 0, 1], W[0, 0, 32], W[0, 0, 33]) == (1.0, 6.0, 24.0, -12.0)
    assert (W[0, 1, 62], W[0, 1, 63]) == (0.0, 0.125)
    M = 4
    B = np.zeros((1, M, K), np.uint16)
    for m, k in enumerate([0, 1, 33, 63]):
        B[0, m, k] = 0x3F80     # 1.0
    C = oracle.gemm_w4a16(Aq, As, B)
    expect = [[1.0, 0.0], [6.0, 0.0], [-12.0, 0.0], [0.0, 0.125]]
    for m in range(M):
        for n in range(N):
            assert oracle.bf16_to_f64(int(C[0, m, n])) == expect[m][n], (m, n)


def test_w4a16_equals_the_bf16_gemm_of_its_exact_bf16_weights():
    """Every weight the codes encode (in the scale range used) is a bf16
    value, so the A16W4 product is the (separately pinned) bf16 oracle's."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 3, 20, 256
    Aq, As = synthetic.w4_weights(L, N, K, seed=51)
    B = synthetic.normal_bf16((L, M, K), seed=51, stream=1, sigma=1.0)
    W = oracle.w4_dequant(Aq, As)
    Wb = np.vectorize(oracle.f64_to_bf16)(W).astype(np.uint16)
    assert np.array_equal((Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), W)
    assert np.array_equal(oracle.gemm_w4a16(Aq, As, B), oracle.gemm(Wb, B))


@pytest.mark.parametrize("L,M,N,K", [(1, 1, 1, 32), (1, 2, 3, 64), (2, 3, 2, 96)])
def test_w4a16_brute_force_exact_rationals(L, M, N, K):
    from split_bf16_gemm_swapped_gb300 import synthetic
    Aq, As = synthetic.w4_weights(L, N, K, seed=61 + K)
    B = synthetic.normal_bf16((L, M, K), seed=61 + K, stream=1, sigma=1.0)
    C = oracle.gemm_w4a16(Aq, As, B)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                s = sum(_exact_w4(Aq, As, l, n, k) * _exact.value(int(B[l, m, k])) for k in range(K))
                assert C[l, m, n] == _exact.round_bf16(s), (l, m, n)


@pytest.mark.parametrize("scale,expect", [(127, 1.0), (130, 8.0), (124, 0.125)])
def test_w4a16_all_ones_closed_form(scale, expect):
    """Every weight code 2 (1.0) with one scale, every activation 1.0:
    C = K * 2^(scale - 127) exactly."""
    L, M, N, K = 1, 2, 3, 1024
    Aq = np.full((L, N, K // 2), 0x22, np.uint8)
    As = np.full((L, N, K // 32), scale, np.uint8)
    B = np.full((L, M, K), 0x3F80, np.uint16)
    C = oracle.gemm_w4a16(Aq, As, B)
    assert np.all(np.vectorize(oracle.bf16_to_f64)(C) == K * expect)


def test_w4a16_pins_catch_planted_mistakes():
    """Altered operands (the mistakes an oracle could make) change the exact
    result: nibbles swapped, one scale per row, scale blocks out of order."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 1, 2, 3, 64
    Aq, As = synthetic.w4_weights(L, N, K, seed=71)
    B = synthetic.normal_bf16((L, M, K), seed=71, stream=1, sigma=1.0)
    exact = np.array([[[_exact.round_bf16(sum(_exact_w4(Aq, As, 0, n, k) * _exact.value(int(B[0, m, k]))
                                             for k in range(K))) for n in range(N)] for m in range(M)]],
                     dtype=np.uint16)
    assert np.array_equal(oracle.gemm_w4a16(Aq, As, B), exact)
    swapped = ((Aq & 0x0F) << 4) | (Aq >> 4)            # high nibble read as the even k
    one_scale = np.repeat(As[:, :, :1], K // 32, axis=2)  # the first block's scale for the whole row
    reversed_blocks = np.ascontiguousarray(As[:, :, ::-1])  # block b scaled by block (nb - 1 - b)
    assert np.any(As[:, :, 0] != As[:, :, 1])
    for name, (q, s) in {"nibbles swapped": (swapped, As), "scale per row": (Aq, one_scale),
                         "scale blocks": (Aq, reversed_blocks)}.items():
        assert not np.array_equal(oracle.gemm_w4a16(q, s, B), exact), name


def test_w4_elements_equal_exact_rationals_one_by_one():
    """The per-element A16W4 path, pinned directly: every output of a small
    batched shape against the exact rational sum rounded once, and on a
    larger shape against the whole-GEMM path (itself pinned above) at the
    first, last and scattered flat indices l*M*N + m*N + n."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 3, 4, 64
    Aq, As = synthetic.w4_weights(L, N, K, seed=81)
    B = synthetic.normal_bf16((L, M, K), seed=81, stream=1, sigma=1.0)
    idx = np.arange(L * M * N)
    got = oracle.w4_elements(Aq, As, B, idx)
    for i in idx:
        l, m, n = i // (M * N), (i // N) % M, i % N
        s = sum(_exact_w4(Aq, As, l, n, k) * _exact.value(int(B[l, m, k])) for k in range(K))
        assert got[i] == _exact.round_bf16(s), (l, m, n)
    L, M, N, K = 2, 5, 300, 512
    Aq, As = synthetic.w4_weights(L, N, K, seed=82)
    B = synthetic.normal_bf16((L, M, K), seed=82, stream=1, sigma=1.0)
    full = oracle.gemm_w4a16(Aq, As, B).reshape(-1)
    idx = np.unique(np.concatenate([[0, 1, N - 1, N, M * N, L * M * N - 1],
                                    np.random.default_rng(5).integers(0, L * M * N, 400)]))
    assert np.array_equal(oracle.w4_elements(Aq, As, B, idx), full[idx])
    # an index read with M and N exchanged would pick other outputs
    swapped = (idx // (M * N)) * M * N + (idx % N) * M + (idx // N) % M
    assert not np.array_equal(full[swapped], full[idx])


# --------------------------------------------------------------------------
# A16W8: E4M3 weights with E8M0 scales per 32 k
# --------------------------------------------------------------------------
def _golden_e4m3():
    rows = []
    for line in (GOLDEN / "e4m3_values.txt").read_text().splitlines():
        if line.startswith("0x"):
            code, value = line.split()[:2]
            rows.append((int(code, 16), float(value)))
    return rows


def test_e4m3_decoding_matches_the_hand_derived_table():
    rows = _golden_e4m3()
    assert len(rows) >= 18
    for code, value in rows:
        got = oracle.e4m3_to_f64(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), hex(code)


def test_e4m3_decoding_matches_torch_on_all_256_codes():
    """Every code against PyTorch's float8_e4m3fn (a library conversion):
    the same value, sign of zero included, and not-a-number for 0x7F, 0xFF."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


_E4M3_TORCH = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).tolist()


def _exact_w8(Aq, As, l, n, k):
    """The weight from PyTorch's E4M3 conversion (independent of the oracle)
    and the scale's power of two, as an exact rational."""
    value = Fraction(_E4M3_TORCH[int(Aq[l, n, k])])
    return value * Fraction(2) ** (int(As[l, n, k // 32]) - 127)


def test_w8_byte_order_and_scale_blocks_on_a_hand_made_row():
    """Code k of a row is byte k; the scale of k is byte k // 32 of the row's
    scales.  One-hot activations pick single weights out of the product."""
    K, N = 64, 2
    Aq = np.zeros((1, N, K), np.uint8)
    As = np.full((1, N, K // 32), 127, np.uint8)
    Aq[0, 0, 0], Aq[0, 0, 1] = 0x38, 0x4B     # 1.0, 5.5
    Aq[0, 0, 33] = 0xBC                        # -1.5, in the second scale block
    As[0, 0, 1] = 130                          # x 2^3
    Aq[0, 1, 63] = 0x01                        # 2^-9
    As[0, 1, 1] = 120                          # x 2^-7
    W = oracle.w8_dequant(Aq, As)
    assert (W[0, 0, 0], W[0, 0, 1], W[0, 0, 33], W[0, 1, 63]) == (1.0, 5.5, -12.0, 2.0 ** -16)
    M = 4
    B = np.zeros((1, M, K), np.uint16)
    for m, k in enumerate([0, 1, 33, 63]):
        B[0, m, k] = 0x3F80
    C = oracle.gemm_w8a16(Aq, As, B)
    expect = [[1.0, 0.0], [5.5, 0.0], [-12.0, 0.0], [0.0, 2.0 ** -16]]
    for m in range(M):
        for n in range(N):
            assert oracle.bf16_to_f64(int(C[0, m, n])) == expect[m][n], (m, n)


@pytest.mark.parametrize("L,M,N,K", [(1, 1, 1, 32), (1, 2, 3, 64), (2, 3, 2, 96)])
def test_w8a16_brute_force_exact_rationals(L, M, N, K):
    from split_bf16_gemm_swapped_gb300 import synthetic
    Aq, As = synthetic.w8_weights(L, N, K, seed=91 + K)
    B = synthetic.normal_bf16((L, M, K), seed=91 + K, stream=1, sigma=1.0)
    C = oracle.gemm_w8a16(Aq, As, B)
    for l in range(L):
        for m in range(M):
            for n in range(N):
                s = sum(_exact_w8(Aq, As, l, n, k) * _exact.value(int(B[l, m, k])) for k in range(K))
                assert C[l, m, n] == _exact.round_bf16(s), (l, m, n)


def test_w8a16_equals_the_bf16_gemm_of_its_exact_bf16_weights():
    """Every weight the 8-bit codes encode (in the scale range used) is a
    bf16 value (4 significant bits), so the A16W8 product is the bf16
    oracle's on those weights."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 2, 3, 20, 256
    Aq, As = synthetic.w8_weights(L, N, K, seed=95)
    B = synthetic.normal_bf16((L, M, K), seed=95, stream=1, sigma=1.0)
    W = oracle.w8_dequant(Aq, As)
    Wb = np.vectorize(oracle.f64_to_bf16)(W).astype(np.uint16)
    assert np.array_equal((Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), W)
    assert np.array_equal(oracle.gemm_w8a16(Aq, As, B), oracle.gemm(Wb, B))


def test_w8a16_all_ones_closed_form():
    """Every weight code 0x38 (1.0) with scale 2^2, every activation 1.0:
    C = 4 K exactly."""
    L, M, N, K = 1, 2, 3, 1024
    Aq = np.full((L, N, K), 0x38, np.uint8)
    As = np.full((L, N, K // 32), 129, np.uint8)
    B = np.full((L, M, K), 0x3F80, np.uint16)
    assert np.all(np.vectorize(oracle.bf16_to_f64)(oracle.gemm_w8a16(Aq, As, B)) == 4.0 * K)


def test_w8a16_pins_catch_planted_mistakes():
    """Altered operands (the mistakes an oracle could make) change the exact
    result: bytes swapped in pairs, one scale per row, scale blocks reversed."""
    from split_bf16_gemm_swapped_gb300 import synthetic
    L, M, N, K = 1, 2, 3, 64
    Aq, As = synthetic.w8_weights(L, N, K, seed=97)
    B = synthetic.normal_bf16((L, M, K), seed=97, stream=1, sigma=1.0)
    exact = np.array([[[_exact.round_bf16(sum(_exact_w8(Aq, As, 0, n, k) * _exact.value(int(B[0, m, k]))
                                             for k in range(K))) for n in range(N)] for m in range(M)]],
                     dtype=np.uint16)
    assert np.array_equal(oracle.gemm_w8a16(Aq, As, B), exact)
    swapped = np.ascontiguousarray(Aq.reshape(L, N, K // 2, 2)[..., ::-1].reshape(L, N, K))
    one_scale = np.repeat(As[:, :, :1], K // 32, axis=2)
    reversed_blocks = np.ascontiguousarray(As[:, :, ::-1])
    assert np.any(As[:, :, 0] != As[:, :, 1])
    for name, (q, s) in {"bytes swapped": (swapped, As), "scale per row": (Aq, one_scale),
                         "scale blocks": (Aq, reversed_blocks)}.items():
        assert not np.array_equal(oracle.gemm_w8a16(q, s, B), exact), name
