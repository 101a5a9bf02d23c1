"""GPU parity: the sm_103a split-K GEMM (through the C ABI) against the CPU
oracle, element by element, on seeded synthetic inputs.

Tolerance: one bf16 ulp of the oracle's value, or 1e-3*sqrt(K)*max|A|*max|B|
for outputs near zero; bit-exact on the closed forms (all-ones, identity
weights, one nonzero per row, small integers).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only collection
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import synthetic, workloads  # noqa: E402
from tests import _tol  # noqa: E402
from tests._gpu import DEV, assert_parity, gemm_gpu, oracle_full, to_dev, to_host  # noqa: E402

ONE = 0x3F80


def _draw(L, M, N, K, seed, outlier_p=0.0, scale=1.0):
    a = synthetic.normal_bf16((L, N, K), seed, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0, outlier_p, scale)
    return a, b


def test_tiny_workload_full_parity():
    w = workloads.TINY
    a, b = w.make_a(), w.make_b()
    c = gemm_gpu(a, b, split_k=w.split_k)
    assert_parity(c, oracle_full(a, b), a, b, w.K)


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 13, 16, 17, 31, 32, 33, 63, 64, 65, 100, 128, 129])
def test_every_split_and_token_tail(split, M):
    L, N, K = 1, 300, 1024          # N=300: two full 128-row tiles and a ragged one
    a, b = _draw(L, M, N, K, seed=1000 + M)
    c = gemm_gpu(a, b, split_k=split)
    assert_parity(c, oracle_full(a, b), a, b, K)


@pytest.mark.parametrize("M,N,K,L,split,kind", [
    (3, 300, 8192, 1, 1, (6, 2, 0, 1)),     # CTAs alone on their SMs: 6 stages, two issuers
    (5, 1000, 4096, 8, 2, (6, 2, 1, 1)),    # the same with a dedicated mailbox
    (8, 2560, 4096, 8, 2, (3, 1, 0, 2)),    # 16 K tiles a CTA: 3 stages, mailbox aliased on the ring
    (16, 1280, 8192, 4, 4, (3, 1, 0, 2)),
])
def test_deep_rings_and_depth_first_mailboxes(M, N, K, L, split, kind):
    """The plans of grids of lone CTAs (deep even rings, two issuers) and of
    long K slices at 2 CTAs/SM (a third stage before a mailbox of their own)
    against the oracle."""
    p = sk.splitk_plan(M, N, K, L, split)
    assert (p.stages, p.mma_issuers, p.mailbox_dedicated, p.ctas_per_sm) == kind
    a, b = _draw(L, M, N, K, seed=2100 + M)
    c = gemm_gpu(a, b, split_k=split)
    assert_parity(c, oracle_full(a, b), a, b, K)
    assert np.array_equal(c, gemm_gpu(a, b, plan=p))


def test_seeded_random_shapes_match_the_oracle():
    """40 seeded shapes (ragged K multiples of 8, ragged N, batches, every
    split and the planner's own), each through whatever plan the planner
    picks, against the oracle."""
    rng = np.random.default_rng(2400)
    kinds = set()
    for i in range(40):
        M = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 20, 32, 40, 64]))
        N = int(rng.integers(1, 9)) * 128 - int(rng.choice([0, 0, 8, 40]))
        K = int(rng.integers(1, 65)) * 128 - 8 * int(rng.integers(0, 3))
        L = int(rng.choice([1, 1, 2]))
        split = int(rng.choice([0, 1, 2, 4, 8]))
        if split and -(-K // 128) < split:
            split = 1
        a, b = _draw(L, M, N, K, seed=2400 + i)
        p = sk.splitk_plan(M, N, K, L, split)
        kinds.add((p.stages, p.mma_issuers, p.mailbox_dedicated, p.reduce_scatter, p.b_resident, p.a_tmem_tiles))
        c = gemm_gpu(a, b, split_k=split)
        assert_parity(c, oracle_full(a, b), a, b, K)
    assert len(kinds) >= 8                  # the draw reaches many plan families


@pytest.mark.parametrize("split", [1, 4])
def test_batched_L_and_ragged_N(split):
    L, M, N, K = 3, 7, 200, 2048
    a, b = _draw(L, M, N, K, seed=77)
    c = gemm_gpu(a, b, split_k=split)
    assert_parity(c, oracle_full(a, b), a, b, K)


@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_all_ones_gives_K_exactly(split):
    L, M, N, K = 2, 5, 384, 2048
    a = np.full((L, N, K), ONE, np.uint16)
    b = np.full((L, M, K), ONE, np.uint16)
    c = gemm_gpu(a, b, split_k=split)
    assert np.all(c == 0x4500)       # 2048 in bf16


@pytest.mark.parametrize("split", [1, 2, 8])
def test_identity_weights_pass_activations_bit_exactly(split):
    L, M, N, K = 2, 20, 250, 1024
    a = np.zeros((L, N, K), np.uint16)
    for n in range(N):
        a[:, n, n] = ONE
    b = synthetic.normal_bf16((L, M, K), 5, synthetic.STREAM_B, 1.0)
    c = gemm_gpu(a, b, split_k=split)
    expect = b[:, :, :N].copy()
    expect[(expect & 0x7FFF) == 0] = 0
    assert np.array_equal(c, expect)


def test_single_nonzero_per_row_bit_exact():
    rng = np.random.default_rng(9)
    L, M, N, K = 1, 9, 256, 2048
    a = np.zeros((L, N, K), np.uint16)
    perm = rng.integers(0, K, size=N)
    a[0, np.arange(N), perm] = rng.integers(0x3C00, 0x4400, size=N).astype(np.uint16)
    b = synthetic.normal_bf16((L, M, K), 6, synthetic.STREAM_B, 1.0)
    c = gemm_gpu(a, b, split_k=4)
    assert np.array_equal(c, oracle.gemm(a, b))


@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_small_integers_are_exact_for_every_split(split):
    rng = np.random.default_rng(split)
    L, M, N, K = 1, 16, 256, 1024
    vals = np.array([0x0000, 0x3F80, 0x4000, 0x4040, 0x4080, 0x40A0, 0x40C0, 0x40E0, 0x4100,
                     0xBF80, 0xC000, 0xC040, 0xC080, 0xC100], np.uint16)   # 0, +-1..8
    a = vals[rng.integers(0, vals.size, size=(L, N, K))]
    b = vals[rng.integers(0, vals.size, size=(L, M, K))]
    c = gemm_gpu(a, b, split_k=split)
    assert np.array_equal(c, oracle.gemm(a, b))


def test_deterministic_run_to_run():
    w = workloads.DECODE_M16.with_(N=1024)
    a, b = w.make_a(), w.make_b()
    ta, tb = to_dev(a), to_dev(b)
    first = None
    for _ in range(10):
        c = to_host(sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k))
        if first is None:
            first = c
        assert np.array_equal(c, first)


def _mailbox_bytes(p, M):
    """Bytes of the plan's dedicated mailbox region (0 when aliased)."""
    ncm = min(M, p.mma_n)
    if p.split_k == 1 or not p.mailbox_dedicated:
        return 0
    if p.reduce_scatter:
        return ncm * 512
    return (p.split_k - 1) * min(4 * p.mailbox_quads, ncm) * 512


def _ring(base, M=None):
    """`base` as the page's ring design: activations ride the weight ring,
    no tensor-memory staging, one MMA issuer."""
    p = sk.Plan.from_buffer_copy(base)
    p.b_resident = 0
    p.b_loader = 0
    p.l2_prefetch = 0
    p.a_tmem_tiles = 0
    p.mma_issuers = 1
    p.tmem_cols = max(32, p.mma_n)
    p.smem_bytes = (1024 + p.stages * (32768 + p.mma_n * 256)
                    + _mailbox_bytes(p, M if M is not None else p.mma_n) + 256)
    return p


def _variant(base, stages, dedicated, quads, M, trigger=0):
    """A rank-0-reduction plan; `quads` is capped to what an aliased mailbox
    (the drained weight ring) holds."""
    p = _ring(base)
    p.reduce_scatter = 0
    p.stages = stages
    p.mailbox_dedicated = dedicated
    p.pdl_trigger = trigger
    ncm = min(M, p.mma_n)
    nq = -(-ncm // 4)
    quads = min(quads, nq) if quads < 4 else min(quads, max(4, nq))
    if not dedicated and p.split_k > 1:
        fits = lambda q: (p.split_k - 1) * min(4 * q, ncm) * 512 <= stages * 32768
        if not fits(quads):
            quads = 4
            while quads + 4 <= nq and fits(quads + 4):
                quads += 4
    p.mailbox_quads = quads
    p.reduce_rounds = -(-nq // quads)
    cols = min(4 * quads, ncm)
    ded = (p.split_k - 1) * cols * 512 if (dedicated and p.split_k > 1) else 0
    p.smem_bytes = 1024 + stages * (32768 + p.mma_n * 256) + ded + 256
    return p


@pytest.mark.parametrize("M", [1, 3, 6, 16, 30, 64, 100, 128])
@pytest.mark.parametrize("split", [2, 8])
def test_reduction_rounds_and_mailbox_placements(M, split):
    """Force 16-column reduction rounds (several rounds once M > 16), with the
    mailbox in its own region and aliased onto rank 0's drained weight ring."""
    L, N, K = 1, 256, 2048
    a, b = _draw(L, M, N, K, seed=500 + M)
    ref = oracle_full(a, b)
    base = sk.splitk_plan(M, N, K, L, split)
    few = min(4, base.mailbox_quads) if base.mailbox_quads < 4 else 4
    for stages, ded, quads, trig in [(2, 1, few, 0), (3, 0, few, 1), (2, 0, base.mailbox_quads, 0),
                                     (4, 1, base.mailbox_quads, 1)]:
        p = _variant(base, stages, ded, quads, M, trig)
        if p.smem_bytes > 232448:
            continue
        c = gemm_gpu(a, b, plan=p)
        assert_parity(c, ref, a, b, K)


def test_no_pdl_flag_gives_identical_bits():
    w = workloads.DECODE_M1.with_(N=1024)
    a, b = w.make_a(), w.make_b()
    p = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
    c0 = gemm_gpu(a, b, plan=p)
    c1 = gemm_gpu(a, b, plan=p, flags=sk.FLAG_NO_PDL)
    assert np.array_equal(c0, c1)


@pytest.mark.parametrize("K,split", [(8, 1), (136, 2), (1000, 4), (1032, 4), (1032, 8), (2040, 8),
                                     (7176, 8), (520, 1)])
def test_ragged_K_tails_and_uneven_slices(K, split):
    """K not a multiple of 128*split: ranks own floor or ceil of the K tiles,
    and TMA reads zeros past K (a whole box past K included)."""
    L, M, N = 2, 5, 200
    a, b = _draw(L, M, N, K, seed=800 + K)
    c = gemm_gpu(a, b, split_k=split)
    assert_parity(c, oracle_full(a, b), a, b, K)


def test_ragged_K_all_ones_is_exact():
    for K, split in [(1000, 4), (1032, 8), (264, 2)]:
        L, M, N = 1, 3, 256
        a = np.full((L, N, K), ONE, np.uint16)
        b = np.full((L, M, K), ONE, np.uint16)
        c = gemm_gpu(a, b, split_k=split)
        expect = oracle.gemm(a[:, :1, :], b[:, :1, :])[0, 0, 0]     # bf16 of K
        assert np.all(c == expect), (K, split)


def _scatter(base, M, stages=None):
    p = _ring(base)
    if stages is not None:
        p.stages = stages
    ncm = min(M, p.mma_n)
    p.reduce_scatter = 1
    p.mailbox_dedicated = 1
    p.mailbox_quads = -(-ncm // 4)
    p.reduce_rounds = 1
    p.smem_bytes = 1024 + p.stages * (32768 + p.mma_n * 256) + ncm * 512 + 256
    return p


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("M", [1, 5, 16, 33, 64, 100, 128])
def test_scattered_reduction_matches_rank0_bit_for_bit(M, split):
    """Each rank summing 128/split rows in rank order gives the bits rank 0
    gives summing the whole tile (same additions, same order)."""
    L, N, K = 2, 300, 2040
    a, b = _draw(L, M, N, K, seed=900 + M + split)
    base = _ring(sk.splitk_plan(M, N, K, L, split), M)
    c0 = gemm_gpu(a, b, plan=base)
    p = _scatter(base, M)
    if p.smem_bytes > 232448:
        p = _scatter(base, M, stages=2)
    c1 = gemm_gpu(a, b, plan=p)
    assert np.array_equal(c0, c1)
    assert_parity(c1, oracle_full(a, b), a, b, K)


@pytest.mark.parametrize("M,N,K,split", [(1, 7168, 2048, 4), (16, 4096, 7168, 8), (5, 300, 1000, 2),
                                         (33, 203, 1032, 4), (64, 256, 2048, 1), (128, 384, 2048, 8)])
def test_bias_epilogue(M, N, K, split):
    """C = B A^T + bias, the bias added in FP32 before the one rounding; both
    reduction modes (rank 0 and scattered) carry it."""
    L = 2
    a, b = _draw(L, M, N, K, seed=1100 + M)
    bias = synthetic.normal_bf16((L, N), 1100 + M, synthetic.STREAM_OUTLIER, 0.5)
    ta, tb = to_dev(a), to_dev(b)
    tbias = to_dev(bias)
    torch.cuda.synchronize()
    tc = sk.splitk_gemm_bf16_bias(ta, tb, tbias, split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    ref = oracle.gemm_bias(a, b, bias)
    from tests import _tol
    ok, rep = _tol.check(to_host(tc), ref, K, _tol.max_abs_bf16(a), _tol.max_abs_bf16(b))
    assert ok, rep
    # a zero bias gives the plain GEMM's bits
    tz = sk.splitk_gemm_bf16_bias(ta, tb, torch.zeros_like(tbias), split_k=split)
    plain = sk.splitk_gemm_bf16(ta, tb, split_k=split)
    torch.cuda.synchronize()
    assert torch.equal(tz.view(torch.int16), plain.view(torch.int16))


def _tmem_cols(mma_n, tiles, issuers=1):
    acc = max(32, mma_n) * issuers
    need = acc if tiles == 0 else (acc + 63) // 64 * 64 + 64 * tiles
    return next(c for c in (32, 64, 128, 256, 512) if c >= need)


def _staged(base, stages, tmem_tiles, issuers=1, b_resident=1, M=None, b_loader=0):
    """`base` with every activation K tile in its own buffer, the first
    `tmem_tiles` weight K tiles staged in tensor memory and `issuers` MMA
    threads; None if the plan cannot hold (shared memory, or tensor memory of
    the CTAs an SM fits)."""
    if stages % issuers:
        return None                   # a stage would have two consumers
    p = sk.Plan.from_buffer_copy(base)
    ded = _mailbox_bytes(base, M if M is not None else base.mma_n)
    if not base.mailbox_dedicated and base.split_k > 1:
        round_bytes = (base.split_k - 1) * min(4 * base.mailbox_quads, base.mma_n) * 512
        if round_bytes > stages * 32768:
            return None
    p.stages = stages
    p.b_resident = b_resident
    p.b_loader = b_loader
    p.a_tmem_tiles = tmem_tiles
    p.mma_issuers = issuers
    p.tmem_cols = _tmem_cols(p.mma_n, tmem_tiles, issuers)
    b_tiles = max(stages, p.k_tiles_per_cta) if b_resident else stages
    p.smem_bytes = 1024 + stages * 32768 + b_tiles * p.mma_n * 256 + ded + 256
    if p.smem_bytes > 232448 or 233472 // (p.smem_bytes + 1024) * p.tmem_cols > 512:
        return None
    return p


@pytest.mark.parametrize("M,split", [(1, 4), (4, 1), (16, 8), (16, 2), (33, 4), (64, 2), (128, 8), (100, 8)])
def test_staged_weights_and_resident_activations_give_the_same_bits(M, split):
    """Weight K tiles copied into tensor memory (tcgen05.cp) and read by the
    MMA from there, and activation tiles loaded all at once, give the bits of
    the plain ring: the same products accumulate in the same order."""
    L, N, K = 2, 300, 2048 + 8 * split
    a, b = _draw(L, M, N, K, seed=1200 + M + split)
    base = _ring(sk.splitk_plan(M, N, K, L, split), M)
    c0 = gemm_gpu(a, b, plan=base)
    assert_parity(c0, oracle_full(a, b), a, b, K)
    ran = 0
    for stages in (2, 3):
        for tiles in (0, 1, 2, 3):
            for loader in (0, 1):
                p = _staged(base, stages, tiles, M=M, b_loader=loader)
                if p is None:
                    continue
                c1 = gemm_gpu(a, b, plan=p)
                assert np.array_equal(c0, c1), (stages, tiles, loader)
                ran += 1
    assert ran >= 1


@pytest.mark.parametrize("M,split", [(1, 4), (3, 1), (16, 8), (16, 2), (33, 4), (64, 2), (100, 8)])
def test_two_mma_issuers(M, split):
    """A second MMA thread takes the odd K tiles into its own accumulator:
    parity with the oracle, exact closed forms, and every staging variant of
    the two-issuer plan gives the same bits (same products, same order)."""
    L, N, K = 2, 300, 2048 + 8 * split
    a, b = _draw(L, M, N, K, seed=1300 + M + split)
    base = sk.splitk_plan(M, N, K, L, split)
    p2 = _staged(base, 2, 0, issuers=2, b_resident=0, M=M)
    assert p2 is not None
    c2 = gemm_gpu(a, b, plan=p2)
    assert_parity(c2, oracle_full(a, b), a, b, K)
    ran = 0
    for stages in (2, 3):
        for tiles in (0, 1, 2, 3):
            p = _staged(base, stages, tiles, issuers=2, M=M, b_loader=tiles % 2)
            if p is None:
                continue
            p.l2_prefetch = 1
            assert np.array_equal(gemm_gpu(a, b, plan=p), c2), (stages, tiles)
            ran += 1
    assert ran >= 1
    ones = np.full((L, N, K), ONE, np.uint16)
    c = gemm_gpu(ones, np.full((L, M, K), ONE, np.uint16), plan=p2)
    assert np.all(c == oracle.gemm(ones[:1, :1, :], np.full((1, 1, K), ONE, np.uint16))[0, 0, 0])


def test_two_issuers_need_an_even_ring():
    """With an odd stage count a ring stage would have two consumers; the
    library refuses such a plan before launching anything."""
    base = _ring(sk.splitk_plan(1, 512, 2048, 1, 4), 1)
    p = sk.Plan.from_buffer_copy(base)
    p.stages = 3
    p.mma_issuers = 2
    p.tmem_cols = _tmem_cols(p.mma_n, 0, 2)
    p.smem_bytes = 1024 + 3 * (32768 + p.mma_n * 256) + _mailbox_bytes(base, 1) + 256
    a, b = _draw(1, 1, 512, 2048, seed=7)
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_gemm_bf16_planned(to_dev(a), to_dev(b), None, p)
    assert e.value.name == "SPLITK_ERR_BAD_PLAN"


@pytest.mark.parametrize("M,K", [(1, 1000), (3, 2056), (8, 1032), (16, 520)])
def test_thread_loaded_activations_with_ragged_K_and_bias(M, K):
    """Activations loaded by the epilogue threads (zeros past K, rows past M
    left unwritten) give the bits of the TMA-loaded plan, with a bias too."""
    L, N, split = 2, 200, 4
    a, b = _draw(L, M, N, K, seed=1400 + M)
    base = sk.splitk_plan(M, N, K, L, split)
    p0 = _staged(base, 2, 0, issuers=2, M=M, b_loader=0)
    p1 = _staged(base, 2, 0, issuers=2, M=M, b_loader=1)
    assert p0 is not None and p1 is not None
    c0 = gemm_gpu(a, b, plan=p0)
    assert np.array_equal(gemm_gpu(a, b, plan=p1), c0)
    assert_parity(c0, oracle_full(a, b), a, b, K)


# --------------------------------------------------------------------------
# A16W4: 4-bit weights decoded on chip
# --------------------------------------------------------------------------
def _w4_draw(L, M, N, K, seed):
    aq, a_s = synthetic.w4_weights(L, N, K, seed)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0)
    return aq, a_s, b


def _u8_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


@pytest.mark.parametrize("M,N,K,split", [(1, 300, 1024, 4), (4, 256, 1024, 1), (16, 200, 2048, 8),
                                         (5, 384, 3072, 4), (32, 256, 1024, 2), (9, 130, 512, 2),
                                         (17, 300, 896, 1)])
def test_w4a16_matches_the_oracle(M, N, K, split):
    L = 2
    aq, a_s, b = _w4_draw(L, M, N, K, seed=1500 + M + K)
    tc = sk.splitk_gemm_w4a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    ref = oracle.gemm_w4a16(aq, a_s, b)
    w = oracle.w4_dequant(aq, a_s)
    max_w = float(np.max(np.abs(w)))
    ok, rep = _tol.check(to_host(tc), ref, K, max_w, _tol.max_abs_bf16(b))
    assert ok, rep


@pytest.mark.parametrize("M", [3, 9])
def test_w4a16_grids_of_several_waves_match_the_oracle(M):
    """512 CTAs: the planner trades TMEM slots for a third CTA per SM."""
    L, N, K, split = 8, 2048, 2048, 4
    aq, a_s, b = _w4_draw(L, M, N, K, seed=1550 + M)
    p = sk.splitk_plan_w4a16(M, N, K, L, split)
    assert (p.a_tmem_tiles, p.mma_issuers, p.ctas_per_sm) == (1, 1, 3)
    tc = sk.splitk_gemm_w4a16_planned(_u8_dev(aq), _u8_dev(a_s), to_dev(b), None, p)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    ref = oracle.gemm_w4a16(aq, a_s, b)
    max_w = float(np.max(np.abs(oracle.w4_dequant(aq, a_s))))
    ok, rep = _tol.check(to_host(tc), ref, K, max_w, _tol.max_abs_bf16(b))
    assert ok, rep


@pytest.mark.parametrize("M,split", [(1, 4), (8, 2), (8, 4), (16, 8), (32, 2)])
def test_w4a16_equals_the_bf16_kernel_on_the_decoded_weights(M, split):
    """The decoded weights are exact bf16 values, so the A16W4 product equals,
    bit for bit, the bf16 kernel's on those weights with as many MMA issuers
    (the same products accumulated in the same order: with two, the even and
    odd K tiles in two accumulators added at the end)."""
    L, N, K = 1, 256, 2048
    aq, a_s, b = _w4_draw(L, M, N, K, seed=1600 + M)
    wb = np.vectorize(oracle.f64_to_bf16)(oracle.w4_dequant(aq, a_s)).astype(np.uint16)
    ta, ts, tb = _u8_dev(aq), _u8_dev(a_s), to_dev(b)
    w4 = sk.splitk_plan_w4a16(M, N, K, L, split)
    for issuers in (1, 2):
        if issuers > w4.a_tmem_tiles:
            continue
        p4 = sk.Plan.from_buffer_copy(w4)
        p4.mma_issuers = issuers
        p4.tmem_cols = _tmem_cols(p4.mma_n, p4.a_tmem_tiles, issuers)
        c4 = to_host(sk.splitk_gemm_w4a16_planned(ta, ts, tb, None, p4))
        cb = gemm_gpu(wb, b, plan=_bf16_plan_like(p4, M, N, K, L, split))
        assert np.array_equal(c4, cb), issuers


def _w4_variant(base, slots, stage, loader, issuers=1, decoders=None):
    """`base` with `slots` TMEM slots, the bf16 shared-memory stage on or
    off, the given activation loader, MMA issuers and decoding warpgroups;
    shared memory grown for the stage and padded until the slots of the CTAs
    sharing an SM fit its TMEM."""
    p = sk.Plan.from_buffer_copy(base)
    if decoders is not None:
        p.w4_decoders = decoders
    p.a_tmem_tiles = slots
    p.mma_issuers = issuers
    p.tmem_cols = _tmem_cols(p.mma_n, slots, issuers)
    p.b_loader = loader
    p.smem_bytes += max(0, stage - base.w4_smem_tiles) * 32768
    p.w4_smem_tiles = stage
    p.smem_bytes = max(p.smem_bytes, 233472 // (512 // p.tmem_cols + 1) + 16) // 16 * 16
    while 233472 // (p.smem_bytes + 1024) * p.tmem_cols > 512:
        p.smem_bytes += 16
    return p


@pytest.mark.parametrize("M,K,variants", [
    (3, 1024 * 4, [(s, 0, ld, i) for s in (1, 2, 3) for ld in (0, 1) for i in (1, 2) if i <= s]),
    (3, 512 * 4, [(s, st, ld, i) for s, st in ((3, 1), (3, 0), (2, 0), (1, 0)) for ld in (0, 1) for i in (1, 2)
                  if i <= s]),
    (1, 256 * 4, [(s, st, ld, i) for s, st in ((1, 1), (1, 0), (2, 0)) for ld in (0, 1) for i in (1, 2) if i <= s]),
])
def test_w4a16_slot_counts_and_activation_loaders_agree(M, K, variants):
    """1, 2 or 3 TMEM slots (tiles decoded ahead), the last tile decoded into
    a bf16 stage in shared memory or into a reused slot, TMA- or
    thread-loaded activations, and padded shared memory all give the same
    bits for a given number of MMA issuers (one or two accumulators)."""
    L, N = 1, 256
    aq, a_s, b = _w4_draw(L, M, N, K, seed=1700 + K)
    base = sk.splitk_plan_w4a16(M, N, K, L, 4)
    ta, ts, tb = _u8_dev(aq), _u8_dev(a_s), to_dev(b)
    outs = {1: [], 2: []}
    for slots, stage, loader, issuers in variants:
        for decoders in (1, 2):            # one or two decoding warpgroups: the same bits
            p = _w4_variant(base, slots, stage, loader, issuers, decoders)
            for _ in range(3):             # repeated: a race shows as a difference
                outs[issuers].append(to_host(sk.splitk_gemm_w4a16_planned(ta, ts, tb, None, p)))
        torch.cuda.synchronize()
        assert sk.splitk_get_status() == 0
    ref = oracle.gemm_w4a16(aq, a_s, b)
    max_w = float(np.max(np.abs(oracle.w4_dequant(aq, a_s))))
    for group in outs.values():
        for o in group[1:]:
            assert np.array_equal(o, group[0])
        if group:
            ok, rep = _tol.check(group[0], ref, K, max_w, _tol.max_abs_bf16(b))
            assert ok, rep


def test_w4a16_one_hot_activations_read_out_every_decoded_weight():
    """With one-hot activations (token m reads k = 32 m + o), C[m][n] is the
    decoded weight w(n, 32 m + o) itself; 32 offsets read out every weight of
    a shape holding all 16 codes and scale codes 2..252 (2 is the smallest
    whose products stay normal), compared bit for bit with the oracle's exact
    dequantisation."""
    L, M, N, K = 1, 32, 256, 1024
    rng = np.random.default_rng(1800)
    aq = rng.integers(0, 256, size=(L, N, K // 2), dtype=np.uint8)
    a_s = rng.integers(2, 253, size=(L, N, K // 32), dtype=np.uint8)
    a_s[0, :, 0] = 2
    a_s[0, :, 1] = 127
    a_s[0, :, 3] = 252                     # largest documented code
    want = np.vectorize(oracle.f64_to_bf16)(oracle.w4_dequant(aq, a_s)).astype(np.uint16)
    want[want == 0x8000] = 0               # a sum holding +0 terms reads a -0 weight as +0
    ta, ts = _u8_dev(aq), _u8_dev(a_s)
    for o in range(32):
        b = np.zeros((L, M, K), np.uint16)
        b[0, np.arange(M), 32 * np.arange(M) + o] = ONE
        c = to_host(sk.splitk_gemm_w4a16(ta, ts, to_dev(b), split_k=2))
        assert np.array_equal(c[0], want[0][:, 32 * np.arange(M) + o].T), o
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0


def _bf16_plan_like(w4, M, N, K, L, split):
    """A bf16 plan accumulating like the A16W4 plan `w4`: the page's ring with
    one issuer, or with two (even and odd K tiles in two accumulators)."""
    ring = _ring(sk.splitk_plan(M, N, K, L, split), M)
    if w4.mma_issuers == 1:
        return ring
    pb = _staged(ring, 2, 0, issuers=2, M=M) or _staged(ring, 4, 0, issuers=2, M=M)
    assert pb is not None
    return pb


def test_w4a16_extreme_scales_equal_the_bf16_kernel():
    """Scale codes from 1 (products of 0.5 that are bf16 subnormals) to 252,
    small activations keeping the sums finite: the A16W4 GEMM equals the bf16
    kernel on the exactly dequantised weights, bit for bit."""
    L, M, N, K, split = 1, 4, 256, 2048, 4
    rng = np.random.default_rng(1900)
    aq = rng.integers(0, 256, size=(L, N, K // 2), dtype=np.uint8)
    codes = np.array([1, 2, 100, 127, 142, 143, 200, 252], np.uint8)
    a_s = codes[rng.integers(0, len(codes), size=(L, N, K // 32))]
    b = synthetic.normal_bf16((L, M, K), 1900, synthetic.STREAM_B, 2.0 ** -20)
    wb = np.vectorize(oracle.f64_to_bf16)(oracle.w4_dequant(aq, a_s)).astype(np.uint16)
    w4 = sk.splitk_plan_w4a16(M, N, K, L, split)
    c4 = to_host(sk.splitk_gemm_w4a16_planned(_u8_dev(aq), _u8_dev(a_s), to_dev(b), None, w4))
    cb = gemm_gpu(wb, b, plan=_bf16_plan_like(w4, M, N, K, L, split))
    assert np.array_equal(c4, cb)


def test_w4a16_activations_of_any_magnitude_equal_the_bf16_kernel():
    """Tokens of 2^100, of 2^-100, beyond f16's range, and one spanning 30
    binades: the A16W4 GEMM equals the bf16 kernel on the dequantised
    weights, bit for bit (every product normal in both)."""
    L, M, N, K, split = 1, 5, 256, 2048, 4
    aq, a_s, _ = _w4_draw(L, M, N, K, seed=1950)
    rng = np.random.default_rng(1950)
    vals = rng.standard_normal((L, M, K))
    vals[0, 0] *= 2.0 ** 100
    vals[0, 1] *= 2.0 ** -100
    vals[0, 2] *= 1e6
    vals[0, 3] *= np.exp2(rng.integers(-10, 20, size=K))
    b = np.vectorize(oracle.f64_to_bf16)(vals).astype(np.uint16)
    wb = np.vectorize(oracle.f64_to_bf16)(oracle.w4_dequant(aq, a_s)).astype(np.uint16)
    w4 = sk.splitk_plan_w4a16(M, N, K, L, split)
    c4 = to_host(sk.splitk_gemm_w4a16_planned(_u8_dev(aq), _u8_dev(a_s), to_dev(b), None, w4))
    cb = gemm_gpu(wb, b, plan=_bf16_plan_like(w4, M, N, K, L, split))
    assert np.array_equal(c4, cb)


def test_w4a16_all_ones_closed_form():
    L, M, N, K = 1, 2, 256, 2048
    aq = np.full((L, N, K // 2), 0x22, np.uint8)          # every weight 1.0 ...
    a_s = np.full((L, N, K // 32), 129, np.uint8)         # ... times 4
    b = np.full((L, M, K), ONE, np.uint16)
    c = to_host(sk.splitk_gemm_w4a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=4))
    torch.cuda.synchronize()
    assert np.all(c == oracle.f64_to_bf16(4.0 * K))


@pytest.mark.parametrize("L,N", [(65535, 128), (1, 65535 * 128)])
def test_w4a16_the_largest_grid_dimensions_index_correctly(L, N):
    """As the bf16 case: weight row n of matrix l has one nonzero 4-bit code,
    s = (l + n) % 7 - 3 (E2M1 holds 0, +-1, +-2, +-3 exactly), at k = 0, with
    scale code 127 (x1), so C[l][m][n] = s * B[l][m][0] exactly."""
    M, K = 2, 128
    s = (np.arange(L)[:, None] + np.arange(N)[None, :]) % 7 - 3                   # [L, N]
    e2m1 = np.array([0xD, 0xC, 0xA, 0x0, 0x2, 0x4, 0x5], np.uint8)                 # -3 .. 3
    aq = np.zeros((L, N, K // 2), np.uint8)
    aq[:, :, 0] = e2m1[s + 3]                                                        # low nibble: k = 0
    a_s = np.full((L, N, K // 32), 127, np.uint8)
    b = (((np.arange(L * M * K) % 13) - 6) * 0.25).astype(np.float32).reshape(L, M, K)
    b_bits = (b.view(np.uint32) >> 16).astype(np.uint16)                            # exact
    expect = s[:, None, :].astype(np.float64) * b[:, :, 0:1].astype(np.float64)    # [L, M, N]
    c = sk.splitk_gemm_w4a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b_bits), split_k=0)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    got = to_host(c).astype(np.uint32) << 16
    assert np.array_equal(got.view(np.float32).astype(np.float64), expect)
    del c
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- persistent plans
def _persistent(M, N, K, L, split, clusters=None, stages=None, quads=None, mma_n=None, b_stages=0):
    """The persistent plan of the shape at `split` (the deepest ring unless
    `stages` is given, reduction rounds of `quads` 4-column groups if given,
    the activations on the weight ring unless `b_stages` gives them a ring
    of their own), with `clusters` as its grid bound if given."""
    props = torch.cuda.get_device_properties(DEV)
    cands = sk.splitk_plan_candidates_for(M, N, K, L, split, props.multi_processor_count,
                                          props.shared_memory_per_multiprocessor,
                                          props.shared_memory_per_block_optin)
    ps = [p for p in cands if p.persistent and (quads is None or p.mailbox_quads == quads)
          and (mma_n is None or p.mma_n == mma_n) and p.b_stages == b_stages]
    assert ps, "no persistent candidate"
    p = max(ps, key=lambda q: q.stages) if stages is None else next(q for q in ps if q.stages == stages)
    p = sk.Plan.from_buffer_copy(p)
    if clusters is not None:
        p.grid[1] = clusters
    return p


@pytest.mark.parametrize("M,N,K,L,split,clusters", [
    (64, 1000, 4096, 2, 4, 3),      # a ragged weight tile; 3 clusters walk 16 tiles
    (128, 384, 2048, 3, 8, 2),
    (100, 700, 3000, 1, 2, 1),      # ragged K and a ragged token tile; one cluster walks all tiles
    (129, 300, 2040, 2, 4, None),   # two token tiles, the second with one column
    (33, 520, 1024, 2, 8, 4),
    (16, 1024, 8192, 2, 4, 5),
    (1, 640, 2048, 1, 2, 2),
])
def test_persistent_kernel_matches_the_oracle(M, N, K, L, split, clusters):
    """Clusters that each walk several output tiles, with the ring running on
    across tiles and two accumulators, against the oracle."""
    a, b = _draw(L, M, N, K, seed=2700 + M + split)
    p = _persistent(M, N, K, L, split, clusters)
    c = gemm_gpu(a, b, plan=p)
    assert_parity(c, oracle_full(a, b), a, b, K)
    assert np.array_equal(c, gemm_gpu(a, b, plan=p))          # run to run


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("M", [5, 64, 128])
def test_persistent_kernel_equals_the_scattered_per_tile_kernel_bit_for_bit(M, split):
    """The same partials (one issuer, the same K slices) summed over ranks in
    the same order: the persistent and the per-tile scattered kernels give
    the same bits, at every ring depth and cluster count."""
    L, N, K = 2, 640, 4096
    a, b = _draw(L, M, N, K, seed=2800 + M + split)
    base = _ring(sk.splitk_plan(M, N, K, L, split), M)
    ref_plan = _scatter(base, M)
    if ref_plan.smem_bytes > 232448:
        ref_plan = _scatter(base, M, stages=2)
    want = gemm_gpu(a, b, plan=ref_plan)
    for stages, clusters in [(None, None), (2, 1), (3, 7)]:
        try:
            p = _persistent(M, N, K, L, split, clusters, stages)
        except StopIteration:
            continue                                          # that depth does not fit
        assert np.array_equal(gemm_gpu(a, b, plan=p), want), (stages, clusters)


@pytest.mark.parametrize("M,split,stages,b_stages,clusters", [
    (128, 8, 4, 2, 3),     # the weight ring twice the activation ring's depth
    (128, 4, 3, 3, 2),     # equal depths, separate rings
    (64, 4, 5, 2, None),
    (100, 2, 2, 5, 1),     # a deeper activation ring; one cluster walks every tile
    (37, 8, 5, 3, 4),      # depths with no common factor
    (16, 2, 5, 3, 5),
])
def test_persistent_activation_ring_of_its_own(M, split, stages, b_stages, clusters):
    """The activations on a ring of their own depth beside the weight ring:
    the same MMAs on the same K tiles in the same order, so the same bits as
    the plan whose activations ride the weight ring, and the oracle's
    values."""
    L, N, K = 2, 520, 3000
    a, b = _draw(L, M, N, K, seed=3200 + M + split)
    p = _persistent(M, N, K, L, split, clusters, stages, b_stages=b_stages)
    assert (p.stages, p.b_stages) == (stages, b_stages)
    c = gemm_gpu(a, b, plan=p)
    assert np.array_equal(c, gemm_gpu(a, b, plan=_persistent(M, N, K, L, split, clusters, 2)))
    assert_parity(c, oracle_full(a, b), a, b, K)


@pytest.mark.parametrize("M,quads", [(100, 4), (128, 16), (64, 8), (37, 4)])
def test_persistent_reduction_rounds(M, quads):
    """A tile reduced in rounds of a few 4-column groups through a smaller
    mailbox (the last round ragged when M is): the same bits as one round a
    tile, and the oracle's values."""
    L, N, K, split = 2, 520, 2048, 4
    a, b = _draw(L, M, N, K, seed=3000 + M)
    tile = next(t for t in (16, 32, 64, 128) if t >= min(M, 128))      # the shape's own token tile
    p = _persistent(M, N, K, L, split, clusters=3, quads=quads, mma_n=tile)
    assert p.reduce_rounds > 1
    c = gemm_gpu(a, b, plan=p)
    one = _persistent(M, N, K, L, split, clusters=3, quads=-(-min(M, tile) // 4), stages=2, mma_n=tile)
    assert np.array_equal(c, gemm_gpu(a, b, plan=one))
    assert_parity(c, oracle_full(a, b), a, b, K)


@pytest.mark.parametrize("M", [100, 128, 129])
def test_persistent_64_token_tiles_share_weight_tiles(M):
    """More than 64 tokens as several 64-token tiles per weight tile (the
    clusters working side by side read each weight tile in turn): the same
    bits as the shape's own token tile, and the oracle's values."""
    L, N, K, split = 2, 520, 2048, 8
    a, b = _draw(L, M, N, K, seed=3100 + M)
    p64 = _persistent(M, N, K, L, split, clusters=5, mma_n=64)
    c = gemm_gpu(a, b, plan=p64)
    own = _persistent(M, N, K, L, split, clusters=3, mma_n=128)
    assert np.array_equal(c, gemm_gpu(a, b, plan=own))
    assert_parity(c, oracle_full(a, b), a, b, K)


def test_persistent_kernel_closed_forms_and_bias():
    """All-ones inputs give C = K exactly; the bias is added before the one
    rounding, as by the oracle."""
    L, M, N, K, split = 2, 64, 1000, 4096, 4
    p = _persistent(M, N, K, L, split, clusters=5)
    ones = np.full((L, N, K), ONE, np.uint16)
    c = gemm_gpu(ones, np.full((L, M, K), ONE, np.uint16), plan=p)
    assert np.all(c == oracle.f64_to_bf16(float(K)))
    # a shape whose plan is persistent (76 tiles: two rounds of 38 clusters), through the bias entry point
    L, M, N, K = 1, 64, 9728 - 100, 1024
    assert sk.splitk_plan(M, N, K, L, split).persistent == 1
    a, b = _draw(L, M, N, K, seed=2900)
    bias = synthetic.normal_bf16((L, N), 2900, synthetic.STREAM_OUTLIER, 0.5)
    tc = sk.splitk_gemm_bf16_bias(to_dev(a), to_dev(b), to_dev(bias), split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert_parity(to_host(tc), oracle.gemm_bias(a, b, bias), a, b, K)


def test_w4a16_scale_codes_outside_the_contract_decode_as_documented():
    """Scale codes 0, 253, 254 and 255 (outside the documented 1..252): a
    block of 32 k with that code, every activation of the block 2^-10 and
    the rest zero, so C[n] = 32 * 2^-10 * w decoded.  Code 0 decodes as a
    zero scale, 253 and 254 as 2^126 and 2^127 (decoded weights past bf16's
    largest finite value are +-Inf), 255 as +Inf (NaN for the zero code)."""
    L, M, N, K = 1, 1, 256, 1024
    aq = np.zeros((L, N, K // 2), np.uint8)
    for n in range(N):                         # row n: every k holds e2m1 code n % 16
        aq[0, n, :] = (n % 16) * 0x11
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    b = np.zeros((L, M, K), np.uint16)
    b[0, 0, 32:64] = 0x3A80                    # 2^-10 on block 1
    for code in (0, 253, 254, 255):
        a_s = np.full((L, N, K // 32), 127, np.uint8)
        a_s[0, :, 1] = code
        c = to_host(sk.splitk_gemm_w4a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=2))
        torch.cuda.synchronize()
        assert sk.splitk_get_status() == 0
        got = (c.astype(np.uint32) << 16).view(np.float32)[0, 0].astype(np.float64)
        for n in range(N):
            w = e2m1[n % 16]
            if code == 0:
                assert got[n] == 0.0, (code, n)
                continue
            if w == 0 and code == 255:
                assert np.isnan(got[n]), (code, n)
                continue
            dec = w * np.inf if code == 255 else w * 2.0 ** (code - 127)
            if np.isfinite(dec) and abs(dec) >= 2.0 ** 128:
                dec = np.copysign(np.inf, w)
            assert got[n] == dec * 32 * 2.0 ** -10, (code, n, got[n], dec)


# ---------------------------------------------------------------- A16W8 (E4M3 weights)
def _w8_draw(L, M, N, K, seed):
    aq, a_s = synthetic.w8_weights(L, N, K, seed)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0)
    return aq, a_s, b


@pytest.mark.parametrize("M,N,K,split", [(1, 300, 1024, 4), (4, 256, 1024, 1), (16, 200, 2048, 8),
                                         (5, 384, 3072, 4), (32, 256, 1024, 2), (17, 300, 896, 1),
                                         (1, 7168, 2048, 4), (16, 4096, 7168, 8)])
def test_w8a16_matches_the_oracle(M, N, K, split):
    L = 2 if N < 1000 else 1
    aq, a_s, b = _w8_draw(L, M, N, K, seed=3200 + M + K)
    tc = sk.splitk_gemm_w8a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=split)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    ref = oracle.gemm_w8a16(aq, a_s, b)
    max_w = float(np.max(np.abs(oracle.w8_dequant(aq, a_s))))
    ok, rep = _tol.check(to_host(tc), ref, K, max_w, _tol.max_abs_bf16(b))
    assert ok, rep


@pytest.mark.parametrize("M,split", [(1, 4), (8, 2), (16, 8), (32, 2)])
def test_w8a16_equals_the_bf16_kernel_on_the_decoded_weights(M, split):
    """Every E4M3 weight times its power of two is an exact bf16 value, so
    the A16W8 product equals, bit for bit, the bf16 kernel's on the decoded
    weights with as many MMA issuers, and with one or two decoding
    warpgroups."""
    L, N, K = 1, 256, 2048
    aq, a_s, b = _w8_draw(L, M, N, K, seed=3300 + M)
    wb = np.vectorize(oracle.f64_to_bf16)(oracle.w8_dequant(aq, a_s)).astype(np.uint16)
    ta, ts, tb = _u8_dev(aq), _u8_dev(a_s), to_dev(b)
    w8 = sk.splitk_plan_w8a16(M, N, K, L, split)
    assert w8.weight_format == sk.WEIGHTS_E4M3_E8M0
    for issuers in (1, 2):
        if issuers > w8.a_tmem_tiles:
            continue
        for decoders in (1, 2):
            p8 = _w4_variant(w8, w8.a_tmem_tiles, w8.w4_smem_tiles, w8.b_loader, issuers, decoders)
            c8 = to_host(sk.splitk_gemm_w8a16_planned(ta, ts, tb, None, p8))
            cb = gemm_gpu(wb, b, plan=_bf16_plan_like(p8, M, N, K, L, split))
            assert np.array_equal(c8, cb), (issuers, decoders)


def test_w8a16_one_hot_activations_read_out_every_decoded_weight():
    """One-hot activations (token m reads k = 32 m + o) make C[m][n] the
    decoded weight w(n, 32 m + o); 32 offsets read out every weight of a
    shape holding all 254 finite codes and scale codes 3..246, compared bit
    for bit with the oracle's exact dequantisation."""
    L, M, N, K = 1, 32, 256, 1024
    rng = np.random.default_rng(3400)
    aq = rng.integers(0, 256, size=(L, N, K), dtype=np.uint8)
    aq[(aq & 0x7F) == 0x7F] ^= 1                   # no not-a-number codes
    aq[0, 0, :254] = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    a_s = rng.integers(3, 247, size=(L, N, K // 32), dtype=np.uint8)
    a_s[0, :, 0] = 3                               # smallest exact scale
    a_s[0, :, 1] = 127
    a_s[0, :, 3] = 246                             # largest exact scale
    want = np.vectorize(oracle.f64_to_bf16)(oracle.w8_dequant(aq, a_s)).astype(np.uint16)
    want[want == 0x8000] = 0                       # a sum holding +0 terms reads a -0 weight as +0
    ta, ts = _u8_dev(aq), _u8_dev(a_s)
    for o in range(32):
        b = np.zeros((L, M, K), np.uint16)
        b[0, np.arange(M), 32 * np.arange(M) + o] = ONE
        c = to_host(sk.splitk_gemm_w8a16(ta, ts, to_dev(b), split_k=2))
        assert np.array_equal(c[0], want[0][:, 32 * np.arange(M) + o].T), o
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0


def test_w8a16_slots_stage_and_decoders_agree():
    """1, 2 or 3 TMEM slots, the bf16 stage, the activation loaders and one
    or two decoding warpgroups: the same bits, run three times each."""
    L, M, N, K = 1, 3, 256, 512 * 4
    aq, a_s, b = _w8_draw(L, M, N, K, seed=3500)
    base = sk.splitk_plan_w8a16(M, N, K, L, 4)
    ta, ts, tb = _u8_dev(aq), _u8_dev(a_s), to_dev(b)
    outs = {1: [], 2: []}
    for slots, stage in ((3, 1), (3, 0), (2, 0), (1, 0)):
        for loader in (0, 1):
            for issuers in (1, 2):
                if issuers > slots:
                    continue
                for decoders in (1, 2):
                    p = _w4_variant(base, slots, stage, loader, issuers, decoders)
                    for _ in range(3):
                        outs[issuers].append(to_host(sk.splitk_gemm_w8a16_planned(ta, ts, tb, None, p)))
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    ref = oracle.gemm_w8a16(aq, a_s, b)
    max_w = float(np.max(np.abs(oracle.w8_dequant(aq, a_s))))
    for group in outs.values():
        for o in group[1:]:
            assert np.array_equal(o, group[0])
        ok, rep = _tol.check(group[0], ref, K, max_w, _tol.max_abs_bf16(b))
        assert ok, rep


def test_w8a16_all_ones_closed_form():
    """Every weight code 0x38 (1.0) with scale 2^2 and every activation 1.0:
    C = 4 K exactly."""
    L, M, N, K = 1, 4, 300, 2048
    aq = np.full((L, N, K), 0x38, np.uint8)
    a_s = np.full((L, N, K // 32), 129, np.uint8)
    b = np.full((L, M, K), ONE, np.uint16)
    c = to_host(sk.splitk_gemm_w8a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=4))
    torch.cuda.synchronize()
    assert np.all(c == oracle.f64_to_bf16(4.0 * K))


@pytest.mark.parametrize("bits", [4, 8])
def test_quantized_code_rings_agree(bits):
    """The packed codes in a ring of 1, 2 or 4 stages instead of all of a
    CTA's 7 tiles at once (each stage refilled once every decoder has read
    it): the same bits, within the oracle's tolerance, with one and two
    decoding warpgroups."""
    L, M, N, K, split = 1, 16, 512, 7168, 8
    if bits == 4:
        aq, a_s, b = _w4_draw(L, M, N, K, seed=3600)
        plan, run, ref = sk.splitk_plan_w4a16, sk.splitk_gemm_w4a16_planned, oracle.gemm_w4a16(aq, a_s, b)
        max_w = float(np.max(np.abs(oracle.w4_dequant(aq, a_s))))
    else:
        aq, a_s, b = _w8_draw(L, M, N, K, seed=3600)
        plan, run, ref = sk.splitk_plan_w8a16, sk.splitk_gemm_w8a16_planned, oracle.gemm_w8a16(aq, a_s, b)
        max_w = float(np.max(np.abs(oracle.w8_dequant(aq, a_s))))
    ta, ts, tb = _u8_dev(aq), _u8_dev(a_s), to_dev(b)
    base = plan(M, N, K, L, split)
    assert base.k_tiles_per_cta == 7
    outs = []
    for decoders in (1, 2):
        for stages in (7, 4, 2, 1):
            p = sk.Plan.from_buffer_copy(base)
            p.smem_bytes += max(0, stages - base.stages) * (8192 if bits == 4 else 16384)
            p.stages = stages
            p.w4_decoders = decoders
            for _ in range(2):
                outs.append(to_host(run(ta, ts, tb, None, p)))
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ok, rep = _tol.check(outs[0], ref, K, max_w, _tol.max_abs_bf16(b))
    assert ok, rep


def test_w8a16_not_a_number_codes_decode_as_documented():
    """The two E4M3 not-a-number codes are outside the contract; the header
    documents that they decode as +-480 times the scale.  One-hot
    activations read them out."""
    L, M, N, K = 1, 4, 128, 128
    aq = np.full((L, N, K), 0x38, np.uint8)          # 1.0 elsewhere
    aq[0, 0:64, 5] = 0x7F
    aq[0, 64:128, 5] = 0xFF
    a_s = np.full((L, N, K // 32), 120, np.uint8)    # 2^-7
    b = np.zeros((L, M, K), np.uint16)
    b[0, 0, 5] = ONE
    c = to_host(sk.splitk_gemm_w8a16(_u8_dev(aq), _u8_dev(a_s), to_dev(b), split_k=1))
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert np.all(c[0, 0, :64] == oracle.f64_to_bf16(480.0 * 2.0 ** -7))
    assert np.all(c[0, 0, 64:] == oracle.f64_to_bf16(-480.0 * 2.0 ** -7))
    assert np.all(c[0, 1:] == 0)
