"""The C ABI on a GPU: argument errors, guard bands around C, the host-I/O
entry point, CUDA-graph capture, and programmatic-dependent-launch chains."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import split_bf16_gemm_swapped_gb300 as sk  # noqa: E402
from split_bf16_gemm_swapped_gb300 import synthetic, workloads  # noqa: E402
from tests._gpu import DEV, assert_parity, gemm_gpu, to_dev, to_host  # noqa: E402


def _draw(L, M, N, K, seed):
    a = synthetic.normal_bf16((L, N, K), seed, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), seed, synthetic.STREAM_B, 1.0)
    return a, b


def test_plan_on_the_device_matches_the_described_device():
    props = torch.cuda.get_device_properties(DEV)
    p = sk.splitk_plan(1, 7168, 2048, 1, 4)
    q = sk.splitk_plan_for(1, 7168, 2048, 1, 4, props.multi_processor_count,
                           props.shared_memory_per_multiprocessor,
                           props.shared_memory_per_block_optin)
    assert p.as_dict() == q.as_dict()


def test_argument_errors_enqueue_nothing():
    lib = sk.load_library()
    ta = torch.zeros((256, 1024), dtype=torch.bfloat16, device=DEV)
    tb = torch.zeros((4, 1024), dtype=torch.bfloat16, device=DEV)
    tc = torch.full((4, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    a, b, c = ta.data_ptr(), tb.data_ptr(), tc.data_ptr()
    assert lib.splitk_gemm_bf16(a, b, c, 4, 256, 1004, 1, 1, s) == -1      # K % 8
    assert lib.splitk_gemm_bf16(a, b, c, 4, 256, 1024, 1, 3, s) == -3      # split 3
    assert lib.splitk_gemm_bf16(a, b, c, 4, 256, 128, 1, 2, s) == -1       # 1 K tile, 2 ranks
    assert lib.splitk_gemm_bf16(a + 2, b, c, 4, 256, 1024, 1, 1, s) == -2  # misaligned A
    assert lib.splitk_gemm_bf16(a, b, c, 0, 256, 1024, 1, 1, s) == -1
    p = sk.splitk_plan(4, 256, 1024, 1, 4)
    bad = sk.Plan.from_buffer_copy(p)
    bad.stages = 9
    assert lib.splitk_gemm_bf16_planned(a, b, c, 4, 256, 1024, 1, ctypes.byref(bad), 0, s) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.smem_bytes += 16
    assert lib.splitk_gemm_bf16_planned(a, b, c, 4, 256, 1024, 1, ctypes.byref(bad), 0, s) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.grid[1] += 1
    assert lib.splitk_gemm_bf16_planned(a, b, c, 4, 256, 1024, 1, ctypes.byref(bad), 0, s) == -10
    torch.cuda.synchronize()
    assert bool((tc == 7.0).all())


def test_a_host_output_tensor_is_refused_before_any_launch():
    a = torch.zeros((256, 1024), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((4, 1024), dtype=torch.bfloat16, device=DEV)
    host_c = torch.full((4, 256), 7.0, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="device"):
        sk.splitk_gemm_bf16(a, b, host_c)
    aq = torch.zeros((256, 512), dtype=torch.uint8, device=DEV)
    a_s = torch.full((256, 32), 127, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError, match="device"):
        sk.splitk_gemm_w4a16(aq, a_s, b, host_c)
    assert bool((host_c == 7.0).all())


@pytest.mark.parametrize("L,N", [(65535, 128), (1, 65535 * 128)])
def test_the_largest_grid_dimensions_index_correctly(L, N):
    """The grid's limits of 65,535 matrices (z) and 65,535 weight tiles (y).
    Weight row n of matrix l has one nonzero, s = (l + n) % 7 - 3, at k = 0,
    so C[l][m][n] = s * B[l][m][0] exactly: B holds multiples of 1/4 in
    [-1.5, 1.5], and every product is a bf16 value.  2.1 GB of weights."""
    M, K = 2, 128
    s = ((np.arange(L)[:, None] + np.arange(N)[None, :]) % 7 - 3).astype(np.float32)     # [L, N]
    b = (((np.arange(L * M * K) % 13) - 6) * 0.25).astype(np.float32).reshape(L, M, K)
    b_bits = (b.view(np.uint32) >> 16).astype(np.uint16)                                  # exact
    expect = s[:, None, :].astype(np.float64) * b[:, :, 0:1].astype(np.float64)          # [L, M, N]
    a = torch.zeros((L, N, K), dtype=torch.bfloat16, device=DEV)
    a[:, :, 0] = torch.from_numpy(s).to(DEV).to(torch.bfloat16)
    p = sk.splitk_plan(M, N, K, L, 0)
    assert tuple(p.grid)[1:] == ((N + 127) // 128, L)
    c = sk.splitk_gemm_bf16(a, to_dev(b_bits), split_k=0)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0, sk.splitk_get_fault()
    got = to_host(c).astype(np.uint32) << 16
    assert np.array_equal(got.view(np.float32).astype(np.float64), expect)
    del a, c
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,split", [(1, 300, 4), (5, 129, 2), (40, 200, 8), (128, 384, 1)])
def test_guard_bands_around_C_are_untouched(M, N, split):
    L, K = 2, 1024
    a, b = _draw(L, M, N, K, seed=M * 7 + N)
    pad = 4096
    buf = torch.full((pad + L * M * N + pad,), float("nan"), dtype=torch.bfloat16, device=DEV)
    canary = buf.view(torch.int16).clone()
    c = buf[pad:pad + L * M * N].view(L, M, N)
    sk.splitk_gemm_bf16(to_dev(a), to_dev(b), c, split_k=split)
    torch.cuda.synchronize()
    now = buf.view(torch.int16)
    assert torch.equal(now[:pad], canary[:pad]) and torch.equal(now[-pad:], canary[-pad:])
    assert_parity(to_host(c), oracle.gemm(a, b), a, b, K)


def test_unaligned_C_and_N_not_multiple_of_8_use_element_stores():
    L, M, N, K = 1, 3, 203, 1024
    a, b = _draw(L, M, N, K, seed=31)
    buf = torch.zeros((L * M * N + 1,), dtype=torch.bfloat16, device=DEV)
    c = buf[1:].view(L, M, N)                          # 2-byte aligned only
    sk.splitk_gemm_bf16(to_dev(a), to_dev(b), c, split_k=2)
    torch.cuda.synchronize()
    assert float(buf[0]) == 0.0
    assert_parity(to_host(c), oracle.gemm(a, b), a, b, K)


def test_host_io_entry_point_matches_the_device_path():
    w = workloads.DECODE_M1
    a, b = w.make_a(), w.make_b()
    ta, tb = to_dev(a), to_dev(b)
    ref = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    b_pin = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    c_pin = torch.zeros((w.L, w.M, w.N), dtype=torch.bfloat16).pin_memory()
    b_dev = torch.empty_like(tb)
    c_dev = torch.empty_like(ref)
    sk.splitk_gemm_bf16_hostio(ta, b_pin, c_pin, b_dev, c_dev, w.split_k)
    torch.cuda.synchronize()
    assert torch.equal(c_pin.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("M,N,K,L,split", [(1, 7168, 2048, 1, 4), (4, 300, 1024, 2, 2), (16, 4096, 7168, 1, 8)])
def test_zero_copy_entry_point_matches_the_device_path(M, N, K, L, split):
    """Activations read from, and the output written to, pinned host memory
    by the kernel itself: the device path's bits."""
    a, b = _draw(L, M, N, K, seed=2200 + M)
    want = gemm_gpu(a, b, split_k=split)
    ta = to_dev(a)
    b_pin = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).pin_memory()
    c_pin = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        sk.splitk_gemm_bf16_zerocopy(ta, b_pin, c_pin, split_k=split)
        torch.cuda.synchronize()
        assert sk.splitk_get_status() == 0
        assert np.array_equal(c_pin.view(torch.int16).numpy().view(np.uint16), want)


def test_zero_copy_refuses_unmapped_buffers_and_unstaged_shapes():
    L, M, N, K = 1, 1, 256, 1024
    a, b = _draw(L, M, N, K, seed=2300)
    ta = to_dev(a)
    b_pin = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    c_pin = torch.empty((L, M, N), dtype=torch.bfloat16).pin_memory()
    pageable_b = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    pageable_c = torch.empty((L, M, N), dtype=torch.bfloat16)
    for bb, cc in ((pageable_b, c_pin), (b_pin, pageable_c)):
        with pytest.raises(sk.SplitKError) as e:
            sk.splitk_gemm_bf16_zerocopy(ta, bb, cc, split_k=2)
        assert e.value.code == -12
    # a shape whose activations the epilogue threads do not load (wide tiles)
    a2, b2 = _draw(1, 64, 256, 8192, seed=2301)
    b2_pin = torch.from_numpy(b2.view(np.int16)).view(torch.bfloat16).pin_memory()
    c2_pin = torch.empty((1, 64, 256), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_gemm_bf16_zerocopy(to_dev(a2), b2_pin, c2_pin, split_k=1)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0


def test_calls_captured_in_a_cuda_graph_replay_identically():
    w = workloads.DECODE_M16.with_(N=1024)
    a, b = w.make_a(), w.make_b()
    ta, tb = to_dev(a), to_dev(b)
    eager = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)      # also caches A's map
    torch.cuda.synchronize()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            sk.splitk_gemm_bf16(ta, tb, out, split_k=w.split_k, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_pdl_chain_matches_serialised_launches():
    """C1 = B0 A1^T feeds the next call as its activations: the second kernel
    must read C1 only after the first one completed (griddepcontrol.wait)."""
    K1, N1, N2, M = 2048, 1024, 512, 8
    a1 = synthetic.normal_bf16((N1, K1), 61, synthetic.STREAM_A, 0.02)
    a2 = synthetic.normal_bf16((N2, N1), 62, synthetic.STREAM_A, 0.02)
    b0 = synthetic.normal_bf16((M, K1), 61, synthetic.STREAM_B, 1.0)
    ta1, ta2, tb0 = to_dev(a1), to_dev(a2), to_dev(b0)
    torch.cuda.synchronize()
    c1 = sk.splitk_gemm_bf16(ta1, tb0, split_k=4)
    c2 = sk.splitk_gemm_bf16(ta2, c1, split_k=4)                # PDL on
    torch.cuda.synchronize()
    p1 = sk.splitk_plan(M, N1, K1, 1, 4)
    p2 = sk.splitk_plan(M, N2, N1, 1, 4)
    d1 = sk.splitk_gemm_bf16_planned(ta1, tb0, None, p1, sk.FLAG_NO_PDL)
    torch.cuda.synchronize()
    d2 = sk.splitk_gemm_bf16_planned(ta2, d1, None, p2, sk.FLAG_NO_PDL)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), d1.view(torch.int16))
    assert torch.equal(c2.view(torch.int16), d2.view(torch.int16))
    assert_parity(to_host(c1), oracle.gemm(a1, b0), a1, b0, K1)


def test_tune_measures_candidates_and_returns_a_plan_that_computes_the_product():
    """splitk_tune times every candidate on this device over a few weight
    copies and returns the fastest; that plan passes the launch check and
    computes the product."""
    M, N, K, L = 2, 1024, 2048, 1
    a = synthetic.normal_bf16((L, N, K), 31, synthetic.STREAM_A, 0.02)
    b = synthetic.normal_bf16((L, M, K), 31, synthetic.STREAM_B, 1.0)
    ta = to_dev(a)
    a_list = [ta] + [ta.clone() for _ in range(3)]
    tb = to_dev(b)
    plan, us = sk.splitk_tune(a_list, tb, split_k=4, reps=8)
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert us > 0 and plan.split_k == 4
    props = torch.cuda.get_device_properties(DEV)
    assert sk.splitk_plan_check_for(plan, M, N, K, L, props.shared_memory_per_multiprocessor,
                                    props.shared_memory_per_block_optin) == 0
    c = sk.splitk_gemm_bf16_planned(a_list[2], tb, None, plan)
    torch.cuda.synchronize()
    assert_parity(to_host(c), oracle.gemm(a, b), a, b, K)


def test_trace_stamps_stay_in_their_buffer_are_ordered_and_stop_when_off():
    """splitk_set_trace: a buffer for fewer CTAs than the grid receives the
    stamps of the first CTAs only; a CTA's stamps taken by one thread are in
    time order, stamps a CTA never reaches stay as they were, words past the
    buffer's CTAs are untouched; tracing off stops every write."""
    w = workloads.DECODE_M1                             # 224 CTAs: 56 tiles x split 4
    a, b = w.make_a(), w.make_b()
    ta, tb = to_dev(a), to_dev(b)
    plan = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
    grid = plan.grid[0] * plan.grid[1] * plan.grid[2]
    traced = 100                                        # CTAs the buffer holds
    SENT = 0x5A5A5A5A5A5A5A5A
    buf = torch.full(((grid + 8) * sk.TRACE_SLOTS,), SENT, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    sk.splitk_set_trace(buf[: traced * sk.TRACE_SLOTS])
    try:
        c = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
        torch.cuda.synchronize()
    finally:
        sk.splitk_set_trace(None)
    assert sk.splitk_get_status() == 0
    assert_parity(to_host(c), oracle.gemm(a, b, threads=8), a, b, w.K)
    t = buf.cpu().numpy().view(np.uint64).reshape(grid + 8, sk.TRACE_SLOTS)
    assert np.all(t[traced:] == SENT)                  # past the buffer: untouched
    f = {name: i for i, name in enumerate(sk.TRACE_FIELDS)}
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    for cta in range(traced):
        r = t[cta]
        sm, rank = int(r[f["sm_rank"]]) & 0xFFFFFFFF, int(r[f["sm_rank"]]) >> 32
        assert sm < sms and rank == cta % w.split_k     # the cluster runs along grid x
        # thread 0: start, map acquired, first ring pass issued, set-up passed,
        # last weight issued, end
        chain = [r[f[k]] for k in ("start", "map_ready", "prefetched", "synced", "weights_issued", "end")]
        assert all(x != SENT for x in chain) and chain == sorted(chain), (cta, chain)
        # epilogue thread 0: accumulator complete, then partials published or summed
        assert r[f["mma_done"]] != SENT and r[f["mma_done"]] <= r[f["reduced"]] != SENT
        if rank == 0:
            assert r[f["reduced"]] <= r[f["stored"]] != SENT
        else:
            assert r[f["stored"]] == SENT               # only rank 0 stores
        assert r[f["start"]] <= r[f["mma_done"]]
    # tracing off: a second call writes nothing
    buf.fill_(SENT)
    c2 = sk.splitk_gemm_bf16(ta, tb, split_k=w.split_k)
    torch.cuda.synchronize()
    assert bool((buf == SENT).all())
    assert torch.equal(c.view(torch.int16), c2.view(torch.int16))


def test_release_frees_the_cache_and_later_calls_rebuild_it():
    """splitk_release frees the device tensor-map pool (and its host mirror);
    the next call encodes the maps again and computes the same bits."""
    a, b = _draw(1, 3, 700, 2048, 91)
    ta, tb = to_dev(a), to_dev(b)
    c1 = sk.splitk_gemm_bf16(ta, tb, split_k=4)
    torch.cuda.synchronize()
    info = sk.splitk_cache_info()
    assert info["device_bytes"] > 0 and info["host_bytes"] > 0 and info["maps"] >= 1
    sk.splitk_release()
    assert sk.splitk_cache_info() == {"device_bytes": 0, "host_bytes": 0, "maps": 0}
    c2 = sk.splitk_gemm_bf16(ta, tb, split_k=4)
    c3 = sk.splitk_gemm_bf16(ta, tb, split_k=2)          # another plan, the same weight map
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert sk.splitk_cache_info()["maps"] == 1
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    ref = oracle.gemm(a, b)
    assert_parity(to_host(c2), ref, a, b, 2048)
    assert_parity(to_host(c3), ref, a, b, 2048)


def test_persistent_plans_chain_with_pdl_and_replay_in_a_graph():
    """Persistent plans (the planner's choice at split 8 for long streams):
    a call whose activations are the previous call's output waits for it
    (programmatic dependent launch), and calls captured in a CUDA graph --
    the first one of the shape inside the capture -- replay bit for bit."""
    M, N1, K1, N2 = 16, 4864, 4096, 4864
    a1 = synthetic.normal_bf16((N1, K1), 71, synthetic.STREAM_A, 0.02)
    a2 = synthetic.normal_bf16((N2, N1), 72, synthetic.STREAM_A, 0.02)
    b0 = synthetic.normal_bf16((M, K1), 71, synthetic.STREAM_B, 1.0)
    ta1, ta2, tb0 = to_dev(a1), to_dev(a2), to_dev(b0)
    p1 = sk.splitk_plan(M, N1, K1, 1, 8)
    p2 = sk.splitk_plan(M, N2, N1, 1, 8)
    assert p1.persistent == 1 and p2.persistent == 1
    torch.cuda.synchronize()
    c1 = sk.splitk_gemm_bf16(ta1, tb0, split_k=8)
    c2 = sk.splitk_gemm_bf16(ta2, c1, split_k=8)               # PDL on
    torch.cuda.synchronize()
    d1 = sk.splitk_gemm_bf16_planned(ta1, tb0, None, p1, sk.FLAG_NO_PDL)
    torch.cuda.synchronize()
    d2 = sk.splitk_gemm_bf16_planned(ta2, d1, None, p2, sk.FLAG_NO_PDL)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), d1.view(torch.int16))
    assert torch.equal(c2.view(torch.int16), d2.view(torch.int16))
    assert_parity(to_host(c1), oracle.gemm(a1, b0), a1, b0, K1)
    # capture: a new weight pointer, so its tensor map is first made inside the capture
    ta3 = ta1.clone()
    out = torch.empty_like(c1)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            sk.splitk_gemm_bf16(ta3, tb0, out, split_k=8, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert sk.splitk_get_status() == 0
    assert torch.equal(out.view(torch.int16), c1.view(torch.int16))


@pytest.mark.parametrize("M,N,K,L,split", [(16, 7168, 16384, 1, 4), (4, 300, 1024, 2, 1), (33, 2048, 2048, 1, 2)])
def test_host_io_copy_kernels_chain_calls_in_order(M, N, K, L, split):
    """splitk_gemm_bf16_hostio with pinned buffers (copy kernels chained to
    the GEMM): three calls back to back on one stream with different
    activations and one set of device and host buffers each return their own
    product, as the device path does; pageable host buffers (the copy
    engines) the same."""
    a, _ = _draw(L, M, N, K, seed=2400 + M)
    ta = to_dev(a)
    bs = [synthetic.normal_bf16((L, M, K), 2400 + M + i, synthetic.STREAM_B, 1.0) for i in range(3)]
    wants = [gemm_gpu(a, b, split_k=split) for b in bs]
    b_dev = torch.empty((L, M, K), dtype=torch.bfloat16, device=DEV)
    c_dev = torch.empty((L, M, N), dtype=torch.bfloat16, device=DEV)
    for pinned in (True, False):
        b_hosts = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16) for b in bs]
        c_hosts = [torch.full((L, M, N), float("nan"), dtype=torch.bfloat16) for _ in bs]
        if pinned:
            b_hosts = [x.pin_memory() for x in b_hosts]
            c_hosts = [x.pin_memory() for x in c_hosts]
        for i in range(3):
            sk.splitk_gemm_bf16_hostio(ta, b_hosts[i], c_hosts[i], b_dev, c_dev, split_k=split)
        torch.cuda.synchronize()
        assert sk.splitk_get_status() == 0
        for i in range(3):
            assert np.array_equal(c_hosts[i].view(torch.int16).numpy().view(np.uint16), wants[i]), (pinned, i)
