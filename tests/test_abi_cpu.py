"""The C ABI without a GPU: the library loads, exports every symbol that
include/splitk.h declares, plans tactics on a described device, and rejects
bad arguments before touching CUDA."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import pytest

import split_bf16_gemm_swapped_gb300 as sk
from split_bf16_gemm_swapped_gb300 import _build

ROOT = Path(__file__).resolve().parent.parent
GB300 = dict(num_sms=152, smem_per_sm=233472, smem_per_block_optin=232448)


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build_splitk()


def declared_symbols():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = h.read_text()
        names |= set(re.findall(r"SPLITK_API\s+[\w\s\*]+?\b(splitk_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert "splitk_gemm_bf16" in names and "splitk_plan" in names
    lib = ctypes.CDLL(str(sk.library_path()))
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


_C_CONSUMER = r"""
#include <stdio.h>
#include "splitk.h"
int main(void) {
    splitk_plan_t p;
    int rc = splitk_plan_for(16, 4096, 7168, 1, 8, 152, 233472, 232448, &p);
    printf("%d %d %d %d %d %d %u %u %u %zu\n", rc, p.mma_n, p.stages, p.split_k, p.a_tmem_tiles,
           p.reduce_scatter, p.grid[0], p.grid[1], p.grid[2], p.smem_bytes);
    printf("%d\n", splitk_gemm_bf16(NULL, NULL, NULL, 1, 128, 128, 1, 1, NULL));
    return 0;
}
"""


def test_the_header_is_plain_c_and_a_c_program_links_the_library(tmp_path):
    """A C11 consumer compiles against include/splitk.h with every warning an
    error, links the library, and plans what the Python binding plans."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(_C_CONSUMER)
    lib = sk.library_path()
    exe = tmp_path / "consumer"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{ROOT / 'include'}",
                    str(src), "-o", str(exe), f"-L{lib.parent}", f"-l:{lib.name}", f"-Wl,-rpath,{lib.parent}"],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    p = sk.splitk_plan_for(16, 4096, 7168, 1, 8, **GB300)
    expect = (f"0 {p.mma_n} {p.stages} {p.split_k} {p.a_tmem_tiles} {p.reduce_scatter} "
              f"{p.grid[0]} {p.grid[1]} {p.grid[2]} {p.smem_bytes}")
    assert out[0] == expect
    assert int(out[1]) == -7                           # SPLITK_ERR_NULL, before any CUDA call


def test_a_missing_library_raises_instead_of_falling_back(monkeypatch, tmp_path):
    """No CPU fallback: without the built library every entry point raises."""
    monkeypatch.setattr(_build, "SPLITK_LIB", tmp_path / "libmissing.so")
    monkeypatch.setattr(sk, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        sk.load_library()
    with pytest.raises(RuntimeError, match="missing"):
        sk.splitk_plan_for(1, 7168, 2048, 1, 4, **GB300)


def test_an_output_on_another_device_is_refused():
    import torch
    a = torch.empty((128, 256), dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError, match="device"):
        sk._out(torch.empty((4, 128), dtype=torch.bfloat16), a, 4, 128, 1)
    assert sk._out(None, a, 4, 128, 1).device == a.device


def test_a16w4_operands_are_checked_before_the_library():
    import torch
    aq = torch.empty((256, 512), dtype=torch.uint8, device="meta")
    a_s = torch.empty((256, 32), dtype=torch.uint8, device="meta")
    b = torch.empty((4, 1024), dtype=torch.bfloat16, device="meta")
    assert sk._w4_dims(aq, a_s, b) == (4, 256, 1024, 1)
    with pytest.raises(TypeError):
        sk._w4_dims(aq, a_s, b.float())                 # activations are bf16
    with pytest.raises(ValueError):
        sk._w4_dims(aq, a_s, b.unsqueeze(0))            # mixed ranks
    with pytest.raises(ValueError):
        sk._w4_dims(aq, a_s[:, :16], b)                 # one scale per 32 k


def test_version_and_strerror():
    assert sk.splitk_version() >= 10000
    for code, name in sk.STATUS.items():
        assert sk.splitk_strerror(code) != "unknown status code", name
    assert sk.splitk_strerror(12345) == "unknown status code"


def test_the_binding_knows_every_status_the_header_declares():
    text = (ROOT / "include" / "splitk.h").read_text()
    enum = text[text.index("enum splitk_status"):]
    enum = enum[:enum.index("};")]
    declared = {int(v): k for k, v in re.findall(r"(SPLITK_\w+)\s*=\s*(-?\d+)", enum)}
    assert declared == sk.STATUS


def _plan(M, N, K, L=1, split=0):
    return sk.splitk_plan_for(M, N, K, L, split, **GB300)


def _per_tile(M, N, K, L=1, split=0):
    """The per-tile kernel's own choice (the second candidate when the plan
    is persistent)."""
    c = sk.splitk_plan_candidates_for(M, N, K, L, split, **GB300)
    return c[1] if c[0].persistent else c[0]


def test_plan_of_the_decode_workloads():
    p = _plan(1, 7168, 2048, 1, 4)
    assert (p.mma_m, p.mma_n, p.split_k, p.k_tiles_per_cta) == (128, 16, 4, 4)
    assert list(p.grid) == [4, 56, 1] and list(p.cluster) == [4, 1, 1]
    assert p.smem_bytes <= GB300["smem_per_block_optin"]
    p = _plan(16, 4096, 7168, 1, 8)
    assert (p.mma_n, p.split_k, p.k_tiles_per_cta) == (16, 8, 7)
    assert list(p.grid) == [8, 32, 1]
    p = _plan(64, 18432, 7168, 1, 2)                # persistent: 144 tiles over 152 / 2 = 76 clusters
    assert (p.mma_n, p.persistent, list(p.grid)) == (64, 1, [2, 76, 1])
    p = _plan(128, 7168, 16384, 2, 8)              # persistent: 152 SMs / 8 = 19 clusters
    assert (p.mma_n, list(p.grid), p.k_tiles_per_cta, p.persistent) == (128, [8, 19, 1], 16, 1)
    # split 8: a 2-deep activation ring of its own buys one reduction round a tile
    assert (p.stages, p.b_stages, p.mailbox_quads, p.reduce_rounds) == (3, 2, 32, 1)
    p4 = _plan(128, 7168, 16384, 2, 4)             # split 4: the activations ride the weight ring
    assert (p4.persistent, p4.stages, p4.b_stages) == (1, 3, 0)
    assert (p4.mailbox_quads, p4.reduce_rounds) == (16, 2)                # two rounds buy a third stage
    assert _plan(16, 4096, 7168, 1, 8).persistent == 0   # 32 tiles deal out unevenly over 19 clusters
    assert _plan(16, 7168, 16384, 2, 8).persistent == 1
    assert _plan(16, 7168, 16384, 2, 4).persistent == 0  # narrow tiles at split 4: the per-tile kernel
    assert _plan(64, 7168, 16384, 2, 4).persistent == 1
    p2 = _plan(128, 7168, 16384, 2, 2)             # split 2, 128 tokens: 64-token tiles, 224 over 76 clusters
    assert (p2.persistent, p2.mma_n, p2.split_k) == (1, 64, 2)
    p64 = _plan(64, 7168, 16384, 2, 2)                   # 112 tiles over 76 clusters: persistent all the same
    assert (p64.persistent, p64.mma_n) == (1, 64)
    p32 = _plan(32, 7168, 16384, 2, 4)                   # 32-token tiles at split 4, evenly dealt: persistent
    assert (p32.persistent, p32.mma_n) == (1, 32)
    pw = _plan(64, 18432, 7168, 1, 2)                     # the wide projection: 144 tiles, even enough
    assert (pw.persistent, pw.mma_n) == (1, 64)
    p32 = _plan(32, 7168, 16384, 2, 2)                   # 32-token tiles at split 2: persistent
    assert (p32.persistent, p32.mma_n) == (1, 32)
    assert _plan(48, 7168, 16384, 2, 2).persistent == 1  # 64-token tiles, uneven rounds: persistent
    assert p.reduce_rounds >= 1 and p.mailbox_quads % 4 == 0


def test_decode_tactics():
    """The staged decode tactic: a 2-stage weight ring, all activation tiles
    resident, the first min(3, k_tiles - 2) weight tiles staged in tensor
    memory, two MMA issuers, early trigger, 2 CTAs per SM.  M=1: rank 0
    reduces; M=16, split 8: each rank reduces 16 rows (scattered)."""
    p = _plan(1, 7168, 2048, 1, 4)
    assert (p.ctas_per_sm, p.stages, p.reduce_scatter, p.mailbox_dedicated) == (2, 2, 0, 1)
    assert (p.b_resident, p.a_tmem_tiles, p.mma_issuers, p.pdl_trigger, p.tmem_cols) == (1, 2, 2, 1, 256)
    assert p.b_loader == 1                         # 1 row x 4 K tiles: 64 loads of 16 bytes
    assert p.l2_prefetch == 0                      # all 4 weight tiles on chip
    assert p.smem_bytes == 1024 + 2 * 32768 + 4 * 16 * 256 + 3 * 512 + 256
    p = _plan(16, 4096, 7168, 1, 8)
    assert (p.ctas_per_sm, p.stages, p.reduce_scatter, p.mailbox_dedicated) == (2, 2, 1, 1)
    assert (p.b_resident, p.a_tmem_tiles, p.mma_issuers, p.pdl_trigger, p.tmem_cols) == (1, 3, 2, 1, 256)
    assert p.b_loader == 0                         # 16 rows x 7 K tiles: TMA
    assert p.l2_prefetch == 1                      # 2 of 7 weight tiles off chip before the wait
    assert p.smem_bytes == 1024 + 2 * 32768 + 7 * 16 * 256 + 16 * 512 + 256
    for p in (_plan(1, 7168, 2048, 1, 4), _plan(16, 4096, 7168, 1, 8)):
        assert 2 * (p.smem_bytes + 1024) <= GB300["smem_per_sm"]
        assert GB300["smem_per_sm"] // (p.smem_bytes + 1024) * p.tmem_cols <= 512


def test_long_k_and_wide_shapes_keep_the_ring():
    """Where all activation tiles do not fit beside the ring at 2 CTAs per SM
    (long K) or tiles are wide, the plan keeps the page's ring design."""
    for args in [(1, 7168, 16384, 2, 4), (32, 7168, 16384, 2, 2), (64, 18432, 7168, 1, 2)]:
        p = _plan(*args)
        assert (p.b_resident, p.a_tmem_tiles, p.mma_issuers, p.pdl_trigger, p.b_loader, p.l2_prefetch) == \
            (0, 0, 1, 0, 0, 0), args


def test_auto_split_fills_the_sms_with_the_smallest_split():
    assert _plan(1, 7168, 2048).split_k == 4       # 56 tiles -> 224 CTAs >= 3/4 of 152
    assert _plan(16, 4096, 7168).split_k == 4      # 32 tiles -> 128 CTAs
    assert _plan(64, 18432, 7168).split_k == 1     # 144 tiles of 64 tokens: no reduction
    assert _plan(8, 7168, 16384, 2).split_k == 2   # 112 tiles -> 224 CTAs
    assert _plan(1, 128, 128).split_k == 1         # K of one tile: no split
    assert _plan(1, 128, 256).split_k == 2         # two K tiles, one tile: split 2


@pytest.mark.parametrize("K,split,k_tiles", [(1000, 4, 2), (1032, 4, 3), (8, 1, 1), (136, 2, 1),
                                             (7168, 8, 7), (7176, 8, 8)])
def test_k_tails_take_ragged_tiles(K, split, k_tiles):
    p = _plan(4, 256, K, 1, split)
    assert p.k_tiles_per_cta == k_tiles


def _check_persistent(p, M, N, K, L, split):
    """The invariants of a persistent plan: a cluster of split CTAs per
    `split` SMs (at most one per output tile), one CTA per SM, two
    accumulators, the scattered mailbox beside a ring of weight and
    activation stages (or a weight ring and an activation ring)."""
    tiles = -(-M // p.mma_n) * -(-N // 128) * L
    assert split >= 2 and p.split_k == split
    assert list(p.grid) == [split, max(1, min(tiles, GB300["num_sms"] // split)), 1]
    assert list(p.cluster) == [split, 1, 1]
    assert (p.reduce_scatter, p.mailbox_dedicated, p.b_resident, p.a_tmem_tiles,
            p.mma_issuers, p.b_loader, p.l2_prefetch, p.ctas_per_sm) == (1, 1, 0, 0, 1, 0, 0, 1)
    assert p.tmem_cols == next(c for c in (32, 64, 128, 256, 512) if c >= 2 * max(32, p.mma_n))
    assert 2 <= p.stages <= 8
    assert p.b_stages == 0 or 2 <= p.b_stages <= 8
    b_ring = p.b_stages or p.stages
    nquads = -(-min(M, p.mma_n) // 4)
    assert p.mailbox_quads == nquads or (p.mailbox_quads % 4 == 0 and p.mailbox_quads < nquads)
    assert p.reduce_rounds == -(-nquads // p.mailbox_quads)
    round_cols = min(min(M, p.mma_n), 4 * p.mailbox_quads)
    budget = min(GB300["smem_per_block_optin"], GB300["smem_per_sm"] - 1024)
    bars = 256 if b_ring == p.stages else 384       # a second set of ring barriers when the depths differ
    assert p.smem_bytes == 1024 + p.stages * 32768 + b_ring * p.mma_n * 256 + round_cols * 512 + bars
    assert p.smem_bytes <= budget
    one_more = 32768 + (0 if p.b_stages else p.mma_n * 256)
    if p.stages < 8:   # the deepest weight ring that fits
        assert p.smem_bytes + one_more > budget
    if p.reduce_rounds > 1:   # rounds only where they buy a deeper ring than one round a tile
        assert 1024 + p.stages * 32768 + b_ring * p.mma_n * 256 + min(M, p.mma_n) * 512 + bars > budget


@pytest.mark.parametrize("M", [1, 4, 16, 17, 32, 33, 64, 65, 128, 129, 1000])
@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_every_plan_fits_and_is_consistent(M, split):
    K = 128 * 8 * 4 - 8 * (M % 5)                  # some ragged K
    p = _plan(M, 7168, K, 2, split)
    assert p.k_tiles_per_cta == -(-(-(-K // 128)) // split)
    # 64-token tiles: the persistent kernel at split 2 with 64 or more tokens
    assert p.mma_n >= min(M, 128) or p.mma_n == 128 or (p.persistent and split == 2 and M >= 64 and p.mma_n == 64)
    if p.persistent:
        _check_persistent(p, M, 7168, K, 2, split)
        return
    assert p.grid[0] == split * -(-M // p.mma_n)
    assert 2 <= p.stages <= 8
    assert p.smem_bytes <= GB300["smem_per_block_optin"]
    assert p.mma_issuers in (1, 2) and p.stages % p.mma_issuers == 0
    assert 0 <= p.a_tmem_tiles <= 3 and (p.a_tmem_tiles == 0 or p.b_resident)
    assert p.b_loader in (0, 1) and (p.b_loader == 0 or p.b_resident)
    acc = max(32, p.mma_n) * p.mma_issuers
    need = acc if p.a_tmem_tiles == 0 else (acc + 63) // 64 * 64 + 64 * p.a_tmem_tiles
    assert p.tmem_cols == next(c for c in (32, 64, 128, 256, 512) if c >= need)
    assert GB300["smem_per_sm"] // (p.smem_bytes + 1024) * p.tmem_cols <= 512
    b_tiles = max(p.stages, p.k_tiles_per_cta) if p.b_resident else p.stages
    # the reduction's mailbox fits where it is placed
    if p.reduce_scatter:
        assert split >= 4 and min(M, p.mma_n) >= 2 and p.mailbox_dedicated == 1
        assert p.smem_bytes == 1024 + p.stages * 32768 + b_tiles * p.mma_n * 256 + min(M, p.mma_n) * 512 + 256
    elif split > 1:
        cols = min(4 * p.mailbox_quads, M, p.mma_n)
        round_bytes = (split - 1) * cols * 128 * 4
        ded = round_bytes if p.mailbox_dedicated else 0
        if not p.mailbox_dedicated:
            assert round_bytes <= p.stages * 32768
        nquads = -(-min(M, p.mma_n) // 4)
        assert p.reduce_rounds == -(-nquads // p.mailbox_quads)
        assert p.smem_bytes == 1024 + p.stages * 32768 + b_tiles * p.mma_n * 256 + ded + 256
    # the f32 staging tile of rank 0 fits in its drained activation ring
    assert min(M, p.mma_n) * 128 * 4 <= b_tiles * p.mma_n * 256


def test_every_plan_of_a_broad_shape_grid_passes_the_launch_check():
    """Whatever the planners write for ~5,000 shapes, the launch-time check
    accepts, within the shared-memory and TMEM budgets of the SM."""
    n = 0
    for M in (1, 2, 3, 5, 8, 13, 16, 24, 32, 48, 64, 100, 128, 200):
        for N in (128, 300, 1000, 7168, 18432):
            for K in (8, 136, 1000, 2048, 7168, 16384, 32768):
                for L in (1, 3):
                    for split in (0, 1, 2, 4, 8):
                        try:
                            p = _plan(M, N, K, L, split)
                        except sk.SplitKError as e:
                            assert e.code in (-1, -4), (M, N, K, L, split, e.code)
                            continue
                        assert _check(p, M, N, K, L) == 0, (M, N, K, L, split, p.as_dict())
                        assert p.smem_bytes <= GB300["smem_per_block_optin"]
                        assert GB300["smem_per_sm"] // (p.smem_bytes + 1024) * p.tmem_cols <= 512
                        n += 1
                        if M <= 32 and K % 128 == 0:
                            try:
                                q = sk.splitk_plan_w4a16_for(M, N, K, L, split, **GB300)
                            except sk.SplitKError as e:
                                assert e.code in (-1, -4), (M, N, K, L, split, e.code)
                                continue
                            assert _check(q, M, N, K, L) == 0, (M, N, K, L, split, q.as_dict())
                            assert GB300["smem_per_sm"] // (q.smem_bytes + 1024) * q.tmem_cols <= 512
    assert n > 3000


@pytest.mark.parametrize("args,code", [
    ((0, 128, 128, 1, 1), -1), ((1, 0, 128, 1, 1), -1), ((1, 128, 0, 1, 1), -1),
    ((1, 128, 128, 0, 1), -1), ((1, 128, 100, 1, 1), -1), ((1, 128, 1024, 1, 3), -3),
    ((1, 128, 1024, 1, 16), -3), ((1, 128, 128, 1, 2), -1), ((1, 128, 1004, 1, 1), -1),
    ((1, 128 * 70000, 128, 1, 1), -1), ((1, 128 * 65535 + 1, 128, 1, 1), -1), ((1, 128, 128, 65536, 1), -1),
    ((1, 128, 2**31 - 120, 1, 0), -1),                 # K past the last signed 32-bit tile coordinate
])
def test_plan_rejects_bad_shapes(args, code):
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_plan_for(*args, **GB300)
    assert e.value.code == code


def test_sizes_near_int_max_plan_without_overflow():
    M = 2**31 - 1
    p = sk.splitk_plan_for(M, 128, 128, 1, 1, **GB300)
    assert tuple(p.grid) == ((M + 127) // 128, 1, 1)
    assert _check(p, M, 128, 128, 1) == 0
    K = 2**31 - 128                                    # the largest K
    p = sk.splitk_plan_for(1, 128, K, 1, 8, **GB300)
    assert p.k_tiles_per_cta == -(-(K // 128) // 8)       # the most any rank owns
    assert _check(p, 1, 128, K, 1) == 0
    assert _check(p, 1, 128, K + 8, 1) == -1


def test_the_largest_grid_dimensions_are_planned():
    p = sk.splitk_plan_for(1, 128 * 65535, 128, 1, 0, **GB300)
    assert tuple(p.grid) == (1, 65535, 1)
    p = sk.splitk_plan_for(1, 128, 128, 65535, 0, **GB300)
    assert tuple(p.grid) == (1, 1, 65535)


def test_gemm_rejects_null_and_misaligned_pointers_before_cuda():
    lib = sk.load_library()
    assert lib.splitk_gemm_bf16(None, 16, 16, 1, 128, 128, 1, 1, None) == -7
    assert lib.splitk_gemm_bf16(16, 16, None, 1, 128, 128, 1, 1, None) == -7
    assert lib.splitk_gemm_bf16(8, 16, 16, 1, 128, 128, 1, 1, None) == -2
    assert lib.splitk_gemm_bf16(16, 24, 16, 1, 128, 128, 1, 1, None) == -2
    assert lib.splitk_gemm_bf16(16, 16, 17, 1, 128, 128, 1, 1, None) == -2


def test_calls_needing_a_device_report_it_without_one():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = sk.load_library()
    plan = sk.Plan()
    assert lib.splitk_plan(1, 128, 128, 1, 1, ctypes.byref(plan)) == -9
    assert lib.splitk_gemm_bf16(16, 16, 16, 1, 128, 128, 1, 1, None) == -9


def test_settings_calls():
    assert sk.load_library().splitk_set_wait_limit_ns(0) == 0
    assert sk.load_library().splitk_debug_inject(0) == 0


def _check(p, M, N, K, L):
    return sk.splitk_plan_check_for(p, M, N, K, L, GB300["smem_per_sm"], GB300["smem_per_block_optin"])


@pytest.mark.parametrize("args", [(1, 7168, 2048, 1, 4), (16, 4096, 7168, 1, 8), (4, 256, 1024, 1, 0),
                                  (64, 18432, 7168, 1, 2), (128, 7168, 16384, 2, 0), (3, 200, 1000, 2, 0)])
def test_candidates_are_valid_distinct_and_start_with_the_plan(args):
    M, N, K, L, split = args
    cands = sk.splitk_plan_candidates_for(M, N, K, L, split, **GB300)
    assert len(cands) >= 2
    assert cands[0].as_dict() == _plan(*args).as_dict()
    seen = set()
    for p in cands:
        assert _check(p, M, N, K, L) == 0, p
        assert split == 0 or p.split_k == split
        assert p.stages % p.mma_issuers == 0
        assert GB300["smem_per_sm"] // (p.smem_bytes + 1024) * p.tmem_cols <= 512
        key = bytes(p)
        assert key not in seen
        seen.add(key)
    # the page's ring always; the staged family where all activation tiles fit
    assert any(not p.b_resident for p in cands)
    if M <= 16 and K <= 8192:
        assert any(p.b_resident and p.a_tmem_tiles for p in cands)
    if split != 1 and min(M, cands[0].mma_n) >= 4:
        assert any(p.reduce_scatter for p in cands)


def test_a_cta_alone_on_its_sm_gets_a_deep_ring_and_two_issuers():
    """Grids of at most one CTA per SM (the split-1 sweep: 112 CTAs) keep as
    many weight tiles in flight as shared memory holds, on an even ring with
    two MMA issuers where mma_n <= 64; fuller grids keep the shallow ring."""
    p = _plan(1, 7168, 16384, 2, 1)
    assert (p.stages, p.mma_issuers, p.ctas_per_sm) == (6, 2, 1)
    assert p.smem_bytes <= GB300["smem_per_block_optin"]
    assert _check(p, 1, 7168, 16384, 2) == 0
    p = _plan(64, 7168, 16384, 2, 1)
    assert (p.stages, p.mma_issuers) == (4, 2)
    p = _plan(128, 7168, 16384, 2, 1)                   # mma_n 128: one issuer
    assert p.mma_issuers == 1
    p = _plan(1, 7168, 16384, 2, 2)                     # 224 CTAs share SMs
    assert p.stages <= 4 and p.ctas_per_sm == 2


def test_long_k_slices_prefer_a_deeper_ring_over_their_own_mailbox():
    """16 K tiles a CTA and more: 3 ring stages with the mailbox aliased on the
    drained ring beat 2 with a dedicated or scattered one at 2 CTAs/SM; not
    when the aliased partials would need more than one reduction round, and
    not on short slices."""
    for M, split in ((8, 2), (16, 2), (16, 4)):
        p = _per_tile(M, 7168, 16384, 2, split)
        assert (p.stages, p.mailbox_dedicated, p.reduce_scatter, p.reduce_rounds, p.ctas_per_sm) == (3, 0, 0, 1, 2)
        assert _check(p, M, 7168, 16384, 2) == 0
    p = _per_tile(128, 7168, 16384, 2, 4)                   # 96 KB of partials: keep the scattered mailbox
    assert (p.stages, p.reduce_scatter) == (2, 1)
    p = _per_tile(8, 7168, 16384, 2, 8)                     # 16 K tiles a CTA
    assert (p.stages, p.mailbox_dedicated) == (3, 0)
    # a few token columns: the scattered mailbox when the dedicated one does
    # not fit beside the third stage; a single column keeps the dedicated one
    for M in (2, 4):
        p = _per_tile(M, 7168, 16384, 2, 8)
        assert (p.stages, p.mailbox_dedicated, p.reduce_scatter, p.ctas_per_sm) == (3, 1, 1, 2)
    p = _per_tile(1, 7168, 16384, 2, 8)
    assert (p.stages, p.mailbox_dedicated, p.reduce_scatter) == (3, 1, 0)
    p = _per_tile(8, 7168, 2048, 4, 2)                      # 8 K tiles a CTA: the dedicated mailbox stays
    assert (p.stages, p.mailbox_dedicated) == (2, 1)


def test_the_planner_writes_every_field():
    """A plan written over stale memory is the same plan (the one-shot GEMM
    calls plan into an uninitialised struct on the stack)."""
    import ctypes
    for args in [(1, 7168, 2048, 1, 4), (16, 4096, 7168, 1, 8), (3, 200, 1000, 2, 0)]:
        stale = sk.Plan()
        ctypes.memset(ctypes.byref(stale), 0xA5, ctypes.sizeof(stale))
        rc = sk.load_library().splitk_plan_for(*args, GB300["num_sms"], GB300["smem_per_sm"],
                                               GB300["smem_per_block_optin"], ctypes.byref(stale))
        assert rc == 0
        assert bytes(stale) == bytes(_plan(*args))
        assert _check(stale, *args[:4]) == 0


def test_plan_check_rejects_what_a_launch_would():
    M, N, K, L = 1, 7168, 2048, 1
    p = _plan(M, N, K, L, 4)
    assert _check(p, M, N, K, L) == 0
    bad = sk.Plan.from_buffer_copy(p)
    bad.stages = 3                                      # odd ring with two issuers
    assert _check(bad, M, N, K, L) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.tmem_cols = 128                                 # not what the layout needs
    assert _check(bad, M, N, K, L) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.b_resident = 0                                  # staged tiles need resident activations
    assert _check(bad, M, N, K, L) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.w4_smem_tiles = 1                               # a bf16 stage of decoded 4-bit weights
    bad.smem_bytes += 32768
    assert _check(bad, M, N, K, L) == -10
    assert _check(p, M, N, K + 8, L) == -10             # another shape
    bad = sk.Plan.from_buffer_copy(p)
    bad.b_stages = 2                                    # an activation ring of its own: persistent plans only
    assert _check(bad, M, N, K, L) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.w4_decoders = 1                                 # a bf16 plan decodes nothing
    assert _check(bad, M, N, K, L) == -10
    w4 = sk.splitk_plan_w4a16_for(M, N, K, L, 4, **GB300)
    assert _check(w4, M, N, K, L) == 0
    for dec in (0, 3):
        bad = sk.Plan.from_buffer_copy(w4)
        bad.w4_decoders = dec
        assert _check(bad, M, N, K, L) == -10
    bad = sk.Plan.from_buffer_copy(p)
    bad.cluster[1] = 2                                  # clusters span the K ranks of one tile only
    assert _check(bad, M, N, K, L) == -10


@pytest.mark.parametrize("args", [(1, 7168, 2048, 1, 4), (16, 4096, 7168, 1, 8), (4, 256, 1024, 1, 0),
                                  (32, 1000, 4096, 2, 0), (3, 300, 512, 1, 2), (1, 7168, 2048, 8, 4)])
def test_w4a16_plans(args):
    M, N, K, L, split = args
    p = sk.splitk_plan_w4a16_for(*args, **GB300)
    assert p.weight_format == sk.WEIGHTS_E2M1_E8M0
    assert p.stages == p.k_tiles_per_cta <= 8 and p.b_resident == 1
    assert p.mma_issuers == (2 if p.a_tmem_tiles >= 2 else 1)
    assert 1 <= p.a_tmem_tiles <= 3 and p.mma_n in (16, 32)
    assert split == 0 or p.split_k == split
    assert GB300["smem_per_sm"] // (p.smem_bytes + 1024) * p.tmem_cols <= 512
    assert _check(p, M, N, K, L) == 0
    bf = sk.Plan.from_buffer_copy(p)
    bf.weight_format = sk.WEIGHTS_BF16          # an A16W4 layout is no bf16 plan
    assert _check(bf, M, N, K, L) == -10
    if p.mma_issuers == 2:
        one = sk.Plan.from_buffer_copy(p)
        one.mma_issuers = 1                     # one issuer fits the same TMEM columns
        assert _check(one, M, N, K, L) == 0
        few = sk.Plan.from_buffer_copy(p)
        few.a_tmem_tiles = 1                    # two issuers need two slots
        few.tmem_cols = 128
        assert _check(few, M, N, K, L) == -10
    # the bf16 stage takes the one tile after the TMEM slots, and only that
    assert p.w4_smem_tiles == (1 if p.k_tiles_per_cta == p.a_tmem_tiles + 1 and M <= 16 else 0)
    st = sk.Plan.from_buffer_copy(p)
    st.w4_smem_tiles = 1 - p.w4_smem_tiles
    st.smem_bytes += 32768
    assert _check(st, M, N, K, L) == (0 if p.k_tiles_per_cta == p.a_tmem_tiles + 1 else -10)
    if p.w4_smem_tiles:
        small = sk.Plan.from_buffer_copy(p)
        small.smem_bytes -= 32768               # no room for the stage
        assert _check(small, M, N, K, L) == -10


def test_w4a16_grids_of_several_waves_trade_tmem_slots_for_residency():
    one = sk.splitk_plan_w4a16_for(1, 7168, 2048, 1, 4, **GB300)    # 224 CTAs: under two waves
    assert one.a_tmem_tiles == 3 and one.ctas_per_sm == 2
    assert one.w4_decoders == 1                                      # 4 K tiles a CTA: one decoding warpgroup
    small_batch = sk.splitk_plan_w4a16_for(16, 4096, 7168, 1, 8, **GB300)
    assert small_batch.k_tiles_per_cta == 7 and small_batch.w4_decoders == 1 and small_batch.ctas_per_sm == 2
    many = sk.splitk_plan_w4a16_for(1, 7168, 2048, 8, 4, **GB300)   # 1792 CTAs
    assert (many.a_tmem_tiles, many.mma_issuers, many.w4_smem_tiles, many.w4_decoders) == (1, 1, 0, 1)
    assert many.ctas_per_sm == 3 and many.ctas_per_sm * many.tmem_cols <= 512
    assert _check(many, 1, 7168, 2048, 8) == 0
    wide = sk.splitk_plan_w4a16_for(16, 4096, 7168, 4, 8, **GB300)  # one slot would not raise residency
    assert wide.a_tmem_tiles == 3 and wide.ctas_per_sm == 2


def test_w4a16_plans_reject_what_the_kernel_cannot_do():
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_plan_w4a16_for(33, 256, 1024, 1, 0, **GB300)      # tiles of more than 32 tokens
    assert e.value.code == -1
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_plan_w4a16_for(1, 256, 1000, 1, 0, **GB300)      # K not a multiple of 128
    assert e.value.code == -1
    with pytest.raises(sk.SplitKError) as e:
        sk.splitk_plan_w4a16_for(1, 256, 128 * 20, 1, 2, **GB300)  # 10 K tiles per CTA
    assert e.value.code == -4
    p = sk.splitk_plan_w4a16_for(1, 256, 128 * 20, 1, 0, **GB300)  # the plan raises the split
    assert p.k_tiles_per_cta <= 8


@pytest.mark.parametrize("args", [(1, 7168, 2048, 1, 4), (16, 4096, 7168, 1, 8), (4, 256, 1024, 1, 0),
                                  (32, 1000, 4096, 2, 0)])
def test_w8a16_plans(args):
    M, N, K, L, split = args
    p = sk.splitk_plan_w8a16_for(*args, **GB300)
    assert p.weight_format == sk.WEIGHTS_E4M3_E8M0
    assert min(2, p.k_tiles_per_cta) <= p.stages <= p.k_tiles_per_cta <= 8 and p.b_resident == 1
    assert 1 <= p.a_tmem_tiles <= 3 and p.mma_n in (16, 32) and p.w4_decoders in (1, 2)
    assert _check(p, M, N, K, L) == 0
    # 16 KiB of codes a K tile: the layout holds the ring of them
    b_tiles = max(2, p.k_tiles_per_cta)
    assert p.smem_bytes >= 1024 + p.stages * 16384 + b_tiles * p.mma_n * 256 + p.w4_smem_tiles * 32768
    # a ring shorter than the CTA's tiles only where all of them would not fit two CTAs an SM
    if p.stages < p.k_tiles_per_cta:
        assert p.smem_bytes + 1024 <= GB300["smem_per_sm"] // 2
        assert p.smem_bytes + 16384 + 1024 > GB300["smem_per_sm"] // 2     # one stage more would not
    # a 4-bit plan of the same shape is not an 8-bit one
    w4 = sk.splitk_plan_w4a16_for(*args, **GB300)
    bad = sk.Plan.from_buffer_copy(w4)
    bad.weight_format = sk.WEIGHTS_E4M3_E8M0
    assert _check(bad, M, N, K, L) in (0, -10)     # accepted only if its shared memory holds 8-bit tiles
    if w4.smem_bytes < p.smem_bytes - 32768:
        assert _check(bad, M, N, K, L) == -10
