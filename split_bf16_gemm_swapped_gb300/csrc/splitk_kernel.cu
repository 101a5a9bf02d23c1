// The split-K BF16 decode GEMM kernel for sm_103a (GB300).
//
//   C[l][m][n] = bf16_rne( sum_k A[l][n][k] * B[l][m][k] )
//
// Method: the vLLM "splitk" API page (module
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.gemm.splitk, class
// SplitKGemm): a thread-block cluster of split_k CTAs shares one output tile;
// rank r accumulates the contiguous K slice [r*K/split_k, (r+1)*K/split_k) in
// FP32; ranks != 0 publish their partials into rank 0's shared memory over
// DSMEM (st.async, completion counted in bytes on rank 0's mbarrier); rank 0
// waits at cluster scope, adds them in rank order, converts once to BF16 and
// stores.  Operands are swapped: 128 weight rows (public N) on the tcgen05
// MMA M dimension, the tokens (public M) on MMA N.
//
// CTA roles (256 threads):
//   warp 0      weight (A) producer: TMA from a tensor map in global memory,
//               L2 evict_first, issued before the programmatic-dependent-launch
//               wait; then launch_dependents (SplitKGemm.weight_warp)
//   warp 1      activation (B) producer: griddepcontrol.wait, then TMA
//               (SplitKGemm.activation_warp)
//   warp 2      TMEM allocation, tcgen05.mma issue (even K tiles when there
//               are two issuers), TMEM release (mma_warp)
//   warp 3      second MMA issuer (odd K tiles, own accumulator) or idle; it
//               keeps warps 4..7 on TMEM lane quadrants 0..3
//   warps 4..7  weight tiles copied into TMEM before the wait (staged tiles)
//               or, for 4- and 8-bit weights, decoded to bf16 into TMEM or a
//               shared-memory stage; activation loads for few rows; then the
//               epilogue: TMEM -> registers, DSMEM publish / rank-0 reduce,
//               BF16 packing, 16-byte stores (epilog_warp)
//
// Every mbarrier wait is bounded by %globaltimer (the Muse Spark AMD dev
// page's _spin_bounded: a timeout records a diagnostic, sets a sticky failed
// flag, and the CTA's later waits give up at once); TMEM is always released.
// A CTA whose shared memory a peer may still address (aliased or multi-round
// mailboxes) leaves only after a final cluster barrier; a
// CTA whose wait failed first drains (bounded) the copies it issued and the
// partials addressed to it, so a failed launch leaves no copy in flight into
// a departed CTA.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>


#include "splitk.h"
#include "splitk_device.cuh"
#include "splitk_internal.h"
#include "splitk_kernel_common.cuh"

namespace splitk {

// The E8M0 scale words of one weight row's K tiles (four codes a tile, one
// per 32 k), all loaded when the decoder starts, so that no tile's decode
// waits on a global load; taken in order, each take shifting the rest down
// (indices stay compile-time: the words stay in registers).
struct ScaleWords {
  uint32_t w[kMaxStages];
  __device__ __forceinline__ void load(const uint32_t* src, bool row_ok, int k_tiles) {
#pragma unroll
    for (int i = 0; i < kMaxStages; ++i) w[i] = (row_ok && i < k_tiles) ? __ldg(src + i) : 0u;
  }
  __device__ __forceinline__ uint32_t take() {
    const uint32_t x = w[0];
#pragma unroll
    for (int i = 0; i + 1 < kMaxStages; ++i) w[i] = w[i + 1];
    return x;
  }
};

// ---- decode of packed weight codes to bf16 (quantized weights)
//
// Decode of the 32-k steps [j0, j1) of one weight row of a packed tile, each
// step one scale block (scale code byte j of `codes`), into 16 words of bf16
// pairs: E2M1 codes are 64 B a row in the 64-byte swizzle (step j is the
// 16-byte chunk at slot j ^ ((row >> 1) & 3)), a byte -> two bf16; E4M3
// codes are 128 B a row in the 128-byte swizzle (step j is chunks 2j and
// 2j + 1 at slots c ^ (row & 7)), two bytes -> two bf16.  Both place the
// code bits in bf16 lanes (exact, a constant power of two apart from the
// code's value) and take one bf16 product by a power of two (two for scale
// codes out of that product's range), exact wherever the scaled weight is a
// bf16 value.
template <int kFmt>
struct QFmt {
  static constexpr int kCodeWords = kFmt == 2 ? 8 : 4;   // 32-bit words of codes a step
  using Scale = dev::BlockScale<kFmt == 2 ? 120 : 126>;
};

template <int kFmt>
__device__ __forceinline__ void q_load_step(uint32_t src, int j, int row, uint32_t (&w)[QFmt<kFmt>::kCodeWords]) {
  if constexpr (kFmt == 2) {
    dev::ld_shared_v4(src + (uint32_t)(((2 * j) ^ (row & 7)) * 16), w[0], w[1], w[2], w[3]);
    dev::ld_shared_v4(src + (uint32_t)(((2 * j + 1) ^ (row & 7)) * 16), w[4], w[5], w[6], w[7]);
  } else {
    dev::ld_shared_v4(src + (uint32_t)((j ^ ((row >> 1) & 3)) * 16), w[0], w[1], w[2], w[3]);
  }
}

// One step's 16 pairs with the block multiplier `m` of the form kTwo.
template <int kFmt, bool kTwo>
__device__ __forceinline__ void q_convert_step(const uint32_t (&w)[QFmt<kFmt>::kCodeWords], uint32_t m,
                                               uint32_t (&r)[16]) {
  using S = typename QFmt<kFmt>::Scale;
  if constexpr (kFmt == 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[2 * i] = S::template apply<kTwo>(dev::e4m3x2_placed<0>(w[i]), m);
      r[2 * i + 1] = S::template apply<kTwo>(dev::e4m3x2_placed<1>(w[i]), m);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w4 = w[i] << 4;
      r[4 * i + 0] = S::template apply<kTwo>(dev::e2m1x2_placed<0>(w[i], w4), m);
      r[4 * i + 1] = S::template apply<kTwo>(dev::e2m1x2_placed<1>(w[i], w4), m);
      r[4 * i + 2] = S::template apply<kTwo>(dev::e2m1x2_placed<2>(w[i], w4), m);
      r[4 * i + 3] = S::template apply<kTwo>(dev::e2m1x2_placed<3>(w[i], w4), m);
    }
  }
}

// Whether every scale code of steps [j0, j1) takes the one-product form
// (the form is chosen once for a row's steps of a tile).
template <int kFmt>
__device__ __forceinline__ bool q_row_fast(uint32_t codes, int j0, int j1) {
  bool fast = true;
#pragma unroll 1
  for (int j = j0; j < j1; ++j) fast = fast && QFmt<kFmt>::Scale::fast((codes >> (8 * j)) & 0xFFu);
  return fast;
}

// Steps [j0, j1) of the row at `src` (j1 - j0 even: 4, or 2 with two
// decoding warpgroups), two at a time through two code buffers, each step's
// codes loaded a step ahead so that the load latency overlaps the previous
// step's conversion; `emit(j, r)` stores step j's 16 words.
template <int kFmt, bool kTwo, class Emit>
__device__ __forceinline__ void q_steps(uint32_t src, int row, uint32_t codes, int j0, int j1, Emit& emit) {
  using S = typename QFmt<kFmt>::Scale;
  uint32_t a[QFmt<kFmt>::kCodeWords], b[QFmt<kFmt>::kCodeWords];
  q_load_step<kFmt>(src, j0, row, a);
#pragma unroll 1
  for (int j = j0; j < j1; j += 2) {
    q_load_step<kFmt>(src, j + 1, row, b);
    uint32_t ra[16], rb[16];
    q_convert_step<kFmt, kTwo>(a, S::template multiplier<kTwo>((codes >> (8 * j)) & 0xFFu), ra);
    emit(j, ra);
    if (j + 2 < j1) q_load_step<kFmt>(src, j + 2, row, a);
    q_convert_step<kFmt, kTwo>(b, S::template multiplier<kTwo>((codes >> (8 * j + 8)) & 0xFFu), rb);
    emit(j + 1, rb);
  }
}

// kFmt: the weight format (0 bf16; 1 E2M1 codes, 2 E4M3 codes, each with
// E8M0 scales per 32 k, decoded on chip).  kDecWG: warpgroups decoding
// quantized weight tiles (1: warps 4..7, the epilogue; 2: also warps 8..11,
// each group decoding half of every tile's K).
template <int MMA_N, int kFmt, int kDecWG>
__global__ void __launch_bounds__(kDecWG == 2 ? kThreadsW4Wide : kThreads, kDecWG == 2 ? 2 : 3)
    splitk_gemm_bf16_kernel(const __grid_constant__ CUtensorMap b_map, const KernelParams p) {
  constexpr bool kQuant = kFmt != 0;                           // quantized weights, decoded on chip
  constexpr uint32_t kQTileBytes = kFmt == 2 ? kW8TileBytes : kW4TileBytes;   // one packed K tile
  constexpr uint32_t kQRowBytes = kFmt == 2 ? kW8RowBytes : kW4RowBytes;      // one row of it
  constexpr uint32_t kBStage = b_stage_bytes(MMA_N);
  constexpr uint32_t kBBox = kBStage / 2;                   // MMA_N rows x 128 B
  constexpr uint32_t kAccCols = tmem_acc_cols(MMA_N);       // TMEM columns of one accumulator
  constexpr uint32_t kIdesc = dev::idesc_bf16_f32(kMmaM, MMA_N);
  constexpr uint32_t kAStage = kQuant ? kQTileBytes : kAStageBytes;   // one weight K tile in shared memory

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + (kAlignSlack - 1)) & ~(kAlignSlack - 1);

  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);
  const int split = p.split;
  const int stages = p.stages;
  // The cluster is the split K ranks of one output tile; rank 0 owns the tile.
  const int rank = split > 1 ? (int)dev::cluster_ctarank() : 0;
  const int m_tile = (int)blockIdx.x / split;
  const int n0 = (int)blockIdx.y * kMmaM;
  const int m0 = m_tile * MMA_N;
  const int l = (int)blockIdx.z;
  // Contiguous K slices: ranks below T % split take one extra tile.
  const int kt_base = p.k_tiles_total / split;
  const int kt_extra = p.k_tiles_total % split;
  const int k_tiles = kt_base + (rank < kt_extra ? 1 : 0);
  const int kt0 = rank * kt_base + (rank < kt_extra ? rank : kt_extra);

  const bool b_res = p.b_resident != 0;
  const int tmem_tiles = p.a_tmem_tiles < k_tiles ? p.a_tmem_tiles : k_tiles;

  // Shared memory: [A ring (quantized weights: a ring of packed tiles)][B ring or all B tiles]
  // [dedicated mailbox?][barriers].
  const uint32_t sA = base;
  const uint32_t sB = sA + (uint32_t)stages * kAStage;
  const uint32_t sQStage = sB + (uint32_t)p.b_region_tiles * kBStage;   // quantized weights: the bf16 stage (if any)
  const uint32_t ring_end = sQStage + (kQuant ? (uint32_t)p.w4_smem_tiles * kAStageBytes : 0u);
  const uint32_t sMail = p.mailbox_dedicated ? ring_end : sA;
  const uint32_t sBar = ring_end + (p.mailbox_dedicated ? p.mailbox_bytes : 0u);
  const uint32_t bar_full0 = sBar;                       // [kMaxStages], count 2
  const uint32_t bar_empty0 = sBar + 8u * kMaxStages;    // [kMaxStages], count 1 (quantized: the decoders)
  const uint32_t bar_mma_done = sBar + 16u * kMaxStages; // count 1
  const uint32_t bar_tmem_empty = bar_mma_done + 8u;     // count 128
  const uint32_t bar_reduce = bar_mma_done + 16u;        // count 1 + tx bytes
  const uint32_t bar_ready = bar_mma_done + 24u;         // count 1 (rank 0 arrives)
  const uint32_t slot_tmem = bar_mma_done + 32u;
  const uint32_t slot_abort = bar_mma_done + 36u;
  const uint32_t bar_b = bar_mma_done + 40u;             // count 1 + tx bytes (resident B)
  const uint32_t bar_slot_full0 = bar_mma_done + 48u;    // quantized [3]: tile decoded into TMEM slot (a warp each)
  const uint32_t bar_slot_empty0 = bar_mma_done + 72u;   // quantized [3]: slot read by the MMAs, count 1
  const uint32_t bar_w4_stage = bar_mma_done + 96u;      // quantized: the bf16 stage decoded (a warp each)

  const Waiter waiter{slot_abort, p.wait_limit_ns};

  // ---- set-up, three warps in parallel: warp 3 initialises the barriers,
  // warp 2 allocates TMEM, and warp 0 acquires A's tensor map (a round trip
  // to global memory) and then issues the first ring pass of weight loads.
  // Every thread arrives on the cluster barrier (a 1-CTA cluster when
  // split_k = 1) once its own set-up is published, and waits on it before
  // touching shared state.  Warp 0 arrives before issuing its loads: an
  // arrival with release semantics after those issues would hold the whole
  // cluster until the loads have landed.
  int a_issued = 0;          // weight tiles thread 0 has issued (for the drain after a failure)
  bool b_issued = false;     // activation tiles issued onto bar_b (resident activations)
  uint64_t a_policy = 0;
  if (warp == 3) {
    if (lane == 0) {
      for (int s = 0; s < stages; ++s) {
        dev::mbar_init(bar_full0 + 8u * s, b_res ? 1u : 2u);   // A (and B when it rides the ring)
        // the stage's MMA commit; quantized weights: every decoding warp,
        // once it has read the stage's codes
        dev::mbar_init(bar_empty0 + 8u * s, kQuant ? (uint32_t)(kEpiWarps * kDecWG) : 1u);
      }
      dev::mbar_init(bar_b, p.b_loader ? (uint32_t)kEpiThreads : 1u);
      dev::mbar_init(bar_mma_done, (uint32_t)p.mma_issuers);
      dev::mbar_init(bar_tmem_empty, kEpiThreads);
      dev::mbar_init(bar_reduce, 1);
      dev::mbar_init(bar_ready, 1);
      if (kQuant) {
        for (int i = 0; i < 3; ++i) {
          dev::mbar_init(bar_slot_full0 + 8u * i, (uint32_t)(kEpiWarps * kDecWG));
          dev::mbar_init(bar_slot_empty0 + 8u * i, 1);
        }
        dev::mbar_init(bar_w4_stage, (uint32_t)(kEpiWarps * kDecWG));
      }
      dev::st_shared_u32(slot_abort, 0u);
      dev::fence_barrier_init();
      stamp(p, kTrBarInit);
    }
    dev::named_bar_sync(2, 64);          // barriers exist for warp 0's loads
  } else if (warp == 0) {
    if (lane == 0) {
      stamp(p, kTrStart);
      dev::tensormap_acquire(p.a_map);   // the weight stream does not depend on the previous kernel
      stamp(p, kTrMapReady);
      a_policy = dev::policy_evict_first();
    }
    dev::named_bar_sync(2, 64);
  } else if (warp == 2) {
    dev::tmem_alloc(slot_tmem, p.tmem_cols);
    dev::tmem_relinquish();
    dev::tc_fence_before();
    if (lane == 0) {
      stamp(p, kTrTmemAlloc);
      // Early trigger: the next kernel may launch once every CTA holds its
      // tensor memory.  (Not before: a CTA of the next kernel that took the
      // columns first would wait for this kernel, which would wait for it.)
      if (p.pdl_trigger_early) dev::griddep_launch_dependents();
    }
  }
  dev::cluster_arrive_release();
  if (kQuant && threadIdx.x == 0) {
    // the first ring pass of packed weight tiles (usually all of the CTA's):
    // one box each, 8 KiB of 4-bit codes or 16 KiB of 8-bit ones
    const int first = k_tiles < stages ? k_tiles : stages;
    for (; a_issued < first; ++a_issued) {
      const uint32_t full = bar_full0 + 8u * a_issued;
      dev::mbar_arrive_expect_tx(full, kQTileBytes);
      dev::tma_load_3d_hint(sA + (uint32_t)a_issued * kQTileBytes, p.a_map, (kt0 + a_issued) * (int)kQRowBytes,
                            n0, l, full, a_policy);
    }
    stamp(p, kTrPrefetched);
  } else if (threadIdx.x == 0) {
    const int first = k_tiles < stages ? k_tiles : stages;
    for (; a_issued < first; ++a_issued) {
      const uint32_t full = bar_full0 + 8u * a_issued;
      const uint32_t dst = sA + (uint32_t)a_issued * kAStageBytes;
      const int k = (kt0 + a_issued) * kCtaK;
      dev::mbar_arrive_expect_tx(full, kAStageBytes);
      dev::tma_load_3d_hint(dst, p.a_map, k, n0, l, full, a_policy);
      dev::tma_load_3d_hint(dst + kABoxBytes, p.a_map, k + kAtomK, n0, l, full, a_policy);
    }
    if (p.l2_prefetch) {
      // The weight tiles that cannot be on chip before the PDL wait returns
      // (past the ring and the tensor-memory tiles) go to L2 now, so their
      // loads after the wait hit L2 instead of waiting for HBM.
      for (int kt = stages + tmem_tiles; kt < k_tiles; ++kt) {
        const int k = (kt0 + kt) * kCtaK;
        dev::tma_prefetch_3d(p.a_map, k, n0, l);
        dev::tma_prefetch_3d(p.a_map, k + kAtomK, n0, l);
      }
    }
    stamp(p, kTrPrefetched);
  }
  // Peers' barriers (and this CTA's TMEM address) exist past this point.
  dev::cluster_wait_acquire();
  dev::tc_fence_after();
  const uint32_t tmem_base = dev::ld_shared_u32(slot_tmem);
  if (threadIdx.x == 0) {
    stamp(p, kTrSynced);
    if (p.trace != nullptr) {
      const uint32_t cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
      if (cta < p.trace_ctas) {
        p.trace[(size_t)cta * kTraceSlots + kTrSmRank] =
            (unsigned long long)smid() | ((unsigned long long)rank << 32);
      }
    }
  }
  if (threadIdx.x == 128) stamp(p, kTrEpiSynced);

  // Decode of the 32-k steps [j0, j1) of weight row `row` of the packed tile
  // in code-ring stage `stage` (q_steps above).
  // The form is chosen for the whole warp (a vote): the steps end in
  // warp-collective stores (tcgen05.st.sync.aligned), which every lane must
  // reach at the same instruction.  The two-product form is exact for every
  // code, so a lane that could use one product loses only time.
  auto q_decode_row = [&](int stage, int row, uint32_t codes, int j0, int j1, auto&& emit) {
    const uint32_t src = sA + (uint32_t)stage * kQTileBytes + (uint32_t)row * kQRowBytes;
    if (__all_sync(0xffffffffu, q_row_fast<kFmt>(codes, j0, j1))) {
      q_steps<kFmt, false>(src, row, codes, j0, j1, emit);
    } else {
      q_steps<kFmt, true>(src, row, codes, j0, j1, emit);
    }
  };
  // Into TMEM columns t_col + 16 j of the thread's lane, or into the bf16
  // stage in shared memory in the 128-byte-swizzled layout of the bf16 path
  // (two boxes of 64 k; 16-byte chunk c of row r of an 8-row atom at chunk
  // c ^ (r % 8)), read by the MMA from there.
  auto q_decode_tmem = [&](int stage, int row, uint32_t codes, uint32_t t_col, int j0, int j1) {
    q_decode_row(stage, row, codes, j0, j1, [&](int j, const uint32_t (&r)[16]) {
      __syncwarp();   // tcgen05.st is warp-collective
      dev::tmem_st_x16(t_col + (uint32_t)(j * 16), r);
    });
  };
  auto q_decode_stage = [&](int stage, int row, uint32_t codes, int j0, int j1) {
    const uint32_t atom = sQStage + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u;
    q_decode_row(stage, row, codes, j0, j1, [&](int j, const uint32_t (&r)[16]) {
      // k = 32 j .. 32 j + 31: box j / 2, chunks 4 (j % 2) .. + 3
      const uint32_t box = atom + (uint32_t)(j >> 1) * kABoxBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int chunk = 4 * (j & 1) + c;
        dev::st_shared_v4(box + (uint32_t)((chunk ^ (row & 7)) * 16), r[4 * c], r[4 * c + 1], r[4 * c + 2],
                          r[4 * c + 3]);
      }
    });
  };
  // the chunks of each tile the epilogue warpgroup decodes (the rest: warps 8..11)
  constexpr int kEpiJ1 = kDecWG == 2 ? 2 : 4;
  // A decoder's wait for packed tile kt at code-ring position `cp`.
  auto code_wait = [&](const RingPos& cp, int kt) {
    waiter.wait<false>(bar_full0 + 8u * (uint32_t)cp.index, cp.phase, kRoleEpiDecode, kt);
  };
  // The decoders' signals, one arrival a warp (a thread arrival each would
  // queue 128 or 256 shared-memory atomics on one barrier per tile): after a
  // warp synchronisation, which orders every lane's prior accesses (and,
  // after each lane's tcgen05 fence or proxy fence, its TMEM or shared-memory
  // stores) before lane 0's release.
  auto warp_arrive = [&](uint32_t bar) {
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(bar);
  };
  // Tile kt's codes (ring stage `stage`) read into registers: the stage may
  // take tile kt + stages (no arrival when there is none).
  auto code_free = [&](int kt, int stage) {
    if (kt + stages < k_tiles) warp_arrive(bar_empty0 + 8u * (uint32_t)stage);
  };

  if (warp == 0) {
    // ---- weight producer
    if (lane == 0) {
      RingPos pos = RingPos::at(a_issued, stages);
      for (int kt = a_issued; kt < k_tiles; ++kt, pos.advance(1, stages)) {
        const int s = pos.index;
        const uint32_t full = bar_full0 + 8u * s;
        // the stage's previous round (kt - stages) consumed
        if (!waiter.wait<false>(bar_empty0 + 8u * s, pos.phase ^ 1u, kRoleWeightTma, kt)) break;
        if constexpr (kQuant) {
          // packed codes: the stage is free once every decoder has read it
          dev::mbar_arrive_expect_tx(full, kQTileBytes);
          dev::tma_load_3d_hint(sA + (uint32_t)s * kQTileBytes, p.a_map, (kt0 + kt) * (int)kQRowBytes, n0, l,
                                full, a_policy);
        } else {
          const uint32_t dst = sA + (uint32_t)s * kAStageBytes;
          const int k = (kt0 + kt) * kCtaK;
          dev::mbar_arrive_expect_tx(full, kAStageBytes);
          dev::tma_load_3d_hint(dst, p.a_map, k, n0, l, full, a_policy);
          dev::tma_load_3d_hint(dst + kABoxBytes, p.a_map, k + kAtomK, n0, l, full, a_policy);
        }
        a_issued = kt + 1;
      }
      stamp(p, kTrWeightsIssued);
      if (!p.pdl_trigger_early) dev::griddep_launch_dependents();
    }
  } else if (warp == 1) {
    // ---- activation producer: B may be the previous kernel's output.
    if (lane == 0) {
      dev::griddep_wait();
      stamp(p, kTrActReady);
      if (b_res && !p.b_loader) {
        // Every activation K tile of this CTA at once, on one barrier.
        dev::mbar_arrive_expect_tx(bar_b, (uint32_t)k_tiles * kBStage);
        b_issued = true;
        for (int kt = 0; kt < k_tiles; ++kt) {
          const uint32_t dst = sB + (uint32_t)kt * kBStage;
          const int k = (kt0 + kt) * kCtaK;
          dev::tma_load_3d(dst, &b_map, k, m0, l, bar_b);
          dev::tma_load_3d(dst + kBBox, &b_map, k + kAtomK, m0, l, bar_b);
        }
      }
      RingPos pos{0, 0u};
      for (int kt = 0; kt < (b_res ? 0 : k_tiles); ++kt, pos.advance(1, stages)) {
        const int s = pos.index;
        const uint32_t full = bar_full0 + 8u * s;
        if (kt >= stages && !waiter.wait<false>(bar_empty0 + 8u * s, pos.phase ^ 1u, kRoleActTma, kt)) {
          break;
        }
        const uint32_t dst = sB + (uint32_t)s * kBStage;
        const int k = (kt0 + kt) * kCtaK;
        dev::mbar_arrive_expect_tx(full, kBStage);
        dev::tma_load_3d(dst, &b_map, k, m0, l, full);
        dev::tma_load_3d(dst + kBBox, &b_map, k + kAtomK, m0, l, full);
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ---- MMA issuers: D[128 x MMA_N] += A[128 x 16] * B[MMA_N x 16]^T, 8 per
    // K tile.  With two issuers (one tcgen05.mma stream per thread is
    // issue-bound at MMA_N <= 64), warp 2 takes the even K tiles into
    // accumulator 0 and warp 3 the odd ones into accumulator 1; the epilogue
    // adds the two.
    const int issuer = warp - 2;
    const int nis = p.mma_issuers;
    if (kQuant && lane == 0 && issuer < nis) {
      // Quantized weights: the epilogue threads decode each weight tile into a TMEM slot
      // (tile kt in slot kt % slots); the MMAs read A from there.  Issuer i
      // takes tiles i, i + nis, ... into its own accumulator.  The decoders
      // finish tiles in order, so an issuer that saw tile kt - nis full also
      // saw every earlier round of tile kt's slot complete (nis <= slots).
      const int slots = p.a_tmem_tiles;
      const uint32_t d_acc = tmem_base + (uint32_t)issuer * kAccCols;
      // descriptors by addition to the buffers' first (smem_desc_advance)
      const uint64_t b_desc0 = dev::smem_desc_sw128(sB), q_desc = dev::smem_desc_sw128(sQStage);
      bool ok = waiter.wait<false>(bar_b, 0u, kRoleMma, -1);
      dev::tc_fence_after();
      RingPos sp = RingPos::at(issuer, slots);                  // TMEM slot of tile kt
      for (int kt = issuer; kt < k_tiles && ok; kt += nis, sp.advance(nis, slots)) {
        const uint32_t first = (uint32_t)(kt >= nis);          // 0: this accumulator's first tile
        const uint64_t b_d = dev::smem_desc_advance(b_desc0, (uint32_t)kt * kBStage);
        if (p.w4_smem_tiles && kt == slots) {
          // the tile decoded into the bf16 stage in shared memory
          ok = waiter.wait<false>(bar_w4_stage, 0u, kRoleMma, kt);
          if (!ok) break;
          dev::tc_fence_after();
          if (kt == k_tiles - 1) stamp(p, kTrLastFull);
#pragma unroll
          for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
            const uint32_t a_off = (uint32_t)(kk >> 2) * kABoxBytes + (uint32_t)(kk & 3) * 32u;
            const uint32_t b_off = (uint32_t)(kk >> 2) * kBBox + (uint32_t)(kk & 3) * 32u;
            dev::mma_bf16(d_acc, dev::smem_desc_advance(q_desc, a_off), dev::smem_desc_advance(b_d, b_off),
                          kIdesc, (first | (uint32_t)kk) != 0u ? 1u : 0u);
          }
          continue;
        }
        const int slot = sp.index;
        ok = waiter.wait<false>(bar_slot_full0 + 8u * slot, sp.phase, kRoleMma, kt);
        if (!ok) break;
        dev::tc_fence_after();
        if (kt == 0) stamp(p, kTrFirstFull);
        if (kt == k_tiles - 1) stamp(p, kTrLastFull);
        const uint32_t t_col = tmem_base + p.tmem_tile_col0 + (uint32_t)slot * kTmemTileCols;
#pragma unroll
        for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
          const uint32_t b_off = (uint32_t)(kk >> 2) * kBBox + (uint32_t)(kk & 3) * 32u;
          dev::mma_bf16_ts(d_acc, t_col + (uint32_t)kk * 8u, dev::smem_desc_advance(b_d, b_off), kIdesc,
                           (first | (uint32_t)kk) != 0u ? 1u : 0u);
        }
        dev::mma_commit(bar_slot_empty0 + 8u * slot);   // slot free once these MMAs have read it
      }
      dev::mma_commit(bar_mma_done);
    }
    if (!kQuant && lane == 0 && issuer < nis) {
      const uint32_t d_acc = tmem_base + (uint32_t)issuer * kAccCols;
      // descriptors by addition to the buffers' first (smem_desc_advance)
      const uint64_t a_desc0 = dev::smem_desc_sw128(sA), b_desc0 = dev::smem_desc_sw128(sB);
      bool ok = true;
      // Before the activations can exist: copy this issuer's share of the
      // first `tmem_tiles` weight K tiles from the ring into tensor memory as
      // they land, so their stages take further tiles and more of the CTA's
      // weights are on chip when the previous kernel completes.
      RingPos cpos = RingPos::at(issuer, stages);
      for (int kt = issuer; kt < tmem_tiles && ok; kt += nis, cpos.advance(nis, stages)) {
        const int s = cpos.index;
        ok = waiter.wait<false>(bar_full0 + 8u * s, cpos.phase, kRoleMma, kt);
        if (!ok) break;
        dev::tc_fence_after();
        const uint64_t a_d = dev::smem_desc_advance(a_desc0, (uint32_t)s * kAStageBytes);
        const uint32_t t_col = tmem_base + p.tmem_tile_col0 + (uint32_t)kt * kTmemTileCols;
#pragma unroll
        for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
          const uint32_t a_off = (uint32_t)(kk >> 2) * kABoxBytes + (uint32_t)(kk & 3) * 32u;
          dev::tmem_cp_128x256b(t_col + (uint32_t)kk * 8u, dev::smem_desc_advance(a_d, a_off));
        }
        dev::mma_commit(bar_empty0 + 8u * s);  // stage free once the copies have read it
      }
      if (ok && b_res) {
        ok = waiter.wait<false>(bar_b, 0u, kRoleMma, -1);
        dev::tc_fence_after();
      }
      RingPos pos = RingPos::at(issuer, stages);
      for (int kt = issuer; kt < k_tiles && ok; kt += nis, pos.advance(nis, stages)) {
        const int s = pos.index;
        const uint32_t first = (uint32_t)(kt >= nis);          // 0: this accumulator's first tile
        const uint64_t b_d = dev::smem_desc_advance(b_desc0, (uint32_t)(b_res ? kt : s) * kBStage);
        if (kt == issuer) stamp(p, kTrFirstFull);
        if (kt < tmem_tiles) {
          // A from tensor memory (copied above, ordered before these MMAs)
          if (kt == k_tiles - 1) stamp(p, kTrLastFull);
          const uint32_t t_col = tmem_base + p.tmem_tile_col0 + (uint32_t)kt * kTmemTileCols;
#pragma unroll
          for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
            const uint32_t b_off = (uint32_t)(kk >> 2) * kBBox + (uint32_t)(kk & 3) * 32u;
            dev::mma_bf16_ts(d_acc, t_col + (uint32_t)kk * 8u, dev::smem_desc_advance(b_d, b_off), kIdesc,
                             (first | (uint32_t)kk) != 0u ? 1u : 0u);
          }
          continue;
        }
        ok = waiter.wait<false>(bar_full0 + 8u * s, pos.phase, kRoleMma, kt);
        if (!ok) break;
        dev::tc_fence_after();
        if (kt == k_tiles - 1) stamp(p, kTrLastFull);
        const uint64_t a_d = dev::smem_desc_advance(a_desc0, (uint32_t)s * kAStageBytes);
#pragma unroll
        for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
          const uint32_t a_off = (uint32_t)(kk >> 2) * kABoxBytes + (uint32_t)(kk & 3) * 32u;
          const uint32_t b_off = (uint32_t)(kk >> 2) * kBBox + (uint32_t)(kk & 3) * 32u;
          dev::mma_bf16(d_acc, dev::smem_desc_advance(a_d, a_off), dev::smem_desc_advance(b_d, b_off), kIdesc,
                        (first | (uint32_t)kk) != 0u ? 1u : 0u);
        }
        dev::mma_commit(bar_empty0 + 8u * s);  // stage free once these MMAs finish
      }
      dev::mma_commit(bar_mma_done);           // this issuer's accumulator complete
    }
    __syncwarp();
  } else if (kDecWG == 2 && warp >= 8) {
    // ---- second decoding warpgroup (quantized weights): chunks 2 and 3 (k 64..127) of
    // every tile's rows, into the same TMEM slots or bf16 stage
    const int row = (int)threadIdx.x - 256;
    const uint32_t t_row2 = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    const int slots = p.a_tmem_tiles;
    const bool row_ok = n0 + row < p.N;
    const uint8_t* srow =
        p.a_scale + ((size_t)l * p.N + (size_t)(row_ok ? n0 + row : 0)) * (size_t)(p.K / 32) + (size_t)kt0 * 4;
    ScaleWords scales;
    scales.load(reinterpret_cast<const uint32_t*>(srow), row_ok, k_tiles);
    RingPos cp{0, 0u}, sp{0, 0u};   // code-ring stage and TMEM slot of tile kt
    for (int kt = 0; kt < k_tiles; ++kt, cp.advance(1, stages), sp.advance(1, slots)) {
      if (p.w4_smem_tiles && kt == slots) {
        code_wait(cp, kt);
        const uint32_t codes = scales.take();
        q_decode_stage(cp.index, row, codes, kEpiJ1, 4);
        code_free(kt, cp.index);
        dev::fence_proxy_async_shared();
        warp_arrive(bar_w4_stage);
        continue;
      }
      const int slot = sp.index;
      // the slot's previous tile (kt - slots) read by the MMAs
      if (kt >= slots) waiter.wait<false>(bar_slot_empty0 + 8u * slot, sp.phase ^ 1u, kRoleEpiDecode, kt);
      code_wait(cp, kt);
      const uint32_t codes = scales.take();
      q_decode_tmem(cp.index, row, codes, t_row2 + p.tmem_tile_col0 + (uint32_t)slot * kTmemTileCols, kEpiJ1, 4);
      code_free(kt, cp.index);
      dev::tmem_wait_st();
      dev::tc_fence_before();
      warp_arrive(bar_slot_full0 + 8u * slot);
    }
  } else if (warp >= 4) {
    // ---- epilogue: thread et owns TMEM lane et = weight row n0 + et.
    const int et = (int)threadIdx.x - 128;
    const uint32_t t_row = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    const int ncols = (p.M - m0) < MMA_N ? (p.M - m0) : MMA_N;    // real token columns
    const bool two_acc = p.mma_issuers > 1 && k_tiles > 1;        // the odd K tiles' accumulator is in use
    const int nquads = (ncols + 3) >> 2;
    const int qr = p.mailbox_quads;                               // quads per round
    const bool owner = rank == 0;
    // Rank 0 stages its f32 tile [ncols][128] in its drained activation ring.
    float* const stage = reinterpret_cast<float*>(smem_raw + (sB - raw));
    const float* const mail = reinterpret_cast<const float*>(smem_raw + (sMail - raw));

    // The bias of the 8 weight rows this thread will store (a parameter like
    // A, read before the accumulator is complete).  Rank-0 stores: rows
    // (et % 16) * 8 of the tile; scattered stores: rows of this rank's slice.
    // Narrow tiles (at most 4 token columns) store each thread's own row:
    // the bias of row n0 + et.
    const bool narrow = !p.reduce_scatter && ncols <= 4;
    float bias8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (p.bias != nullptr && narrow) {
      if (n0 + et < p.N) bias8[0] = __uint_as_float((uint32_t)__ldg(p.bias + (size_t)l * (size_t)p.N + (size_t)(n0 + et)) << 16);
    } else if (p.bias != nullptr) {
      const int nb = n0 + (p.reduce_scatter ? rank * (kMmaM / split) + (et % (kMmaM / split / 8)) * 8
                                            : (et & 15) * 8);
      const uint16_t* bp = p.bias + (size_t)l * (size_t)p.N + (size_t)nb;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (nb + e < p.N) bias8[e] = __uint_as_float((uint32_t)__ldg(bp + e) << 16);
      }
    }

    // The activations of all of the CTA's K tiles, loaded by the epilogue
    // threads (idle until the accumulator is complete) with 16-byte loads
    // through L2 and stored in the 128-byte-swizzled layout the MMA reads:
    // 16-byte chunk c of row r of an 8-row atom lands at chunk c ^ (r % 8).
    // Columns past K are zero (the weights there are zero-filled, and
    // 0 * garbage could be NaN); rows past M are left unwritten -- they
    // only feed accumulator columns that are never read.
    auto load_activations = [&]() {
      dev::griddep_wait();
      const int cpr = k_tiles * (kCtaK / 8);           // 16-byte chunks per row
      for (int i = et; i < ncols * cpr; i += kEpiThreads) {
        const int r = i / cpr;
        const int ci = i - r * cpr;
        const int kt = ci >> 4, half = (ci >> 3) & 1, c = ci & 7;
        const int k = (kt0 + kt) * kCtaK + half * kAtomK + c * 8;
        uint32_t x0 = 0, x1 = 0, x2 = 0, x3 = 0;
        if (k < p.K) {
          dev::ld_global_cg_v4(p.b + ((size_t)l * p.M + (size_t)(m0 + r)) * (size_t)p.K + (size_t)k, x0, x1, x2, x3);
        }
        dev::st_shared_v4(sB + (uint32_t)kt * kBStage + (uint32_t)half * kBBox + (uint32_t)(r >> 3) * 1024u +
                              (uint32_t)(r & 7) * 128u + (uint32_t)((c ^ (r & 7)) * 16),
                          x0, x1, x2, x3);
      }
      dev::fence_proxy_async_shared();   // generic-proxy stores, read by tcgen05.mma
      dev::mbar_arrive(bar_b);
      if (et == 0) stamp(p, kTrActReady);
    };

    if constexpr (kQuant) {
      // Quantized weights: thread et decodes weight row n0 + et of each K tile into TMEM
      // lane et (with a second decoding warpgroup: chunks 0 and 1 of each
      // tile, the other group chunks 2 and 3).  The first `slots` tiles are
      // decoded before the previous kernel completes; with the epilogue
      // loading the activations, that load comes next, then the remaining
      // tiles as the MMAs free their slots.
      const int slots = p.a_tmem_tiles;
      const bool row_ok = n0 + et < p.N;
      const uint8_t* srow =
          p.a_scale + ((size_t)l * p.N + (size_t)(row_ok ? n0 + et : 0)) * (size_t)(p.K / 32) + (size_t)kt0 * 4;
      ScaleWords scales;
      scales.load(reinterpret_cast<const uint32_t*>(srow), row_ok, k_tiles);
      RingPos cp{0, 0u}, sp{0, 0u};   // code-ring stage and TMEM slot of tile kt
      for (int kt = 0; kt < k_tiles; ++kt, cp.advance(1, stages), sp.advance(1, slots)) {
        if (kt == slots && p.b_loader && !p.w4_smem_tiles) load_activations();
        if (p.w4_smem_tiles && kt == slots) {
          // the tile after the TMEM slots: decoded before the wait into the
          // bf16 stage in shared memory
          code_wait(cp, kt);
          const uint32_t codes = scales.take();
          q_decode_stage(cp.index, et, codes, 0, kEpiJ1);
          code_free(kt, cp.index);
          dev::fence_proxy_async_shared();   // generic-proxy stores, read by tcgen05.mma
          warp_arrive(bar_w4_stage);
          if (p.b_loader) load_activations();   // the stage is the last tile
          continue;
        }
        const int slot = sp.index;
        // the slot's previous tile (kt - slots) read by the MMAs
        if (kt >= slots) waiter.wait<false>(bar_slot_empty0 + 8u * slot, sp.phase ^ 1u, kRoleEpiDecode, kt);
        code_wait(cp, kt);
        const uint32_t codes = scales.take();
        q_decode_tmem(cp.index, et, codes, t_row + p.tmem_tile_col0 + (uint32_t)slot * kTmemTileCols, 0, kEpiJ1);
        code_free(kt, cp.index);
        dev::tmem_wait_st();
        dev::tc_fence_before();
        warp_arrive(bar_slot_full0 + 8u * slot);
      }
      if (p.b_loader && k_tiles <= slots) load_activations();
    } else if (p.b_loader) {
      load_activations();
    }

    waiter.wait<false>(bar_mma_done, 0u, kRoleEpiMma, 0);
    __syncwarp();
    dev::tc_fence_after();
    if (et == 0) stamp(p, kTrMmaDone);

    if (p.reduce_scatter) {
      // Scattered reduction: rank r sums and stores weight rows
      // [r*R, (r+1)*R) of the tile, R = 128 / split.  Each rank's partial of
      // those rows lands in rank r's mailbox, [source rank][R rows][column]
      // or [source rank][column][R rows] (below; its own by shared stores,
      // the others' by st.async), and every
      // element is summed over source ranks 0, 1, ... in order: the same
      // additions in the same order as rank 0 makes in the gathered mode,
      // with 1/split of the DSMEM bytes arriving at each SM.
      const int R = kMmaM / split;
      const int my_lo = rank * R;
      float* const mb = reinterpret_cast<float*>(smem_raw + (sMail - raw));
      if (et == 0) {
        dev::mbar_arrive_expect_tx(bar_reduce, (uint32_t)((split - 1) * ncols * R) * 4u);
      }
      // Thread et holds weight row et and sends it to the rank that sums it.
      // Whole quads of columns (ncols % 4 == 0): the mailbox is [source][row]
      // [column] and the row's columns go as 16-byte st.async, a quarter of
      // the remote stores.  Otherwise [source][column][row] with 4-byte ones
      // (a warp's 32 rows of one column are 128 contiguous bytes).
      const int dst_rank = et / R;
      const bool publish = !(p.inject & kInjectSkipPublish);
      const bool by_row = (ncols & 3) == 0;
      const uint32_t slot = by_row ? (uint32_t)((rank * R + (et - dst_rank * R)) * ncols) * 4u
                                   : ((uint32_t)(rank * ncols) * (uint32_t)R + (uint32_t)(et - dst_rank * R)) * 4u;
      const uint32_t r_bar = dev::mapa(bar_reduce, (uint32_t)dst_rank);
      const uint32_t r_mail = dev::mapa(sMail, (uint32_t)dst_rank) + slot;
#pragma unroll 1
      for (int g = 0; g * 16 < ncols; ++g) {
        uint32_t v[16];
        __syncwarp();   // tcgen05.ld is warp-collective
        load_acc16(t_row + (uint32_t)(g * 16), kAccCols, two_acc, v);
        if (by_row) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = g * 16 + 4 * q;
            if (col >= ncols) break;                          // warp-uniform
            if (dst_rank == rank) {
              dev::st_shared_v4(sMail + slot + (uint32_t)col * 4u, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else if (publish) {
              dev::st_async_v4(r_mail + (uint32_t)col * 4u, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], r_bar);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = g * 16 + e;
            if (col >= ncols) break;                          // warp-uniform
            if (dst_rank == rank) {
              *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(mb) + slot + (size_t)col * R * 4) = v[e];
            } else if (publish) {
              dev::st_async_b32(r_mail + (uint32_t)(col * R) * 4u, v[e], r_bar);
            }
          }
        }
      }
      // TMEM reads are done: let warp 2 release it.
      dev::tc_fence_before();
      dev::mbar_arrive(bar_tmem_empty);
      if (et == 0) stamp(p, kTrReduced);
      dev::named_bar_sync(1, kEpiThreads);                  // own slot complete
      waiter.wait<true>(bar_reduce, 0u, kRoleEpiReduce, 0);
      if (by_row) {
        // One weight row and 4 token columns per item: sum the sources in
        // rank order, four bf16 stores (one per token row of C).
        const int nq = ncols >> 2;
        const int items = R * nq;
#pragma unroll 1
        for (int it = et; it < items; it += kEpiThreads) {
          const int r = it / nq;
          const int c4 = (it - r * nq) * 4;
          const float* src = mb + (size_t)r * ncols + c4;
          float4 x = *reinterpret_cast<const float4*>(src);
#pragma unroll 1
          for (int sr = 1; sr < split; ++sr) {
            const float4 a4 = *reinterpret_cast<const float4*>(src + (size_t)sr * R * ncols);
            x.x += a4.x; x.y += a4.y; x.z += a4.z; x.w += a4.w;
          }
          const int n = n0 + my_lo + r;
          if (n >= p.N) continue;
          const float bv = p.bias != nullptr
                               ? __uint_as_float((uint32_t)__ldg(p.bias + (size_t)l * (size_t)p.N + (size_t)n) << 16)
                               : 0.0f;
          uint16_t* dst = p.c + ((size_t)((size_t)l * p.M + (size_t)(m0 + c4)) * (size_t)p.N + (size_t)n);
          dst[0] = (uint16_t)(dev::pack_bf16x2(x.x + bv, 0.0f) & 0xFFFFu);
          dst[(size_t)p.N] = (uint16_t)(dev::pack_bf16x2(x.y + bv, 0.0f) & 0xFFFFu);
          dst[(size_t)2 * p.N] = (uint16_t)(dev::pack_bf16x2(x.z + bv, 0.0f) & 0xFFFFu);
          dst[(size_t)3 * p.N] = (uint16_t)(dev::pack_bf16x2(x.w + bv, 0.0f) & 0xFFFFu);
        }
        if (et == 0) stamp(p, kTrStored);
      } else {
      // 8 weight rows of one token column per item: sum the sources in rank
      // order, pack bf16 pairs, one 16-byte store.
      const int chunks = R / 8;
      const int items = ncols * chunks;
#pragma unroll 1
      for (int it = et; it < items; it += kEpiThreads) {
        const int m = it / chunks;
        const int c8 = (it - m * chunks) * 8;
        const float* src = mb + (size_t)m * R + c8;
        float4 x = *reinterpret_cast<const float4*>(src);
        float4 y = *reinterpret_cast<const float4*>(src + 4);
#pragma unroll 1
        for (int sr = 1; sr < split; ++sr) {
          const float* ps = src + (size_t)sr * ncols * R;
          const float4 a4 = *reinterpret_cast<const float4*>(ps);
          const float4 b4 = *reinterpret_cast<const float4*>(ps + 4);
          x.x += a4.x; x.y += a4.y; x.z += a4.z; x.w += a4.w;
          y.x += b4.x; y.y += b4.y; y.z += b4.z; y.w += b4.w;
        }
        const int n = n0 + my_lo + c8;
        if (n >= p.N) continue;
        x.x += bias8[0]; x.y += bias8[1]; x.z += bias8[2]; x.w += bias8[3];
        y.x += bias8[4]; y.y += bias8[5]; y.z += bias8[6]; y.w += bias8[7];
        const uint32_t q0 = dev::pack_bf16x2(x.x, x.y), q1 = dev::pack_bf16x2(x.z, x.w);
        const uint32_t q2 = dev::pack_bf16x2(y.x, y.y), q3 = dev::pack_bf16x2(y.z, y.w);
        uint16_t* dst = p.c + ((size_t)((size_t)l * p.M + (size_t)(m0 + m)) * (size_t)p.N + (size_t)n);
        if (p.vec_store && n + 8 <= p.N) {
          dev::st_global_v4(dst, q0, q1, q2, q3);
        } else {
          store8_clipped(dst, n, p.N, q0, q1, q2, q3);
        }
      }
      if (et == 0) stamp(p, kTrStored);
      }
    } else if (narrow) {
      // One round, each thread its own weight row: peers send each live
      // column with a 4-byte st.async into rank 0's mailbox [peer-1][column]
      // [row]; rank 0 adds peers 1, 2, ... in rank order (the same additions
      // as the wide path) and stores its row's outputs itself.
      uint32_t v[4];
      __syncwarp();   // tcgen05.ld is warp-collective
      load_acc4(t_row, kAccCols, two_acc, v);
      if (split > 1 && !owner) {
        bool publish = !(p.inject & kInjectSkipPublish);
        if (publish && !p.mailbox_dedicated) {
          publish = waiter.wait<true>(bar_ready, 0u, kRoleEpiReady, 0);
        }
        dev::tc_fence_before();
        dev::mbar_arrive(bar_tmem_empty);
        if (publish) {
          const uint32_t r_bar = dev::mapa(bar_reduce, 0u);
          const uint32_t r_mail =
              dev::mapa(sMail, 0u) + (uint32_t)((rank - 1) * ncols) * kColumnBytes + (uint32_t)et * 4u;
#pragma unroll
          for (int col = 0; col < 4; ++col) {
            if (col < ncols) dev::st_async_b32(r_mail + (uint32_t)col * kColumnBytes, v[col], r_bar);
          }
        }
        if (et == 0) stamp(p, kTrReduced);
      } else {
        if (split > 1) {
          if (et == 0) {
            dev::mbar_arrive_expect_tx(bar_reduce, (uint32_t)(split - 1) * (uint32_t)ncols * kColumnBytes);
          }
          if (!p.mailbox_dedicated && et >= 1 && et < split) {
            dev::mbar_arrive_remote(dev::mapa(bar_ready, (uint32_t)et));
          }
        }
        float x[4];
#pragma unroll
        for (int col = 0; col < 4; ++col) x[col] = __uint_as_float(v[col]);
        dev::tc_fence_before();
        dev::mbar_arrive(bar_tmem_empty);
        if (split > 1) {
          waiter.wait<true>(bar_reduce, 0u, kRoleEpiReduce, 0);
#pragma unroll 1
          for (int peer = 1; peer < split; ++peer) {
            const float* mp = mail + (size_t)((peer - 1) * ncols) * kEpiThreads + et;
#pragma unroll
            for (int col = 0; col < 4; ++col) {
              if (col < ncols) x[col] += mp[(size_t)col * kEpiThreads];
            }
          }
        }
        if (et == 0) stamp(p, kTrReduced);
        const int n = n0 + et;
        if (n < p.N) {
          uint16_t* dst = p.c + ((size_t)l * p.M + (size_t)m0) * (size_t)p.N + (size_t)n;
#pragma unroll
          for (int col = 0; col < 4; ++col) {
            if (col < ncols) dst[(size_t)col * p.N] = (uint16_t)(dev::pack_bf16x2(x[col] + bias8[0], 0.0f) & 0xFFFFu);
          }
        }
        if (et == 0) stamp(p, kTrStored);
      }
    } else {
      int round = 0;
      // A round whose reduction wait failed leaves its barrier phase open:
      // rank 0 then arms no further round (an arrival on a phase with no
      // pending arrivals is undefined).
      bool reduce_ok = true;
      for (int qb = 0; qb < nquads; qb += qr, ++round) {
        const int q_end = (nquads - qb) < qr ? nquads : qb + qr;
        const int c_lo = qb * 4;
        // Mailbox of a round: [peer - 1][column - c_lo][row], f32; only the
        // round's real token columns [c_lo, c_hi) travel.
        const int c_hi = (ncols < q_end * 4) ? ncols : q_end * 4;
        const int rc = c_hi - c_lo;
        // The aliased mailbox (and any later round) waits for rank 0 to free it.
        const bool need_ready = split > 1 && !(p.mailbox_dedicated && round == 0);
        if (split > 1 && owner) {
          if (et == 0 && reduce_ok) {
            dev::mbar_arrive_expect_tx(bar_reduce, (uint32_t)(split - 1) * (uint32_t)rc * kColumnBytes);
          }
          // One thread per peer, in parallel: a release arrival waits for the
          // issuing thread's earlier memory operations, so arrivals issued one
          // after another from a single thread would serialise into round trips.
          if (need_ready && et >= 1 && et < split) {
            dev::mbar_arrive_remote(dev::mapa(bar_ready, (uint32_t)et));
          }
        }
        const uint32_t r_bar = dev::mapa(bar_reduce, 0u);
        const uint32_t r_mail = dev::mapa(sMail, 0u) + (uint32_t)((rank - 1) * rc) * kColumnBytes;
        bool publish = split > 1 && !owner && !(p.inject & kInjectSkipPublish);
        bool first_group = true;

        // 16 token columns per TMEM load; quads of 4 columns within.
  #pragma unroll 1
        for (int g = qb >> 2; g * 4 < q_end; ++g, first_group = false) {
          uint32_t v[16];
          __syncwarp();   // tcgen05.ld is warp-collective
          load_acc16(t_row + (uint32_t)(g * 16), kAccCols, two_acc, v);
          if (split > 1 && !owner) {
            if (first_group && publish && need_ready) {
              publish = waiter.wait<true>(bar_ready,
                                          (uint32_t)((round - (p.mailbox_dedicated ? 1 : 0)) & 1),
                                          kRoleEpiReady, round);
            }
            if (publish) {
              // Thread et sends row et of each live column; a warp's 32 rows
              // of one column are 128 contiguous bytes of the mailbox.
  #pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int col = g * 16 + e;
                if (col >= c_lo && col < c_hi) {                  // warp-uniform
                  dev::st_async_b32(r_mail + (uint32_t)(col - c_lo) * kColumnBytes + (uint32_t)et * 4u, v[e],
                                    r_bar);
                }
              }
            }
          } else {
            float x[16];
  #pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(v[e]);
            if (split > 1) {
              if (first_group && reduce_ok) {
                reduce_ok = waiter.wait<true>(bar_reduce, (uint32_t)(round & 1), kRoleEpiReduce, round);
              }
              // rank 0's partial + peers 1, 2, ... in rank order; each peer's
              // 16 columns are loaded together.
  #pragma unroll 1
              for (int peer = 1; peer < split; ++peer) {
                const float* mp = mail + ((size_t)((peer - 1) * rc + (g * 16 - c_lo)) * kEpiThreads + et);
                float w[16];
  #pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int c0 = g * 16 + 4 * j;
                  if (c0 >= c_lo && c0 < c_hi) {                  // live quad (warp-uniform)
  #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      w[4 * j + i] = (c0 + i < c_hi) ? mp[(size_t)(4 * j + i) * kEpiThreads] : 0.0f;
                    }
                  } else {
                    w[4 * j] = w[4 * j + 1] = w[4 * j + 2] = w[4 * j + 3] = 0.0f;
                  }
                }
  #pragma unroll
                for (int e = 0; e < 16; ++e) x[e] += w[e];
              }
            }
  #pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int col = g * 16 + e;
              if (col >= c_lo && col < c_hi) stage[(size_t)col * kMmaM + et] = x[e];
            }
          }
        }
        // Every rank-0 thread has read this round before the mailbox is reused.
        if (split > 1 && owner && q_end < nquads) dev::named_bar_sync(1, kEpiThreads);
      }
      // TMEM reads are done: let warp 2 release it.
      dev::tc_fence_before();
      dev::mbar_arrive(bar_tmem_empty);
      if (et == 0) stamp(p, kTrReduced);

      if (owner) {
        // Rank 0 stores the tile: 16 vectors of 8 bf16 per token row, packed in
        // pairs (low half first) and coalesced along n.
        dev::named_bar_sync(1, kEpiThreads);
        const int total = ncols * (kMmaM / 8);
  #pragma unroll 1
        for (int idx = et; idx < total; idx += kEpiThreads) {
          const int row = idx >> 4;
          const int c8 = (idx & 15) * 8;
          const int n = n0 + c8;
          if (n >= p.N) continue;
          float4 x = *reinterpret_cast<const float4*>(stage + row * kMmaM + c8);
          float4 y = *reinterpret_cast<const float4*>(stage + row * kMmaM + c8 + 4);
          x.x += bias8[0]; x.y += bias8[1]; x.z += bias8[2]; x.w += bias8[3];
          y.x += bias8[4]; y.y += bias8[5]; y.z += bias8[6]; y.w += bias8[7];
          const uint32_t q0 = dev::pack_bf16x2(x.x, x.y), q1 = dev::pack_bf16x2(x.z, x.w);
          const uint32_t q2 = dev::pack_bf16x2(y.x, y.y), q3 = dev::pack_bf16x2(y.z, y.w);
          uint16_t* dst = p.c + ((size_t)((size_t)l * p.M + (size_t)(m0 + row)) * (size_t)p.N + (size_t)n);
          if (p.vec_store && n + 8 <= p.N) {
            dev::st_global_v4(dst, q0, q1, q2, q3);
          } else {
            store8_clipped(dst, n, p.N, q0, q1, q2, q3);
          }
        }
        if (et == 0) stamp(p, kTrStored);
      }
    }
  }

  // ---- teardown
  if (dev::ld_shared_u32(slot_abort) != 0u) {
    // A wait failed somewhere in this CTA, so consumers may have stopped
    // waiting for copies that are still landing in this CTA's shared memory:
    // let them land (bounded) before the CTA leaves.  For each ring stage
    // the last round issued is the one to wait for; earlier rounds completed
    // before the stage was refilled.
    const unsigned long long drain_ns = 10000000ull;   // 10 ms
    if (threadIdx.x == 0) {
      for (int s = 0; s < a_issued && s < stages; ++s) {
        const int round = (a_issued - 1 - s) / stages;   // of the last tile issued to stage s
        drain_wait(bar_full0 + 8u * s, (uint32_t)(round & 1), drain_ns);
      }
    }
    if (warp == 1 && lane == 0 && b_issued) drain_wait(bar_b, 0u, drain_ns);
    // the peers' partials of a dedicated single-round (or scattered) reduction,
    // which no final cluster barrier covers
    const int tq = (((p.M - m0) < MMA_N ? (p.M - m0) : MMA_N) + 3) >> 2;
    if (threadIdx.x == 128 && split > 1 && p.mailbox_dedicated && tq <= p.mailbox_quads &&
        (p.reduce_scatter || rank == 0)) {
      drain_wait(bar_reduce, 0u, drain_ns);
    }
  }
  if (warp == 2) {
    waiter.wait<false>(bar_mma_done, 0u, kRoleTmemRelease, 0, 4);
    waiter.wait<false>(bar_tmem_empty, 0u, kRoleTmemRelease, 1, 4);
    dev::tc_fence_after();
    __syncwarp();
    dev::tmem_dealloc(tmem_base, p.tmem_cols);
  }
  // With a dedicated mailbox and a single reduction round, rank 0 never
  // addresses a peer's shared memory and its reduction wait proves every
  // peer's bytes have landed: each CTA leaves as soon as it is done, so a
  // peer's shared memory is free for the next kernel's CTAs while rank 0 is
  // still reducing.  (A peer later than rank 0's whole wait limit would
  // publish into a departed CTA; the limit is chosen so that never happens.)
  const int tile_quads = (((p.M - m0) < MMA_N ? (p.M - m0) : MMA_N) + 3) >> 2;
  const bool final_barrier = split > 1 && !(p.mailbox_dedicated && tile_quads <= p.mailbox_quads);
  if (final_barrier) {
    // No CTA leaves while a peer may still address its shared memory.  The
    // arrival is relaxed (a release would wait for the tile's global
    // stores): rank 0's remote arrivals on the peers' barriers were observed
    // by the peers before they published, and rank 0 has received every
    // peer's bytes.  A CTA whose wait failed fences its remote operations
    // first instead.
    if (dev::ld_shared_u32(slot_abort) != 0u) dev::fence_acq_rel_cluster();
    __syncwarp();
    dev::cluster_arrive_relaxed();
    dev::cluster_wait_acquire();
  }
  if (threadIdx.x == 0) stamp(p, kTrEnd);
}

// ---------------------------------------------------------------- host side
namespace {

template <int MMA_N, int kFmt, int kDecWG = 1>
cudaError_t launch_t(const LaunchArgs& la, const CUtensorMap& b_map, const KernelParams& p,
                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = la.grid;
  cfg.blockDim = dim3(kDecWG == 2 ? kThreadsW4Wide : kThreads, 1, 1);
  cfg.dynamicSmemBytes = la.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeClusterDimension;
  attrs[n].val.clusterDim.x = la.cluster_x;
  attrs[n].val.clusterDim.y = 1;
  attrs[n].val.clusterDim.z = 1;
  ++n;
  if (la.pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, splitk_gemm_bf16_kernel<MMA_N, kFmt, kDecWG>, b_map, p);
}

template <int MMA_N, int kFmt, int kDecWG = 1>
cudaError_t prepare_t(int max_dynamic_smem) {
  return cudaFuncSetAttribute(splitk_gemm_bf16_kernel<MMA_N, kFmt, kDecWG>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
}

template <int kFmt>
cudaError_t launch_quantized(const LaunchArgs& la, const CUtensorMap& b_map, const KernelParams& p,
                             cudaStream_t stream) {
  // quantized weights: decode-sized tiles only
  if (la.w4_decoders == 2) {
    switch (la.mma_n) {
      case 16: return launch_t<16, kFmt, 2>(la, b_map, p, stream);
      case 32: return launch_t<32, kFmt, 2>(la, b_map, p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (la.mma_n) {
    case 16: return launch_t<16, kFmt>(la, b_map, p, stream);
    case 32: return launch_t<32, kFmt>(la, b_map, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int kFmt>
cudaError_t prepare_quantized(int max_dynamic_smem) {
  cudaError_t e;
  if ((e = prepare_t<16, kFmt>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_t<32, kFmt>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_t<16, kFmt, 2>(max_dynamic_smem)) != cudaSuccess) return e;
  return prepare_t<32, kFmt, 2>(max_dynamic_smem);
}

}  // namespace

cudaError_t launch_kernel(const LaunchArgs& la, const CUtensorMap& b_map, const KernelParams& p,
                          cudaStream_t stream) {
  if (la.fmt == 1) return launch_quantized<1>(la, b_map, p, stream);
  if (la.fmt == 2) return launch_quantized<2>(la, b_map, p, stream);
  switch (la.mma_n) {
    case 16: return launch_t<16, 0>(la, b_map, p, stream);
    case 32: return launch_t<32, 0>(la, b_map, p, stream);
    case 64: return launch_t<64, 0>(la, b_map, p, stream);
    case 128: return launch_t<128, 0>(la, b_map, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_kernels(int max_dynamic_smem) {
  cudaError_t e;
  if ((e = prepare_t<16, 0>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_t<32, 0>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_t<64, 0>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_t<128, 0>(max_dynamic_smem)) != cudaSuccess) return e;
  if ((e = prepare_quantized<1>(max_dynamic_smem)) != cudaSuccess) return e;
  return prepare_quantized<2>(max_dynamic_smem);
}

cudaError_t read_and_clear_fault(int* out_words) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out_words, g_fault, sizeof(int) * kFaultWords);
  if (e != cudaSuccess) return e;
  int zeros[kFaultWords] = {0};
  return cudaMemcpyToSymbol(g_fault, zeros, sizeof(zeros));
}

}  // namespace splitk
