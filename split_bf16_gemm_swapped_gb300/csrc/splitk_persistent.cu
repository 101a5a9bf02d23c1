// The persistent split-K kernel for sm_103a: the same GEMM as
// splitk_gemm_bf16_kernel, C[l][m][n] = bf16_rne( sum_k A[l][n][k] * B[l][m][k] ),
// for grids of many output tiles per split-K cluster (wide tiles, long K,
// splits of 2 and more).
//
// The per-tile kernel reduces a tile's partials only after its whole K slice
// has streamed, and with one CTA per SM nothing streams meanwhile: at wide
// tiles and large splits the memory pipe idles for the reduction.  Here a
// cluster of split CTAs (one per SM) stays resident and walks the output
// tiles cy, cy + clusters, cy + 2 clusters, ... (cy = the cluster's index),
// every rank taking its K slice of each.  The weight and activation rings run
// on across tiles, and the tile's accumulator alternates between two TMEM
// buffers, so the MMAs of tile j + 1 and the loads behind them proceed while
// the epilogue reduces tile j.  The two rings have their own depths: at wide
// tiles an activation K tile is as large as a weight K tile but comes from
// L2, so a shallower activation ring leaves shared memory for more weight
// tiles in flight from DRAM.
//
// Reduction: the page's rank order, scattered as in the per-tile kernel's
// reduce_scatter mode -- rank r sums weight rows [r*R, (r+1)*R), R = 128 /
// split, over source ranks 0, 1, ..., split-1 in that order (the same FP32
// additions as rank 0 makes in the gathered mode, so the same bits).  Each
// rank has one mailbox holding the columns of one reduction round (a whole
// tile, or a group of its columns when the mailbox is smaller), laid out
// [source][R rows][columns] for rounds of whole column quads (each row sent
// as 16-byte st.async) and [source][columns][R rows] otherwise (4-byte
// st.async); before publishing a round into a peer's mailbox a rank waits
// until every peer has signalled (a remote mbarrier arrival) that it has
// read its mailbox of the previous round.
//
// CTA roles (256 threads):
//   warp 0      weight producer: TMA, L2 evict_first, the first ring pass
//               issued before the cluster barrier and the PDL wait
//   warp 1      activation producer: griddepcontrol.wait, then TMA into the
//               activation ring
//   warp 2      TMEM (two accumulators) and the tcgen05.mma issue
//   warp 3      barrier initialisation, then idle (it keeps warps 4..7 on
//               TMEM lane quadrants 0..3)
//   warps 4..7  epilogue: TMEM -> registers, DSMEM publish, rank-ordered sum
//               of the CTA's rows, bf16 packing, 16-byte stores
//
// Every wait is bounded as in the per-tile kernel (a timeout records the
// fault, the CTA's later waits give up at once); TMEM is always released;
// the CTAs of a cluster leave together after a final cluster barrier.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "splitk.h"
#include "splitk_device.cuh"
#include "splitk_internal.h"
#include "splitk_kernel_common.cuh"

namespace splitk {

template <int MMA_N, bool kOneRing>
__global__ void __launch_bounds__(kThreads, 1)
    splitk_persistent_kernel(const __grid_constant__ CUtensorMap b_map, const KernelParams p) {
  constexpr uint32_t kBStage = b_stage_bytes(MMA_N);
  constexpr uint32_t kBBox = kBStage / 2;                   // MMA_N rows x 128 B
  constexpr uint32_t kAccCols = tmem_acc_cols(MMA_N);       // TMEM columns of one accumulator
  constexpr uint32_t kIdesc = dev::idesc_bf16_f32(kMmaM, MMA_N);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + (kAlignSlack - 1)) & ~(kAlignSlack - 1);

  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);
  const int split = p.split;
  const int a_stages = p.stages;     // weight ring depth
  const int b_stages = p.b_stages;   // activation ring depth
  // Rings of one depth (kOneRing) share their barriers: one full barrier per
  // stage that both producers arrive on, one MMA commit per K tile.  A
  // compile-time choice: a second wait and commit on the MMA issuer's path
  // measured 2-6 % slower, and a run-time test of the depths 1.5-2.5 %.
  constexpr bool one_ring = kOneRing;
  const int rank = (int)dev::cluster_ctarank();
  // Output tiles: m (token tiles) fastest, then n, then l.  The clusters
  // working at the same time then share each weight tile's reads when there
  // are several token tiles (the later reads hit L2), and activation tiles
  // in L2 either way.
  const int m_tiles = (p.M + MMA_N - 1) / MMA_N;
  const int n_tiles = (p.N + kMmaM - 1) / kMmaM;
  const long long tiles = (long long)m_tiles * n_tiles * p.L;
  const int cy = (int)blockIdx.y;
  const int clusters = (int)gridDim.y;
  const int my_tiles = cy < tiles ? (int)((tiles - cy + clusters - 1) / clusters) : 0;
  // Contiguous K slices: ranks below T % split take one extra tile.
  const int kt_base = p.k_tiles_total / split;
  const int kt_extra = p.k_tiles_total % split;
  const int k_tiles = kt_base + (rank < kt_extra ? 1 : 0);
  const int kt0 = rank * kt_base + (rank < kt_extra ? rank : kt_extra);

  // Shared memory: [A ring][B ring][mailbox][barriers].
  const uint32_t sA = base;
  const uint32_t sB = sA + (uint32_t)a_stages * kAStageBytes;
  const uint32_t sMail = sB + (uint32_t)b_stages * kBStage;
  const uint32_t sBar = sMail + p.mailbox_bytes;
  const uint32_t bar_a_full0 = sBar;                        // [kMaxStages] weight tile landed, count 1 (2: one ring)
  const uint32_t bar_a_empty0 = sBar + 8u * kMaxStages;     // [kMaxStages] its MMAs done (commit), count 1
  // [kMaxStages] activation tile landed / its MMAs done, count 1 (one ring: the weight ring's)
  const uint32_t bar_b_full0 = one_ring ? bar_a_full0 : sBar + 16u * kMaxStages;
  const uint32_t bar_b_empty0 = one_ring ? bar_a_empty0 : sBar + 24u * kMaxStages;
  const uint32_t bar_acc_full0 = sBar + (one_ring ? 16u : 32u) * kMaxStages;   // [2] accumulator complete, count 1
  const uint32_t bar_acc_empty0 = bar_acc_full0 + 16u;      // [2] accumulator read, count 128
  const uint32_t bar_reduce = bar_acc_full0 + 32u;          // count 1 + tx bytes of the peers
  const uint32_t bar_ready = bar_acc_full0 + 40u;           // count split - 1 (one per peer)
  const uint32_t slot_tmem = bar_acc_full0 + 48u;
  const uint32_t slot_abort = bar_acc_full0 + 52u;
  const uint32_t bar_mma_done = bar_acc_full0 + 56u;        // every MMA issued has completed, count 1

  const Waiter waiter{slot_abort, p.wait_limit_ns};

  auto tile_coords = [&](int j, int* n0, int* m0, int* l) {
    const long long t = (long long)cy + (long long)j * clusters;
    const long long r = t / m_tiles;
    *m0 = (int)(t - r * m_tiles) * MMA_N;
    *n0 = (int)(r % n_tiles) * kMmaM;
    *l = (int)(r / n_tiles);
  };

  // ---- set-up: warp 3 initialises the barriers, warp 2 allocates TMEM,
  // warp 0 acquires A's tensor map and issues the first ring pass of weight
  // loads (they depend on nothing the previous kernel writes).
  int a_issued = 0;      // weight K tiles issued so far (over all tiles)
  int b_issued = 0;      // activation K tiles issued so far
  uint64_t a_policy = 0;
  const int total_kt = my_tiles * k_tiles;
  if (warp == 3) {
    if (lane == 0) {
      for (int s = 0; s < a_stages; ++s) {
        dev::mbar_init(bar_a_full0 + 8u * s, one_ring ? 2u : 1u);
        dev::mbar_init(bar_a_empty0 + 8u * s, 1u);
      }
      for (int s = 0; !one_ring && s < b_stages; ++s) {
        dev::mbar_init(bar_b_full0 + 8u * s, 1u);
        dev::mbar_init(bar_b_empty0 + 8u * s, 1u);
      }
      for (int i = 0; i < 2; ++i) {
        dev::mbar_init(bar_acc_full0 + 8u * i, 1u);
        dev::mbar_init(bar_acc_empty0 + 8u * i, (uint32_t)kEpiThreads);
      }
      dev::mbar_init(bar_reduce, 1u);
      dev::mbar_init(bar_ready, (uint32_t)(split - 1));
      dev::mbar_init(bar_mma_done, 1u);
      dev::st_shared_u32(slot_abort, 0u);
      dev::fence_barrier_init();
      stamp(p, kTrBarInit);
    }
    dev::named_bar_sync(2, 64);
  } else if (warp == 0) {
    if (lane == 0) {
      stamp(p, kTrStart);
      dev::tensormap_acquire(p.a_map);
      stamp(p, kTrMapReady);
      // Weights are read once (evict first), or once per token tile by
      // clusters working side by side (kept for the later reads).
      a_policy = m_tiles == 1 ? dev::policy_evict_first() : dev::policy_evict_normal();
    }
    dev::named_bar_sync(2, 64);
  } else if (warp == 2) {
    dev::tmem_alloc(slot_tmem, p.tmem_cols);
    dev::tmem_relinquish();
    dev::tc_fence_before();
    if (lane == 0) stamp(p, kTrTmemAlloc);
  }
  dev::cluster_arrive_release();
  if (threadIdx.x == 0) {
    const int first = total_kt < a_stages ? total_kt : a_stages;
    int j = 0, kt = 0, n0 = 0, m0 = 0, l = 0;
    if (first > 0) tile_coords(0, &n0, &m0, &l);
    for (; a_issued < first; ++a_issued, ++kt) {
      if (kt == k_tiles) {
        kt = 0;
        tile_coords(++j, &n0, &m0, &l);
      }
      const uint32_t full = bar_a_full0 + 8u * a_issued;
      const uint32_t dst = sA + (uint32_t)a_issued * kAStageBytes;
      const int k = (kt0 + kt) * kCtaK;
      dev::mbar_arrive_expect_tx(full, kAStageBytes);
      dev::tma_load_3d_hint(dst, p.a_map, k, n0, l, full, a_policy);
      dev::tma_load_3d_hint(dst + kABoxBytes, p.a_map, k + kAtomK, n0, l, full, a_policy);
    }
    stamp(p, kTrPrefetched);
  }
  dev::cluster_wait_acquire();
  dev::tc_fence_after();
  const uint32_t tmem_base = dev::ld_shared_u32(slot_tmem);
  if (threadIdx.x == 0) {
    stamp(p, kTrSynced);
    if (p.trace != nullptr) {
      const uint32_t cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
      if (cta < p.trace_ctas) {
        uint32_t sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        p.trace[(size_t)cta * kTraceSlots + kTrSmRank] = (unsigned long long)sm | ((unsigned long long)rank << 32);
      }
    }
  }

  int reduce_armed = -1;  // epilogue thread 0: parity of a reduction phase armed but not seen complete
  if (warp == 0) {
    // ---- weight producer: the ring continues across tiles
    if (lane == 0) {
      // ring position and (output tile, K tile) of global load g, kept by
      // additions; the tile's coordinates recomputed once per output tile
      RingPos pos = RingPos::at(a_issued, a_stages);
      int j = a_issued / k_tiles;
      int kt = a_issued - j * k_tiles;
      int n0 = 0, m0 = 0, l = 0;
      if (a_issued < total_kt) tile_coords(j, &n0, &m0, &l);
      for (int g = a_issued; g < total_kt; ++g, pos.advance(1, a_stages)) {
        if (kt == k_tiles) {
          kt = 0;
          tile_coords(++j, &n0, &m0, &l);
        }
        const int s = pos.index;
        if (!waiter.wait<false>(bar_a_empty0 + 8u * s, pos.phase ^ 1u, kRoleWeightTma, g)) break;
        const uint32_t full = bar_a_full0 + 8u * s;
        const uint32_t dst = sA + (uint32_t)s * kAStageBytes;
        const int k = (kt0 + kt) * kCtaK;
        dev::mbar_arrive_expect_tx(full, kAStageBytes);
        dev::tma_load_3d_hint(dst, p.a_map, k, n0, l, full, a_policy);
        dev::tma_load_3d_hint(dst + kABoxBytes, p.a_map, k + kAtomK, n0, l, full, a_policy);
        a_issued = g + 1;
        ++kt;
      }
      stamp(p, kTrWeightsIssued);
      dev::griddep_launch_dependents();
    }
  } else if (warp == 1) {
    // ---- activation producer: B may be the previous kernel's output
    if (lane == 0) {
      dev::griddep_wait();
      stamp(p, kTrActReady);
      RingPos pos{0, 0u};
      int j = 0, kt = 0, n0 = 0, m0 = 0, l = 0;
      if (total_kt > 0) tile_coords(0, &n0, &m0, &l);
      for (int g = 0; g < total_kt; ++g, pos.advance(1, b_stages)) {
        if (kt == k_tiles) {
          kt = 0;
          tile_coords(++j, &n0, &m0, &l);
        }
        const int s = pos.index;
        if (g >= b_stages && !waiter.wait<false>(bar_b_empty0 + 8u * s, pos.phase ^ 1u, kRoleActTma, g)) {
          break;
        }
        const uint32_t full = bar_b_full0 + 8u * s;
        const uint32_t dst = sB + (uint32_t)s * kBStage;
        const int k = (kt0 + kt) * kCtaK;
        dev::mbar_arrive_expect_tx(full, kBStage);
        dev::tma_load_3d(dst, &b_map, k, m0, l, full);
        dev::tma_load_3d(dst + kBBox, &b_map, k + kAtomK, m0, l, full);
        b_issued = g + 1;
        ++kt;
      }
    }
  } else if (warp == 2) {
    // ---- MMA issuer: tile j accumulates into buffer j & 1, once the
    // epilogue has read that buffer's previous tile (j - 2)
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      RingPos pa{0, 0u}, pb{0, 0u};                  // weight / activation ring positions of load g
      const uint64_t a_desc0 = dev::smem_desc_sw128(sA), b_desc0 = dev::smem_desc_sw128(sB);
      for (int j = 0; j < my_tiles && ok; ++j) {
        const int buf = j & 1;
        const int use = j >> 1;
        if (use > 0) {
          ok = waiter.wait<false>(bar_acc_empty0 + 8u * buf, (uint32_t)((use - 1) & 1), kRoleMmaAccFree, j);
          if (!ok) break;
          dev::tc_fence_after();
        }
        const uint32_t d_acc = tmem_base + (uint32_t)buf * kAccCols;
        for (int kt = 0; kt < k_tiles; ++kt, ++g, pa.advance(1, a_stages), pb.advance(1, b_stages)) {
          ok = waiter.wait<false>(bar_a_full0 + 8u * pa.index, pa.phase, kRoleMma, g) &&
               (one_ring || waiter.wait<false>(bar_b_full0 + 8u * pb.index, pb.phase, kRoleMma, g));
          if (!ok) break;
          dev::tc_fence_after();
          if (g == 0) stamp(p, kTrFirstFull);
          // the stages' descriptors by addition to the rings' first
          const uint64_t a_d = dev::smem_desc_advance(a_desc0, (uint32_t)pa.index * kAStageBytes);
          const uint64_t b_d = dev::smem_desc_advance(b_desc0, (uint32_t)pb.index * kBStage);
#pragma unroll
          for (int kk = 0; kk < kCtaK / kMmaK; ++kk) {
            const uint32_t a_off = (uint32_t)(kk >> 2) * kABoxBytes + (uint32_t)(kk & 3) * 32u;
            const uint32_t b_off = (uint32_t)(kk >> 2) * kBBox + (uint32_t)(kk & 3) * 32u;
            dev::mma_bf16(d_acc, dev::smem_desc_advance(a_d, a_off), dev::smem_desc_advance(b_d, b_off), kIdesc,
                          (kt | kk) != 0 ? 1u : 0u);
          }
          // both stages free once these MMAs finish
          dev::mma_commit(bar_a_empty0 + 8u * pa.index);
          if (!one_ring) dev::mma_commit(bar_b_empty0 + 8u * pb.index);
        }
        if (!ok) break;
        dev::mma_commit(bar_acc_full0 + 8u * buf);   // tile j's accumulator complete
      }
      stamp(p, kTrLastFull);
      dev::mma_commit(bar_mma_done);                 // tracks every MMA this thread issued
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- epilogue: thread et owns TMEM lane et = weight row n0 + et of each tile.
    // A tile is reduced in rounds of p.mailbox_quads 4-column groups (one
    // round when the mailbox holds all of a tile's columns): each round the
    // ranks publish those columns, sum and store them, and signal the peers
    // that the mailbox is free for the next round (of this tile or the next).
    // After a failed wait (or once the CTA's failure flag is set) a thread
    // goes quiet: it arms, waits for and addresses no barrier or mailbox any
    // more -- re-arming the reduction barrier while its phase is still open
    // would arrive on a phase with no pending arrivals -- but it still runs
    // the loop to the end, so that all 128 threads meet every named barrier.
    // The output is then undefined.
    bool quiet = false;
    const int et = (int)threadIdx.x - 128;
    const uint32_t t_row = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    const int R = kMmaM / split;
    const int my_lo = rank * R;
    const int dst_rank = et / R;
    const int qr = p.mailbox_quads;                          // 4-column groups per round
    const bool publish = !(p.inject & kInjectSkipPublish);
    float* const mb = reinterpret_cast<float*>(smem_raw + (sMail - raw));
    const uint32_t r_bar = dev::mapa(bar_reduce, (uint32_t)dst_rank);
    const uint32_t r_mail0 = dev::mapa(sMail, (uint32_t)dst_rank);
    int gr = 0;                                              // reduction rounds so far (all tiles)
    for (int j = 0; j < my_tiles; ++j) {
      const int buf = j & 1;
      int n0, m0, l;
      tile_coords(j, &n0, &m0, &l);
      const int ncols = (p.M - m0) < MMA_N ? (p.M - m0) : MMA_N;
      const int nquads = (ncols + 3) >> 2;
      // the bias of the 8 weight rows this thread will store
      float bias8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (p.bias != nullptr) {
        const int nb = n0 + my_lo + (et % (R / 8)) * 8;
        const uint16_t* bp = p.bias + (size_t)l * (size_t)p.N + (size_t)nb;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (nb + e < p.N) bias8[e] = __uint_as_float((uint32_t)__ldg(bp + e) << 16);
        }
      }
      if (dev::ld_shared_u32(slot_abort) != 0u) quiet = true;
      if (!quiet && !waiter.wait<false>(bar_acc_full0 + 8u * buf, (uint32_t)((j >> 1) & 1), kRoleEpiMma, j)) {
        quiet = true;
      }
      __syncwarp();
      dev::tc_fence_after();
      if (j == 0 && et == 0) stamp(p, kTrMmaDone);
      for (int qb = 0; qb < nquads; qb += qr, ++gr) {
        const int c_lo = qb * 4;
        const int c_hi = ncols < (qb + qr) * 4 ? ncols : (qb + qr) * 4;
        const int rc = c_hi - c_lo;
        const bool last_round_of_tile = qb + qr >= nquads;
        if (et == 0 && !quiet) {
          dev::mbar_arrive_expect_tx(bar_reduce, (uint32_t)((split - 1) * rc * R) * 4u);
          reduce_armed = gr & 1;
        }
        // The peers' mailboxes hold the previous round until each peer has read it.
        if (gr > 0 && publish && !quiet &&
            !waiter.wait<true>(bar_ready, (uint32_t)((gr - 1) & 1), kRoleEpiReady, gr)) {
          quiet = true;
        }
        const bool send = publish && !quiet;
        // Rounds of whole column quads: the mailbox is [source][row][column]
        // and each thread sends its row's columns as 16-byte st.async (a
        // quarter of the remote stores).  Otherwise [source][column][row]:
        // thread et's value of column c goes to [rank][c - c_lo][et - dst_rank*R]
        // of the rank that sums row et, a warp's rows of one column contiguous.
        const bool by_row = (rc & 3) == 0;
        const uint32_t slot = by_row ? (uint32_t)((rank * R + (et - dst_rank * R)) * rc) * 4u
                                     : ((uint32_t)(rank * rc) * (uint32_t)R + (uint32_t)(et - dst_rank * R)) * 4u;
#pragma unroll 1
        for (int g = c_lo >> 4; g * 16 < c_hi; ++g) {
          uint32_t v[16];
          __syncwarp();   // tcgen05.ld is warp-collective
          load_acc16(t_row + (uint32_t)buf * kAccCols + (uint32_t)(g * 16), 0u, false, v);
          if (by_row) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int col = g * 16 + 4 * q;
              if (col < c_lo || col >= c_hi) continue;           // warp-uniform
              const uint32_t off = slot + (uint32_t)(col - c_lo) * 4u;
              if (dst_rank == rank) {
                dev::st_shared_v4(sMail + off, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              } else if (send) {
                dev::st_async_v4(r_mail0 + off, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], r_bar);
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int col = g * 16 + e;
              if (col < c_lo || col >= c_hi) continue;           // warp-uniform
              const uint32_t off = slot + (uint32_t)((col - c_lo) * R) * 4u;
              if (dst_rank == rank) {
                *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(mb) + off) = v[e];
              } else if (send) {
                dev::st_async_b32(r_mail0 + off, v[e], r_bar);
              }
            }
          }
        }
        if (last_round_of_tile) {
          // this buffer's TMEM reads are done: the MMAs of tile j + 2 may use it
          dev::tc_fence_before();
          dev::mbar_arrive(bar_acc_empty0 + 8u * buf);
        }
        dev::named_bar_sync(1, kEpiThreads);                // own slot complete
        if (!quiet) {
          if (waiter.wait<true>(bar_reduce, (uint32_t)(gr & 1), kRoleEpiReduce, gr)) {
            if (et == 0) reduce_armed = -1;
          } else {
            quiet = true;
          }
        }
        if (by_row) {
          // 8 weight rows x 4 token columns per item: sum the sources in rank
          // order, then per column pack bf16 pairs and one 16-byte store.
          const int nq = rc >> 2;
          const int items = (R >> 3) * nq;
#pragma unroll 1
          for (int it = et; it < items; it += kEpiThreads) {
            const int rb = it / nq;
            const int c4 = (it - rb * nq) * 4;
            const float* src = mb + (size_t)(rb * 8) * rc + c4;
            float4 x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = *reinterpret_cast<const float4*>(src + (size_t)i * rc);
#pragma unroll 1
            for (int sr = 1; sr < split; ++sr) {
              const float* ps = src + (size_t)sr * R * rc;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 a4 = *reinterpret_cast<const float4*>(ps + (size_t)i * rc);
                x[i].x += a4.x; x[i].y += a4.y; x[i].z += a4.z; x[i].w += a4.w;
              }
            }
            const int n = n0 + my_lo + rb * 8;
            if (n >= p.N) continue;
            float b8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (p.bias != nullptr) {
              const uint16_t* bp = p.bias + (size_t)l * (size_t)p.N + (size_t)n;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                if (n + e < p.N) b8[e] = __uint_as_float((uint32_t)__ldg(bp + e) << 16);
              }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float v8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) v8[i] = (c == 0 ? x[i].x : c == 1 ? x[i].y : c == 2 ? x[i].z : x[i].w) + b8[i];
              const uint32_t q0 = dev::pack_bf16x2(v8[0], v8[1]), q1 = dev::pack_bf16x2(v8[2], v8[3]);
              const uint32_t q2 = dev::pack_bf16x2(v8[4], v8[5]), q3 = dev::pack_bf16x2(v8[6], v8[7]);
              uint16_t* dst =
                  p.c + ((size_t)((size_t)l * p.M + (size_t)(m0 + c_lo + c4 + c)) * (size_t)p.N + (size_t)n);
              if (p.vec_store && n + 8 <= p.N) {
                dev::st_global_v4(dst, q0, q1, q2, q3);
              } else {
                store8_clipped(dst, n, p.N, q0, q1, q2, q3);
              }
            }
          }
        } else {
        // 8 weight rows of one token column per item: sum the sources in rank
        // order, pack bf16 pairs, one 16-byte store.
        const int chunks = R / 8;
        const int items = rc * chunks;
#pragma unroll 1
        for (int it = et; it < items; it += kEpiThreads) {
          const int mc = it / chunks;
          const int c8 = (it - mc * chunks) * 8;
          const float* src = mb + (size_t)mc * R + c8;
          float4 x = *reinterpret_cast<const float4*>(src);
          float4 y = *reinterpret_cast<const float4*>(src + 4);
#pragma unroll 1
          for (int sr = 1; sr < split; ++sr) {
            const float* ps = src + (size_t)sr * rc * R;
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
          uint16_t* dst = p.c + ((size_t)((size_t)l * p.M + (size_t)(m0 + c_lo + mc)) * (size_t)p.N + (size_t)n);
          if (p.vec_store && n + 8 <= p.N) {
            dev::st_global_v4(dst, q0, q1, q2, q3);
          } else {
            store8_clipped(dst, n, p.N, q0, q1, q2, q3);
          }
        }
        }
        // Every thread has read the mailbox: the peers may publish the next round.
        dev::named_bar_sync(1, kEpiThreads);
        const bool more = !(j == my_tiles - 1 && last_round_of_tile);
        if (more && et >= 1 && et < split && !quiet) {
          dev::mbar_arrive_remote(dev::mapa(bar_ready, (uint32_t)((rank + et) % split)));
        }
      }
      if (j == my_tiles - 1 && et == 0) stamp(p, kTrStored);
    }
  }

  // ---- teardown
  if (dev::ld_shared_u32(slot_abort) != 0u) {
    // A wait failed somewhere in this CTA: let the copies this CTA issued
    // land (bounded) before it leaves.  For each ring stage the last round
    // issued is the one to wait for.
    const unsigned long long drain_ns = 10000000ull;   // 10 ms
    const int issued = warp == 0 ? a_issued : warp == 1 ? b_issued : 0;
    const int ring = warp == 0 ? a_stages : b_stages;
    const uint32_t full0 = warp == 0 ? bar_a_full0 : bar_b_full0;
    if ((warp == 0 || warp == 1) && lane == 0) {
      for (int s = 0; s < issued && s < ring; ++s) {
        const int round = (issued - 1 - s) / ring;
        drain_wait(full0 + 8u * s, (uint32_t)(round & 1), drain_ns);
      }
    }
    // the peers' partials of a reduction this CTA stopped waiting for
    if (threadIdx.x == 128 && reduce_armed >= 0) drain_wait(bar_reduce, (uint32_t)reduce_armed, drain_ns);
  }
  if (warp == 2) {
    // every MMA issued has completed before tensor memory is released
    if (lane == 0) {
      if (!waiter.wait<false>(bar_mma_done, 0u, kRoleTmemRelease, 0, 4)) {
        drain_wait(bar_mma_done, 0u, 10000000ull);
      }
    }
    __syncwarp();
  }
  // No CTA leaves while a peer may still address its shared memory.  The
  // arrival is relaxed (a release would wait for the tile's global stores);
  // every peer's bytes addressed to this CTA were received through its
  // reduction waits.  A CTA whose wait failed fences its remote operations
  // first instead.
  if (dev::ld_shared_u32(slot_abort) != 0u) dev::fence_acq_rel_cluster();
  __syncwarp();
  dev::cluster_arrive_relaxed();
  dev::cluster_wait_acquire();
  if (warp == 2) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem_base, p.tmem_cols);
  }
  if (threadIdx.x == 0) stamp(p, kTrEnd);
}

// ---------------------------------------------------------------- host side
namespace {

template <int MMA_N>
cudaError_t launch_p(const LaunchArgs& la, const CUtensorMap& b_map, const KernelParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = la.grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
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
  if (p.b_stages == p.stages) return cudaLaunchKernelEx(&cfg, splitk_persistent_kernel<MMA_N, true>, b_map, p);
  return cudaLaunchKernelEx(&cfg, splitk_persistent_kernel<MMA_N, false>, b_map, p);
}

template <int MMA_N>
cudaError_t max_clusters_p(unsigned cluster_x, size_t smem, int* out) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_x, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cluster_x;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, splitk_persistent_kernel<MMA_N, true>, &cfg);
}

}  // namespace

cudaError_t launch_persistent(const LaunchArgs& la, const CUtensorMap& b_map, const KernelParams& p,
                              cudaStream_t stream) {
  switch (la.mma_n) {
    case 16: return launch_p<16>(la, b_map, p, stream);
    case 32: return launch_p<32>(la, b_map, p, stream);
    case 64: return launch_p<64>(la, b_map, p, stream);
    case 128: return launch_p<128>(la, b_map, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t max_active_clusters_persistent(int mma_n, unsigned cluster_x, size_t smem, int* out) {
  switch (mma_n) {
    case 16: return max_clusters_p<16>(cluster_x, smem, out);
    case 32: return max_clusters_p<32>(cluster_x, smem, out);
    case 64: return max_clusters_p<64>(cluster_x, smem, out);
    case 128: return max_clusters_p<128>(cluster_x, smem, out);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_persistent(int max_dynamic_smem) {
  const void* fns[] = {
      (const void*)splitk_persistent_kernel<16, true>,  (const void*)splitk_persistent_kernel<16, false>,
      (const void*)splitk_persistent_kernel<32, true>,  (const void*)splitk_persistent_kernel<32, false>,
      (const void*)splitk_persistent_kernel<64, true>,  (const void*)splitk_persistent_kernel<64, false>,
      (const void*)splitk_persistent_kernel<128, true>, (const void*)splitk_persistent_kernel<128, false>};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t read_and_clear_fault_persistent(int* out_words) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out_words, g_fault, sizeof(int) * kFaultWords);
  if (e != cudaSuccess) return e;
  int zeros[kFaultWords] = {0};
  return cudaMemcpyToSymbol(g_fault, zeros, sizeof(zeros));
}

}  // namespace splitk
