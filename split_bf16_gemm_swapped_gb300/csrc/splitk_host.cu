// Host side of the C ABI (include/splitk.h): tactic planning, tensor-map
// caches, argument checks and launch.
//
// The page's launcher (SplitKGemm.__call__ on the vLLM "splitk" API page)
// launches grid (ceil(Mk/mma_m), ceil(Nk/mma_n) * split_k, L) with a
// (1, split_k, 1) cluster, 256 threads, the whole shared memory of the SM and
// PDL, and takes A's tensor map as a device address.  Here the cluster runs
// along grid x (grid = (split_k * m_tiles, n_tiles, L)) so the CTAs that
// share a weight tile are launched next to each other, shared memory is sized
// from the occupancy the grid needs instead of taking the whole SM, and the
// device tensor maps of A live in a pool owned by this library.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "splitk.h"
#include "splitk_internal.h"

namespace splitk {

// Scratch of splitk_gemm_bf16_noalloc: room for the one CUDA tensor map of A
// that a launch reads besides its operands.  A file-scope device array, so
// every GPU that loads this library holds these bytes until the process
// exits and the entry point never allocates.  In host code the name stands
// for the device symbol; its device address comes from cudaGetSymbolAddress.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMapPoolSlots = 4096;     // 512 KiB of device tensor maps
constexpr size_t kBMapCacheMax = 1024;

std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<unsigned> g_inject{0};
std::atomic<unsigned long long*> g_trace{nullptr};
std::atomic<unsigned> g_trace_ctas{0};


bool valid_split(int s) { return s == 1 || s == 2 || s == 4 || s == 8; }

int choose_mma_n(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

// Activation tiles the B region holds: the ring's stages, or every K tile
// of the CTA (at least as many as stages, so rank 0's f32 staging tile of
// min(M, mma_n) x 128 always fits once the region is drained).
int b_region_tiles_for(int stages, int b_resident, int k_tiles) {
  return b_resident ? std::max(stages, k_tiles) : stages;
}

size_t smem_bytes_for(int mma_n, int stages, uint32_t dedicated_mailbox_bytes, int b_region_tiles) {
  return (size_t)kAlignSlack + (size_t)stages * kAStageBytes +
         (size_t)b_region_tiles * b_stage_bytes(mma_n) + dedicated_mailbox_bytes + kBarRegionBytes;
}

// Bytes of one reduction round: (split - 1) peers x the round's token
// columns (at most 4 per quad, at most the tile's real columns) x 128 rows.
uint32_t mailbox_round_bytes(int split, int quads, int ncols_max) {
  const int cols = std::min(quads * 4, ncols_max);
  return (uint32_t)(split - 1) * (uint32_t)cols * kColumnBytes;
}

// Bytes of one packed K tile of quantized weights (E2M1: 8 KiB, E4M3: 16 KiB).
inline uint32_t q_tile_bytes(int fmt) { return fmt == SPLITK_WEIGHTS_E4M3_E8M0 ? kW8TileBytes : kW4TileBytes; }
inline bool is_quantized(int fmt) { return fmt == SPLITK_WEIGHTS_E2M1_E8M0 || fmt == SPLITK_WEIGHTS_E4M3_E8M0; }

// Shared memory of a quantized-weight plan's layout: all packed weight
// tiles, all activation tiles (at least 2: rank 0's f32 staging tile reuses
// them), the mailbox and the barriers.
// code_stages: the ring of packed weight tiles (at most k_tiles)
size_t smem_bytes_w4(int mma_n, int k_tiles, int code_stages, uint32_t dedicated_mailbox_bytes, int smem_tiles,
                     int fmt) {
  return (size_t)kAlignSlack + (size_t)code_stages * q_tile_bytes(fmt) +
         (size_t)std::max(2, k_tiles) * b_stage_bytes(mma_n) + (size_t)smem_tiles * kAStageBytes +
         dedicated_mailbox_bytes + kBarRegionBytes;
}

// Mailbox bytes of a dedicated single-round reduction (rank 0 or scattered).
uint32_t w4_mailbox_bytes(int split, int reduce_scatter, int ncols_max) {
  if (split == 1) return 0u;
  if (reduce_scatter) return (uint32_t)ncols_max * kColumnBytes;
  return mailbox_round_bytes(split, (ncols_max + 3) / 4, ncols_max);
}

// CTAs of this kernel that shared memory lets onto one SM (each CTA also
// reserves 1 KiB of the SM's shared memory).
int resident_by_smem(size_t smem_per_sm, size_t smem) { return (int)(smem_per_sm / (smem + 1024)); }

// Token columns one reduction round of a persistent plan moves: all of a
// tile's, or `quads` 4-column groups.
int persistent_round_cols(int ncols_max, int quads) { return std::min(ncols_max, 4 * quads); }

// Shared memory of a persistent plan: the weight ring (`stages` K tiles), the
// activation ring (`b_stages` K tiles, or `stages` when 0), the scattered
// mailbox of one reduction round's token columns and the barriers (a second
// set of full/empty barriers when the two rings' depths differ).
size_t smem_bytes_persistent(int mma_n, int stages, int b_stages, int round_cols) {
  return (size_t)kAlignSlack + (size_t)stages * kAStageBytes +
         (size_t)(b_stages != 0 ? b_stages : stages) * b_stage_bytes(mma_n) + (size_t)round_cols * kColumnBytes +
         (b_stages != 0 && b_stages != stages ? kBarRegionBytesPersistent : kBarRegionBytes);
}

// 128-wide K tiles covering K; the last one may be ragged (TMA reads zeros
// past K).
inline int total_k_tiles(int K) { return (int)(((long long)K + kCtaK - 1) / kCtaK); }

// The largest K: the kernel's K coordinates (TMA takes signed 32-bit ones)
// reach the end of the last 128-wide tile.
constexpr int kMaxK = 0x7FFFFFFF - kCtaK + 1;

// Tiles of `tile` rows covering `rows` (64-bit: rows may be near INT_MAX).
inline long long tiles_of(int rows, int tile) { return ((long long)rows + tile - 1) / tile; }

// Split-K choice from GB300 measurements (decode shapes and the long-K
// sweep, back to back): rank 0's reduction costs more as the split and the
// tile's token columns grow, so take the smallest split whose grid fills
// about 3/4 of the SMs (1/2 for tiles of 64 or more tokens), with at least
// one K tile per rank.
int auto_split(int T, long long tiles, int num_sms, int mma_n) {
  const double fill = (mma_n >= 64 ? 0.5 : 0.75) * (double)num_sms;
  int best = 1;
  for (int s : {1, 2, 4, 8}) {
    if (s > T) break;
    best = s;
    if ((double)(tiles * s) >= fill) return s;
  }
  return best;
}

// The staged decode tactic, for grids of narrow tiles (mma_n <= 32) that are
// resident at 2 CTAs per SM with few K tiles per CTA: the activations of all
// of a CTA's K tiles in their own buffer, loaded at once after the
// programmatic-dependent-launch wait; a 2-stage weight ring whose first
// min(3, k_tiles - 2) tiles (both of 2) are copied into tensor memory as they
// land, so that up to 5 weight K tiles are on chip before the wait returns,
// the rest prefetched into L2; two MMA
// issuers (a thread issues one tcgen05.mma about every 46 cycles at these
// widths); and the early trigger.  Measured on GB300 (back to back, weights
// rotated past L2): single-token decode 7.1 -> 5.8 us, small-batch decode
// 12.0 -> 11.8 us.  `ded` is the mailbox region the ring plan chose.
bool stage_for_decode(splitk_plan_t* out, int ncols_max, long long ctas, int num_sms, size_t smem_per_sm,
                      size_t smem_optin, uint32_t ded) {
  const int kt = out->k_tiles_per_cta;
  if (out->mma_n > 32 || kt < 2 || ctas > 2LL * num_sms) return false;
  // an aliased mailbox round must fit the 2-stage ring
  if (!out->reduce_scatter && out->split_k > 1 && !out->mailbox_dedicated &&
      mailbox_round_bytes(out->split_k, out->mailbox_quads, ncols_max) > 2u * kAStageBytes) {
    return false;
  }
  // All of them when the ring holds them anyway (2 tiles: measured faster),
  // else as many as leave the 2 ring stages to the tiles after them.
  const int tiles = kt <= 2 ? kt : std::min(kMaxTmemTiles, kt - 2);
  const uint32_t cols = tmem_cols_for(out->mma_n, tiles, 2);
  const size_t smem = smem_bytes_for(out->mma_n, 2, ded, b_region_tiles_for(2, 1, kt));
  const size_t budget = std::min(smem_optin, smem_per_sm / 2 - 1024);
  if (smem > budget || (size_t)resident_by_smem(smem_per_sm, smem) * cols > 512u) return false;
  out->stages = 2;
  out->b_resident = 1;
  out->a_tmem_tiles = tiles;
  out->mma_issuers = 2;
  out->tmem_cols = cols;
  out->pdl_trigger = 1;
  out->smem_bytes = smem;
  out->ctas_per_sm = 2;
  // Few activation rows: the idle epilogue threads load them (at most 4
  // 16-byte loads each) sooner than a TMA queued behind weight loads
  // (single-token decode 5.8 -> 5.5 us; 16 rows x 7 tiles is slower).
  out->b_loader = ncols_max * kt * (kCtaK / 8) <= 4 * kEpiThreads ? 1 : 0;
  // Tiles that stay off chip until the wait go to L2 at CTA start
  // (small-batch decode: 11.6 -> 11.1 us).
  out->l2_prefetch = kt > 2 + tiles ? 1 : 0;
  return true;
}

// The persistent plan for a shape and a split of 2 or more: one CTA per SM
// with the deepest ring (2 to 8 stages) that fits beside the scattered
// mailbox, the mailbox holding a whole tile's columns or, when a smaller one
// leaves room for a deeper ring, reduction rounds of 16, 8 or 4 4-column
// groups; two accumulators in TMEM; one cluster per `split` SMs (at most one
// per output tile).  Nonzero `stages` / `quads` fix the ring depth / round;
// nonzero `b_stages` gives the activations a ring of their own that deep
// (`stages` then counts weight tiles alone).
bool persistent_plan(int M, int N, int K, int L, int split, int stages, int b_stages, int quads, int num_sms,
                     size_t smem_per_sm, size_t smem_optin, splitk_plan_t* out, int mma_n_want = 0) {
  if (split < 2 || !valid_split(split)) return false;
  const int T = total_k_tiles(K);
  if (T < split) return false;
  const int mma_n = mma_n_want != 0 ? mma_n_want : choose_mma_n(M);
  if (mma_n != 16 && mma_n != 32 && mma_n != 64 && mma_n != 128) return false;
  const int ncols_max = std::min(M, mma_n);
  const int nquads_max = (ncols_max + 3) / 4;
  if (b_stages != 0 && (b_stages < 2 || b_stages > kMaxStages)) return false;
  const size_t budget = std::min(smem_optin, smem_per_sm - 1024);
  auto deepest = [&](int qr) {
    int st = kMaxStages;
    while (st > 2 && smem_bytes_persistent(mma_n, st, b_stages, persistent_round_cols(ncols_max, qr)) > budget) --st;
    return st;
  };
  int qr = quads;
  if (qr == 0) {
    // one round a tile unless fewer columns a round buy a deeper ring
    qr = nquads_max;
    for (int q : {16, 8, 4}) {
      if (q < nquads_max && (stages == 0 ? deepest(q) > deepest(qr) : false)) qr = q;
    }
  }
  if (qr < 1 || qr > mma_n / 4 || (qr % 4 != 0 && qr < nquads_max)) return false;
  qr = std::min(qr, nquads_max);
  const int round_cols = persistent_round_cols(ncols_max, qr);
  const int st = stages != 0 ? stages : deepest(qr);
  if (st < 2 || st > kMaxStages || smem_bytes_persistent(mma_n, st, b_stages, round_cols) > budget) return false;
  const long long tiles = tiles_of(M, mma_n) * tiles_of(N, kMmaM) * L;
  const long long clusters = std::max<long long>(1, std::min<long long>(tiles, num_sms / split));
  std::memset(out, 0, sizeof(*out));
  out->mma_m = kMmaM;
  out->mma_n = mma_n;
  out->stages = st;
  out->split_k = split;
  out->k_tiles_per_cta = (T + split - 1) / split;
  out->mailbox_dedicated = 1;
  out->mailbox_quads = qr;
  out->reduce_rounds = (nquads_max + qr - 1) / qr;
  out->grid[0] = (unsigned)split;
  out->grid[1] = (unsigned)std::min<long long>(clusters, 65535);
  out->grid[2] = 1;
  out->cluster[0] = (unsigned)split;
  out->cluster[1] = 1;
  out->cluster[2] = 1;
  out->b_stages = b_stages;
  out->smem_bytes = smem_bytes_persistent(mma_n, st, b_stages, round_cols);
  out->ctas_per_sm = 1;
  out->reduce_scatter = 1;
  out->mma_issuers = 1;
  out->tmem_cols = pow2_at_least(2u * tmem_acc_cols(mma_n));
  out->weight_format = SPLITK_WEIGHTS_BF16;
  out->persistent = 1;
  return true;
}

int plan_ring_impl(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                   size_t smem_optin, splitk_plan_t* out);

// The plan: the per-tile kernel's (plan_ring_impl), or the persistent kernel,
// whose reduction overlaps the next tile's stream, where that measured
// faster on GB300 (the K = 16384 sweep, back to back, the same box): split 8
// at every tile width (M = 1..16: 0.82-0.95 -> 0.97-0.99 of the HBM copy
// bandwidth; M = 64: 0.55 -> 0.87), and split 4 for tiles of 32 to 128
// tokens (M = 64: 0.80 -> 0.82; the wide projection 0.68 -> 0.88), when the
// grid exceeds one CTA per SM and the output tiles deal out evenly (at least
// 90 %) over one cluster per `split` SMs; at split 8 with a reduction in
// rounds, the activations on a ring of their own so that one round does.
int plan_impl(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
              size_t smem_optin, splitk_plan_t* out) {
  const int rc = plan_ring_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_optin, out);
  if (rc != SPLITK_OK) return rc;
  const int split = out->split_k;
  // Split 2 with at least 64 tokens: 64-token tiles where they deal out
  // evenly (M = 128 sweep point, twice the tiles: 0.73 -> 0.77 of the HBM
  // copy bandwidth; the wide projection, 144 tiles: 46.1 -> 45.5 us).
  const bool two_wide = split == 2 && M >= 64;
  const int pers_n = two_wide ? 64 : 0;
  const long long tiles = tiles_of(M, pers_n != 0 ? pers_n : out->mma_n) * tiles_of(N, kMmaM) * L;
  const long long clusters = std::max(1, num_sms / split);
  const long long rounds = (tiles + clusters - 1) / clusters;
  const bool balanced = (double)tiles >= 0.9 * (double)(rounds * clusters);
  // Split 2 at 32- and 64-token tiles: the persistent kernel measured faster
  // even with uneven rounds (112 tiles over 76 clusters: M = 32 sweep point
  // 77.4 -> 75.1 us, M = 64 79.1 -> 77.0 us).  Split 4 from 32-token tiles
  // when the tiles deal out evenly (M = 32: 76.8 -> 76.0 us).
  const bool two_uneven = split == 2 && (out->mma_n == 32 || out->mma_n == 64);
  if ((((split == 8 || (split == 4 && out->mma_n >= 32) || two_wide) && balanced) || two_uneven) &&
      tiles * split > num_sms) {
    splitk_plan_t p;
    if (persistent_plan(M, N, K, L, split, 0, 0, 0, num_sms, smem_per_sm, smem_optin, &p, pers_n)) {
      // At split 8 a tile reduced in two rounds waits twice on all seven
      // peers; an activation ring of 2 stages of its own leaves room for a
      // mailbox of the whole tile at the same weight ring depth (M = 128
      // sweep point: 109.6 -> 96.9 us; at split 4 the shallower activation
      // ring costs more than the second round: 93.0 -> 97.4 us).
      splitk_plan_t one;
      const int nquads_max = (std::min(M, p.mma_n) + 3) / 4;
      if (split == 8 && p.reduce_rounds > 1 &&
          persistent_plan(M, N, K, L, split, p.stages, 2, nquads_max, num_sms, smem_per_sm, smem_optin, &one,
                          p.mma_n)) {
        p = one;
      }
      *out = p;
    }
  }
  return SPLITK_OK;
}

int plan_ring_impl(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                   size_t smem_optin, splitk_plan_t* out) {
  if (!out) return SPLITK_ERR_NULL;
  std::memset(out, 0, sizeof(*out));   // fields a bf16 plan does not use stay 0
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  if (split_k != 0 && !valid_split(split_k)) return SPLITK_ERR_UNSUPPORTED_SPLIT;
  if (num_sms < 1 || smem_optin < 1 || smem_per_sm < 1) return SPLITK_ERR_UNSUPPORTED_DEVICE;
  // K's row stride must be a multiple of 16 bytes (TMA).
  if (K % 8 != 0 || K > kMaxK) return SPLITK_ERR_INVALID_SHAPE;
  const int T = total_k_tiles(K);
  const int mma_n = choose_mma_n(M);
  const long long m_tiles = tiles_of(M, mma_n);
  const long long n_tiles = ((long long)N + kMmaM - 1) / kMmaM;
  if (n_tiles > 65535 || L > 65535) return SPLITK_ERR_INVALID_SHAPE;
  int split = split_k;
  if (split == 0) split = auto_split(T, m_tiles * n_tiles * L, num_sms, mma_n);
  if (split > T) return SPLITK_ERR_INVALID_SHAPE;      // every rank owns a K tile
  if (m_tiles * split > 0x7FFFFFFFLL) return SPLITK_ERR_INVALID_SHAPE;
  const int k_tiles = (T + split - 1) / split;          // the most any rank owns

  // Shared memory is sized so the whole grid is resident at once (up to 2
  // CTAs per SM), with as deep a ring as that leaves.  Measured on GB300 for
  // the decode shapes: 3 stages at 2 CTAs/SM beat 2 stages at 3 CTAs/SM
  // (where the next kernel's grid could be co-resident), because a stage
  // that is already in flight when the previous kernel completes shortens
  // the critical path more than early residency does.
  const long long ctas = (long long)split * m_tiles * n_tiles * L;
  int per_sm = (int)std::min<long long>(2, std::max<long long>(1, (ctas + num_sms - 1) / num_sms));
  const int ncols_max = std::min(M, mma_n);
  const int nquads_max = (ncols_max + 3) / 4;
  const uint32_t ded_bytes =
      split > 1 ? mailbox_round_bytes(split, nquads_max, ncols_max) : 0u;
  const bool prefer_dedicated = split > 1 && ded_bytes <= 16u * 1024u;

  // Scattered reduction (each rank sums 128/split rows) moves 1/split of the
  // DSMEM bytes into each SM; measured on GB300 it wins from split 4 and 16
  // token columns up whenever its own mailbox (min(M, mma_n) * 512 B) fits at
  // the same residency (M=16 decode, split 8: 12.9 us vs 14.2 us).
  const bool try_scatter = split >= 4 && ncols_max >= 16;
  const uint32_t scatter_bytes = (uint32_t)ncols_max * kColumnBytes;

  // A ring plan: `stages` deep, mailbox `mode` (2 scattered, 1 dedicated,
  // 0 aliased on rank 0's drained ring, or none without a split).
  auto fill = [&](int stages, int mode, int per_sm_v, int issuers) {
    // Aliased: one round when the partials fit the drained ring, else rounds
    // of whole 16-column groups (4 quads; at least one group always fits a
    // 2-stage ring).
    int quads = nquads_max;
    if (split > 1 && mode == 0 && mailbox_round_bytes(split, quads, ncols_max) > (uint32_t)stages * kAStageBytes) {
      quads = 4;
      while (mailbox_round_bytes(split, quads + 4, ncols_max) <= (uint32_t)stages * kAStageBytes) quads += 4;
    }
    const uint32_t ded = mode == 2 ? scatter_bytes : mode == 1 ? ded_bytes : 0u;
    out->mma_m = kMmaM;
    out->mma_n = mma_n;
    out->stages = stages;
    out->split_k = split;
    out->k_tiles_per_cta = k_tiles;
    out->mailbox_dedicated = split > 1 && mode != 0 ? 1 : 0;
    out->mailbox_quads = quads;
    out->reduce_rounds = split > 1 ? (nquads_max + quads - 1) / quads : 0;
    out->grid[0] = (unsigned)(split * m_tiles);
    out->grid[1] = (unsigned)n_tiles;
    out->grid[2] = (unsigned)L;
    out->cluster[0] = (unsigned)split;
    out->cluster[1] = 1;
    out->cluster[2] = 1;
    out->smem_bytes = smem_bytes_for(mma_n, stages, ded, stages);
    out->ctas_per_sm = per_sm_v;
    // The early trigger when the grid leaves SMs free: the next launch's CTAs
    // start their weight streams there while this one finishes (K = 16384
    // sweep, split 1, 112 CTAs: M = 1..16 0.940-0.949 -> 0.952-0.960 of the
    // HBM copy bandwidth, unchanged from 32 tokens).  With every SM busy it
    // measured slower (split 4, M = 16: 75.1 -> 76.2 us).
    out->pdl_trigger = ctas < num_sms ? 1 : 0;
    out->reduce_scatter = mode == 2 ? 1 : 0;
    out->b_resident = 0;
    out->a_tmem_tiles = 0;
    out->mma_issuers = issuers;
    out->tmem_cols = tmem_cols_for(mma_n, 0, issuers);
    out->b_loader = 0;
    out->l2_prefetch = 0;
    out->weight_format = SPLITK_WEIGHTS_BF16;
    return ded;
  };
  const int split_mode = split == 1 ? 0 : try_scatter ? 2 : prefer_dedicated ? 1 : 0;

  // Short K slices of narrow tiles: the staged decode tactic
  // (stage_for_decode), with the mailbox measured best for it: scattered from
  // 16 token columns and split 4, else a dedicated one when small.
  {
    const uint32_t ded = fill(2, split_mode, 2, 1);
    if (stage_for_decode(out, ncols_max, ctas, num_sms, smem_per_sm, smem_optin, ded)) return SPLITK_OK;
  }

  for (; per_sm >= 1; --per_sm) {
    const size_t budget = std::min(smem_optin, smem_per_sm / (size_t)per_sm - 1024);
    // A CTA alone on its SM (a grid of at most one CTA per SM) keeps as many
    // weight tiles in flight as its shared memory holds, with two MMA issuers
    // on an even ring where one issuer's tcgen05.mma stream is issue-bound
    // (mma_n <= 64).  Measured on GB300, the split-1 sweep (112 CTAs, K 16384):
    // M=1 0.86 -> 0.95 of the HBM copy bandwidth with 6 stages, M=16
    // 0.85 -> 0.92, M=64 0.85 -> 0.88 (4 stages, all that fit).
    const bool deep = per_sm == 1 && ctas <= num_sms;
    const bool deep_two = deep && mma_n <= 64;
    const int stages_cap = std::min(kMaxStages, std::max(2, deep ? k_tiles : std::min(k_tiles, 4)));
    // Mailbox modes in order of preference (measured on the decode shapes):
    // scattered, dedicated, aliased.  On short K slices the first mode that
    // fits at any depth wins; on long ones (16 K tiles a CTA and more) the
    // deepest ring does, with the first mode that fits at that depth: a stage
    // more in flight outweighs the mailbox placement there (K = 16384 sweep
    // at 2 CTAs/SM: M=8, split 2 0.93 -> 0.99, M=16, split 4 0.91 -> 0.93 and
    // M=2, split 8 0.87 -> 0.92 of the HBM copy bandwidth with 3 aliased
    // stages instead of 2 with their own mailbox).
    int modes[3];
    int n_modes = 0;
    if (split_mode == 2) modes[n_modes++] = 2;
    if (split > 1 && prefer_dedicated) modes[n_modes++] = 1;
    // A few token columns (2-15): the scattered mailbox before the aliased
    // one when the dedicated one does not fit (K = 16384 sweep at 3 stages,
    // split 8: M=2 0.90 -> 0.92, M=4 0.89 -> 0.91; a single column keeps the
    // dedicated mailbox, measured best).
    if (split_mode != 2 && split >= 4 && ncols_max >= 2) modes[n_modes++] = 2;
    modes[n_modes++] = 0;
    auto fits = [&](int mode, int stages) {
      if (deep_two && stages % 2 != 0) return false;
      const uint32_t ded = mode == 2 ? scatter_bytes : mode == 1 ? ded_bytes : 0u;
      return smem_bytes_for(mma_n, stages, ded, stages) <= budget;
    };
    auto choose = [&](bool depth_first) {
      for (int i = 0; i < (depth_first ? stages_cap - 1 : n_modes); ++i) {
        for (int j = 0; j < (depth_first ? n_modes : stages_cap - 1); ++j) {
          const int stages = stages_cap - (depth_first ? i : j);
          const int mode = modes[depth_first ? j : i];
          if (!fits(mode, stages)) continue;
          // ... but not into an aliased mailbox that needs more than one
          // reduction round (M=128, split 4: 0.55 -> 0.52 that way)
          if (depth_first && mode == 0 && split > 1 && mode != modes[0] &&
              mailbox_round_bytes(split, nquads_max, ncols_max) > (uint32_t)stages * kAStageBytes) {
            continue;
          }
          fill(stages, mode, per_sm, deep_two ? 2 : 1);
          return true;
        }
      }
      return false;
    };
    if ((k_tiles >= 16 && choose(true)) || choose(false)) return SPLITK_OK;
  }
  return SPLITK_ERR_NO_FIT;
}

// The quantized-weight plan (A16W4, or A16W8 with fmt = E4M3): decode-sized
// tiles (mma_n 16 or 32), the split of the bf16 planner (raised until a
// CTA's K slice is at most 8 tiles; their packed codes go through a ring of
// code stages, all at once where two CTAs still share an SM), min(3,
// k_tiles) TMEM slots for decoded
// tiles (measured: more slots, decoded before the PDL wait, beat more CTAs
// per SM), resident activations loaded by TMA, the early trigger, and a
// dedicated single-round mailbox (scattered from split 4 and 16 token
// columns).  Shared memory is padded when needed so that the
// CTAs fitting an SM can hold their TMEM.
int plan_w4_impl(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm, size_t smem_optin,
                 splitk_plan_t* out, int fmt = SPLITK_WEIGHTS_E2M1_E8M0) {
  if (!out) return SPLITK_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || L < 1 || M > 32 || K % kCtaK != 0 || K > kMaxK) return SPLITK_ERR_INVALID_SHAPE;
  if (split_k != 0 && !valid_split(split_k)) return SPLITK_ERR_UNSUPPORTED_SPLIT;
  if (num_sms < 1 || smem_optin < 1 || smem_per_sm < 1) return SPLITK_ERR_UNSUPPORTED_DEVICE;
  const int T = K / kCtaK;
  const int mma_n = choose_mma_n(M);
  const long long m_tiles = tiles_of(M, mma_n);
  const long long n_tiles = ((long long)N + kMmaM - 1) / kMmaM;
  if (n_tiles > 65535 || L > 65535) return SPLITK_ERR_INVALID_SHAPE;
  int split = split_k != 0 ? split_k : auto_split(T, m_tiles * n_tiles * L, num_sms, mma_n);
  while (split_k == 0 && split < 8 && (T + split - 1) / split > kMaxStages && split * 2 <= T) split *= 2;
  if (split > T) return SPLITK_ERR_INVALID_SHAPE;
  const int kt = (T + split - 1) / split;
  if (kt > kMaxStages) return SPLITK_ERR_NO_FIT;
  const int ncols_max = std::min(M, mma_n);
  splitk_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.mma_m = kMmaM;
  p.mma_n = mma_n;
  p.stages = kt;
  p.split_k = split;
  p.k_tiles_per_cta = kt;
  p.mailbox_dedicated = split > 1 ? 1 : 0;
  p.mailbox_quads = (ncols_max + 3) / 4;
  p.reduce_rounds = split > 1 ? 1 : 0;
  p.grid[0] = (unsigned)(split * m_tiles);
  p.grid[1] = (unsigned)n_tiles;
  p.grid[2] = (unsigned)L;
  p.cluster[0] = (unsigned)split;
  p.cluster[1] = 1;
  p.cluster[2] = 1;
  p.pdl_trigger = 1;
  p.reduce_scatter = split >= 4 && ncols_max >= 16 ? 1 : 0;
  p.b_resident = 1;
  p.a_tmem_tiles = std::min(kMaxTmemTiles, kt);
  // two MMA issuers (even and odd K tiles into two accumulators) where
  // there are two slots: a lone issuer's tcgen05.mma stream is issue-bound
  p.mma_issuers = p.a_tmem_tiles >= 2 ? 2 : 1;
  p.tmem_cols = tmem_cols_for(mma_n, p.a_tmem_tiles, p.mma_issuers);
  p.b_loader = 0;             // the epilogue threads are busy decoding (measured: TMA is faster here)
  p.l2_prefetch = 0;
  p.weight_format = fmt;
  const uint32_t ded = w4_mailbox_bytes(split, p.reduce_scatter, ncols_max);
  // One tile past the TMEM slots: decode it into a bf16 stage in shared
  // memory, before the PDL wait, if that still fits 2 CTAs per SM
  // (the single-token decode case: 4 K tiles per CTA, 3 slots).
  // The ring of packed tiles: all of the CTA's at once, unless fewer let two
  // CTAs share an SM (8-bit codes: 16 KiB a tile; small-batch decode, 7
  // tiles a CTA, would otherwise run one CTA per SM, its 32 clusters of 8
  // in three waves).
  int code_stages = kt;
  while (code_stages > 2 && smem_bytes_w4(mma_n, kt, code_stages, ded, 0, fmt) + 1024 > smem_per_sm / 2) {
    --code_stages;
  }
  p.stages = code_stages;
  p.w4_smem_tiles = kt == p.a_tmem_tiles + 1 &&
                            smem_bytes_w4(mma_n, kt, code_stages, ded, 1, fmt) + 1024 <= smem_per_sm / 2
                        ? 1
                        : 0;
  // One decoding warpgroup.  The decode (about four instructions a weight
  // pair) is bound by the SM's instruction issue, which a second warpgroup
  // (384 threads a CTA, at most 2 CTAs an SM by registers) barely raises
  // while it takes registers the next kernel's CTAs could use.  Measured on
  // GB300: small-batch decode (7 tiles a CTA) 11.47 us with two groups,
  // 11.29 with one; M=16, L=4 45.2 -> 44.1 us; single-token decode 7.14 ->
  // 6.27 us.  Plans may still ask for two (w4_decoders = 2).
  p.w4_decoders = 1;
  // Shared memory padded when needed so that the CTAs fitting an SM can
  // hold their TMEM.
  auto padded_smem = [&](size_t smem, uint32_t tmem_cols) {
    const int per_sm_max = std::max(1, (int)(512u / tmem_cols));
    if (resident_by_smem(smem_per_sm, smem) > per_sm_max) {
      smem = std::max(smem, (smem_per_sm / (size_t)(per_sm_max + 1) + 16u) & ~(size_t)15u);
      while (resident_by_smem(smem_per_sm, smem) > per_sm_max) smem += 16;
    }
    return smem;
  };
  size_t smem = padded_smem(smem_bytes_w4(mma_n, kt, code_stages, ded, p.w4_smem_tiles, fmt), p.tmem_cols);
  // Grids of more than two waves: one TMEM slot and one issuer when that lets
  // more CTAs share an SM (at most 3 by registers), so that their decodes
  // overlap (single-token decode, L=8: 49.1 -> 46.2 us).
  const long long ctas = (long long)split * m_tiles * n_tiles * L;
  if (ctas > 2LL * num_sms && p.a_tmem_tiles > 1) {
    const uint32_t cols1 = tmem_cols_for(mma_n, 1, 1);
    const size_t smem1 = padded_smem(smem_bytes_w4(mma_n, kt, code_stages, ded, 0, fmt), cols1);
    if (std::min(3, resident_by_smem(smem_per_sm, smem1)) > std::min(2, resident_by_smem(smem_per_sm, smem))) {
      p.a_tmem_tiles = 1;
      p.mma_issuers = 1;
      p.tmem_cols = cols1;
      p.w4_smem_tiles = 0;
      p.w4_decoders = 1;        // 256 threads: a third CTA fits an SM's registers
      smem = smem1;
    }
  }
  if (smem > smem_optin) return SPLITK_ERR_NO_FIT;
  p.smem_bytes = smem;
  p.ctas_per_sm = std::min(p.w4_decoders == 2 ? 2 : 3, resident_by_smem(smem_per_sm, smem));
  *out = p;
  return SPLITK_OK;
}

// Re-derives everything a plan implies and checks it against the shape.
int check_plan_w4(const splitk_plan_t& pl, int M, int N, int K, int L, size_t smem_optin, size_t smem_per_sm,
                  uint32_t* dedicated_bytes) {
  if (pl.mma_m != kMmaM || (pl.mma_n != 16 && pl.mma_n != 32)) return SPLITK_ERR_BAD_PLAN;
  if (!valid_split(pl.split_k)) return SPLITK_ERR_UNSUPPORTED_SPLIT;
  if (M > 32 || K % kCtaK != 0 || K > kMaxK || K / kCtaK < pl.split_k) return SPLITK_ERR_INVALID_SHAPE;
  const int T = K / kCtaK;
  const int kt = (T + pl.split_k - 1) / pl.split_k;
  if (pl.k_tiles_per_cta != kt || pl.stages < 1 || pl.stages > kt) return SPLITK_ERR_BAD_PLAN;
  if (kt > kMaxStages) return SPLITK_ERR_NO_FIT;
  if (pl.b_stages != 0 || pl.persistent != 0) return SPLITK_ERR_BAD_PLAN;
  if (pl.w4_decoders != 1 && pl.w4_decoders != 2) return SPLITK_ERR_BAD_PLAN;
  const long long m_tiles = tiles_of(M, pl.mma_n);
  const long long n_tiles = ((long long)N + kMmaM - 1) / kMmaM;
  if (n_tiles > 65535 || L > 65535) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.grid[0] != (unsigned)(pl.split_k * m_tiles) || pl.grid[1] != (unsigned)n_tiles ||
      pl.grid[2] != (unsigned)L || pl.cluster[0] != (unsigned)pl.split_k || pl.cluster[1] != 1 ||
      pl.cluster[2] != 1) {
    return SPLITK_ERR_BAD_PLAN;
  }
  const int ncols_max = std::min(M, pl.mma_n);
  if (pl.split_k > 1 && (!pl.mailbox_dedicated || pl.mailbox_quads != (ncols_max + 3) / 4)) return SPLITK_ERR_BAD_PLAN;
  if (pl.reduce_scatter != 0 && (pl.reduce_scatter != 1 || pl.split_k < 2)) return SPLITK_ERR_BAD_PLAN;
  if (pl.b_resident != 1 || pl.l2_prefetch != 0) return SPLITK_ERR_BAD_PLAN;
  if (pl.a_tmem_tiles < 1 || pl.a_tmem_tiles > kMaxTmemTiles) return SPLITK_ERR_BAD_PLAN;
  // An issuer waits on a slot's next round only after its own previous tile
  // (nis tiles back) is full, which orders it after the slot's previous
  // round when the slots are at least as many as the issuers; otherwise a
  // phase-parity wait could return a round early.
  if (pl.mma_issuers < 1 || pl.mma_issuers > 2 || pl.mma_issuers > pl.a_tmem_tiles) return SPLITK_ERR_BAD_PLAN;
  if (pl.b_loader != 0 && pl.b_loader != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.pdl_trigger != 0 && pl.pdl_trigger != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.tmem_cols != tmem_cols_for(pl.mma_n, pl.a_tmem_tiles, pl.mma_issuers)) return SPLITK_ERR_BAD_PLAN;
  // the bf16 stage takes exactly the tile after the TMEM slots, which are
  // then each used once (a slot reused after the stage would be waited on a
  // round it never had)
  if (pl.w4_smem_tiles != 0 && (pl.w4_smem_tiles != 1 || kt != pl.a_tmem_tiles + 1)) return SPLITK_ERR_BAD_PLAN;
  const uint32_t ded = w4_mailbox_bytes(pl.split_k, pl.reduce_scatter, ncols_max);
  if (pl.smem_bytes < smem_bytes_w4(pl.mma_n, kt, pl.stages, ded, pl.w4_smem_tiles, pl.weight_format) ||
      pl.smem_bytes % 16 != 0) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.smem_bytes > smem_optin) return SPLITK_ERR_NO_FIT;
  if ((size_t)resident_by_smem(smem_per_sm, pl.smem_bytes) * pl.tmem_cols > 512u) return SPLITK_ERR_BAD_PLAN;
  *dedicated_bytes = ded;
  return SPLITK_OK;
}

// Re-derives everything a persistent plan implies and checks it.
int check_plan_persistent(const splitk_plan_t& pl, int M, int N, int K, int L, size_t smem_optin,
                          size_t smem_per_sm, uint32_t* dedicated_bytes) {
  if (pl.persistent != 1 || pl.mma_m != kMmaM) return SPLITK_ERR_BAD_PLAN;
  if (pl.mma_n != 16 && pl.mma_n != 32 && pl.mma_n != 64 && pl.mma_n != 128) return SPLITK_ERR_BAD_PLAN;
  if (!valid_split(pl.split_k)) return SPLITK_ERR_UNSUPPORTED_SPLIT;
  if (pl.split_k < 2) return SPLITK_ERR_BAD_PLAN;
  if (K % 8 != 0 || K > kMaxK || total_k_tiles(K) < pl.split_k) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.k_tiles_per_cta != (total_k_tiles(K) + pl.split_k - 1) / pl.split_k) return SPLITK_ERR_BAD_PLAN;
  if (pl.stages < 2 || pl.stages > kMaxStages) return SPLITK_ERR_BAD_PLAN;
  if (pl.b_stages != 0 && (pl.b_stages < 2 || pl.b_stages > kMaxStages)) return SPLITK_ERR_BAD_PLAN;
  if (L > 65535) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.grid[0] != (unsigned)pl.split_k || pl.grid[1] < 1 || pl.grid[1] > 65535 || pl.grid[2] != 1 ||
      pl.cluster[0] != (unsigned)pl.split_k || pl.cluster[1] != 1 || pl.cluster[2] != 1) {
    return SPLITK_ERR_BAD_PLAN;
  }
  const int ncols_max = std::min(M, pl.mma_n);
  const int nquads_max = (ncols_max + 3) / 4;
  // rounds of whole 16-column groups (or all of a tile's columns at once)
  if (pl.mailbox_quads < 1 || pl.mailbox_quads > nquads_max ||
      (pl.mailbox_quads % 4 != 0 && pl.mailbox_quads != nquads_max) ||
      pl.reduce_rounds != (nquads_max + pl.mailbox_quads - 1) / pl.mailbox_quads) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.reduce_scatter != 1 || pl.mailbox_dedicated != 1 || pl.b_resident != 0 || pl.a_tmem_tiles != 0 ||
      pl.mma_issuers != 1 || pl.b_loader != 0 || pl.l2_prefetch != 0 || pl.pdl_trigger != 0) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.tmem_cols != pow2_at_least(2u * tmem_acc_cols(pl.mma_n))) return SPLITK_ERR_BAD_PLAN;
  const int round_cols = persistent_round_cols(ncols_max, pl.mailbox_quads);
  const size_t smem = smem_bytes_persistent(pl.mma_n, pl.stages, pl.b_stages, round_cols);
  if (smem != pl.smem_bytes) return SPLITK_ERR_BAD_PLAN;
  if (smem > smem_optin) return SPLITK_ERR_NO_FIT;
  if ((size_t)resident_by_smem(smem_per_sm, smem) * pl.tmem_cols > 512u) return SPLITK_ERR_BAD_PLAN;
  *dedicated_bytes = (uint32_t)round_cols * kColumnBytes;
  return SPLITK_OK;
}

int check_plan(const splitk_plan_t& pl, int M, int N, int K, int L, size_t smem_optin,
               size_t smem_per_sm, uint32_t* dedicated_bytes) {
  if (is_quantized(pl.weight_format)) {
    return check_plan_w4(pl, M, N, K, L, smem_optin, smem_per_sm, dedicated_bytes);
  }
  if (pl.weight_format != SPLITK_WEIGHTS_BF16 || pl.w4_smem_tiles != 0 || pl.w4_decoders != 0) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.persistent != 0) return check_plan_persistent(pl, M, N, K, L, smem_optin, smem_per_sm, dedicated_bytes);
  if (pl.mma_m != kMmaM) return SPLITK_ERR_BAD_PLAN;
  if (pl.mma_n != 16 && pl.mma_n != 32 && pl.mma_n != 64 && pl.mma_n != 128) return SPLITK_ERR_BAD_PLAN;
  if (!valid_split(pl.split_k)) return SPLITK_ERR_UNSUPPORTED_SPLIT;
  if (K % 8 != 0 || K > kMaxK || total_k_tiles(K) < pl.split_k) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.k_tiles_per_cta != (total_k_tiles(K) + pl.split_k - 1) / pl.split_k) return SPLITK_ERR_BAD_PLAN;
  if (pl.stages < 2 || pl.stages > kMaxStages) return SPLITK_ERR_BAD_PLAN;
  const long long m_tiles = tiles_of(M, pl.mma_n);
  const long long n_tiles = ((long long)N + kMmaM - 1) / kMmaM;
  if (m_tiles * pl.split_k > 0x7FFFFFFFLL) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.b_stages != 0) return SPLITK_ERR_BAD_PLAN;
  if (n_tiles > 65535 || L > 65535) return SPLITK_ERR_INVALID_SHAPE;
  if (pl.grid[0] != (unsigned)(pl.split_k * m_tiles) || pl.grid[1] != (unsigned)n_tiles ||
      pl.grid[2] != (unsigned)L || pl.cluster[0] != (unsigned)pl.split_k || pl.cluster[1] != 1 ||
      pl.cluster[2] != 1) {
    return SPLITK_ERR_BAD_PLAN;
  }
  const int ncols_max = std::min(M, pl.mma_n);
  const int nquads_max = (ncols_max + 3) / 4;
  if (pl.mailbox_quads < 1 || pl.mailbox_quads > pl.mma_n / 4 ||
      (pl.mailbox_quads % 4 != 0 && pl.mailbox_quads < nquads_max)) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.pdl_trigger != 0 && pl.pdl_trigger != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.reduce_scatter != 0 && pl.reduce_scatter != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.b_resident != 0 && pl.b_resident != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.a_tmem_tiles < 0 || pl.a_tmem_tiles > kMaxTmemTiles || pl.a_tmem_tiles > pl.k_tiles_per_cta ||
      (pl.a_tmem_tiles > 0 && !pl.b_resident)) {
    return SPLITK_ERR_BAD_PLAN;
  }
  if (pl.mma_issuers != 1 && pl.mma_issuers != 2) return SPLITK_ERR_BAD_PLAN;
  // Each ring stage must have one consumer that waits its rounds in order: a
  // phase-parity wait issued a round early returns at once, and its tile's
  // copy could then still be landing when the CTA exits.  Issuer i takes the
  // K tiles i, i + issuers, ..., so stage s belongs to issuer s % issuers
  // exactly when the stage count is a multiple of the issuer count.
  if (pl.stages % pl.mma_issuers != 0) return SPLITK_ERR_BAD_PLAN;
  if (pl.b_loader != 0 && (pl.b_loader != 1 || !pl.b_resident)) return SPLITK_ERR_BAD_PLAN;
  if (pl.l2_prefetch != 0 && pl.l2_prefetch != 1) return SPLITK_ERR_BAD_PLAN;
  if (pl.tmem_cols != tmem_cols_for(pl.mma_n, pl.a_tmem_tiles, pl.mma_issuers)) return SPLITK_ERR_BAD_PLAN;
  uint32_t ded = 0;
  if (pl.reduce_scatter) {
    // every rank's slice of every source rank, one round, own region
    if (pl.split_k < 2 || !pl.mailbox_dedicated || pl.mailbox_quads < nquads_max) return SPLITK_ERR_BAD_PLAN;
    ded = (uint32_t)ncols_max * kColumnBytes;
  } else if (pl.split_k > 1) {
    const uint32_t round_bytes = mailbox_round_bytes(pl.split_k, pl.mailbox_quads, ncols_max);
    if (pl.mailbox_dedicated) {
      ded = round_bytes;
    } else if (round_bytes > (uint32_t)pl.stages * kAStageBytes) {
      return SPLITK_ERR_BAD_PLAN;
    }
  }
  const size_t smem =
      smem_bytes_for(pl.mma_n, pl.stages, ded, b_region_tiles_for(pl.stages, pl.b_resident, pl.k_tiles_per_cta));
  if (smem != pl.smem_bytes) return SPLITK_ERR_BAD_PLAN;
  if (smem > smem_optin) return SPLITK_ERR_NO_FIT;
  // tcgen05.alloc waits for free columns: however many CTAs fit an SM, their
  // allocations together must fit its 512 columns, or a CTA could wait on
  // one that waits on it (a cluster peer, or the next kernel's CTA that
  // waits for this kernel to complete).
  if ((size_t)resident_by_smem(smem_per_sm, smem) * pl.tmem_cols > 512u) return SPLITK_ERR_BAD_PLAN;
  *dedicated_bytes = ded;
  return SPLITK_OK;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

// A 3-D bf16 tensor [d2][d1][d0] (d0 contiguous) read in boxes of
// {64, rows, 1} with the 128-byte swizzle; out-of-range rows read as zero.
bool encode_3d(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2u, d0 * d1 * 2u};
  cuuint32_t box[3] = {(cuuint32_t)kAtomK, box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Quantized weight codes [L][N][row_bytes] read in boxes of one packed K
// tile by 128 rows: A16W4 {64 B, 128, 1} with the 64-byte swizzle, A16W8
// {128 B, 128, 1} with the 128-byte swizzle (each decoding thread reads its
// row conflict-free); out-of-range rows read as zero codes.
bool encode_3d_w4(CUtensorMap* map, const void* ptr, uint64_t row_bytes, uint64_t d1, uint64_t d2,
                  int fmt = SPLITK_WEIGHTS_E2M1_E8M0) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool w8 = fmt == SPLITK_WEIGHTS_E4M3_E8M0;
  cuuint64_t dims[3] = {row_bytes, d1, d2};
  cuuint64_t strides[2] = {row_bytes, row_bytes * d1};
  cuuint32_t box[3] = {w8 ? kW8RowBytes : kW4RowBytes, (cuuint32_t)kMmaM, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, w8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct AKey {
  uintptr_t ptr;
  int N, K, L;
  int fmt;                    // SPLITK_WEIGHTS_*
  bool operator==(const AKey& o) const {
    return ptr == o.ptr && N == o.N && K == o.K && L == o.L && fmt == o.fmt;
  }
};
struct BKey {
  uintptr_t ptr;
  int M, K, L, rows;
  bool operator==(const BKey& o) const {
    return ptr == o.ptr && M == o.M && K == o.K && L == o.L && rows == o.rows;
  }
};
inline uint64_t mix(uint64_t h, uint64_t v) {
  h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
  return h;
}
struct AKeyHash {
  size_t operator()(const AKey& k) const {
    return (size_t)mix(mix(mix(mix(mix(0, k.ptr), (uint64_t)k.N), (uint64_t)k.K), (uint64_t)k.L), (uint64_t)k.fmt);
  }
};
struct BKeyHash {
  size_t operator()(const BKey& k) const {
    return (size_t)mix(mix(mix(mix(mix(0, k.ptr), (uint64_t)k.M), (uint64_t)k.K), (uint64_t)k.L),
                       (uint64_t)k.rows);
  }
};

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  size_t smem_per_sm = 0;
  size_t smem_optin = 0;
  CUtensorMap* d_pool = nullptr;   // device tensor maps of A
  CUtensorMap* h_pool = nullptr;   // pinned mirror, never rewritten once used
  int used = 0;
  std::unordered_map<AKey, int, AKeyHash> a_slots;
  std::unordered_map<BKey, CUtensorMap, BKeyHash> b_maps;
  int max_clusters[9] = {};        // persistent kernel: clusters of 2, 4, 8 resident at once (0: unknown)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
// Device address of g_noalloc_scratch per device (null until looked up).
void* g_noalloc_addr[kMaxDevices] = {};

// Caller holds g_mu.  Returns the current device's state, initialised.
int current_device(DeviceState** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SPLITK_ERR_UNSUPPORTED_DEVICE;
  }
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0, optin = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return SPLITK_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return SPLITK_ERR_UNSUPPORTED_DEVICE;
    if (!encode_fn()) return SPLITK_ERR_CUDA;
    if (prepare_kernels(optin) != cudaSuccess || prepare_persistent(optin) != cudaSuccess) {
      cudaGetLastError();
      return SPLITK_ERR_CUDA;
    }
    st.num_sms = sms;
    st.smem_optin = (size_t)optin;
    st.smem_per_sm = (size_t)per_sm;
    // Clusters of the persistent kernel that fit the device at once, one CTA
    // an SM (the shared memory of its plans), queried here rather than at a
    // launch that may be part of a graph capture.
    for (int split : {2, 4, 8}) {
      int fit = 0;
      if (max_active_clusters_persistent(128, (unsigned)split, (size_t)optin, &fit) != cudaSuccess) {
        cudaGetLastError();
        fit = 0;
      }
      st.max_clusters[split] = fit;
    }
    st.ready = true;
  }
  *out = &st;
  if (dev_out) *dev_out = dev;
  return SPLITK_OK;
}

// Caller holds g_mu.  Device address of A's tensor map, encoding and
// copying it on `stream` the first time.
int a_map_for(DeviceState& st, const void* a, int N, int K, int L, cudaStream_t stream,
              const CUtensorMap** out, int fmt = SPLITK_WEIGHTS_BF16) {
  AKey key{(uintptr_t)a, N, K, L, fmt};
  auto it = st.a_slots.find(key);
  if (it != st.a_slots.end()) {
    *out = st.d_pool + it->second;
    return SPLITK_OK;
  }
  if (!st.d_pool) {
    if (cudaMalloc((void**)&st.d_pool, sizeof(CUtensorMap) * kMapPoolSlots) != cudaSuccess) {
      cudaGetLastError();
      st.d_pool = nullptr;
      return SPLITK_ERR_CUDA;
    }
    if (cudaMallocHost((void**)&st.h_pool, sizeof(CUtensorMap) * kMapPoolSlots) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(st.d_pool);
      st.d_pool = nullptr;
      st.h_pool = nullptr;
      return SPLITK_ERR_CUDA;
    }
    st.used = 0;
  }
  if (st.used >= kMapPoolSlots) return SPLITK_ERR_CACHE_FULL;
  const int slot = st.used;
  const bool encoded =
      fmt == SPLITK_WEIGHTS_E2M1_E8M0   ? encode_3d_w4(&st.h_pool[slot], a, (uint64_t)K / 2u, (uint64_t)N, (uint64_t)L)
      : fmt == SPLITK_WEIGHTS_E4M3_E8M0 ? encode_3d_w4(&st.h_pool[slot], a, (uint64_t)K, (uint64_t)N, (uint64_t)L, fmt)
                                        : encode_3d(&st.h_pool[slot], a, (uint64_t)K, (uint64_t)N, (uint64_t)L,
                                                    (uint32_t)kMmaM);
  if (!encoded) return SPLITK_ERR_CUDA;
  // Outside a graph capture the copy completes before this returns, so a
  // launch on any stream may use the slot from now on; inside a capture it
  // becomes a node of the graph, ordered before the kernel on `stream`.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  const cudaError_t copied =
      cap == cudaStreamCaptureStatusNone
          ? cudaMemcpy(st.d_pool + slot, st.h_pool + slot, sizeof(CUtensorMap), cudaMemcpyHostToDevice)
          : cudaMemcpyAsync(st.d_pool + slot, st.h_pool + slot, sizeof(CUtensorMap),
                            cudaMemcpyHostToDevice, stream);
  if (copied != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  st.used = slot + 1;
  st.a_slots.emplace(key, slot);
  *out = st.d_pool + slot;
  return SPLITK_OK;
}

int b_map_for(DeviceState& st, const void* b, int M, int K, int L, int rows, CUtensorMap* out) {
  BKey key{(uintptr_t)b, M, K, L, rows};
  auto it = st.b_maps.find(key);
  if (it != st.b_maps.end()) {
    *out = it->second;
    return SPLITK_OK;
  }
  CUtensorMap m;
  if (!encode_3d(&m, b, (uint64_t)K, (uint64_t)M, (uint64_t)L, (uint32_t)rows)) return SPLITK_ERR_CUDA;
  if (st.b_maps.size() >= kBMapCacheMax) st.b_maps.clear();
  st.b_maps.emplace(key, m);
  *out = m;
  return SPLITK_OK;
}

int check_pointers(const void* a, const void* b, const void* c) {
  if (!a || !b || !c) return SPLITK_ERR_NULL;
  if (((uintptr_t)a & 15u) || ((uintptr_t)b & 15u) || ((uintptr_t)c & 1u)) return SPLITK_ERR_MISALIGNED;
  return SPLITK_OK;
}

// The kernel's parameters for a checked plan.
void fill_params(const splitk_plan_t& pl, int M, int N, int K, int L, uint32_t ded, const CUtensorMap* a_map,
                 const void* b, void* c, const void* bias, KernelParams* p, const void* a_scale = nullptr) {
  p->a_map = a_map;
  p->a_scale = static_cast<const uint8_t*>(a_scale);
  p->b = static_cast<const uint16_t*>(b);
  p->c = static_cast<uint16_t*>(c);
  p->bias = static_cast<const uint16_t*>(bias);
  p->M = M;
  p->N = N;
  p->K = K;
  p->L = L;
  p->split = pl.split_k;
  p->stages = pl.stages;
  p->b_stages = pl.persistent != 0 && pl.b_stages != 0 ? pl.b_stages : pl.stages;
  p->k_tiles_total = total_k_tiles(K);
  p->mailbox_dedicated = pl.split_k > 1 ? pl.mailbox_dedicated : 0;
  p->mailbox_bytes = ded;
  p->mailbox_quads = pl.mailbox_quads;
  p->vec_store = ((N % 8) == 0 && ((uintptr_t)c & 15u) == 0) ? 1 : 0;
  p->wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p->inject = g_inject.load(std::memory_order_relaxed);
  p->pdl_trigger_early = pl.pdl_trigger;
  p->reduce_scatter = pl.reduce_scatter;
  p->b_resident = pl.b_resident;
  p->b_region_tiles = is_quantized(pl.weight_format)
                          ? std::max(2, pl.k_tiles_per_cta)
                          : b_region_tiles_for(pl.stages, pl.b_resident, pl.k_tiles_per_cta);
  p->a_tmem_tiles = pl.a_tmem_tiles;
  p->tmem_cols = pl.tmem_cols;
  p->tmem_tile_col0 = tmem_tile_col0(pl.mma_n, pl.mma_issuers);
  p->mma_issuers = pl.mma_issuers;
  p->b_loader = pl.b_loader;
  p->w4_smem_tiles = pl.w4_smem_tiles;
  p->l2_prefetch = pl.l2_prefetch;
  p->trace = g_trace.load(std::memory_order_relaxed);
  p->trace_ctas = p->trace ? g_trace_ctas.load(std::memory_order_relaxed) : 0u;
}

LaunchArgs launch_args(const splitk_plan_t& pl, bool pdl) {
  LaunchArgs la;
  la.mma_n = pl.mma_n;
  la.fmt = pl.weight_format == SPLITK_WEIGHTS_E2M1_E8M0 ? 1 : pl.weight_format == SPLITK_WEIGHTS_E4M3_E8M0 ? 2 : 0;
  la.persistent = pl.persistent != 0;
  la.w4_decoders = pl.w4_decoders == 2 ? 2 : 1;
  la.grid = dim3(pl.grid[0], pl.grid[1], pl.grid[2]);
  la.cluster_x = (unsigned)pl.split_k;
  la.smem_bytes = pl.smem_bytes;
  la.pdl = pdl;
  return la;
}

// Caller holds g_mu.  Launches a checked plan: the per-tile kernel, or the
// persistent one with as many clusters as the device holds at once (at most
// the plan's grid[1] and the output tiles; the kernel is correct for any
// number, as each cluster walks the tiles that many apart).
cudaError_t launch_plan(DeviceState& st, const splitk_plan_t& pl, const LaunchArgs& la0, const CUtensorMap& b_map,
                        const KernelParams& p, int M, int N, int L, cudaStream_t stream) {
  if (!la0.persistent) return launch_kernel(la0, b_map, p, stream);
  LaunchArgs la = la0;
  const int fit = pl.split_k >= 2 && pl.split_k <= 8 ? st.max_clusters[pl.split_k] : 0;
  const long long tiles = tiles_of(M, pl.mma_n) * tiles_of(N, kMmaM) * L;
  long long g = std::min<long long>((long long)pl.grid[1], tiles);
  if (fit > 0) g = std::min<long long>(g, fit);       // 0: unknown, the plan's own bound
  la.grid = dim3((unsigned)pl.split_k, (unsigned)std::max<long long>(1, g), 1u);
  return launch_persistent(la, b_map, p, stream);
}

// Caller holds g_mu.
int launch_locked(DeviceState& st, const void* a, const void* b, void* c, int M, int N, int K, int L,
                  const splitk_plan_t& pl, unsigned flags, cudaStream_t stream,
                  const void* bias = nullptr, const void* a_scale = nullptr) {
  uint32_t ded = 0;
  int rc = check_plan(pl, M, N, K, L, st.smem_optin, st.smem_per_sm, &ded);
  if (rc != SPLITK_OK) return rc;
  // the quantized kernels need their scales; the bf16 kernel takes none
  if (is_quantized(pl.weight_format) != (a_scale != nullptr)) return SPLITK_ERR_BAD_PLAN;
  const CUtensorMap* a_map = nullptr;
  rc = a_map_for(st, a, N, K, L, stream, &a_map, pl.weight_format);
  if (rc != SPLITK_OK) return rc;
  CUtensorMap b_map;
  rc = b_map_for(st, b, M, K, L, pl.mma_n, &b_map);
  if (rc != SPLITK_OK) return rc;

  KernelParams p;
  fill_params(pl, M, N, K, L, ded, a_map, b, c, bias, &p, a_scale);
  const LaunchArgs la = launch_args(pl, (flags & SPLITK_FLAG_NO_PDL) == 0);
  if (launch_plan(st, pl, la, b_map, p, M, N, L, stream) != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  return SPLITK_OK;
}

int gemm_auto(const void* a, const void* b, void* c, int M, int N, int K, int L, int split_k,
              unsigned flags, cudaStream_t stream, const void* bias = nullptr) {
  int rc = check_pointers(a, b, c);
  if (rc != SPLITK_OK) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  splitk_plan_t pl;
  rc = plan_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a, b, c, M, N, K, L, pl, flags, stream, bias);
}

// Every valid tactic for a shape on a described device: the plan's own
// choice first, then the page's ring (2-8 stages, one or two MMA issuers,
// either PDL trigger) and the staged family (2 stages, 0-3 weight tiles in
// tensor memory, resident activations loaded by TMA or by the epilogue
// threads, L2 prefetch of the tiles left off chip), for each split and each
// reduction (rank 0 with its own or an aliased mailbox, scattered).  Each
// candidate passes check_plan.
int enumerate_plans(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                    size_t smem_optin, std::vector<splitk_plan_t>* out) {
  splitk_plan_t base;
  std::memset(&base, 0, sizeof(base));
  int rc = plan_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_optin, &base);
  if (rc != SPLITK_OK) return rc;
  out->push_back(base);
  if (base.persistent) {
    // the per-tile kernel's own choice next, for comparison
    splitk_plan_t ring;
    if (plan_ring_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_optin, &ring) == SPLITK_OK) {
      out->push_back(ring);
    }
  }
  const int T = total_k_tiles(K);
  const int mma_n = base.mma_n;
  const long long m_tiles = tiles_of(M, mma_n);
  const long long n_tiles = ((long long)N + kMmaM - 1) / kMmaM;
  const int ncols_max = std::min(M, mma_n);
  const int nquads_max = (ncols_max + 3) / 4;
  auto same = [](const splitk_plan_t& x, const splitk_plan_t& y) { return std::memcmp(&x, &y, sizeof(x)) == 0; };
  for (int split : {1, 2, 4, 8}) {
    if ((split_k != 0 && split != split_k) || split > T) continue;
    const int kt = (T + split - 1) / split;
    for (int mode = 0; mode < 3; ++mode) {               // 0 own mailbox, 1 aliased, 2 scattered
      if (split == 1 && mode != 0) continue;
      if (mode == 2 && ncols_max < 4) continue;
      for (int b_res = 0; b_res <= 1; ++b_res) {
        for (int stages = 2; stages <= (b_res ? 2 : kMaxStages); ++stages) {
          if (stages > std::max(2, kt)) continue;
          for (int tiles = 0; tiles <= (b_res ? std::min(kMaxTmemTiles, kt) : 0); ++tiles) {
            for (int issuers = 1; issuers <= 2; ++issuers) {
              if (stages % issuers) continue;
              for (int trig = 0; trig <= 1; ++trig) {
                for (int loader = 0; loader <= b_res; ++loader) {
                  for (int pf = 0; pf <= (b_res && kt > stages + tiles ? 1 : 0); ++pf) {
                    splitk_plan_t p;
                    std::memset(&p, 0, sizeof(p));
                    p.mma_m = kMmaM;
                    p.mma_n = mma_n;
                    p.stages = stages;
                    p.split_k = split;
                    p.k_tiles_per_cta = kt;
                    p.grid[0] = (unsigned)(split * m_tiles);
                    p.grid[1] = (unsigned)n_tiles;
                    p.grid[2] = (unsigned)L;
                    p.cluster[0] = (unsigned)split;
                    p.cluster[1] = 1;
                    p.cluster[2] = 1;
                    p.pdl_trigger = trig;
                    p.reduce_scatter = mode == 2 ? 1 : 0;
                    p.b_resident = b_res;
                    p.a_tmem_tiles = tiles;
                    p.mma_issuers = issuers;
                    p.tmem_cols = tmem_cols_for(mma_n, tiles, issuers);
                    p.b_loader = loader;
                    p.l2_prefetch = pf;
                    uint32_t ded = 0;
                    int quads = nquads_max;
                    if (split == 1) {
                      p.mailbox_dedicated = 0;
                    } else if (mode == 0) {
                      p.mailbox_dedicated = 1;
                      ded = mailbox_round_bytes(split, quads, ncols_max);
                    } else if (mode == 1) {
                      p.mailbox_dedicated = 0;
                      if (mailbox_round_bytes(split, quads, ncols_max) > (uint32_t)stages * kAStageBytes) {
                        quads = 4;
                        while (quads + 4 <= nquads_max &&
                               mailbox_round_bytes(split, quads + 4, ncols_max) <= (uint32_t)stages * kAStageBytes) {
                          quads += 4;
                        }
                      }
                    } else {
                      p.mailbox_dedicated = 1;
                      ded = (uint32_t)ncols_max * kColumnBytes;
                    }
                    p.mailbox_quads = quads;
                    p.reduce_rounds = split > 1 ? (nquads_max + quads - 1) / quads : 0;
                    p.smem_bytes = smem_bytes_for(mma_n, stages, ded, b_region_tiles_for(stages, b_res, kt));
                    p.ctas_per_sm = std::min(3, resident_by_smem(smem_per_sm, p.smem_bytes));
                    uint32_t ded_check = 0;
                    if (p.ctas_per_sm < 1 || check_plan(p, M, N, K, L, smem_optin, smem_per_sm, &ded_check) != SPLITK_OK) {
                      continue;
                    }
                    bool dup = false;
                    for (const auto& q : *out) dup = dup || same(p, q);
                    if (!dup) out->push_back(p);
                  }
                }
              }
            }
          }
        }
      }
    }
    // the persistent kernel at every ring depth and reduction round that
    // fit, at the shape's token tile and (for more than 64 tokens) at
    // 64-token tiles, several of which share each weight tile; the
    // activations on the weight ring or on a ring of their own
    for (int tile_n : {mma_n, 64}) {
      if (tile_n != mma_n && M <= 64) continue;
      const int nq = (std::min(M, tile_n) + 3) / 4;
      for (int stages = 2; split >= 2 && stages <= kMaxStages; ++stages) {
        for (int b_stages = 0; b_stages <= kMaxStages; b_stages += b_stages == 0 ? 2 : 1) {
          for (int quads : {nq, 16, 8, 4}) {
            if (quads > nq || (quads != nq && quads % 4 != 0)) continue;
            splitk_plan_t p;
            uint32_t ded_check = 0;
            if (!persistent_plan(M, N, K, L, split, stages, b_stages, quads, num_sms, smem_per_sm, smem_optin, &p,
                                 tile_n) ||
                check_plan(p, M, N, K, L, smem_optin, smem_per_sm, &ded_check) != SPLITK_OK) {
              continue;
            }
            bool dup = false;
            for (const auto& q : *out) dup = dup || same(p, q);
            if (!dup) out->push_back(p);
          }
        }
      }
    }
  }
  return SPLITK_OK;
}

// The device address of page-locked, device-mapped host memory, or null.
void* mapped_device_pointer(const void* host) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
  return at.devicePointer;
}

}  // namespace
}  // namespace splitk

using namespace splitk;

extern "C" {

SPLITK_API int splitk_plan_for(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                               size_t smem_per_block_optin, splitk_plan_t* out) {
  return plan_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_per_block_optin, out);
}

SPLITK_API int splitk_plan(int M, int N, int K, int L, int split_k, splitk_plan_t* out) {
  if (!out) return SPLITK_ERR_NULL;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return plan_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, out);
}

SPLITK_API int splitk_gemm_bf16(const void* a, const void* b, void* c, int M, int N, int K, int L,
                                int split_k, splitk_stream_t stream) {
  return gemm_auto(a, b, c, M, N, K, L, split_k, 0u, reinterpret_cast<cudaStream_t>(stream));
}

SPLITK_API int splitk_gemm_bf16_bias(const void* a, const void* b, const void* bias, void* c, int M,
                                     int N, int K, int L, int split_k, splitk_stream_t stream) {
  if (!bias) return SPLITK_ERR_NULL;
  if ((uintptr_t)bias & 1u) return SPLITK_ERR_MISALIGNED;
  return gemm_auto(a, b, c, M, N, K, L, split_k, 0u, reinterpret_cast<cudaStream_t>(stream), bias);
}

SPLITK_API int splitk_gemm_bf16_planned(const void* a, const void* b, void* c, int M, int N, int K,
                                        int L, const splitk_plan_t* plan, unsigned flags,
                                        splitk_stream_t stream) {
  if (!plan) return SPLITK_ERR_NULL;
  int rc = check_pointers(a, b, c);
  if (rc != SPLITK_OK) return rc;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a, b, c, M, N, K, L, *plan, flags, reinterpret_cast<cudaStream_t>(stream));
}

SPLITK_API int splitk_gemm_bf16_hostio(const void* a, const void* b_host, void* c_host, void* b_dev,
                                       void* c_dev, int M, int N, int K, int L, int split_k,
                                       splitk_stream_t stream) {
  if (!b_host || !c_host) return SPLITK_ERR_NULL;
  int rc = check_pointers(a, b_dev, c_dev);
  if (rc != SPLITK_OK) return rc;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  splitk_plan_t pl;
  rc = plan_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl);
  if (rc != SPLITK_OK) return rc;
  const size_t b_bytes = (size_t)L * (size_t)M * (size_t)K * 2u;
  const size_t c_bytes = (size_t)L * (size_t)M * (size_t)N * 2u;
  // Page-locked, device-mapped host buffers: the copies are kernels chained
  // to the GEMM by programmatic dependent launch, so the GEMM streams its
  // weights while the activations arrive and the copy-out is resident when
  // it completes.  Otherwise (pageable memory, odd alignment) the copy
  // engines, in stream order.
  void* b_mapped = mapped_device_pointer(b_host);
  void* c_mapped = mapped_device_pointer(c_host);
  const bool kernels = b_mapped != nullptr && c_mapped != nullptr &&
                       (((uintptr_t)b_mapped | (uintptr_t)b_dev | (uintptr_t)c_mapped | (uintptr_t)c_dev) & 15u) == 0;
  cudaError_t e = kernels ? launch_pdl_copy(b_mapped, b_dev, b_bytes, st->num_sms, s)
                          : cudaMemcpyAsync(b_dev, b_host, b_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  rc = launch_locked(*st, a, b_dev, c_dev, M, N, K, L, pl, 0u, s);
  if (rc != SPLITK_OK) return rc;
  e = kernels ? launch_pdl_copy(c_dev, c_mapped, c_bytes, st->num_sms, s)
              : cudaMemcpyAsync(c_host, c_dev, c_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  return SPLITK_OK;
}

SPLITK_API int splitk_gemm_bf16_zerocopy(const void* a, const void* b_host, void* c_host, int M, int N, int K,
                                         int L, int split_k, splitk_stream_t stream) {
  if (!a || !b_host || !c_host) return SPLITK_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  void* b_dev = mapped_device_pointer(b_host);
  void* c_dev = mapped_device_pointer(c_host);
  if (!b_dev || !c_dev) return SPLITK_ERR_NOT_MAPPED;
  rc = check_pointers(a, b_dev, c_dev);
  if (rc != SPLITK_OK) return rc;
  splitk_plan_t pl;
  rc = plan_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl);
  if (rc != SPLITK_OK) return rc;
  // the epilogue threads' loads read the host memory; TMA is not used on it
  if (!pl.b_resident) return SPLITK_ERR_NO_FIT;
  pl.b_loader = 1;
  return launch_locked(*st, a, b_dev, c_dev, M, N, K, L, pl, 0u, reinterpret_cast<cudaStream_t>(stream));
}

SPLITK_API int splitk_gemm_bf16_noalloc(const void* a, const void* b, void* c, int M, int N, int K,
                                        int L, int split_k, splitk_stream_t stream) {
  int rc = check_pointers(a, b, c);
  if (rc != SPLITK_OK) return rc;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  // The call needs one tensor map of scratch; the array holds that much.
  if (sizeof(CUtensorMap) > kNoAllocScratchBytes) return SPLITK_ERR_SCRATCH;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int dev = -1;
  rc = current_device(&st, &dev);
  if (rc != SPLITK_OK) return rc;
  // The tensor map is copied from a host variable of this call: a graph
  // would copy it again at every replay, after the call has returned.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return SPLITK_ERR_CAPTURE;
  splitk_plan_t pl;
  rc = plan_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl);
  if (rc != SPLITK_OK) return rc;
  uint32_t ded = 0;
  rc = check_plan(pl, M, N, K, L, st->smem_optin, st->smem_per_sm, &ded);
  if (rc != SPLITK_OK) return rc;
  if (pl.weight_format != SPLITK_WEIGHTS_BF16) return SPLITK_ERR_BAD_PLAN;
  // Set-up, once per device, with that device current: the device address of
  // the scratch array.
  if (g_noalloc_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return SPLITK_ERR_CUDA;
    }
    g_noalloc_addr[dev] = addr;
  }
  CUtensorMap* scratch_map = static_cast<CUtensorMap*>(g_noalloc_addr[dev]);
  // A's tensor map goes into the scratch array on the stream (the whole map is
  // rewritten, so nothing in the array has to start at zero); B's is a launch
  // parameter.  Both are encoded here, on the host, without caching.
  CUtensorMap a_map, b_map;
  if (!encode_3d(&a_map, a, (uint64_t)K, (uint64_t)N, (uint64_t)L, (uint32_t)kMmaM) ||
      !encode_3d(&b_map, b, (uint64_t)K, (uint64_t)M, (uint64_t)L, (uint32_t)pl.mma_n)) {
    return SPLITK_ERR_CUDA;
  }
  // The source is a pageable local: cudaMemcpyAsync returns only once it has
  // been staged, so it may go out of scope afterwards.  The same device
  // address is rewritten by every call; the kernel orders this generic-proxy
  // write before its TMA loads with fence.proxy.tensormap::generic.acquire at
  // its start, which the copy precedes in stream order.
  if (cudaMemcpyAsync(scratch_map, &a_map, sizeof(CUtensorMap), cudaMemcpyHostToDevice, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  KernelParams p;
  fill_params(pl, M, N, K, L, ded, scratch_map, b, c, nullptr, &p);
  const LaunchArgs la = launch_args(pl, true);
  if (launch_plan(*st, pl, la, b_map, p, M, N, L, s) != cudaSuccess) {
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  return SPLITK_OK;
}

SPLITK_API int splitk_plan_w4a16_for(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                                     size_t smem_per_block_optin, splitk_plan_t* out) {
  return plan_w4_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_per_block_optin, out);
}

SPLITK_API int splitk_plan_w4a16(int M, int N, int K, int L, int split_k, splitk_plan_t* out) {
  if (!out) return SPLITK_ERR_NULL;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return plan_w4_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, out);
}

SPLITK_API int splitk_gemm_w4a16_planned(const void* a_q, const void* a_scale, const void* b, void* c, int M,
                                         int N, int K, int L, const splitk_plan_t* plan, unsigned flags,
                                         splitk_stream_t stream) {
  if (!plan || !a_scale) return SPLITK_ERR_NULL;
  int rc = check_pointers(a_q, b, c);
  if (rc != SPLITK_OK) return rc;
  if ((uintptr_t)a_scale & 3u) return SPLITK_ERR_MISALIGNED;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  if (plan->weight_format != SPLITK_WEIGHTS_E2M1_E8M0) return SPLITK_ERR_BAD_PLAN;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a_q, b, c, M, N, K, L, *plan, flags, reinterpret_cast<cudaStream_t>(stream), nullptr,
                       a_scale);
}

SPLITK_API int splitk_gemm_w4a16(const void* a_q, const void* a_scale, const void* b, void* c, int M, int N,
                                 int K, int L, int split_k, splitk_stream_t stream) {
  if (!a_scale) return SPLITK_ERR_NULL;
  int rc = check_pointers(a_q, b, c);
  if (rc != SPLITK_OK) return rc;
  if ((uintptr_t)a_scale & 3u) return SPLITK_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  splitk_plan_t pl;
  rc = plan_w4_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a_q, b, c, M, N, K, L, pl, 0u, reinterpret_cast<cudaStream_t>(stream), nullptr,
                       a_scale);
}

SPLITK_API int splitk_plan_w8a16_for(int M, int N, int K, int L, int split_k, int num_sms, size_t smem_per_sm,
                                     size_t smem_per_block_optin, splitk_plan_t* out) {
  return plan_w4_impl(M, N, K, L, split_k, num_sms, smem_per_sm, smem_per_block_optin, out, SPLITK_WEIGHTS_E4M3_E8M0);
}

SPLITK_API int splitk_plan_w8a16(int M, int N, int K, int L, int split_k, splitk_plan_t* out) {
  if (!out) return SPLITK_ERR_NULL;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return plan_w4_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, out,
                      SPLITK_WEIGHTS_E4M3_E8M0);
}

SPLITK_API int splitk_gemm_w8a16_planned(const void* a_q, const void* a_scale, const void* b, void* c, int M,
                                         int N, int K, int L, const splitk_plan_t* plan, unsigned flags,
                                         splitk_stream_t stream) {
  if (!plan || !a_scale) return SPLITK_ERR_NULL;
  int rc = check_pointers(a_q, b, c);
  if (rc != SPLITK_OK) return rc;
  if ((uintptr_t)a_scale & 3u) return SPLITK_ERR_MISALIGNED;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  if (plan->weight_format != SPLITK_WEIGHTS_E4M3_E8M0) return SPLITK_ERR_BAD_PLAN;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a_q, b, c, M, N, K, L, *plan, flags, reinterpret_cast<cudaStream_t>(stream), nullptr,
                       a_scale);
}

SPLITK_API int splitk_gemm_w8a16(const void* a_q, const void* a_scale, const void* b, void* c, int M, int N,
                                 int K, int L, int split_k, splitk_stream_t stream) {
  if (!a_scale) return SPLITK_ERR_NULL;
  int rc = check_pointers(a_q, b, c);
  if (rc != SPLITK_OK) return rc;
  if ((uintptr_t)a_scale & 3u) return SPLITK_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  splitk_plan_t pl;
  rc = plan_w4_impl(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &pl,
                    SPLITK_WEIGHTS_E4M3_E8M0);
  if (rc != SPLITK_OK) return rc;
  return launch_locked(*st, a_q, b, c, M, N, K, L, pl, 0u, reinterpret_cast<cudaStream_t>(stream), nullptr,
                       a_scale);
}

SPLITK_API int splitk_plan_check_for(const splitk_plan_t* plan, int M, int N, int K, int L,
                                     size_t smem_per_sm, size_t smem_per_block_optin) {
  if (!plan) return SPLITK_ERR_NULL;
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  uint32_t ded = 0;
  return check_plan(*plan, M, N, K, L, smem_per_block_optin, smem_per_sm, &ded);
}

SPLITK_API int splitk_plan_candidates_for(int M, int N, int K, int L, int split_k, int num_sms,
                                          size_t smem_per_sm, size_t smem_per_block_optin,
                                          splitk_plan_t* out, int max_out) {
  if (max_out > 0 && !out) return SPLITK_ERR_NULL;
  std::vector<splitk_plan_t> all;
  const int rc = enumerate_plans(M, N, K, L, split_k, num_sms, smem_per_sm, smem_per_block_optin, &all);
  if (rc != SPLITK_OK) return rc;
  for (int i = 0; i < (int)all.size() && i < max_out; ++i) out[i] = all[(size_t)i];
  return (int)all.size();
}

SPLITK_API int splitk_tune(const void* const* a_list, int n_a, const void* b, void* c, int M, int N, int K,
                           int L, int split_k, int reps, splitk_stream_t stream, splitk_plan_t* best,
                           float* best_us_per_call) {
  if (!a_list || n_a < 1 || !best) return SPLITK_ERR_NULL;
  for (int i = 0; i < n_a; ++i) {
    const int rc = check_pointers(a_list[i], b, c);
    if (rc != SPLITK_OK) return rc;
  }
  if (M < 1 || N < 1 || K < 1 || L < 1) return SPLITK_ERR_INVALID_SHAPE;
  if (reps < 1) reps = 64;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  int rc = current_device(&st, nullptr);
  if (rc != SPLITK_OK) return rc;
  std::vector<splitk_plan_t> cands;
  rc = enumerate_plans(M, N, K, L, split_k, st->num_sms, st->smem_per_sm, st->smem_optin, &cands);
  if (rc != SPLITK_OK) return rc;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    cudaGetLastError();
    return SPLITK_ERR_CUDA;
  }
  float best_ms = -1.0f;
  for (const splitk_plan_t& p : cands) {
    // one pass over the weights to warm the tensor maps and the code
    for (int i = 0; i < n_a && rc == SPLITK_OK; ++i) rc = launch_locked(*st, a_list[i], b, c, M, N, K, L, p, 0u, s);
    if (rc == SPLITK_OK && cudaEventRecord(e0, s) != cudaSuccess) rc = SPLITK_ERR_CUDA;
    for (int r = 0; r < reps && rc == SPLITK_OK; ++r) {
      rc = launch_locked(*st, a_list[r % n_a], b, c, M, N, K, L, p, 0u, s);
    }
    float ms = 0.0f;
    if (rc == SPLITK_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)) {
      rc = SPLITK_ERR_CUDA;
    }
    if (rc != SPLITK_OK) break;
    if (best_ms < 0.0f || ms < best_ms) {
      best_ms = ms;
      *best = p;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != SPLITK_OK) {
    cudaGetLastError();
    return rc;
  }
  if (best_us_per_call) *best_us_per_call = best_ms * 1000.0f / (float)reps;
  return SPLITK_OK;
}

SPLITK_API int splitk_get_fault(splitk_fault_t* out) {
  int words[kFaultWords] = {0};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return SPLITK_ERR_UNSUPPORTED_DEVICE;
    }
    int words_p[kFaultWords] = {0};
    if (read_and_clear_fault(words) != cudaSuccess || read_and_clear_fault_persistent(words_p) != cudaSuccess) {
      cudaGetLastError();
      return SPLITK_ERR_CUDA;
    }
    if (words[0] == 0) std::memcpy(words, words_p, sizeof(words));
  }
  if (out) {
    out->code = words[0];
    out->role = words[1];
    out->index = words[2];
    out->parity = words[3];
    out->block[0] = words[4];
    out->block[1] = words[5];
    out->block[2] = words[6];
    out->cluster_rank = words[7];
  }
  return words[0] == 0 ? SPLITK_OK : SPLITK_ERR_TIMEOUT;
}

SPLITK_API int splitk_get_status(void) { return splitk_get_fault(nullptr); }

SPLITK_API int splitk_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : (unsigned long long)ns);
  return SPLITK_OK;
}

SPLITK_API int splitk_debug_inject(unsigned flags) {
  g_inject.store(flags & kInjectSkipPublish);
  return SPLITK_OK;
}

SPLITK_API int splitk_set_trace(void* device_buffer, size_t bytes) {
  if (device_buffer && ((uintptr_t)device_buffer & 7u)) return SPLITK_ERR_MISALIGNED;
  const size_t ctas = device_buffer ? bytes / (sizeof(unsigned long long) * kTraceSlots) : 0;
  g_trace_ctas.store((unsigned)std::min<size_t>(ctas, 0xFFFFFFFFu));
  g_trace.store(ctas ? static_cast<unsigned long long*>(device_buffer) : nullptr);
  return SPLITK_OK;
}

SPLITK_API int splitk_cache_info(size_t* device_bytes, size_t* host_bytes, int* maps) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SPLITK_ERR_UNSUPPORTED_DEVICE;
  }
  const DeviceState& st = g_dev[dev];
  const size_t pool = sizeof(CUtensorMap) * (size_t)kMapPoolSlots;
  if (device_bytes) *device_bytes = st.d_pool ? pool : 0u;
  if (host_bytes) *host_bytes = st.h_pool ? pool : 0u;
  if (maps) *maps = st.d_pool ? st.used : 0;
  return SPLITK_OK;
}

SPLITK_API void splitk_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int prev = -1;
  bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& st = g_dev[d];
    if (!st.ready) continue;
    if (cudaSetDevice(d) == cudaSuccess) {
      cudaDeviceSynchronize();
      if (st.d_pool) cudaFree(st.d_pool);
      if (st.h_pool) cudaFreeHost(st.h_pool);
    }
    st.d_pool = nullptr;
    st.h_pool = nullptr;
    st.used = 0;
    st.a_slots.clear();
    st.b_maps.clear();
  }
  if (have_prev) cudaSetDevice(prev);
  cudaGetLastError();
}

SPLITK_API const char* splitk_strerror(int code) {
  switch (code) {
    case SPLITK_OK: return "success";
    case SPLITK_ERR_INVALID_SHAPE: return "invalid shape (M, N, K, L >= 1; K a multiple of 8 with at least one 128-wide K tile per split rank; N, K, L and the grid within their limits)";
    case SPLITK_ERR_MISALIGNED: return "misaligned pointer (A and B need 16 bytes, C 2 bytes)";
    case SPLITK_ERR_UNSUPPORTED_SPLIT: return "split_k must be 0, 1, 2, 4 or 8";
    case SPLITK_ERR_NO_FIT: return "no tactic fits the shared-memory budget";
    case SPLITK_ERR_CUDA: return "a CUDA call failed";
    case SPLITK_ERR_TIMEOUT: return "a bounded wait in the kernel ran out";
    case SPLITK_ERR_NULL: return "null pointer argument";
    case SPLITK_ERR_CACHE_FULL: return "device tensor-map pool full; call splitk_release()";
    case SPLITK_ERR_UNSUPPORTED_DEVICE: return "no CUDA device of compute capability 10.3";
    case SPLITK_ERR_BAD_PLAN: return "plan does not match the shape";
    case SPLITK_ERR_SCRATCH: return "the call needs more scratch than the allocation-free array holds";
    case SPLITK_ERR_NOT_MAPPED: return "host buffer is not page-locked and mapped into the device address space";
    case SPLITK_ERR_CAPTURE: return "the allocation-free entry point cannot run inside a CUDA graph capture";
    default: return "unknown status code";
  }
}

SPLITK_API int splitk_version(void) { return 10000; }

}  // extern "C"
