// Internal declarations shared by the kernel and the host translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace splitk {

// Tile constants.  The weight tile is 128 rows (tcgen05 MMA M for one CTA);
// a K tile is 128 wide and arrives as two TMA boxes of 64 bf16 = 128 bytes,
// the width of the 128-byte swizzle ("two evict_first boxes per K tile",
// box {64, mma_m} in the page's SplitKGemm docstring); one bf16 tcgen05 MMA
// consumes K = 16.
constexpr int kMmaM = 128;
constexpr int kCtaK = 128;
constexpr int kAtomK = 64;
constexpr int kMmaK = 16;
constexpr int kThreads = 256;      // warps 0..7
constexpr int kThreadsW4Wide = 384;   // A16W4 with a second decoding warpgroup (warps 8..11)
constexpr int kEpiThreads = 128;   // warps 4..7, one per TMEM lane / weight row
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kMaxStages = 8;
constexpr uint32_t kAStageBytes = kMmaM * kCtaK * 2;        // 32 KiB
constexpr uint32_t kABoxBytes = kMmaM * kAtomK * 2;         // 16 KiB
constexpr uint32_t kBarRegionBytes = 256;
constexpr uint32_t kBarRegionBytesPersistent = 384;        // two rings' full/empty barriers
constexpr uint32_t kAlignSlack = 1024;                      // swizzle-128B atoms
constexpr uint32_t kColumnBytes = kEpiThreads * 4;          // one token column of f32 partials
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
// Longest a waiting thread sleeps in one mbarrier try_wait before it looks
// at the clock and the CTA's failure flag again.
constexpr uint32_t kWaitHintNs = 1000000u;

__host__ __device__ constexpr uint32_t b_stage_bytes(int mma_n) { return (uint32_t)mma_n * kCtaK * 2; }

// A16W4 weights: a K tile of 128 rows x 128 four-bit codes is 128 rows of 64
// bytes (one TMA box, 64-byte swizzle); its 4 scale codes per row (one per 32
// k) are read by the decoding threads.
constexpr uint32_t kW4TileBytes = kMmaM * kCtaK / 2;       // 8 KiB
constexpr uint32_t kW4RowBytes = kCtaK / 2;                 // 64
// A16W8 weights: 128 rows x 128 E4M3 codes = 128 rows of 128 bytes (one TMA
// box, 128-byte swizzle), the same 4 scale codes per row and K tile.
constexpr uint32_t kW8TileBytes = kMmaM * kCtaK;           // 16 KiB
constexpr uint32_t kW8RowBytes = kCtaK;                     // 128

// Tensor memory: one accumulator per MMA issuer, max(32, mma_n) columns
// each, from column 0; weight K tiles staged in tensor memory (64 columns
// each: 128 lanes x 128 bf16) from the next 64-column boundary.  Allocations
// are powers of two.
constexpr int kMaxTmemTiles = 3;
constexpr uint32_t kTmemTileCols = 64;
__host__ __device__ constexpr uint32_t tmem_acc_cols(int mma_n) { return mma_n < 32 ? 32u : (uint32_t)mma_n; }
__host__ __device__ constexpr uint32_t tmem_tile_col0(int mma_n, int issuers) {
  return (tmem_acc_cols(mma_n) * (uint32_t)issuers + 63u) & ~63u;
}
__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  return v <= 32u ? 32u : v <= 64u ? 64u : v <= 128u ? 128u : v <= 256u ? 256u : 512u;
}
__host__ __device__ constexpr uint32_t tmem_cols_for(int mma_n, int tmem_tiles, int issuers) {
  return pow2_at_least(tmem_tiles == 0 ? tmem_acc_cols(mma_n) * (uint32_t)issuers
                                       : tmem_tile_col0(mma_n, issuers) + kTmemTileCols * (uint32_t)tmem_tiles);
}

// Fault record in device memory (one per device, see splitk_fault_t).
constexpr int kFaultWords = 8;

// Fault roles.
enum Role : int {
  kRoleWeightTma = 0,
  kRoleActTma = 1,
  kRoleMma = 2,
  kRoleTmemRelease = 3,
  kRoleEpiMma = 4,
  kRoleEpiReduce = 5,
  kRoleEpiReady = 6,
  kRoleEpiDecode = 7,
  kRoleMmaAccFree = 8,   // persistent kernel: MMA issuer waiting for an accumulator to be read
};

constexpr unsigned kInjectSkipPublish = 0x1u;

struct KernelParams {
  const CUtensorMap* a_map;   // device address of A's tensor map
  uint16_t* c;                // C[L][M][N] bf16 bits
  const uint16_t* bias;       // [L][N] bf16 bits added before rounding, or null
  const uint16_t* b;          // activations B[L][M][K] (read directly when b_loader = 1)
  const uint8_t* a_scale;     // A16W4: scale codes [L][N][K/32] (null for bf16 weights)
  int M, N, K, L;
  int split;                  // cluster size along K
  int stages;                 // ring depth (persistent kernel: of the weight ring)
  int b_stages;               // persistent kernel: depth of the activation ring
  int k_tiles_total;          // 128-wide K tiles over all of K (last may be ragged)
  int mailbox_dedicated;      // 1: own region after the ring, 0: rank 0's A ring
  uint32_t mailbox_bytes;     // size of the dedicated region (0 if aliased)
  int mailbox_quads;          // 4-column groups per reduction round: a multiple of 4, or all
  int vec_store;              // 16-byte stores of C allowed
  unsigned long long wait_limit_ns;
  unsigned inject;
  int pdl_trigger_early;      // launch_dependents once TMEM is held, not after the weights
  int reduce_scatter;         // each rank sums and stores 128/split rows
  int b_resident;             // 1: all activation K tiles in their own buffer, one barrier
  int b_region_tiles;         // activation tiles the B region holds (ring stages or all)
  int a_tmem_tiles;           // leading weight K tiles moved into TMEM before the PDL wait
  uint32_t tmem_cols;         // TMEM columns allocated per CTA
  uint32_t tmem_tile_col0;    // TMEM column of the first staged weight tile
  int mma_issuers;            // 1 or 2 threads issuing MMAs (2: even/odd K tiles)
  int b_loader;               // 0: TMA (activation warp); 1: epilogue threads
  int w4_smem_tiles;          // A16W4: 1 = the tile after the TMEM slots is decoded into a bf16 stage in shared memory
  int l2_prefetch;            // 1: weight tiles not on chip before the PDL wait prefetched to L2
  unsigned long long* trace;  // per-CTA %globaltimer stamps, or null
  unsigned trace_ctas;        // CTAs the trace buffer holds
};

// Trace record of one CTA: kTraceSlots u64 words (see splitk_set_trace).
constexpr int kTraceSlots = 16;
enum TraceSlot : int {
  kTrSmRank = 0,        // %smid | cluster rank << 32
  kTrStart = 1,         // thread 0, first instruction
  kTrSynced = 2,        // thread 0, after the CTA/cluster barrier of the set-up
  kTrWeightsIssued = 3, // weight producer, after its last TMA issue
  kTrActReady = 4,      // activation producer, after griddepcontrol.wait
  kTrFirstFull = 5,     // MMA issuer, first stage landed
  kTrLastFull = 6,      // MMA issuer, last stage landed
  kTrMmaDone = 7,       // epilogue thread 0, accumulator complete
  kTrReduced = 8,       // epilogue thread 0: partials published (peer) / summed (rank 0)
  kTrStored = 9,        // epilogue thread 0 of rank 0, after its stores
  kTrEnd = 10,          // thread 0, after the final barrier
  kTrBarInit = 11,      // thread 0, mbarriers initialised and fenced
  kTrMapReady = 12,     // thread 0, A's tensor map acquired
  kTrPrefetched = 13,   // thread 0, weight loads of the first ring pass issued
  kTrTmemAlloc = 14,    // warp 2, TMEM allocated
  kTrEpiSynced = 15,    // epilogue thread 0, after the set-up barrier
};

struct LaunchArgs {
  int mma_n;
  int fmt;                    // 0 bf16 weights, 1 E2M1 codes, 2 E4M3 codes (with E8M0 scales)
  bool persistent;            // the persistent kernel (grid = (split, clusters, 1))
  int w4_decoders;            // A16W4: decoding warpgroups (1 or 2)
  dim3 grid;
  unsigned cluster_x;
  size_t smem_bytes;
  bool pdl;
};

// Defined in splitk_kernel.cu.
cudaError_t launch_kernel(const LaunchArgs& la, const CUtensorMap& b_map,
                          const KernelParams& p, cudaStream_t stream);
// A copy of `bytes` bytes (both pointers 16-byte aligned, either may be the
// device mapping of page-locked host memory) as a kernel in the stream's
// programmatic-dependent-launch chain (splitk_copy.cu).
cudaError_t launch_pdl_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t stream);
cudaError_t prepare_kernels(int max_dynamic_smem);
cudaError_t read_and_clear_fault(int* out_words);

// Defined in splitk_persistent.cu.
cudaError_t launch_persistent(const LaunchArgs& la, const CUtensorMap& b_map,
                              const KernelParams& p, cudaStream_t stream);
cudaError_t max_active_clusters_persistent(int mma_n, unsigned cluster_x, size_t smem, int* out);
cudaError_t prepare_persistent(int max_dynamic_smem);
cudaError_t read_and_clear_fault_persistent(int* out_words);

}  // namespace splitk
