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
constexpr int kEpiThreads = 128;   // warps 4..7, one per TMEM lane / weight row
constexpr int kMaxStages = 8;
constexpr uint32_t kAStageBytes = kMmaM * kCtaK * 2;        // 32 KiB
constexpr uint32_t kABoxBytes = kMmaM * kAtomK * 2;         // 16 KiB
constexpr uint32_t kBarRegionBytes = 256;
constexpr uint32_t kAlignSlack = 1024;                      // swizzle-128B atoms
constexpr uint32_t kQuadBytes = kEpiThreads * 4 * 4;        // one 4-column group
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;

__host__ __device__ constexpr uint32_t b_stage_bytes(int mma_n) { return (uint32_t)mma_n * kCtaK * 2; }
__host__ __device__ constexpr int max_quads_per_round(int mma_n) { return mma_n / 4 < 8 ? mma_n / 4 : 8; }

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
};

constexpr unsigned kInjectSkipPublish = 0x1u;

struct KernelParams {
  const CUtensorMap* a_map;   // device address of A's tensor map
  uint16_t* c;                // C[L][M][N] bf16 bits
  int M, N, K, L;
  int split;                  // cluster size along K
  int stages;                 // ring depth
  int k_tiles;                // K tiles per CTA
  int mailbox_dedicated;      // 1: own region after the ring, 0: rank 0's A ring
  uint32_t mailbox_bytes;     // size of the dedicated region (0 if aliased)
  int mailbox_quads;          // 4-column groups per reduction round
  int vec_store;              // 16-byte stores of C allowed
  unsigned long long wait_limit_ns;
  unsigned inject;
};

struct LaunchArgs {
  int mma_n;
  dim3 grid;
  unsigned cluster_x;
  size_t smem_bytes;
  bool pdl;
};

// Defined in splitk_kernel.cu.
cudaError_t launch_kernel(const LaunchArgs& la, const CUtensorMap& b_map,
                          const KernelParams& p, cudaStream_t stream);
cudaError_t prepare_kernels(int max_dynamic_smem);
cudaError_t read_and_clear_fault(int* out_words);

}  // namespace splitk
