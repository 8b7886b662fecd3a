// kernel_params.h -- parameter blocks shared by the host planner
// (agmm_api.cpp) and the sm_103a kernels (agmm_kernels.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace agmm {

constexpr int kMaxShards = 8;
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;       // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr int kTileM = 128;         // MMA M (one CTA, 128 TMEM lanes)
constexpr int kTileK = 64;          // k per stage: one 128-byte swizzle row of bf16
constexpr int kASlotBytes = kTileM * kTileK * 2;  // 16 KiB
constexpr int kStatusBytes = 256;   // status words at the start of the workspace
constexpr int kTraceSlots = 16;     // u64 slots per CTA in the optional trace
constexpr int kCtlBytes = 1024;     // per-CTA control block: barriers, flags, swap-path chunk table
constexpr int kMaxSwapChunks = 32;  // swap path: at most 256 rows in chunks of >= 8 rows
constexpr int kMaxSplits = 16;      // swap path: largest cluster (non-portable size 16)

enum Path : int { kPathRows = 0, kPathSwap = 1 };

// Status word layout (int32 at the workspace base):
//   [0] first error code (0 = none), [1] role that gave up, [2] stage, [3] tile.
enum StatusRole : int { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleDrain = 4, kRoleStore = 5 };

struct __align__(128) KernelParams {
  CUtensorMap xmap[kMaxShards];  // shard r: [m_pd, k] bf16, box {64, box_rows}, 128B swizzle
  CUtensorMap ymap;              // Y: K-major box {64, rows}; MN-major box {64, 64} or,
                                 // with y3d, {64, 64, blocks} over dims {64, k, n / 64}
  void* out;                     // O [P*m_pd, n], bf16 or f32
  int* status;                   // status words (may be null)
  int64_t m_pd;                  // rows per shard
  int64_t ldo;                   // row stride of O in elements (= n)
  int P;
  int my_id;
  int box_rows;                  // rows per chunk (a power of two, 8..128)
  int box_shift;                 // log2(box_rows)
  int whole_shards;              // chunks cover whole shards in ring first-visit order
  int total_chunks;              // chunks in the ring-ordered row sequence
  int num_m_tiles;               // row path: 128-row tiles of chunks
  int num_mc_tiles;              // row path: cluster rows = ceil(num_m_tiles / CTAs per cluster)
  int num_n_tiles;               // n tiles
  int num_k_blocks;              // k / 64
  int group_m;                   // row path: row tiles per raster group
  int num_tiles;                 // row path: num_mc_tiles * num_n_tiles (cluster tiles)
  int stages;                    // pipeline depth (<= kMaxStages)
  int mma_n;                     // MMA N
  int tmem_cols;                 // TMEM columns allocated (power of two >= 32)
  int splits;                    // swap path: k splits = cluster size
  uint32_t b_slot_bytes;         // bytes of one B-operand stage slot (multiple of 1024)
  uint64_t wait_limit_cycles;    // bound on every wait, in SM clock cycles
  int test_drop_first_arrive;    // test hook: producer skips its first arrival
  uint64_t* trace;               // optional [CTAs][kTraceSlots] timestamps (null: off)
  // Rows path work (hybrid stream-K).  Cluster tiles [0, dp_tiles) are dealt
  // round-robin to the clusters whole.  The k blocks of the remaining tiles
  // (sk units) are divided evenly: cluster c takes units [c*U/C, (c+1)*U/C).
  // A tile's k blocks may so be spread over consecutive clusters: the one
  // holding k block 0 owns the tile; the others (contributors) each leave a
  // float32 partial in sk_partials[cluster][cluster rank] and count themselves
  // in sk_flags[tile - dp_tiles][cluster rank].  The owner waits for them,
  // adds the partials in k order and resets the counter to 0.  Each cluster
  // works through its stream-K units first, then its whole tiles (the
  // gathered-LHS variant: its whole tiles first).
  int dp_tiles;
  int sk_min_units;              // unused on the device; planner bookkeeping
  int* sk_flags;                 // [sk tiles][cluster rank] arrival counters (zero between runs)
  float* sk_partials;            // [clusters][cluster rank][BN/32][8][128][4]
  // Swap path with k splits: float32 partials in device memory
  // [row group][n tile][split][quad][128 lanes][4] (null: the partials go
  // through distributed shared memory instead).
  float* swap_partials;
  int group_chunks;  // swap path: ring chunks per row group (blockIdx.z)
  int pdl;  // launched with programmatic stream serialization (host side only)
  int f16;  // X, Y and a 16-bit O are fp16 (else bf16)
  // Optional by-product: the gathered LHS.  xcatmap[r] views rows
  // [r*m_pd, (r+1)*m_pd) of the caller's [P*m_pd, k] buffer with the shard
  // maps' box; each X box is stored there once, by the n tile whose share of
  // the k range holds it (swapped tiles: the MMA thread TMA-stores the landed
  // boxes when store_xcat is set; row tiles: the epilogue warps of the
  // KernelKey::store variant copy them from the shards, see xcat below).
  CUtensorMap xcatmap[kMaxShards];
  int store_xcat;
  int y3d;                       // Y [k, n]: one 3-D box per load instead of one 2-D box per 64 columns
  void* xcat;                    // row tiles: the gathered LHS [P*m_pd, k], written by the epilogue warps
  int64_t ldx;                   // its row stride and the shards' in elements (= k)
  const void* xsrc[kMaxShards];  // row tiles: the shards, read by that copy
};

struct GatherParams {
  const uint4* src[kMaxShards];  // shard r, m_pd*k bf16
  uint4* dst;                    // [P*m_pd, k] bf16
  int64_t vec_per_shard;         // m_pd*k*2 / 16
};

// Kernel variant: path, Y storage (true: [n, k] -> K-major tiles), float32
// output, and the row path's n tile (128 or 256; the swap path uses 128).
struct KernelKey {
  int path;
  bool y_kmajor;
  bool out_f32;
  int bn;
  int cm;     // row path: CTAs per cluster along M (two: neighbouring row tiles)
  bool pair;  // cm == 2: one cta_group::2 MMA per pair, each CTA holding half the Y tile
              // (a two-CTA cluster is always a pair; no copy is multicast)
  int atoms = 1;  // swap path: k blocks per pipeline stage (1 or 2)
  bool store = false;  // row path: the variant whose epilogue warps also copy
                       // the X rows to the gathered LHS (agmm_run_gather)
};

// One instantiation of the fused kernel, chosen by select_*_kernel from a key
// (nullptr: no such variant); each group of variants lives in its own
// translation unit (agmm_select_*.cu).
using KernelFn = void (*)(KernelParams);
KernelFn select_swap_kernel(const KernelKey& k);
KernelFn select_rows_kernel_a1(const KernelKey& k);
KernelFn select_rows_kernel_a2(const KernelKey& k);

// Largest dynamic shared memory a CTA may request (227 KiB on sm_100-class parts).
constexpr size_t kMaxDynSmem = 232448;

// Sets the kernel's shared-memory and cluster attributes and reports how many
// clusters of `cluster_x` CTAs can be co-resident (1-CTA clusters: CTAs/SM).
cudaError_t prepare_agmm_kernel(const KernelKey& key, size_t smem_bytes, int cluster_x,
                                int* max_active);

cudaError_t launch_agmm_kernel(const KernelKey& key, const KernelParams& p, dim3 grid,
                               int cluster_x, size_t smem_bytes, bool cooperative,
                               cudaStream_t stream);

cudaError_t launch_gather_kernel(const GatherParams& g, int P, int blocks_per_shard,
                                 cudaStream_t stream);

}  // namespace agmm
