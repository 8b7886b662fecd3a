// agmm_fused_kernel.cuh -- the sm_103a kernel of the fused all-gather matmul,
// instantiated by agmm_select_*.cu (one translation unit per group of
// variants, so that they compile in parallel).
//
//   O = concat_r(X_r) @ Ycan  (tpu_inference "all_gather_matmul.py": the
//   all_gather_matmul docstring, _do_mxu with preferred_element_type=float32,
//   _do_o_local_copy for the output row placement)
//
// One warp-specialised CTA of 6 warps:
//   warp 0      runs the load loop converged; one elected lane issues TMA
//               loads of X chunks (through the per-shard tensor-map table, in
//               ring order) and Y tiles into a multi-stage shared-memory ring
//               guarded by full/empty mbarriers;
//   warp 1      allocates tensor memory and runs the MMA loop converged; one
//               elected lane issues tcgen05.mma (bf16 x bf16 or fp16 x fp16 ->
//               f32 accumulators in TMEM) and tcgen05.commit; on swapped
//               tiles it also TMA-stores the landed X boxes to a gathered-LHS
//               buffer before releasing each stage, when asked;
//   warps 2-5   drain TMEM with tcgen05.ld, round to the output dtype and store
//               each row at its rank-order offset; on row tiles writing the
//               gathered LHS they also copy a share of each tile's X rows to it
//               while the tile's main loop runs (the ring is not involved).
// Issuing from converged warps keeps the copy and MMA operands warp-uniform;
// a loop that a single lane runs alone pays for moving them to uniform
// registers at every issue.  Both loops test the next stage's barrier while
// they issue the current stage.
//
// Two tile orientations:
//   rows path  MMA M = 128 gathered rows (ring-ordered chunks) per CTA, MMA
//              N = n tile; clusters of two CTAs multiply as a cta_group::2
//              pair, each CTA loading and holding half the Y tile (no load is
//              multicast); persistent clusters walk the tile list, TMEM holds
//              two accumulators so the epilogue of one tile overlaps the main
//              loop of the next.
//   swap path  (the whole gathered LHS fits in one MMA N <= 256) MMA M = 128
//              columns of n, MMA N = the gathered rows of one row group; k is
//              split across the CTAs of a thread-block cluster and the float32
//              partials are summed in a fixed rank order (through an
//              L2-resident workspace, or distributed shared memory), so each
//              byte of Y comes from device memory once.
//
// Every mbarrier wait is bounded (KernelParams::wait_limit_cycles).  A wait that
// runs out raises a shared abort flag and records AGMM_ERR_TIMEOUT in the
// status words; all roles then leave their loops, wait (bounded) for their own
// TMA and MMA work in flight, and the CTA frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"
#include "ptx_sm103.cuh"
#include "ring_schedule.h"

namespace agmm {
namespace {

constexpr int kStatusTimeout = 5;  // AGMM_ERR_TIMEOUT

// Offsets inside the control block.
__device__ __forceinline__ uint32_t bar_full(uint32_t ctl, int s) { return ctl + 8u * s; }
__device__ __forceinline__ uint32_t bar_empty(uint32_t ctl, int s) {
  return ctl + 8u * (kMaxStages + s);
}
__device__ __forceinline__ uint32_t bar_acc_full(uint32_t ctl, int a) {
  return ctl + 8u * (2 * kMaxStages + a);
}
__device__ __forceinline__ uint32_t bar_acc_empty(uint32_t ctl, int a) {
  return ctl + 8u * (2 * kMaxStages + 2 + a);
}
__device__ __forceinline__ uint32_t bar_drain(uint32_t ctl) {
  return ctl + 8u * (2 * kMaxStages + 4);
}
// Stream-K hand-offs among the epilogue warps: the owner thread's go-ahead
// (1 arrival) and the contributors' "partial stored" (128 arrivals).
__device__ __forceinline__ uint32_t bar_owner_go(uint32_t ctl) { return ctl + 8u * (2 * kMaxStages + 5); }
__device__ __forceinline__ uint32_t bar_published(uint32_t ctl) { return ctl + 8u * (2 * kMaxStages + 6); }
// Swapped tiles, k splits reduced through distributed shared memory: the
// owner's receive barrier (1 arrival with the expected bytes, then the
// other ranks' bulk copies).
__device__ __forceinline__ uint32_t bar_recv(uint32_t ctl) { return ctl + 8u * (2 * kMaxStages + 7); }
constexpr int kAbortOffset = 8 * (3 * kMaxStages + 8);  // int
constexpr int kTmemOffset = kAbortOffset + 16;          // uint32
constexpr int kChunkTabOffset = 512;                    // int4[kMaxSwapChunks]: shard, src_row, valid, out_row
static_assert(kTmemOffset + 4 <= kChunkTabOffset, "control block overlap");
static_assert(kChunkTabOffset + kMaxSwapChunks * 16 <= kCtlBytes, "control block too small");

enum WaitResult : int { kWaitOk = 1, kWaitTimeout = 0, kWaitAborted = -1 };

// Bounded wait for the phase of `bar` with the given parity.  When `waited`
// is given, the time spent blocked is added to it (trace only).
template <bool kClusterScope = false>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
  if constexpr (kClusterScope)
    return ptx::mbar_try_wait_cluster(bar, parity);
  else
    return ptx::mbar_try_wait(bar, parity);
}

// Suspend-time hint of the waits' retries: a waiting thread sleeps until the
// phase completes or this long passes (the abort flag and the bound are
// checked between sleeps).
constexpr uint32_t kSleepHintNs = 20000;

template <bool kClusterScope = false>
__device__ __forceinline__ bool try_wait_sleep(uint32_t bar, uint32_t parity) {
  if constexpr (kClusterScope)
    return ptx::mbar_try_wait_cluster_sleep(bar, parity, kSleepHintNs);
  else
    return ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs);
}

// The bound is in SM clock cycles (the host converts the time limit at the
// device's peak clock, so a wait lasts at least that long).  The first test
// returns at once; the retries sleep on the barrier rather than poll it.
template <bool kClusterScope = false>
__device__ __forceinline__ int wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_cycles, uint64_t* waited = nullptr) {
  if (try_wait_scoped<kClusterScope>(bar, parity)) return kWaitOk;
  const uint64_t t0 = ptx::clock_cycles();
  for (;;) {
    if (try_wait_sleep<kClusterScope>(bar, parity)) {
      if (waited) *waited += ptx::clock_cycles() - t0;
      return kWaitOk;
    }
    if (*abort) return kWaitAborted;
    if (ptx::clock_cycles() - t0 > limit_cycles) return kWaitTimeout;
  }
}

// Bounded wait that polls with the non-blocking test: for barriers completed
// by another CTA's bulk copies, where a blocked try_wait may wake late.
__device__ __forceinline__ int wait_phase_poll(uint32_t bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_cycles) {
  const uint64_t t0 = ptx::clock_cycles();
  for (int i = 0;; ++i) {
    if (ptx::mbar_test_wait(bar, parity)) return kWaitOk;
    if ((i & 15) == 15) {
      if (*abort) return kWaitAborted;
      if (ptx::clock_cycles() - t0 > limit_cycles) return kWaitTimeout;
    }
  }
}

// Trace slot written by one thread (not lane 0 of each warp).
__device__ __forceinline__ void trace_value(const KernelParams& p, int slot, uint64_t v) {
  if (p.trace != nullptr) p.trace[(size_t)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) * kTraceSlots + slot] = v;
}

// Bounded wait that ignores the abort flag: used to drain work in flight.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_cycles) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::clock_cycles();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (ptx::clock_cycles() - t0 > limit_cycles) return false;
  }
}

__device__ __noinline__ void record_failure(const KernelParams& p, volatile int* abort, int result,
                                            int role, int stage, int tile) {
  *abort = 1;
  if (result == kWaitTimeout && p.status != nullptr) {
    if (atomicCAS(p.status, 0, kStatusTimeout) == 0) {
      p.status[1] = role;
      p.status[2] = stage;
      p.status[3] = tile;
    }
  }
}

// Opt-in device trace: %globaltimer stamps per CTA (16 slots of u64).
__device__ __forceinline__ void trace(const KernelParams& p, int slot) {
  if (p.trace != nullptr && (threadIdx.x & 31) == 0) {
    const uint32_t cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    p.trace[(size_t)cta * kTraceSlots + slot] = ptx::globaltimer_ns();
  }
}

__device__ __forceinline__ uint32_t lane_base_of(uint32_t tmem_base, int warp) {
  return tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
}

// Row-path tile order: ring-ordered row tiles, grouped by group_m so that a
// wave of CTAs shares a band of X rows and sweeps n inside it (L2 reuse).
__device__ __forceinline__ void decode_row_tile(const KernelParams& p, int tile, int& mt, int& nt) {
  const int per_group = p.group_m * p.num_n_tiles;
  const int grp = tile / per_group;
  const int first_m = grp * p.group_m;
  const int gm = min(p.num_mc_tiles - first_m, p.group_m);
  const int r = tile - grp * per_group;
  mt = first_m + r % gm;
  nt = r / gm;
}

enum SegRole : int { kSegWhole = 0, kSegOwner = 1, kSegContrib = 2 };

struct Segment {
  int tile;      // cluster tile
  int mt, nt;    // this CTA's row tile, n tile
  int kb0, kb1;  // k blocks [kb0, kb1)
  int role;      // whole tile, owner of a split tile, or contributor
};

// The rows-path work of one cluster: its contiguous share of the stream-K
// units (see KernelParams) and its data-parallel tiles.  The plain kernel
// takes the shared tiles first (kSkFirst): a stream-K owner's fix-up (waiting
// for its contributors' partials, then summing them) then runs on the
// epilogue warps while the main loop works through the whole tiles, instead
// of ending the launch, and every contributor's share is done early.  The
// variant that also copies the gathered LHS takes its whole tiles first: its
// epilogue warps copy each segment's share of X before draining the segment,
// and behind short stream-K segments that copy would hold up the
// contributors' hand-offs.
struct SegmentIter {
  int cid, nclusters, kblocks, dp_tiles, next_dp;
  int64_t u, hi;

  __device__ __forceinline__ void init(const KernelParams& p, int cluster_id, int clusters) {
    cid = cluster_id;
    nclusters = clusters;
    kblocks = p.num_k_blocks;
    dp_tiles = p.dp_tiles;
    next_dp = cluster_id;
    const int64_t units = (int64_t)(p.num_tiles - p.dp_tiles) * kblocks;
    const int64_t base = (int64_t)p.dp_tiles * kblocks;
    u = base + units * cluster_id / clusters;
    hi = base + units * (cluster_id + 1) / clusters;
  }

  template <bool kSkFirst>
  __device__ __forceinline__ bool next(const KernelParams& p, int cm, int crank, Segment& s) {
    if (u < hi && (kSkFirst || next_dp >= dp_tiles)) {
      const int t = (int)(u / kblocks);
      s.tile = t;
      s.kb0 = (int)(u - (int64_t)t * kblocks);
      const int64_t left = hi - u;
      s.kb1 = (int)min((int64_t)kblocks, (int64_t)s.kb0 + left);
      s.role = (s.kb0 == 0) ? (s.kb1 == kblocks ? kSegWhole : kSegOwner) : kSegContrib;
      u += s.kb1 - s.kb0;
    } else if (next_dp < dp_tiles) {
      s.tile = next_dp;
      s.kb0 = 0;
      s.kb1 = kblocks;
      s.role = kSegWhole;
      next_dp += nclusters;
    } else {
      return false;
    }
    int mc;
    decode_row_tile(p, s.tile, mc, s.nt);
    s.mt = mc * cm + crank;
    return true;
  }
};

// First stream-K unit of cluster c.
__device__ __forceinline__ int64_t sk_first_unit(const KernelParams& p, int c, int clusters) {
  const int64_t units = (int64_t)(p.num_tiles - p.dp_tiles) * p.num_k_blocks;
  return (int64_t)p.dp_tiles * p.num_k_blocks + units * c / clusters;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Two float32 values rounded (to nearest even) to the 16-bit output type:
// bf16, or fp16 when f16.
// Both conversions are computed and one is selected: no branch.
__device__ __forceinline__ uint32_t pack_16x2(float lo, float hi, bool f16) {
  __half2 h = __floats2half2_rn(lo, hi);
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  const uint32_t hu = *reinterpret_cast<uint32_t*>(&h);
  const uint32_t bu = *reinterpret_cast<uint32_t*>(&b);
  return f16 ? hu : bu;
}


// Store 32 consecutive f32 accumulator values of one output row.
template <bool kF32>
__device__ __forceinline__ void store_row32(void* out, int64_t ldo, int64_t row, int64_t col,
                                            const uint32_t (&v)[32], bool f16) {
  if constexpr (kF32) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(out) + row * ldo + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row * ldo + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dst[i] = make_uint4(pack_16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1]), f16),
                          pack_16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3]), f16),
                          pack_16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5]), f16),
                          pack_16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7]), f16));
    }
  }
}

// Swapped tiles: writes output slots [s0, s0 + ns) of this CTA's row group
// (gathered-row slots: chunk c0 + slot / box_rows, row slot % box_rows) for
// the n tile's 128 columns, from float32 sums staged in shared memory as
// stg[slot][128], rounded to the output type, as 16-byte stores along each
// output row.  Threads t = 0..T-1 share the work.
template <bool kF32>
__device__ __forceinline__ void store_slots(const KernelParams& p, const float* stg, int s0, int ns,
                                            const int4* chunk_tab, int c0, int nt, int t, int T) {
  constexpr int kPieces = kF32 ? kTileM / 4 : kTileM / 8;  // 16-byte pieces per 128-column row
  for (int u = t; u < ns * kPieces; u += T) {
    const int sl = u / kPieces;
    const int pc = u - sl * kPieces;
    const int cj = s0 + sl;
    const int4 e = chunk_tab[c0 + (cj >> p.box_shift)];
    const int r = cj & (p.box_rows - 1);
    if (r >= e.z) continue;
    const float* src = stg + (size_t)sl * kTileM;
    const int64_t row = (int64_t)e.w + r;
    const int64_t col = (int64_t)nt * kTileM;
    if constexpr (kF32) {
      const float4 v = *reinterpret_cast<const float4*>(src + pc * 4);
      *reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * p.ldo + col + pc * 4) = v;
    } else {
      const float4 a = *reinterpret_cast<const float4*>(src + pc * 8);
      const float4 b = *reinterpret_cast<const float4*>(src + pc * 8 + 4);
      const bool f16 = p.f16 != 0;
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.ldo + col + pc * 8) =
          make_uint4(pack_16x2(a.x, a.y, f16), pack_16x2(a.z, a.w, f16), pack_16x2(b.x, b.y, f16),
                     pack_16x2(b.z, b.w, f16));
    }
  }
}

// Swap path, device-memory mode: owner `split` of one (n tile, row group)
// sums quads [q0, q0 + items/128) of every rank's slot.  A quad is four
// gathered-row slots of all 128 columns, stored [quad][128 lanes][4 floats].
struct OwnerSlice {
  const float4* gslot;  // rank 0's slot of this (n tile, row group)
  size_t slot_quads;    // quads per rank's slot
  int q0;               // first quad owned
  int items;            // owned (quad, column) pairs
};

// The (quad, column) items are spread over all warps.  Each thread issues
// every rank's 16-byte load for kH items before summing (kH x kS loads in
// flight, at most 24), then adds them in rank order and stages the sums in
// shared memory, stg[slot - 4 * q0][128] (written out by store_slots).
template <int kS>
__device__ __forceinline__ void owner_sum_global(const OwnerSlice& os, float* stg) {
  constexpr int kH = (24 / kS) < 1 ? 1 : ((24 / kS) > 4 ? 4 : (24 / kS));
#pragma unroll 1
  for (int i = threadIdx.x; i < os.items; i += kH * kThreads) {
    float4 part[kH][kS];
#pragma unroll
    for (int h = 0; h < kH; ++h) {
      const int it = i + h * kThreads;
      if (it < os.items) {
        const size_t q = (size_t)(os.q0 + (it >> 7));
        const int t = it & (kTileM - 1);
#pragma unroll
        for (int rk = 0; rk < kS; ++rk) part[h][rk] = __ldcg(os.gslot + ((size_t)rk * os.slot_quads + q) * kTileM + t);
      }
    }
#pragma unroll
    for (int h = 0; h < kH; ++h) {
      const int it = i + h * kThreads;
      if (it < os.items) {
        const int q = os.q0 + (it >> 7);
        const int t = it & (kTileM - 1);
        float4 sum = part[h][0];
#pragma unroll
        for (int rk = 1; rk < kS; ++rk) {
          sum.x += part[h][rk].x;
          sum.y += part[h][rk].y;
          sum.z += part[h][rk].z;
          sum.w += part[h][rk].w;
        }
        float* dst = stg + (size_t)(q - os.q0) * 4 * kTileM + t;
        dst[0] = sum.x;
        dst[kTileM] = sum.y;
        dst[2 * kTileM] = sum.z;
        dst[3 * kTileM] = sum.w;
      }
    }
  }
}

// Swap path, shared-memory mode: the owner's sum of its quads [q0, q0 +
// items/128) over the kS ranks, in rank order, from its own partial (rank
// `split`, send[quad][lane]) and the copies the others sent
// (recv[rank][quad - q0][lane], qmax quads per rank); staged like
// owner_sum_global.  All threads of the CTA share the (quad, lane) items.
template <int kS>
__device__ __forceinline__ void owner_sum_smem(const float4* send, const float4* recv, int qmax, int split, int q0,
                                               int items, float* stg) {
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int q = q0 + (it >> 7);
    const int t = it & (kTileM - 1);
    float4 part[kS];
#pragma unroll
    for (int rk = 0; rk < kS; ++rk)
      part[rk] = rk == split ? send[q * kTileM + t] : recv[(rk * qmax + (q - q0)) * kTileM + t];
    float4 sum = part[0];
#pragma unroll
    for (int rk = 1; rk < kS; ++rk) {
      sum.x += part[rk].x;
      sum.y += part[rk].y;
      sum.z += part[rk].z;
      sum.w += part[rk].w;
    }
    float* dst = stg + (q - q0) * 4 * kTileM + t;
    dst[0] = sum.x;
    dst[kTileM] = sum.y;
    dst[2 * kTileM] = sum.z;
    dst[3 * kTileM] = sum.w;
  }
}

// Row tiles writing the gathered LHS: the epilogue warps (128 threads, t =
// 0..127) copy k blocks [kb_a, kb_b) of row tile mt's X rows from the shards
// to their rows of the gathered LHS, 16 bytes per load and store.  Each n
// tile copies its own share of the k blocks, so every (row, k block) is
// written once; the copy reads the shards directly (mostly from L2, where the
// main loop is streaming the same rows) and never touches the shared-memory
// ring.
__device__ __noinline__ void copy_x_rows(const KernelParams& p, const RingGeom& geom, int mt, int kb_a, int kb_b,
                                         int lane, int t) {
  if (kb_b <= kb_a || mt >= p.num_m_tiles) return;
  const int cpt = kTileM / p.box_rows;
  // lane j < cpt holds chunk j of the row tile (valid 0: none)
  int shard = 0, valid = 0;
  int64_t src_row = 0, out_row = 0;
  if (lane < cpt && (int64_t)mt * cpt + lane < p.total_chunks) {
    const RingChunk ch = ring_chunk(geom, (int64_t)mt * cpt + lane);
    shard = ch.shard;
    valid = ch.valid;
    src_row = ch.src_row;
    out_row = ch.out_row;
  }
  // Warp w copies rows [32w, 32w + 32) of the tile; lane l first resolves row
  // 32w + l (its chunk's shard, source and output rows), then the warp walks
  // the rows kU at a time, each lane taking one 16-byte piece of each row, so
  // that kU loads are in flight per thread without per-piece divisions.
  const int r_mine = (t & ~31) + lane;
  const int j_mine = r_mine >> p.box_shift;
  const int rr_mine = r_mine & (p.box_rows - 1);
  const int sh = __shfl_sync(0xffffffffu, shard, j_mine);
  const int vl = __shfl_sync(0xffffffffu, valid, j_mine);
  const int64_t sr = __shfl_sync(0xffffffffu, src_row, j_mine);
  const int64_t orow = __shfl_sync(0xffffffffu, out_row, j_mine);
  const bool ok_mine = rr_mine < vl;
  const uint16_t* const src_mine =
      static_cast<const uint16_t*>(p.xsrc[sh]) + (sr + rr_mine) * p.ldx + (int64_t)kb_a * kTileK;
  uint16_t* const dst_mine = static_cast<uint16_t*>(p.xcat) + (orow + rr_mine) * p.ldx + (int64_t)kb_a * kTileK;
  const int ppr = (kb_b - kb_a) * (kTileK / 8);  // 16-byte pieces per row
  constexpr int kU = 16;                          // rows (loads) in flight per thread
  for (int pc = lane; pc - lane < ppr; pc += 32) {
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += kU) {
      uint4 v[kU];
      uint16_t* dst[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint16_t* s_ = reinterpret_cast<const uint16_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(src_mine), r0 + u));
        uint16_t* d_ = reinterpret_cast<uint16_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst_mine), r0 + u));
        const bool ok = __shfl_sync(0xffffffffu, ok_mine ? 1 : 0, r0 + u) != 0 && pc < ppr;
        dst[u] = ok ? d_ + (int64_t)pc * 8 : nullptr;
        if (ok) v[u] = __ldg(reinterpret_cast<const uint4*>(s_ + (int64_t)pc * 8));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (dst[u] != nullptr) __stcs(reinterpret_cast<uint4*>(dst[u]), v[u]);  // streaming: not re-read
    }
  }
}

// ----------------------------------------------------------------------------
// The fused kernel.  kPath: kPathRows / kPathSwap.  kYK: Y stored [n, k]
// (K-major tiles); otherwise Y is [k, n] and its tiles are MN-major.  kF32:
// float32 output.  kBN: n tile of the rows path (the swap path uses 128).
// ----------------------------------------------------------------------------
template <int kPath, bool kYK, bool kF32, int kBN, int kCM, bool kPair, int kAtoms, bool kStore>
__global__ void __launch_bounds__(kThreads, 1) agmm_fused_sm103a(const __grid_constant__ KernelParams p) {
  // Clusters exist only as CTA pairs of the rows path: no copy is multicast.
  static_assert(kCM == 1 || (kCM == 2 && kPair), "two-CTA clusters multiply as a CTA pair");
  static_assert(!kPair || (kCM == 2 && kPath == kPathRows), "CTA pairs are clusters of two on the rows path");
  static_assert(kAtoms == 1 || kAtoms == 2, "one or two k blocks per pipeline stage");
  static_assert(!kStore || kPath == kPathRows, "the epilogue's copy of the gathered LHS serves row tiles");
  // The leader's accumulator-release barrier receives the follower's
  // epilogue arrivals (release at cluster scope): its wait acquires at
  // cluster scope.  Stage barriers are fed by TMA and tcgen05.commit.
  constexpr bool kCS = kPair;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int S = p.stages;
  // A stage holds `A` k blocks, each laid out as a one-block stage.  With two
  // per stage the producer and the MMA issuer hand off once per two blocks:
  // their barrier operations cost as much as a block's MMAs at these tile
  // sizes.
  constexpr int A = kAtoms;
  const uint32_t a_slot = (uint32_t)A * kASlotBytes;
  const uint32_t b_slot = (uint32_t)A * p.b_slot_bytes;
  const uint32_t a0 = base;
  const uint32_t b0 = base + (uint32_t)S * a_slot;
  const uint32_t ctl = b0 + (uint32_t)S * b_slot;
  uint8_t* ctl_ptr = base_ptr + (ctl - base);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl_ptr + kAbortOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl_ptr + kTmemOffset);
  int4* chunk_tab = reinterpret_cast<int4*>(ctl_ptr + kChunkTabOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RingGeom geom = make_ring_geom(p.P, p.m_pd, p.my_id, p.box_rows, p.whole_shards);
  const uint64_t limit = p.wait_limit_cycles;

  if (warp == 0) trace(p, 0);
  // The next kernel in the stream may start its prologue on free SMs; it waits
  // (griddepcontrol.wait) for this grid to finish before touching memory.
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
  if (warp == 0) {
    // The lanes of warp 0 initialise one barrier each (lane L: full[L] for L
    // < S, empty[L - S], then the accumulator, drain and hand-off barriers)
    // and each fences its own initialisation; the tensor maps are prefetched
    // by lane as well.
    const int b = lane;
    if (b < S) {
      // a pair: both producers count their bytes on the leader's barrier
      ptx::mbar_init(bar_full(ctl, b), kPair ? 2 : 1);
    } else if (b < 2 * S) {
      // the MMA frees the stage (a pair: the leader's MMA, for both CTAs)
      ptx::mbar_init(bar_empty(ctl, b - S), 1);
    } else if (b < 2 * S + 2) {
      ptx::mbar_init(bar_acc_full(ctl, b - 2 * S), 1);
    } else if (b < 2 * S + 4) {
      // a pair: both CTAs' epilogues drain the accumulator the leader fills
      ptx::mbar_init(bar_acc_empty(ctl, b - 2 * S - 2), kPair ? 256 : 128);
    } else if (b == 2 * S + 4) {
      ptx::mbar_init(bar_drain(ctl), 1);
    } else if (b == 2 * S + 5) {
      ptx::mbar_init(bar_owner_go(ctl), 1);
    } else if (b == 2 * S + 6) {
      ptx::mbar_init(bar_published(ctl), 128);
    } else if (b == 2 * S + 7) {
      ptx::mbar_init(bar_recv(ctl), 1);
    }
    if (lane < p.P) ptx::prefetch_tensormap(&p.xmap[lane]);
    if (lane == 31) ptx::prefetch_tensormap(&p.ymap);
    if (lane == 0) *abort_flag = 0;
    ptx::fence_mbar_init();
    __syncwarp();
    if (lane == 0 && kPath == kPathSwap && p.splits > 1 && p.swap_partials == nullptr) {
      // this owner's quads of each other rank's partial (see the reduction)
      const int gc = min(p.group_chunks, p.total_chunks - (int)blockIdx.z * p.group_chunks);
      const int Q = gc * p.box_rows / 4;
      const int mine = (int)(((int64_t)(blockIdx.x + 1) * Q) / p.splits) - (int)(((int64_t)blockIdx.x * Q) / p.splits);
      ptx::mbar_arrive_expect_tx(bar_recv(ctl), (uint32_t)((p.splits - 1) * mine) * (uint32_t)kTileM * 16u);
    }
  }
  if constexpr (kPath == kPathSwap) {
    // The ring-ordered chunk table, computed once per CTA (each row group of
    // the swap path keeps its chunks of the gathered LHS in one MMA N).
    if (warp == 2 && lane < p.total_chunks) {
      const RingChunk ch = ring_chunk(geom, lane);
      chunk_tab[lane] = make_int4(ch.shard, (int)ch.src_row, ch.valid, (int)ch.out_row);
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), (uint32_t)p.tmem_cols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(tmem_slot), (uint32_t)p.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (kCM > 1) {
    // The pair's MMAs read both CTAs' shared memory and signal both CTAs'
    // barriers: none may do so before every CTA has initialised them.
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait();
  }
  // Swapped tiles reducing their k splits through distributed shared memory:
  // the other ranks copy into this CTA's receive buffer and signal its
  // receive barrier; the matching wait comes before the first such copy.
  const bool swap_bulk = kPath == kPathSwap && p.splits > 1 && p.swap_partials == nullptr;
  if (swap_bulk) ptx::cluster_arrive_relaxed();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touched only shared memory, tensor memory and the
  // parameter block; from here on the previous grid's writes must be visible.
  ptx::griddep_wait();
  if (warp == 0) {
    trace(p, 1);
    if (p.trace != nullptr && lane == 0) {
      const uint32_t cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
      p.trace[(size_t)cta * kTraceSlots + 12] = ptx::smid();
      p.trace[(size_t)cta * kTraceSlots + 13] = ptx::cluster_ctarank();
    }
  }

  // Work of this CTA.  Rows path: tiles blockIdx.x, +gridDim.x, ...
  // Swap path: n tile blockIdx.y, k split blockIdx.x (= rank in the cluster).
  const int swap_nt = (kPath == kPathSwap) ? (int)blockIdx.y : 0;
  const int split = (kPath == kPathSwap) ? (int)blockIdx.x : 0;
  // Swap path row group blockIdx.z: ring chunks [swap_c0, swap_c0 + swap_nch).
  const int swap_c0 = (kPath == kPathSwap) ? (int)blockIdx.z * p.group_chunks : 0;
  const int swap_nch = (kPath == kPathSwap) ? min(p.group_chunks, p.total_chunks - swap_c0) : 0;
  const int swap_cl = (kPath == kPathSwap) ? (int)(blockIdx.z * gridDim.y + blockIdx.y) : 0;  // cluster index
  const int kb_begin = (kPath == kPathSwap) ? (int)((int64_t)split * p.num_k_blocks / p.splits) : 0;
  const int kb_end =
      (kPath == kPathSwap) ? (int)((int64_t)(split + 1) * p.num_k_blocks / p.splits) : p.num_k_blocks;
  const int crank = (kCM > 1) ? (int)(blockIdx.x % kCM) : 0;  // rank in the cluster
  const int cluster_id = (int)(blockIdx.x / kCM);
  const int nclusters = (int)(gridDim.x / kCM);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; one elected lane issues the copies and
    // the barrier arrivals.
    {
      const bool leader = ptx::elect_one();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool dropped = false;
      bool ok = true;
      bool traced_first = false;
      uint64_t waited_empty = 0;
      uint64_t* wait_acc = p.trace ? &waited_empty : nullptr;
      const int cpt = kTileM / p.box_rows;
      SegmentIter iter;
      if constexpr (kPath == kPathRows) iter.init(p, cluster_id, nclusters);
      bool swap_pending = true;
      for (int tile = 0; ok; ++tile) {
        int mt = 0, nt = swap_nt;
        int kb0 = kb_begin, kb1 = kb_end;
        int shard_j[16];
        int row_j[16];
        int nchunks = 0;
        uint32_t bytes;
        if constexpr (kPath == kPathRows) {
          Segment sg;
          if (!iter.template next<!kStore>(p, kCM, crank, sg)) break;
          mt = sg.mt;
          nt = sg.nt;
          kb0 = sg.kb0;
          kb1 = sg.kb1;
          for (int j = 0; j < cpt; ++j) {
            const int64_t gc = (int64_t)mt * cpt + j;
            if (mt < p.num_m_tiles && gc < p.total_chunks) {
              const RingChunk ch = ring_chunk(geom, gc);
              shard_j[nchunks] = ch.shard;
              row_j[nchunks] = (int)ch.src_row;
              ++nchunks;
            }
          }
          // a pair CTA receives only its half of the Y tile
          bytes = (uint32_t)nchunks * p.box_rows * 128u + (uint32_t)(kPair ? kBN / 2 : kBN) * 128u;
        } else {
          if (!swap_pending) break;
          swap_pending = false;
          bytes = (uint32_t)kASlotBytes + (uint32_t)swap_nch * p.box_rows * 128u;
        }
        // One X box per stage (the usual row tile of one 128-row chunk) is
        // kept in registers rather than the chunk arrays.
        const CUtensorMap* xmap0 = (kPath == kPathRows && nchunks > 0) ? &p.xmap[shard_j[0]] : nullptr;
        const int xrow0 = (kPath == kPathRows && nchunks > 0) ? row_j[0] : 0;
        // The next stage's empty barrier is tested while this stage's copies
        // are issued, so its latency is off the loop's critical path.
        bool empty_ready = false;
        for (int kb = kb0; kb < kb1; kb += A) {
          const int na = min(A, kb1 - kb);  // k blocks in this stage
          if (!empty_ready) {
            int res = wait_phase(bar_empty(ctl, stage), phase ^ 1u, abort_flag, limit, wait_acc);
            res = __shfl_sync(0xffffffffu, res, 0);
            if (res != kWaitOk) {
              if (leader) record_failure(p, abort_flag, res, kRoleProducer, stage, tile);
              ok = false;
              break;
            }
          }
          const int next_stage = (stage + 1 == S) ? 0 : stage + 1;
          const uint32_t next_phase = (stage + 1 == S) ? (phase ^ 1u) : phase;
          empty_ready = kb + A < kb1 && ptx::mbar_test_wait(bar_empty(ctl, next_stage), next_phase ^ 1u);
          // A pair follower's copies complete on the leader's barrier.
          const bool to_leader = kPair && crank == 1;
          const uint32_t full = to_leader ? ptx::map_shared_rank(bar_full(ctl, stage), 0) : bar_full(ctl, stage);
          // test hook: the first arrival is dropped, so the MMA thread's wait
          // on this stage runs out
          const bool drop = p.test_drop_first_arrive && !dropped;
          if (drop) dropped = true;
          if (!drop && !to_leader) {
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          if (!drop && leader) {
            if (to_leader)
              ptx::mbar_arrive_expect_tx_remote(full, bytes * (uint32_t)na);
            else
              ptx::mbar_arrive_expect_tx(full, bytes * (uint32_t)na);
            const uint32_t a_dst0 = a0 + (uint32_t)stage * a_slot;
            const uint32_t b_dst0 = b0 + (uint32_t)stage * b_slot;
#pragma unroll
            for (int at = 0; at < A; ++at) {
            if (at >= na) break;
            const uint32_t a_dst = a_dst0 + (uint32_t)at * kASlotBytes;
            const uint32_t b_dst = b_dst0 + (uint32_t)at * p.b_slot_bytes;
            const int k0 = (kb + at) * kTileK;
            if constexpr (kPath == kPathRows) {
              if (nchunks == 1) {
                if (to_leader)
                  ptx::tma_load_2d_pair(a_dst, xmap0, full, k0, xrow0);
                else
                  ptx::tma_load_2d(a_dst, xmap0, full, k0, xrow0);
              } else {
                for (int j = 0; j < nchunks; ++j) {
                  if (to_leader)
                    ptx::tma_load_2d_pair(a_dst + (uint32_t)j * p.box_rows * 128u, &p.xmap[shard_j[j]], full, k0,
                                          row_j[j]);
                  else
                    ptx::tma_load_2d(a_dst + (uint32_t)j * p.box_rows * 128u, &p.xmap[shard_j[j]], full, k0,
                                     row_j[j]);
                }
              }
              if constexpr (kCM == 1) {
                if constexpr (kYK) {
                  ptx::tma_load_2d(b_dst, &p.ymap, full, k0, nt * kBN);
                } else if (p.y3d) {
                  ptx::tma_load_3d(b_dst, &p.ymap, full, 0, k0, nt * (kBN / 64));
                } else {
#pragma unroll
                  for (int a = 0; a < kBN / 64; ++a)
                    ptx::tma_load_2d(b_dst + (uint32_t)a * 8192u, &p.ymap, full, nt * kBN + a * 64, k0);
                }
              } else if constexpr (kPair) {
                // This CTA's half of the Y tile's N rows, into its own slot.
                if constexpr (kYK) {
                  if (to_leader)
                    ptx::tma_load_2d_pair(b_dst, &p.ymap, full, k0, nt * kBN + crank * (kBN / 2));
                  else
                    ptx::tma_load_2d(b_dst, &p.ymap, full, k0, nt * kBN + crank * (kBN / 2));
                } else if (p.y3d) {
                  constexpr int kBoxes = kBN / 64 / 2;
                  if (to_leader)
                    ptx::tma_load_3d_pair(b_dst, &p.ymap, full, 0, k0, nt * (kBN / 64) + crank * kBoxes);
                  else
                    ptx::tma_load_3d(b_dst, &p.ymap, full, 0, k0, nt * (kBN / 64) + crank * kBoxes);
                } else {
                  constexpr int kBoxes = kBN / 64 / 2;
#pragma unroll
                  for (int aa = 0; aa < kBoxes; ++aa) {
                    if (to_leader)
                      ptx::tma_load_2d_pair(b_dst + (uint32_t)aa * 8192u, &p.ymap, full,
                                            nt * kBN + (crank * kBoxes + aa) * 64, k0);
                    else
                      ptx::tma_load_2d(b_dst + (uint32_t)aa * 8192u, &p.ymap, full,
                                       nt * kBN + (crank * kBoxes + aa) * 64, k0);
                  }
                }
              }
            } else {
              if constexpr (kYK) {
                ptx::tma_load_2d(a_dst, &p.ymap, full, k0, nt * kTileM);
              } else if (p.y3d) {
                ptx::tma_load_3d(a_dst, &p.ymap, full, 0, k0, nt * (kTileM / 64));
              } else {
#pragma unroll
                for (int a = 0; a < kTileM / 64; ++a)
                  ptx::tma_load_2d(a_dst + (uint32_t)a * 8192u, &p.ymap, full, nt * kTileM + a * 64, k0);
              }
              const uint32_t chunk_bytes = (uint32_t)p.box_rows * 128u;
              for (int c = 0; c < swap_nch; ++c) {
                const int4 e = chunk_tab[swap_c0 + c];
                ptx::tma_load_2d(b_dst + (uint32_t)c * chunk_bytes, &p.xmap[e.x], full, k0, e.y);
              }
            }
            }  // k blocks of the stage
          }
          if (!traced_first) {
            trace(p, 2);
            traced_first = true;
          }
          stage = next_stage;
          phase = next_phase;
        }
      }
      trace(p, 3);
      if (leader) {
        if (kPath == kPathRows) trace_value(p, 10, waited_empty);
        // Wait for the TMA loads still in flight (only on an abort can a load
        // be unconsumed; a consumed stage's phase has already completed).
        for (int s = 0; s < S; ++s)
          if ((armed >> s) & 1u)
            if (!wait_drain(bar_full(ctl, s), (armed_parity >> s) & 1u, limit))
              record_failure(p, abort_flag, kWaitTimeout, kRoleDrain, s, -1);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (kPair && crank == 1) {
      // Pair follower: the leader's MMA thread works for both CTAs; the
      // follower's copies complete on the leader's stage barriers.
    } else {
      // The whole warp runs the loop; one elected lane issues the MMAs,
      // commits and bulk copies.
      const bool issuer = ptx::elect_one();
      constexpr int kN = (kPath == kPathRows) ? kBN : 0;
      const int mma_n = (kPath == kPathRows) ? kN : p.mma_n;
      // rows path: A = X chunks (K-major), B = Y; swap path: A = Y, B = X chunks.
      const bool a_mn = (kPath == kPathSwap) && !kYK;
      const bool b_mn = (kPath == kPathRows) && !kYK;
      // a pair MMA spans both CTAs' 128 rows: M = 256
      const uint32_t idesc = ptx::idesc_f16kind_f32(kPair ? 2 * kTileM : kTileM, mma_n, a_mn, b_mn, p.f16 != 0);
      constexpr uint16_t kPairMask = 3;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      uint64_t waited_full = 0, waited_accfree = 0;
      uint64_t* wf = p.trace ? &waited_full : nullptr;
      uint64_t* wa = p.trace ? &waited_accfree : nullptr;
      SegmentIter iter;
      if constexpr (kPath == kPathRows) iter.init(p, cluster_id, nclusters);
      const uint32_t chunk_bytes = (uint32_t)p.box_rows * 128u;
      bool stored_any = false;
      for (int tile = 0; ok; ++tile, ++it) {
        int kb0 = kb_begin, kb1 = kb_end;
        // Gathered-LHS by-product: every CTA that loads an X box may store
        // it, so each (X rows, k block) is stored by the one n tile whose
        // share of the k range holds that k block: n tile t stores k blocks
        // [t*K/T, (t+1)*K/T) of its range, and the stores are spread evenly.
        // (row tiles: the store variant's epilogue warps copy it instead)
        bool store = false;
        int st_lo = 0, st_hi = 0;
        if constexpr (kPath == kPathRows) {
          Segment sg;
          if (!iter.template next<!kStore>(p, kCM, crank, sg)) break;
          kb0 = sg.kb0;
          kb1 = sg.kb1;
        } else {
          if (it > 0) break;
          store = p.store_xcat != 0;
          const int span = kb_end - kb_begin;
          st_lo = kb_begin + (int)((int64_t)swap_nt * span / p.num_n_tiles);
          st_hi = kb_begin + (int)((int64_t)(swap_nt + 1) * span / p.num_n_tiles);
        }
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        int res = wait_phase<kCS>(bar_acc_empty(ctl, acc), acc_phase ^ 1u, abort_flag, limit, wa);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res != kWaitOk) {
          if (issuer) record_failure(p, abort_flag, res, kRoleMma, -1, tile);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * mma_n);
        // The next stage's full barrier is tested while this stage's MMAs
        // are issued, so its latency is off the loop's critical path.
        bool full_ready = false;
        for (int kb = kb0; kb < kb1; kb += A) {
          const int na = min(A, kb1 - kb);  // k blocks in this stage
          // (a pair: this barrier also counts the follower's copies)
          if (!full_ready) {
            res = wait_phase(bar_full(ctl, stage), phase, abort_flag, limit, wf);
            res = __shfl_sync(0xffffffffu, res, 0);
            if (res != kWaitOk) {
              if (issuer) record_failure(p, abort_flag, res, kRoleMma, stage, tile);
              ok = false;
              break;
            }
          }
          ptx::tc_fence_after();
          if (it == 0 && kb == kb0) trace(p, 4);
          const uint32_t a_addr0 = a0 + (uint32_t)stage * a_slot;
          const uint32_t b_addr0 = b0 + (uint32_t)stage * b_slot;
          const int next_stage = (stage + 1 == S) ? 0 : stage + 1;
          const uint32_t next_phase = (stage + 1 == S) ? (phase ^ 1u) : phase;
          full_ready = kb + A < kb1 && ptx::mbar_test_wait(bar_full(ctl, next_stage), next_phase);
          bool stored_stage = false;
#pragma unroll
          for (int at = 0; at < A; ++at) {
          if (at >= na) break;
          const int kbb = kb + at;
          const uint32_t a_addr = a_addr0 + (uint32_t)at * kASlotBytes;
          const uint32_t b_addr = b_addr0 + (uint32_t)at * p.b_slot_bytes;
          const bool store_kb = kPath == kPathSwap && store && kbb >= st_lo && kbb < st_hi && issuer;
          if (store_kb) {
            // The landed X boxes go out to the gathered LHS as they are; the
            // per-shard maps clip a box at its shard's last row.
            for (int c = 0; c < swap_nch; ++c) {
              const int4 e = chunk_tab[swap_c0 + c];
              ptx::tma_store_2d(&p.xcatmap[e.x], b_addr + (uint32_t)c * chunk_bytes, kbb * kTileK, e.y);
            }
            ptx::bulk_commit();
            stored_any = true;
            stored_stage = true;
          }
          // K-major operand: the 16-element k step moves 32 bytes inside the
          // 128-byte swizzle row; MN-major operand: it moves 16 rows of 128 B.
          // A descriptor's address field counts 16-byte units.
          const uint64_t a_desc0 =
              a_mn ? ptx::smem_desc_sw128(a_addr, 8192u, 1024u) : ptx::smem_desc_sw128(a_addr, 16u, 1024u);
          const uint64_t b_desc0 =
              b_mn ? ptx::smem_desc_sw128(b_addr, 8192u, 1024u) : ptx::smem_desc_sw128(b_addr, 16u, 1024u);
          const uint64_t a_step = a_mn ? 2048u / 16u : 32u / 16u;
          const uint64_t b_step = b_mn ? 2048u / 16u : 32u / 16u;
          if (issuer) {
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              const uint64_t a_desc = a_desc0 + a_step * (uint64_t)kk;
              const uint64_t b_desc = b_desc0 + b_step * (uint64_t)kk;
              const uint32_t accumulate = (kbb > kb0 || kk > 0) ? 1u : 0u;
              if constexpr (kPair)
                ptx::mma_bf16_pair(d_tmem, a_desc, b_desc, idesc, accumulate);
              else
                ptx::mma_bf16(d_tmem, a_desc, b_desc, idesc, accumulate);
            }
          }
          }  // k blocks of the stage
          if (issuer) {
            // the stores must have read the stage before it is released
            if (stored_stage) ptx::bulk_wait_read_all();
            // frees the stage (a pair: in both CTAs, whose producers fill
            // their halves of it) once these MMAs finish
            if constexpr (kPair)
              ptx::mma_commit_pair(bar_empty(ctl, stage), kPairMask);
            else
              ptx::mma_commit(bar_empty(ctl, stage));
          }
          stage = next_stage;
          phase = next_phase;
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if (issuer) {
          if constexpr (kPair)
            ptx::mma_commit_pair(bar_acc_full(ctl, acc), kPairMask);
          else
            ptx::mma_commit(bar_acc_full(ctl, acc));
        }
      }
      if (issuer) {
        if (stored_any) ptx::bulk_wait_all();
        trace_value(p, 14, waited_full);
        trace_value(p, 15, waited_accfree);
        // Every MMA this thread issued has finished once the drain barrier fires.
        if constexpr (kPair)
          ptx::mma_commit_pair(bar_drain(ctl), kPairMask);
        else
          ptx::mma_commit(bar_drain(ctl));
        if (!wait_drain(bar_drain(ctl), 0, limit))
          record_failure(p, abort_flag, kWaitTimeout, kRoleDrain, -1, -1);
      }
      trace(p, 5);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int trow = q * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    if constexpr (kPath == kPathRows) {
      const int cpt = kTileM / p.box_rows;
      int it = 0;
      uint64_t waited_accfull = 0;
      uint64_t* we = p.trace ? &waited_accfull : nullptr;
      SegmentIter iter;
      iter.init(p, cluster_id, nclusters);
      const size_t slot_floats = (size_t)kTileM * kBN;
      uint32_t owner_parity = 0, publish_parity = 0;
      for (int tile = 0;; ++tile, ++it) {
        Segment sg;
        if (!iter.template next<!kStore>(p, kCM, crank, sg)) break;
        if constexpr (kStore) {
          // while this segment's main loop runs: its share of the gathered LHS
          const int st_lo = (int)((int64_t)sg.nt * p.num_k_blocks / p.num_n_tiles);
          const int st_hi = (int)((int64_t)(sg.nt + 1) * p.num_k_blocks / p.num_n_tiles);
          copy_x_rows(p, geom, sg.mt, max(st_lo, sg.kb0), min(st_hi, sg.kb1), lane, trow);
        }
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        int res = kWaitOk;
        if (lane == 0) res = wait_phase(bar_acc_full(ctl, acc), acc_phase, abort_flag, limit, we);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res != kWaitOk) {
          if (lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, acc, tile);
          break;
        }
        ptx::tc_fence_after();
        if (it == 0) trace(p, 6);
        const int64_t gc = (int64_t)sg.mt * cpt + trow / p.box_rows;
        const int r = trow % p.box_rows;
        int64_t out_row = -1;
        if (sg.mt < p.num_m_tiles && gc < p.total_chunks) {
          const RingChunk ch = ring_chunk(geom, gc);
          if (r < ch.valid) out_row = ch.out_row + r;
        }
        const uint32_t tbase = lane_base + (uint32_t)(acc * kBN);
        // Contributors of an owned tile: the following clusters whose first
        // stream-K unit falls inside this tile, in k order.
        int ncontrib = 0;
        if (sg.role == kSegOwner) {
          const int64_t tile_end = (int64_t)(sg.tile + 1) * p.num_k_blocks;
          while (cluster_id + 1 + ncontrib < nclusters &&
                 sk_first_unit(p, cluster_id + 1 + ncontrib, nclusters) < tile_end)
            ++ncontrib;
          if (threadIdx.x == 64) {
            int wres = kWaitOk;
            const int* flag = p.sk_flags + (size_t)(sg.tile - p.dp_tiles) * kCM + crank;
            const uint64_t t0 = ptx::clock_cycles();
            while (ld_acquire_gpu(flag) < ncontrib) {
              if (*abort_flag) { wres = kWaitAborted; break; }
              if (ptx::clock_cycles() - t0 > limit) { wres = kWaitTimeout; break; }
              __nanosleep(32);
            }
            if (wres == kWaitOk) {
              *const_cast<volatile int*>(flag) = 0;  // ready for the next run
            } else {
              record_failure(p, abort_flag, wres, kRoleEpilogue, -2, sg.tile);
              if (wres == kWaitTimeout && p.status != nullptr && p.status[3] == sg.tile) {
                p.status[4] = ncontrib;
                p.status[5] = ld_acquire_gpu(flag);
                p.status[6] = cluster_id;
                p.status[7] = crank;
              }
            }
            ptx::mbar_arrive(bar_owner_go(ctl));  // release the other epilogue threads either way
          }
          __syncwarp();
          int gres = kWaitOk;
          if (lane == 0) gres = wait_phase(bar_owner_go(ctl), owner_parity, abort_flag, limit);
          gres = __shfl_sync(0xffffffffu, gres, 0);
          owner_parity ^= 1u;
          if (gres != kWaitOk && lane == 0) record_failure(p, abort_flag, gres, kRoleEpilogue, -3, sg.tile);
        }
        // Partial slot layout [BN/32][8][128 rows][4 floats]: a warp's 16-byte
        // accesses cover 512 contiguous bytes.
        float4* my_slot = (sg.role == kSegContrib)
                              ? reinterpret_cast<float4*>(p.sk_partials + ((size_t)cluster_id * kCM + crank) * slot_floats)
                              : nullptr;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
          ptx::tmem_ld_wait();
          if (c == kBN / 32 - 1) {
            ptx::tc_fence_before();
            // TMEM buffer may be reused (a pair's leader refills both CTAs')
            if (kPair && crank == 1)
              ptx::mbar_arrive_remote(ptx::map_shared_rank(bar_acc_empty(ctl, acc), 0));
            else
              ptx::mbar_arrive(bar_acc_empty(ctl, acc));
          }
          if (sg.role == kSegContrib) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              my_slot[((size_t)c * 8 + i) * kTileM + trow] =
                  make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                              __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            continue;
          }
          // Owner: own partial + contributor 1 + contributor 2 + ... (k order);
          // two contributors' loads are in flight together.
          for (int j = 0; j < ncontrib; j += 2) {
            const float4* s0 = reinterpret_cast<const float4*>(
                p.sk_partials + ((size_t)(cluster_id + 1 + j) * kCM + crank) * slot_floats);
            const float4* s1 = reinterpret_cast<const float4*>(
                p.sk_partials + ((size_t)(cluster_id + 2 + j) * kCM + crank) * slot_floats);
            float4 q0[8], q1[8];
            const bool two = j + 1 < ncontrib;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              q0[i] = __ldcg(s0 + ((size_t)c * 8 + i) * kTileM + trow);
              if (two) q1[i] = __ldcg(s1 + ((size_t)c * 8 + i) * kTileM + trow);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) + q0[i].x);
              v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + q0[i].y);
              v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + q0[i].z);
              v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + q0[i].w);
            }
            if (two) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) + q1[i].x);
                v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + q1[i].y);
                v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + q1[i].z);
                v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + q1[i].w);
              }
            }
          }
          if (out_row >= 0) store_row32<kF32>(p.out, p.ldo, out_row, (int64_t)sg.nt * kBN + c * 32, v, p.f16 != 0);
        }
        if (sg.role == kSegContrib) {
          // Publish: every thread fences its stores and arrives; one thread
          // waits for all 128 and counts the partial for the owner.
          __threadfence();
          ptx::mbar_arrive(bar_published(ctl));
          if (threadIdx.x == 64) {
            const int pres = wait_phase(bar_published(ctl), publish_parity, abort_flag, limit);
            if (pres == kWaitOk)
              atomicAdd(p.sk_flags + (size_t)(sg.tile - p.dp_tiles) * kCM + crank, 1);
            else
              record_failure(p, abort_flag, pres, kRoleEpilogue, -4, sg.tile);
          }
          publish_parity ^= 1u;
        }
      }
      trace(p, 7);
      if (warp == 2 && lane == 0) trace_value(p, 9, waited_accfull);
    } else {
      // Swap path: wait for this CTA's float32 partial [n 128][row slots].
      int res = kWaitOk;
      if (lane == 0) res = wait_phase(bar_acc_full(ctl, 0), 0, abort_flag, limit);
      res = __shfl_sync(0xffffffffu, res, 0);
      if (res != kWaitOk) {
        if (lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, 0, swap_nt);
      } else {
        ptx::tc_fence_after();
        trace(p, 6);
      }
    }
  }

  if constexpr (kPath == kPathSwap) {
    // Reduction of the k splits of this CTA's (n tile, row group).  The
    // accumulator holds 128 n columns (TMEM lanes) x ncols gathered-row slots
    // (TMEM columns): chunks c0.. of the ring-ordered chunk table, box_rows
    // slots each.  A quad is 4 slots of all 128 lanes ([lane][4 floats], 2
    // KiB); owner o (rank o of the cluster) sums quads [o*Q/S, (o+1)*Q/S) of
    // every rank's partial in rank order, so every output element has one
    // fixed reduction order whatever the route.
    //   one split:      the CTA stores its accumulator directly;
    //   device memory:  each rank stores its partial to its own slot in an
    //                   L2-resident workspace with coalesced 16-byte stores;
    //                   a cluster barrier (release/acquire) orders them
    //                   before the owners' loads;
    //   shared memory:  each rank drains its partial into its own pipeline
    //                   memory (idle after its main loop), then bulk-copies
    //                   owner o's quads into slot [rank] of owner o's receive
    //                   buffer (past the control block), counted on o's
    //                   receive barrier; owners wait only for their bytes, so
    //                   early ranks' copies land while late ranks still work.
    const int ncols = swap_nch * p.box_rows;
    const int S = p.splits;
    const int groups = (ncols + 15) >> 4;
    const int Q = ncols >> 2;
    const int q_lo = (int)(((int64_t)split * Q) / S);
    const int q_hi = (int)(((int64_t)(split + 1) * Q) / S);
    // Slot size of the device-memory mode: the widest row group's columns.
    const int slot_groups = (p.group_chunks * p.box_rows + 15) >> 4;
    const size_t slot_quads = (size_t)slot_groups * 4;
    const bool global_mode = S > 1 && p.swap_partials != nullptr;
    constexpr uint32_t kQuadBytes = (uint32_t)kTileM * 16u;
    float4* gslot = global_mode ? reinterpret_cast<float4*>(p.swap_partials) +
                                      ((size_t)swap_cl * S) * slot_quads * kTileM
                                : nullptr;
    const int tl = (warp & 3) * 32 + lane;  // epilogue thread: TMEM lane = n column
    __syncwarp();
    trace(p, 8);
    // staged sums, [slot][128 columns] float32 (pipeline memory, idle now)
    float* const stg = reinterpret_cast<float*>(base_ptr);
    if (S == 1) {
      if (warp >= 2) {
        if (!*abort_flag) {
          const uint32_t tbase = lane_base_of(tmem_base, warp);
#pragma unroll 1
          for (int g = 0; g < groups; ++g) {
            uint32_t v[16];
            ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 16), v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (g * 16 + i < ncols) stg[(size_t)(g * 16 + i) * kTileM + tl] = __uint_as_float(v[i]);
          }
          ptx::tc_fence_before();
        }
        // the four epilogue warps' slots staged (every thread arrives, also
        // on an abort, so the bounded wait below cannot be stranded)
        ptx::mbar_arrive(bar_published(ctl));
        int res = kWaitOk;
        if (lane == 0) res = wait_phase(bar_published(ctl), 0, abort_flag, limit);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res == kWaitOk && !*abort_flag)
          store_slots<kF32>(p, stg, 0, ncols, chunk_tab, swap_c0, swap_nt, tl, kTileM);
      }
    } else if (global_mode) {
      if (warp >= 2) {
        float4* mine = gslot + (size_t)split * slot_quads * kTileM + tl;
        const uint32_t tbase = lane_base_of(tmem_base, warp);
#pragma unroll 1
        for (int g = 0; g < groups; g += 2) {
          uint32_t v[2][16];
          ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 16), v[0]);
          if (g + 1 < groups) ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)((g + 1) * 16), v[1]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (g + h < groups) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                mine[((size_t)(g + h) * 4 + q4) * kTileM] =
                    make_float4(__uint_as_float(v[h][4 * q4]), __uint_as_float(v[h][4 * q4 + 1]),
                                __uint_as_float(v[h][4 * q4 + 2]), __uint_as_float(v[h][4 * q4 + 3]));
            }
          }
        }
        ptx::tc_fence_before();
      }
      __syncwarp();
      ptx::cluster_sync_all();  // partials delivered
      trace(p, 9);
      // one decision for the whole CTA, so the barrier below is reached by all
      if (__syncthreads_or(*abort_flag) == 0) {
        const OwnerSlice os{gslot, slot_quads, q_lo, (q_hi - q_lo) * kTileM};
        switch (S) {
#define AGMM_OWNER_CASE(N) \
  case N:                  \
    owner_sum_global<N>(os, stg); \
    break;
          AGMM_OWNER_CASE(2) AGMM_OWNER_CASE(3) AGMM_OWNER_CASE(4) AGMM_OWNER_CASE(5) AGMM_OWNER_CASE(6)
          AGMM_OWNER_CASE(7) AGMM_OWNER_CASE(8) AGMM_OWNER_CASE(9) AGMM_OWNER_CASE(10) AGMM_OWNER_CASE(11)
          AGMM_OWNER_CASE(12) AGMM_OWNER_CASE(13) AGMM_OWNER_CASE(14) AGMM_OWNER_CASE(15) AGMM_OWNER_CASE(16)
#undef AGMM_OWNER_CASE
          default:
            break;
        }
        __syncthreads();
        store_slots<kF32>(p, stg, q_lo * 4, (q_hi - q_lo) * 4, chunk_tab, swap_c0, swap_nt, threadIdx.x, kThreads);
      }
    } else {
      // shared-memory mode: send buffer [quad][lane][16 B] at the start of
      // the pipeline memory, receive buffer [rank][qmax quads][lane][16 B]
      // past the control block
      const int qmax = (Q + S - 1) / S;
      const uint32_t send = base;
      const uint32_t recv = ctl + (uint32_t)kCtlBytes;
      if (warp >= 2) {
        if (!*abort_flag) {
          const uint32_t tbase = lane_base_of(tmem_base, warp);
          const uint32_t lane_off = (uint32_t)tl * 16u;
#pragma unroll 1
          for (int g = 0; g < groups; g += 2) {
            uint32_t v[2][16];
            ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 16), v[0]);
            if (g + 1 < groups) ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)((g + 1) * 16), v[1]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const int q = (g + h) * 4 + q4;
                if (g + h < groups && q < Q)
                  ptx::st_shared_v4(send + (uint32_t)q * kQuadBytes + lane_off, v[h][4 * q4], v[h][4 * q4 + 1],
                                    v[h][4 * q4 + 2], v[h][4 * q4 + 3]);
              }
            }
          }
          ptx::tc_fence_before();
        }
        // the bulk copies read what the generic stores wrote
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar_published(ctl));
      }
      __syncwarp();
      // every owner has initialised its receive barrier
      ptx::cluster_wait();
      trace(p, 9);
      if (warp == 2) {
        int res = kWaitOk;
        if (lane == 0) res = wait_phase_poll(bar_published(ctl), 0, abort_flag, limit);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res != kWaitOk) {
          if (lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, -5, swap_nt);
        } else if (!*abort_flag && ptx::elect_one()) {
          for (int o = 0; o < S; ++o) {
            const int lo = (int)(((int64_t)o * Q) / S);
            const int hi = (int)(((int64_t)(o + 1) * Q) / S);
            if (o == split || hi <= lo) continue;
            ptx::bulk_copy_to_cluster(ptx::map_shared_rank(recv + (uint32_t)(split * qmax) * kQuadBytes, (uint32_t)o),
                                      send + (uint32_t)lo * kQuadBytes, (uint32_t)(hi - lo) * kQuadBytes,
                                      ptx::map_shared_rank(bar_recv(ctl), (uint32_t)o));
          }
        }
        __syncwarp();
      }
      {
        // every warp waits for this owner's bytes, then all threads sum
        int res = kWaitOk;
        if (lane == 0) res = wait_phase_poll(bar_recv(ctl), 0, abort_flag, limit);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res != kWaitOk && lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, -6, swap_nt);
        // one decision for the whole CTA, so the barrier below is reached by all
        if (__syncthreads_or(*abort_flag) == 0) {
          // sums staged in this CTA's own (unused) receive slot, [slot][128]
          const float4* const sendv = reinterpret_cast<const float4*>(base_ptr);
          const float4* const recvv = reinterpret_cast<const float4*>(base_ptr + (recv - base));
          float* const own = reinterpret_cast<float*>(base_ptr + (recv - base)) + (size_t)split * qmax * 4 * kTileM;
          const int items = (q_hi - q_lo) * kTileM;
          switch (S) {
#define AGMM_OWNER_CASE(N) \
  case N:                  \
    owner_sum_smem<N>(sendv, recvv, qmax, split, q_lo, items, own); \
    break;
            AGMM_OWNER_CASE(2) AGMM_OWNER_CASE(3) AGMM_OWNER_CASE(4) AGMM_OWNER_CASE(5) AGMM_OWNER_CASE(6)
            AGMM_OWNER_CASE(7) AGMM_OWNER_CASE(8) AGMM_OWNER_CASE(9) AGMM_OWNER_CASE(10) AGMM_OWNER_CASE(11)
            AGMM_OWNER_CASE(12) AGMM_OWNER_CASE(13) AGMM_OWNER_CASE(14) AGMM_OWNER_CASE(15) AGMM_OWNER_CASE(16)
#undef AGMM_OWNER_CASE
            default:
              break;
          }
          __syncthreads();
          store_slots<kF32>(p, own, q_lo * 4, (q_hi - q_lo) * 4, chunk_tab, swap_c0, swap_nt, threadIdx.x, kThreads);
        }
      }
      __syncwarp();
      // No CTA leaves while copies out of or into its shared memory may run:
      // each arrives once its own bytes are in (relaxed: it publishes no
      // memory through this barrier).
      ptx::cluster_arrive_relaxed();
      ptx::cluster_wait();
    }
    trace(p, 10);
  }

  if constexpr (kPath == kPathRows && kCM > 1) {
    // The pair leader's MMAs read this CTA's shared memory and its commits
    // arrive on this CTA's barriers until the last one: leave only after both
    // CTAs have drained.
    __syncwarp();
    ptx::cluster_sync_all();
  }
  __syncthreads();
  if (warp == 0) trace(p, 11);
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (kPair)
      ptx::tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
    else
      ptx::tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
}

}  // namespace
}  // namespace agmm

// Pointer to one instantiation of the fused kernel for a kernel key (the
// key's y_kmajor and out_f32 pick among the four layouts of a variant).
#define AGMM_FUSED_PICK(PATH, BN, CM, PAIR, AT, ST)                                                   \
  (k.y_kmajor ? (k.out_f32 ? &agmm_fused_sm103a<PATH, true, true, BN, CM, PAIR, AT, ST>                \
                           : &agmm_fused_sm103a<PATH, true, false, BN, CM, PAIR, AT, ST>)              \
              : (k.out_f32 ? &agmm_fused_sm103a<PATH, false, true, BN, CM, PAIR, AT, ST>               \
                           : &agmm_fused_sm103a<PATH, false, false, BN, CM, PAIR, AT, ST>))
