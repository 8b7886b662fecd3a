// agmm_kernels.cu -- sm_103a kernels of the fused all-gather matmul.
//
//   O = concat_r(X_r) @ Ycan  (tpu_inference "all_gather_matmul.py": the
//   all_gather_matmul docstring, _do_mxu with preferred_element_type=float32,
//   _do_o_local_copy for the output row placement)
//
// One warp-specialised CTA of 6 warps:
//   warp 0      one elected thread issues TMA loads of X chunks (through the
//               per-shard tensor-map table, in ring order) and Y tiles into a
//               multi-stage shared-memory ring guarded by full/empty mbarriers;
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma
//               (bf16 x bf16 -> f32 accumulators in TMEM) and tcgen05.commit;
//   warps 2-5   drain TMEM with tcgen05.ld, round to the output dtype and store
//               each row at its rank-order offset.
//
// Two tile orientations:
//   rows path  MMA M = 128 gathered rows (ring-ordered chunks), MMA N = n tile;
//              persistent CTAs walk the tile list, TMEM holds two accumulators
//              so the epilogue of one tile overlaps the main loop of the next.
//   swap path  (the whole gathered LHS fits in one MMA N <= 256) MMA M = 128
//              columns of n, MMA N = every gathered row; k is split across the
//              CTAs of a thread-block cluster and the float32 partials are
//              summed in a fixed rank order through distributed shared memory,
//              so Y is read from device memory exactly once.
//
// Every mbarrier wait is bounded (KernelParams::wait_limit_ns).  A wait that
// runs out raises a shared abort flag and records AGMM_ERR_TIMEOUT in the
// status words; all roles then leave their loops, wait (bounded) for their own
// TMA and MMA work in flight, and the CTA frees its tensor memory and returns.
#include <cuda_bf16.h>

#include "kernel_params.h"
#include "ptx_sm103.cuh"
#include "ring_schedule.h"

namespace agmm {
namespace {

constexpr int kCtlBytes = 256;  // barriers + flags after the stage slots
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
constexpr int kAbortOffset = 8 * (2 * kMaxStages + 5);  // int
constexpr int kTmemOffset = kAbortOffset + 16;          // uint32

enum WaitResult : int { kWaitOk = 1, kWaitTimeout = 0, kWaitAborted = -1 };

// Bounded wait for the phase of `bar` with the given parity.
__device__ __forceinline__ int wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return kWaitOk;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return kWaitOk;
    if ((it & 15u) == 0u) {
      if (*abort) return kWaitAborted;
      if (ptx::globaltimer_ns() - t0 > limit_ns) return kWaitTimeout;
    }
  }
}

// Bounded wait that ignores the abort flag: used to drain work in flight.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u && ptx::globaltimer_ns() - t0 > limit_ns) return false;
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

// Row-path tile order: ring-ordered row tiles, grouped by group_m so that a
// wave of CTAs shares a band of X rows and sweeps n inside it (L2 reuse).
__device__ __forceinline__ void decode_row_tile(const KernelParams& p, int tile, int& mt, int& nt) {
  const int per_group = p.group_m * p.num_n_tiles;
  const int grp = tile / per_group;
  const int first_m = grp * p.group_m;
  const int gm = min(p.num_m_tiles - first_m, p.group_m);
  const int r = tile - grp * per_group;
  mt = first_m + r % gm;
  nt = r / gm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store 32 consecutive f32 accumulator values of one output row.
template <bool kF32>
__device__ __forceinline__ void store_row32(void* out, int64_t ldo, int64_t row, int64_t col,
                                            const uint32_t (&v)[32]) {
  if constexpr (kF32) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(out) + row * ldo + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * ldo + col);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dst[i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i + 0]), __uint_as_float(v[8 * i + 1])),
                          pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                          pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                          pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
    }
  }
}

// Store 4 consecutive values of one output row.
template <bool kF32>
__device__ __forceinline__ void store_row4(void* out, int64_t ldo, int64_t row, int64_t col,
                                           float4 s) {
  if constexpr (kF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + row * ldo + col) = s;
  } else {
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + row * ldo + col) =
        make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
  }
}

// ----------------------------------------------------------------------------
// The fused kernel.  kPath: kPathRows / kPathSwap.  kYK: Y stored [n, k]
// (K-major tiles); otherwise Y is [k, n] and its tiles are MN-major.  kF32:
// float32 output.  kBN: n tile of the rows path (the swap path uses 128).
// ----------------------------------------------------------------------------
template <int kPath, bool kYK, bool kF32, int kBN>
__global__ void __launch_bounds__(kThreads, 1) agmm_fused_sm103a(const __grid_constant__ KernelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int S = p.stages;
  const uint32_t a0 = base;
  const uint32_t b0 = base + (uint32_t)S * kASlotBytes;
  const uint32_t ctl = b0 + (uint32_t)S * p.b_slot_bytes;
  uint8_t* ctl_ptr = base_ptr + (ctl - base);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl_ptr + kAbortOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl_ptr + kTmemOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RingGeom geom = make_ring_geom(p.P, p.m_pd, p.my_id, p.box_rows);
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar_full(ctl, s), 1);
      ptx::mbar_init(bar_empty(ctl, s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar_acc_full(ctl, a), 1);
      ptx::mbar_init(bar_acc_empty(ctl, a), 128);
    }
    ptx::mbar_init(bar_drain(ctl), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int r = 0; r < p.P; ++r) ptx::prefetch_tensormap(&p.xmap[r]);
    ptx::prefetch_tensormap(&p.ymap);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), (uint32_t)p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Work of this CTA.  Rows path: tiles blockIdx.x, +gridDim.x, ...
  // Swap path: n tile blockIdx.y, k split blockIdx.x (= rank in the cluster).
  const int swap_nt = (kPath == kPathSwap) ? (int)blockIdx.y : 0;
  const int split = (kPath == kPathSwap) ? (int)blockIdx.x : 0;
  const int kb_begin = (kPath == kPathSwap) ? (int)((int64_t)split * p.num_k_blocks / p.splits) : 0;
  const int kb_end =
      (kPath == kPathSwap) ? (int)((int64_t)(split + 1) * p.num_k_blocks / p.splits) : p.num_k_blocks;
  const int tile_first = (kPath == kPathSwap) ? 0 : (int)blockIdx.x;
  const int tile_step = (kPath == kPathSwap) ? 1 : (int)gridDim.x;
  const int tile_count = (kPath == kPathSwap) ? 1 : p.num_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool dropped = false;
      bool ok = true;
      const int cpt = kTileM / p.box_rows;
      for (int tile = tile_first; ok && tile < tile_count; tile += tile_step) {
        int mt = 0, nt = swap_nt;
        int shard_j[16];
        int row_j[16];
        int nchunks = 0;
        uint32_t bytes;
        if constexpr (kPath == kPathRows) {
          decode_row_tile(p, tile, mt, nt);
          for (int j = 0; j < cpt; ++j) {
            const int64_t gc = (int64_t)mt * cpt + j;
            if (gc < p.total_chunks) {
              const RingChunk ch = ring_chunk(geom, gc);
              shard_j[nchunks] = ch.shard;
              row_j[nchunks] = (int)ch.src_row;
              ++nchunks;
            }
          }
          bytes = (uint32_t)nchunks * p.box_rows * 128u + (uint32_t)kBN * 128u;
        } else {
          bytes = (uint32_t)kASlotBytes + (uint32_t)p.total_chunks * p.box_rows * 128u;
        }
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          const int res = wait_phase(bar_empty(ctl, stage), phase ^ 1u, abort_flag, limit);
          if (res != kWaitOk) {
            record_failure(p, abort_flag, res, kRoleProducer, stage, tile);
            ok = false;
            break;
          }
          const uint32_t full = bar_full(ctl, stage);
          if (p.test_drop_first_arrive && !dropped) {
            dropped = true;  // the MMA thread's wait on this stage runs out
          } else {
            ptx::mbar_arrive_expect_tx(full, bytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            const uint32_t a_dst = a0 + (uint32_t)stage * kASlotBytes;
            const uint32_t b_dst = b0 + (uint32_t)stage * p.b_slot_bytes;
            const int k0 = kb * kTileK;
            if constexpr (kPath == kPathRows) {
              for (int j = 0; j < nchunks; ++j)
                ptx::tma_load_2d(a_dst + (uint32_t)j * p.box_rows * 128u, &p.xmap[shard_j[j]], full,
                                 k0, row_j[j]);
              if constexpr (kYK) {
                ptx::tma_load_2d(b_dst, &p.ymap, full, k0, nt * kBN);
              } else {
#pragma unroll
                for (int a = 0; a < kBN / 64; ++a)
                  ptx::tma_load_2d(b_dst + (uint32_t)a * 8192u, &p.ymap, full, nt * kBN + a * 64, k0);
              }
            } else {
              if constexpr (kYK) {
                ptx::tma_load_2d(a_dst, &p.ymap, full, k0, nt * kTileM);
              } else {
#pragma unroll
                for (int a = 0; a < kTileM / 64; ++a)
                  ptx::tma_load_2d(a_dst + (uint32_t)a * 8192u, &p.ymap, full, nt * kTileM + a * 64, k0);
              }
              for (int c = 0; c < p.total_chunks; ++c) {
                const RingChunk ch = ring_chunk(geom, c);
                ptx::tma_load_2d(b_dst + (uint32_t)c * p.box_rows * 128u, &p.xmap[ch.shard], full, k0,
                                 (int)ch.src_row);
              }
            }
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wait for this thread's TMA loads still in flight (only on an abort can
      // a load be unconsumed; a consumed stage's phase has already completed).
      for (int s = 0; s < S; ++s)
        if ((armed >> s) & 1u)
          if (!wait_drain(bar_full(ctl, s), (armed_parity >> s) & 1u, limit))
            record_failure(p, abort_flag, kWaitTimeout, kRoleDrain, s, -1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr int kN = (kPath == kPathRows) ? kBN : 0;
      const int mma_n = (kPath == kPathRows) ? kN : p.mma_n;
      // rows path: A = X chunks (K-major), B = Y; swap path: A = Y, B = X chunks.
      const bool a_mn = (kPath == kPathSwap) && !kYK;
      const bool b_mn = (kPath == kPathRows) && !kYK;
      const uint32_t idesc = ptx::idesc_bf16_f32(kTileM, mma_n, a_mn, b_mn);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int tile = tile_first; ok && tile < tile_count; tile += tile_step, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        int res = wait_phase(bar_acc_empty(ctl, acc), acc_phase ^ 1u, abort_flag, limit);
        if (res != kWaitOk) {
          record_failure(p, abort_flag, res, kRoleMma, -1, tile);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * mma_n);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          res = wait_phase(bar_full(ctl, stage), phase, abort_flag, limit);
          if (res != kWaitOk) {
            record_failure(p, abort_flag, res, kRoleMma, stage, tile);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = a0 + (uint32_t)stage * kASlotBytes;
          const uint32_t b_addr = b0 + (uint32_t)stage * p.b_slot_bytes;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk) {
            // K-major operand: the 16-element k step moves 32 bytes inside the
            // 128-byte swizzle row; MN-major operand: it moves 16 rows of 128 B.
            const uint64_t a_desc =
                a_mn ? ptx::smem_desc_sw128(a_addr + kk * 2048u, 8192u, 1024u)
                     : ptx::smem_desc_sw128(a_addr + kk * 32u, 16u, 1024u);
            const uint64_t b_desc =
                b_mn ? ptx::smem_desc_sw128(b_addr + kk * 2048u, 8192u, 1024u)
                     : ptx::smem_desc_sw128(b_addr + kk * 32u, 16u, 1024u);
            ptx::mma_bf16(d_tmem, a_desc, b_desc, idesc, (kb > kb_begin || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(bar_empty(ctl, stage));  // frees the stage once these MMAs finish
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(bar_acc_full(ctl, acc));  // accumulator ready for the epilogue
      }
      // Every MMA this thread issued has finished once the drain barrier fires.
      ptx::mma_commit(bar_drain(ctl));
      if (!wait_drain(bar_drain(ctl), 0, limit))
        record_failure(p, abort_flag, kWaitTimeout, kRoleDrain, -1, -1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int trow = q * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    if constexpr (kPath == kPathRows) {
      const int cpt = kTileM / p.box_rows;
      int it = 0;
      for (int tile = tile_first; tile < tile_count; tile += tile_step, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        int res = kWaitOk;
        if (lane == 0) res = wait_phase(bar_acc_full(ctl, acc), acc_phase, abort_flag, limit);
        res = __shfl_sync(0xffffffffu, res, 0);
        if (res != kWaitOk) {
          if (lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, acc, tile);
          break;
        }
        ptx::tc_fence_after();
        int mt, nt;
        decode_row_tile(p, tile, mt, nt);
        const int64_t gc = (int64_t)mt * cpt + trow / p.box_rows;
        const int r = trow % p.box_rows;
        int64_t out_row = -1;
        if (gc < p.total_chunks) {
          const RingChunk ch = ring_chunk(geom, gc);
          if (r < ch.valid) out_row = ch.out_row + r;
        }
        const uint32_t tbase = lane_base + (uint32_t)(acc * kBN);
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(c * 32), v);
          ptx::tmem_ld_wait();
          if (c == kBN / 32 - 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_acc_empty(ctl, acc));  // TMEM buffer may be reused
          }
          if (out_row >= 0) store_row32<kF32>(p.out, p.ldo, out_row, (int64_t)nt * kBN + c * 32, v);
        }
      }
    } else {
      // Swap path, part 1: this CTA's float32 partial [n 128][rows mma_n] goes
      // from TMEM into shared memory as red[col][128] (col = gathered-row slot).
      int res = kWaitOk;
      if (lane == 0) res = wait_phase(bar_acc_full(ctl, 0), 0, abort_flag, limit);
      res = __shfl_sync(0xffffffffu, res, 0);
      if (res != kWaitOk) {
        if (lane == 0) record_failure(p, abort_flag, res, kRoleEpilogue, 0, swap_nt);
      } else {
        ptx::tc_fence_after();
        float* red = reinterpret_cast<float*>(base_ptr);
#pragma unroll 1
        for (int cb = 0; cb < p.mma_n / 32; ++cb) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(lane_base + (uint32_t)(cb * 32), v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) red[(cb * 32 + i) * kTileM + trow] = __uint_as_float(v[i]);
        }
        ptx::tc_fence_before();
      }
    }
  }

  if constexpr (kPath == kPathSwap) {
    // Part 2: rank `split` of the cluster owns gathered-row slots [c0, c1) and
    // sums every rank's partial for them in rank order 0..splits-1.
    __syncwarp();
    if (p.splits > 1) ptx::cluster_sync_all(); else __syncthreads();
    if (warp >= 2 && !*abort_flag) {
      const int tid = threadIdx.x - 64;
      const int lane4 = (tid & 31) * 4;
      const int ncols = p.total_chunks * p.box_rows;
      const int c0 = (int)((int64_t)split * ncols / p.splits);
      const int c1 = (int)((int64_t)(split + 1) * ncols / p.splits);
      const uint32_t red_addr = base;
      const float* red = reinterpret_cast<const float*>(base_ptr);
      for (int col = c0 + (tid >> 5); col < c1; col += 4) {
        const int chunk = col / p.box_rows;
        const int r = col - chunk * p.box_rows;
        const RingChunk ch = ring_chunk(geom, chunk);
        if (r >= ch.valid) continue;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t off = (uint32_t)((col * kTileM + lane4) * 4);
        if (p.splits > 1) {
          for (int rk = 0; rk < p.splits; ++rk) {
            const float4 v = ptx::ld_shared_cluster_v4(ptx::map_shared_rank(red_addr + off, (uint32_t)rk));
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
          }
        } else {
          s = *reinterpret_cast<const float4*>(red + col * kTileM + lane4);
        }
        store_row4<kF32>(p.out, p.ldo, ch.out_row + r, (int64_t)swap_nt * kTileM + lane4, s);
      }
    }
    if (p.splits > 1) ptx::cluster_sync_all();  // keep shared memory alive for remote readers
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
}

// Copies shard r (blockIdx.y) to rows [r*m_pd, (r+1)*m_pd) of the gathered
// buffer: the decomposed path's all-gather (AllGather-GEMM tutorial, local
// store phase), here a device-local copy.
__global__ void __launch_bounds__(256) agmm_gather_rows(const __grid_constant__ GatherParams g) {
  const int r = blockIdx.y;
  const uint4* __restrict__ src = g.src[r];
  uint4* __restrict__ dst = g.dst + (int64_t)r * g.vec_per_shard;
  const int64_t n = g.vec_per_shard;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 v0 = __ldg(src + i);
    const uint4 v1 = __ldg(src + i + stride);
    const uint4 v2 = __ldg(src + i + 2 * stride);
    const uint4 v3 = __ldg(src + i + 3 * stride);
    dst[i] = v0;
    dst[i + stride] = v1;
    dst[i + 2 * stride] = v2;
    dst[i + 3 * stride] = v3;
  }
  for (; i < n; i += stride) dst[i] = __ldg(src + i);
}

using KernelFn = void (*)(KernelParams);

KernelFn select_kernel(const KernelKey& k) {
#define AGMM_PICK(PATH, BN)                                                                   \
  (k.y_kmajor ? (k.out_f32 ? &agmm_fused_sm103a<PATH, true, true, BN>                         \
                           : &agmm_fused_sm103a<PATH, true, false, BN>)                       \
              : (k.out_f32 ? &agmm_fused_sm103a<PATH, false, true, BN>                        \
                           : &agmm_fused_sm103a<PATH, false, false, BN>))
  if (k.path == kPathSwap) return AGMM_PICK(kPathSwap, 128);
  if (k.bn == 256) return AGMM_PICK(kPathRows, 256);
  if (k.bn == 128) return AGMM_PICK(kPathRows, 128);
  return nullptr;
#undef AGMM_PICK
}

}  // namespace

cudaError_t prepare_agmm_kernel(const KernelKey& key, size_t smem_bytes, int cluster_x,
                                int* max_active) {
  KernelFn fn = select_kernel(key);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  if (cluster_x > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (max_active) {
    if (cluster_x > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)cluster_x, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem_bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)cluster_x;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(max_active, fn, &cfg);
    } else {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_active, fn, kThreads, smem_bytes);
    }
  }
  return e;
}

cudaError_t launch_agmm_kernel(const KernelKey& key, const KernelParams& p, dim3 grid, int cluster_x,
                               size_t smem_bytes, cudaStream_t stream) {
  KernelFn fn = select_kernel(key);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (cluster_x > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, fn, p);
}

cudaError_t launch_gather_kernel(const GatherParams& g, int P, int blocks_per_shard,
                                 cudaStream_t stream) {
  agmm_gather_rows<<<dim3((unsigned)blocks_per_shard, (unsigned)P, 1), 256, 0, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace agmm
