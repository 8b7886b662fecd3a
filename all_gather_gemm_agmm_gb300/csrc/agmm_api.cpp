// agmm_api.cpp -- the C ABI of include/agmm.h: argument validation, tile
// planning, the per-shard TMA descriptor table, and kernel launches.
//
// Validation follows validate_inputs of tpu_inference "all_gather_matmul.py"
// (k % 128, n % 128), with its m rules relaxed (see agmm.h).  The descriptor
// table follows the per-peer descriptor idea of jax mosaic gpu
// "launch_context.py" (_get_tma_desc: one 128-byte descriptor per peer base
// pointer, at most 8 peers): descriptors are encoded on the host and passed to
// the kernel as a __grid_constant__ parameter block.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "agmm.h"
#include "kernel_params.h"
#include "ring_schedule.h"

using namespace agmm;

namespace {

thread_local std::string g_last_error;

agmm_status_t fail(agmm_status_t s, const std::string& msg) {
  g_last_error = msg;
  if (std::getenv("AGMM_LOG")) std::fprintf(stderr, "[agmm] %s: %s\n", agmm_status_string(s), msg.c_str());
  return s;
}

agmm_status_t fail_cuda(cudaError_t e, const char* what) {
  return fail(AGMM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

constexpr int64_t kMaxElems = (int64_t)1 << 40;

int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
bool encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer, bool f16, std::string* err) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

// Y stored [k, n] as a 3-D tensor: dims {64 n, k, n / 64}, byte strides
// {n * 2, 128}; a box {64, 64, blocks} brings `blocks` 64-column blocks of
// one 64-row k block, each an 8 KiB MN-major swizzled block, in one copy.
bool encode_y_mn3d(CUtensorMap* map, const void* ptr, uint64_t n, uint64_t k, uint32_t blocks, bool f16,
                   std::string* err) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t dims[3] = {64, k, n / 64};
  cuuint64_t strides[2] = {n * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kTileK, blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled (3-D Y) failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

}  // namespace

struct agmm_plan_s {
  int P = 0;
  int64_t m_pd = 0, k = 0, n = 0;
  agmm_dtype_t dtype = AGMM_BF16;
  int rhs_t = 0;
  int device = 0;
  int num_sms = 0;
  KernelKey key{};
  int whole_shards = 0;
  int box_rows = 0, total_chunks = 0, num_m_tiles = 0, num_mc_tiles = 0, num_n_tiles = 0, num_k_blocks = 0;
  int group_m = 1, num_tiles = 0, stages = 0, mma_n = 0, tmem_cols = 0, splits = 1;
  uint32_t b_slot_bytes = 0;
  int atoms = 1;  // k blocks per pipeline stage (1 or 2)
  size_t smem_bytes = 0;
  dim3 grid{1, 1, 1};
  int cluster_x = 1;
  int dp_tiles = 0, sk_tiles = 0;
  int max_clusters = 0;  // co-resident clusters (rows path)
  bool swap_dsmem = false;  // swap path: k-split partials through DSMEM
  int row_groups = 1;       // swap path: row groups of the gathered rows (grid z)
  bool f16 = false;         // fp16 operands (else bf16)
  int clock_khz = 2100000;  // peak SM clock of the planned device
  int group_chunks = 0;     // swap path: ring chunks per row group
  bool stream_k = true;     // rows path: share a ragged last wave's k blocks
  bool stream_k_asked = false;  // rows path: the configuration set stream-K on (no fill rule)
  int config_source = 0;    // agmm_plan_info_t::config_source
  size_t tail_bytes = 0;  // workspace bytes for tail counters and partials
  // descriptor cache: tensor maps depend only on the X and Y pointers
  bool cache_valid = false;
  const void* cache_x[kMaxShards] = {};
  const void* cache_y = nullptr;
  const void* cache_xcat = nullptr;  // buffer the gathered-LHS maps describe
  KernelParams params{};
  agmm_plan_s* sub = nullptr;  // unfused path: P = 1 over the gathered buffer
  agmm_tile_config_t user_cfg{};  // the caller's configuration (fields 0 when none)
  size_t out_elem = 2;
  int64_t M() const { return (int64_t)P * m_pd; }
};

namespace {

size_t gathered_bytes(const agmm_plan_s* pl) { return ((size_t)pl->M() * (size_t)pl->k * 2 + 255) / 256 * 256; }

agmm_status_t validate_shape(int P, int64_t m_pd, int64_t k, int64_t n, int dtype, int rhs_t) {
  if (P < 1 || P > AGMM_MAX_SHARDS)
    return fail(AGMM_ERR_INVALID_ARG, "P must be in [1, 8] (per-peer descriptor tables hold at most 8)");
  if (m_pd < 1 || m_pd > ((int64_t)1 << 31) - 1)
    return fail(AGMM_ERR_INVALID_ARG, "m_per_device must be in [1, 2^31)");
  if (k < 128 || k % 128 != 0) return fail(AGMM_ERR_INVALID_ARG, "k must be a positive multiple of 128");
  if (n < 128 || n % 128 != 0) return fail(AGMM_ERR_INVALID_ARG, "n must be a positive multiple of 128");
  if (k > ((int64_t)1 << 31) - 1 || n > ((int64_t)1 << 31) - 1)
    return fail(AGMM_ERR_INVALID_ARG, "k and n must be below 2^31");
  const int64_t M = (int64_t)P * m_pd;
  if (M > kMaxElems / k || k > kMaxElems / n || M > kMaxElems / n)
    return fail(AGMM_ERR_INVALID_ARG, "problem exceeds 2^40 elements in an operand");
  if (dtype < AGMM_BF16 || dtype > AGMM_F16_F32OUT) return fail(AGMM_ERR_INVALID_ARG, "unknown dtype");
  if (rhs_t != 0 && rhs_t != 1) return fail(AGMM_ERR_INVALID_ARG, "rhs_transpose must be 0 or 1");
  return AGMM_OK;
}

// tcgen05.alloc blocks until the SM has the columns free, so the CTAs that
// shared memory lets share an SM must fit in its 512 TMEM columns together;
// otherwise a CTA could wait on a CTA of another cluster that waits on it.
// Pads the request so that at most 512 / tmem_cols CTAs are resident per SM
// (228 KiB of shared memory per SM, 1 KiB of it reserved per CTA).
size_t tmem_safe_smem(size_t smem, int tmem_cols) {
  constexpr size_t kSmemPerSm = 233472;
  const size_t fit = (size_t)(512 / std::max(32, tmem_cols));
  const size_t floor_bytes = kSmemPerSm / (fit + 1) + 1;  // fit + 1 CTAs would not fit
  return std::min(kMaxDynSmem, std::max(smem, floor_bytes));
}

// The tuned table: measured tile configurations for exact shapes, written by
// the package's tuner (tune.py) from its timing runs on GB300.
struct TunedEntry {
  int P;
  int64_t m_pd, k, n;
  int rhs_t, f16;
  agmm_tile_config_t cfg;
};
const TunedEntry kTunedTable[] = {
#include "tuned_sm103.inc"
    {0, 0, 0, 0, 0, 0, {}}  // end marker
};

const agmm_tile_config_t* tuned_lookup(int P, int64_t m_pd, int64_t k, int64_t n, int rhs_t, bool f16) {
  for (const TunedEntry& e : kTunedTable)
    if (e.P == P && e.m_pd == m_pd && e.k == k && e.n == n && e.rhs_t == rhs_t && e.f16 == (f16 ? 1 : 0))
      return &e.cfg;
  return nullptr;
}

bool on_off_ok(int v) { return v == AGMM_CFG_AUTO || v == AGMM_CFG_OFF || v == AGMM_CFG_ON; }

agmm_status_t validate_config(const agmm_tile_config_t* c) {
  if (!c) return AGMM_OK;
  const bool box_ok = c->box_rows == 0 || c->box_rows == 8 || c->box_rows == 16 || c->box_rows == 32 ||
                      c->box_rows == 64 || c->box_rows == 128;
  const bool rg_ok = c->row_groups == 0 || (c->row_groups >= 1 && c->row_groups <= 256 &&
                                            (c->row_groups & (c->row_groups - 1)) == 0);
  if (c->path < 0 || c->path > 2) return fail(AGMM_ERR_INVALID_ARG, "config.path must be 0, 1 or 2");
  if (c->chunks < 0 || c->chunks > 2) return fail(AGMM_ERR_INVALID_ARG, "config.chunks must be 0, 1 or 2");
  if (!box_ok) return fail(AGMM_ERR_INVALID_ARG, "config.box_rows must be 0, 8, 16, 32, 64 or 128");
  if (c->tile_n != 0 && c->tile_n != 128 && c->tile_n != 256)
    return fail(AGMM_ERR_INVALID_ARG, "config.tile_n must be 0, 128 or 256");
  if (c->cluster_m < 0 || c->cluster_m > 2) return fail(AGMM_ERR_INVALID_ARG, "config.cluster_m must be 0, 1 or 2");
  if (!on_off_ok(c->cta_pair) || !on_off_ok(c->stream_k) || !on_off_ok(c->dsmem_reduce) ||
      !on_off_ok(c->tuned_table))
    return fail(AGMM_ERR_INVALID_ARG, "on/off config fields take AGMM_CFG_AUTO, AGMM_CFG_OFF or AGMM_CFG_ON");
  if (c->stages != 0 && (c->stages < 2 || c->stages > kMaxStages))
    return fail(AGMM_ERR_INVALID_ARG, "config.stages must be 0 or in [2, 8]");
  if (c->group_m < 0 || c->group_m > 65536) return fail(AGMM_ERR_INVALID_ARG, "config.group_m must be in [0, 65536]");
  if (!rg_ok) return fail(AGMM_ERR_INVALID_ARG, "config.row_groups must be 0 or a power of two up to 256");
  if (c->splits < 0 || c->splits > 16) return fail(AGMM_ERR_INVALID_ARG, "config.splits must be in [0, 16]");
  return AGMM_OK;
}

// AGMM_* environment overrides (tests and experiments) as a config; values
// out of range are ignored.
agmm_tile_config_t env_config() {
  agmm_tile_config_t c{};
  auto on_off = [](const char* name) {
    const char* v = std::getenv(name);
    if (!v || !*v) return AGMM_CFG_AUTO;
    return std::atoi(v) != 0 ? AGMM_CFG_ON : AGMM_CFG_OFF;
  };
  const int path = env_int("AGMM_PATH", -1);  // 0: row tiles, 1: swapped tiles
  if (path == kPathRows || path == kPathSwap) c.path = path == kPathRows ? 1 : 2;
  const char* ch = std::getenv("AGMM_CHUNKS");  // half | whole
  if (ch && std::strcmp(ch, "half") == 0) c.chunks = 1;
  if (ch && std::strcmp(ch, "whole") == 0) c.chunks = 2;
  const int bn = env_int("AGMM_BN", 0);
  if (bn == 128 || bn == 256) c.tile_n = bn;
  const int cm = env_int("AGMM_CM", 0);
  if (cm == 1 || cm == 2) c.cluster_m = cm;
  c.cta_pair = on_off("AGMM_PAIR");
  const int st = env_int("AGMM_STAGES", 0);
  if (st >= 1) c.stages = std::min(kMaxStages, std::max(2, st));
  const int gm = env_int("AGMM_GROUP_M", 0);
  if (gm >= 1) c.group_m = std::min(gm, 65536);
  c.stream_k = on_off("AGMM_STREAMK");
  const int rg = env_int("AGMM_ROWGROUPS", 0);
  if (rg >= 1) c.row_groups = rg;
  const int sk = env_int("AGMM_SPLITK", 0);
  if (sk >= 1) c.splits = std::min(sk, 16);
  c.dsmem_reduce = on_off("AGMM_SWAP_DSMEM");
  c.tuned_table = on_off("AGMM_TUNED");
  return c;
}

bool any_tile_field(const agmm_tile_config_t& c) {
  return c.path || c.chunks || c.box_rows || c.tile_n || c.cluster_m || c.cta_pair || c.stages || c.group_m ||
         c.stream_k || c.row_groups || c.splits || c.dsmem_reduce;
}

// Fields of `top` that are set replace those of `base`.
void overlay(agmm_tile_config_t* base, const agmm_tile_config_t& top) {
  auto pick = [](int& b, int t) {
    if (t != 0) b = t;
  };
  pick(base->path, top.path);
  pick(base->chunks, top.chunks);
  pick(base->box_rows, top.box_rows);
  pick(base->tile_n, top.tile_n);
  pick(base->cluster_m, top.cluster_m);
  pick(base->cta_pair, top.cta_pair);
  pick(base->stages, top.stages);
  pick(base->group_m, top.group_m);
  pick(base->stream_k, top.stream_k);
  pick(base->row_groups, top.row_groups);
  pick(base->splits, top.splits);
  pick(base->dsmem_reduce, top.dsmem_reduce);
  pick(base->tuned_table, top.tuned_table);
}

// The configuration a plan is built from: the caller's set fields, then the
// environment's, then the tuned table's entry for the exact shape.  Fields
// the caller set are strict (an infeasible one fails the plan); the others
// fall back to the planner's rules when they cannot hold.
struct ResolvedConfig {
  agmm_tile_config_t cfg{};
  agmm_tile_config_t strict{};
  int source = 0;
};

ResolvedConfig resolve_config(const agmm_plan_s* pl, const agmm_tile_config_t* user) {
  ResolvedConfig r;
  const agmm_tile_config_t env = env_config();
  if (user) r.strict = *user;
  const int table_switch = user && user->tuned_table ? user->tuned_table : env.tuned_table;
  const agmm_tile_config_t* tuned =
      table_switch == AGMM_CFG_OFF ? nullptr : tuned_lookup(pl->P, pl->m_pd, pl->k, pl->n, pl->rhs_t, pl->f16);
  if (tuned) {
    r.cfg = *tuned;
    r.source = 1;
  }
  overlay(&r.cfg, env);
  overlay(&r.cfg, r.strict);
  if (any_tile_field(env) || any_tile_field(r.strict)) r.source = 2;
  return r;
}

// Tile planning for a device with `num_sms` SMs (pure host logic), from the
// resolved configuration `c`; fields of `strict` that are set must hold.
agmm_status_t choose_tiles(agmm_plan_s* pl, const agmm_tile_config_t& c, const agmm_tile_config_t& strict) {
  const int whole_lo = c.chunks == 2 ? 1 : 0;
  const int whole_hi = c.chunks == 1 ? 0 : 1;
  const int bh_top = c.box_rows ? c.box_rows : 128;
  const int bh_bottom = c.box_rows ? c.box_rows : 8;
  // Swap path: the whole ring-ordered row sequence (chunks padded to their box
  // height) fits in one MMA N of at most 256.  Candidates: half-shard chunks
  // (the ring's half split) or whole-shard chunks, each with box heights 8..128.
  // Cost: padded rows (MMA N, reduction volume) plus 16 rows per chunk (one
  // TMA box per chunk and stage).  Ties keep the half split and larger boxes.
  int best_bh = -1, best_whole = 0;
  int64_t best_cost = 0;
  for (int whole = whole_lo; whole <= whole_hi; ++whole) {
    for (int bh = bh_top; bh >= bh_bottom; bh >>= 1) {
      const RingGeom g = make_ring_geom(pl->P, pl->m_pd, 0, bh, whole);
      const int64_t pad = ring_padded_rows(g);
      const int64_t cost = pad + 16 * ring_total_chunks(g);
      if (pad <= 256 && (best_bh < 0 || cost < best_cost)) {
        best_bh = bh;
        best_whole = whole;
        best_cost = cost;
      }
    }
  }
  if (best_bh < 0 && strict.path == 2)
    return fail(AGMM_ERR_UNSUPPORTED, "swapped tiles need the gathered rows, padded to box heights, within 256");
  const int64_t budget = (int64_t)kMaxDynSmem - 1024 - kCtlBytes;
  pl->num_k_blocks = (int)(pl->k / kTileK);
  if (best_bh > 0 && c.path != 1) {
    pl->key.path = kPathSwap;
    pl->key.bn = kTileM;
    pl->key.cm = 1;
    pl->key.pair = false;
    pl->box_rows = best_bh;
    pl->whole_shards = best_whole;
    pl->total_chunks = (int)ring_total_chunks(make_ring_geom(pl->P, pl->m_pd, 0, best_bh, best_whole));
    pl->num_n_tiles = (int)(pl->n / kTileM);
    pl->num_m_tiles = 1;
    pl->num_tiles = pl->num_n_tiles;
    // Row groups: the chunks may be divided into G groups (blockIdx.z), each
    // its own MMA N.  More groups re-read Y (once per group) and each CTA
    // reads fewer X rows per k block; they leave more CTAs per n tile, so k
    // needs fewer splits, and the split-K partials (splits x rows x n floats,
    // written and read back) shrink.  Per-CTA cost model, in bytes moved
    // per SM: k blocks x (Y box + X rows) + 4.4 x the partial's bytes (a
    // partial is written and read back at about half the load rate).
    const int max_splits = std::min(16, pl->num_k_blocks);
    auto pick_groups = [&](int force_g, int* out_g, int* out_s) {
      double best_model = -1.0;
      for (int G = 1; G <= pl->total_chunks; G *= 2) {
        if (force_g > 0 && G != force_g) continue;
        const int cpg = (pl->total_chunks + G - 1) / G;
        if ((G - 1) * cpg >= pl->total_chunks) continue;  // the last group would be empty
        const int gcols = cpg * pl->box_rows;
        int S = pl->num_sms / (pl->num_n_tiles * G);
        S = std::max(1, std::min(S, max_splits));
        if (c.splits > 0) S = std::max(1, std::min(c.splits, max_splits));
        const int kb = (pl->num_k_blocks + S - 1) / S;
        const int mn = (gcols + 31) / 32 * 32;
        const double model = (double)kb * (kASlotBytes + 128.0 * mn) + (S > 1 ? 4.4 * 512.0 * gcols : 0.0);
        if (best_model < 0 || model < best_model * 0.97) {
          best_model = model;
          *out_g = G;
          *out_s = S;
        }
        if (force_g == 0 && G >= 8) break;
      }
      return best_model >= 0;
    };
    int best_g = 1, best_s = 1;
    if (!pick_groups(c.row_groups, &best_g, &best_s)) {
      if (strict.row_groups != 0)
        return fail(AGMM_ERR_UNSUPPORTED, "config.row_groups leaves a row group empty for this shape");
      pick_groups(0, &best_g, &best_s);
    }
    pl->row_groups = best_g;
    pl->group_chunks = (pl->total_chunks + best_g - 1) / best_g;
    pl->mma_n = (pl->group_chunks * pl->box_rows + 31) / 32 * 32;
    pl->b_slot_bytes = (uint32_t)pl->mma_n * 128u;
    // Two k blocks per stage halve the barrier hand-offs per block, as long
    // as at least three stages still fit (MMA N <= 128); wider tiles keep
    // one block per stage and their deeper ring.
    pl->atoms = budget / (2 * (kASlotBytes + (int64_t)pl->b_slot_bytes)) >= 3 ? 2 : 1;
    pl->key.atoms = pl->atoms;
    const int64_t stage_bytes = (kASlotBytes + pl->b_slot_bytes) * pl->atoms;
    pl->stages = (int)std::min<int64_t>(kMaxStages, budget / stage_bytes);
    if (c.stages) pl->stages = std::min(pl->stages, c.stages);
    // The k splits (cluster size); plan_impl lowers them until one wave of
    // clusters covers every (n tile, row group).
    pl->splits = best_s;
    // k-split partials go through device memory (L2) unless dsmem_reduce
    // routes them through distributed shared memory.
    pl->swap_dsmem = c.dsmem_reduce == AGMM_CFG_ON;
    pl->tmem_cols = pow2_ceil(std::max(32, pl->mma_n));
    pl->group_m = 1;
  } else {
    pl->key.path = kPathRows;
    // Chunking: half-shard (the ring's half split) or whole-shard chunks, box
    // heights 8..128.  Within 3% of the fewest 128-row tiles, take the largest
    // box (fewest TMA boxes per stage); ties keep the half split.
    int64_t min_tiles = -1;
    for (int whole = whole_lo; whole <= whole_hi; ++whole)
      for (int bh = bh_top; bh >= bh_bottom; bh >>= 1) {
        const RingGeom g = make_ring_geom(pl->P, pl->m_pd, 0, bh, whole);
        const int64_t t = (ring_total_chunks(g) + kTileM / bh - 1) / (kTileM / bh);
        if (min_tiles < 0 || t < min_tiles) min_tiles = t;
      }
    int bh_best = -1, whole_best = 0;
    int64_t tiles_best = -1;
    for (int whole = whole_lo; whole <= whole_hi; ++whole)
      for (int bh = bh_top; bh >= bh_bottom; bh >>= 1) {
        const RingGeom g = make_ring_geom(pl->P, pl->m_pd, 0, bh, whole);
        const int64_t t = (ring_total_chunks(g) + kTileM / bh - 1) / (kTileM / bh);
        if (t * 100 > min_tiles * 103 && t > min_tiles) continue;
        if (bh > bh_best) {
          bh_best = bh;
          whole_best = whole;
          tiles_best = t;
        }
      }
    if (tiles_best > (int64_t)1 << 30) return fail(AGMM_ERR_INVALID_ARG, "too many row tiles");
    // Clusters of two CTAs on neighbouring row tiles multiply as a
    // cta_group::2 pair: each CTA holds its 128 rows and half the Y tile, 32
    // KiB per k block and SM, and reads half the Y operand per MMA.  No copy
    // is multicast; a two-CTA cluster is always a pair, so cta_pair off means
    // one-CTA clusters.
    int cm = c.cluster_m ? c.cluster_m : (tiles_best >= 2 ? 2 : 1);
    if (c.cta_pair == AGMM_CFG_ON && cm != 2 && strict.cta_pair == AGMM_CFG_ON)
      return fail(AGMM_ERR_UNSUPPORTED, "config.cta_pair needs cluster_m 2");
    if (c.cta_pair == AGMM_CFG_OFF && cm == 2) {
      if (strict.cta_pair == AGMM_CFG_OFF && strict.cluster_m == 2)
        return fail(AGMM_ERR_UNSUPPORTED, "a two-CTA cluster multiplies as a CTA pair: cta_pair off needs cluster_m 1");
      if (strict.cluster_m != 2) cm = 1;
    }
    // 256-wide tiles, unless they would not give half the clusters a whole
    // tile (stream-K then splits most of the work): 128-wide tiles double
    // the tile count.
    int bn = (pl->n % 256 == 0) ? 256 : 128;
    if (bn == 256) {
      const int64_t tiles256 = (tiles_best + cm - 1) / cm * (pl->n / 256);
      if (2 * tiles256 < pl->num_sms / cm) bn = 128;
    }
    if (c.tile_n) {
      if (pl->n % c.tile_n == 0)
        bn = c.tile_n;
      else if (strict.tile_n)
        return fail(AGMM_ERR_UNSUPPORTED, "config.tile_n does not divide n");
    }
    pl->key.bn = bn;
    pl->box_rows = bh_best;
    pl->whole_shards = whole_best;
    pl->total_chunks = (int)ring_total_chunks(make_ring_geom(pl->P, pl->m_pd, 0, bh_best, whole_best));
    pl->num_m_tiles = (int)tiles_best;
    pl->num_n_tiles = (int)(pl->n / bn);
    pl->key.cm = cm;
    pl->key.pair = cm == 2;
    pl->num_mc_tiles = (pl->num_m_tiles + cm - 1) / cm;
    if ((int64_t)pl->num_mc_tiles * pl->num_n_tiles > ((int64_t)1 << 31) - 1)
      return fail(AGMM_ERR_INVALID_ARG, "too many output tiles");
    pl->num_tiles = pl->num_mc_tiles * pl->num_n_tiles;
    pl->mma_n = bn;
    pl->b_slot_bytes = (uint32_t)(pl->key.pair ? bn / 2 : bn) * 128u;
    // 128-wide tiles take two k blocks per stage whenever three such stages
    // fit: the producer's and the MMA issuer's barrier operations per stage
    // cost more than a 128-wide k block's MMAs (about 256 cycles), and two
    // blocks per stage halve them per block (P4 m128 sweep point: 24.7 ->
    // 22.0 us).  256-wide tiles keep one block per stage and their deeper
    // ring: their MMAs take about as long as the hand-offs, and with two
    // blocks per stage only three stages fit (c4_quarter: 262 -> 269 us).
    pl->atoms = bn == 128 && budget / (2 * (kASlotBytes + (int64_t)pl->b_slot_bytes)) >= 3 ? 2 : 1;
    const int env_atoms = env_int("AGMM_ATOMS", 0);
    if (env_atoms == 1 || env_atoms == 2) pl->atoms = env_atoms;
    pl->key.atoms = pl->atoms;
    const int64_t stage_bytes = (kASlotBytes + pl->b_slot_bytes) * pl->atoms;
    pl->stages = (int)std::min<int64_t>(kMaxStages, budget / stage_bytes);
    if (c.stages) pl->stages = std::min(pl->stages, c.stages);
    pl->splits = 1;
    pl->tmem_cols = 2 * bn;
    pl->group_m = c.group_m ? c.group_m : 8;
    pl->stream_k = c.stream_k != AGMM_CFG_OFF;
    pl->stream_k_asked = c.stream_k == AGMM_CFG_ON;
  }
  pl->smem_bytes = tmem_safe_smem(1024 + (size_t)pl->stages * (kASlotBytes + pl->b_slot_bytes) * pl->atoms + kCtlBytes,
                                  pl->tmem_cols);
  return AGMM_OK;
}

// Rows path: persistent clusters, one CTA per SM, at most `max_clusters`
// co-resident.  Whole waves of cluster tiles are dealt round-robin; when the
// tile count is not a multiple of the clusters, the last one to two waves' k
// blocks are divided evenly over the clusters (stream-K), so no SM idles in a
// ragged last wave -- unless that wave already fills two thirds of the
// clusters: its idle clusters then cost less than stream-K's fix-up at the
// end of the launch (an owner waits for its contributors' partials and sums
// them), measured at about a third of a tile's time.  A configuration that
// sets stream-K on keeps it whatever the fill.
void size_rows_grid(agmm_plan_s* pl, int max_clusters) {
  const int cm = pl->key.cm;
  int G = std::max(1, std::min(pl->num_sms / cm, max_clusters));
  const int T = pl->num_tiles;
  int dp = T;
  if (T % G != 0 && pl->stream_k && (pl->stream_k_asked || 3 * (T % G) < 2 * G)) {
    // Stream-K over the ragged last wave alone keeps its tiles together in
    // raster order (L2 reuse) as long as a tile is shared by at most about
    // three clusters; a thinner last wave also takes the wave before it.
    const int W = T / G;
    const int R = T - W * G;
    dp = (W >= 1 && 3 * R >= G) ? W * G : (W >= 1 ? (W - 1) * G : 0);
    // at least 4 k blocks per cluster share
    const int64_t units = (int64_t)(T - dp) * pl->num_k_blocks;
    if (units < (int64_t)G * 4) G = (int)std::max<int64_t>(1, units / 4);
  }
  if (dp == T) G = std::min(G, T);
  pl->dp_tiles = dp;
  pl->sk_tiles = T - dp;
  pl->grid = dim3((unsigned)(G * cm), 1, 1);
  pl->tail_bytes = pl->sk_tiles > 0 ? (size_t)(pl->sk_tiles * cm * 4 + 255) / 256 * 256 +
                                          (size_t)G * cm * kTileM * (size_t)pl->key.bn * 4
                                    : 0;
  pl->cluster_x = cm;
}

agmm_status_t plan_impl(int P, int64_t m_pd, int64_t k, int64_t n, agmm_dtype_t dtype, int rhs_t,
                        const agmm_tile_config_t* config, bool with_sub, agmm_plan_s** out) {
  agmm_status_t st = validate_shape(P, m_pd, k, n, (int)dtype, rhs_t);
  if (st != AGMM_OK) return st;
  if ((st = validate_config(config)) != AGMM_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return fail_cuda(e, "cudaDeviceGetAttribute");
  int clock_khz = 0;
  if (cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess || clock_khz <= 0) {
    (void)cudaGetLastError();
    clock_khz = 2100000;  // above the part's 2.07 GHz peak
  }
  if (major != 10 || minor != 3)
    return fail(AGMM_ERR_UNSUPPORTED, "this library is built for sm_103a only; device is sm_" +
                                          std::to_string(major) + std::to_string(minor));
  agmm_plan_s* pl = new (std::nothrow) agmm_plan_s();
  if (!pl) return fail(AGMM_ERR_NOMEM, "plan allocation");
  pl->P = P;
  pl->m_pd = m_pd;
  pl->k = k;
  pl->n = n;
  pl->dtype = dtype;
  pl->rhs_t = rhs_t;
  pl->device = dev;
  pl->num_sms = sms;
  pl->clock_khz = clock_khz;
  pl->key.y_kmajor = rhs_t != 0;
  pl->key.out_f32 = dtype == AGMM_BF16_F32OUT || dtype == AGMM_F16_F32OUT;
  pl->f16 = dtype == AGMM_F16 || dtype == AGMM_F16_F32OUT;
  pl->out_elem = pl->key.out_f32 ? 4 : 2;
  const ResolvedConfig rc = resolve_config(pl, config);
  pl->config_source = rc.source;
  st = choose_tiles(pl, rc.cfg, rc.strict);
  if (st != AGMM_OK) {
    delete pl;
    return st;
  }
  // Attributes and co-residency.  Swap path: the largest cluster (k split)
  // for which one wave of clusters covers every n tile; rows path: one
  // persistent CTA per SM.
  const int swap_stages = pl->stages;  // the swapped tiles' depth before the reduction's buffers
  for (;;) {
    if (pl->key.path == kPathSwap) {
      // k splits reduced through distributed shared memory: each rank's
      // partial (Q quads of 128 x 4 floats, Q = the widest row group's slots
      // / 4) is drained into its own pipeline memory, and a receive buffer of
      // splits x ceil(Q / splits) quads follows the control block.  Fewer
      // stages until both fit; if they cannot, the device-memory route (which
      // needs neither buffer) with the same splits.
      const int64_t stage_bytes = (kASlotBytes + pl->b_slot_bytes) * pl->atoms;
      const int64_t Q = (int64_t)pl->group_chunks * pl->box_rows / 4;
      const int64_t quad = (int64_t)kTileM * 16;
      const bool bulk = pl->splits > 1 && pl->swap_dsmem;
      const int64_t recv = bulk ? pl->splits * ((Q + pl->splits - 1) / pl->splits) * quad : 0;
      const int64_t avail = (int64_t)kMaxDynSmem - 1024 - kCtlBytes - recv;
      if (bulk) {
        int st = swap_stages;
        while (st > 2 && (int64_t)st * stage_bytes > avail) --st;
        if ((int64_t)st * stage_bytes > avail || (int64_t)st * stage_bytes < Q * quad) {
          pl->swap_dsmem = false;
          pl->stages = swap_stages;
          continue;
        }
        pl->stages = st;
      } else {
        pl->stages = swap_stages;
      }
      pl->smem_bytes =
          tmem_safe_smem(1024 + (size_t)pl->stages * stage_bytes + kCtlBytes + (size_t)recv, pl->tmem_cols);
    }
    int active = 0;
    const int cluster = pl->key.path == kPathSwap ? pl->splits : pl->key.cm;
    e = prepare_agmm_kernel(pl->key, pl->smem_bytes, cluster, &active);
    if (e != cudaSuccess) {
      delete pl;
      return fail_cuda(e, "kernel attribute setup");
    }
    if (pl->key.path == kPathRows) {
      // the variant that also copies the gathered LHS runs on the same grid
      KernelKey sk = pl->key;
      sk.store = true;
      int active_store = 0;
      e = prepare_agmm_kernel(sk, pl->smem_bytes, cluster, &active_store);
      if (e != cudaSuccess) {
        delete pl;
        return fail_cuda(e, "kernel attribute setup (store variant)");
      }
      active = std::min(active, active_store);
      if (active <= 0) {
        delete pl;
        return fail(AGMM_ERR_UNSUPPORTED, "row kernel cannot be resident");
      }
      pl->max_clusters = cluster > 1 ? active : active * pl->num_sms;
      break;
    }
    if (pl->splits == 1) active *= pl->num_sms;  // CTAs per SM -> CTAs per device
    const int needed = pl->key.path == kPathSwap ? pl->num_n_tiles * pl->row_groups : 1;
    if (active >= needed || (pl->splits == 1 && active > 0)) break;
    if (pl->splits <= 1) {
      delete pl;
      return fail(AGMM_ERR_UNSUPPORTED, "kernel cannot be resident with the planned shared memory");
    }
    --pl->splits;
  }
  if (pl->key.path == kPathSwap) {
    pl->grid = dim3((unsigned)pl->splits, (unsigned)pl->num_n_tiles, (unsigned)pl->row_groups);
    pl->cluster_x = pl->splits;
    if (pl->splits > 1 && !pl->swap_dsmem) {
      const int64_t groups = (pl->group_chunks * (int64_t)pl->box_rows + 15) / 16;
      pl->tail_bytes = (size_t)pl->num_n_tiles * pl->row_groups * pl->splits * groups * 4 * kTileM * 16;
    }
    if (pl->splits == 1) pl->swap_dsmem = false;
  } else {
    size_rows_grid(pl, pl->max_clusters);
  }
  KernelParams& kp = pl->params;
  kp.m_pd = m_pd;
  kp.ldo = n;
  kp.P = P;
  kp.box_rows = pl->box_rows;
  kp.whole_shards = pl->whole_shards;
  kp.box_shift = 0;
  while ((1 << kp.box_shift) < pl->box_rows) ++kp.box_shift;
  kp.total_chunks = pl->total_chunks;
  kp.group_chunks = pl->key.path == kPathSwap ? pl->group_chunks : pl->total_chunks;
  kp.num_m_tiles = pl->num_m_tiles;
  kp.num_mc_tiles = pl->num_mc_tiles;
  kp.num_n_tiles = pl->num_n_tiles;
  kp.num_k_blocks = pl->num_k_blocks;
  kp.group_m = pl->group_m;
  kp.num_tiles = pl->num_tiles;
  kp.stages = pl->stages;
  kp.mma_n = pl->mma_n;
  kp.tmem_cols = pl->tmem_cols;
  kp.splits = pl->splits;
  kp.b_slot_bytes = pl->b_slot_bytes;
  // The kernels bound their waits in SM cycles: a limit converted at the
  // peak clock (kHz = cycles per millisecond) lasts at least that long.
  kp.wait_limit_cycles = (uint64_t)std::max(1, env_int("AGMM_WAIT_LIMIT_MS", 2000)) * (uint64_t)pl->clock_khz;
  kp.test_drop_first_arrive = env_int("AGMM_TEST_DROP_ARRIVE", 0) != 0;
  kp.pdl = env_int("AGMM_PDL", 1) != 0;
  kp.f16 = pl->f16 ? 1 : 0;
  kp.dp_tiles = pl->dp_tiles;
  if (config) pl->user_cfg = *config;
  if (with_sub && P > 1) {
    st = plan_impl(1, pl->M(), k, n, dtype, rhs_t, nullptr, false, &pl->sub);
    if (st != AGMM_OK) {
      delete pl;
      return st;
    }
  }
  *out = pl;
  return AGMM_OK;
}

// ws_bytes: the workspace bytes the call uses (agmm_workspace_bytes); the
// workspace must not overlap O, Y or a shard.
agmm_status_t check_run_args(agmm_plan_s* pl, const void* const* xs, const void* y, void* o, int my_id,
                             void* ws, size_t ws_bytes) {
  if (!pl) return fail(AGMM_ERR_INVALID_ARG, "plan is NULL");
  if (!xs || !y || !o || !ws) return fail(AGMM_ERR_INVALID_ARG, "a pointer argument is NULL");
  if (my_id < 0 || my_id >= pl->P) return fail(AGMM_ERR_INVALID_ARG, "my_id must be in [0, P)");
  const size_t xbytes = (size_t)pl->m_pd * (size_t)pl->k * 2;
  const size_t ybytes = (size_t)pl->k * (size_t)pl->n * 2;
  const size_t obytes = (size_t)pl->M() * (size_t)pl->n * pl->out_elem;
  for (int r = 0; r < pl->P; ++r) {
    if (!xs[r]) return fail(AGMM_ERR_INVALID_ARG, "shard pointer " + std::to_string(r) + " is NULL");
    if (!aligned16(xs[r])) return fail(AGMM_ERR_ALIGNMENT, "shard " + std::to_string(r) + " is not 16-byte aligned");
    if (overlaps(xs[r], xbytes, o, obytes)) return fail(AGMM_ERR_INVALID_ARG, "O overlaps a shard");
    if (overlaps(xs[r], xbytes, ws, ws_bytes))
      return fail(AGMM_ERR_INVALID_ARG, "the workspace overlaps shard " + std::to_string(r));
  }
  if (!aligned16(y) || !aligned16(o) || !aligned16(ws))
    return fail(AGMM_ERR_ALIGNMENT, "Y, O and the workspace must be 16-byte aligned");
  if (overlaps(y, ybytes, o, obytes)) return fail(AGMM_ERR_INVALID_ARG, "O overlaps Y");
  if (overlaps(y, ybytes, ws, ws_bytes)) return fail(AGMM_ERR_INVALID_ARG, "the workspace overlaps Y");
  if (overlaps(o, obytes, ws, ws_bytes)) return fail(AGMM_ERR_INVALID_ARG, "the workspace overlaps O");
  return AGMM_OK;
}

// status: the device status words; tail_ws: tail_bytes of workspace for the
// split tail tiles (counters, then partials).
agmm_status_t launch_fused(agmm_plan_s* pl, const void* const* xs, const void* y, void* o, int my_id,
                           void* status, void* tail_ws, cudaStream_t stream, void* xcat = nullptr) {
  KernelParams& kpx = pl->params;
  // swapped tiles: the MMA thread stores the X boxes when asked; row tiles:
  // the epilogue warps of the store variant copy the rows to xcat
  kpx.store_xcat = xcat != nullptr && pl->key.path == kPathSwap ? 1 : 0;
  kpx.xcat = xcat;
  kpx.ldx = pl->k;
  for (int r = 0; r < kMaxShards; ++r) kpx.xsrc[r] = r < pl->P ? xs[r] : nullptr;
  if (xcat != nullptr && xcat != pl->cache_xcat) {
    // per-shard views of the gathered buffer: a store is clipped at its shard
    std::string err;
    for (int r = 0; r < pl->P; ++r) {
      const void* base = static_cast<const uint8_t*>(xcat) + (size_t)r * pl->m_pd * pl->k * 2;
      if (!encode_2d(&kpx.xcatmap[r], base, (uint64_t)pl->k, (uint64_t)pl->m_pd, kTileK, (uint32_t)pl->box_rows,
                     pl->f16, &err)) {
        pl->cache_xcat = nullptr;
        return fail(AGMM_ERR_CUDA, "gathered-LHS tensor map: " + err);
      }
    }
    pl->cache_xcat = xcat;
  }
  bool same = pl->cache_valid && pl->cache_y == y;
  for (int r = 0; same && r < pl->P; ++r) same = pl->cache_x[r] == xs[r];
  KernelParams& kp = pl->params;
  if (!same) {
    std::string err;
    for (int r = 0; r < pl->P; ++r) {
      if (!encode_2d(&kp.xmap[r], xs[r], (uint64_t)pl->k, (uint64_t)pl->m_pd, kTileK, (uint32_t)pl->box_rows, pl->f16, &err)) {
        pl->cache_valid = false;
        return fail(AGMM_ERR_CUDA, "shard tensor map: " + err);
      }
    }
    bool ok;
    const uint32_t y_rows =
        pl->key.path == kPathSwap ? (uint32_t)kTileM : (uint32_t)(pl->key.bn / pl->key.cm);
    kp.y3d = 0;
    if (pl->rhs_t) {  // Y [n, k]: K-major boxes of y_rows n-rows
      ok = encode_2d(&kp.ymap, y, (uint64_t)pl->k, (uint64_t)pl->n, kTileK, y_rows, pl->f16, &err);
    } else {
      // Y [k, n]: MN-major 64 n x 64 k blocks, all of one load (y_rows
      // columns) in one 3-D box; one 2-D box per block if the driver
      // refuses the 3-D map.
      ok = env_int("AGMM_Y3D", 1) != 0 &&
           encode_y_mn3d(&kp.ymap, y, (uint64_t)pl->n, (uint64_t)pl->k, y_rows / 64, pl->f16, &err);
      if (ok) {
        kp.y3d = 1;
      } else {
        if (!err.empty() && std::getenv("AGMM_LOG")) std::fprintf(stderr, "[agmm] %s; using 2-D boxes\n", err.c_str());
        err.clear();
        ok = encode_2d(&kp.ymap, y, (uint64_t)pl->n, (uint64_t)pl->k, 64, kTileK, pl->f16, &err);
      }
    }
    if (!ok) {
      pl->cache_valid = false;
      return fail(AGMM_ERR_CUDA, "Y tensor map: " + err);
    }
    for (int r = 0; r < pl->P; ++r) pl->cache_x[r] = xs[r];
    pl->cache_y = y;
    pl->cache_valid = true;
  }
  kp.out = o;
  kp.status = static_cast<int*>(status);
  kp.my_id = my_id;
  kp.swap_partials = (pl->key.path == kPathSwap && pl->tail_bytes > 0) ? static_cast<float*>(tail_ws) : nullptr;
  if (pl->sk_tiles > 0) {
    kp.sk_flags = static_cast<int*>(tail_ws);
    kp.sk_partials = reinterpret_cast<float*>(static_cast<uint8_t*>(tail_ws) +
                                              (pl->sk_tiles * pl->key.cm * 4 + 255) / 256 * 256);
  } else {
    kp.sk_flags = nullptr;
    kp.sk_partials = nullptr;
  }
  // Row tiles writing the gathered LHS run the variant whose epilogue copies it.
  KernelKey key = pl->key;
  key.store = xcat != nullptr && pl->key.path == kPathRows;
  // Stream-K owners wait for other CTAs.  Without clusters a cooperative
  // launch guarantees that every CTA of the grid is resident at once; with
  // clusters the planner sized the grid to the co-resident cluster count, and
  // the owners' waits are bounded in any case.
  cudaError_t e = launch_agmm_kernel(key, kp, pl->grid, pl->cluster_x, pl->smem_bytes,
                                     pl->sk_tiles > 0 && pl->cluster_x == 1, stream);
  if (e != cudaSuccess) return fail_cuda(e, "fused kernel launch");
  return AGMM_OK;
}

}  // namespace

namespace agmm {

// Records a failure for agmm_last_error (used by other translation units).
agmm_status_t set_last_error(agmm_status_t status, const char* message) { return fail(status, message); }

// The unfused path on an explicit scratch region of scratch_bytes bytes, with
// the status words and split-tail counters cleared first on `stream`.  Used by
// the allocation-free entry point.
agmm_status_t run_unfused_on_scratch(agmm_plan_s* plan, const void* const* x_shards, const void* y, void* o,
                                     int my_id, void* scratch, size_t scratch_bytes, cudaStream_t s) {
  if (!plan) return fail(AGMM_ERR_INVALID_ARG, "plan is NULL");
  const size_t need = agmm_workspace_bytes(plan, 1);
  if (need > scratch_bytes)
    return fail(AGMM_ERR_INVALID_ARG, "this problem needs " + std::to_string(need) +
                                          " bytes of scratch but the static scratch holds " +
                                          std::to_string(scratch_bytes) + "; use agmm_run_unfused");
  agmm_status_t st = check_run_args(plan, x_shards, y, o, my_id, scratch, need);
  if (st != AGMM_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  agmm_plan_s* gemm = plan->P == 1 ? plan : plan->sub;
  uint8_t* tail = plan->P == 1 ? base + kStatusBytes : base + kStatusBytes + gathered_bytes(plan);
  cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes, s);
  if (e == cudaSuccess && gemm->sk_tiles > 0)
    e = cudaMemsetAsync(tail, 0, (size_t)(gemm->sk_tiles * gemm->key.cm * 4 + 255) / 256 * 256, s);
  if (e != cudaSuccess) return fail_cuda(e, "scratch clear");
  if (plan->P == 1) return launch_fused(plan, x_shards, y, o, 0, base, tail, s);
  uint8_t* gathered = base + kStatusBytes;
  for (int r = 0; r < plan->P; ++r)
    if (overlaps(x_shards[r], (size_t)plan->m_pd * plan->k * 2, gathered, gathered_bytes(plan)))
      return fail(AGMM_ERR_INVALID_ARG, "the scratch overlaps a shard");
  GatherParams g{};
  for (int r = 0; r < plan->P; ++r) g.src[r] = static_cast<const uint4*>(x_shards[r]);
  g.dst = reinterpret_cast<uint4*>(gathered);
  g.vec_per_shard = plan->m_pd * plan->k * 2 / 16;
  const int64_t want = (g.vec_per_shard + 4 * 256 - 1) / (4 * 256);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)plan->num_sms * 8 / plan->P + 1));
  e = launch_gather_kernel(g, plan->P, blocks, s);
  if (e != cudaSuccess) return fail_cuda(e, "gather kernel launch");
  const void* one[1] = {gathered};
  return launch_fused(plan->sub, one, y, o, 0, base, tail, s);
}

}  // namespace agmm

extern "C" {

agmm_status_t agmm_plan_config(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                               int rhs_transpose, const agmm_tile_config_t* config, agmm_plan_t* out_plan) {
  if (!out_plan) return fail(AGMM_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  agmm_plan_s* pl = nullptr;
  agmm_status_t st = plan_impl(P, m_per_device, k, n, dtype, rhs_transpose, config, true, &pl);
  if (st == AGMM_OK) *out_plan = pl;
  return st;
}

agmm_status_t agmm_plan(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                        int rhs_transpose, agmm_plan_t* out_plan) {
  return agmm_plan_config(P, m_per_device, k, n, dtype, rhs_transpose, nullptr, out_plan);
}

void agmm_destroy(agmm_plan_t plan) {
  if (!plan) return;
  agmm_destroy(plan->sub);
  delete plan;
}

size_t agmm_workspace_bytes(agmm_plan_t plan, int unfused) {
  if (!plan) return 0;
  if (!unfused || plan->P == 1) return kStatusBytes + plan->tail_bytes;
  return kStatusBytes + gathered_bytes(plan) + plan->sub->tail_bytes;
}

agmm_status_t agmm_run(agmm_plan_t plan, const void* const* x_shards, const void* y, void* o, int my_id,
                       void* workspace, void* stream) {
  agmm_status_t st = check_run_args(plan, x_shards, y, o, my_id, workspace, agmm_workspace_bytes(plan, 0));
  if (st != AGMM_OK) return st;
  return launch_fused(plan, x_shards, y, o, my_id, workspace, static_cast<uint8_t*>(workspace) + kStatusBytes,
                      static_cast<cudaStream_t>(stream));
}

agmm_status_t agmm_run_gather(agmm_plan_t plan, const void* const* x_shards, const void* y, void* o, void* xcat,
                              int my_id, void* workspace, void* stream) {
  agmm_status_t st = check_run_args(plan, x_shards, y, o, my_id, workspace, agmm_workspace_bytes(plan, 0));
  if (st != AGMM_OK) return st;
  if (!xcat) return fail(AGMM_ERR_INVALID_ARG, "xcat is NULL");
  if (!aligned16(xcat)) return fail(AGMM_ERR_ALIGNMENT, "xcat must be 16-byte aligned");
  const size_t gbytes = (size_t)plan->M() * plan->k * 2;
  const size_t xbytes = (size_t)plan->m_pd * plan->k * 2;
  for (int r = 0; r < plan->P; ++r)
    if (overlaps(x_shards[r], xbytes, xcat, gbytes)) return fail(AGMM_ERR_INVALID_ARG, "xcat overlaps a shard");
  if (overlaps(y, (size_t)plan->k * plan->n * 2, xcat, gbytes) ||
      overlaps(o, (size_t)plan->M() * plan->n * plan->out_elem, xcat, gbytes) ||
      overlaps(workspace, agmm_workspace_bytes(plan, 0), xcat, gbytes))
    return fail(AGMM_ERR_INVALID_ARG, "xcat overlaps Y, O or the workspace");
  return launch_fused(plan, x_shards, y, o, my_id, workspace, static_cast<uint8_t*>(workspace) + kStatusBytes,
                      static_cast<cudaStream_t>(stream), xcat);
}

agmm_status_t agmm_run_unfused(agmm_plan_t plan, const void* const* x_shards, const void* y, void* o,
                               int my_id, void* workspace, void* stream) {
  agmm_status_t st = check_run_args(plan, x_shards, y, o, my_id, workspace, agmm_workspace_bytes(plan, 1));
  if (st != AGMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan->P == 1)
    return launch_fused(plan, x_shards, y, o, 0, workspace, static_cast<uint8_t*>(workspace) + kStatusBytes, s);
  uint8_t* gathered = static_cast<uint8_t*>(workspace) + kStatusBytes;
  const size_t gbytes = gathered_bytes(plan);
  for (int r = 0; r < plan->P; ++r)
    if (overlaps(x_shards[r], (size_t)plan->m_pd * plan->k * 2, gathered, gbytes))
      return fail(AGMM_ERR_INVALID_ARG, "the workspace overlaps a shard");
  GatherParams g{};
  for (int r = 0; r < plan->P; ++r) g.src[r] = static_cast<const uint4*>(x_shards[r]);
  g.dst = reinterpret_cast<uint4*>(gathered);
  g.vec_per_shard = plan->m_pd * plan->k * 2 / 16;
  const int64_t want = (g.vec_per_shard + 4 * 256 - 1) / (4 * 256);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)plan->num_sms * 8 / plan->P + 1));
  cudaError_t e = launch_gather_kernel(g, plan->P, blocks, s);
  if (e != cudaSuccess) return fail_cuda(e, "gather kernel launch");
  const void* one[1] = {gathered};
  return launch_fused(plan->sub, one, y, o, 0, workspace, gathered + gbytes, s);
}

agmm_status_t agmm_run_host(agmm_plan_t plan, const void* const* x_host, const void* y_host, void* o_host,
                            void* const* x_dev, void* y_dev, void* o_dev, int my_id, void* workspace,
                            void* stream) {
  if (!plan || !x_host || !y_host || !o_host || !x_dev)
    return fail(AGMM_ERR_INVALID_ARG, "a pointer argument is NULL");
  for (int r = 0; r < plan->P; ++r)
    if (!x_host[r] || !x_dev[r]) return fail(AGMM_ERR_INVALID_ARG, "a shard pointer is NULL");
  agmm_status_t st = check_run_args(plan, const_cast<const void* const*>(x_dev), y_dev, o_dev, my_id, workspace,
                                    agmm_workspace_bytes(plan, 0));
  if (st != AGMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xbytes = (size_t)plan->m_pd * plan->k * 2;
  cudaError_t e;
  for (int r = 0; r < plan->P; ++r)
    if ((e = cudaMemcpyAsync(x_dev[r], x_host[r], xbytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return fail_cuda(e, "shard upload");
  if ((e = cudaMemcpyAsync(y_dev, y_host, (size_t)plan->k * plan->n * 2, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return fail_cuda(e, "Y upload");
  st = launch_fused(plan, const_cast<const void* const*>(x_dev), y_dev, o_dev, my_id, workspace,
                    static_cast<uint8_t*>(workspace) + kStatusBytes, s);
  if (st != AGMM_OK) return st;
  if ((e = cudaMemcpyAsync(o_host, o_dev, (size_t)plan->M() * plan->n * plan->out_elem, cudaMemcpyDeviceToHost,
                           s)) != cudaSuccess)
    return fail_cuda(e, "O download");
  return AGMM_OK;
}

agmm_status_t agmm_query_status(agmm_plan_t plan, void* workspace, void* stream) {
  (void)plan;
  if (!workspace) return fail(AGMM_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e, "stream synchronize");
  int words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if ((e = cudaMemcpy(words, workspace, sizeof words, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e, "status read");
  if (words[0] == 0) return AGMM_OK;
  if ((e = cudaMemset(workspace, 0, sizeof words)) != cudaSuccess) return fail_cuda(e, "status clear");
  static const char* roles[] = {"?", "producer", "mma", "epilogue", "drain", "store"};
  const char* role = (words[1] >= 1 && words[1] <= 5) ? roles[words[1]] : roles[0];
  return fail(words[0] == AGMM_ERR_TIMEOUT ? AGMM_ERR_TIMEOUT : AGMM_ERR_CUDA,
              std::string("device wait ran out in the ") + role + " role (stage " + std::to_string(words[2]) +
                  ", tile " + std::to_string(words[3]) + "; detail " + std::to_string(words[4]) + " " +
                  std::to_string(words[5]) + " " + std::to_string(words[6]) + " " + std::to_string(words[7]) + ")");
}

size_t agmm_trace_bytes(agmm_plan_t plan) {
  if (!plan) return 0;
  const size_t ctas = (size_t)plan->grid.x * plan->grid.y * plan->grid.z;
  return ctas * kTraceSlots * sizeof(uint64_t);
}

agmm_status_t agmm_set_trace(agmm_plan_t plan, void* trace, size_t bytes) {
  if (!plan) return fail(AGMM_ERR_INVALID_ARG, "plan is NULL");
  if (trace == nullptr) {
    plan->params.trace = nullptr;
    return AGMM_OK;
  }
  if (bytes < agmm_trace_bytes(plan)) return fail(AGMM_ERR_INVALID_ARG, "trace buffer too small");
  if ((reinterpret_cast<uintptr_t>(trace) & 7u) != 0) return fail(AGMM_ERR_ALIGNMENT, "trace buffer not 8-byte aligned");
  plan->params.trace = static_cast<uint64_t*>(trace);
  return AGMM_OK;
}

agmm_status_t agmm_plan_info(agmm_plan_t plan, agmm_plan_info_t* info) {
  if (!plan || !info) return fail(AGMM_ERR_INVALID_ARG, "NULL argument");
  info->path = plan->key.path;
  info->box_rows = plan->box_rows;
  info->whole_shards = plan->whole_shards;
  info->chunks = plan->total_chunks;
  info->tile_m = kTileM;
  info->tile_n = plan->mma_n;
  info->tile_k = kTileK;
  info->stages = plan->stages;
  info->splits = plan->splits;
  info->num_tiles = plan->num_tiles;
  info->num_ctas = (int)(plan->grid.x * plan->grid.y * plan->grid.z);
  info->group_m = plan->group_m;
  info->num_sms = plan->num_sms;
  info->smem_bytes = plan->smem_bytes;
  info->row_groups = plan->key.path == kPathSwap ? plan->row_groups : 1;
  info->cluster_m = plan->key.path == kPathSwap ? 1 : plan->key.cm;
  info->cta_pair = plan->key.pair ? 1 : 0;
  info->stream_k_tiles = plan->key.path == kPathSwap ? 0 : plan->sk_tiles;
  info->dsmem_reduce = plan->key.path == kPathSwap && plan->swap_dsmem ? 1 : 0;
  info->config_source = plan->config_source;
  info->k_blocks_per_stage = plan->atoms;
  return AGMM_OK;
}

agmm_status_t agmm_plan_preview(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                                int rhs_transpose, const agmm_tile_config_t* config, int num_sms,
                                agmm_plan_info_t* info) {
  if (!info) return fail(AGMM_ERR_INVALID_ARG, "info is NULL");
  if (num_sms < 1 || num_sms > 4096) return fail(AGMM_ERR_INVALID_ARG, "num_sms must be in [1, 4096]");
  agmm_status_t st = validate_shape(P, m_per_device, k, n, (int)dtype, rhs_transpose);
  if (st != AGMM_OK) return st;
  if ((st = validate_config(config)) != AGMM_OK) return st;
  agmm_plan_s pl;
  pl.P = P;
  pl.m_pd = m_per_device;
  pl.k = k;
  pl.n = n;
  pl.dtype = dtype;
  pl.rhs_t = rhs_transpose;
  pl.num_sms = num_sms;
  pl.key.y_kmajor = rhs_transpose != 0;
  pl.key.out_f32 = dtype == AGMM_BF16_F32OUT || dtype == AGMM_F16_F32OUT;
  pl.f16 = dtype == AGMM_F16 || dtype == AGMM_F16_F32OUT;
  const ResolvedConfig rc = resolve_config(&pl, config);
  st = choose_tiles(&pl, rc.cfg, rc.strict);
  if (st != AGMM_OK) return st;
  // the row path's grid as if every cluster were resident
  if (pl.key.path == kPathRows) size_rows_grid(&pl, num_sms / pl.key.cm);
  info->path = pl.key.path;
  info->box_rows = pl.box_rows;
  info->whole_shards = pl.whole_shards;
  info->chunks = pl.total_chunks;
  info->tile_m = kTileM;
  info->tile_n = pl.mma_n;
  info->tile_k = kTileK;
  info->stages = pl.stages;
  info->splits = pl.splits;
  info->num_tiles = pl.num_tiles;
  info->num_ctas = pl.key.path == kPathSwap ? pl.splits * pl.num_n_tiles * pl.row_groups
                                            : (int)(pl.grid.x * pl.grid.y * pl.grid.z);
  info->group_m = pl.group_m;
  info->num_sms = num_sms;
  info->smem_bytes = pl.smem_bytes;
  info->row_groups = pl.key.path == kPathSwap ? pl.row_groups : 1;
  info->cluster_m = pl.key.path == kPathSwap ? 1 : pl.key.cm;
  info->cta_pair = pl.key.pair ? 1 : 0;
  info->stream_k_tiles = pl.key.path == kPathSwap ? 0 : pl.sk_tiles;
  info->dsmem_reduce = pl.key.path == kPathSwap && pl.swap_dsmem ? 1 : 0;
  info->config_source = rc.source;
  info->k_blocks_per_stage = pl.atoms;
  return AGMM_OK;
}

agmm_status_t agmm_ring_chunks(int P, int64_t m_per_device, int my_id, int box_rows, int whole_shards,
                               int32_t* shard, int64_t* src_row, int64_t* out_row, int32_t* valid,
                               int64_t max_chunks, int64_t* n_chunks) {
  if (P < 1 || P > AGMM_MAX_SHARDS || m_per_device < 1 || my_id < 0 || my_id >= P || box_rows < 1 ||
      box_rows > 256 || !n_chunks || max_chunks < 0)
    return fail(AGMM_ERR_INVALID_ARG, "bad ring description arguments");
  if (whole_shards != 0 && whole_shards != 1) return fail(AGMM_ERR_INVALID_ARG, "whole_shards must be 0 or 1");
  const RingGeom g = make_ring_geom(P, m_per_device, my_id, box_rows, whole_shards);
  const int64_t total = ring_total_chunks(g);
  *n_chunks = total;
  for (int64_t c = 0; c < total && c < max_chunks; ++c) {
    const RingChunk ch = ring_chunk(g, c);
    if (shard) shard[c] = ch.shard;
    if (src_row) src_row[c] = ch.src_row;
    if (out_row) out_row[c] = ch.out_row;
    if (valid) valid[c] = ch.valid;
  }
  return AGMM_OK;
}

const char* agmm_status_string(agmm_status_t status) {
  switch (status) {
    case AGMM_OK: return "AGMM_OK";
    case AGMM_ERR_INVALID_ARG: return "AGMM_ERR_INVALID_ARG";
    case AGMM_ERR_UNSUPPORTED: return "AGMM_ERR_UNSUPPORTED";
    case AGMM_ERR_ALIGNMENT: return "AGMM_ERR_ALIGNMENT";
    case AGMM_ERR_CUDA: return "AGMM_ERR_CUDA";
    case AGMM_ERR_TIMEOUT: return "AGMM_ERR_TIMEOUT";
    case AGMM_ERR_NOMEM: return "AGMM_ERR_NOMEM";
  }
  return "AGMM_ERR_UNKNOWN";
}

const char* agmm_last_error(void) { return g_last_error.c_str(); }

int agmm_version(void) { return AGMM_VERSION; }

}  // extern "C"
