/*
 * agmm.h -- C ABI of the GB300 (sm_103a) fused all-gather matmul.
 *
 * Operation (tpu_inference "all_gather_matmul.py", all_gather_matmul
 * docstring and _all_gather_kernel; AllGather-GEMM tutorial,
 * torch_allgather_gemm):
 *
 *     O = concat(X_0, ..., X_{P-1}) @ Ycan
 *     Ycan = Y            (rhs_transpose == 0, Y stored [k, n])
 *          = transpose(Y) (rhs_transpose != 0, Y stored [n, k])
 *
 * On one GPU the P "ranks" of the pages are P separate shard buffers
 * X_r [m_per_device, k] in the same device memory.  The kernel reads them
 * through a per-shard TMA descriptor table in the pages' bidirectional ring
 * order (ring step s consumes the left half of shard (my_id + s) mod P and the
 * right half of shard (my_id - s) mod P, _do_o_local_copy), accumulates in
 * float32 in tensor memory (preferred_element_type=float32 in _do_mxu) and
 * writes row block r of O at rows [r*m_per_device, (r+1)*m_per_device).  The
 * gathered left-hand side is never written to device memory by agmm_run.
 *
 * Layout: every matrix is dense row-major bf16 (AGMM_BF16*) or fp16
 * (AGMM_F16*; the AllGather-GEMM tutorial's float16 tensors).  O is
 * [P*m_per_device, n] in the input type, or float32 (the *_F32OUT types).
 *
 * Ownership: the caller owns every device buffer (shards, Y, O, workspace)
 * and the stream.  A plan owns host memory only.
 *
 * Errors: every call returns a status; nothing throws across this boundary.
 * agmm_last_error() gives a message for the last failing call of the calling
 * thread.  Runs are asynchronous on the given stream; a device-side timeout
 * is reported later through agmm_query_status().
 *
 * Threads: a plan caches tensor-map descriptors and is not safe for
 * concurrent use from several host threads.  Distinct plans are independent.
 */
#ifndef AGMM_H_
#define AGMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AGMM_VERSION 1
#define AGMM_MAX_SHARDS 8 /* per-peer descriptor tables are capped at 8 peers
                             (jax mosaic gpu launch_context.py, _get_tma_desc) */

typedef enum {
  AGMM_OK = 0,
  AGMM_ERR_INVALID_ARG = 1, /* a size, index or pointer is out of range         */
  AGMM_ERR_UNSUPPORTED = 2, /* no sm_103a device, or a shape this build rejects */
  AGMM_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned          */
  AGMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed                */
  AGMM_ERR_TIMEOUT = 5,     /* a device-side wait ran past its limit            */
  AGMM_ERR_NOMEM = 6        /* host allocation failed                           */
} agmm_status_t;

typedef enum {
  AGMM_BF16 = 0,        /* bf16 inputs, float32 accumulation, bf16 output    */
  AGMM_BF16_F32OUT = 1, /* bf16 inputs, float32 accumulation, float32 output */
  AGMM_F16 = 2,         /* fp16 inputs, float32 accumulation, fp16 output    */
  AGMM_F16_F32OUT = 3   /* fp16 inputs, float32 accumulation, float32 output */
} agmm_dtype_t;

typedef struct agmm_plan_s* agmm_plan_t;

/* What the planner chose (for tests, tracing and the benchmark). */
typedef struct {
  int path;          /* 0: row tiles (MMA M spans gathered rows);
                        1: swapped tiles (MMA M spans n, gathered rows are MMA N) */
  int box_rows;      /* rows per X tensor-map box (a "chunk")                    */
  int whole_shards;  /* 0: chunks follow the ring's left/right half split;
                        1: chunks cover whole shards in ring first-visit order   */
  int chunks;        /* chunks in the whole ring-ordered row sequence            */
  int tile_m;        /* MMA M                                                    */
  int tile_n;        /* MMA N                                                    */
  int tile_k;        /* k elements per k block (one TMA box of X rows)           */
  int stages;        /* shared-memory pipeline depth                             */
  int splits;        /* k splits reduced inside a thread-block cluster           */
  int num_tiles;     /* output tiles                                             */
  int num_ctas;      /* CTAs launched by agmm_run                                */
  int group_m;       /* row tiles per raster group                               */
  int num_sms;       /* SMs of the planned device                                */
  size_t smem_bytes; /* dynamic shared memory per CTA                            */
  int row_groups;    /* swapped tiles: groups of chunks, one MMA N each (else 1) */
  int cluster_m;     /* row tiles: CTAs per cluster sharing a Y tile (else 1)    */
  int cta_pair;      /* row tiles: 1 when a cluster multiplies as a CTA pair
                        (always so for a two-CTA cluster)                       */
  int stream_k_tiles;/* row tiles: output tiles whose k blocks are shared        */
  int dsmem_reduce;  /* swapped tiles: 1 when k-split partials go through
                        distributed shared memory, 0 through device memory     */
  int config_source; /* 0: the planner's rules; 1: the tuned table (an entry
                        measured for this exact shape); 2: a caller's config or
                        AGMM_* environment overrides set at least one field     */
  int k_blocks_per_stage; /* k blocks per pipeline stage: 1, or 2 where two fit
                        three times (one barrier hand-off per two blocks)       */
} agmm_plan_info_t;

/*
 * Tile configuration for agmm_plan_config and agmm_plan_preview.
 * all_gather_matmul (tpu_inference "all_gather_matmul.py") takes its block
 * sizes bn and bk as optional arguments and fills the missing ones from a
 * table of tuned sizes keyed by shape, dtype and mesh size
 * (get_tuned_block_sizes); this struct is that argument.  Every field left at
 * 0 (AGMM_CFG_AUTO) is chosen by the planner: from the tuned table when it
 * holds an entry for the exact (P, m_per_device, k, n, rhs_transpose, input
 * type), else by its rules.  On/off fields take AGMM_CFG_OFF or
 * AGMM_CFG_ON.  Fields that belong to the other tile path are ignored.
 */
#define AGMM_CFG_AUTO 0
#define AGMM_CFG_OFF 1
#define AGMM_CFG_ON 2
typedef struct {
  int path;         /* 1: row tiles; 2: swapped tiles (needs every gathered row,
                       padded to box heights, within 256)                     */
  int chunks;       /* 1: the ring's half-shard chunks; 2: whole-shard chunks */
  int box_rows;     /* X rows per TMA box: 8, 16, 32, 64 or 128               */
  int tile_n;       /* row tiles: MMA N, 128 or 256 (n must be a multiple)    */
  int cluster_m;    /* row tiles: 1, or 2 neighbouring row tiles per cluster,
                       which multiply as one cta_group::2 pair, each CTA
                       loading half of the shared Y tile                     */
  int cta_pair;     /* row tiles: on = two-CTA clusters (needs cluster_m 2 or
                       auto); off = one-CTA clusters (a two-CTA cluster is
                       always a pair, so cluster_m 2 with cta_pair off is
                       AGMM_ERR_UNSUPPORTED)                                  */
  int stages;       /* pipeline stages, 2..8: an upper bound that shared
                       memory may lower (a swapped k-split reduction through
                       distributed shared memory takes room for its receive
                       buffer)                                                */
  int group_m;      /* row tiles: row-tile (pairs) per raster group, >= 1     */
  int stream_k;     /* row tiles: on = share a ragged last wave's k blocks
                       (stream-K); auto = the same unless that wave fills at
                       least two thirds of the clusters; off = whole tiles   */
  int row_groups;   /* swapped tiles: groups of chunks (1, 2, 4, ...), each a
                       separate MMA N; no group may be empty                  */
  int splits;       /* swapped tiles: k splits per cluster, 1..16: an upper
                       bound, lowered until every cluster is resident         */
  int dsmem_reduce; /* swapped tiles: on = reduce the k splits through
                       distributed shared memory instead of device memory     */
  int tuned_table;  /* off = ignore the tuned table for this plan             */
} agmm_tile_config_t;

/*
 * agmm_plan -- validate a problem and choose tiles for the current device.
 *
 * Arguments follow all_gather_matmul's problem statement: P shards (the mesh
 * axis size), m_per_device rows per shard, contraction length k, n output
 * columns (the page's n_per_device), dtype, rhs_transpose.
 *
 * Accepted: 1 <= P <= 8; m_per_device >= 1; k >= 128 and k % 128 == 0;
 * n >= 128 and n % 128 == 0 (validate_inputs' k and n rules); P*m_per_device*k,
 * k*n and P*m_per_device*n below 2^40 elements.  validate_inputs' rules that
 * m be a multiple of 16*P are relaxed: any m_per_device >= 1 is accepted and
 * an odd shard is split as floor(m/2) left rows and the rest right rows.
 *
 * Returns AGMM_ERR_INVALID_ARG (with *out_plan = NULL) for a rejected shape,
 * AGMM_ERR_UNSUPPORTED when the current device is not sm_103, AGMM_ERR_CUDA
 * when no device can be queried, AGMM_ERR_NOMEM on host allocation failure.
 * Shape validation happens before any CUDA call.
 */
agmm_status_t agmm_plan(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                        int rhs_transpose, agmm_plan_t* out_plan);

/*
 * agmm_plan_config -- agmm_plan with a tile configuration.  Fields of
 * `config` that are set take precedence over the AGMM_* environment
 * overrides, which take precedence over the tuned table.  NULL behaves like
 * agmm_plan.  Returns AGMM_ERR_INVALID_ARG for a field outside its range, and
 * AGMM_ERR_UNSUPPORTED when a set field cannot hold for this shape (swapped
 * tiles for more than 256 padded rows, tile_n not dividing n, a CTA pair
 * without a 2-CTA cluster or a 2-CTA cluster without the pair, an empty row
 * group, a box height whose swapped
 * rows exceed 256).
 */
agmm_status_t agmm_plan_config(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                               int rhs_transpose, const agmm_tile_config_t* config, agmm_plan_t* out_plan);

/* Release a plan.  NULL is a no-op. */
void agmm_destroy(agmm_plan_t plan);

/*
 * Bytes of device workspace agmm_run (unfused == 0) or agmm_run_unfused
 * (unfused != 0) needs.  The first 256 bytes hold the device status words;
 * the unfused path adds the gathered [P*m_per_device, k] buffer (input type) at
 * offset 256.  The workspace must be zero-filled before its first use and
 * must not be shared by runs that overlap on the device.  Returns 0 for NULL.
 * After agmm_query_status has reported AGMM_ERR_TIMEOUT, zero-fill the whole
 * workspace again before its next use: a run that gave up may leave split
 * counters behind it.
 */
size_t agmm_workspace_bytes(agmm_plan_t plan, int unfused);

/*
 * agmm_run -- the fused all-gather matmul, asynchronous on `stream`.
 *
 *   x_shards  host array of P device pointers; shard r is [m_per_device, k]
 *   y         device pointer, [k, n] or (rhs_transpose) [n, k]
 *   o         device pointer, [P*m_per_device, n]; must not overlap an input
 *   my_id     this rank's index in [0, P): ring step 0 starts at shard my_id
 *   workspace device pointer to agmm_workspace_bytes(plan, 0) bytes; must
 *             not overlap O, Y or a shard
 *   stream    a cudaStream_t (NULL: the legacy default stream)
 *
 * Every device pointer must be 16-byte aligned (TMA: global addresses and
 * strides are multiples of 16 bytes).  The result does not depend on my_id.
 * Returns AGMM_ERR_INVALID_ARG / AGMM_ERR_ALIGNMENT for bad arguments (nothing
 * is launched), AGMM_ERR_CUDA if the launch fails.
 */
agmm_status_t agmm_run(agmm_plan_t plan, const void* const* x_shards, const void* y, void* o,
                       int my_id, void* workspace, void* stream);

/*
 * agmm_run_gather -- agmm_run that also writes the gathered left-hand side.
 *
 * Source: tpu_inference "all_gather_matmul.py", the module's note on
 * splitting a large n (one all-gather matmul returns its output block and
 * the gathered x; the next block is then a plain matmul of that x), and the
 * kernel's x scratch output, which holds the shards a device received.
 *
 * Same arguments and result as agmm_run, plus
 *   xcat  device pointer to [P*m_per_device, k] elements of the input type,
 *         row-major, 16-byte aligned, caller-owned; on return (stream order)
 *         it holds concat(X_0, ..., X_{P-1}) in rank order, bit for bit.
 * Each (rows, k block) piece is stored by one of the CTAs that load it: n
 * tile t stores the k blocks in the t-th share of the k
 * range, so the gathered rows are written once, never read back, and the
 * store work is spread over all n tiles.  On row tiles the epilogue warps of
 * each CTA copy their rows' share from the shards while the tile's main loop
 * runs; on swapped tiles the MMA thread stores the landed boxes.  xcat
 * must not overlap the shards, Y, O or the workspace (AGMM_ERR_INVALID_ARG).
 * The workspace is agmm_workspace_bytes(plan, 0) bytes, as for agmm_run.
 */
agmm_status_t agmm_run_gather(agmm_plan_t plan, const void* const* x_shards, const void* y, void* o, void* xcat,
                              int my_id, void* workspace, void* stream);

/*
 * agmm_run_unfused -- the decomposed comparison path: a gather kernel copies
 * shard r to rows [r*m_per_device, (r+1)*m_per_device) of a scratch buffer in
 * the workspace (the decomposed approach of the AllGather-GEMM tutorial), then
 * the same tensor-core GEMM runs on it as a single shard.  Same arguments and
 * result as agmm_run; workspace is agmm_workspace_bytes(plan, 1) bytes.
 */
agmm_status_t agmm_run_unfused(agmm_plan_t plan, const void* const* x_shards, const void* y,
                               void* o, int my_id, void* workspace, void* stream);

/*
 * agmm_run_unfused_noalloc -- agmm_run_unfused without a caller workspace and
 * without allocating device memory.  The pages have no counterpart; this is a
 * convenience of this library for callers that cannot allocate at the point
 * where they run the product: code under a framework allocator that has
 * reserved the device's memory for itself (a cudaMalloc of its own there can
 * fail or fragment that pool), and latency-critical loops that cannot afford
 * cudaMalloc's and cudaFree's implicit device synchronisation.
 *
 * The scratch is one file-scope device array of AGMM_STATIC_SCRATCH_BYTES (64
 * MiB) that every GPU loading this library holds until the process exits.  A
 * problem whose agmm_workspace_bytes(plan, 1) exceeds it is rejected with
 * AGMM_ERR_INVALID_ARG (nothing is launched).  The first call on a device,
 * with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for later calls on that device: make
 * that first call before any stream capture, and note that a device reset
 * (cudaDeviceReset) invalidates the kept address, so no call may follow a
 * reset in the same process.  Each call clears the scratch's status words and
 * counters on `stream`, then gathers and multiplies; no call allocates or
 * frees memory.  All calls share the one array, which keeps the last call's
 * contents: calls that overlap on the device (different streams without
 * ordering) race and corrupt each other.  Device-side wait timeouts of these
 * calls are recorded in the shared scratch and are not reported to the
 * caller.  Arguments, alignment rules and result are those of agmm_run.
 */
#define AGMM_STATIC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB */
agmm_status_t agmm_run_unfused_noalloc(agmm_plan_t plan, const void* const* x_shards, const void* y,
                                       void* o, int my_id, void* stream);

/*
 * agmm_run_host -- agmm_run from host memory: copies each host shard to
 * x_dev[r] and the host Y to y_dev, runs, and copies O back to o_host, all
 * asynchronously on `stream` (host buffers should be pinned for overlap; the
 * caller synchronizes before reading o_host).  Device buffers as in agmm_run.
 */
agmm_status_t agmm_run_host(agmm_plan_t plan, const void* const* x_host, const void* y_host,
                            void* o_host, void* const* x_dev, void* y_dev, void* o_dev, int my_id,
                            void* workspace, void* stream);

/*
 * Synchronize `stream`, read the device status words in `workspace` and
 * clear them.  Returns AGMM_OK, AGMM_ERR_TIMEOUT if a kernel gave up on a
 * wait since the last query, or AGMM_ERR_CUDA if the stream reports an error.
 */
agmm_status_t agmm_query_status(agmm_plan_t plan, void* workspace, void* stream);

/*
 * Optional device trace: after agmm_set_trace(plan, buf, bytes) every
 * agmm_run of this plan writes, per CTA, 16 unsigned 64-bit slots to the
 * device buffer `buf` (agmm_trace_bytes(plan) bytes, 8-byte aligned): %globaltimer
 * nanoseconds (the stamps themselves cost a few hundred cycles each) at
 * kernel entry (0), after set-up (1), first and last TMA issue
 * (2, 3), first operand arrival at the MMA thread (4), last MMA commit (5),
 * first accumulator seen by the epilogue (6), rows-path epilogue done (7),
 * swap-path reduction barriers (8, 9), reduction stored (10), exit (11), plus
 * the SM id (12) and cluster rank (13).  On the row path slots 9, 10, 14 and
 * 15 instead hold SM clock cycles spent blocked: epilogue waiting for an
 * accumulator (9), producer waiting for a free stage (10), MMA thread waiting
 * for operands (14) and for a free accumulator (15).  Pass NULL to switch it
 * off.  The buffer stays owned by the caller and must outlive the runs that
 * use it.
 */
size_t agmm_trace_bytes(agmm_plan_t plan);
agmm_status_t agmm_set_trace(agmm_plan_t plan, void* trace, size_t bytes);

/* Fill *info with the plan's choices. */
agmm_status_t agmm_plan_info(agmm_plan_t plan, agmm_plan_info_t* info);

/*
 * agmm_plan_preview -- the tile choice agmm_plan would start from on a device
 * with num_sms SMs, computed on the host alone: no CUDA call, so it works
 * without a GPU (tests, tooling).  Same shape arguments and validation as
 * agmm_plan.  The device-dependent steps that agmm_plan adds afterwards are
 * absent: lowering the k splits until every cluster is resident, and
 * sizing the row path's persistent grid.  So `splits` is an upper bound and
 * `num_ctas` is the grid before them.  `config` (NULL allowed) acts as in
 * agmm_plan_config, with the same errors.  Returns AGMM_ERR_INVALID_ARG for a
 * NULL info or num_sms outside [1, 4096].
 */
agmm_status_t agmm_plan_preview(int P, int64_t m_per_device, int64_t k, int64_t n, agmm_dtype_t dtype,
                                int rhs_transpose, const agmm_tile_config_t* config, int num_sms,
                                agmm_plan_info_t* info);

/*
 * The ring-ordered row sequence, host side (no device needed).  For box
 * height box_rows the sequence is cut into chunks; chunk c covers rows
 * [src_row[c], src_row[c] + valid[c]) of shard shard[c], which land at rows
 * [out_row[c], out_row[c] + valid[c]) of O.  With whole_shards == 0 chunks
 * follow ring step s = 0..P-1: left half of shard (my_id+s) mod P, then right
 * half of shard (my_id-s) mod P.  With whole_shards == 1 each shard is one
 * run of chunks, shards in the order the bidirectional ring first delivers
 * them: my_id, my_id+1, my_id-1, my_id+2, ... (mod P); the planner uses this
 * when the halves are too small to fill a TMA box.  Writes at most max_chunks
 * entries and stores the full count in *n_chunks.
 */
agmm_status_t agmm_ring_chunks(int P, int64_t m_per_device, int my_id, int box_rows,
                               int whole_shards, int32_t* shard, int64_t* src_row,
                               int64_t* out_row, int32_t* valid, int64_t max_chunks,
                               int64_t* n_chunks);

/* Static description of a status code. */
const char* agmm_status_string(agmm_status_t status);

/* Detail of the calling thread's last failing call ("" if none). */
const char* agmm_last_error(void);

/* AGMM_VERSION of the loaded library. */
int agmm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AGMM_H_ */
