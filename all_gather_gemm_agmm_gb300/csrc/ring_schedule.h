// ring_schedule.h -- the bidirectional ring order of the all-gather matmul,
// as row "chunks" that one TMA box each brings into shared memory.
//
// Source: tpu_inference "all_gather_matmul.py", _all_gather_kernel.  Each
// shard is split into a left half of m_per_device // 2 rows
// (m_per_device_per_direction) and a right half of the remaining rows.  At
// ring step s (outer step s+1 of the Pallas grid) a device holds the left half
// that started at device (my_id + s) mod P -- left halves travel to the left
// neighbour -- and the right half that started at device (my_id - s) mod P.
// _do_o_local_copy writes them to output rows
//   left : m/2 * 2*((my_id + s) mod P)       ... i.e. rows of shard (my_id+s)
//   right: m/2 * (2*((my_id - s) mod P) + 1)  ... i.e. rows of shard (my_id-s)
// which is rank-order concatenation.
//
// On one GPU every shard is already resident, so the ring becomes the order in
// which row chunks are visited: step 0 takes shard my_id, step s the left half
// of shard (my_id+s) mod P and the right half of shard (my_id-s) mod P.  Each
// half is cut into chunks of box_rows rows (the last one ragged).
//
// Whole-shard mode (for shards whose halves are too small to fill a TMA box)
// keeps the ring's shard order at shard granularity: shards in the order the
// bidirectional ring first delivers them -- my_id, my_id+1, my_id-1, my_id+2,
// my_id-2, ... (mod P) -- each cut into chunks of box_rows rows.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define AGMM_HD __host__ __device__ __forceinline__
#else
#define AGMM_HD inline
#endif

namespace agmm {

struct RingGeom {
  int P;
  int my_id;
  int box_rows;   // rows per chunk (TMA box height)
  int chunks_l;   // chunks in a left half  = ceil(half_l / box_rows)
  int chunks_r;   // chunks in a right half = ceil(half_r / box_rows)
  int64_t m_pd;   // rows per shard
  int64_t half_l; // m_pd / 2 (floor): m_per_device_per_direction; 0 in whole-shard mode
  int whole;      // whole-shard mode
};

struct RingChunk {
  int shard;       // source shard
  int valid;       // rows of this chunk that belong to its half (<= box_rows)
  int64_t src_row; // first row inside the shard
  int64_t out_row; // first output row: shard * m_pd + src_row
};

AGMM_HD int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

AGMM_HD RingGeom make_ring_geom(int P, int64_t m_pd, int my_id, int box_rows, int whole = 0) {
  RingGeom g;
  g.P = P;
  g.my_id = my_id;
  g.box_rows = box_rows;
  g.m_pd = m_pd;
  g.whole = whole;
  g.half_l = whole ? 0 : m_pd / 2;
  g.chunks_l = (int)ceil_div64(g.half_l, box_rows);
  g.chunks_r = (int)ceil_div64(m_pd - g.half_l, box_rows);
  return g;
}

// Offset of the t-th shard the bidirectional ring delivers: 0, +1, -1, +2, ...
AGMM_HD int ring_first_visit(int my_id, int t, int P) {
  const int off = (t & 1) ? (t + 1) / 2 : -(t / 2);
  int s = (my_id + off) % P;
  return s < 0 ? s + P : s;
}

AGMM_HD int64_t ring_total_chunks(const RingGeom& g) {
  return (int64_t)g.P * (g.chunks_l + g.chunks_r);
}

// Chunk c of the ring-ordered sequence (0 <= c < ring_total_chunks(g) < 2^31;
// 32-bit index arithmetic keeps this cheap on the device).
AGMM_HD RingChunk ring_chunk(const RingGeom& g, int64_t c64) {
  const int c = (int)c64;
  const int per_step = g.chunks_l + g.chunks_r;
  const int s = c / per_step;
  const int w = c - s * per_step;
  RingChunk ch;
  int64_t seg_end;
  if (g.whole) {
    ch.shard = ring_first_visit(g.my_id, s, g.P);
    ch.src_row = (int64_t)w * g.box_rows;
    seg_end = g.m_pd;
  } else if (w < g.chunks_l) {
    ch.shard = g.my_id + s;
    if (ch.shard >= g.P) ch.shard -= g.P;
    ch.src_row = (int64_t)w * g.box_rows;
    seg_end = g.half_l;
  } else {
    ch.shard = g.my_id - s;
    if (ch.shard < 0) ch.shard += g.P;
    ch.src_row = g.half_l + (int64_t)(w - g.chunks_l) * g.box_rows;
    seg_end = g.m_pd;
  }
  const int64_t rem = seg_end - ch.src_row;
  ch.valid = (int)(rem < g.box_rows ? rem : g.box_rows);
  ch.out_row = (int64_t)ch.shard * g.m_pd + ch.src_row;
  return ch;
}

// Rows the chunk sequence occupies when every chunk is padded to box_rows.
AGMM_HD int64_t ring_padded_rows(const RingGeom& g) { return ring_total_chunks(g) * g.box_rows; }

}  // namespace agmm
