// ta_layout.h -- definitions shared by the host launcher and the kernels:
// tile sizes, the workspace layout and the records the plan kernel leaves
// for the attention kernel.
#pragma once

#include <cstddef>
#include <cstdint>

namespace ta {

// A Q tile is kBlockM packed rows: floor(kBlockM / g) q rows times the g q
// heads of one kv head (row index = q_row * g + head_in_group, the packing
// of the "Q_load" block of the page "tree_attn.py"), attended against kv
// tiles of kBlockN columns.  A work unit is two consecutive Q tiles of one
// (sequence, kv head) -- tile A, then tile B -- that stream the same K/V
// tiles through one CTA.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kKvBoxRows = 128;  // kv rows per TMA box (one box per kv tile)
constexpr int kMaxGroup = 128;   // largest supported h_q / h_kv
constexpr int kPageSize = 16;    // kv slots per page of a paged KV cache
constexpr int kTilesPerUnit = 2; // Q tiles per work unit

// Tile classes computed by the plan kernel for each (Q tile, kv tile); a kv
// tile's class byte holds tile A's class in bits 0-1 and tile B's in 2-3.
constexpr uint8_t kTileEmpty = 0;    // no (row, column) pair visible: skipped
constexpr uint8_t kTilePartial = 1;  // some visible: the mask is evaluated per element
constexpr uint8_t kTileFull = 2;     // every valid row sees every column: no mask

// Device status bits (WsHeader::error).
constexpr unsigned int DEVERR_TIMEOUT = 1u;     // a bounded wait expired
constexpr unsigned int DEVERR_BAD_INDPTR = 2u;  // index arrays violate the layout rules

constexpr int kCostBuckets = 512;  // LPT ordering resolution (tiles per item)

struct WsHeader {
  unsigned int queue_head;  // next work item (attention kernel)
  unsigned int queue_done;  // attention CTAs finished (the last one resets the queue)
  unsigned int error;       // DEVERR_* bits, cleared by tree_attn_device_status
  unsigned int num_pairs;   // (sequence, unit) pairs found by the plan kernel
  unsigned int num_items;   // work records * h_kv, 0 if the index arrays are invalid
  unsigned int reserved;    // unused (zero)
  unsigned int pad[10];
};
static_assert(sizeof(WsHeader) == 64, "header size");

// Everything the attention kernel needs about one (sequence, unit) pair --
// or, with split-KV, about one chunk of a pair's kv tiles -- written by the
// plan kernel so that a work item costs one 64-byte load.
struct ItemRec {
  int32_t part;       // split-KV: this chunk's partial-state slot (-1: not split)
  int32_t r0;         // the unit's first q row within its sequence
  int32_t q_row0;     // global index of the unit's first q row
  int32_t nq;         // q rows of the sequence inside this unit (1 .. 2R)
  int32_t qo, kv;     // q rows / kv rows of the sequence (tree start = kv - tl)
  int32_t tl;         // tree nodes
  int32_t tile_lo;    // first kv tile of this item's range (0 unless split)
  int32_t kv_base;    // kv_indptr[b]
  int32_t tree_base;  // mn_indptr[b]
  int32_t n_tiles;    // kv tiles of this item's range non-empty for tile A or B
  int32_t class_off;  // byte offset of the pair's kv-tile class bytes (16-aligned)
  int32_t kvt;        // kv tiles of the sequence
  int32_t n_a, n_b;   // of those, the ones non-empty for tile A / for tile B
  uint32_t cls;       // if kvt <= kInlineTiles: tile j's class byte in bits 4j .. 4j+3
};
constexpr int kInlineTiles = 8;

// Class byte of kv tile j of a record (inline bits for short sequences, else
// the class table).
__host__ __device__ inline int tile_class(const ItemRec& r, const uint8_t* classes, int j) {
  if (r.kvt <= kInlineTiles) return (r.cls >> (4 * j)) & 15;
  return classes[r.class_off + j];
}
static_assert(sizeof(ItemRec) == 64, "item record size");

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// q rows per Q tile for group size g, and per work unit.
inline int rows_per_item(int g) { return kBlockM / g; }
inline int rows_per_unit(int g) { return kTilesPerUnit * rows_per_item(g); }

constexpr int kMaxChunks = 16;  // split-KV: chunks per (sequence, unit) at most
// split-KV: the least kv tiles of a chunk when the chunk length is chosen
// automatically (a chunk's fixed costs -- its Q tiles, its partial state
// written and read back -- stay small against its kv tiles)
constexpr int kMinChunkTiles = 8;

struct WsLayout {
  int64_t max_pairs;    // upper bound on (sequence, unit) pairs
  int64_t max_records;  // upper bound on work records (pairs, or pair chunks when split)
  int64_t class_bytes;  // bound on the class table
  size_t off_sorted, off_classes, off_rope, off_krot;
  size_t off_merge, off_part_o, off_part_lse;   // split-KV only (else empty)
  size_t total;
};

// Workspace layout for the given sizes (all offsets 256-byte aligned):
//   header | ItemRec sorted[max_records] (longest-first order)
//   | uint8 classes[]
//   and with RoPE: | float2 rope_cs[total_kv][head_dim / 2] (cos / sin of
//                    every kv token's position; q rows read their own node's)
//                  | rotated k [total_kv][h_kv][head_dim] (storage dtype)
//   and with split-KV: | int4 merge[max_pairs] (per pair: q_row0, nq, chunks,
//                        first record) | float part_o[max_records][h_kv][2 x 128][d]
//                        | float part_lse[max_records][h_kv][2 x 128]
//                        (packed rows of tile A, then of tile B)
// ``max_chunks`` (1..kMaxChunks) caps the split-KV chunks of a pair; 1 lays
// out the unsplit workspace.
inline WsLayout make_ws_layout(int64_t batch, int64_t total_q, int64_t total_kv, int g,
                               int h_kv, int head_dim, bool rotary, int max_chunks = 1) {
  WsLayout L{};
  const int64_t U = rows_per_unit(g);
  const bool split = max_chunks > 1;
  L.max_pairs = ceil_div(total_q, U) + batch;
  L.max_records = L.max_pairs * (split ? max_chunks : 1);
  L.class_bytes = L.max_pairs * round_up(ceil_div(total_kv, kBlockN), 16);
  size_t off = 256;
  L.off_sorted = off;
  off += round_up(L.max_records * (int64_t)sizeof(ItemRec), 256);
  L.off_classes = off;
  off += round_up(L.class_bytes, 256);
  L.off_rope = off;
  if (rotary) off += round_up(total_kv * (int64_t)(head_dim / 2) * 8, 256);
  L.off_krot = off;
  if (rotary) off += round_up(total_kv * (int64_t)h_kv * head_dim * 2, 256);
  L.off_merge = off;
  if (split) off += round_up(L.max_pairs * 16, 256);
  L.off_part_o = off;
  if (split)
    off += round_up(L.max_records * h_kv * kTilesPerUnit * kBlockM * (int64_t)head_dim * 4, 256);
  L.off_part_lse = off;
  if (split) off += round_up(L.max_records * h_kv * kTilesPerUnit * kBlockM * 4, 256);
  L.total = off;
  return L;
}

}  // namespace ta
