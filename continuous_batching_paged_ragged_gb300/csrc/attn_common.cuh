// Definitions shared by the attention translation units: the per-pass workspace header, the prefill
// work-item record and the prefill launch entry.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kBS = 16;          // tokens per cache block
constexpr int kHeadsTile = 8;    // query heads per KV head handled by one decode MMA tile (G <= 8)

// Rows with at least this many new tokens (a prefill chunk) go to the tensor-core tile kernel; shorter
// rows (decode, short chunks) to the split-K decode kernel.  The choice depends on the row alone, so a
// row's result does not depend on the rest of the batch.
constexpr int kPrefillMinQlen = 16;
constexpr int kPrefillRows = 128;  // MMA rows of a prefill Q tile: (query position, query head) pairs
constexpr int kPrefillKeys = 128;  // keys per K/V tile (64 at head_dim 256, prefill_tile_keys)
constexpr int kPrefillBuckets = 1024;
// An item whose keys span more K/V tiles than this runs as two chunks of keys (split-KV) that the
// second chunk to finish merges, when its row alone cannot keep every CTA busy for the item's length; the
// split depends on the row (and the SM count) alone.
constexpr int kPrefillSplitTiles = 24;

// Query positions per prefill Q tile: the G query heads of a KV head are packed into the MMA rows.
__host__ __device__ constexpr int prefill_positions(int group) { return kPrefillRows / group; }
// Keys per prefill K/V tile: at head_dim 256 a Q tile's output takes 256 tensor memory columns, its scores the
// next 64 (a 128-key tile's would not fit beside them), and 64-key tiles keep the K/V rings in shared memory.
__host__ __device__ constexpr int prefill_tile_keys(int head_dim) { return head_dim == 256 ? 64 : kPrefillKeys; }

struct WsHeader {
  int32_t n_tasks;   // decode tasks of the pass
  int32_t work;      // dynamic decode tasks handed out so far (each CTA's first two are static)
  int32_t done;      // decode CTAs of the current launch that have finished
  int32_t n_items;   // prefill items of the pass
  int32_t pwork;     // dynamic prefill items handed out so far (each CTA's first is static)
  int32_t pdone;     // prefill CTAs of the current launch that have finished
  int32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// A prefill work entry: one KV head, up to prefill_item_positions(G, d) consecutive query positions of one
// row, all of its keys or one of two chunks of them.
//   x: row (block-table row)
//   y: KV head | positions << 8 | chunk << 20 | split << 21
//   z: first query token (packed)     w: keys visible to the item's first position, minus one
// Position i of the item attends causally to keys 0 .. w + i.  A split item's two entries share a slot
// (the partial results and the merge handshake).
__host__ __device__ constexpr int prefill_rec_y(int g, int npos, int chunk, int split) {
  return g | (npos << 8) | (chunk << 20) | (split << 21);
}

struct PrefillArgs {
  const CUtensorMap* kv_map;  // device copy is passed by value below; this one is host-side
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int4* items;
  const int32_t* items_slot;  // per work entry: the split item's slot, or -1
  int2* pf_sync;              // per slot: {chunks finished, first chunk's partial published}
  float2* pf_ml;              // per slot: [256 rows] (running max, running sum) of the first chunk
  float* pf_o;                // per slot and Q tile: [head_dim][128 rows] unnormalised output of the first chunk
  WsHeader* hdr;
  int32_t* err;
  int layer_row0_k, layer_row0_v;
  int max_blocks, num_q_heads, num_kv_heads, num_blocks, head_dim;
  int num_sms;
  int64_t max_items;
};

// Launch the prefill tile kernel for one layer (programmatic dependent launch on `stream`).
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// Whether the tile kernel serves this head shape (otherwise every row takes the decode path).
bool prefill_supported(int head_dim, int group);
// Query positions per prefill item (the Q tiles of one item share their K/V tiles).
int prefill_item_positions(int group, int head_dim);

}  // namespace pkv
