// Ragged paged GQA attention: per-pass plan, persistent split-K decode, cross-split merge.
//
// What is computed ("Continuous Batching Is Not a Bigger Batch", sections "What the scheduler does on one
// step" and "Where the batch size actually comes from"): for every query token of every row, causal
// attention over that row's keys in the paged cache, query head h reading KV head h / G (grouped-query
// attention), scores scaled by 1/sqrt(d).  "Static batching" ("Ragged batches", "Bottleneck, and what
// follows") is why the keys are read from blocks in place, with no padding to the widest row.
//
// How (GB300 design, not from the pages):
//  * plan_kernel (once per pass): per packed query token its row and causal context length, and the pass's
//    task list, largest first.  A task is one split of one (token, KV head): `split_blocks` consecutive
//    16-token blocks.  The split count of a token depends only on its own context, so results are
//    bit-identical whatever else is in the batch, whatever the row order and wherever the blocks sit
//    physically.  Rows with 16 or more new tokens become prefill work entries instead (longest first).
//  * decode_kernel (decode.cuh): persistent CTAs of four streaming warps, a combiner warp and a scheduler
//    warp.  The scheduler warp queues tasks (one static, the rest from a global counter); each task's
//    blocks are dealt to the streaming warps, which stream K and V through their own TMA rings and run
//    the G query heads' contraction on warp MMAs with an online softmax; the combiner warp folds the four
//    warps' shares and finishes the token (fp16 output, or a split partial, or the merge of all of them).
//    Its fp16-cache instances compile here, the 8-bit ones in decode_e4m3.cu.
//  * Cross-split merge: a token whose context fits one split gets its fp16 output from the decode
//    directly.  Otherwise each split leaves an unnormalised partial (m, l, o), and the CTA that finishes the
//    token's last split merges them with log-sum-exp weights inside the same launch (a separate merge
//    launch cost more than the merge: its CTAs cannot start until the decode's have left the SMs).
//    Tokens with more than 32 splits are merged by merge_kernel, launched behind the decode, which
//    spreads one token's merge over many CTAs.
//  * Prefill rows run on the tcgen05 tile kernel (prefill.cu) ahead of the decode; on the 8-bit cache
//    their blocks are first dequantized into an fp16 shadow in the workspace (dequant_prefill_rows_kernel).
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "attn_common.cuh"

#include "decode.cuh"

namespace pkv {


// ---------------------------------------------------------------------------------------------------
// Merge of tokens with more than kFusedMergeSplits splits (long contexts).  Grid (token, KV head, chunk
// of 32 partial elements of one head); 256 threads = 8 element threads (a float4 each) x 32 split groups.
// Split group sg folds splits sg, sg + 32, ... into a running (max, sum, o) with four splits' loads in
// flight; then the 32 groups' results are combined in group order.  A fixed order throughout, so the
// result depends only on the token's own splits.
// ---------------------------------------------------------------------------------------------------
struct MergeParams {
  const float* part_o;
  const float2* part_ml;
  const int32_t* tok_ctx;
  __half* out;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int split_blocks;
  int max_splits;
};

constexpr int kMergeGroups = 32;  // split groups of the long-context merge

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  __shared__ float4 s_o[kMergeGroups][8];
  __shared__ float2 s_ml[kMergeGroups];
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int t = blockIdx.x, g = blockIdx.y;
  const int ctx = __ldg(p.tok_ctx + t);
  const int e0 = blockIdx.z * 32;  // the chunk's first element: head e0 / D, dims e0 % D ..
  if (ctx <= 0 || e0 >= p.group * D) return;
  const int nblk = (ctx + kBS - 1) / kBS;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  if (nsplit <= kFusedMergeSplits) return;
  const int tid = threadIdx.x, e4 = tid & 7, sg = tid >> 3;
  const int h = e0 / D;
  const size_t sb = ((size_t)t * p.num_kv_heads + g) * p.max_splits;
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fold = [&](float2 ml, float4 o) {
    const float nM = fmaxf(M, ml.x);
    const float a = exp2f(M - nM), f = exp2f(ml.x - nM);
    M = nM;
    L = L * a + ml.y * f;
    acc.x = acc.x * a + o.x * f;
    acc.y = acc.y * a + o.y * f;
    acc.z = acc.z * a + o.z * f;
    acc.w = acc.w * a + o.w * f;
  };
  constexpr int U = 4;
  int s = sg;
  for (; s + (U - 1) * kMergeGroups < nsplit; s += U * kMergeGroups) {
    float2 ml[U];
    float4 o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t pi = (sb + s + u * kMergeGroups) * kHeadsTile;
      ml[u] = __ldcg(p.part_ml + pi + h);
      o[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + pi * D + e0) + e4);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) fold(ml[u], o[u]);
  }
  for (; s < nsplit; s += kMergeGroups) {
    const size_t pi = (sb + s) * kHeadsTile;
    fold(__ldcg(p.part_ml + pi + h), __ldcg(reinterpret_cast<const float4*>(p.part_o + pi * D + e0) + e4));
  }
  s_o[sg][e4] = acc;
  if (e4 == 0) s_ml[sg] = make_float2(M, L);
  __syncthreads();
  if (sg != 0) return;
  M = -INFINITY;
  L = 0.f;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q = 0; q < kMergeGroups; ++q)
    if (s_ml[q].x != -INFINITY) fold(s_ml[q], s_o[q][e4]);  // groups past nsplit hold nothing
  const float il = 1.f / L;
  const __half2 lo = __floats2half2_rn(acc.x * il, acc.y * il);
  const __half2 hi = __floats2half2_rn(acc.z * il, acc.w * il);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&lo);
  v.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.num_q_heads + (size_t)g * p.group) * D + e0 + 4 * e4) = v;
}

// ---------------------------------------------------------------------------------------------------
// Plan: token table, task list, counters.  One CTA (block-wide scans over the tokens).
// ---------------------------------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive prefix over warps
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  *total = warp_sums[(blockDim.x >> 5) - 1];
  return before + x - v;
}

struct PlanParams {
  const int32_t* context_lens;
  const int32_t* qsl;
  int num_seqs, num_tokens, max_ctx, split_blocks, num_kv_heads;
  int prefill_min_qlen;  // rows with at least this many new tokens become prefill items (0: none)
  int prefill_pos;       // query positions per prefill item
  int prefill_keys;      // keys per prefill K/V tile
  int prefill_ctas;      // CTAs of the prefill tile kernel at most (the SM count)
  int32_t* tok_row;
  int32_t* tok_ctx;
  int32_t* merge_cnt;
  int4* tasks;
  int4* items;
  int32_t* items_slot;
  int2* pf_sync;
  int max_slots;
  int32_t* pf_base;  // 8-bit cache: [num_seqs + 1] first fp16 shadow block of each row (rows that are not prefill
                     // rows hold none), then the total; or null
  WsHeader* hdr;
  int32_t* err;
};

__device__ __forceinline__ bool row_meta_ok(int q_len, int ctx, int max_ctx) {
  return q_len >= 1 && ctx >= q_len && ctx <= max_ctx;
}

// Prefill items of row b in plan order, one per position block: `fn(n, npos, first token, w)` with n the
// item's K/V tiles and w the keys visible to its first position minus one.
template <typename F>
__device__ __forceinline__ void for_row_items(const PlanParams& p, int b, F fn) {
  const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1), ctx = __ldg(p.context_lens + b);
  const int q_len = q1 - q0;
  if (p.prefill_min_qlen <= 0 || q_len < p.prefill_min_qlen || !row_meta_ok(q_len, ctx, p.max_ctx)) return;
  for (int qb = 0; qb * p.prefill_pos < q_len; ++qb) {
    const int npos = min(p.prefill_pos, q_len - qb * p.prefill_pos);
    const int w = ctx - q_len + qb * p.prefill_pos;
    fn((w + npos + p.prefill_keys - 1) / p.prefill_keys, npos, q0 + qb * p.prefill_pos, w);
  }
}

// K/V tiles of the two chunks of an item of n tiles (the first chunk takes the extra tile).
__device__ __forceinline__ int split_first(int n) { return (n + 1) / 2; }

// K/V tiles of all of row b's prefill items, over every KV head.
__device__ __forceinline__ int64_t row_prefill_tiles(const PlanParams& p, int b) {
  int64_t t = 0;
  for_row_items(p, b, [&](int n, int, int, int) { t += n; });
  return t * p.num_kv_heads;
}

// An item runs as two chunks of keys when it is long (more than kPrefillSplitTiles tiles) and its row alone
// cannot keep every CTA busy for as long as the item takes (row tiles / CTAs < the item's tiles): a long
// chunk on a short prompt splits, the items of a chunk that fills the GPU by itself do not (no handshake).
// It depends on the row and the device alone, so a row's result does not depend on the rest of the batch.
__device__ __forceinline__ bool split_item(const PlanParams& p, int n, int64_t row_tiles) {
  return n > kPrefillSplitTiles && (int64_t)n * p.prefill_ctas > row_tiles;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
  __shared__ int warp_sums[32];
  __shared__ int hist[kPrefillBuckets];
  __shared__ int n_slots;
  __shared__ int tail_at[kMaxSplitBlocks + 1];  // per last-split size: its task count, then its next slot
  __shared__ int n_dec;
  dev::griddep_wait();
  for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
    const int q0 = __ldg(p.qsl + i), q1 = __ldg(p.qsl + i + 1), ctx = __ldg(p.context_lens + i);
    if (q1 < q0 || (i == 0 && q0 != 0) || (i == p.num_seqs - 1 && q1 != p.num_tokens))
      dev::set_error(p.err, PKV_DEVERR_QSL);
    if (!row_meta_ok(q1 - q0, ctx, p.max_ctx)) dev::set_error(p.err, PKV_DEVERR_ROW_META);
  }
  for (int i = threadIdx.x; i < p.num_tokens * p.num_kv_heads; i += blockDim.x) p.merge_cnt[i] = 0;
  for (int i = threadIdx.x; i < kPrefillBuckets; i += blockDim.x) hist[i] = 0;
  for (int i = threadIdx.x; i <= kMaxSplitBlocks; i += blockDim.x) tail_at[i] = 0;
  for (int i = threadIdx.x; i < p.max_slots; i += blockDim.x) p.pf_sync[i] = make_int2(0, 0);
  if (threadIdx.x == 0) n_slots = 0;
  __syncthreads();

  // ---- decode tasks: tokens of rows that are not prefill items ----
  // Largest first: every token's full splits in token order, then the short last splits by decreasing
  // size.  The CTAs that take the last tasks of a launch then hold little work each, so the launch ends
  // nearly together on every SM.  (The order decides which CTA computes a split, never the result.)
  int carry = 0;
  for (int base = 0; base < p.num_tokens; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int nblk = 0, row = 0, c = 0;
    if (t < p.num_tokens) {
      const int b = dev::row_of_token(p.qsl, p.num_seqs, t);
      const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1), ctx = __ldg(p.context_lens + b);
      const int q_len = q1 - q0;
      const bool prefill = p.prefill_min_qlen > 0 && q_len >= p.prefill_min_qlen;
      if (t >= q0 && t < q1 && row_meta_ok(q_len, ctx, p.max_ctx) && !prefill) c = ctx - q_len + (t - q0) + 1;
      p.tok_row[t] = b;
      p.tok_ctx[t] = c;  // 0: no decode work (prefill row or invalid metadata)
      row = b;
      nblk = (c + kBS - 1) / kBS;
    }
    const int nfull = nblk / p.split_blocks, tail = nblk % p.split_blocks;
    if (tail > 0) atomicAdd(&tail_at[tail], p.num_kv_heads);
    const int cnt = nfull * p.num_kv_heads;
    int total = 0;
    const int off = carry + block_exclusive_scan(cnt, warp_sums, &total);
    for (int g = 0; g < p.num_kv_heads && cnt > 0; ++g)
      for (int s = 0; s < nfull; ++s) p.tasks[off + g * nfull + s] = make_int4(t, g | (s << 8), row, c);
    carry += total;
    __syncthreads();  // warp_sums is reused by the next chunk
  }
  if (threadIdx.x == 0) {  // each last-split size's first slot, largest size first
    int at = carry;
    for (int sz = kMaxSplitBlocks; sz >= 1; --sz) {
      const int n = tail_at[sz];
      tail_at[sz] = at;
      at += n;
    }
    n_dec = at;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < p.num_tokens; t += blockDim.x) {
    const int c = p.tok_ctx[t];  // written by this thread above
    const int nblk = (c + kBS - 1) / kBS, nfull = nblk / p.split_blocks, tail = nblk % p.split_blocks;
    if (tail > 0) {
      const int at = atomicAdd(&tail_at[tail], p.num_kv_heads), row = p.tok_row[t];
      for (int g = 0; g < p.num_kv_heads; ++g) p.tasks[at + g] = make_int4(t, g | (nfull << 8), row, c);
    }
  }

  // ---- prefill work entries, bucketed by K/V tile count, longest first; long items in two chunks ----
  auto bucket_of = [](int cost) { return kPrefillBuckets - 1 - min(cost, kPrefillBuckets - 1); };
  for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x) {
    const int64_t row_tiles = row_prefill_tiles(p, b);
    for_row_items(p, b, [&](int n, int, int, int) {
      if (split_item(p, n, row_tiles)) {
        atomicAdd(&hist[bucket_of(split_first(n))], p.num_kv_heads);
        atomicAdd(&hist[bucket_of(n - split_first(n))], p.num_kv_heads);
      } else {
        atomicAdd(&hist[bucket_of(n)], p.num_kv_heads);
      }
    });
  }
  __syncthreads();
  int n_items = 0;
  for (int base = 0; base < kPrefillBuckets; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < kPrefillBuckets ? hist[i] : 0;
    int total = 0;
    const int off = n_items + block_exclusive_scan(v, warp_sums, &total);
    __syncthreads();
    if (i < kPrefillBuckets) hist[i] = off;  // first slot of the bucket
    n_items += total;
    __syncthreads();
  }
  for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x) {
    const int64_t row_tiles = row_prefill_tiles(p, b);
    for_row_items(p, b, [&](int n, int npos, int t0, int w) {
      const bool split = split_item(p, n, row_tiles);
      const int slot = split ? atomicAdd(&n_slots, p.num_kv_heads) : -1;
      for (int chunk = 0; chunk < (split ? 2 : 1); ++chunk) {
        const int cost = split ? (chunk == 0 ? split_first(n) : n - split_first(n)) : n;
        const int at = atomicAdd(&hist[bucket_of(cost)], p.num_kv_heads);
        for (int g = 0; g < p.num_kv_heads; ++g) {
          p.items[at + g] = make_int4(b, prefill_rec_y(g, npos, chunk, split ? 1 : 0), t0, w);
          p.items_slot[at + g] = split ? slot + g : -1;
        }
      }
    });
  }

  // ---- 8-bit cache: the prefill rows' blocks, numbered row after row in the fp16 shadow ----
  if (p.pf_base != nullptr) {
    int nsh = 0;
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
      const int b = base + threadIdx.x;
      int nb = 0;
      if (b < p.num_seqs) {
        const int q_len = __ldg(p.qsl + b + 1) - __ldg(p.qsl + b), ctx = __ldg(p.context_lens + b);
        if (p.prefill_min_qlen > 0 && q_len >= p.prefill_min_qlen && row_meta_ok(q_len, ctx, p.max_ctx))
          nb = (ctx + kBS - 1) / kBS;
      }
      int total = 0;
      const int off = nsh + block_exclusive_scan(nb, warp_sums, &total);
      if (b < p.num_seqs) p.pf_base[b] = off;
      nsh += total;
      __syncthreads();
    }
    if (threadIdx.x == 0) p.pf_base[p.num_seqs] = nsh;
  }

  if (threadIdx.x == 0) {
    p.hdr->n_tasks = n_dec;
    p.hdr->work = 0;
    p.hdr->done = 0;
    p.hdr->n_items = n_items;
    p.hdr->pwork = 0;
    p.hdr->pdone = 0;
  }
  __threadfence();
  dev::griddep_launch_dependents();
}

// ---------------------------------------------------------------------------------------------------
// Workspace layout and launches
// ---------------------------------------------------------------------------------------------------
struct WsLayout {
  size_t hdr, tok_row, tok_ctx, merge_cnt, tasks, items, items_slot, pf_sync, pf_ml, pf_o, part_ml, part_o, total;
  // 8-bit cache with prefill rows: the rows' first shadow block, the shadow block tables and the fp16 shadow
  size_t pf_base = 0, shadow_bt = 0, shadow = 0;
  int64_t shadow_blocks = 0;
  int max_splits;
  int64_t max_tasks;
  int prefill_min_qlen;  // 0: every row takes the decode path
  int prefill_pos;
  int64_t max_items;
};

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

static WsLayout ws_layout(const pkv_config& c, int num_seqs, int num_tokens, int max_blocks) {
  WsLayout w;
  w.max_splits = (max_blocks + c.split_blocks - 1) / c.split_blocks;
  w.max_tasks = (int64_t)num_tokens * c.num_kv_heads * w.max_splits;
  const int group = c.num_q_heads / c.num_kv_heads;
  // the tile kernel reads fp16 K/V: on an 8-bit cache it reads the prefill rows' blocks from an fp16 shadow
  const bool prefill = prefill_supported(c.head_dim, group) && c.num_kv_heads < 256;
  w.prefill_min_qlen = prefill ? kPrefillMinQlen : 0;
  w.prefill_pos = prefill_item_positions(group, c.head_dim);
  // a prefill row has >= prefill_min_qlen tokens, every other row >= 1: at most R such rows, holding at most
  // num_tokens - (num_seqs - R) tokens
  int64_t rows = 0, toks = 0;
  if (prefill && num_seqs > 0) {
    rows = std::min<int64_t>(num_seqs, (int64_t)(num_tokens - num_seqs) / (kPrefillMinQlen - 1));
    toks = num_tokens - (num_seqs - rows);
  }
  w.max_items = rows > 0 ? (int64_t)c.num_kv_heads * ((toks + w.prefill_pos - 1) / w.prefill_pos + rows) : 0;
  size_t off = 0;
  w.hdr = off;
  off += sizeof(WsHeader);
  w.tok_row = off;
  off += up256((size_t)num_tokens * 4);
  w.tok_ctx = off;
  off += up256((size_t)num_tokens * 4);
  w.merge_cnt = off;
  off += up256((size_t)num_tokens * c.num_kv_heads * 4);
  w.tasks = off;
  off += up256((size_t)w.max_tasks * sizeof(int4));
  // prefill: up to two work entries per item (split-KV), one partial slot per item
  w.items = off;
  off += up256((size_t)w.max_items * 2 * sizeof(int4));
  w.items_slot = off;
  off += up256((size_t)w.max_items * 2 * sizeof(int32_t));
  w.pf_sync = off;
  off += up256((size_t)w.max_items * sizeof(int2));
  w.pf_ml = off;
  off += up256((size_t)w.max_items * kPrefillRows * 2 * sizeof(float2));
  w.pf_o = off;
  off += up256((size_t)w.max_items * kPrefillRows * 2 * c.head_dim * sizeof(float));
  const size_t parts = w.max_splits > 1 ? (size_t)w.max_tasks : 0;  // one partial per (token, KV head, split)
  w.part_ml = off;
  off += up256(parts * kHeadsTile * sizeof(float2));
  w.part_o = off;
  off += up256(parts * 32 * (c.head_dim / 4) * sizeof(float));
  if (c.kv_dtype == PKV_KV_E4M3 && rows > 0) {
    // the prefill rows hold at most `rows` x max_blocks blocks, and at most the pool's when no two rows
    // share one; more than that is refused by the dequantizing kernel (reported, never written)
    w.shadow_blocks = std::min<int64_t>((int64_t)c.num_blocks, rows * (int64_t)max_blocks);
    w.pf_base = off;
    off += up256((size_t)(num_seqs + 1) * 4);
    w.shadow_bt = off;
    off += up256((size_t)num_seqs * max_blocks * 4);
    w.shadow = off;
    off += up256((size_t)2 * w.shadow_blocks * c.num_kv_heads * kBS * c.head_dim * 2);
  }
  w.total = off;
  return w;
}


static cudaError_t launch_plan(pkv_pool* pool, char* ws, const WsLayout& w, const int32_t* context_lens,
                               const int32_t* qsl, int num_seqs, int num_tokens, int max_blocks, cudaStream_t s) {
  const pkv_config& c = pool->cfg;
  PlanParams p;
  p.context_lens = context_lens;
  p.qsl = qsl;
  p.num_seqs = num_seqs;
  p.num_tokens = num_tokens;
  p.max_ctx = max_blocks * kBS;
  p.split_blocks = c.split_blocks;
  p.num_kv_heads = c.num_kv_heads;
  p.prefill_min_qlen = w.prefill_min_qlen;
  p.prefill_pos = w.prefill_pos;
  p.prefill_keys = prefill_tile_keys(c.head_dim);
  p.prefill_ctas = pool->num_sms;
  p.tok_row = reinterpret_cast<int32_t*>(ws + w.tok_row);
  p.tok_ctx = reinterpret_cast<int32_t*>(ws + w.tok_ctx);
  p.merge_cnt = reinterpret_cast<int32_t*>(ws + w.merge_cnt);
  p.tasks = reinterpret_cast<int4*>(ws + w.tasks);
  p.items = reinterpret_cast<int4*>(ws + w.items);
  p.items_slot = reinterpret_cast<int32_t*>(ws + w.items_slot);
  p.pf_sync = reinterpret_cast<int2*>(ws + w.pf_sync);
  p.max_slots = (int)w.max_items;
  p.pf_base = w.shadow_blocks > 0 ? reinterpret_cast<int32_t*>(ws + w.pf_base) : nullptr;
  p.hdr = reinterpret_cast<WsHeader*>(ws + w.hdr);
  p.err = pool->dev_error;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p);
}

// ---------------------------------------------------------------------------------------------------
// 8-bit cache, prefill rows: the tile kernel reads fp16 tiles, so every block of a prefill row is first
// dequantized (exactly) into an fp16 shadow in the workspace, and the row's shadow block table is written
// alongside.  The plan numbered the prefill rows' blocks row after row (pf_base, monotone, with the total at
// the end); a CTA takes shadow blocks in turn, finds its row by binary search over pf_base staged in shared
// memory, and dequantizes the block's Hkv x 16 rows with all its threads.  Keys past the context in a last
// block are written as zeros.
// ---------------------------------------------------------------------------------------------------
struct DequantParams {
  const unsigned char* codes_k;  // this layer's codes [num_blocks][Hkv][16][D]
  const unsigned char* codes_v;
  const unsigned char* scales;   // this layer's scale records [num_blocks][Hkv][2][16]
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* pf_base;        // [num_seqs + 1]
  int32_t* shadow_bt;            // [num_seqs][max_blocks]
  uint4* shadow_k;               // [shadow_blocks][Hkv][16][D] fp16
  uint4* shadow_v;
  int32_t* err;
  int64_t shadow_blocks;
  int num_seqs, max_blocks, num_kv_heads, num_blocks;
};

constexpr int kDequantMaxRows = 48 * 1024 - 1;  // pf_base staged in shared memory: (rows + 1) x 4 bytes <= 192 KB

template <int D>
__global__ void __launch_bounds__(256) dequant_prefill_rows_kernel(const DequantParams p) {
  extern __shared__ int32_t sbase[];  // [num_seqs + 1]
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  constexpr int CPR = D / 8;  // 16-byte fp16 chunks (8 codes) per row
  for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) sbase[i] = p.pf_base[i];
  __syncthreads();
  const int64_t want = sbase[p.num_seqs];
  // rows sharing blocks can hold more than the shadow: the excess is refused and reported (the tile kernel
  // then finds an out-of-range id in their tables and reports it too)
  if (want > p.shadow_blocks && blockIdx.x == 0 && threadIdx.x == 0) dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
  const int total = (int)min(want, p.shadow_blocks);
  const int per_block = p.num_kv_heads * kBS * CPR;
  for (int sb = blockIdx.x; sb < total; sb += gridDim.x) {
    int lo = 0, hi = p.num_seqs - 1;  // the row: the last b with sbase[b] <= sb (rows before it hold fewer)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sbase[mid] <= sb) lo = mid; else hi = mid - 1;
    }
    const int b = lo, j = sb - sbase[b];
    const int ctx = __ldg(p.context_lens + b);
    const int id = __ldg(p.block_tables + (int64_t)b * p.max_blocks + j);
    const bool ok = id >= 0 && id < p.num_blocks;
    if (threadIdx.x == 0) {
      p.shadow_bt[(int64_t)b * p.max_blocks + j] = sb;
      if (!ok) dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
    }
    for (int i = threadIdx.x; i < per_block; i += blockDim.x) {
      const int h = i / (kBS * CPR), r = (i / CPR) % kBS, c = i % CPR;
      const bool live = ok && j * kBS + r < ctx;
      const int64_t src = (ok ? (int64_t)id : 0) * p.num_kv_heads + h;
      const int64_t dst = (((int64_t)sb * p.num_kv_heads + h) * kBS + r) * CPR + c;
      const unsigned char* rec = p.scales + src * 32;
      const uint2 zero = make_uint2(0, 0);
      const uint2 ck = live ? __ldg(reinterpret_cast<const uint2*>(p.codes_k + (src * kBS + r) * D) + c) : zero;
      const uint2 cv = live ? __ldg(reinterpret_cast<const uint2*>(p.codes_v + (src * kBS + r) * D) + c) : zero;
      p.shadow_k[dst] = dev::e4m3x8_dequant(ck, live ? __ldg(rec + r) : 127u);
      p.shadow_v[dst] = dev::e4m3x8_dequant(cv, live ? __ldg(rec + 16 + r) : 127u);
    }
  }
}

template <int D>
static cudaError_t launch_dequant(const DequantParams& dq, int num_sms, cudaStream_t s) {
  static bool attr = false;
  const size_t smem = (size_t)(dq.num_seqs + 1) * 4;
  if (!attr && smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(dequant_prefill_rows_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (kDequantMaxRows + 1) * 4);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(dequant_prefill_rows_kernel<D>, dim3((unsigned)(num_sms * 2)), dim3(256), smem, s, dq);
}

// Inputs of an append fused into the decode launch (k == nullptr: not fused).
struct FusedAppend {
  const void* k = nullptr;
  const void* v = nullptr;
  const int64_t* slots = nullptr;
};

// decode (+ merge of very long tokens) and prefill tiles for one layer on a planned workspace
static pkv_status launch_attention(pkv_pool* pool, int layer, const void* q, const int32_t* block_tables,
                                   const int32_t* context_lens, const int32_t* qsl, int max_blocks, int num_seqs,
                                   int num_tokens, void* out, char* ws,
                                   const WsLayout& w, cudaStream_t s, int* launches,
                                   const FusedAppend& fa = FusedAppend()) {
  const pkv_config& c = pool->cfg;
  DecodeParams p;
  p.kv_map = c.kv_dtype == PKV_KV_E4M3 ? pool->kv_map : pool->run_map;  // fp16: one copy per run
  p.q = static_cast<const __half*>(q);
  p.block_tables = block_tables;
  p.qsl = qsl;
  p.tasks = reinterpret_cast<const int4*>(ws + w.tasks);
  p.hdr = reinterpret_cast<WsHeader*>(ws + w.hdr);
  p.out = static_cast<__half*>(out);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  p.merge_cnt = reinterpret_cast<int32_t*>(ws + w.merge_cnt);
  p.err = pool->dev_error;
  p.k_in = static_cast<const __half*>(fa.k);
  p.v_in = static_cast<const __half*>(fa.v);
  p.slots = fa.slots;
  p.cache_k = static_cast<__half*>(pkv_pool_layer_ptr(pool, layer, 0));
  p.cache_v = static_cast<__half*>(pkv_pool_layer_ptr(pool, layer, 1));
  const bool f8 = c.kv_dtype == PKV_KV_E4M3;
  p.scales = static_cast<unsigned char*>(pkv_pool_scales_ptr(pool, layer));
  p.num_slots = (int64_t)c.num_blocks * c.block_size;
  // TMA rows per (layer, K/V) pool: one per token (fp16) or per 128 code bytes (8-bit)
  const int64_t toks_per_pool = (int64_t)c.num_blocks * c.num_kv_heads * c.block_size;
  // (the 8-bit d 256 map addresses tokens, with the two halves of a key as its middle dimension)
  const int rows_per_pool = (int)(f8 && c.head_dim != 256 ? toks_per_pool * c.head_dim / 128 : toks_per_pool);
  p.layer_row0_k = (layer * 2) * rows_per_pool;
  p.layer_row0_v = (layer * 2 + 1) * rows_per_pool;
  p.max_blocks = max_blocks;
  p.num_q_heads = c.num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.num_blocks = c.num_blocks;
  p.split_blocks = c.split_blocks;
  p.max_splits = w.max_splits;
  p.max_tasks = (int)w.max_tasks;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  const int group = c.num_q_heads / c.num_kv_heads;
  // Prefill rows exist only if some row has at least prefill_min_qlen new tokens.  Their tile kernel goes
  // first; the decode kernel follows in its tail (late_wait).
  p.late_wait = 0;
  cudaError_t e;
  if (w.prefill_min_qlen > 0 && num_tokens - num_seqs >= w.prefill_min_qlen - 1) {
    PrefillArgs a;
    a.kv_map = &pool->kv_map;
    a.block_tables = block_tables;
    a.layer_row0_k = p.layer_row0_k;
    a.layer_row0_v = p.layer_row0_v;
    a.num_blocks = c.num_blocks;
    if (f8) {  // the prefill rows' blocks, dequantized into the workspace's fp16 shadow (its map is prepared)
      char* shadow = ws + w.shadow;
      const uint64_t srows = (uint64_t)2 * w.shadow_blocks * c.num_kv_heads * kBS;
      if (pool->shadow_base != shadow || pool->shadow_rows != srows)
        return fail(PKV_ERR_INVALID_ARG, "8-bit cache: the shadow tensor map was not prepared for this workspace");
      DequantParams dq;
      dq.codes_k = static_cast<const unsigned char*>(pkv_pool_layer_ptr(pool, layer, 0));
      dq.codes_v = static_cast<const unsigned char*>(pkv_pool_layer_ptr(pool, layer, 1));
      dq.scales = p.scales;
      dq.block_tables = block_tables;
      dq.context_lens = context_lens;
      dq.pf_base = reinterpret_cast<const int32_t*>(ws + w.pf_base);
      dq.shadow_bt = reinterpret_cast<int32_t*>(ws + w.shadow_bt);
      dq.shadow_k = reinterpret_cast<uint4*>(shadow);
      dq.shadow_v = reinterpret_cast<uint4*>(shadow + srows / 2 * c.head_dim * 2);
      dq.err = p.err;
      dq.shadow_blocks = w.shadow_blocks;
      dq.num_seqs = num_seqs;
      dq.max_blocks = max_blocks;
      dq.num_kv_heads = c.num_kv_heads;
      dq.num_blocks = c.num_blocks;
      e = c.head_dim == 64    ? launch_dequant<64>(dq, pool->num_sms, s)
          : c.head_dim == 128 ? launch_dequant<128>(dq, pool->num_sms, s)
                              : launch_dequant<256>(dq, pool->num_sms, s);
      if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
      *launches += 1;
      a.kv_map = &pool->shadow_map;
      a.block_tables = dq.shadow_bt;
      a.layer_row0_k = 0;
      a.layer_row0_v = (int)(srows / 2);
      a.num_blocks = (int)w.shadow_blocks;
    }
    a.q = q;
    a.out = out;
    a.items = reinterpret_cast<const int4*>(ws + w.items);
    a.items_slot = reinterpret_cast<const int32_t*>(ws + w.items_slot);
    a.pf_sync = reinterpret_cast<int2*>(ws + w.pf_sync);
    a.pf_ml = reinterpret_cast<float2*>(ws + w.pf_ml);
    a.pf_o = reinterpret_cast<float*>(ws + w.pf_o);
    a.hdr = p.hdr;
    a.err = p.err;
    a.max_blocks = max_blocks;
    a.num_q_heads = c.num_q_heads;
    a.num_kv_heads = c.num_kv_heads;
    a.head_dim = c.head_dim;
    a.num_sms = pool->num_sms;
    a.max_items = 2 * w.max_items;
    e = launch_prefill(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    *launches += 1;
    p.late_wait = 1;
  }
  if (f8) {
    e = launch_decode_e4m3(c.head_dim, group, p, pool->num_sms, w.max_tasks, s);
  } else {
    switch (c.head_dim) {
      case 64: e = launch_decode_g<64, kKvF16>(group, p, pool->num_sms, w.max_tasks, s); break;
      case 128: e = launch_decode_g<128, kKvF16>(group, p, pool->num_sms, w.max_tasks, s); break;
      case 256: e = launch_decode_g<256, kKvF16>(group, p, pool->num_sms, w.max_tasks, s); break;
      default: return fail(PKV_ERR_UNSUPPORTED, "head_dim");
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  *launches += 1;
  if (w.max_splits > kFusedMergeSplits) {
    MergeParams m{p.part_o, p.part_ml, reinterpret_cast<const int32_t*>(ws + w.tok_ctx), p.out, c.num_q_heads, c.num_kv_heads, group, c.split_blocks,
                  w.max_splits};
    const dim3 grid(num_tokens, c.num_kv_heads, (group * c.head_dim) / 32);
    switch (c.head_dim) {
      case 64: e = launch_pdl(merge_kernel<64>, grid, dim3(256), 0, s, m); break;
      case 128: e = launch_pdl(merge_kernel<128>, grid, dim3(256), 0, s, m); break;
      default: e = launch_pdl(merge_kernel<256>, grid, dim3(256), 0, s, m); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    *launches += 1;
  }
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_attention_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_tokens,
                                                int32_t max_blocks_per_seq) {
  if (!pool || num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 1) return 0;
  return ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq).total;
}

static pkv_status check_common(pkv_pool* pool, const int32_t* context_lens, const int32_t* qsl, int32_t num_seqs,
                               int32_t num_tokens, int32_t max_blocks) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (num_seqs < 0 || num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be >= 0");
  if (num_tokens > 0 && num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "tokens without rows");
  if (num_seqs > num_tokens) return fail(PKV_ERR_INVALID_ARG, "every row needs at least one query token");
  if (max_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  if (num_tokens > 0 && (!context_lens || !qsl)) return fail(PKV_ERR_INVALID_ARG, "metadata pointers must be non-NULL");
  const pkv_config& c = pool->cfg;
  if (c.split_blocks > kMaxSplitBlocks)
    return fail(PKV_ERR_UNSUPPORTED, "split_blocks above " + std::to_string(kMaxSplitBlocks));
  const int64_t splits = ((int64_t)max_blocks + c.split_blocks - 1) / c.split_blocks;
  if (splits >= (1 << 23) || (int64_t)num_tokens * c.num_kv_heads * splits >= (1ll << 31))
    return fail(PKV_ERR_UNSUPPORTED, "too many splits in one pass; raise split_blocks");
  return PKV_OK;
}

static pkv_status check_workspace(pkv_pool* pool, void* workspace, size_t ws_bytes, int32_t num_seqs, int32_t num_tokens,
                                  int32_t max_blocks) {
  if (num_tokens > 0 && !workspace) return fail(PKV_ERR_INVALID_ARG, "workspace must be non-NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks);
  if (ws_bytes < w.total)
    return fail(PKV_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(w.total) + " bytes");
  return PKV_OK;
}

static pkv_status check_io(const void* q, const void* out, const int32_t* block_tables) {
  if (!q || !out || !block_tables) return fail(PKV_ERR_INVALID_ARG, "q, out and block_tables must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (q == out) return fail(PKV_ERR_INVALID_ARG, "out may not alias q");
  return PKV_OK;
}

// The plan remembered for `workspace`, or null.
static const PlanKey* find_plan(const pkv_pool* pool, const void* workspace) {
  for (auto it = pool->plans.rbegin(); it != pool->plans.rend(); ++it)
    if (it->workspace == workspace) return &*it;
  return nullptr;
}

static void forget_plan(pkv_pool* pool, const void* workspace) {
  for (auto it = pool->plans.begin(); it != pool->plans.end(); ++it)
    if (it->workspace == workspace) {
      pool->plans.erase(it);
      return;
    }
}

static void remember_plan(pkv_pool* pool, const PlanKey& key) {
  forget_plan(pool, key.workspace);
  pool->plans.push_back(key);
  if (pool->plans.size() > kMaxPlans) pool->plans.erase(pool->plans.begin());
}

// A call on a planned workspace: the plan must have been issued on this workspace with the same metadata
// pointers and sizes, and (when both the plan and this call ran under PKV_VALIDATE=1) the same
// context_lens / query_start_loc contents.
static pkv_status check_plan(const pkv_pool* pool, const void* workspace, const int32_t* context_lens,
                             const int32_t* qsl, int32_t num_seqs, int32_t num_tokens, int32_t max_blocks,
                             const MetaCheck& mc) {
  const PlanKey* k = find_plan(pool, workspace);
  if (!k || k->context_lens != context_lens || k->query_start_loc != qsl || k->num_seqs != num_seqs ||
      k->num_tokens != num_tokens || k->max_blocks_per_seq != max_blocks)
    return fail(PKV_ERR_INVALID_ARG, "no matching plan: call pkv_attention_plan for this workspace and metadata");
  if (mc.ran && k->summed && mc.sum != k->meta_sum)
    return fail(PKV_ERR_INVALID_ARG, "PKV_VALIDATE: context_lens / query_start_loc changed since pkv_attention_plan "
                "on this workspace; plan the pass again");
  return PKV_OK;
}

// Host-side refusals of the 8-bit cache's prefill path, made before anything is launched: the dequantizing
// kernel stages one int per row in shared memory, and the fp16 shadow's tensor map is encoded here (once per
// workspace placement) so that a failed encode launches nothing either.
static pkv_status prepare_prefill_shadow(pkv_pool* pool, char* ws, const WsLayout& w, int num_seqs, int num_tokens) {
  const pkv_config& c = pool->cfg;
  if (c.kv_dtype != PKV_KV_E4M3 || w.prefill_min_qlen <= 0 || num_tokens - num_seqs < w.prefill_min_qlen - 1)
    return PKV_OK;
  if (num_seqs > kDequantMaxRows)
    return fail(PKV_ERR_UNSUPPORTED, "8-bit cache: prefill rows in a pass of more than 49151 rows");
  char* shadow = ws + w.shadow;
  const uint64_t srows = (uint64_t)2 * w.shadow_blocks * c.num_kv_heads * kBS;
  if (pool->shadow_base != shadow || pool->shadow_rows != srows) {
    const pkv_status st = encode_f16_rows(&pool->shadow_map, shadow, srows, c.head_dim);
    if (st != PKV_OK) {
      pool->shadow_base = nullptr;
      return st;
    }
    pool->shadow_base = shadow;
    pool->shadow_rows = srows;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_attention_plan(pkv_pool* pool, const int32_t* context_lens, const int32_t* query_start_loc,
                                         int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq);
  if (st == PKV_OK) st = check_workspace(pool, workspace, workspace_bytes, num_seqs, num_tokens, max_blocks_per_seq);
  MetaCheck mc;
  if (st == PKV_OK) st = validate_metadata(pool, nullptr, max_blocks_per_seq, context_lens, query_start_loc, num_seqs,
                                           num_tokens, nullptr, stream, &mc);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  forget_plan(pool, workspace);
  PlanKey key{workspace, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq, mc.ran, mc.sum};
  if (num_tokens == 0) {
    remember_plan(pool, key);
    return PKV_OK;
  }
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  st = prepare_prefill_shadow(pool, static_cast<char*>(workspace), w, num_seqs, num_tokens);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_plan(pool, static_cast<char*>(workspace), w, context_lens, query_start_loc, num_seqs,
                              num_tokens, max_blocks_per_seq, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  remember_plan(pool, key);
  pool->last_launches = 1;
  return PKV_OK;
}

extern "C" pkv_status pkv_attention(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq);
  if (st == PKV_OK) st = check_workspace(pool, workspace, workspace_bytes, num_seqs, num_tokens, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  if (layer < 0 || layer >= pool->cfg.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_tokens == 0) return PKV_OK;
  st = check_io(q, out, block_tables);
  MetaCheck mc;
  if (st == PKV_OK) st = validate_metadata(pool, block_tables, max_blocks_per_seq, context_lens, query_start_loc,
                                           num_seqs, num_tokens, nullptr, stream, &mc);
  if (st == PKV_OK) st = check_plan(pool, workspace, context_lens, query_start_loc, num_seqs, num_tokens,
                                    max_blocks_per_seq, mc);
  if (st != PKV_OK) return st;
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  st = prepare_prefill_shadow(pool, static_cast<char*>(workspace), w, num_seqs, num_tokens);
  if (st != PKV_OK) return st;
  int launches = 0;
  st = launch_attention(pool, layer, q, block_tables, context_lens, query_start_loc, max_blocks_per_seq, num_seqs, num_tokens, out,
                        static_cast<char*>(workspace), w, (cudaStream_t)stream, &launches);
  pool->last_launches = launches;
  return st;
}

// ---------------------------------------------------------------------------------------------------
// kv_append + attention of one layer as one call.  When no row of the pass can take the prefill path
// (every row has fewer than kPrefillMinQlen new tokens), the append runs inside the decode launch: tiles
// take this pass's keys and values from the inputs and each token is written to the cache by the warp
// whose block holds its position, so the attention waits for no separate append.  Otherwise it is the
// append kernel followed by the attention.
// ---------------------------------------------------------------------------------------------------
extern "C" pkv_status pkv_attention_append(pkv_pool* pool, int32_t layer, const void* q, const void* k,
                                           const void* v, const int64_t* slot_mapping, const int32_t* block_tables,
                                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                                           const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                                           void* out, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq);
  if (st == PKV_OK) st = check_workspace(pool, workspace, workspace_bytes, num_seqs, num_tokens, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  if (layer < 0 || layer >= pool->cfg.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_tokens == 0) return PKV_OK;
  st = check_io(q, out, block_tables);
  if (st != PKV_OK) return st;
  if (!k || !v || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  MetaCheck mc;
  st = validate_metadata(pool, block_tables, max_blocks_per_seq, context_lens, query_start_loc, num_seqs, num_tokens,
                         slot_mapping, stream, &mc);
  if (st == PKV_OK) st = check_plan(pool, workspace, context_lens, query_start_loc, num_seqs, num_tokens,
                                    max_blocks_per_seq, mc);
  if (st != PKV_OK) return st;
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  st = prepare_prefill_shadow(pool, static_cast<char*>(workspace), w, num_seqs, num_tokens);
  if (st != PKV_OK) return st;
  int launches = 0;
  // Prefill rows possible (they read the cache), or on an 8-bit cache a row with 16 or more new tokens
  // (quantizing its rows once beats re-quantizing them in every tile that holds them): append first.
  const bool long_rows = num_tokens - num_seqs >= kPrefillMinQlen - 1;
  if (w.max_items > 0 || (pool->cfg.kv_dtype == PKV_KV_E4M3 && long_rows)) {
    st = pkv_append(pool, layer, k, v, slot_mapping, num_tokens, stream);
    if (st != PKV_OK) return st;
    launches = pool->last_launches;
    st = launch_attention(pool, layer, q, block_tables, context_lens, query_start_loc, max_blocks_per_seq, num_seqs, num_tokens,
                          out, static_cast<char*>(workspace), w, (cudaStream_t)stream, &launches);
  } else {
    FusedAppend fa;
    fa.k = k;
    fa.v = v;
    fa.slots = slot_mapping;
    st = launch_attention(pool, layer, q, block_tables, context_lens, query_start_loc, max_blocks_per_seq, num_seqs, num_tokens,
                          out, static_cast<char*>(workspace), w, (cudaStream_t)stream, &launches, fa);
  }
  pool->last_launches = launches;
  return st;
}

// ---------------------------------------------------------------------------------------------------
// Allocation-free variant of the attention call.
//
// Some callers cannot hand the library a workspace: an engine that has already reserved every byte of
// device memory for its own pools, or a caller that may not issue cudaMalloc (which can synchronise the
// whole device) while a pass is in flight.  For them the split-K scratch -- the per-token table, the
// task list, the merge counters and the partial (m, l, o) results -- lives in one fixed array compiled
// into this library.  Each device that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------------------------------
namespace pkv {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address in the current context.  In host code the symbol name itself is only a
// host-side stand-in and must never reach a kernel.  The address is looked up (cudaGetSymbolAddress, with the
// device current) the first time a context calls, and cached per (device, context): a context created
// after cudaDeviceReset loads the library's module again, so it gets its own lookup.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

static CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && f) fn = reinterpret_cast<CtxGetCurrentFn>(f);
  }
  return fn;
}

struct ScratchAddr {
  int device;
  CUcontext ctx;
  void* ptr;
};

// The cached address for (device, context), or null when that context has not looked it up yet.
static void* noalloc_scratch_cached(int device, CUcontext ctx, std::vector<ScratchAddr>& cache) {
  for (const ScratchAddr& a : cache)
    if (a.device == device && a.ctx == ctx) return a.ptr;
  return nullptr;
}

static pkv_status noalloc_scratch_ptr(int device, cudaStream_t stream, void** out) {
  static std::mutex mu;
  static std::vector<ScratchAddr> cache;
  *out = nullptr;
  // a runtime call on the stream makes the device's context current on this thread (the runtime does this
  // lazily), and the capture status is needed below anyway
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return fail(PKV_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS || !ctx) return fail(PKV_ERR_CUDA, "cuCtxGetCurrent found no current context");
  std::lock_guard<std::mutex> lock(mu);
  if (void* p = noalloc_scratch_cached(device, ctx, cache)) {
    *out = p;
    return PKV_OK;
  }
  if (cap != cudaStreamCaptureStatusNone)
    return fail(PKV_ERR_INVALID_ARG, "the first pkv_attention_noalloc call on a device (and context) must come before "
                "any stream capture: it looks up the built-in scratch array's address");
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch array");
  cache.push_back(ScratchAddr{device, ctx, ptr});
  *out = ptr;
  return PKV_OK;
}

}  // namespace pkv

extern "C" pkv_status pkv_attention_noalloc(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                                            const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                                            void* out, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  if (layer < 0 || layer >= pool->cfg.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_tokens == 0) return PKV_OK;
  st = check_io(q, out, block_tables);
  if (st == PKV_OK) st = validate_metadata(pool, block_tables, max_blocks_per_seq, context_lens, query_start_loc,
                                           num_seqs, num_tokens, nullptr, stream);
  if (st != PKV_OK) return st;
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  if (w.total > kNoAllocScratchBytes)
    return fail(PKV_ERR_OUT_OF_RANGE, "pass needs " + std::to_string(w.total) + " bytes of scratch; the built-in "
                "array holds " + std::to_string(kNoAllocScratchBytes) + " (use pkv_attention with a workspace)");
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (device != pool->device) return fail(PKV_ERR_INVALID_ARG, "the pool's device must be the current device");
  cudaStream_t s = (cudaStream_t)stream;
  void* scratch = nullptr;
  st = noalloc_scratch_ptr(device, s, &scratch);
  if (st != PKV_OK) return st;
  // What must start at zero -- the task and split counters -- is cleared by the plan kernel on every call;
  // everything else is written before it is read.
  char* ws = static_cast<char*>(scratch);
  st = prepare_prefill_shadow(pool, ws, w, num_seqs, num_tokens);
  if (st != PKV_OK) return st;
  e = launch_plan(pool, ws, w, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  int launches = 1;
  st = launch_attention(pool, layer, q, block_tables, context_lens, query_start_loc, max_blocks_per_seq, num_seqs, num_tokens, out,
                        ws, w, s, &launches);
  pool->last_launches = launches;
  return st;
}
