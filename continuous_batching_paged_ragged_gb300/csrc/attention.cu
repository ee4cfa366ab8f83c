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
//    task list.  A task is one split of one (token, KV head): `split_blocks` consecutive 16-token blocks.
//    The split count of a token depends only on its own context, so results are bit-identical whatever
//    else is in the batch, whatever the row order and wherever the blocks sit physically.
//  * decode_kernel: persistent; a CTA of 4 warps takes one task at a time from a global counter, and
//    the task's blocks are dealt round-robin to its warps (block i to warp i % 4).  Every warp streams its
//    blocks' K and V runs through its own shared-memory ring with 2-D TMA tile copies (128-byte swizzle)
//    that its lane 0 issues: independent issuers per SM are what keep HBM busy, and sharing a task four
//    ways keeps all of them busy even when a pass has few tasks.  The KV head's G <= 8 query heads ride
//    along, so each K/V block is read from HBM exactly once.  Per 16-key block the group contraction runs
//    on the tensor cores with warp MMAs: S^T[16 keys x 8 heads] = K Q^T and O^T[d x 8 heads] += V^T P^T,
//    operands fetched from the swizzled ring with ldmatrix; the online softmax (running max and sum in
//    the log2 domain, fp32) reduces across the lanes that share a head with warp shuffles.  At the end of
//    a task the four warps' (m, l, o) are combined with log-sum-exp weights through shared memory.
//  * Cross-split merge: a token whose context fits one split gets its fp16 output from the decode
//    directly.  Otherwise each split leaves an unnormalised partial (m, l, o); the CTA that finishes the
//    token's last split merges them with log-sum-exp weights, inside the same launch (a separate merge
//    launch cost more than the merge: its CTAs cannot start until the decode's have left the SMs).
//    Tokens with more than 32 splits are merged by merge_kernel, launched behind the decode, which
//    spreads one token's merge over many CTAs.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

#include "attn_common.cuh"

namespace pkv {

constexpr int kFusedMergeSplits = 32;  // tokens with up to this many splits are merged inside the decode
constexpr int kMaxSplitBlocks = 32;   // upper bound on split_blocks (a split's block ids fit one warp)

// Ring slots per warp: runs (a block's K or V for one KV head, or a task's q) in flight.
#ifndef PKV_DECODE_RING
#define PKV_DECODE_RING(D) ((D) == 256 ? 2 : ((D) == 128 ? 3 : 5))
#endif

constexpr int kSmemPerSM = 228 * 1024;  // shared memory of one SM
constexpr int kSmemReservedPerCTA = 1024;

template <int D, int G>
struct DecodeTraits {
  static constexpr int NW = 4;                     // warps per CTA; block i of a task goes to warp i % NW
  static constexpr int NTHREADS = NW * 32;
  static constexpr int RUN = kBS * D * 2;          // one (block, KV head) run of K or V = D/64 TMA boxes
  static constexpr int BOXES = D / 64;
  static constexpr int NR = PKV_DECODE_RING(D);    // ring slots (runs in flight) per warp
  static constexpr int KS = D / 16;                // MMA k-steps over the head dimension (scores)
  static constexpr int MT = D / 16;                // MMA m-tiles over the head dimension (values)
  static constexpr int OV = MT * 4;                // fp32 output values per lane
  static constexpr int OFF_BAR = NW * NR * RUN;    // [NW][NR] run barriers after the rings
  static constexpr int OFF_CO = OFF_BAR + NW * NR * 8;         // combine: [NW][OV][32 lanes] fp32 o
  static constexpr int OFF_CM = OFF_CO + NW * OV * 32 * 4;     // combine: [NW][8 heads] running max
  static constexpr int OFF_CL = OFF_CM + NW * kHeadsTile * 4;  // combine: [NW][8 heads] running sum
  static constexpr int OFF_IDX = OFF_CL + NW * kHeadsTile * 4; // [4] task indices, merge target, its splits
  static constexpr int SMEM = OFF_IDX + 32 + 1024;  // + slack to align the rings to 1024 bytes
  static constexpr int FIT = kSmemPerSM / (SMEM + kSmemReservedPerCTA);
  static constexpr int MINB = FIT < 4 ? FIT : 4;   // CTAs per SM (shared memory bound)
  static_assert(D % 64 == 0 && G >= 1 && G <= kHeadsTile, "shape");
  static_assert(RUN % 1024 == 0, "swizzled boxes need 1024-byte aligned slots");
  static_assert(8 * D * 2 <= RUN && KS % 2 == 0, "a task's q (8 rows) fits one slot");
  static_assert(MINB >= 1, "shared memory");
};

struct DecodeParams {
  CUtensorMap kv_map;  // the pool as TMA rows of head_dim values (64-byte aligned: first member)
  const __half* q;
  const int32_t* block_tables;
  const int32_t* tok_row;
  const int32_t* tok_ctx;
  const int4* tasks;   // {token, kv head | split << 8, row, causal context}
  WsHeader* hdr;
  __half* out;
  float* part_o;       // [num_tokens * num_kv_heads * max_splits][8 heads][D]
  float2* part_ml;     // [num_tokens * num_kv_heads * max_splits][8 heads]
  int32_t* merge_cnt;  // [num_tokens * num_kv_heads] splits finished; zero between launches
  int32_t* err;
  // Append fused into the attention (k_in != nullptr): keys and values of this pass's tokens are taken
  // from k_in / v_in [T][Hkv][D] wherever a tile holds them, and the warp holding a token's own
  // position writes that token into the cache at slots[t].
  const __half* k_in;
  const __half* v_in;
  const int64_t* slots;
  const int32_t* qsl;
  __half* cache_k;     // this layer's K pool [num_blocks][Hkv][16][D]
  __half* cache_v;
  int64_t num_slots;
  // Launched right behind the prefill kernel of the same pass: its inputs were final once that kernel
  // passed its own dependency wait, so the decode runs in the prefill's tail (on SMs the prefill has left)
  // and waits for it only at its end, so that whatever follows sees both complete.
  int late_wait;
  int layer_row0_k;    // TMA row of (layer, K, block 0, head 0, slot 0)
  int layer_row0_v;    // TMA row of (layer, V, block 0, head 0, slot 0)
  int max_blocks;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int split_blocks;
  int max_splits;
  float scale_log2;  // log2(e) / sqrt(head_dim)
};

// Byte offset of 16-byte chunk c (8 dims) of key row r inside a ring slot written by 64-value TMA boxes
// with the 128-byte swizzle: box c / 8, row r at 128 bytes, chunk slot (c % 8) XOR (r % 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------------------------------
// Per-warp stream.  Measured on this access pattern (scattered 4 KB runs): one issuing thread per CTA
// tops out near 6 GB/s whatever the ring depth, while 12-16 issuing warps per SM reach 5.6-6 TB/s -- so
// every warp streams its own runs.  The next task's metadata loads overlap the current task's compute,
// and the next task's first runs enter the ring before the current task ends.
// ---------------------------------------------------------------------------------------------------
struct TaskMeta {
  int t, g, s, row, ctx, nsplit;
  int nbw;  // blocks of the split dealt to this warp: blocks warp, warp + NW, ...
  int ids;  // lane j holds the physical id of this warp's block j (j < nbw <= 8)
  int nst;  // fused append: the row's first position appended this pass (its token is t - (ctx-1 - nst))
};

template <int NW>
__device__ __forceinline__ void task_from_record(const DecodeParams& p, int4 rec, int warp, TaskMeta& m) {
  m.t = rec.x;
  m.g = rec.y & 0xFF;
  m.s = rec.y >> 8;
  m.row = rec.z;
  m.ctx = rec.w;
  const int nblk = (m.ctx + kBS - 1) / kBS;
  const int nb = m.t >= 0 ? min(p.split_blocks, nblk - m.s * p.split_blocks) : 0;
  m.nbw = nb > warp ? (nb - warp + NW - 1) / NW : 0;
  m.nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
}

__device__ __forceinline__ int4 load_record(const DecodeParams& p, int idx, int n_tasks) {
  return idx < n_tasks ? __ldcg(p.tasks + idx) : make_int4(-1, 0, 0, 0);
}

// First position of the row that this pass appends (fused append only): the row's first token sits at
// position ctx - 1 - (t - query_start_loc[row]).
__device__ __forceinline__ int load_nst(const DecodeParams& p, const TaskMeta& m) {
  if (p.k_in == nullptr || m.t < 0) return 1 << 30;
  return m.ctx - 1 - (m.t - __ldcg(p.qsl + m.row));
}

template <int NW>
__device__ __forceinline__ int load_ids(const DecodeParams& p, const TaskMeta& m, int warp, int lane) {
  int id = 0;
  if (lane < m.nbw) {
    id = __ldcg(p.block_tables + (int64_t)m.row * p.max_blocks + m.s * p.split_blocks + warp + NW * lane);
    if (id < 0 || id >= p.num_blocks) {
      dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
      id = 0;  // keep the copy in bounds; this token's output is flagged as invalid
    }
  }
  return id;
}

template <int D, int G>
struct Worker {
  using T = DecodeTraits<D, G>;
  const DecodeParams& p;
  unsigned char* ring;   // this warp's NR slots (1024-byte aligned)
  uint64_t* bars;        // this warp's NR barriers
  const volatile int* idx_ring;  // the CTA's task indices: task k at [k % 4]
  uint64_t pol;
  int warp, lane;
  int n_tasks;
  int k = 0;             // the CTA's sequence number of the current task
  int issued = 0;        // runs issued into the ring so far
  int consumed = 0;      // runs taken out of the ring so far
  int icur = 0;          // 0: the issue cursor is in the current task, 1: in the next one
  int ir = 0;            // run index of the issue cursor: 0 q, 1 + 2j K of block j, 2 + 2j V of block j
  int nstage = 0;        // next task's metadata: 0 nothing, 1 record loaded, 2 ids loaded
  int4 nxt_rec;
  TaskMeta cur, nxt;
  bool ok = true;

  __device__ Worker(const DecodeParams& p_, unsigned char* ring_, uint64_t* bars_, const int* idx_ring_,
                    int warp_, int lane_)
      : p(p_), ring(ring_), bars(bars_), idx_ring(idx_ring_), warp(warp_), lane(lane_) {
    pol = dev::l2_policy_evict_first();
    n_tasks = __ldcg(&p.hdr->n_tasks);
    task_from_record<T::NW>(p, load_record(p, idx_ring[0], n_tasks), warp, cur);
    cur.ids = load_ids<T::NW>(p, cur, warp, lane);
    cur.nst = load_nst(p, cur);
  }

  static __device__ __forceinline__ int runs(const TaskMeta& m) { return m.t >= 0 && m.nbw > 0 ? 1 + 2 * m.nbw : 0; }

  // Advance the next task's metadata by one dependent load (called between blocks so each load's
  // latency hides behind compute); full == true finishes it now.
  __device__ __forceinline__ void prefetch_next(bool full) {
    if (nstage == 0) {
      nxt_rec = load_record(p, idx_ring[(k + 1) & 3], n_tasks);
      nstage = 1;
      if (!full) return;
    }
    if (nstage == 1) {
      task_from_record<T::NW>(p, nxt_rec, warp, nxt);
      nxt.ids = load_ids<T::NW>(p, nxt, warp, lane);
      nxt.nst = load_nst(p, nxt);
      nstage = 2;
    }
  }
  __device__ __forceinline__ void issue_run(const TaskMeta& m, int r) {
    const int slot = issued % T::NR;
    unsigned char* dst = ring + slot * T::RUN;
    if (r == 0) {
      if (lane == 0) {
        dev::mbar_arrive_expect_tx(&bars[slot], G * D * 2);
        dev::bulk_g2s(dst, p.q + ((size_t)m.t * p.num_q_heads + (size_t)m.g * G) * D, G * D * 2, &bars[slot], pol);
      }
    } else {
      const int id = __shfl_sync(0xffffffffu, m.ids, (r - 1) >> 1);
      if (lane == 0) {
        const int row = (((r - 1) & 1) ? p.layer_row0_v : p.layer_row0_k) + (id * p.num_kv_heads + m.g) * kBS;
        dev::mbar_arrive_expect_tx(&bars[slot], T::RUN);
#pragma unroll
        for (int b = 0; b < T::BOXES; ++b) dev::tma_load_2d(dst + b * 2048, &p.kv_map, b * 64, row, &bars[slot], pol);
      }
    }
    ++issued;
  }
  // Issue the next run of the stream (current task, then the next task), if there is one.
  __device__ __forceinline__ bool issue_next() {
    if (icur == 0) {
      if (ir < runs(cur)) {
        issue_run(cur, ir++);
        return true;
      }
      icur = 1;
      ir = 0;
    }
    prefetch_next(true);
    if (ir < runs(nxt)) {
      issue_run(nxt, ir++);
      return true;
    }
    return false;
  }
  // Top the ring up.  It runs dry when the warp had no blocks in the task just finished (a short split
  // deals nothing to some warps), since only consuming a run issues the next one.
  __device__ __forceinline__ void fill() {
    while (issued - consumed < T::NR && issue_next()) {
    }
  }
  // Wait for the oldest run in the ring; returns its slot's shared-memory address.
  __device__ __forceinline__ uint32_t wait_run() {
    const int slot = consumed % T::NR;
    if (!dev::mbar_wait(&bars[slot], (consumed / T::NR) & 1)) {
      if (lane == 0) dev::set_error(p.err, PKV_DEVERR_WAIT_TIMEOUT);
      ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    return dev::smem_addr(ring + slot * T::RUN);
  }
  // The warp is done with the oldest run: recycle its slot for the next run of the stream.
  __device__ __forceinline__ void release_run() {
    __syncwarp();
    ++consumed;
    if (ok) issue_next();
  }
  // Move to the next task; the issue cursor is already inside it.
  __device__ __forceinline__ void advance() {
    prefetch_next(true);
    cur = nxt;
    ++k;
    icur = 0;
    nstage = 0;
  }
  // Before leaving early (a wait gave up): let the copies still in flight land, each wait bounded.
  __device__ __forceinline__ void drain() {
    for (; consumed < issued; ++consumed) dev::mbar_wait(&bars[consumed % T::NR], (consumed / T::NR) & 1);
  }
};

// Output element held by register r of `lane` in the O^T fragment layout: its dim and its head.
__device__ __forceinline__ void frag_coord(int lane, int r, int& dim, int& head) {
  dim = 16 * (r >> 2) + (lane >> 2) + ((r & 2) ? 8 : 0);
  head = ((lane & 3) << 1) + (r & 1);
}
// ... and back: the lane and register holding (dim, head).
__device__ __forceinline__ void frag_slot(int dim, int head, int& lane, int& r) {
  lane = ((dim & 7) << 2) | (head >> 1);
  r = ((dim >> 4) << 2) | (((dim >> 3) & 1) << 1) | (head & 1);
}

// Merge a token's split partials (all of them final) into its fp16 output, with log-sum-exp weights in
// split order, so the result does not depend on which CTA merges.  The partials were written by other
// CTAs during this launch: they are read from L2 (.cg), never from a possibly stale L1 line.
template <int D, int G, int NT>
__device__ __forceinline__ void merge_splits(const DecodeParams& p, int tg, int nsplit) {
  constexpr int NG = G * D / 4;            // groups of 4 consecutive dims of one head
  constexpr int EG = (NG + NT - 1) / NT;   // groups per thread
  constexpr int U = EG >= 4 ? 2 : 4;       // splits whose loads are in flight together
  const int t = tg / p.num_kv_heads, g = tg % p.num_kv_heads;
  const size_t sb = (size_t)tg * p.max_splits;
  float M[EG], L[EG];
  float4 acc[EG];
#pragma unroll
  for (int j = 0; j < EG; ++j) {
    M[j] = -INFINITY;
    L[j] = 0.f;
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s0 = 0; s0 < nsplit; s0 += U) {
    float2 ml[EG][U];
    float4 o[EG][U];
#pragma unroll
    for (int j = 0; j < EG; ++j) {
      const int e4 = threadIdx.x + j * NT;
      const int h = (4 * e4) / D, dim = (4 * e4) % D;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (e4 < NG && s0 + u < nsplit) {
          const size_t pi = (sb + s0 + u) * kHeadsTile + h;
          ml[j][u] = __ldcg(p.part_ml + pi);
          o[j][u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + pi * D + dim));
        }
      }
    }
#pragma unroll
    for (int j = 0; j < EG; ++j) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (s0 + u < nsplit) {
          const float nM = fmaxf(M[j], ml[j][u].x);
          const float a = exp2f(M[j] - nM), f = exp2f(ml[j][u].x - nM);
          M[j] = nM;
          L[j] = L[j] * a + ml[j][u].y * f;
          acc[j].x = acc[j].x * a + o[j][u].x * f;
          acc[j].y = acc[j].y * a + o[j][u].y * f;
          acc[j].z = acc[j].z * a + o[j][u].z * f;
          acc[j].w = acc[j].w * a + o[j][u].w * f;
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < EG; ++j) {
    const int e4 = threadIdx.x + j * NT;
    if (e4 >= NG) continue;
    const int h = (4 * e4) / D, dim = (4 * e4) % D;
    const float il = 1.f / L[j];
    const __half2 lo = __floats2half2_rn(acc[j].x * il, acc[j].y * il);
    const __half2 hi = __floats2half2_rn(acc[j].z * il, acc[j].w * il);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&lo);
    v.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.num_q_heads + (size_t)g * G + h) * D + dim) = v;
  }
}

template <int D, int G>
__device__ __forceinline__ void worker_loop(const DecodeParams& p, unsigned char* smem, int warp, int lane) {
  using T = DecodeTraits<D, G>;
  uint64_t* all_bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  float* co = reinterpret_cast<float*>(smem + T::OFF_CO);
  float* cm = reinterpret_cast<float*>(smem + T::OFF_CM);
  float* cl = reinterpret_cast<float*>(smem + T::OFF_CL);
  int* idx_ring = reinterpret_cast<int*>(smem + T::OFF_IDX);
  // The first task's record and block ids are loaded before the dependency wait: the plan kernel that
  // wrote the task list released its dependents only after its writes (and a fence), and block tables
  // are final before the plan; they are read through L2, never a possibly stale L1 line.  The task
  // counters, q and the cache (written by the append just before) are touched only after the wait.
  Worker<D, G> w(p, smem + warp * T::NR * T::RUN, all_bars + warp * T::NR, idx_ring, warp, lane);
  if (!p.late_wait) dev::griddep_wait();
  dev::griddep_launch_dependents();
  // one CTA-uniform decision (a racing error-word update must not split the CTA)
  if (__syncthreads_or(threadIdx.x == 0 && dev::pool_poisoned(p.err))) return;
  // Split completion (thread 0 only): after writing a split's partial the CTA counts it on the token's
  // counter, and the CTA that completes the count merges the token.  The count's result is examined only
  // at the end of the CTA's next task, so its round trip never stalls the stream.
  int pend_tg = -1, pend_prev = 0, pend_ns = 0;
  auto resolve_pending = [&]() {  // thread 0: publish the token this CTA must merge, or -1
    int tg = -1;
    if (pend_tg >= 0 && pend_prev == pend_ns - 1) {
      tg = pend_tg;
      p.merge_cnt[tg] = 0;       // ready for the next launch on this plan
      dev::fence_acq_rel_gpu();  // acquire: the other splits' partials, released with their counts
    }
    idx_ring[4] = tg;
    idx_ring[5] = pend_ns;
    pend_tg = -1;
  };

  const int qh = lane >> 2;        // head whose q this lane feeds to the MMA (B operand column); key row too
  const int h0 = (lane & 3) << 1;  // heads of this lane's score / output columns: h0, h0 + 1
  int pending = 0;                 // thread 0: index of the task two ahead, published at the task's end
  bool cta_ok = true;              // CTA-uniform: no wait gave up
  while (w.cur.t >= 0) {           // uniform: every warp reads the same index
    if (threadIdx.x == 0) pending = 2 * (int)gridDim.x + atomicAdd(&p.hdr->work, 1);
    const TaskMeta d = w.cur;
    w.fill();
    w.prefetch_next(false);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[T::MT][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    if (d.nbw > 0 && w.ok) {
      // ---- q as the MMA B operand (Q^T: k = dims, n = heads), from the task's first ring run ----
      // Rows G..7 of the 8-row tile hold stale bytes; they only feed score and output columns of heads
      // >= G, which are never written out.
      uint32_t qb[T::KS][2];
      const uint32_t qs = w.wait_run();
#pragma unroll
      for (int k2 = 0; k2 < T::KS / 2; ++k2) {
        uint32_t r4[4];
        dev::ldsm_x4(qs + (lane & 7) * (D * 2) + (4 * k2 + (lane >> 3)) * 16, r4);
        qb[2 * k2][0] = r4[0];
        qb[2 * k2][1] = r4[1];
        qb[2 * k2 + 1][0] = r4[2];
        qb[2 * k2 + 1][1] = r4[3];
      }
      w.release_run();

      for (int j = 0; j < d.nbw && w.ok; ++j) {
        const int bpos = (d.s * p.split_blocks + warp + T::NW * j) * kBS;  // the block's first position
        const int ntok = min(kBS, d.ctx - bpos);
        // fused append: positions ov0 .. bpos + ntok - 1 of the block are this pass's tokens; their rows
        // come from the inputs (the cache may not hold them yet), and the block holding the token's own
        // position writes it into the cache
        const int ov0 = max(bpos, d.nst), nov = bpos + ntok - ov0;
        auto override_rows = [&](uint32_t base, const __half* src) {
          for (int idx = lane; idx < nov * (D / 8); idx += 32) {
            const int rr = ov0 - bpos + idx / (D / 8), cc = idx % (D / 8);
            const int tk = d.t - (d.ctx - 1 - (bpos + rr));
            const uint4 v = __ldcg(reinterpret_cast<const uint4*>(src + ((size_t)tk * p.num_kv_heads + d.g) * D) + cc);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(rr, cc)), "r"(v.x), "r"(v.y),
                         "r"(v.z), "r"(v.w)
                         : "memory");
          }
          __syncwarp();
        };
        if (nov > 0 && d.ctx - 1 < bpos + kBS) {
          const int64_t slot = __ldcg(p.slots + d.t);
          if (slot != -1) {
            if (slot < 0 || slot >= p.num_slots) {
              if (lane == 0) dev::set_error(p.err, PKV_DEVERR_SLOT_RANGE);
            } else {
              const size_t src = ((size_t)d.t * p.num_kv_heads + d.g) * D;
              const size_t dst = (((size_t)(slot >> 4) * p.num_kv_heads + d.g) * kBS + (slot & 15)) * D;
              for (int cc = lane; cc < D / 8; cc += 32) {
                reinterpret_cast<uint4*>(p.cache_k + dst)[cc] = __ldcg(reinterpret_cast<const uint4*>(p.k_in + src) + cc);
                reinterpret_cast<uint4*>(p.cache_v + dst)[cc] = __ldcg(reinterpret_cast<const uint4*>(p.v_in + src) + cc);
              }
            }
          }
        }
        // ---- S^T[16 keys x 8 heads] = K Q^T on the tensor cores ----
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const uint32_t ks_base = w.wait_run();
          if (nov > 0) override_rows(ks_base, p.k_in);
          const int kr = (lane & 7) + ((lane >> 3) & 1) * 8;  // key row this lane addresses for ldmatrix
#pragma unroll
          for (int ks = 0; ks < T::KS; ++ks) {
            uint32_t a[4];
            dev::ldsm_x4(ks_base + swz(kr, 2 * ks + (lane >> 4)), a);
            dev::mma_16816(sc, a, qb[ks][0], qb[ks][1]);
          }
          if (nov > 0) dev::fence_proxy_async_smem();  // the override precedes the slot's next TMA write
          w.release_run();
        }
        w.prefetch_next(false);  // one dependent metadata load of the next task per block, hidden by compute
        // ---- online softmax (log2 domain); the lane holds keys qh, qh + 8 for heads h0, h0 + 1 ----
        const bool v0 = qh < ntok, v1 = qh + 8 < ntok;
        const float s0 = v0 ? sc[0] * p.scale_log2 : -INFINITY;  // key qh,     head h0
        const float s1 = v0 ? sc[1] * p.scale_log2 : -INFINITY;  // key qh,     head h0 + 1
        const float s2 = v1 ? sc[2] * p.scale_log2 : -INFINITY;  // key qh + 8, head h0
        const float s3 = v1 ? sc[3] * p.scale_log2 : -INFINITY;  // key qh + 8, head h0 + 1
        float b0 = fmaxf(s0, s2), b1 = fmaxf(s1, s3);
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
          b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, m));
          b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, m));
        }
        const float n0 = fmaxf(m0, b0), n1 = fmaxf(m1, b1);
        const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
        m0 = n0;
        m1 = n1;
        const float p0 = exp2f(s0 - n0), p1 = exp2f(s1 - n1), p2 = exp2f(s2 - n0), p3 = exp2f(s3 - n1);
        l0 = l0 * a0 + p0 + p2;
        l1 = l1 * a1 + p1 + p3;
#pragma unroll
        for (int mt = 0; mt < T::MT; ++mt) {
          o[mt][0] *= a0;
          o[mt][1] *= a1;
          o[mt][2] *= a0;
          o[mt][3] *= a1;
        }
        // P^T as the B operand (k = keys, n = heads): transpose the [keys x heads] 8x8 fragments
        const __half2 pk0 = __floats2half2_rn(p0, p1), pk1 = __floats2half2_rn(p2, p3);
        const uint32_t pb0 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk0));
        const uint32_t pb1 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk1));
        // ---- O^T[d x 8 heads] += V^T P^T on the tensor cores ----
        {
          const uint32_t vs_base = w.wait_run();
          if (ntok < kBS) {  // rows past the context may hold anything: zero them so 0 * garbage cannot poison O
            for (int idx = lane; idx < (kBS - ntok) * (D / 8); idx += 32) {
              const int r = ntok + idx / (D / 8), c = idx % (D / 8);
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vs_base + swz(r, c)), "r"(0) : "memory");
            }
            __syncwarp();
          }
          if (nov > 0) override_rows(vs_base, p.v_in);
          const int mat = lane >> 3;                      // ldmatrix matrix this lane addresses
          const int vr = (lane & 7) + ((mat >> 1) << 3);  // its key row
#pragma unroll
          for (int mt = 0; mt < T::MT; ++mt) {
            uint32_t a[4];
            dev::ldsm_x4_t(vs_base + swz(vr, 2 * mt + (mat & 1)), a);
            dev::mma_16816(o[mt], a, pb0, pb1);
          }
          if (ntok < kBS || nov > 0) dev::fence_proxy_async_smem();  // generic writes precede the next TMA write
          w.release_run();
        }
      }
    }

    // ---- publish this warp's share of the split; a warp with no blocks publishes (-inf, 0, 0) ----
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, m);
      l1 += __shfl_xor_sync(0xffffffffu, l1, m);
    }
#pragma unroll
    for (int r = 0; r < T::OV; ++r) co[(warp * T::OV + r) * 32 + lane] = o[r >> 2][r & 3];
    if (lane < 4) {
      cm[warp * kHeadsTile + h0] = m0;
      cm[warp * kHeadsTile + h0 + 1] = m1;
      cl[warp * kHeadsTile + h0] = l0;
      cl[warp * kHeadsTile + h0 + 1] = l1;
    }
    if (threadIdx.x == 0) {
      idx_ring[(w.k + 2) & 3] = pending;
      resolve_pending();
    }
    if (!__syncthreads_and(w.ok)) {  // a wait gave up somewhere in the CTA: stop together
      cta_ok = false;
      break;
    }
    if (idx_ring[4] >= 0) merge_splits<D, G, T::NTHREADS>(p, idx_ring[4], idx_ring[5]);

    // ---- combine the warps' shares with log-sum-exp weights; write the output or the split's partial ----
    const size_t pidx = ((size_t)d.t * p.num_kv_heads + d.g) * p.max_splits + d.s;
    for (int e = threadIdx.x; e < G * D; e += T::NTHREADS) {
      const int h = e / D, dim = e % D;
      int ln, r;
      frag_slot(dim, h, ln, r);
      float M = cm[h];
#pragma unroll
      for (int v = 1; v < T::NW; ++v) M = fmaxf(M, cm[v * kHeadsTile + h]);
      float L = 0.f, acc = 0.f;
#pragma unroll
      for (int v = 0; v < T::NW; ++v) {
        const float f = exp2f(cm[v * kHeadsTile + h] - M);
        L += cl[v * kHeadsTile + h] * f;
        acc += co[(v * T::OV + r) * 32 + ln] * f;
      }
      if (d.nsplit == 1) {
        p.out[((size_t)d.t * p.num_q_heads + (size_t)d.g * G + h) * D + dim] = __float2half_rn(acc / L);
      } else {
        p.part_o[(pidx * kHeadsTile + h) * D + dim] = acc;
        if (dim == 0) p.part_ml[pidx * kHeadsTile + h] = make_float2(M, L);
      }
    }
    __syncthreads();  // the combine buffers are free again; the partial is written
    if (threadIdx.x == 0 && d.nsplit > 1 && d.nsplit <= kFusedMergeSplits) {
      pend_tg = d.t * p.num_kv_heads + d.g;
      pend_prev = dev::atom_add_release_gpu(p.merge_cnt + pend_tg, 1);  // releases the CTA's partial
      pend_ns = d.nsplit;
    }
    w.advance();
  }
  if (cta_ok) {  // the CTA's last split may still complete a token
    if (threadIdx.x == 0) resolve_pending();
    __syncthreads();
    if (idx_ring[4] >= 0) merge_splits<D, G, T::NTHREADS>(p, idx_ring[4], idx_ring[5]);
  }
  if (!w.ok || w.consumed < w.issued) w.drain();
}

template <int D, int G>
__global__ void __launch_bounds__(DecodeTraits<D, G>::NTHREADS, DecodeTraits<D, G>::MINB)
decode_kernel(const __grid_constant__ DecodeParams p) {
  using T = DecodeTraits<D, G>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  int* idx_ring = reinterpret_cast<int*>(smem + T::OFF_IDX);
  // set-up that reads nothing written by earlier kernels runs before the dependency wait
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int i = 0; i < T::NR; ++i) dev::mbar_init(&bars[warp * T::NR + i], 1);
    dev::fence_mbar_init();
  }
  if (threadIdx.x == 0) {  // the first two tasks are static: no counter round trip before the first copy
    idx_ring[0] = blockIdx.x;
    idx_ring[1] = blockIdx.x + gridDim.x;
  }
  __syncthreads();
  worker_loop<D, G>(p, smem, warp, lane);  // waits for the previous kernel itself, after its first loads
  // the last CTA out resets the task counter for the next launch on this plan
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.hdr->done, 1) == (int)gridDim.x - 1) {
      p.hdr->work = 0;
      p.hdr->done = 0;
      __threadfence();
    }
  }
  if (p.late_wait) dev::griddep_wait();  // complete only after the prefill kernel ahead of it
}

// ---------------------------------------------------------------------------------------------------
// Merge of tokens with more than kFusedMergeSplits splits.  Grid (token, KV head, chunk of partial
// elements), 256 threads = SG split groups x (256 / SG) element threads; element e of a partial is head
// e / D, dim e % D.
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

template <int D, int SG>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  constexpr int TE = 256 / SG;                        // threads along the elements
  constexpr int EPC = SG == 1 ? kHeadsTile * D : TE;  // elements per CTA
  constexpr int EPT = EPC / TE;              // elements per thread
  __shared__ float sM[kHeadsTile], sL[kHeadsTile];
  __shared__ float red[256];
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int t = blockIdx.x, g = blockIdx.y;
  const int ctx = __ldg(p.tok_ctx + t);
  if (ctx <= 0) return;
  const int nblk = (ctx + kBS - 1) / kBS;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  if (nsplit <= kFusedMergeSplits || (int)blockIdx.z * EPC >= p.group * D) return;
  const size_t sb = ((size_t)t * p.num_kv_heads + g) * p.max_splits;
  const int tid = threadIdx.x;
  // per-head max and sum over the splits: thread (head tid % 8, split stride group tid / 8)
  {
    const int h = tid & 7;
    float M = -INFINITY;
    for (int s = tid >> 3; s < nsplit; s += 32) M = fmaxf(M, p.part_ml[(sb + s) * kHeadsTile + h].x);
    red[tid] = M;
    __syncthreads();
    if (tid < 8) {
      float x = red[tid];
      for (int k = 1; k < 32; ++k) x = fmaxf(x, red[tid + 8 * k]);
      sM[tid] = x;
    }
    __syncthreads();
    M = sM[h];
    float L = 0.f;
    for (int s = tid >> 3; s < nsplit; s += 32) {
      const float2 ml = p.part_ml[(sb + s) * kHeadsTile + h];
      L += ml.y * exp2f(ml.x - M);
    }
    __syncthreads();
    red[tid] = L;
    __syncthreads();
    if (tid < 8) {
      float x = 0.f;
      for (int k = 0; k < 32; ++k) x += red[tid + 8 * k];
      sL[tid] = x;
    }
    __syncthreads();
  }
  const int te = tid % TE, sg = tid / TE;
  const int E = p.group * D;  // elements that belong to real query heads
  float acc[EPT];
  int heads[EPT];
#pragma unroll
  for (int k = 0; k < EPT; ++k) {
    const int e = blockIdx.z * EPC + te + k * TE;
    heads[k] = min(e / D, kHeadsTile - 1);
    acc[k] = 0.f;
  }
  for (int s = sg; s < nsplit; s += SG) {
    const float* po = p.part_o + (sb + s) * kHeadsTile * D;
    const float2* pml = p.part_ml + (sb + s) * kHeadsTile;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int e = blockIdx.z * EPC + te + k * TE;
      if (e < E) acc[k] += po[e] * exp2f(pml[heads[k]].x - sM[heads[k]]);
    }
  }
#pragma unroll
  for (int k = 0; k < EPT; ++k) {
    if constexpr (SG > 1) {
      __syncthreads();
      red[tid] = acc[k];
      __syncthreads();
      if (sg != 0) continue;
      for (int j = 1; j < SG; ++j) acc[k] += red[te + j * TE];
    }
    const int e = blockIdx.z * EPC + te + k * TE;
    if (e < E)
      p.out[((size_t)t * p.num_q_heads + (size_t)g * p.group + heads[k]) * D + e % D] =
          __float2half_rn(acc[k] / sL[heads[k]]);
  }
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
  int32_t* tok_row;
  int32_t* tok_ctx;
  int32_t* merge_cnt;
  int4* tasks;
  int4* items;
  int32_t* items_slot;
  int2* pf_sync;
  int max_slots;
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
    fn((w + npos + kPrefillKeys - 1) / kPrefillKeys, npos, q0 + qb * p.prefill_pos, w);
  }
}

// K/V tiles of the two chunks of an item of n tiles (the first chunk takes the extra tile).
__device__ __forceinline__ int split_first(int n) { return (n + 1) / 2; }

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
  __shared__ int warp_sums[32];
  __shared__ int hist[kPrefillBuckets];
  __shared__ int n_slots;
  dev::griddep_wait();
  for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
    const int q0 = __ldg(p.qsl + i), q1 = __ldg(p.qsl + i + 1), ctx = __ldg(p.context_lens + i);
    if (q1 < q0 || (i == 0 && q0 != 0) || (i == p.num_seqs - 1 && q1 != p.num_tokens))
      dev::set_error(p.err, PKV_DEVERR_QSL);
    if (!row_meta_ok(q1 - q0, ctx, p.max_ctx)) dev::set_error(p.err, PKV_DEVERR_ROW_META);
  }
  for (int i = threadIdx.x; i < p.num_tokens * p.num_kv_heads; i += blockDim.x) p.merge_cnt[i] = 0;
  for (int i = threadIdx.x; i < kPrefillBuckets; i += blockDim.x) hist[i] = 0;
  for (int i = threadIdx.x; i < p.max_slots; i += blockDim.x) p.pf_sync[i] = make_int2(0, 0);
  if (threadIdx.x == 0) n_slots = 0;

  // ---- decode tasks: tokens of rows that are not prefill items ----
  // Pass 0 lists each token's short last split, pass 1 its full splits in token order: tokens then
  // complete, and get merged, all through the launch rather than together at its end, and the launch
  // ends on equal-sized tasks.
  int carry = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int base = 0; base < p.num_tokens; base += blockDim.x) {
      const int t = base + threadIdx.x;
      int nblk = 0, row = 0, c = 0;
      if (t < p.num_tokens) {
        if (pass == 0) {
          const int b = dev::row_of_token(p.qsl, p.num_seqs, t);
          const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1), ctx = __ldg(p.context_lens + b);
          const int q_len = q1 - q0;
          const bool prefill = p.prefill_min_qlen > 0 && q_len >= p.prefill_min_qlen;
          if (t >= q0 && t < q1 && row_meta_ok(q_len, ctx, p.max_ctx) && !prefill) c = ctx - q_len + (t - q0) + 1;
          p.tok_row[t] = b;
          p.tok_ctx[t] = c;  // 0: no decode work (prefill row or invalid metadata)
          row = b;
        } else {
          c = p.tok_ctx[t];
          row = p.tok_row[t];
        }
        nblk = (c + kBS - 1) / kBS;
      }
      const int nfull = nblk / p.split_blocks;
      const int ntail = nblk % p.split_blocks ? 1 : 0;
      const int cnt = (pass == 0 ? ntail : nfull) * p.num_kv_heads;
      int total = 0;
      const int off = carry + block_exclusive_scan(cnt, warp_sums, &total);
      if (cnt > 0) {
        if (pass == 0) {
          for (int g = 0; g < p.num_kv_heads; ++g) p.tasks[off + g] = make_int4(t, g | (nfull << 8), row, c);
        } else {
          for (int g = 0; g < p.num_kv_heads; ++g)
            for (int s = 0; s < nfull; ++s) p.tasks[off + g * nfull + s] = make_int4(t, g | (s << 8), row, c);
        }
      }
      carry += total;
      __syncthreads();  // warp_sums is reused by the next chunk
    }
  }

  // ---- prefill work entries, bucketed by K/V tile count, longest first; long items in two chunks ----
  auto bucket_of = [](int cost) { return kPrefillBuckets - 1 - min(cost, kPrefillBuckets - 1); };
  for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x)
    for_row_items(p, b, [&](int n, int, int, int) {
      if (n > kPrefillSplitTiles) {
        atomicAdd(&hist[bucket_of(split_first(n))], p.num_kv_heads);
        atomicAdd(&hist[bucket_of(n - split_first(n))], p.num_kv_heads);
      } else {
        atomicAdd(&hist[bucket_of(n)], p.num_kv_heads);
      }
    });
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
  for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x)
    for_row_items(p, b, [&](int n, int npos, int t0, int w) {
      const bool split = n > kPrefillSplitTiles;
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

  if (threadIdx.x == 0) {
    p.hdr->n_tasks = carry;
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
  const bool prefill = prefill_supported(c.head_dim, group) && c.num_kv_heads < 256;
  w.prefill_min_qlen = prefill ? kPrefillMinQlen : 0;
  w.prefill_pos = prefill_item_positions(group);
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
  w.total = off;
  return w;
}

template <int D, int G>
static cudaError_t launch_decode(const DecodeParams& p, int num_sms, int64_t max_tasks, cudaStream_t stream) {
  using T = DecodeTraits<D, G>;
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, G>, T::NTHREADS, T::SMEM);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
  }
  int64_t grid = (int64_t)num_sms * per_sm;  // persistent: one CTA per resident slot, one task at a time
  if (grid > max_tasks) grid = max_tasks;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_kernel<D, G>, dim3((unsigned)grid), dim3(T::NTHREADS), T::SMEM, stream, p);
}

template <int D>
static cudaError_t launch_decode_g(int group, const DecodeParams& p, int num_sms, int64_t max_tasks,
                                   cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode<D, 1>(p, num_sms, max_tasks, stream);
    case 2: return launch_decode<D, 2>(p, num_sms, max_tasks, stream);
    case 4: return launch_decode<D, 4>(p, num_sms, max_tasks, stream);
    case 6: return launch_decode<D, 6>(p, num_sms, max_tasks, stream);
    case 8: return launch_decode<D, 8>(p, num_sms, max_tasks, stream);
    default: return cudaErrorInvalidValue;
  }
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
  p.tok_row = reinterpret_cast<int32_t*>(ws + w.tok_row);
  p.tok_ctx = reinterpret_cast<int32_t*>(ws + w.tok_ctx);
  p.merge_cnt = reinterpret_cast<int32_t*>(ws + w.merge_cnt);
  p.tasks = reinterpret_cast<int4*>(ws + w.tasks);
  p.items = reinterpret_cast<int4*>(ws + w.items);
  p.items_slot = reinterpret_cast<int32_t*>(ws + w.items_slot);
  p.pf_sync = reinterpret_cast<int2*>(ws + w.pf_sync);
  p.max_slots = (int)w.max_items;
  p.hdr = reinterpret_cast<WsHeader*>(ws + w.hdr);
  p.err = pool->dev_error;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p);
}

// Inputs of an append fused into the decode launch (k == nullptr: not fused).
struct FusedAppend {
  const void* k = nullptr;
  const void* v = nullptr;
  const int64_t* slots = nullptr;
  const int32_t* qsl = nullptr;
};

// decode (+ merge of very long tokens) and prefill tiles for one layer on a planned workspace
static pkv_status launch_attention(pkv_pool* pool, int layer, const void* q, const int32_t* block_tables,
                                   int max_blocks, int num_seqs, int num_tokens, void* out, char* ws,
                                   const WsLayout& w, cudaStream_t s, int* launches,
                                   const FusedAppend& fa = FusedAppend()) {
  const pkv_config& c = pool->cfg;
  DecodeParams p;
  p.kv_map = pool->kv_map;
  p.q = static_cast<const __half*>(q);
  p.block_tables = block_tables;
  p.tok_row = reinterpret_cast<const int32_t*>(ws + w.tok_row);
  p.tok_ctx = reinterpret_cast<const int32_t*>(ws + w.tok_ctx);
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
  p.qsl = fa.qsl;
  p.cache_k = static_cast<__half*>(pkv_pool_layer_ptr(pool, layer, 0));
  p.cache_v = static_cast<__half*>(pkv_pool_layer_ptr(pool, layer, 1));
  p.num_slots = (int64_t)c.num_blocks * c.block_size;
  const int rows_per_pool = c.num_blocks * c.num_kv_heads * c.block_size;
  p.layer_row0_k = (layer * 2) * rows_per_pool;
  p.layer_row0_v = (layer * 2 + 1) * rows_per_pool;
  p.max_blocks = max_blocks;
  p.num_q_heads = c.num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.num_blocks = c.num_blocks;
  p.split_blocks = c.split_blocks;
  p.max_splits = w.max_splits;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  const int group = c.num_q_heads / c.num_kv_heads;
  // Prefill rows exist only if some row has at least prefill_min_qlen new tokens.  Their tile kernel goes
  // first; the decode kernel follows in its tail (late_wait).
  p.late_wait = 0;
  cudaError_t e;
  if (w.prefill_min_qlen > 0 && num_tokens - num_seqs >= w.prefill_min_qlen - 1) {
    PrefillArgs a;
    a.kv_map = &pool->kv_map;
    a.q = q;
    a.out = out;
    a.block_tables = block_tables;
    a.items = reinterpret_cast<const int4*>(ws + w.items);
    a.items_slot = reinterpret_cast<const int32_t*>(ws + w.items_slot);
    a.pf_sync = reinterpret_cast<int2*>(ws + w.pf_sync);
    a.pf_ml = reinterpret_cast<float2*>(ws + w.pf_ml);
    a.pf_o = reinterpret_cast<float*>(ws + w.pf_o);
    a.hdr = p.hdr;
    a.err = p.err;
    a.layer_row0_k = p.layer_row0_k;
    a.layer_row0_v = p.layer_row0_v;
    a.max_blocks = max_blocks;
    a.num_q_heads = c.num_q_heads;
    a.num_kv_heads = c.num_kv_heads;
    a.num_blocks = c.num_blocks;
    a.head_dim = c.head_dim;
    a.num_sms = pool->num_sms;
    a.max_items = 2 * w.max_items;
    e = launch_prefill(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    *launches += 1;
    p.late_wait = 1;
  }
  switch (c.head_dim) {
    case 64: e = launch_decode_g<64>(group, p, pool->num_sms, w.max_tasks, s); break;
    case 128: e = launch_decode_g<128>(group, p, pool->num_sms, w.max_tasks, s); break;
    case 256: e = launch_decode_g<256>(group, p, pool->num_sms, w.max_tasks, s); break;
    default: return fail(PKV_ERR_UNSUPPORTED, "head_dim");
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  *launches += 1;
  if (w.max_splits > kFusedMergeSplits) {
    MergeParams m{p.part_o, p.part_ml, p.tok_ctx, p.out, c.num_q_heads, c.num_kv_heads, group, c.split_blocks,
                  w.max_splits};
    const dim3 grid(num_tokens, c.num_kv_heads, (kHeadsTile * c.head_dim) / 64);
    switch (c.head_dim) {
      case 64: e = launch_pdl(merge_kernel<64, 4>, grid, dim3(256), 0, s, m); break;
      case 128: e = launch_pdl(merge_kernel<128, 4>, grid, dim3(256), 0, s, m); break;
      default: e = launch_pdl(merge_kernel<256, 4>, grid, dim3(256), 0, s, m); break;
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

extern "C" pkv_status pkv_attention_plan(pkv_pool* pool, const int32_t* context_lens, const int32_t* query_start_loc,
                                         int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq);
  if (st == PKV_OK) st = check_workspace(pool, workspace, workspace_bytes, num_seqs, num_tokens, max_blocks_per_seq);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  pool->plan = PlanKey{workspace, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq};
  if (num_tokens == 0) return PKV_OK;
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  cudaError_t e = launch_plan(pool, static_cast<char*>(workspace), w, context_lens, query_start_loc, num_seqs,
                              num_tokens, max_blocks_per_seq, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    pool->plan = PlanKey{};
    return cuda_fail(e, "plan launch");
  }
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
  if (st != PKV_OK) return st;
  const PlanKey& k = pool->plan;
  if (k.workspace != workspace || k.context_lens != context_lens || k.query_start_loc != query_start_loc ||
      k.num_seqs != num_seqs || k.num_tokens != num_tokens || k.max_blocks_per_seq != max_blocks_per_seq)
    return fail(PKV_ERR_INVALID_ARG, "no matching plan: call pkv_attention_plan for this workspace and metadata");
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  int launches = 0;
  st = launch_attention(pool, layer, q, block_tables, max_blocks_per_seq, num_seqs, num_tokens, out,
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
  const PlanKey& pk = pool->plan;
  if (pk.workspace != workspace || pk.context_lens != context_lens || pk.query_start_loc != query_start_loc ||
      pk.num_seqs != num_seqs || pk.num_tokens != num_tokens || pk.max_blocks_per_seq != max_blocks_per_seq)
    return fail(PKV_ERR_INVALID_ARG, "no matching plan: call pkv_attention_plan for this workspace and metadata");
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  int launches = 0;
  if (w.max_items > 0) {  // prefill rows possible: they read the cache, so append first
    st = pkv_append(pool, layer, k, v, slot_mapping, num_tokens, stream);
    if (st != PKV_OK) return st;
    launches = pool->last_launches;
    st = launch_attention(pool, layer, q, block_tables, max_blocks_per_seq, num_seqs, num_tokens, out,
                          static_cast<char*>(workspace), w, (cudaStream_t)stream, &launches);
  } else {
    FusedAppend fa;
    fa.k = k;
    fa.v = v;
    fa.slots = slot_mapping;
    fa.qsl = query_start_loc;
    st = launch_attention(pool, layer, q, block_tables, max_blocks_per_seq, num_seqs, num_tokens, out,
                          static_cast<char*>(workspace), w, (cudaStream_t)stream, &launches, fa);
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

// The array's device address, looked up once per device with that device current.  In host code the
// symbol name itself is only a host-side stand-in and must never reach a kernel.
static void* noalloc_scratch_ptr(int device, cudaError_t* err) {
  static std::mutex mu;
  static void* cached[128] = {};
  *err = cudaSuccess;
  if (device < 0 || device >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[device]) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    cached[device] = ptr;
  }
  return cached[device];
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
  if (st != PKV_OK) return st;
  const WsLayout w = ws_layout(pool->cfg, num_seqs, num_tokens, max_blocks_per_seq);
  if (w.total > kNoAllocScratchBytes)
    return fail(PKV_ERR_OUT_OF_RANGE, "pass needs " + std::to_string(w.total) + " bytes of scratch; the built-in "
                "array holds " + std::to_string(kNoAllocScratchBytes) + " (use pkv_attention with a workspace)");
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (device != pool->device) return fail(PKV_ERR_INVALID_ARG, "the pool's device must be the current device");
  void* scratch = noalloc_scratch_ptr(device, &e);
  if (!scratch) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch array");
  // What must start at zero -- the task and split counters -- is cleared by the plan kernel on every call;
  // everything else is written before it is read.
  char* ws = static_cast<char*>(scratch);
  cudaStream_t s = (cudaStream_t)stream;
  e = launch_plan(pool, ws, w, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq, s);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  int launches = 1;
  st = launch_attention(pool, layer, q, block_tables, max_blocks_per_seq, num_seqs, num_tokens, out, ws, w, s,
                        &launches);
  pool->last_launches = launches;
  return st;
}
