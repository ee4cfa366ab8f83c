// The persistent split-K decode kernel: per-pass tasks (one split of one (token, KV head)) taken by
// persistent CTAs of four streaming warps, a combiner warp and a scheduler warp; the cache is streamed
// through per-warp TMA rings and the group contraction runs on warp MMAs.  Templated on the head
// dimension, the query heads per KV head and the cache format (fp16 values or 8-bit E4M3 codes with a
// power-of-two scale per cached row), so each format's instances compile in their own translation unit.
// How it fits the pass (plan, merge of long tokens, prefill, entry points) is described in attention.cu.
#pragma once

#include <cuda_fp16.h>

#include <cmath>

#include "attn_common.cuh"

namespace pkv {
constexpr int kFusedMergeSplits = 32;  // tokens with up to this many splits are merged inside the decode
constexpr int kMaxSplitBlocks = 32;   // upper bound on split_blocks (a split's block ids fit one warp)

// Ring slots per streaming warp: runs (a block's K or V for one KV head) in flight; fewer where the shared
// memory of two CTAs per SM does not hold them.  The 8-bit cache's runs are half as long and its warps go
// through them faster: its rings take every slot that fits (measured on the long-context decode: halving
// them nearly doubles the time).
#ifndef PKV_DECODE_RING
#define PKV_DECODE_RING(D) ((D) == 256 ? 2 : ((D) == 128 ? 5 : 8))
#endif

constexpr int kSmemPerSM = 228 * 1024;  // shared memory of one SM
constexpr int kSmemReservedPerCTA = 1024;
constexpr int kStaticTasks = 1;         // each CTA's first task comes without a counter (see Scheduler)
constexpr int kEagerClaimBlocks = 8;    // past tasks this small, the scheduler claims as early as slots allow

// One task as the scheduler warp hands it to the streaming warps and the combiner warp (shared memory).
struct TaskEntry {
  int4 rec;  // {token (-1: no more tasks), kv head | split << 8, row, causal context}
  int nst;   // the row's first position appended this pass
  int nb;    // blocks in the split
  int rot;   // block i of the split goes to streaming warp (i + rot) % 4 (a function of the row alone)
  int pad;
  int ids[kMaxSplitBlocks];  // the split's physical block ids
};

// Cache formats of the decode kernel (template parameter KV).
constexpr int kKvF16 = 0;   // fp16 values
constexpr int kKvE4M3 = 1;  // E4M3 codes with one power-of-two scale per cached (token, KV head) row

template <int D, int G, int KV>
struct DecodeTraits {
  static constexpr int NW = 4;                     // streaming warps; then the combiner and the scheduler
  static constexpr int NTHREADS = (NW + 2) * 32;
  static constexpr bool F8 = KV == kKvE4M3;
  static constexpr int RUN = kBS * D * (F8 ? 1 : 2);  // one (block, KV head) run of K or V
  static constexpr int BOXROWS = kBS * D / 128;    // 8-bit: 128-byte rows of a run (its box height)
  static constexpr int SCL = F8 ? 32 : 0;          // 8-bit: scale record per slot (the K and V scales of a block)
  static constexpr int RING = F8 ? 16 : PKV_DECODE_RING(D);  // 8-bit: as many slots as fit, up to 16
  static constexpr int KS = D / 16;                // MMA k-steps over the head dimension (scores)
  static constexpr int MT = D / 16;                // MMA m-tiles over the head dimension (values)
  static constexpr int OV = MT * 4;                // fp32 output values per lane (8-head fragment)
  static constexpr int LG = (G + 1) / 2;           // lanes l with (l & 3) < LG hold real heads
  static constexpr int SHL = 8 * LG;               // such lanes
  static constexpr int QD = 3;                     // task queue depth
  static constexpr int QB = G * D * 2;             // a streaming warp's q buffer (the G heads' rows)
  // everything but the rings: q buffers, shares, staging, queue, the other barriers, flag, alignment slack
  static constexpr int REST = NW * QB + NW * OV * SHL * 4 + NW * kHeadsTile * 8 + G * D * 4 + 64 +
                              QD * (int)sizeof(TaskEntry) + (3 * NW + 3 * QD + 1) * 8 + 8 + 16 + 1024;
  static constexpr int SLOT = RUN + SCL + 8;       // a ring slot with its scale record and its barrier
  static constexpr int NR_FIT = (kSmemPerSM / 2 - kSmemReservedPerCTA - REST) / (NW * SLOT);
  static constexpr int NR = RING < NR_FIT ? RING : (NR_FIT < 2 ? 2 : NR_FIT);
  static constexpr int OFF_QB = NW * NR * RUN;                       // [NW] q buffers
  static constexpr int OFF_SHARE = OFF_QB + NW * QB;                 // [NW][OV][SHL] fp32 o shares
  static constexpr int OFF_SML = OFF_SHARE + NW * OV * SHL * 4;      // [NW][8] float2 (m, l) shares
  static constexpr int OFF_STG = OFF_SML + NW * kHeadsTile * 8;      // combiner staging [G][D] fp32
  static constexpr int OFF_MML = OFF_STG + G * D * 4;                // staged split's (m, l): [8] float2
  static constexpr int OFF_Q = OFF_MML + 64;                         // [QD] TaskEntry
  static constexpr int OFF_BAR = OFF_Q + QD * (int)sizeof(TaskEntry);
  // barriers: ring [NW][NR], share_full [NW], share_empty [NW], queue full [QD], queue empty [QD], q [NW],
  // queue half-done [QD], the combiner's partial copy
  static constexpr int NBARS = NW * NR + 3 * NW + 3 * QD + 1;
  static constexpr int OFF_FLAG = OFF_BAR + (NBARS * 8 + 15) / 16 * 16;  // the CTA's abort flag
  static constexpr int OFF_SCL = OFF_FLAG + 16;                      // 8-bit: [NW][NR] scale records
  static constexpr int SMEM = OFF_SCL + NW * NR * SCL + 1024;        // + slack to align the rings to 1024 bytes
  static constexpr int FIT = kSmemPerSM / (SMEM + kSmemReservedPerCTA);
  // CTAs per SM (shared memory bound).  The 8-bit d = 256 kernel with 8 query heads per KV head holds too
  // much in registers for two CTAs (it spills); like its fp16 twin, which shared memory limits to one, it
  // runs one CTA per SM with the whole register file.
  static constexpr int MINB = (F8 && D == 256 && G > 6) ? 1 : (FIT < 3 ? FIT : 3);
  // Lean blocks two at a time (one softmax step and one rescale of O per pair): measured faster for the 8-bit
  // cache at head_dim 256 (the long-context decode, 7.3 against 8.9 ms a step), whose warps are bound by their
  // turnaround per block; slower on the 5-slot fp16 rings and the 256-row batch, so only there.
  static constexpr bool PAIRS = F8 && D == 256;
  static_assert(D % 64 == 0 && G >= 1 && G <= kHeadsTile, "shape");
  static_assert(RUN % 1024 == 0, "swizzled boxes need 1024-byte aligned slots");
  static_assert(KS % 2 == 0 && QB % 128 == 0, "k-steps in pairs; q buffers stay 16-byte aligned");
  static_assert(OFF_Q % 16 == 0 && OFF_BAR % 8 == 0 && OFF_STG % 16 == 0 && OFF_MML % 16 == 0, "alignment");
  static_assert(NR <= RING && SMEM <= NW * NR * SLOT + REST + 64, "shared-memory budget");
  static_assert(!F8 || (RUN % 1024 == 0 && BOXROWS <= 256), "8-bit runs are whole swizzle atoms, one box each");
  static_assert(OFF_SCL % 16 == 0, "scale records are bulk-copy destinations");
  static_assert(MINB >= 1, "shared memory");
};

struct DecodeParams {
  CUtensorMap kv_map;  // fp16: the pool as whole runs; 8-bit: as rows of codes (64-byte aligned: first member)
  const __half* q;
  const int32_t* block_tables;
  const int32_t* qsl;  // query_start_loc
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
  __half* cache_k;     // this layer's K pool [num_blocks][Hkv][16][D] (8-bit cache: E4M3 codes, one byte each)
  __half* cache_v;
  unsigned char* scales;  // 8-bit cache: this layer's scale records [num_blocks][Hkv][2 (K, V)][16]
  int64_t num_slots;
  // Launched right behind the prefill kernel of the same pass: its inputs were final once that kernel
  // passed its own dependency wait, so the decode runs in the prefill's tail (on SMs the prefill has left)
  // and waits for it only at its end, so that whatever follows sees both complete.
  int late_wait;
  int layer_row0_k;    // TMA row of (layer, K, block 0, head 0, slot 0) (8-bit: rows of 128 code bytes)
  int layer_row0_v;    // TMA row of (layer, V, block 0, head 0, slot 0)
  int max_blocks;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int split_blocks;
  int max_splits;
  int max_tasks;     // entries of the task list (loads stay below it; n_tasks of them are this pass's)
  float scale_log2;  // log2(e) / sqrt(head_dim)
};

// Byte offset of 16-byte chunk c (8 dims) of key row r inside a ring slot written by 64-value TMA boxes
// with the 128-byte swizzle: box c / 8, row r at 128 bytes, chunk slot (c % 8) XOR (r % 8).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The same for the 8-bit cache: byte offset of 16-byte chunk c (16 codes) of key row r inside a ring slot
// holding a run as rows of 128 bytes with the 128-byte swizzle (row R = byte / 128 at 128 R, its chunk
// slot (chunk % 8) XOR (R % 8)).
template <int D>
__device__ __forceinline__ uint32_t swz8(int r, int c) {
  if constexpr (D == 256) return swz(r, c);  // one 16-key x 128-byte box per half of the key (fp16's layout)
  const int x = r * D + 16 * c, R = x >> 7;
  return (uint32_t)(R * 128 + ((((x >> 4) & 7) ^ (R & 7)) << 4));
}

// Wait for phase `parity` of `bar`.  Gives up (false) as soon as another warp of the CTA has given up (the
// abort flag), or after more than 2^16 polls and ~1 s of %globaltimer time; then it records
// PKV_DEVERR_WAIT_TIMEOUT and raises the abort flag, so that every warp of the CTA unwinds.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* err) {
  if (dev::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = dev::globaltimer_ns();
  for (uint32_t polls = 1;; ++polls) {
    if (dev::mbar_try_wait(bar, parity)) return true;
    if ((polls & 31u) == 0) {
      if (*abort) return false;
      if (polls > dev::kWaitMinPolls && (int64_t)(dev::globaltimer_ns() - t0) > dev::kWaitLimitNs) {
        dev::set_error(err, PKV_DEVERR_WAIT_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Shared-memory map of one decode CTA.
template <int D, int G, int KV>
struct DecodeSmem {
  using T = DecodeTraits<D, G, KV>;
  unsigned char* ring;  // [NW][NR] slots of RUN bytes
  unsigned char* qbuf;  // [NW][QB]
  float* sh_o;          // [NW][OV][SHL]
  float2* sh_ml;        // [NW][8]
  float* stg;           // [G][D] fp32 (or [G][D] fp16 for a final output)
  float2* mml;          // [8] (m, l) of the staged split
  TaskEntry* queue;     // [QD]
  uint64_t* ring_bar;   // [NW][NR]
  uint64_t* share_full;
  uint64_t* share_empty;
  uint64_t* qfull;
  uint64_t* qempty;
  uint64_t* qbar;       // [NW] the q buffers' barriers
  uint64_t* qmid;       // [QD] every streaming warp has consumed half of its runs of the entry's task
  uint64_t* pbar;       // the combiner's copy of another split's partial into stg / mml
  volatile int* abort;
  unsigned char* scl;   // 8-bit: [NW][NR] scale records, 32 bytes each
  __device__ explicit DecodeSmem(unsigned char* s) {
    ring = s;
    qbuf = s + T::OFF_QB;
    sh_o = reinterpret_cast<float*>(s + T::OFF_SHARE);
    sh_ml = reinterpret_cast<float2*>(s + T::OFF_SML);
    stg = reinterpret_cast<float*>(s + T::OFF_STG);
    mml = reinterpret_cast<float2*>(s + T::OFF_MML);
    queue = reinterpret_cast<TaskEntry*>(s + T::OFF_Q);
    ring_bar = reinterpret_cast<uint64_t*>(s + T::OFF_BAR);
    share_full = ring_bar + T::NW * T::NR;
    share_empty = share_full + T::NW;
    qfull = share_empty + T::NW;
    qempty = qfull + T::QD;
    qbar = qempty + T::QD;
    qmid = qbar + T::NW;
    pbar = qmid + T::QD;
    abort = reinterpret_cast<volatile int*>(s + T::OFF_FLAG);
    scl = s + T::OFF_SCL;
  }
};

// A task as a streaming warp sees it.
struct TaskView {
  int t, g, s, row, ctx, nsplit, nst;
  int nbw;          // blocks of the split dealt to this warp: task-local blocks bw, bw + 4, ...
  int bw;
  int nlean;        // the warp's leading blocks that are full and hold no row of this pass (see Streamer)
  const int* ids;   // shared memory: the split's block ids
};

__device__ __forceinline__ int warp_blocks(int nb, int bw) { return nb > bw ? (nb - bw + 3) / 4 : 0; }

// ---------------------------------------------------------------------------------------------------
// Streaming warp: takes the CTA's tasks in queue order, streams the K and V runs of its share of each
// task's blocks through its own ring with TMA, and computes the group contraction on the tensor cores.
// At the end of a task it leaves its unnormalised (m, l, o) in its share slot for the combiner warp and
// goes straight on: the next task's first runs are already in its ring.  Measured on this access pattern
// (scattered 4 KB runs): one issuing thread per CTA cannot keep HBM busy, many independent issuers per
// SM can -- hence every streaming warp issues its own copies.
// ---------------------------------------------------------------------------------------------------
template <int D, int G, int KV>
struct Streamer {
  using T = DecodeTraits<D, G, KV>;
  const DecodeParams& p;
  const DecodeSmem<D, G, KV>& sm;
  unsigned char* ring;   // this warp's NR slots (1024-byte aligned)
  uint64_t* bars;        // this warp's NR barriers
  unsigned char* scl;    // 8-bit: this warp's NR scale records
  uint64_t pol;
  int warp, lane;
  int k = 0;             // the CTA's sequence number of the current task
  int issued = 0;        // runs issued into the ring so far
  int consumed = 0;      // runs taken out of the ring so far
  int icur = 0;          // 0: the issue cursor is in the current task, 1: in the next one
  int ir = 0;            // run index of the issue cursor: 2j K of block j, 2j + 1 V of block j
  bool has_nxt = false;
  TaskView cur, nxt;
  bool ok = true;
  // The task's q does not travel through the ring: it has its own buffer, filled with the next task's q
  // as soon as that task is published, so no task starts by waiting for it.
  unsigned char* qbuf;
  uint64_t* qbar;
  int q_seq = -1;        // task whose q was last issued into the buffer
  int q_used = 0;        // q loads taken out of the buffer so far
  bool q_busy = false;   // the buffer holds (or awaits) a q not yet taken
  bool cur_q_done = false;  // the current task's q is taken (or the task needs none): the buffer may refill
  int half_left = 0;     // runs of the current task still to consume before the half-way signal (0: sent)

  __device__ Streamer(const DecodeParams& p_, const DecodeSmem<D, G, KV>& sm_, int warp_, int lane_)
      : p(p_), sm(sm_), warp(warp_), lane(lane_) {
    ring = sm.ring + warp * T::NR * T::RUN;
    bars = sm.ring_bar + warp * T::NR;
    scl = sm.scl + warp * T::NR * T::SCL;
    qbuf = sm.qbuf + warp * T::QB;
    qbar = sm.qbar + warp;
    pol = dev::l2_policy_evict_first();
  }

  // Task kk of the queue (waits until the scheduler warp has published it).
  __device__ void take(int kk, TaskView& v) {
    const bool got = cta_wait(&sm.qfull[kk % T::QD], (kk / T::QD) & 1, sm.abort, p.err);
    ok = __all_sync(0xffffffffu, got) && ok;
    if (!ok) {
      v.t = -1;
      v.nbw = 0;
      return;
    }
    const TaskEntry* e = &sm.queue[kk % T::QD];
    const int4 rec = e->rec;
    v.t = rec.x;
    v.g = rec.y & 0xFF;
    v.s = rec.y >> 8;
    v.row = rec.z;
    v.ctx = rec.w;
    v.nst = e->nst;
    const int nblk = (v.ctx + kBS - 1) / kBS;
    v.nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
    v.bw = (warp - e->rot) & 3;
    v.nbw = v.t >= 0 ? warp_blocks(e->nb, v.bw) : 0;
    v.ids = e->ids;
    // A block is on the lean path when all its 16 keys are inside the context and none is this pass's (with
    // the append fused, the pass's rows come from the inputs): blocks below position `from`.  The same rule
    // holds without the fused append, so both calls pair the same blocks and give the same bits.  Blocks rise
    // with j, so the lean ones are the warp's first nlean.
    const int from = min(v.nst, v.ctx);
    const int first = v.s * p.split_blocks + v.bw;  // absolute index of the warp's block 0
    const int nfull = from / kBS - first;             // blocks first, first + NW, ... below from / 16
    v.nlean = (!T::PAIRS || nfull <= 0) ? 0 : min(v.nbw, (nfull + T::NW - 1) / T::NW);
  }
  static __device__ __forceinline__ int runs(const TaskView& v) { return v.t >= 0 ? 2 * v.nbw : 0; }
  __device__ __forceinline__ int block_pos(const TaskView& v, int j) const {
    return (v.s * p.split_blocks + v.bw + T::NW * j) * kBS;
  }
  // Run r of the warp's stream within a task: the lean blocks go in pairs, K of both then V of both; the rest
  // (an odd lean block, then the blocks holding the context's end or this pass's rows) one by one, K then V.
  static __device__ __forceinline__ void run_of(const TaskView& v, int r, int& j, int& isv) {
    const int pr = 4 * (v.nlean >> 1);
    if (r < pr) {
      j = 2 * (r >> 2) + (r & 1);
      isv = (r >> 1) & 1;
    } else {
      j = 2 * (v.nlean >> 1) + ((r - pr) >> 1);
      isv = (r - pr) & 1;
    }
  }


  __device__ __forceinline__ void issue_slot(const TaskView& v, int r, int slot) {
    unsigned char* dst = ring + slot * T::RUN;
    if (lane != 0) return;
    int j, isv;
    run_of(v, r, j, isv);
    r = isv;  // below, r & 1 tells V from K
    const int id = v.ids[v.bw + T::NW * j];
    if constexpr (T::F8) {
      // the codes as one box; a K run brings the block's 32-byte scale record (K and V scales) along
      dev::mbar_arrive_expect_tx(&bars[slot], T::RUN + ((r & 1) ? 0 : T::SCL));
      if constexpr (D == 256) {  // two boxes: the keys' first and second 128 code bytes (rows are tokens)
        const int tok = ((r & 1) ? p.layer_row0_v : p.layer_row0_k) + (id * p.num_kv_heads + v.g) * kBS;
        dev::tma_load_3d(dst, &p.kv_map, 0, 0, tok, &bars[slot], pol);
        dev::tma_load_3d(dst + 2048, &p.kv_map, 0, 1, tok, &bars[slot], pol);
      } else {
        const int row = ((r & 1) ? p.layer_row0_v : p.layer_row0_k) + (id * p.num_kv_heads + v.g) * T::BOXROWS;
        dev::tma_load_2d(dst, &p.kv_map, 0, row, &bars[slot], pol);
      }
      if (!(r & 1))
        dev::bulk_g2s(scl + slot * T::SCL, p.scales + ((size_t)id * p.num_kv_heads + v.g) * T::SCL, T::SCL,
                      &bars[slot], pol);
    } else {
      const int row = ((r & 1) ? p.layer_row0_v : p.layer_row0_k) + (id * p.num_kv_heads + v.g) * kBS;
      dev::mbar_arrive_expect_tx(&bars[slot], T::RUN);
      dev::tma_load_3d(dst, &p.kv_map, 0, row, 0, &bars[slot], pol);  // the run's D / 64 sub-tiles, one copy
    }
  }
  // Task kk's q into the warp's q buffer (which must be free).
  __device__ __forceinline__ void issue_q(const TaskView& v, int kk) {
    if (lane == 0) {
      dev::fence_proxy_async_smem();  // the warp's reads of the previous q precede this copy
      dev::mbar_arrive_expect_tx(qbar, G * D * 2);
      dev::bulk_g2s(qbuf, p.q + ((size_t)v.t * p.num_q_heads + (size_t)v.g * G) * D, G * D * 2, qbar, pol);
    }
    q_seq = kk;
    q_busy = true;
  }
  // Whether the scheduler has published task kk (never waits).
  __device__ __forceinline__ bool published(int kk) const {
    return __all_sync(0xffffffffu, dev::mbar_test_wait(&sm.qfull[kk % T::QD], (kk / T::QD) & 1));
  }
  // The next task's q as soon as its entry is published; never waits for the entry.
  __device__ __forceinline__ void prefetch_q() {
    if (!cur_q_done || q_busy || q_seq == k + 1 || cur.t < 0 || !ok) return;
    if (!has_nxt) {
      if (!published(k + 1)) return;
      take(k + 1, nxt);
      has_nxt = true;
    }
    if (ok && nxt.t >= 0 && nxt.nbw > 0) issue_q(nxt, k + 1);
  }
  // The current task's q as MMA B fragments (Q^T: k = dims, n = heads).  The buffer holds the G heads' rows;
  // the columns of heads G..7 repeat head 0 (they feed score and output columns that are never written out).
  // Then the buffer is free for the next task's q.
  __device__ __forceinline__ void load_q(uint32_t (&qb)[T::KS][2]) {
    if (q_seq != k) issue_q(cur, k);  // not prefetched
    const bool got = cta_wait(qbar, q_used & 1, sm.abort, p.err);
    ok = __all_sync(0xffffffffu, got) && ok;
    if (!ok) return;
    const uint32_t qs = dev::smem_addr(qbuf);
    if constexpr (T::F8) {
      // The 8-bit K fragments hold dims 4t .. 4t + 3 of a 16-dim step as MMA k indices 2t, 2t + 1, 2t + 8,
      // 2t + 9 (the order ldmatrix delivers bytes in); q takes the same order, which leaves every dot
      // product as it is.
#pragma unroll
      for (int ks = 0; ks < T::KS; ++ks)
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                     : "=r"(qb[ks][0]), "=r"(qb[ks][1])
                     : "r"(qs + ((lane >> 2) < G ? lane >> 2 : 0) * (D * 2) + (16 * ks + 4 * (lane & 3)) * 2));
    } else {
#pragma unroll
      for (int k2 = 0; k2 < T::KS / 2; ++k2) {
        uint32_t r4[4];
        dev::ldsm_x4(qs + ((lane & 7) < G ? lane & 7 : 0) * (D * 2) + (4 * k2 + (lane >> 3)) * 16, r4);
        qb[2 * k2][0] = r4[0];
        qb[2 * k2][1] = r4[1];
        qb[2 * k2 + 1][0] = r4[2];
        qb[2 * k2 + 1][1] = r4[3];
      }
    }
    ++q_used;
    q_busy = false;
    cur_q_done = true;
    __syncwarp();  // every lane's reads precede the next copy into the buffer
    prefetch_q();
  }
  __device__ __forceinline__ void issue_run(const TaskView& v, int r) {
    issue_slot(v, r, issued % T::NR);
    ++issued;
  }
  // Issue the next run of the stream (current task, then the next one), if there is one.  Crossing into
  // the next task never waits for it to be published: the task in hand comes first, and a later release
  // tries again.
  __device__ __forceinline__ bool issue_next() {
    if (icur == 0) {
      if (ir < runs(cur)) {
        issue_run(cur, ir++);
        return true;
      }
      icur = 1;
      ir = 0;
    }
    if (!has_nxt) {
      if (cur.t < 0 || !published(k + 1)) return false;
      take(k + 1, nxt);
      has_nxt = true;
      prefetch_q();
    }
    if (ok && ir < runs(nxt)) {
      issue_run(nxt, ir++);
      return true;
    }
    return false;
  }
  // Top the ring up.  It runs dry when the warp had no blocks in the task just finished, since only
  // consuming a run issues the next one.
  __device__ __forceinline__ void fill() {
    while (ok && issued - consumed < T::NR && issue_next()) {
    }
  }
  // 8-bit: the scale record of the oldest run in the ring (valid once wait_run() has returned for a K run).
  __device__ __forceinline__ unsigned char* run_scales() const { return scl + (consumed % T::NR) * T::SCL; }
  // Wait for the oldest run in the ring; returns its slot's shared-memory address.
  __device__ __forceinline__ uint32_t wait_run() {
    const int slot = consumed % T::NR;
    const bool got = cta_wait(&bars[slot], (consumed / T::NR) & 1, sm.abort, p.err);
    ok = __all_sync(0xffffffffu, got) && ok;
    return dev::smem_addr(ring + slot * T::RUN);
  }
  // Half-way through the current task (half of this warp's runs consumed; at once for a warp with none): the
  // scheduler warp claims the CTA's next task once every streaming warp is there (see Scheduler).
  __device__ __forceinline__ void task_start() {
    half_left = runs(cur) / 2;
    if (half_left == 0 && lane == 0) dev::mbar_arrive(&sm.qmid[k % T::QD]);
  }
  // The warp is done with the oldest run: recycle its slot for the next run of the stream.
  __device__ __forceinline__ void release_run() {
    __syncwarp();
    ++consumed;
    if (ok) issue_next();
    if (half_left > 0 && --half_left == 0 && lane == 0) dev::mbar_arrive(&sm.qmid[k % T::QD]);
  }
  // Before the dependency wait: the first task, and its first K/V runs wherever nothing that the previous
  // kernel writes can be in them (positions the appended tokens never reach, or rows that are replaced
  // from the appended inputs anyway).  q comes after the wait.
  __device__ void prologue() {
    take(0, cur);
    if (!ok) return;
    cur_q_done = cur.nbw == 0;
    while (issued < T::NR && issued < runs(cur)) {
      int jb, isv;
      run_of(cur, issued, jb, isv);
      const int bpos = block_pos(cur, jb);
      if (!(p.k_in != nullptr || p.late_wait || bpos + kBS <= cur.nst)) break;
      issue_slot(cur, issued, issued);
      ++issued;
    }
    ir = issued;
  }
  __device__ void after_wait() {
    if (ok && runs(cur) > 0) issue_q(cur, 0);
  }
  // The copies issued but not consumed must land before the CTA leaves (each wait bounded).
  __device__ void drain() {
    for (; consumed < issued; ++consumed) dev::mbar_wait(&bars[consumed % T::NR], (consumed / T::NR) & 1);
    if (q_busy) dev::mbar_wait(qbar, q_used & 1);
  }
  __device__ __forceinline__ void advance() {
    if (!has_nxt) take(k + 1, nxt);
    if (icur == 0) ir = 0;
    cur = nxt;
    has_nxt = false;
    icur = 0;
    ++k;
    cur_q_done = cur.nbw == 0;  // a task with no blocks for this warp needs no q
  }
};

template <int D, int G, int KV>
__device__ __forceinline__ void stream_loop(const DecodeParams& p, const DecodeSmem<D, G, KV>& sm, Streamer<D, G, KV>& w) {
  using T = DecodeTraits<D, G, KV>;
  const int lane = w.lane, warp = w.warp;
  const int qh = lane >> 2;        // head whose q this lane feeds to the MMA (B operand column); key row too
  const int h0 = (lane & 3) << 1;  // heads of this lane's score / output columns: h0, h0 + 1
  int shares = 0;                  // shares this warp has handed to the combiner warp
  float* my_o = sm.sh_o + warp * T::OV * T::SHL;
  float2* my_ml = sm.sh_ml + warp * kHeadsTile;
  // This lane's ldmatrix row offsets inside a ring slot, hoisted out of the block loop.  fp16: chunk c of a
  // 64-value box sits at swz(r, c); the chunks 2x + hi of the four k-steps of one box differ only in x, and
  // the next box adds 2048.  8-bit: one offset per 32 dims of codes.
  uint32_t koff[4], voff[4];
  uint32_t k8off[T::F8 ? D / 32 : 1], v8off[T::F8 ? D / 32 : 1];
  {
    const int kr = (lane & 7) + ((lane >> 3) & 1) * 8, vmat = lane >> 3, vr = (lane & 7) + ((vmat >> 1) << 3);
#pragma unroll
    for (int x4 = 0; x4 < 4; ++x4) {
      koff[x4] = swz(kr, 2 * x4 + (lane >> 4));
      voff[x4] = swz(vr, 2 * x4 + (vmat & 1));
    }
#pragma unroll
    for (int i = 0; i < (T::F8 ? D / 32 : 1); ++i) {
      k8off[i] = T::F8 ? swz8<D>(kr, 2 * i + (lane >> 4)) : 0u;
      v8off[i] = T::F8 ? swz8<D>(vr, 2 * i + (vmat & 1)) : 0u;
    }
  }
  while (w.ok && w.cur.t >= 0) {
    const TaskView d = w.cur;
    w.task_start();
    w.fill();
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[T::MT][4];
#pragma unroll
    for (int mt = 0; mt < T::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    if (d.nbw > 0 && w.ok) {
      // ---- q as the MMA B operand (Q^T: k = dims, n = heads) ----
      uint32_t qb[T::KS][2];
      w.load_q(qb);

      // ---- the lean blocks, two at a time: both blocks' scores, one softmax step for the pair (one max
      // reduction, one rescale of O), then both blocks' products.  Their runs sit in the ring in that order. ----
      int j = 0;
      if constexpr (T::PAIRS) {
        for (; j + 1 < d.nlean && w.ok; j += 2) {
          float x[2][4];            // scaled scores: [block][key qh head h0, key qh h0 + 1, key qh + 8 h0, .. h0 + 1]
          uint32_t evb[2][2];       // 8-bit: value scale bytes of keys qh, qh + 8
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kb = w.wait_run();
            if (!w.ok) break;
            float ks0 = p.scale_log2, ks1 = p.scale_log2;
            if constexpr (T::F8) {
              const unsigned char* rec = w.run_scales();
              ks0 *= dev::scale_of_byte(rec[qh]);
              ks1 *= dev::scale_of_byte(rec[qh + 8]);
              evb[u][0] = rec[16 + qh];
              evb[u][1] = rec[24 + qh];
#pragma unroll
              for (int i = 0; i < D / 32; ++i) {
                uint32_t r[4];
                dev::ldsm_x4(kb + k8off[i], r);
                uint32_t a0[4], a1[4];
                dev::e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
                dev::e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
                dev::e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
                dev::e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
                dev::mma_16816(sc, a0, qb[2 * i][0], qb[2 * i][1]);
                dev::mma_16816(sd, a1, qb[2 * i + 1][0], qb[2 * i + 1][1]);
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < T::KS; ++ks) {
                uint32_t a[4];
                dev::ldsm_x4(kb + koff[ks & 3] + (ks >> 2) * 2048, a);
                dev::mma_16816((ks & 1) ? sd : sc, a, qb[ks][0], qb[ks][1]);
              }
            }
            x[u][0] = (sc[0] + sd[0]) * ks0;
            x[u][1] = (sc[1] + sd[1]) * ks0;
            x[u][2] = (sc[2] + sd[2]) * ks1;
            x[u][3] = (sc[3] + sd[3]) * ks1;
            w.release_run();
          }
          if (!w.ok) break;
          // ---- one online-softmax step for the pair (log2 domain) ----
          float b0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
          float b1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
          for (int m = 4; m < 32; m <<= 1) {
            b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, m));
            b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, m));
          }
          const float n0 = fmaxf(m0, b0), n1 = fmaxf(m1, b1);
          const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
          m0 = n0;
          m1 = n1;
          float pw[2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            pw[u][0] = exp2f(x[u][0] - n0);
            pw[u][1] = exp2f(x[u][1] - n1);
            pw[u][2] = exp2f(x[u][2] - n0);
            pw[u][3] = exp2f(x[u][3] - n1);
          }
          l0 = l0 * a0 + ((pw[0][0] + pw[0][2]) + (pw[1][0] + pw[1][2]));
          l1 = l1 * a1 + ((pw[0][1] + pw[0][3]) + (pw[1][1] + pw[1][3]));
#pragma unroll
          for (int mt = 0; mt < T::MT; ++mt) {
            o[mt][0] *= a0;
            o[mt][1] *= a1;
            o[mt][2] *= a0;
            o[mt][3] *= a1;
          }
          // ---- O^T[d x 8 heads] += V^T P^T for both blocks ----
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float s0 = 1.f, s1 = 1.f;
            if constexpr (T::F8) {  // the value scale of each key rides on its weight (an exact power of two)
              s0 = dev::scale_of_byte(evb[u][0]);
              s1 = dev::scale_of_byte(evb[u][1]);
            }
            const __half2 pk0 = __floats2half2_rn(pw[u][0] * s0, pw[u][1] * s0);
            const __half2 pk1 = __floats2half2_rn(pw[u][2] * s1, pw[u][3] * s1);
            const uint32_t pb0 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk0));
            const uint32_t pb1 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk1));
            const uint32_t vb = w.wait_run();
            if (!w.ok) break;
            if constexpr (T::F8) {
#pragma unroll
              for (int i = 0; i < D / 32; ++i) {
                uint32_t r[4];
                dev::ldsm_x4_t(vb + v8off[i], r);
                uint32_t ae[4], ao[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) dev::e4m3x4_to_f16x2x2(__byte_perm(r[q], 0, 0x3120), ae[q], ao[q]);
                dev::mma_16816(o[2 * i], ae, pb0, pb1);
                dev::mma_16816(o[2 * i + 1], ao, pb0, pb1);
              }
            } else {
#pragma unroll
              for (int mt = 0; mt < T::MT; ++mt) {
                uint32_t a[4];
                dev::ldsm_x4_t(vb + voff[mt & 3] + (mt >> 2) * 2048, a);
                dev::mma_16816(o[mt], a, pb0, pb1);
              }
            }
            w.release_run();
          }
          w.prefetch_q();  // the next task's q, once the scheduler has published it
        }
      }
      // ---- the rest one by one: an odd lean block, then the blocks holding the context's end or rows of
      // this pass (masking, the fused append's rows from the inputs, the token's own write to the cache) ----
      for (; j < d.nbw && w.ok; ++j) {
        const int bpos = w.block_pos(d, j);  // the block's first position
        const int ntok = min(kBS, d.ctx - bpos);
        // fused append: positions ov0 .. bpos + ntok - 1 of the block are this pass's tokens; their rows
        // come from the inputs (the cache may not hold them yet), and the block holding the token's own
        // position writes it into the cache
        const int ov0 = max(bpos, d.nst), nov = p.k_in != nullptr ? bpos + ntok - ov0 : 0;
        const bool own = nov > 0 && d.ctx - 1 < bpos + kBS;  // the block holds the token's own position
        // Up to 32 16-byte chunks of new rows (one decode token's row at d <= 256): every lane loads its
        // chunk now, while the block's K and V tiles are in flight, so no dependent global load sits between
        // a tile's arrival and its use; more rows (a short chunk) are read after the tile lands.
        const bool pf = nov > 0 && nov * (D / 8) <= 32;
        const int prr = ov0 - bpos + lane / (D / 8), pcc = lane % (D / 8);  // this lane's row and chunk
        uint4 pk = make_uint4(0, 0, 0, 0), pv = pk;
        if (pf && lane < nov * (D / 8)) {
          const size_t src = ((size_t)(d.t - (d.ctx - 1 - (bpos + prr))) * p.num_kv_heads + d.g) * D;
          pk = __ldcg(reinterpret_cast<const uint4*>(p.k_in + src) + pcc);
          pv = __ldcg(reinterpret_cast<const uint4*>(p.v_in + src) + pcc);
        }
        const int64_t slot = own ? __ldcg(p.slots + d.t) : -1;
        auto override_rows = [&](uint32_t base, const __half* src, const uint4& pre) {
          if (pf) {
            if (lane < nov * (D / 8))
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + swz(prr, pcc)), "r"(pre.x),
                           "r"(pre.y), "r"(pre.z), "r"(pre.w)
                           : "memory");
            __syncwarp();
            return;
          }
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
        // 8-bit cache: this pass's rows of the block quantized from the inputs, exactly as the append would
        // store them -- the codes into the slot at `base` (if codes), the scale bytes into `rec` at rec_off
        // (if rec).  A row's D / 8 lanes are consecutive and lane-aligned, so its largest magnitude is one
        // group reduction; every lane of the warp takes part.
        auto quant_rows = [&](uint32_t base, const __half* src, bool codes, unsigned char* rec, int rec_off) {
          constexpr int CPR = D / 8;
          for (int it = 0; it * 32 < nov * CPR; ++it) {
            const int idx = it * 32 + lane;
            const bool in = idx < nov * CPR;
            const int rr = ov0 - bpos + idx / CPR, cc = idx % CPR;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (in) {
              const int tk = d.t - (d.ctx - 1 - (bpos + rr));
              raw = __ldcg(reinterpret_cast<const uint4*>(src + ((size_t)tk * p.num_kv_heads + d.g) * D) + cc);
            }
            const int sb = dev::e4m3_scale_byte(dev::row_amax_bits<CPR>(dev::f16x8_amax_bits(raw)));
            if (in && codes) {
              const uint2 c = dev::e4m3_encode8(raw, sb);
              asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(base + swz8<D>(rr, cc >> 1) + (cc & 1) * 8),
                           "r"(c.x), "r"(c.y)
                           : "memory");
            }
            if (in && rec != nullptr && cc == 0) rec[rec_off + rr] = (unsigned char)sb;
          }
          __syncwarp();
        };
        uint2 ck = make_uint2(0, 0), cv = ck;  // 8-bit, prefetched rows: this lane's codes and its row's scales
        int sbk = 127, sbv = 127;
        // ---- S^T[16 keys x 8 heads] = K Q^T on the tensor cores ----
        // Two accumulators (even and odd k-steps) halve the chain of dependent MMAs; summed at the end.
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
        float ks0 = p.scale_log2, ks1 = p.scale_log2;  // score scale of keys qh and qh + 8
        uint32_t ev0 = 127, ev1 = 127;                 // 8-bit: scale bytes of their values
        {
          const uint32_t ks_base = w.wait_run();
          if (!w.ok) break;
          const int kr = (lane & 7) + ((lane >> 3) & 1) * 8;  // key row this lane addresses for ldmatrix
          if constexpr (T::F8) {
            unsigned char* rec = w.run_scales();  // the block's K and V scales arrived with the K run
            if (nov > 0) {
              if (pf) {
                constexpr int CPR = D / 8;
                sbk = dev::e4m3_scale_byte(dev::row_amax_bits<CPR>(dev::f16x8_amax_bits(pk)));
                sbv = dev::e4m3_scale_byte(dev::row_amax_bits<CPR>(dev::f16x8_amax_bits(pv)));
                if (lane < nov * CPR) {
                  ck = dev::e4m3_encode8(pk, sbk);
                  cv = dev::e4m3_encode8(pv, sbv);
                  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(ks_base + swz8<D>(prr, pcc >> 1) + (pcc & 1) * 8),
                               "r"(ck.x), "r"(ck.y)
                               : "memory");
                  if (pcc == 0) {
                    rec[prr] = (unsigned char)sbk;
                    rec[16 + prr] = (unsigned char)sbv;
                  }
                }
                __syncwarp();
              } else {
                quant_rows(ks_base, p.k_in, true, rec, 0);
                quant_rows(0, p.v_in, false, rec, 16);
              }
            }
            ks0 = p.scale_log2 * dev::scale_of_byte(rec[qh]);
            ks1 = p.scale_log2 * dev::scale_of_byte(rec[qh + 8]);
            ev0 = rec[16 + qh];
            ev1 = rec[24 + qh];
            // 16 keys x 32 dims of codes per ldmatrix; the fragments keep the byte order (see load_q)
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
              uint32_t r[4];
              dev::ldsm_x4(ks_base + swz8<D>(kr, 2 * i + (lane >> 4)), r);
              uint32_t a0[4], a1[4];  // {key g lo, key g + 8 lo, key g hi, key g + 8 hi}
              dev::e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
              dev::e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
              dev::e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
              dev::e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
              dev::mma_16816(sc, a0, qb[2 * i][0], qb[2 * i][1]);
              dev::mma_16816(sd, a1, qb[2 * i + 1][0], qb[2 * i + 1][1]);
            }
          } else {
            if (nov > 0) override_rows(ks_base, p.k_in, pk);
#pragma unroll
            for (int ks = 0; ks < T::KS; ++ks) {
              uint32_t a[4];
              dev::ldsm_x4(ks_base + swz(kr, 2 * ks + (lane >> 4)), a);
              dev::mma_16816((ks & 1) ? sd : sc, a, qb[ks][0], qb[ks][1]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[i] += sd[i];
          if (nov > 0) dev::fence_proxy_async_smem();  // the override precedes the slot's next TMA write
          w.release_run();
        }
        // ---- online softmax (log2 domain); the lane holds keys qh, qh + 8 for heads h0, h0 + 1 ----
        const bool v0 = qh < ntok, v1 = qh + 8 < ntok;
        const float s0 = v0 ? sc[0] * ks0 : -INFINITY;  // key qh,     head h0
        const float s1 = v0 ? sc[1] * ks0 : -INFINITY;  // key qh,     head h0 + 1
        const float s2 = v1 ? sc[2] * ks1 : -INFINITY;  // key qh + 8, head h0
        const float s3 = v1 ? sc[3] * ks1 : -INFINITY;  // key qh + 8, head h0 + 1
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
        // P^T as the B operand (k = keys, n = heads): transpose the [keys x heads] 8x8 fragments.  8-bit: the
        // value scale of each key rides on its weight (an exact power of two), so V^T holds the bare codes.
        float sv0 = 1.f, sv1 = 1.f;
        if constexpr (T::F8) {
          sv0 = v0 ? dev::scale_of_byte(ev0) : 0.f;
          sv1 = v1 ? dev::scale_of_byte(ev1) : 0.f;
        }
        const __half2 pk0 = __floats2half2_rn(p0 * sv0, p1 * sv0), pk1 = __floats2half2_rn(p2 * sv1, p3 * sv1);
        const uint32_t pb0 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk0));
        const uint32_t pb1 = dev::movmatrix_t(*reinterpret_cast<const uint32_t*>(&pk1));
        // ---- O^T[d x 8 heads] += V^T P^T on the tensor cores ----
        {
          const uint32_t vs_base = w.wait_run();
          if (!w.ok) break;
          const int mat = lane >> 3;                      // ldmatrix matrix this lane addresses
          const int vr = (lane & 7) + ((mat >> 1) << 3);  // its key row
          if constexpr (T::F8) {
            if (ntok < kBS) {  // rows past the context may hold anything (NaN codes): zero them
              for (int idx = lane; idx < (kBS - ntok) * (D / 16); idx += 32) {
                const int r = ntok + idx / (D / 16), c = idx % (D / 16);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vs_base + swz8<D>(r, c)), "r"(0) : "memory");
              }
              __syncwarp();
            }
            if (nov > 0) {
              if (pf) {
                if (lane < nov * (D / 8))
                  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(vs_base + swz8<D>(prr, pcc >> 1) + (pcc & 1) * 8),
                               "r"(cv.x), "r"(cv.y)
                               : "memory");
                __syncwarp();
              } else {
                quant_rows(vs_base, p.v_in, true, nullptr, 0);
              }
            }
            // 16 keys x 32 dims per transposing ldmatrix: a lane's word holds keys 2t, 2t + 1 at dims 2g, 2g + 1;
            // regrouped by dim, the even dims feed one MMA (o[2i]) and the odd dims another (o[2i + 1])
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
              uint32_t r[4];
              dev::ldsm_x4_t(vs_base + swz8<D>(vr, 2 * i + (mat & 1)), r);
              uint32_t ae[4], ao[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) dev::e4m3x4_to_f16x2x2(__byte_perm(r[j], 0, 0x3120), ae[j], ao[j]);
              dev::mma_16816(o[2 * i], ae, pb0, pb1);
              dev::mma_16816(o[2 * i + 1], ao, pb0, pb1);
            }
          } else {
            if (ntok < kBS) {  // rows past the context may hold anything: zero them so 0 * garbage cannot poison O
              for (int idx = lane; idx < (kBS - ntok) * (D / 8); idx += 32) {
                const int r = ntok + idx / (D / 8), c = idx % (D / 8);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vs_base + swz(r, c)), "r"(0) : "memory");
              }
              __syncwarp();
            }
            if (nov > 0) override_rows(vs_base, p.v_in, pv);
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
              uint32_t a[4];
              dev::ldsm_x4_t(vs_base + swz(vr, 2 * mt + (mat & 1)), a);
              dev::mma_16816(o[mt], a, pb0, pb1);
            }
          }
          if (ntok < kBS || nov > 0) dev::fence_proxy_async_smem();  // generic writes precede the next TMA write
          w.release_run();
        }
        w.prefetch_q();  // the next task's q, once the scheduler has published it
        // ---- fused append: the token's own key and value into the cache ----
        if (own && slot != -1) {
          if (slot < 0 || slot >= p.num_slots) {
            if (lane == 0) dev::set_error(p.err, PKV_DEVERR_SLOT_RANGE);
          } else if constexpr (T::F8) {
            constexpr int CPR = D / 8;
            const size_t row = ((size_t)(slot >> 4) * p.num_kv_heads + d.g) * kBS + (slot & 15);
            uint2* dk = reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(p.cache_k) + row * D);
            uint2* dv = reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(p.cache_v) + row * D);
            unsigned char* rec = p.scales + ((size_t)(slot >> 4) * p.num_kv_heads + d.g) * T::SCL;
            if (pf) {  // the lanes holding the last new row hold the token's own codes
              if (lane < nov * CPR && prr == d.ctx - 1 - bpos) {
                dk[pcc] = ck;
                dv[pcc] = cv;
                if (pcc == 0) {
                  rec[slot & 15] = (unsigned char)sbk;
                  rec[16 + (slot & 15)] = (unsigned char)sbv;
                }
              }
            } else {
              const bool in = lane < CPR;
              const size_t src = ((size_t)d.t * p.num_kv_heads + d.g) * D;
              const uint4 zero = make_uint4(0, 0, 0, 0);
              const uint4 rk = in ? __ldcg(reinterpret_cast<const uint4*>(p.k_in + src) + lane) : zero;
              const uint4 rv = in ? __ldcg(reinterpret_cast<const uint4*>(p.v_in + src) + lane) : zero;
              const int bk = dev::e4m3_scale_byte(dev::row_amax_bits<CPR>(dev::f16x8_amax_bits(rk)));
              const int bv = dev::e4m3_scale_byte(dev::row_amax_bits<CPR>(dev::f16x8_amax_bits(rv)));
              if (in) {
                dk[lane] = dev::e4m3_encode8(rk, bk);
                dv[lane] = dev::e4m3_encode8(rv, bv);
                if (lane == 0) {
                  rec[slot & 15] = (unsigned char)bk;
                  rec[16 + (slot & 15)] = (unsigned char)bv;
                }
              }
            }
          } else {
            const size_t dst = (((size_t)(slot >> 4) * p.num_kv_heads + d.g) * kBS + (slot & 15)) * D;
            if (pf) {  // the lanes holding the last new row hold the token's own row
              if (lane < nov * (D / 8) && prr == d.ctx - 1 - bpos) {
                reinterpret_cast<uint4*>(p.cache_k + dst)[pcc] = pk;
                reinterpret_cast<uint4*>(p.cache_v + dst)[pcc] = pv;
              }
            } else {
              const size_t src = ((size_t)d.t * p.num_kv_heads + d.g) * D;
              for (int cc = lane; cc < D / 8; cc += 32) {
                reinterpret_cast<uint4*>(p.cache_k + dst)[cc] = __ldcg(reinterpret_cast<const uint4*>(p.k_in + src) + cc);
                reinterpret_cast<uint4*>(p.cache_v + dst)[cc] = __ldcg(reinterpret_cast<const uint4*>(p.v_in + src) + cc);
              }
            }
          }
        }
      }
    }
    if (!w.ok) break;

    // ---- hand this warp's share of the split to the combiner warp ----
    if (d.nbw > 0) {
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, m);
        l1 += __shfl_xor_sync(0xffffffffu, l1, m);
      }
      if (shares > 0) {  // the slot is free once the combiner warp has taken the previous share
        const bool got = cta_wait(&sm.share_empty[warp], (shares - 1) & 1, sm.abort, p.err);
        if (!__all_sync(0xffffffffu, got)) {
          w.ok = false;
          break;
        }
      }
      const int hg = lane & 3;
      if (hg < T::LG) {
        const int ci = (lane >> 2) * T::LG + hg;
#pragma unroll
        for (int r = 0; r < T::OV; ++r) my_o[r * T::SHL + ci] = o[r >> 2][r & 3];
        if (lane < T::LG) {
          my_ml[h0] = make_float2(m0, l0);
          my_ml[h0 + 1] = make_float2(m1, l1);
        }
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&sm.share_full[warp]);
      ++shares;
    }
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(&sm.qempty[w.k % T::QD]);  // done with the task's queue entry
    w.advance();
  }
}

// Output element held by register r of `lane` in the O^T fragment layout: its dim and its head.  fp16
// cache: m-tile mt = r / 4 covers dims 16 mt .. 16 mt + 15, the lane's rows at g = lane / 4 and g + 8.
// 8-bit cache: m-tiles 2i and 2i + 1 cover dims 32 i .. 32 i + 31, the even dims in the first and the odd
// ones in the second; the lane's rows are dims 32 i + 2g (+ 16) and the next odd one.
template <int KV>
__device__ __forceinline__ void frag_coord(int lane, int r, int& dim, int& head) {
  const int mt = r >> 2, g = lane >> 2;
  if constexpr (KV == kKvE4M3) dim = 32 * (mt >> 1) + ((r & 2) ? 16 : 0) + 2 * g + (mt & 1);
  else dim = 16 * mt + g + ((r & 2) ? 8 : 0);
  head = ((lane & 3) << 1) + (r & 1);
}

// ---------------------------------------------------------------------------------------------------
// Scheduler warp: publishes the CTA's tasks into the queue.  The first is static and published before the
// dependency wait: task blockIdx.x, one of the largest (the list is ordered largest first).  Every later task
// is claimed from a global counter -- the second at once, each next one once the streaming warps have
// finished the task two entries back -- so the tasks go out largest first to whichever CTA is ready: a
// greedy longest-first schedule, which ends the launch more evenly than pairing two static tasks per CTA
// (2 % on the 256-row decode).  A CTA holds one task it has not started.
// ---------------------------------------------------------------------------------------------------
template <int D, int G, int KV>
struct Scheduler {
  using T = DecodeTraits<D, G, KV>;
  const DecodeParams& p;
  const DecodeSmem<D, G, KV>& sm;
  int lane;
  int n_tasks = 0;
  int filled = 0;        // queue entries published so far (task sequence numbers 0 .. filled-1)
  bool ended = false;    // an end-of-work entry has been published
  int last_nb = 1 << 30; // blocks of the task published last
  int last_idx = 0;      // list index of the task published last

  __device__ Scheduler(const DecodeParams& p_, const DecodeSmem<D, G, KV>& sm_, int lane_) : p(p_), sm(sm_), lane(lane_) {}

  // Publish task indices idx[0 .. n-1] as the next n queue entries, the loads of all of them in flight
  // together; an index past the task list ends the work (nothing after it is published).
  template <int N>
  __device__ void publish(const int (&idx)[N]) {
    int4 rec[N];
#pragma unroll
    for (int j = 0; j < N; ++j)  // past the list: the end of the work, with nothing to load
      rec[j] = idx[j] < n_tasks && idx[j] < p.max_tasks ? __ldcg(p.tasks + idx[j]) : make_int4(-1, 0, 0, 0);
    int id[N], q0[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
      id[j] = 0;
      q0[j] = 0;
      if (rec[j].x >= 0) {
        const int s = rec[j].y >> 8, nblk = (rec[j].w + kBS - 1) / kBS;
        if (lane < min(p.split_blocks, nblk - s * p.split_blocks))
          id[j] = __ldcg(p.block_tables + (int64_t)rec[j].z * p.max_blocks + s * p.split_blocks + lane);
        q0[j] = __ldcg(p.qsl + rec[j].z);
      }
    }
    const int first = filled;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      if (ended) break;
      TaskEntry* e = &sm.queue[filled % T::QD];
      int nb = 0, nst = 0, rot = 0;
      if (rec[j].x >= 0) {
        const int g = rec[j].y & 0xFF, s = rec[j].y >> 8, ctx = rec[j].w;
        nb = min(p.split_blocks, (ctx + kBS - 1) / kBS - s * p.split_blocks);
        if (lane < nb) {
          int v = id[j];
          if (v < 0 || v >= p.num_blocks) {
            dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
            v = 0;  // keep the copy in bounds; this token's output is flagged as invalid
          }
          e->ids[lane] = v;
        }
        const int qi = rec[j].x - q0[j];  // the token's index among its row's new tokens
        nst = ctx - 1 - qi;
        rot = (qi + g + s) & 3;  // row-local, so the dealing (and the result) does not depend on the batch
      }
      if (lane == 0) {
        e->rec = rec[j];
        e->nst = nst;
        e->nb = nb;
        e->rot = rot;
      }
      // Append fused: the split holding the token's own position reads its key and value rows from the
      // inputs (and its slot) in the middle of its last block, where the load's latency is exposed; bring
      // them into L2 now, a task or more before they are needed.
      if (p.k_in != nullptr && rec[j].x >= 0 && nb > 0 &&
          (rec[j].y >> 8) == ((rec[j].w + kBS - 1) / kBS - 1) / p.split_blocks) {
        constexpr int LINES = D * 2 / 128;  // 128-byte lines of one row
        const size_t row = ((size_t)rec[j].x * p.num_kv_heads + (rec[j].y & 0xFF)) * D;
        if (lane < LINES) dev::prefetch_l2(p.k_in + row + lane * 64);
        else if (lane < 2 * LINES) dev::prefetch_l2(p.v_in + row + (lane - LINES) * 64);
        else if (lane == 2 * LINES) dev::prefetch_l2(p.slots + rec[j].x);
      }
      ++filled;
      ended = rec[j].x < 0;
      last_nb = nb;
    }
    __syncwarp();
    if (lane == 0)
      for (int f = first; f < filled; ++f) dev::mbar_arrive(&sm.qfull[f % T::QD]);
  }
  // Before the dependency wait: the static entries (they touch no counter).
  __device__ void prologue() {
    n_tasks = __ldcg(&p.hdr->n_tasks);
    static_assert(kStaticTasks == 1, "one static task");
    const int idx[kStaticTasks] = {(int)blockIdx.x};
    last_idx = idx[0];
    publish(idx);
  }
  __device__ void run() {
    static_assert(kStaticTasks < T::QD, "queue");
    static_assert(T::QD == 3, "entry m reuses the slot of task m - 3");
    while (!ended) {
      // Entry m is claimed once every streaming warp is half-way through task m - 1 (and entry m's slot, last
      // used by task m - 3, is free): late enough that the next task goes to the CTA that will be free first
      // (a CTA holding one unstarted task for a whole task's time unbalanced the launch: the busiest CTA held
      // 1.3x the average), early enough that the claim, the task's record and its first K/V runs arrive
      // before the warps run dry.  Once the list has reached small tasks (it is ordered largest first) a CTA
      // can hold one more without unbalancing the launch: those are claimed as soon as the slot is free.
      const int m = filled;
      // A long list (many tasks per CTA) balances itself; there the next task is claimed as soon as the
      // previous one has been handed on, for the deepest look-ahead.
      const bool small = last_nb <= kEagerClaimBlocks || n_tasks > 4 * (int)gridDim.x;
      // Near the end of the list (this CTA's last claim was within two grids of it), the counter is read
      // before waiting: once every task has been claimed (the counter may lag, never run ahead) the end of
      // the work is published at once, and the warps finish without waiting for a claim that can only come
      // back empty.
      bool out = false;
      if (last_idx + 2 * (int)gridDim.x >= n_tasks) {
        int seen = 0;
        if (lane == 0) seen = dev::ld_relaxed_gpu(&p.hdr->work);
        out = kStaticTasks * (int)gridDim.x + __shfl_sync(0xffffffffu, seen, 0) >= n_tasks;
      }
      if (!out && !small && !cta_wait(&sm.qmid[(m - 1) % T::QD], ((m - 1) / T::QD) & 1, sm.abort, p.err)) return;
      const int gate = m - T::QD;
      if (gate >= 0 && !cta_wait(&sm.qempty[gate % T::QD], (gate / T::QD) & 1, sm.abort, p.err)) return;
      int c = 0;
      if (lane == 0 && !out) c = atomicAdd(&p.hdr->work, 1);
      const int idx[1] = {out ? n_tasks : kStaticTasks * (int)gridDim.x + __shfl_sync(0xffffffffu, c, 0)};
      last_idx = idx[0];
      publish(idx);
    }
  }
};

// ---------------------------------------------------------------------------------------------------
// Combiner warp: combines the streaming warps' shares of every task with log-sum-exp weights and writes a
// one-split token's fp16 output.  A split of a multi-split token is finished one of two ways:
//  * every other split of the token was already counted when the combiner took the task (an acquire load
//    of the token's counter as the task starts): it merges the token at the task's end -- the other splits'
//    partials from L2 (with one other split, copied into shared memory while the task streams), its own
//    from shared memory or registers -- and resets the counter.  Under the largest-first task order this is the usual case for a token's last,
//    small split.
//  * otherwise it writes its unnormalised partial and counts it on the token's counter at once (the release
//    waits for the partial's stores; the combiner has the slack), examines the count's result when it takes
//    the next task (or the end of the work), and the warp that completes the count merges the token there,
//    while the next task streams.  Counting at once lets the count reach the token's other splits while they
//    run, so that near the end of the launch the last split usually merges at its end with nothing to load.
// Traces of a 256-row decode layer showed the last CTAs spending ~4 us after their last block on merges whose
// loads (and a count's round trip) came after the shares; both are now off that path.
// Nothing here stalls the streaming warps.
// ---------------------------------------------------------------------------------------------------
// One step of the split fold (log-sum-exp): the running (M, L) take split (m, l) in; a scales what was
// accumulated, f the split's values.  Shared by every merge path so their bits agree.
__device__ __forceinline__ void fold_weights(float& M, float& L, float2 ml, float& a, float& f) {
  const float nM = fmaxf(M, ml.x);
  a = exp2f(M - nM);
  f = exp2f(ml.x - nM);
  M = nM;
  L = fmaf(ml.y, f, L * a);
}
__device__ __forceinline__ float fold_value(float acc, float a, float v, float f) { return fmaf(v, f, acc * a); }

template <int D, int G, int KV>
struct Combiner {
  using T = DecodeTraits<D, G, KV>;
  static constexpr int NG = G * D / 4;         // groups of 4 consecutive dims of one head (the G heads)
  static constexpr int EG = (NG + 31) / 32;    // groups per lane
  static constexpr int R = EG <= 6 ? 2 : 1;    // other splits whose loads are in flight together
  const DecodeParams& p;
  const DecodeSmem<D, G, KV>& sm;
  int lane;

  __device__ Combiner(const DecodeParams& p_, const DecodeSmem<D, G, KV>& sm_, int lane_) : p(p_), sm(sm_), lane(lane_) {}

  // Merge the nsplit partials of token-head tg (all final) into its fp16 output with log-sum-exp weights in
  // split order, so the result does not depend on which CTA merges or how.  Split `own` (-1: none) is this
  // warp's and was never written out: its o is in the staging buffer stg ([G][D] fp32), its (m, l) in mml.
  // The others are read from L2 (.cg): they were written by other CTAs during this launch.
  __device__ void merge(int tg, int nsplit, int own) {
    const size_t sb = (size_t)tg * p.max_splits;
    float M[EG], L[EG];
    float4 acc[EG];
#pragma unroll
    for (int j = 0; j < EG; ++j) {
      M[j] = -INFINITY;
      L[j] = 0.f;
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int nrem = nsplit - (own >= 0 ? 1 : 0);  // splits read from L2
    for (int s0 = 0, r0 = 0; s0 < nsplit;) {
      // this round: the next n splits read from L2 (and the own split, if it falls among them), in order
      const int n = min(R, nrem - r0);
      const bool own_in = own >= s0 && own <= s0 + n;
      const int s1 = min(nsplit, s0 + n + (own_in ? 1 : 0));
      float4 o[R][EG];
      float2 ml[R][EG];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        if (u >= n) break;
        const int su = s0 + u + (own_in && own <= s0 + u ? 1 : 0);
#pragma unroll
        for (int j = 0; j < EG; ++j) {
          const int e4 = lane + 32 * j;
          if (e4 < NG) {
            ml[u][j] = __ldcg(p.part_ml + (sb + su) * kHeadsTile + (4 * e4) / D);
            o[u][j] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (sb + su) * kHeadsTile * D) + e4);
          }
        }
      }
      int u = 0;
      for (int s = s0; s < s1; ++s) {
#pragma unroll
        for (int j = 0; j < EG; ++j) {
          const int e4 = lane + 32 * j;
          if (e4 >= NG) continue;
          float2 m;
          float4 v;
          if (s == own) {
            m = sm.mml[(4 * e4) / D];
            v = reinterpret_cast<const float4*>(sm.stg)[e4];
          } else {
            // u < n <= R: pick the register copy without dynamic indexing
            m = ml[0][j];
            v = o[0][j];
#pragma unroll
            for (int q = 1; q < R; ++q)
              if (u == q) {
                m = ml[q][j];
                v = o[q][j];
              }
          }
          float a, f;
          fold_weights(M[j], L[j], m, a, f);
          acc[j].x = fold_value(acc[j].x, a, v.x, f);
          acc[j].y = fold_value(acc[j].y, a, v.y, f);
          acc[j].z = fold_value(acc[j].z, a, v.z, f);
          acc[j].w = fold_value(acc[j].w, a, v.w, f);
        }
        if (s != own) ++u;
      }
      s0 = s1;
      r0 += n;
    }
    const int t = tg / p.num_kv_heads, g = tg % p.num_kv_heads;
#pragma unroll
    for (int j = 0; j < EG; ++j) {
      const int e4 = lane + 32 * j;
      if (e4 >= NG) continue;
      const float il = 1.f / L[j];
      const __half2 lo = __floats2half2_rn(acc[j].x * il, acc[j].y * il);
      const __half2 hi = __floats2half2_rn(acc[j].z * il, acc[j].w * il);
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(&lo);
      v.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.num_q_heads + (size_t)g * G) * D + 4 * e4) = v;
    }
  }
  // A two-split token, merged at the end of its split `own`: this warp's result in registers (acc in fragment
  // order, (M0, L0) / (M1, L1) for the lane's two heads), the other split's partial copied into the staging
  // buffers (stg [G][D] fp32, mml [8]) while the task streamed.  The same fold as merge, element by element,
  // in split order, so the bits do not depend on which path merged.  The fp16 result is staged over stg and
  // written out coalesced.
  __device__ void merge_two(int tg, int own, float (&acc)[T::OV], float M0, float L0, float M1, float L1) {
    const bool real = (lane & 3) < T::LG;
    if (real) {
#pragma unroll
      for (int r = 0; r < T::OV; ++r) {
        int dim, head;
        frag_coord<KV>(lane, r, dim, head);
        if (head >= G) continue;
        const float2 mo = (r & 1) ? make_float2(M1, L1) : make_float2(M0, L0), mp = sm.mml[head];
        const float vo = acc[r], vp = sm.stg[head * D + dim];
        float M = -INFINITY, L = 0.f, x = 0.f;
        float a, f;
        fold_weights(M, L, own == 0 ? mo : mp, a, f);
        x = fold_value(x, a, own == 0 ? vo : vp, f);
        fold_weights(M, L, own == 0 ? mp : mo, a, f);
        x = fold_value(x, a, own == 0 ? vp : vo, f);
        acc[r] = x * (1.f / L);
      }
    }
    __syncwarp();  // every lane has read the partial before the fp16 result goes over it
    if (real) {
      __half* sh = reinterpret_cast<__half*>(sm.stg);
#pragma unroll
      for (int r = 0; r < T::OV; ++r) {
        int dim, head;
        frag_coord<KV>(lane, r, dim, head);
        if (head < G) sh[head * D + dim] = __float2half_rn(acc[r]);
      }
    }
    __syncwarp();
    const int t = tg / p.num_kv_heads, g = tg % p.num_kv_heads;
    uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)t * p.num_q_heads + (size_t)g * G) * D);
    for (int c = lane; c < G * D / 8; c += 32) dst[c] = reinterpret_cast<const uint4*>(sm.stg)[c];
  }
  // A count issued earlier (acquire-release): lane 0 holds the counter's old value.  The warp that
  // completes a token's count merges it: returns whether that is this warp.
  __device__ bool completes_count(int tg, int nsplit, int prev_lane0) {
    const int prev = __shfl_sync(0xffffffffu, prev_lane0, 0);
    if (prev != nsplit - 1) return false;
    if (lane == 0) p.merge_cnt[tg] = 0;  // ready for the next launch on this plan
    __syncwarp();
    return true;
  }

  __device__ void run() {
    uint32_t taken = 0;               // bit w: parity of the shares taken from streaming warp w so far
    // the merge due when the next task (or the end of the work) is in hand: token pm_tg's, with this warp's split
    // pm_own staged in shared memory (or -1), and (pm_cnt) only if the count issued for it completes the token
    int pm_tg = -1, pm_ns = 0, pm_own = -1, ct_prev = 0;
    bool pm_cnt = false;
    uint32_t pcopies = 0;  // partial copies into the staging buffers so far (pbar phases)
    const int hg = lane & 3;
    const bool real = hg < T::LG;     // this lane's fragment columns hold real heads
    const int ci = (lane >> 2) * T::LG + hg;
    for (int k = 0;; ++k) {
      // ---- the task's description; then its queue slot may be refilled ----
      if (!cta_wait(&sm.qfull[k % T::QD], (k / T::QD) & 1, sm.abort, p.err)) return;
      const TaskEntry* e = &sm.queue[k % T::QD];
      const int4 rec = e->rec;
      const int nb = e->nb, rot = e->rot;
      __syncwarp();
      // ---- the merge left by the previous task (its count examined now): it runs while this task streams ----
      if (pm_tg >= 0) {
        if (!pm_cnt || completes_count(pm_tg, pm_ns, ct_prev)) merge(pm_tg, pm_ns, pm_own);
        pm_tg = -1;
      }
      if (rec.x < 0) break;
      if (lane == 0) dev::mbar_arrive(&sm.qempty[k % T::QD]);
      const int t = rec.x, g = rec.y & 0xFF, s = rec.y >> 8, ctx = rec.w;
      const int nblk = (ctx + kBS - 1) / kBS;
      const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
      const int tg = t * p.num_kv_heads + g;
      const bool multi = nsplit > 1 && nsplit <= kFusedMergeSplits;
      int done_lane0 = 0;  // splits of the token counted so far
      if (multi && lane == 0) done_lane0 = dev::ld_acquire_gpu(p.merge_cnt + tg);
      // Every other split already counted: this task merges the token at its end.  With one other split (the
      // usual case: a token's last, small split, under the largest-first order) that split's partial is copied
      // into the staging buffers now, while the task streams.
      const bool m2 = multi && __shfl_sync(0xffffffffu, done_lane0, 0) == nsplit - 1;
      const bool pre = m2 && nsplit == 2;
      if (pre) {
        __syncwarp();  // every read of the staging buffers (the merge above) precedes the copy over them
        if (lane == 0) {
          const size_t pidx = (size_t)tg * p.max_splits + (1 - s);
          dev::fence_proxy_async_smem();
          dev::fence_proxy_async_global();  // the counts' acquire precedes the copy's reads
          dev::mbar_arrive_expect_tx(sm.pbar, G * D * 4 + kHeadsTile * 8);
          dev::bulk_g2s_plain(sm.stg, p.part_o + pidx * kHeadsTile * D, G * D * 4, sm.pbar);
          dev::bulk_g2s_plain(sm.mml, p.part_ml + pidx * kHeadsTile, kHeadsTile * 8, sm.pbar);
        }
      }
      // an abort below must not leave the CTA with the copy in flight
      auto bail = [&]() {
        if (pre) dev::mbar_wait(sm.pbar, pcopies & 1);
      };
      // ---- combine the shares in warp order (a fixed order: the result does not depend on timing) ----
      float acc[T::OV];
#pragma unroll
      for (int r = 0; r < T::OV; ++r) acc[r] = 0.f;
      float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
      for (int w = 0; w < T::NW; ++w) {
        if (warp_blocks(nb, (w - rot) & 3) == 0) continue;
        if (!cta_wait(&sm.share_full[w], (taken >> w) & 1, sm.abort, p.err)) {
          bail();
          return;
        }
        taken ^= 1u << w;
        if (real) {
          const float2 ma = sm.sh_ml[w * kHeadsTile + 2 * hg], mb = sm.sh_ml[w * kHeadsTile + 2 * hg + 1];
          float a0 = 1.f, f0 = 0.f, a1 = 1.f, f1 = 0.f;
          if (ma.x != -INFINITY) {
            const float nM = fmaxf(M0, ma.x);
            a0 = exp2f(M0 - nM);
            f0 = exp2f(ma.x - nM);
            M0 = nM;
            L0 = L0 * a0 + ma.y * f0;
          }
          if (mb.x != -INFINITY) {
            const float nM = fmaxf(M1, mb.x);
            a1 = exp2f(M1 - nM);
            f1 = exp2f(mb.x - nM);
            M1 = nM;
            L1 = L1 * a1 + mb.y * f1;
          }
          const float* so = sm.sh_o + w * T::OV * T::SHL;
#pragma unroll
          for (int r = 0; r < T::OV; ++r) acc[r] = acc[r] * ((r & 1) ? a1 : a0) + so[r * T::SHL + ci] * ((r & 1) ? f1 : f0);
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&sm.share_empty[w]);
      }
      // ---- stage the result in shared memory (the fragment layout is not the output layout) ----
      if (real) {
        if (nsplit == 1) {
          __half* sh = reinterpret_cast<__half*>(sm.stg);
          const float i0 = 1.f / L0, i1 = 1.f / L1;
#pragma unroll
          for (int r = 0; r < T::OV; ++r) {
            int dim, head;
            frag_coord<KV>(lane, r, dim, head);
            if (head < G) sh[head * D + dim] = __float2half_rn(acc[r] * ((r & 1) ? i1 : i0));
          }
        } else if (!pre) {
#pragma unroll
          for (int r = 0; r < T::OV; ++r) {
            int dim, head;
            frag_coord<KV>(lane, r, dim, head);
            if (head < G) sm.stg[head * D + dim] = acc[r];
          }
          if (lane < T::LG) {
            sm.mml[2 * lane] = make_float2(M0, L0);
            sm.mml[2 * lane + 1] = make_float2(M1, L1);
          }
        }
      }
      // ---- this task's token, if every other split of it was counted before it started (its own split from
      // shared memory): with two splits now (nothing left to load), otherwise when the next task is in hand ----
      if (m2 && lane == 0) p.merge_cnt[tg] = 0;  // nobody else counts this token again in this launch
      __syncwarp();
      if (pre) {
        const bool got = cta_wait(sm.pbar, pcopies & 1, sm.abort, p.err);
        ++pcopies;
        if (!__all_sync(0xffffffffu, got)) {
          dev::mbar_wait(sm.pbar, (pcopies - 1) & 1);
          return;
        }
        merge_two(tg, s, acc, M0, L0, M1, L1);
      } else if (m2) {
        pm_tg = tg;
        pm_ns = nsplit;
        pm_own = s;
        pm_cnt = false;
      }
      // ---- the output, or the split's partial (unless merged above), counted at once: its count then
      // reaches the token's other splits while they run, and the one that starts (or finishes) last merges
      // with no count of its own ----
      __syncwarp();
      if (nsplit == 1) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)t * p.num_q_heads + (size_t)g * G) * D);
        for (int c = lane; c < G * D / 8; c += 32) dst[c] = reinterpret_cast<const uint4*>(sm.stg)[c];
      } else if (m2) {
      } else {
        const size_t pidx = (size_t)tg * p.max_splits + s;
        float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * kHeadsTile * D);
        for (int c = lane; c < G * D / 4; c += 32) dst[c] = reinterpret_cast<const float4*>(sm.stg)[c];
        if (real && lane < T::LG) {
          if (2 * lane < G) p.part_ml[pidx * kHeadsTile + 2 * lane] = make_float2(M0, L0);
          if (2 * lane + 1 < G) p.part_ml[pidx * kHeadsTile + 2 * lane + 1] = make_float2(M1, L1);
        }
        if (multi) {
          __syncwarp();  // every lane's stores precede the release below
          if (lane == 0) ct_prev = dev::atom_add_acq_rel_gpu(p.merge_cnt + tg, 1);
          pm_tg = tg;
          pm_ns = nsplit;
          pm_own = -1;
          pm_cnt = true;
        }
      }
      __syncwarp();  // the staging buffers are free again
    }
  }
};

template <int D, int G, int KV>
__global__ void __launch_bounds__(DecodeTraits<D, G, KV>::NTHREADS, DecodeTraits<D, G, KV>::MINB)
decode_kernel(const __grid_constant__ DecodeParams p) {
  using T = DecodeTraits<D, G, KV>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DecodeSmem<D, G, KV> sm(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // set-up that reads nothing written by earlier kernels runs before the dependency wait
  if (threadIdx.x == 0) {
    for (int i = 0; i < T::NW * T::NR; ++i) dev::mbar_init(&sm.ring_bar[i], 1);
    for (int i = 0; i < T::NW; ++i) {
      dev::mbar_init(&sm.share_full[i], 1);
      dev::mbar_init(&sm.share_empty[i], 1);
    }
    for (int i = 0; i < T::QD; ++i) {
      dev::mbar_init(&sm.qfull[i], 1);
      dev::mbar_init(&sm.qempty[i], T::NW + 1);  // the streaming warps and the combiner
    }
    for (int i = 0; i < T::NW; ++i) dev::mbar_init(&sm.qbar[i], 1);
    for (int i = 0; i < T::QD; ++i) dev::mbar_init(&sm.qmid[i], T::NW);  // the streaming warps
    dev::mbar_init(sm.pbar, 1);
    *sm.abort = 0;
    dev::fence_mbar_init();
  }
  __syncwarp();
  __syncthreads();
  // The static tasks' records and block ids are read before the dependency wait: the plan kernel that
  // wrote the task list released its dependents only after its writes (and a fence), and block tables are
  // final before the plan; they are read through L2, never a possibly stale L1 line.  So are the first K/V
  // runs wherever no appended token can be in them.  q, the task counter and the partials are touched only
  // after the wait.
  Streamer<D, G, KV> w(p, sm, warp, lane);
  Scheduler<D, G, KV> sch(p, sm, lane);
  if (warp < T::NW) w.prologue(); else if (warp == T::NW + 1) sch.prologue();
  if (!p.late_wait) dev::griddep_wait();
  dev::griddep_launch_dependents();
  if (warp < T::NW) w.after_wait();  // the first task's q (in bounds even if the pool turns out poisoned)
  // one CTA-uniform decision (a racing error-word update must not split the CTA); every warp arrives
  // converged at each CTA barrier (its predicate is computed first)
  int pz = 0;
  if (threadIdx.x == 0) pz = dev::pool_poisoned(p.err) ? 1 : 0;
  __syncwarp();
  const bool poisoned = __syncthreads_or(pz);
  if (warp < T::NW) {
    if (!poisoned) stream_loop<D, G, KV>(p, sm, w);
    w.drain();
  } else if (!poisoned) {
    if (warp == T::NW) Combiner<D, G, KV>(p, sm, lane).run();
    else sch.run();
  }
  // The last CTA out resets the task counter for the next launch on this plan.  No fence on either side: a
  // CTA's claims are atomics whose results it has used before this barrier (performed at L2 before its count
  // below is issued), and the next launch reads the counters only after its dependency wait, which sees every
  // write of this grid.  This sits on the critical path of every launch (the last CTA's exit).
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (atomicAdd(&p.hdr->done, 1) == (int)gridDim.x - 1) {
      p.hdr->work = 0;
      p.hdr->done = 0;
    }
  }
  if (p.late_wait) dev::griddep_wait();  // complete only after the prefill kernel ahead of it
}

template <int D, int G, int KV>
static cudaError_t launch_decode(const DecodeParams& p, int num_sms, int64_t max_tasks, cudaStream_t stream) {
  using T = DecodeTraits<D, G, KV>;
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, G, KV>, T::NTHREADS, T::SMEM);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
  }
  int64_t grid = (int64_t)num_sms * per_sm;  // persistent: one CTA per resident slot, one task at a time
  if (grid > max_tasks) grid = max_tasks;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_kernel<D, G, KV>, dim3((unsigned)grid), dim3(T::NTHREADS), T::SMEM, stream, p);
}

template <int D, int KV>
static cudaError_t launch_decode_g(int group, const DecodeParams& p, int num_sms, int64_t max_tasks,
                                   cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode<D, 1, KV>(p, num_sms, max_tasks, stream);
    case 2: return launch_decode<D, 2, KV>(p, num_sms, max_tasks, stream);
    case 4: return launch_decode<D, 4, KV>(p, num_sms, max_tasks, stream);
    case 6: return launch_decode<D, 6, KV>(p, num_sms, max_tasks, stream);
    case 8: return launch_decode<D, 8, KV>(p, num_sms, max_tasks, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The 8-bit cache's instances live in their own translation unit (decode_e4m3.cu).
cudaError_t launch_decode_e4m3(int head_dim, int group, const DecodeParams& p, int num_sms, int64_t max_tasks,
                               cudaStream_t stream);

}  // namespace pkv
