// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// What is computed ("Continuous Batching Is Not a Bigger Batch", section "What the scheduler does on one
// step": a prompt is consumed in chunks under the per-pass token budget): for each new token of a row
// with many new tokens, causal attention over the row's keys in the paged cache -- query i of a chunk of
// q_len on top of ctx - q_len cached tokens sees keys 0 .. ctx - q_len + i -- for every query head, the
// head h reading KV head h / G, scores scaled by 1/sqrt(d), fp32 softmax, fp16 output.
//
// How (GB300 design):
//  * A Q tile is 128 MMA rows = P = 128 / G consecutive query positions x the G query heads of one KV
//    head (row r = position r / G, head r % G): every K/V tile is read once for the whole group, and
//    the causal diagonal wastes at most P keys per tile.  A work item is two adjacent Q tiles of one row
//    and KV head; they share every 128-key K/V tile.  (At head_dim 256 an item is one Q tile on 64-key
//    tiles, PfTraits below: the warps, columns and shared memory of one group.)
//  * Persistent CTAs of 11 warps.  Warp 9 streams K and V tiles from the paged pool with 2-D TMA copies
//    (128-byte swizzle) into rings of 3 K and 2 V slots, block ids fetched a tile ahead.  Warps 8 and 10
//    each issue, from one thread, one Q tile's MMAs S = Q K^T (M 128, N 128, K d) and O += P V (M 128,
//    N d, K 128), fp32 accumulators in tensor memory (per Q tile: S and O, 256 columns; 512 in all).
//    Warpgroups 0 and 1 (softmax) each own one Q tile, one S/O row per thread (TMEM lane = thread):
//    they load S with tcgen05.ld, apply the causal mask and an online softmax in the log2 domain, and
//    store P as fp16 over the S they just read (tcgen05.st); the product takes P straight from tensor
//    memory.  Per group the order is S(j), P(j)V, S(j + 1), P(j + 1)V, ...: while one group runs its
//    softmax the tensor core works on the other group's products and scores.
//  * Measured on GB300: one thread issues a 128 x 128 x 16 tcgen05.mma about every 113 cycles whatever N up
//    to 128, two issuing warps one every ~64 (the tensor core's rate).  Hence one issuing warp per Q tile,
//    and 128-wide score tiles (not 64).
//  * The running max is lazy: O (in TMEM) and the running sum are rescaled only when a row's max grows
//    by more than 8 (a factor 256), which keeps P <= 256 and the arithmetic exact up to rounding.
//  * Items are taken longest first (the plan sorts them by K/V tile count) from a global counter.
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "attn_common.cuh"

namespace pkv {

namespace {

constexpr int kKSlots = 3;             // K ring depth
constexpr int kVSlots = 2;             // V ring depth
constexpr int kWG = 2;                 // softmax warpgroups (Q tiles per item) at most
constexpr int kBarItem = 1, kBarQ = 2, kBarEpi = 3;  // named barriers (0 is __syncthreads)
constexpr float kRescaleLog2 = 8.f;    // lazy rescale threshold (log2 units)

// Per head dim: d <= 128 runs two Q tiles per item on 128-key K/V tiles (per Q tile S 128 + O 128 tensor
// memory columns: 512 in all); d = 256 runs one Q tile on 64-key tiles (S 64 + O 256 columns), which also
// keeps the Q tile (64 KB) and the K/V rings within shared memory.
template <int D, int G>
struct PfTraits {
  static constexpr int WG = D == 256 ? 1 : 2;         // softmax warpgroups = Q tiles per item
  static constexpr int KEYS = prefill_tile_keys(D);   // keys per K/V tile
  static constexpr int NH = KEYS / 64;                // 64-key halves of a row of scores
  static constexpr int MMA0 = 4 * WG;                 // issues group 0's MMAs and hands out items
  static constexpr int TMA = 4 * WG + 1;              // streams K/V tiles
  static constexpr int MMA1 = 4 * WG + 2;             // issues group 1's MMAs (two groups only)
  static constexpr int THREADS = (5 * WG + 1) * 32;   // softmax groups, the TMA warp, an MMA warp per group
  static constexpr int Q_THREADS = 5 * WG * 32;       // the Q-tile barrier: softmax groups + MMA warps
  static constexpr int SOFTMAX_THREADS = 4 * WG * 32;
  static constexpr int DH = D / 64;                   // 64-column halves of a row (128-byte swizzle atoms)
  static constexpr int P = prefill_positions(G);      // query positions per Q tile
  static constexpr int QTILE = DH * 128 * 128;        // 128 rows x D fp16
  static constexpr int KVTILE = DH * KEYS * 128;      // KEYS keys x D fp16
  static constexpr int OFF_Q = 0;                     // [WG]
  static constexpr int OFF_K = OFF_Q + WG * QTILE;    // [kKSlots]
  static constexpr int OFF_V = OFF_K + kKSlots * KVTILE;  // [kVSlots]
  static constexpr int OFF_BAR = OFF_V + kVSlots * KVTILE;
  static constexpr int OFF_MISC = OFF_BAR + 256;      // TMEM base, item record, abort flag, slot, merge order
  static constexpr int SMEM = OFF_MISC + 64 + 1024;   // + slack to align to 1024 bytes
  // tensor memory of group w: S (KEYS columns; P, as fp16, overwrites its first KEYS / 2), then O (D columns)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t SO = D == 256 ? 256 : 128;  // O's first column, past S's
  __host__ __device__ static constexpr uint32_t s_col(int w) { return 256u * (uint32_t)w; }
  static constexpr uint32_t IDESC_S = dev::umma_idesc_f16(128, KEYS, false, false);
  static constexpr uint32_t IDESC_PV = dev::umma_idesc_f16(128, D, false, true);
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(WG * 256 <= (int)TMEM_COLS && SO + D <= 256u * (3 - WG), "tensor memory");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct PfParams {
  CUtensorMap kv_map;
  const __half* q;
  __half* out;
  const int32_t* block_tables;
  const int4* items;
  const int32_t* items_slot;
  int2* pf_sync;
  float2* pf_ml;
  float* pf_o;
  WsHeader* hdr;
  int32_t* err;
  int layer_row0_k, layer_row0_v;
  int max_blocks, num_q_heads, num_kv_heads, num_blocks;
  float scale_log2;
};

struct Bars {
  uint64_t* kfull;    // [kKSlots]  K tile landed (TMA bytes)
  uint64_t* kfree;    // [kKSlots]  the scores that read the slot's K tile have completed (tcgen05.commit)
  uint64_t* vfull;    // [kVSlots]  V tile landed
  uint64_t* vfree;    // [kVSlots]  the products that read the slot's V tile have completed
  uint64_t* s_done;   // [kWG]      S of the group's current tile written (and every earlier MMA done)
  uint64_t* p_ready;  // [kWG]      P written over S, O rescaled (128 arrivals)
  uint64_t* pv_done;  // [kWG]      the group's product of its current tile completed
  uint64_t* zfill;    // [1]        the last tile's V rows past the item's keys zeroed (128 arrivals; one phase per
                      //            entry that holds an item's partial last tile)
  uint32_t* tmem_base;
  int4* item;
  volatile int* abort;
  volatile int* slot;   // the current entry's split slot (-1: not split)
  volatile int* order;  // split entries: 0 if this chunk finished first, 1 if it merges
};

// Bounded wait that, once any wait of the CTA has given up, no longer waits at all: every thread then
// runs through the remaining (bounded) loops with garbage and the CTA stays in step at its barriers.
__device__ __forceinline__ void pf_wait(const Bars& sh, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*sh.abort) return;
  if (!dev::mbar_wait(bar, parity)) {
    *sh.abort = 1;
    dev::set_error(err, PKV_DEVERR_WAIT_TIMEOUT);
  }
}

// Byte offset of 16-byte chunk c (8 fp16) of row r in a 128-row tile stored as 64-column halves of
// 16 KB with the 128-byte swizzle.
__device__ __forceinline__ uint32_t qtile_off(int r, int c) {
  return (uint32_t)((c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// The work entry's geometry as seen by each of the item's Q tiles.
struct ItemGeo {
  int row, g, t0, w0;   // row, KV head, first token, keys visible to the first position minus one
  int npos[kWG];        // positions of each Q tile (0: the tile is empty)
  int n[kWG];           // K/V tiles each Q tile needs
  int n_all;            // K/V tiles of the item
  int kend_all;         // keys of the item
  int zfill_wg;         // the group that zeroes V rows past the item's keys in the last tile
  int split, chunk;     // split-KV: this entry is chunk `chunk` of 2
  int tb, te;           // K/V tiles [tb, te) of the item that this entry processes
};

template <class T>
__device__ __forceinline__ ItemGeo item_geo(const int4 rec) {
  constexpr int P = T::P;
  ItemGeo it;
  it.row = rec.x;
  it.g = rec.y & 0xFF;
  const int npos = (rec.y >> 8) & 0x1FF;
  it.chunk = (rec.y >> 20) & 1;
  it.split = (rec.y >> 21) & 1;
  it.t0 = rec.z;
  it.w0 = rec.w;
  it.n_all = 0;
  it.kend_all = 0;
  it.zfill_wg = 0;
#pragma unroll
  for (int w = 0; w < kWG; ++w) {
    it.npos[w] = w < T::WG ? max(0, min(P, npos - w * P)) : 0;
    const int kend = it.w0 + w * P + it.npos[w];
    it.n[w] = it.npos[w] > 0 ? (kend + T::KEYS - 1) / T::KEYS : 0;
    if (it.npos[w] > 0) {
      it.n_all = it.n[w];
      it.kend_all = kend;
      it.zfill_wg = w;
    }
  }
  const int h = (it.n_all + 1) / 2;  // the first chunk takes the extra tile
  it.tb = it.split && it.chunk ? h : 0;
  it.te = it.split && !it.chunk ? h : it.n_all;
  return it;
}

// ---- TMA warp: K/V tiles of the item into the rings, block ids fetched one tile ahead ---------------
template <int D, int G>
__device__ void tma_warp(const PfParams& p, unsigned char* smem, const Bars& sh, int lane) {
  using T = PfTraits<D, G>;
  constexpr int BPT = T::KEYS / kBS;  // blocks per K/V tile
  static_assert(BPT * T::DH <= 32, "one box per lane");
  const uint64_t pol = dev::l2_policy_evict_last();
  int gt = 0;  // CTA-wide index of the next K/V tile
  while (true) {
    dev::named_bar_sync(kBarItem, T::THREADS);
    const volatile int* vi = reinterpret_cast<volatile int*>(sh.item);
    const int4 rec = make_int4(vi[0], vi[1], vi[2], vi[3]);
    if (rec.x < 0) break;
    const ItemGeo it = item_geo<T>(rec);
    const int n = it.te - it.tb;  // tiles of this entry: item tiles tb .. te - 1
    const int nblk = (it.kend_all + kBS - 1) / kBS;
    const int32_t* bt = p.block_tables + (int64_t)it.row * p.max_blocks;
    auto load_ids = [&](int u) {
      const int j = it.tb + u;  // lane i < blocks of tile j: physical id of the tile's block i
      int id = 0;
      if (lane < min(BPT, nblk - j * BPT)) {
        id = __ldg(bt + j * BPT + lane);
        if (id < 0 || id >= p.num_blocks) {
          dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          id = 0;
        }
      }
      return id;
    };
    // TMA of tile j's K (v = false) or V (v = true) into its ring slot, once the MMAs that read the tile
    // a ring-length earlier from that slot have completed.  One 2 KB box (16 keys x 64 columns) per lane:
    // a single issuing thread would be the bottleneck.
    auto issue = [&](int u, bool v, int id) {
      const int j = it.tb + u, gi = gt + u;
      const int slots = v ? kVSlots : kKSlots;
      const int slot = gi % slots;
      if (gi >= slots) pf_wait(sh, v ? &sh.vfree[slot] : &sh.kfree[slot], ((gi - slots) / slots) & 1, p.err);
      const int nb = min(BPT, nblk - j * BPT);
      unsigned char* dst = smem + (v ? T::OFF_V : T::OFF_K) + slot * T::KVTILE;
      uint64_t* full = v ? &sh.vfull[slot] : &sh.kfull[slot];
      const int row0 = v ? p.layer_row0_v : p.layer_row0_k;
      if (lane == 0) dev::mbar_arrive_expect_tx(full, (uint32_t)(nb * T::DH * 2048));
      __syncwarp();
      const int blk = lane / T::DH, h = lane % T::DH;
      const int bid = __shfl_sync(0xffffffffu, id, blk & 31);
      if (lane < nb * T::DH)
        dev::tma_load_2d(dst + h * (T::KEYS * 128) + blk * 2048, &p.kv_map, h * 64,
                         row0 + (bid * p.num_kv_heads + it.g) * kBS, full, pol);
    };
    // K runs one tile ahead of V: a K slot is released by the scores, earlier than a V slot by the products
    int id_next = n > 0 ? load_ids(0) : 0, id_prev = 0;
    for (int t = 0; t <= n; ++t) {
      const int id_cur = id_next;
      if (t + 1 < n) id_next = load_ids(t + 1);
      if (t < n) issue(t, false, id_cur);
      if (t >= 1) issue(t - 1, true, id_prev);
      id_prev = id_cur;
    }
    gt += n;
  }
}

// ---- MMA warps: one per Q-tile group, each issuing its group's MMAs from one thread ------------------
// Measured on GB300: one issuing thread sustains one 128 x 128 x 16 MMA per ~113 cycles, two issuing warps
// together one per ~64 (the tensor core's rate).  So each group's scores and products come from its own warp;
// the K and V ring slots are released once both warps' MMAs that read them have completed (two arrivals).
// The first MMA warp also hands out the items.
template <int D, int G, int w>
__device__ void mma_warp(const PfParams& p, unsigned char* smem, const Bars& sh, int lane, int n_items) {
  using T = PfTraits<D, G>;
  const uint32_t sbase = dev::smem_addr(smem);
  const uint32_t tmem = *sh.tmem_base;
  // base descriptors (this group's Q tile, K slot 0, V slot 0): the others differ only in the start address
  const uint64_t dq = dev::umma_desc_sw128(sbase + T::OFF_Q + w * T::QTILE, 16, 1024);
  const uint64_t dk0 = dev::umma_desc_sw128(sbase + T::OFF_K, 16, 1024);
  const uint64_t dv0 = dev::umma_desc_sw128(sbase + T::OFF_V, T::KEYS * 128, 1024);
  int gt = 0;            // CTA-wide index of the next K/V tile
  int cw[kWG] = {0, 0};  // per Q-tile group: tiles processed so far (barrier phases)
  int nz = 0;            // entries so far whose item's partial last tile was zero-filled (zfill phases)
  bool first = true;
  while (true) {
    int4 rec = make_int4(-1, 0, 0, 0);
    if constexpr (w == 0) {
      if (lane == 0) {
        const int idx = first ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&p.hdr->pwork, 1);
        int slot = -1;
        if (idx < n_items) {
          rec = __ldg(p.items + idx);
          slot = __ldg(p.items_slot + idx);
        }
        *sh.item = rec;
        *sh.slot = slot;
      }
      first = false;
      rec.x = __shfl_sync(0xffffffffu, rec.x, 0);
      rec.y = __shfl_sync(0xffffffffu, rec.y, 0);
      rec.z = __shfl_sync(0xffffffffu, rec.z, 0);
      rec.w = __shfl_sync(0xffffffffu, rec.w, 0);
      __syncwarp();
      dev::named_bar_arrive(kBarItem, T::THREADS);
    } else {
      dev::named_bar_sync(kBarItem, T::THREADS);
      const volatile int* vi = reinterpret_cast<volatile int*>(sh.item);
      rec = make_int4(vi[0], vi[1], vi[2], vi[3]);
    }
    if (rec.x < 0) break;
    const ItemGeo it = item_geo<T>(rec);
    const int n = it.te - it.tb;  // tiles of this entry; u below is the entry's tile, tb + u the item's
    int ne[kWG];                  // tiles of this entry per group
#pragma unroll
    for (int g = 0; g < kWG; ++g) ne[g] = g < T::WG ? max(0, min(it.te, it.n[g]) - it.tb) : 0;
    const int zf = it.zfill_wg;
    // this entry holds the item's last tile and it is partial: group zf zeroes its V rows past the keys
    const bool zfe = it.te == it.n_all && it.kend_all - (it.n_all - 1) * T::KEYS < T::KEYS;

    auto issue_s = [&](int j) {  // S_w(u = j) = Q_w K^T; commits every earlier MMA of this warp too
      const uint64_t dk = dk0 + (uint64_t)((((gt + j) % kKSlots) * T::KVTILE) >> 4);
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          dev::umma_f16_ss(tmem + T::s_col(w), dq + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                           dk + (uint64_t)(((kk >> 2) * (T::KEYS * 128) + (kk & 3) * 32) >> 4), T::IDESC_S, kk > 0);
        dev::umma_commit(&sh.s_done[w]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int j) {  // O_w (+)= P_w(j) V(j), P from tensor memory
      const uint64_t dv = dv0 + (uint64_t)((((gt + j) % kVSlots) * T::KVTILE) >> 4);
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < T::KEYS / 16; ++kk)
          dev::umma_f16_ts(tmem + T::s_col(w) + T::SO, tmem + T::s_col(w) + 8 * kk, dv + (uint64_t)((kk * 2048) >> 4),
                           T::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        dev::umma_commit(&sh.pv_done[w]);
      }
      __syncwarp();
    };
    auto commit = [&](uint64_t* bar) {
      if (lane == 0) dev::umma_commit(bar);
      __syncwarp();
    };

    dev::named_bar_sync(kBarQ, T::Q_THREADS);  // the Q tiles are in shared memory
    dev::tc_fence_after();
    pf_wait(sh, &sh.kfull[gt % kKSlots], (gt / kKSlots) & 1, p.err);
    if (ne[w] > 0) issue_s(0);
    commit(&sh.kfree[gt % kKSlots]);
    for (int j = 0; j < n; ++j) {
      const int gi = gt + j;
      const bool last = j == n - 1;
      pf_wait(sh, &sh.vfull[gi % kVSlots], (gi / kVSlots) & 1, p.err);
      if (!last) pf_wait(sh, &sh.kfull[(gi + 1) % kKSlots], ((gi + 1) / kKSlots) & 1, p.err);
      if (j < ne[w]) {
        pf_wait(sh, &sh.p_ready[w], (cw[w] + j) & 1, p.err);
        // the last tile: the other group zeroes V rows past the item's keys (its own P is ready after that).  A
        // barrier of its own, one phase per such entry, since this warp does not follow the other group tile by
        // tile (a parity wait on its P barrier could match a phase two tiles old).
        if (last && zfe && zf != w) pf_wait(sh, sh.zfill, nz & 1, p.err);
        dev::tc_fence_after();
        // this group's product of tile j, then (P has been read) its scores of tile j + 1 over the same S
        issue_pv(j);
        if (j + 1 < ne[w]) issue_s(j + 1);
      }
      if (!last) commit(&sh.kfree[(gi + 1) % kKSlots]);
      commit(&sh.vfree[gi % kVSlots]);
    }
    gt += n;
#pragma unroll
    for (int g = 0; g < kWG; ++g) cw[g] += ne[g];
    if (zfe) ++nz;
  }
}

// ---- softmax warpgroups: one S / O row per thread ---------------------------------------------------
template <int D, int G>
__device__ void softmax_group(const PfParams& p, unsigned char* smem, const Bars& sh, int wg, int warp, int lane) {
  using T = PfTraits<D, G>;
  const int r = (warp & 3) * 32 + lane;  // this thread's tile row and TMEM lane
  const uint32_t tl = *sh.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + T::s_col(wg);  // lane, group columns
  const uint32_t sQa = dev::smem_addr(smem + T::OFF_Q + wg * T::QTILE);
  int cw = 0;  // tiles processed by this group so far (barrier phases)
  int gt = 0;  // K/V tiles of the CTA so far (V slot / phase of the zero-fill wait)
  while (true) {
    dev::named_bar_sync(kBarItem, T::THREADS);
    const volatile int* vi = reinterpret_cast<volatile int*>(sh.item);
    const int4 rec = make_int4(vi[0], vi[1], vi[2], vi[3]);
    if (rec.x < 0) break;
    const ItemGeo it = item_geo<T>(rec);
    const int slot = *sh.slot;
    const int n = max(0, min(it.te, wg ? it.n[1] : it.n[0]) - it.tb);  // this group's tiles of the entry
    const int pos = r / G, hq = r % G;
    const int npos = wg ? it.npos[1] : it.npos[0];
    const bool valid = r < T::P * G && pos < npos;
    const int first_pos = wg * T::P;
    const int lim = valid ? it.w0 + first_pos + pos : 0;  // last key this row sees (padding rows: key 0)
    const size_t tok = (size_t)(it.t0 + first_pos + pos);

    // ---- Q tile: row r = (position, head), 128-byte swizzle ----
    if (n > 0) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (tok * p.num_q_heads + (size_t)it.g * G + hq) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sQa + qtile_off(r, c)), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      dev::fence_proxy_async_smem();
    }
    dev::named_bar_arrive(kBarQ, T::Q_THREADS);

    float m_ref = -INFINITY, l = 0.f;
    for (int u = 0; u < n; ++u) {
      const int c = cw + u, j = it.tb + u;  // j: the item's tile
      // S(j) written; its commit also covers the product of tile j - 1, so O is settled
      pf_wait(sh, &sh.s_done[wg], c & 1, p.err);
      dev::tc_fence_after();
      const int kb = j * T::KEYS;
      // Whether every valid row of the warp sees the whole tile (warp-uniform): the causal mask costs a
      // compare and a select per score, so only the tiles that reach a row's diagonal take the masked code.
      // Then every key of the tile is one of the item's (the TMA wrote it), and the warp's padding rows
      // (zero q) score 0 on each.  A warp of padding rows alone keeps the mask (key 0 only).
      const bool full = __any_sync(0xffffffffu, valid) && __all_sync(0xffffffffu, !valid || kb + T::KEYS - 1 <= lim);
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      auto tile = [&](auto full_tag) {
        constexpr bool kFull = decltype(full_tag)::value;
        // masked max of one 64-column half of raw scores (the scale is positive, so it commutes with max)
        auto half_max = [&](const uint32_t (&s)[2][32], int h) {
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float x = __uint_as_float(s[k][e]);
              mx4[e & 3] = fmaxf(mx4[e & 3], (kFull || kb + 64 * h + 32 * k + e <= lim) ? x : -INFINITY);
            }
          return fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
        };
        // P = 2^(s * scale_log2 - m_ref) of one half as packed fp16; one FFMA and one MUFU per score
        auto half_exp = [&](const uint32_t (&s)[2][32], int h, uint32_t (&pk)[32], float (&sum4)[4]) {
          const float nm = -m_ref;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k = 2 * e;  // key 64 h + k of the tile
            float x0 = __uint_as_float(s[k >> 5][k & 31]), x1 = __uint_as_float(s[(k + 1) >> 5][(k + 1) & 31]);
            if constexpr (!kFull) {
              if (kb + 64 * h + k > lim) x0 = -INFINITY;
              if (kb + 64 * h + k + 1 > lim) x1 = -INFINITY;
            }
            const float p0 = dev::ex2_approx(fmaf(x0, p.scale_log2, nm));
            const float p1 = dev::ex2_approx(fmaf(x1, p.scale_log2, nm));
            sum4[e & 3] += p0 + p1;
            const __half2 hh = __floats2half2_rn(p0, p1);
            pk[e] = *reinterpret_cast<const uint32_t*>(&hh);
          }
        };
        auto load_half = [&](int h, uint32_t (&s)[2][32]) {
          dev::tmem_ld32(tl + 64 * h, s[0]);
          dev::tmem_ld32(tl + 64 * h + 32, s[1]);
          dev::tmem_wait_ld();
        };
        // Common case (the reference is settled): one pass over S, both halves' P kept in registers and
        // stored only once neither half moves the row max past the lazy threshold, so S is still intact
        // for the two-pass path when one does.
        bool done = false;
        if (u > 0) {
          bool ok;
          if constexpr (T::NH == 2) {
            uint32_t pk0[32], pk1[32];
            {
              uint32_t s[2][32];
              load_half(0, s);
              ok = !__any_sync(0xffffffffu, half_max(s, 0) > m_ref + kRescaleLog2);
              if (ok) half_exp(s, 0, pk0, sum4);
            }
            if (ok) {
              uint32_t s[2][32];
              load_half(1, s);
              ok = !__any_sync(0xffffffffu, half_max(s, 1) > m_ref + kRescaleLog2);
              if (ok) half_exp(s, 1, pk1, sum4);
            }
            if (ok) {
              dev::tmem_st32(tl, pk0);
              dev::tmem_st32(tl + 32, pk1);
            }
          } else {  // one 64-key half
            uint32_t pk0[32];
            uint32_t s[2][32];
            load_half(0, s);
            ok = !__any_sync(0xffffffffu, half_max(s, 0) > m_ref + kRescaleLog2);
            if (ok) {
              half_exp(s, 0, pk0, sum4);
              dev::tmem_st32(tl, pk0);
            }
          }
          if (ok) {
            done = true;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) sum4[i] = 0.f;
          }
        }
        if (!done) {
          // ---- two passes: the row max first (and, past the first tile, the lazy rescale), then P ----
          float mx;
          {
            uint32_t s[2][32];
            load_half(0, s);
            mx = half_max(s, 0);
            if constexpr (T::NH == 2) {
              load_half(1, s);
              mx = fmaxf(mx, half_max(s, 1));
            }
          }
          if (u == 0) {
            m_ref = mx;
          } else {
            const bool need = mx > m_ref + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
              const float alpha = need ? exp2f(m_ref - mx) : 1.f;
#pragma unroll
              for (int k = 0; k < D / 32; ++k) {
                uint32_t o[32];
                dev::tmem_ld32(tl + T::SO + 32 * k, o);
                dev::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                dev::tmem_st32(tl + T::SO + 32 * k, o);
              }
              if (need) {
                l *= alpha;
                m_ref = mx;
              }
            }
          }
          // P over the first 64 columns of S: the first half's columns, already read when the second
          // half is loaded
#pragma unroll
          for (int h = 0; h < T::NH; ++h) {
            uint32_t s[2][32], pk[32];
            load_half(h, s);
            half_exp(s, h, pk, sum4);
            dev::tmem_st32(tl + 32 * h, pk);
          }
        }
      };
      if (full) tile(std::true_type{}); else tile(std::false_type{});
      l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      // ---- the item's last tile: V rows past its keys hold stale bytes; zero them (0 * NaN = NaN) ----
      if (wg == it.zfill_wg && j == it.n_all - 1) {
        const int kl = it.kend_all - kb;
        if (kl < T::KEYS) {
          const int gi = gt + u, vs = gi % kVSlots;
          pf_wait(sh, &sh.vfull[vs], (gi / kVSlots) & 1, p.err);
          const uint32_t sv = dev::smem_addr(smem + T::OFF_V + vs * T::KVTILE);
          for (int idx = r; idx < (T::KEYS - kl) * T::DH * 8; idx += 128) {
            const int kr = kl + idx / (T::DH * 8), rest = idx % (T::DH * 8);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sv + (rest >> 3) * (T::KEYS * 128) + kr * 128 +
                                                                            (rest & 7) * 16),
                         "r"(0)
                         : "memory");
          }
          dev::fence_proxy_async_smem();
          dev::mbar_arrive(sh.zfill);  // the other group's product of this tile waits for it
        }
      }
      dev::fence_proxy_async_smem();
      dev::tmem_wait_st();
      dev::tc_fence_before();
      dev::mbar_arrive(&sh.p_ready[wg]);
    }
    // ---- epilogue: O / l -> fp16, or for a split item the chunk handshake ----
    __half* dst = p.out + (tok * p.num_q_heads + (size_t)it.g * G + hq) * D;
    if (n > 0) {
      pf_wait(sh, &sh.pv_done[wg], (cw + n - 1) & 1, p.err);
      dev::tc_fence_after();
    }
    auto store_row = [&](int k, const float (&v)[32]) {  // 32 output columns of this row, fp16
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t h2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hh = __floats2half2_rn(v[c8 * 8 + 2 * e], v[c8 * 8 + 2 * e + 1]);
          h2[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        *reinterpret_cast<uint4*>(dst + 32 * k + 8 * c8) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
      }
    };
    if (!it.split) {
      if (n > 0) {
        const float il = 1.f / l;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          uint32_t o[32];
          dev::tmem_ld32(tl + T::SO + 32 * k, o);
          dev::tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * il;
          if (valid) store_row(k, v);
        }
      }
    } else {
      // The chunk that finishes first publishes its unnormalised (m, l, O); the other merges them in
      // chunk order (the result does not depend on which chunk finished first) and writes fp16.
      const size_t prow = (size_t)slot * (2 * kPrefillRows) + wg * kPrefillRows + r;
      // the partial O of this (slot, Q tile) is stored column by column, [D][128 rows]: a warp's 32 rows of one
      // column are 32 consecutive floats, so every store and load of the handshake is one coalesced line
      float* pcol = p.pf_o + ((size_t)slot * 2 + wg) * ((size_t)D * kPrefillRows) + r;
      const int2* sync = p.pf_sync + slot;
      if (threadIdx.x == 0) *sh.order = atomicAdd(const_cast<int*>(&sync->x), 1);
      dev::named_bar_sync(kBarEpi, T::SOFTMAX_THREADS);
      const int order = *sh.order;
      const float m_own = n > 0 ? m_ref : -INFINITY, l_own = n > 0 ? l : 0.f;
      if (order == 0) {
        p.pf_ml[prow] = make_float2(m_own, l_own);
        if (n > 0) {
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            uint32_t o[32];
            dev::tmem_ld32(tl + T::SO + 32 * k, o);
            dev::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) pcol[(size_t)(32 * k + e) * kPrefillRows] = __uint_as_float(o[e]);
          }
        }
        dev::named_bar_sync(kBarEpi, T::SOFTMAX_THREADS);  // every row published
        if (threadIdx.x == 0) {
          __threadfence();
          atomicExch(const_cast<int*>(&sync->y), 1);
        }
      } else {
        if (threadIdx.x == 0) {  // bounded wait for the other chunk's partial
          const uint64_t t0 = dev::globaltimer_ns();
          uint32_t polls = 0;
          while (atomicAdd(const_cast<int*>(&sync->y), 0) == 0) {
            if ((++polls & 255u) == 0 && polls > dev::kWaitMinPolls && (int64_t)(dev::globaltimer_ns() - t0) > dev::kWaitLimitNs) {
              *sh.abort = 1;
              dev::set_error(p.err, PKV_DEVERR_WAIT_TIMEOUT);
              break;
            }
          }
          __threadfence();
        }
        dev::named_bar_sync(kBarEpi, T::SOFTMAX_THREADS);
        const float2 mlo = __ldcg(p.pf_ml + prow);
        // chunk 0 first, whichever of the two this is
        const float m0 = it.chunk ? mlo.x : m_own, l0 = it.chunk ? mlo.y : l_own;
        const float m1 = it.chunk ? m_own : mlo.x, l1 = it.chunk ? l_own : mlo.y;
        const float M = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M), f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
        const float il = 1.f / (l0 * f0 + l1 * f1);
        const bool other_has = mlo.x != -INFINITY;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          uint32_t o[32];
          if (n > 0) {
            dev::tmem_ld32(tl + T::SO + 32 * k, o);
            dev::tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          float v[32], ot[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) ot[e] = other_has ? __ldcg(pcol + (size_t)(32 * k + e) * kPrefillRows) : 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float own = __uint_as_float(o[e]);
            const float a0 = it.chunk ? ot[e] : own, a1 = it.chunk ? own : ot[e];
            v[e] = (a0 * f0 + a1 * f1) * il;
          }
          if (valid) store_row(k, v);
        }
        dev::named_bar_sync(kBarEpi, T::SOFTMAX_THREADS);
        if (threadIdx.x == 0) *const_cast<int2*>(sync) = make_int2(0, 0);  // ready for the next launch
      }
    }
    if (n > 0) dev::tc_fence_before();
    cw += n;
    gt += it.te - it.tb;  // K/V tiles of this entry (ring position shared with the TMA and MMA warps)
  }
}

template <int D, int G>
__global__ void __launch_bounds__(PfTraits<D, G>::THREADS, 1) prefill_kernel(const __grid_constant__ PfParams p) {
  using T = PfTraits<D, G>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  Bars sh;
  sh.kfull = bars;
  sh.kfree = sh.kfull + kKSlots;
  sh.vfull = sh.kfree + kKSlots;
  sh.vfree = sh.vfull + kVSlots;
  sh.s_done = sh.vfree + kVSlots;
  sh.p_ready = sh.s_done + kWG;
  sh.pv_done = sh.p_ready + kWG;
  sh.zfill = sh.pv_done + kWG;
  sh.tmem_base = reinterpret_cast<uint32_t*>(smem + T::OFF_MISC);
  sh.item = reinterpret_cast<int4*>(smem + T::OFF_MISC + 16);
  sh.abort = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 32);
  sh.slot = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 36);
  sh.order = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 40);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKSlots; ++i) {
      dev::mbar_init(&sh.kfull[i], 1);
      dev::mbar_init(&sh.kfree[i], T::WG);  // one commit per MMA warp
    }
    for (int i = 0; i < kVSlots; ++i) {
      dev::mbar_init(&sh.vfull[i], 1);
      dev::mbar_init(&sh.vfree[i], T::WG);
    }
    for (int w = 0; w < kWG; ++w) {
      dev::mbar_init(&sh.s_done[w], 1);
      dev::mbar_init(&sh.p_ready[w], 128);
      dev::mbar_init(&sh.pv_done[w], 1);
    }
    dev::mbar_init(sh.zfill, 128);
    dev::fence_mbar_init();
    *sh.abort = 0;
  }
  if (warp == 0) {
    dev::tmem_alloc(sh.tmem_base, T::TMEM_COLS);
    dev::tmem_relinquish();
  }
  dev::tc_fence_before();
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const bool poisoned = __syncthreads_or(threadIdx.x == 0 && dev::pool_poisoned(p.err));
  dev::tc_fence_after();
  const int n_items = poisoned ? 0 : p.hdr->n_items;
  if (warp == T::MMA0) mma_warp<D, G, 0>(p, smem, sh, lane, n_items);
  else if (warp == T::MMA1) mma_warp<D, G, T::WG - 1>(p, smem, sh, lane, n_items);  // only with two groups
  else if (warp == T::TMA) tma_warp<D, G>(p, smem, sh, lane);
  else softmax_group<D, G>(p, smem, sh, warp >> 2, warp, lane);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  if (warp == 0) dev::tmem_dealloc(*sh.tmem_base, T::TMEM_COLS);
  // The last CTA out resets the item counter for the next launch on this plan.  No fence on either side (as
  // in the decode kernel): the CTA's claims were used before the barrier above, and the next launch reads
  // the counters only after its dependency wait, which sees every write of this grid.
  if (threadIdx.x == 0) {
    if (atomicAdd(&p.hdr->pdone, 1) == (int)gridDim.x - 1) {
      p.hdr->pwork = 0;
      p.hdr->pdone = 0;
    }
  }
}

template <int D, int G>
cudaError_t launch_t(const PfParams& p, int num_sms, int64_t max_items, cudaStream_t stream) {
  using T = PfTraits<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int64_t grid = num_sms;  // one CTA per SM (shared memory and tensor memory bound)
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  return launch_pdl(prefill_kernel<D, G>, dim3((unsigned)grid), dim3(T::THREADS), T::SMEM, stream, p);
}

template <int D>
cudaError_t launch_d(int group, const PfParams& p, int num_sms, int64_t max_items, cudaStream_t s) {
  switch (group) {
    case 1: return launch_t<D, 1>(p, num_sms, max_items, s);
    case 2: return launch_t<D, 2>(p, num_sms, max_items, s);
    case 4: return launch_t<D, 4>(p, num_sms, max_items, s);
    case 6: return launch_t<D, 6>(p, num_sms, max_items, s);
    case 8: return launch_t<D, 8>(p, num_sms, max_items, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) &&
         (group == 1 || group == 2 || group == 4 || group == 6 || group == 8);
}

int prefill_item_positions(int group, int head_dim) { return (head_dim == 256 ? 1 : kWG) * prefill_positions(group); }

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PfParams p;
  p.kv_map = *a.kv_map;
  p.q = static_cast<const __half*>(a.q);
  p.out = static_cast<__half*>(a.out);
  p.block_tables = a.block_tables;
  p.items = a.items;
  p.items_slot = a.items_slot;
  p.pf_sync = a.pf_sync;
  p.pf_ml = a.pf_ml;
  p.pf_o = a.pf_o;
  p.hdr = a.hdr;
  p.err = a.err;
  p.layer_row0_k = a.layer_row0_k;
  p.layer_row0_v = a.layer_row0_v;
  p.max_blocks = a.max_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.head_dim));
  const int group = a.num_q_heads / a.num_kv_heads;
  switch (a.head_dim) {
    case 64: return launch_d<64>(group, p, a.num_sms, a.max_items, stream);
    case 128: return launch_d<128>(group, p, a.num_sms, a.max_items, stream);
    case 256: return launch_d<256>(group, p, a.num_sms, a.max_items, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
