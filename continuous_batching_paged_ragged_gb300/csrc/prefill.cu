// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// What is computed ("Continuous Batching Is Not a Bigger Batch", section "What the scheduler does on one
// step": a prompt is consumed in chunks under the per-pass token budget): for each new token of a row
// with many new tokens, causal attention over the row's keys in the paged cache -- query i of a chunk of
// q_len on top of ctx - q_len cached tokens sees keys 0 .. ctx - q_len + i -- for every query head, the
// head h reading KV head h / G, scores scaled by 1/sqrt(d), fp32 softmax, fp16 output.
//
// How (GB300 design):
//  * Work item = one KV head and P = 128 / G consecutive query positions of one row.  Its G query heads
//    are packed into the 128 MMA rows (row r = position r / G, head r % G), so every K/V tile is read
//    once for all heads of the group and the causal diagonal wastes at most P keys per tile.
//  * Persistent CTAs of 5 warps.  Warp 4 (control) streams K/V tiles of 128 keys from the paged pool
//    with 2-D TMA copies (128-byte swizzle) into a 2-stage ring and issues, from one thread, the MMAs
//    S = Q K^T (M 128, N 128, K d) and O += P V (M 128, N d, K 128) with fp32 accumulators in tensor
//    memory.  Warps 0-3 (softmax) own one S row each (TMEM lane = thread): they load S with tcgen05.ld,
//    apply the causal mask and an online softmax in the log2 domain, and write P as fp16 into a swizzled
//    shared-memory tile that the next MMA reads.  The running max is lazy: O (in TMEM) and the running
//    sum are rescaled only when a row's max grows by more than 8 (a factor 256), which keeps P <= 256
//    and the arithmetic exact up to rounding.
//  * Items are taken longest first (the plan sorts them by K/V tile count) from a global counter.
#include <cuda_fp16.h>

#include <cmath>

#include "attn_common.cuh"

namespace pkv {

namespace {

constexpr int kStages = 2;
constexpr int kThreads = 160;          // 4 softmax warps + 1 control warp
constexpr int kBarItem = 1, kBarQ = 2, kBarP = 3;  // named barriers (0 is __syncthreads)
constexpr float kRescaleLog2 = 8.f;    // lazy rescale threshold (log2 units)

template <int D, int G>
struct PfTraits {
  static constexpr int DH = D / 64;                 // 64-wide column halves of a row (128-byte swizzle atoms)
  static constexpr int P = prefill_positions(G);    // query positions per item
  static constexpr int TILE = DH * 128 * 128;       // bytes of a 128-row x D fp16 tile (Q, K or V)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + TILE;       // stage s: K at OFF_KV + 2 s TILE, V after it
  static constexpr int OFF_P = OFF_KV + kStages * 2 * TILE;  // P: 128 rows x 128 keys fp16 (32 KB)
  static constexpr int OFF_BAR = OFF_P + 2 * 128 * 128;      // kfull[2], vfull[2], s_done, pv_done
  static constexpr int OFF_MISC = OFF_BAR + 64;              // TMEM base, item record, abort flag
  static constexpr int SMEM = OFF_MISC + 64 + 1024;          // + slack to align to 1024 bytes
  static constexpr uint32_t TMEM_COLS = 256;                 // S: columns 0..127, O: 128..128+D-1
  static constexpr uint32_t IDESC_S = dev::umma_idesc_f16(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = dev::umma_idesc_f16(128, D, false, true);
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(128 + D <= (int)TMEM_COLS, "TMEM columns");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct PfParams {
  CUtensorMap kv_map;
  const __half* q;
  __half* out;
  const int32_t* block_tables;
  const int4* items;
  WsHeader* hdr;
  int32_t* err;
  int layer_row0_k, layer_row0_v;
  int max_blocks, num_q_heads, num_kv_heads, num_blocks;
  float scale_log2;
};

struct Shared {
  uint64_t* kfull;
  uint64_t* vfull;
  uint64_t* s_done;
  uint64_t* pv_done;
  uint32_t* tmem_base;
  int4* item;
  volatile int* abort;
};

// Bounded wait that, once any wait of the CTA has given up, no longer waits at all: every thread then
// runs through the remaining (bounded) loop with garbage and the CTA stays in step at its barriers.
__device__ __forceinline__ void pf_wait(const Shared& sh, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*sh.abort) return;
  if (!dev::mbar_wait(bar, parity)) {
    *sh.abort = 1;
    dev::set_error(err, PKV_DEVERR_WAIT_TIMEOUT);
  }
}

// Byte offset of 16-byte chunk c (8 fp16) of row r in a 128-row tile stored as 64-column halves with the
// 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---- control warp: TMA producer and MMA issuer ----------------------------------------------------
template <int D, int G>
__device__ void control_warp(const PfParams& p, unsigned char* smem, const Shared& sh, int lane, int n_items) {
  using T = PfTraits<D, G>;
  const uint32_t sbase = dev::smem_addr(smem);
  const uint32_t tS = *sh.tmem_base, tO = tS + 128;
  const uint64_t pol = dev::l2_policy_evict_last();
  int gidx = 0;  // CTA-wide index of the next K/V tile (ring stage gidx % 2, barrier phases)
  bool first = true;
  while (true) {
    int4 rec = make_int4(-1, 0, 0, 0);
    if (lane == 0) {
      const int idx = first ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&p.hdr->pwork, 1);
      if (idx < n_items) rec = __ldg(p.items + idx);
      *sh.item = rec;
    }
    first = false;
    rec.x = __shfl_sync(0xffffffffu, rec.x, 0);
    rec.y = __shfl_sync(0xffffffffu, rec.y, 0);
    rec.w = __shfl_sync(0xffffffffu, rec.w, 0);
    __syncwarp();
    dev::named_bar_arrive(kBarItem, kThreads);
    if (rec.x < 0) break;
    const int row = rec.x, g = rec.y & 0xFFFF, npos = rec.y >> 16;
    const int kend = rec.w + npos;                    // keys the item's last position sees
    const int n = (kend + kPrefillKeys - 1) / kPrefillKeys;
    const int nblk = (kend + kBS - 1) / kBS;
    const int32_t* bt = p.block_tables + (int64_t)row * p.max_blocks;

    auto issue_tile = [&](int j, int gi) {
      const int stage = gi % kStages;
      const int nb = min(8, nblk - j * 8);
      int id = 0;
      if (lane < nb) {
        id = __ldg(bt + j * 8 + lane);
        if (id < 0 || id >= p.num_blocks) {
          dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          id = 0;
        }
      }
      unsigned char* sk = smem + T::OFF_KV + stage * 2 * T::TILE;
      unsigned char* sv = sk + T::TILE;
      if (lane == 0) {
        dev::mbar_arrive_expect_tx(&sh.kfull[stage], (uint32_t)(nb * T::DH * 2048));
        dev::mbar_arrive_expect_tx(&sh.vfull[stage], (uint32_t)(nb * T::DH * 2048));
      }
      for (int i = 0; i < nb; ++i) {
        const int bid = __shfl_sync(0xffffffffu, id, i);
        if (lane == 0) {
          const int rk = p.layer_row0_k + (bid * p.num_kv_heads + g) * kBS;
          const int rv = p.layer_row0_v + (bid * p.num_kv_heads + g) * kBS;
#pragma unroll
          for (int h = 0; h < T::DH; ++h) {
            dev::tma_load_2d(sk + h * 16384 + i * 2048, &p.kv_map, h * 64, rk, &sh.kfull[stage], pol);
            dev::tma_load_2d(sv + h * 16384 + i * 2048, &p.kv_map, h * 64, rv, &sh.vfull[stage], pol);
          }
        }
      }
    };
    auto issue_s = [&](int gi) {  // S = Q K^T into TMEM columns 0..127
      const int stage = gi % kStages;
      const uint32_t sq = sbase + T::OFF_Q, sk = sbase + T::OFF_KV + stage * 2 * T::TILE;
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          dev::umma_f16_ss(tS, dev::umma_desc_sw128(sq + off, 16, 1024), dev::umma_desc_sw128(sk + off, 16, 1024),
                           T::IDESC_S, kk > 0);
        }
        dev::umma_commit(sh.s_done);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int gi, bool acc) {  // O (+)= P V into TMEM columns 128..128+D-1
      const int stage = gi % kStages;
      const uint32_t sp = sbase + T::OFF_P, sv = sbase + T::OFF_KV + stage * 2 * T::TILE + T::TILE;
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kPrefillKeys / 16; ++kk) {
          const uint32_t offp = (kk >> 2) * 16384 + (kk & 3) * 32;
          dev::umma_f16_ss(tO, dev::umma_desc_sw128(sp + offp, 16, 1024),
                           dev::umma_desc_sw128(sv + kk * 2048, 16384, 1024), T::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
        }
        dev::umma_commit(sh.pv_done);
      }
      __syncwarp();
    };

    // the ring's stages are free once the previous item's last P V has completed
    if (gidx > 0) pf_wait(sh, sh.pv_done, (gidx - 1) & 1, p.err);
    issue_tile(0, gidx);
    if (n > 1) issue_tile(1, gidx + 1);
    dev::named_bar_sync(kBarQ, kThreads);  // Q is in shared memory
    dev::tc_fence_after();
    pf_wait(sh, &sh.kfull[gidx % kStages], (gidx / kStages) & 1, p.err);
    issue_s(gidx);
    for (int j = 0; j < n; ++j) {
      const int gi = gidx + j;
      dev::named_bar_sync(kBarP, kThreads);  // P(j) written, O rescaled, S(j) read
      dev::tc_fence_after();
      pf_wait(sh, &sh.vfull[gi % kStages], (gi / kStages) & 1, p.err);
      issue_pv(gi, j > 0);
      if (j + 1 < n) {
        pf_wait(sh, &sh.kfull[(gi + 1) % kStages], ((gi + 1) / kStages) & 1, p.err);
        issue_s(gi + 1);
      }
      if (j + 2 < n) {  // tile j's stage is free once P(j) V(j) has completed
        pf_wait(sh, sh.pv_done, gi & 1, p.err);
        issue_tile(j + 2, gi + 2);
      }
    }
    gidx += n;
  }
  // leave no copy in flight: every issued tile was consumed by an MMA the softmax warps waited for
}

// ---- softmax warps: one S / O row per thread ------------------------------------------------------
template <int D, int G>
__device__ void softmax_warps(const PfParams& p, unsigned char* smem, const Shared& sh, int warp, int lane) {
  using T = PfTraits<D, G>;
  const int r = warp * 32 + lane;  // this thread's tile row and TMEM lane
  const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = *sh.tmem_base + lane_addr, tO = tS + 128;
  unsigned char* sQ = smem + T::OFF_Q;
  unsigned char* sP = smem + T::OFF_P;
  const uint32_t sQa = dev::smem_addr(sQ), sPa = dev::smem_addr(sP);
  int gidx = 0;
  while (true) {
    dev::named_bar_sync(kBarItem, kThreads);
    const volatile int* vi = reinterpret_cast<volatile int*>(sh.item);
    const int4 rec = make_int4(vi[0], vi[1], vi[2], vi[3]);
    if (rec.x < 0) break;
    const int g = rec.y & 0xFFFF, npos = rec.y >> 16, t0 = rec.z, w = rec.w;
    const int kend = w + npos;
    const int n = (kend + kPrefillKeys - 1) / kPrefillKeys;
    const int pos = r / G, hq = r % G;
    const bool valid = r < T::P * G && pos < npos;
    const int lim = valid ? w + pos : 0;  // last key this row sees (a padding row sees key 0 only)

    // ---- Q tile: row r = (position, head), 128-byte swizzle ----
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)(t0 + pos) * p.num_q_heads + (size_t)g * G + hq) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sQa + tile_off(r, c)), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      dev::fence_proxy_async_smem();
      dev::named_bar_arrive(kBarQ, kThreads);
    }

    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j) {
      const int gi = gidx + j;
      pf_wait(sh, sh.s_done, gi & 1, p.err);
      dev::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int k = 0; k < 4; ++k) dev::tmem_ld32(tS + 32 * k, s[k]);
      dev::tmem_wait_ld();
      // ---- scale to the log2 domain, causal mask, row max ----
      const int kb = j * kPrefillKeys;
      const bool full = kb + kPrefillKeys - 1 <= lim;
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x = __uint_as_float(s[k][c]) * p.scale_log2;
          if (!full && kb + 32 * k + c > lim) x = -INFINITY;
          s[k][c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      // ---- lazy rescale of the running state ----
      float alpha = 1.f;
      if (j == 0) {
        m_ref = mx;
      } else {
        pf_wait(sh, sh.pv_done, (gi - 1) & 1, p.err);  // P(j-1) V(j-1) done: P tile free, O settled
        dev::tc_fence_after();
        const bool need = mx > m_ref + kRescaleLog2;
        if (need) alpha = exp2f(m_ref - mx);
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            uint32_t o[32];
            dev::tmem_ld32(tO + 32 * k, o);
            dev::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            dev::tmem_st32(tO + 32 * k, o);
          }
          dev::tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_ref = mx;
        }
      }
      // ---- P = exp2(s - m_ref) as fp16 into the swizzled P tile (row r, keys contiguous) ----
      float sum = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < kPrefillKeys / 8; ++c8) {
        uint32_t h2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c8 * 8 + 2 * e;
          const float p0 = exp2f(__uint_as_float(s[c >> 5][c & 31]) - m_ref);
          const float p1 = exp2f(__uint_as_float(s[(c + 1) >> 5][(c + 1) & 31]) - m_ref);
          sum += p0 + p1;
          const __half2 hh = __floats2half2_rn(p0, p1);
          h2[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sPa + tile_off(r, c8)), "r"(h2[0]), "r"(h2[1]),
                     "r"(h2[2]), "r"(h2[3])
                     : "memory");
      }
      l += sum;
      // ---- last tile: V rows past the item's keys hold stale bytes; zero them (0 * NaN would poison O) ----
      const int kl = kend - kb;
      if (j == n - 1 && kl < kPrefillKeys) {
        const int stage = gi % kStages;
        pf_wait(sh, &sh.vfull[stage], (gi / kStages) & 1, p.err);
        const uint32_t sv = dev::smem_addr(smem + T::OFF_KV + stage * 2 * T::TILE + T::TILE);
        for (int idx = r; idx < (kPrefillKeys - kl) * T::DH * 8; idx += 128) {
          const int kr = kl + idx / (T::DH * 8), rest = idx % (T::DH * 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sv + (rest >> 3) * 16384 + kr * 128 +
                                                                          (rest & 7) * 16),
                       "r"(0)
                       : "memory");
        }
      }
      dev::fence_proxy_async_smem();
      dev::tc_fence_before();
      dev::named_bar_arrive(kBarP, kThreads);
    }
    // ---- epilogue: O / l -> fp16 ----
    const int gl = gidx + n - 1;
    pf_wait(sh, sh.pv_done, gl & 1, p.err);
    dev::tc_fence_after();
    const float il = 1.f / l;
    __half* dst = p.out + ((size_t)(t0 + pos) * p.num_q_heads + (size_t)g * G + hq) * D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      uint32_t o[32];
      dev::tmem_ld32(tO + 32 * k, o);
      dev::tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t h2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(o[c8 * 8 + 2 * e]) * il,
                                                 __uint_as_float(o[c8 * 8 + 2 * e + 1]) * il);
            h2[e] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          *reinterpret_cast<uint4*>(dst + 32 * k + 8 * c8) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
        }
      }
    }
    dev::tc_fence_before();
    gidx += n;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PfParams p) {
  using T = PfTraits<D, G>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared sh;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  sh.kfull = bars;
  sh.vfull = bars + 2;
  sh.s_done = bars + 4;
  sh.pv_done = bars + 5;
  sh.tmem_base = reinterpret_cast<uint32_t*>(smem + T::OFF_MISC);
  sh.item = reinterpret_cast<int4*>(smem + T::OFF_MISC + 16);
  sh.abort = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 6; ++i) dev::mbar_init(&bars[i], 1);
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
  if (warp == 4) control_warp<D, G>(p, smem, sh, lane, n_items);
  else softmax_warps<D, G>(p, smem, sh, warp, lane);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  if (warp == 0) dev::tmem_dealloc(*sh.tmem_base, T::TMEM_COLS);
  // the last CTA out resets the item counter for the next launch on this plan
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.hdr->pdone, 1) == (int)gridDim.x - 1) {
      p.hdr->pwork = 0;
      p.hdr->pdone = 0;
      __threadfence();
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
  return launch_pdl(prefill_kernel<D, G>, dim3((unsigned)grid), dim3(kThreads), T::SMEM, stream, p);
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
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 6 || group == 8);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PfParams p;
  p.kv_map = *a.kv_map;
  p.q = static_cast<const __half*>(a.q);
  p.out = static_cast<__half*>(a.out);
  p.block_tables = a.block_tables;
  p.items = a.items;
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
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
