// Ragged paged GQA attention: per-pass plan, split-K decode partials, cross-split merge.
//
// What is computed ("Continuous Batching Is Not a Bigger Batch", sections "What the scheduler does on one
// step" and "Where the batch size actually comes from"): for every query token of every row, causal
// attention over that row's keys in the paged cache, query head h reading KV head h / G (grouped-query
// attention), scores scaled by 1/sqrt(d).  "Static batching" ("Ragged batches", "Bottleneck, and what
// follows") is why the keys are read from blocks in place, with no padding to the widest row.
//
// How (GB300 design, not from the pages):
//  * plan_kernel (once per pass): per packed query token, its row and its causal context length.
//  * decode_kernel: one CTA per (token, KV head, split of `split_blocks` blocks).  The CTA holds all G
//    query heads of the KV head, so each K/V block is read from HBM exactly once.  A producer warp
//    streams whole (block, KV head) runs of K and V into a shared-memory ring with 1-D bulk (TMA) copies
//    completing on mbarriers; four consumer warps each take every fourth block, compute scores with
//    packed fp32 FMAs, reduce across lanes with warp shuffles, and keep an online softmax (running max
//    and sum in the log2 domain) plus an fp32 accumulator.  The warps are combined through shared memory.
//    A token whose context fits one split writes fp16 output directly; otherwise the split writes an
//    unnormalised partial (m, l, o) to the workspace.
//  * merge_kernel: for tokens with more than one split, log-sum-exp combine of the partials -> fp16.
// The split count of a token depends only on its own context length, so results are bit-identical
// whatever else is in the batch and whatever the row order or physical block placement.
#include <cuda_fp16.h>

#include <cmath>
#include <string>

#include "pkv_internal.cuh"

namespace pkv {

constexpr int kBS = 16;

__host__ __device__ constexpr int next_pow2(int x) { return x <= 1 ? 1 : 2 * next_pow2((x + 1) / 2); }
__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int G>
struct DecodeTraits {
  static constexpr int NCW = 4;                  // consumer warps
  static constexpr int NTHREADS = (NCW + 1) * 32;  // + one producer warp
  static constexpr int DG = D / 16;              // lanes sharing one key row in the score phase (16 dims each)
  static constexpr int TPW = 32 / DG;            // key rows per warp step
  static constexpr int STEPS = kBS / TPW;        // warp steps per block
  static constexpr int DPL = D / 32;             // output dims per lane in the value phase
  static constexpr int RUN = kBS * D * 2;        // bytes of one (block, KV head) run of K (or V)
  static constexpr int NSTAGE = D == 256 ? 6 : 8;
  static constexpr int GP = next_pow2(G);        // heads padded to a power of two for the reduction
  static constexpr int R = GP > DG ? GP / DG : 1;    // heads a lane owns after the reduce-scatter
  static constexpr int REP = DG > GP ? DG / GP : 1;  // lanes holding the same head (replicas)
  static constexpr int RING = NSTAGE * 2 * RUN;
  static constexpr int OFF_P = RING;                                   // [NCW][kBS][GP] probabilities
  static constexpr int OFF_A = OFF_P + NCW * kBS * GP * 4;             // [NCW][GP] rescale factors
  static constexpr int OFF_M = OFF_A + NCW * GP * 4;                   // [NCW][GP] running max
  static constexpr int OFF_L = OFF_M + NCW * GP * 4;                   // [NCW][GP] running sum
  static constexpr int OFF_BAR = align_up(OFF_L + NCW * GP * 4, 8);
  static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8;
  static_assert(D % 16 == 0 && DG <= 32 && kBS % TPW == 0, "head_dim");
  static_assert(NCW * G * D * 4 <= RING, "combine staging must fit in the ring");
  static_assert(DPL % 2 == 0, "value phase works on float2 pairs");
};

struct DecodeParams {
  const __half* q;
  const __half* kpool;
  const __half* vpool;
  const int32_t* block_tables;
  const int32_t* tok_row;
  const int32_t* tok_ctx;
  __half* out;
  float* part_o;
  float2* part_ml;
  int32_t* err;
  int max_blocks;
  int num_q_heads;
  int num_kv_heads;
  int num_blocks;
  int split_blocks;
  int max_splits;
  float scale_log2;  // log2(e) / sqrt(head_dim)
};

// Reduce-scatter of GP values over the DG lanes of a key row (lane bits below DG): halving exchanges
// while more than one head remains per lane, then plain all-reduce.  Afterwards v[0 .. R-1] are the
// full sums of heads head_base(lane) + r.
template <int CNT, int M>
struct ReduceScatter {
  template <int N>
  static __device__ __forceinline__ void run(float (&v)[N], int lane) {
    if constexpr (M >= 1) {
      if constexpr (CNT > 1) {
        constexpr int H = CNT / 2;
        const bool up = (lane & M) != 0;
#pragma unroll
        for (int j = 0; j < H; ++j) {
          const float send = up ? v[j] : v[j + H];
          const float keep = up ? v[j + H] : v[j];
          v[j] = keep + __shfl_xor_sync(0xffffffffu, send, M);
        }
        ReduceScatter<H, M / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
        ReduceScatter<1, M / 2>::run(v, lane);
      }
    }
  }
  static __device__ __forceinline__ int head_base(int lane) {
    if constexpr (M >= 1 && CNT > 1) {
      constexpr int H = CNT / 2;
      return ((lane & M) ? H : 0) + ReduceScatter<H, M / 2>::head_base(lane);
    } else {
      return 0;
    }
  }
};

__device__ __forceinline__ void h8_to_f2(const uint4& raw, float2* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) f[e] = __half22float2(h[e]);
}

template <int D, int G>
__global__ void __launch_bounds__(DecodeTraits<D, G>::NTHREADS)
decode_kernel(const DecodeParams p) {
  using T = DecodeTraits<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::NSTAGE;

  dev::griddep_wait();
  dev::griddep_launch_dependents();

  const int t = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int ctx = __ldg(p.tok_ctx + t);
  if (ctx <= 0) return;  // token handled elsewhere or its row is invalid
  const int nblk = (ctx + kBS - 1) / kBS;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  if (s >= nsplit) return;
  const int first = s * p.split_blocks;
  const int nb = min(p.split_blocks, nblk - first);
  const int row = __ldg(p.tok_row + t);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < T::NSTAGE; ++i) {
      dev::mbar_init(&full[i], 1);
      dev::mbar_init(&empty[i], 1);
    }
    dev::fence_mbar_init();
  }
  // one CTA-uniform decision (a racing error-word update must not split the CTA)
  if (__syncthreads_or(threadIdx.x == 0 && dev::pool_poisoned(p.err))) return;

  if (warp == T::NCW) {
    // ---------------- producer warp: stream K/V runs of this split into the ring ----------------
    const int32_t* bt = p.block_tables + (int64_t)row * p.max_blocks + first;
    const size_t blk_stride = (size_t)p.num_kv_heads * kBS * D;
    const size_t head_off = (size_t)g * kBS * D;
    const uint64_t pol = dev::l2_policy_evict_first();
    bool ok = true;
    for (int base = 0; base < nb && ok; base += 32) {
      int blk = 0;
      if (base + lane < nb) {
        blk = __ldg(bt + base + lane);
        if (blk < 0 || blk >= p.num_blocks) {
          dev::set_error(p.err, PKV_DEVERR_BLOCK_RANGE);
          blk = 0;  // keep the copy in bounds; the output of this token is flagged as invalid
        }
      }
      const int cnt = min(32, nb - base);
      for (int k = 0; k < cnt; ++k) {
        const int b = __shfl_sync(0xffffffffu, blk, k);
        if (lane == 0 && ok) {
          const int idx = base + k;
          const int slot = idx % T::NSTAGE, round = idx / T::NSTAGE;
          if (round > 0 && !dev::mbar_wait(&empty[slot], (round - 1) & 1)) {
            dev::set_error(p.err, PKV_DEVERR_WAIT_TIMEOUT);
            ok = false;
          } else {
            unsigned char* dst = smem + slot * 2 * T::RUN;
            const size_t src = (size_t)b * blk_stride + head_off;
            dev::mbar_arrive_expect_tx(&full[slot], 2 * T::RUN);
            dev::bulk_g2s(dst, p.kpool + src, T::RUN, &full[slot], pol);
            dev::bulk_g2s(dst + T::RUN, p.vpool + src, T::RUN, &full[slot], pol);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int tq = lane / T::DG;  // key row within a warp step
  const int dg = lane % T::DG;  // 16-dim slice: dims [8 dg, 8 dg + 8) and [D/2 + 8 dg, D/2 + 8 dg + 8)
  using RS = ReduceScatter<T::GP, T::DG / 2>;
  const int hbase = RS::head_base(lane);
  const bool primary = (dg % T::REP) == 0;

  float2 qr[G][8];
  {
    const __half* qb = p.q + ((size_t)t * p.num_q_heads + (size_t)g * G) * D;
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(qb + j * D + (dg + c * T::DG) * 8);
        float2 f[4];
        h8_to_f2(raw, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) qr[j][c * 4 + e] = make_float2(f[e].x * p.scale_log2, f[e].y * p.scale_log2);
      }
    }
  }

  float m_run[T::R], l_run[T::R];
#pragma unroll
  for (int r = 0; r < T::R; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.f;
  }
  float2 o[G][T::DPL / 2];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int e = 0; e < T::DPL / 2; ++e) o[j][e] = make_float2(0.f, 0.f);

  float* Pw = reinterpret_cast<float*>(smem + T::OFF_P) + warp * kBS * T::GP;
  float* Aw = reinterpret_cast<float*>(smem + T::OFF_A) + warp * T::GP;
  bool timed_out = false;

  for (int i = warp; i < nb; i += T::NCW) {
    const int slot = i % T::NSTAGE, round = i / T::NSTAGE;
    if (!dev::mbar_wait(&full[slot], round & 1)) {
      if (lane == 0) dev::set_error(p.err, PKV_DEVERR_WAIT_TIMEOUT);
      timed_out = true;
      break;
    }
    const __half* Ks = reinterpret_cast<const __half*>(smem + slot * 2 * T::RUN);
    const __half* Vs = Ks + kBS * D;
    const int ntok = min(kBS, ctx - (first + i) * kBS);

    // scores (log2 domain) of this block's keys
    float sc[T::STEPS][T::R];
#pragma unroll
    for (int st = 0; st < T::STEPS; ++st) {
      const int tok = st * T::TPW + tq;
      float2 kf[8];
      h8_to_f2(*reinterpret_cast<const uint4*>(Ks + tok * D + dg * 8), kf);
      h8_to_f2(*reinterpret_cast<const uint4*>(Ks + tok * D + (dg + T::DG) * 8), kf + 4);
      float v[T::GP];
#pragma unroll
      for (int j = 0; j < T::GP; ++j) {
        if (j < G) {
          float2 a = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 8; ++e) a = __ffma2_rn(qr[j][e], kf[e], a);
          v[j] = a.x + a.y;
        } else {
          v[j] = 0.f;
        }
      }
      RS::run(v, lane);
#pragma unroll
      for (int r = 0; r < T::R; ++r) sc[st][r] = tok < ntok ? v[r] : -INFINITY;
    }

    // online softmax update per head
#pragma unroll
    for (int r = 0; r < T::R; ++r) {
      float bm = sc[0][r];
#pragma unroll
      for (int st = 1; st < T::STEPS; ++st) bm = fmaxf(bm, sc[st][r]);
#pragma unroll
      for (int m = T::DG; m < 32; m <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, m));
      const float mn = fmaxf(m_run[r], bm);
      const float alpha = exp2f(m_run[r] - mn);
      float ls = 0.f;
#pragma unroll
      for (int st = 0; st < T::STEPS; ++st) {
        const float pv = exp2f(sc[st][r] - mn);
        sc[st][r] = pv;
        ls += pv;
      }
      l_run[r] = l_run[r] * alpha + ls;
      m_run[r] = mn;
      const int h = hbase + r;
      if (primary && h < G) {
#pragma unroll
        for (int st = 0; st < T::STEPS; ++st) Pw[(st * T::TPW + tq) * T::GP + h] = sc[st][r];
        if (tq == 0) Aw[h] = alpha;
      }
    }
    __syncwarp();

    // value accumulation: lane owns dims [lane * DPL, lane * DPL + DPL)
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float a = Aw[j];
#pragma unroll
      for (int e = 0; e < T::DPL / 2; ++e) o[j][e] = __fmul2_rn(o[j][e], make_float2(a, a));
    }
#pragma unroll 4
    for (int tk = 0; tk < ntok; ++tk) {
      float2 vf[T::DPL / 2];
      const __half2* vrow = reinterpret_cast<const __half2*>(Vs + tk * D + lane * T::DPL);
#pragma unroll
      for (int e = 0; e < T::DPL / 2; ++e) vf[e] = __half22float2(vrow[e]);
      const float* prow = Pw + tk * T::GP;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float pj = prow[j];
        const float2 pp = make_float2(pj, pj);
#pragma unroll
        for (int e = 0; e < T::DPL / 2; ++e) o[j][e] = __ffma2_rn(pp, vf[e], o[j][e]);
      }
    }
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(&empty[slot]);
  }
  (void)timed_out;

  // ---------------- combine the four warps ----------------
  float* Mw = reinterpret_cast<float*>(smem + T::OFF_M);
  float* Lw = reinterpret_cast<float*>(smem + T::OFF_L);
#pragma unroll
  for (int r = 0; r < T::R; ++r) {
    float l = l_run[r];
#pragma unroll
    for (int m = T::DG; m < 32; m <<= 1) l += __shfl_xor_sync(0xffffffffu, l, m);
    const int h = hbase + r;
    if (primary && tq == 0 && h < G) {
      Mw[warp * T::GP + h] = m_run[r];
      Lw[warp * T::GP + h] = l;
    }
  }
  dev::named_bar_sync(1, T::NCW * 32);  // every consumer is done with the ring
  float* Ow = reinterpret_cast<float*>(smem);  // [NCW][G][D], reusing the ring
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int e = 0; e < T::DPL / 2; ++e)
      *reinterpret_cast<float2*>(Ow + (warp * G + j) * D + lane * T::DPL + 2 * e) = o[j][e];
  dev::named_bar_sync(1, T::NCW * 32);

  for (int e = threadIdx.x; e < G * D; e += T::NCW * 32) {
    const int j = e / D, dim = e - j * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < T::NCW; ++w) M = fmaxf(M, Mw[w * T::GP + j]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < T::NCW; ++w) {
      const float f = exp2f(Mw[w * T::GP + j] - M);
      L += Lw[w * T::GP + j] * f;
      O += Ow[(w * G + j) * D + dim] * f;
    }
    const int h = g * G + j;
    if (nsplit == 1) {
      p.out[((size_t)t * p.num_q_heads + h) * D + dim] = __float2half_rn(O / L);
    } else {
      const size_t pi = ((size_t)t * p.max_splits + s) * p.num_q_heads + h;
      p.part_o[pi * D + dim] = O;
      if (dim == 0) p.part_ml[pi] = make_float2(M, L);
    }
  }
}

struct MergeParams {
  const float* part_o;
  const float2* part_ml;
  const int32_t* tok_ctx;
  __half* out;
  int num_q_heads;
  int split_blocks;
  int max_splits;
};

// One CTA per (token, query head) of a token with more than one split.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int t = blockIdx.x, h = blockIdx.y;
  const int ctx = __ldg(p.tok_ctx + t);
  if (ctx <= 0) return;
  const int nblk = (ctx + kBS - 1) / kBS;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  if (nsplit <= 1) return;
  const size_t base = (size_t)t * p.max_splits * p.num_q_heads + h;
  const float2* ml = p.part_ml + base;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[(size_t)s * p.num_q_heads].x);
  for (int dim = threadIdx.x; dim < D; dim += 128) {
    float L = 0.f, O = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float2 v = ml[(size_t)s * p.num_q_heads];
      const float f = exp2f(v.x - M);
      L += v.y * f;
      O += p.part_o[(base + (size_t)s * p.num_q_heads) * D + dim] * f;
    }
    p.out[((size_t)t * p.num_q_heads + h) * D + dim] = __float2half_rn(O / L);
  }
}

// Per packed token: its row and causal context (keys it sees); 0 marks a token no kernel should touch.
// Also validates the per-row metadata, recording violations in the device error word.
__global__ void __launch_bounds__(256) plan_kernel(const int32_t* __restrict__ context_lens,
                                                   const int32_t* __restrict__ qsl, int num_seqs, int num_tokens,
                                                   int max_ctx, int32_t* __restrict__ tok_row,
                                                   int32_t* __restrict__ tok_ctx, int32_t* err) {
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int n = max(num_seqs, num_tokens);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < num_seqs) {
      const int q0 = __ldg(qsl + i), q1 = __ldg(qsl + i + 1), ctx = __ldg(context_lens + i);
      if (q1 < q0 || (i == 0 && q0 != 0) || (i == num_seqs - 1 && q1 != num_tokens))
        dev::set_error(err, PKV_DEVERR_QSL);
      if (q1 - q0 < 1 || ctx < q1 - q0 || ctx > max_ctx) dev::set_error(err, PKV_DEVERR_ROW_META);
    }
    if (i < num_tokens) {
      const int b = dev::row_of_token(qsl, num_seqs, i);
      const int q0 = __ldg(qsl + b), q1 = __ldg(qsl + b + 1), ctx = __ldg(context_lens + b);
      const int q_len = q1 - q0;
      int c = 0;
      if (i >= q0 && i < q1 && q_len >= 1 && ctx >= q_len && ctx <= max_ctx) c = ctx - q_len + (i - q0) + 1;
      tok_row[i] = b;
      tok_ctx[i] = c;
    }
  }
}

// ---------------------------------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------------------------------
struct WsLayout {
  size_t tok_row, tok_ctx, part_ml, part_o, total;
  int max_splits;
};

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

static WsLayout ws_layout(const pkv_config& c, int num_tokens, int max_blocks) {
  WsLayout w;
  w.max_splits = (max_blocks + c.split_blocks - 1) / c.split_blocks;
  size_t off = 0;
  w.tok_row = off;
  off += up256((size_t)num_tokens * 4);
  w.tok_ctx = off;
  off += up256((size_t)num_tokens * 4);
  const size_t parts = w.max_splits > 1 ? (size_t)num_tokens * w.max_splits * c.num_q_heads : 0;
  w.part_ml = off;
  off += up256(parts * sizeof(float2));
  w.part_o = off;
  off += up256(parts * c.head_dim * sizeof(float));
  w.total = off;
  return w;
}

template <int D, int G>
static cudaError_t launch_decode(const DecodeParams& p, int num_tokens, int num_kv_heads, int max_splits,
                                 cudaStream_t stream) {
  using T = DecodeTraits<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(decode_kernel<D, G>, dim3(num_tokens, num_kv_heads, max_splits), dim3(T::NTHREADS), T::SMEM,
                    stream, p);
}

template <int D>
static cudaError_t launch_decode_g(int group, const DecodeParams& p, int num_tokens, int num_kv_heads,
                                   int max_splits, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode<D, 1>(p, num_tokens, num_kv_heads, max_splits, stream);
    case 2: return launch_decode<D, 2>(p, num_tokens, num_kv_heads, max_splits, stream);
    case 4: return launch_decode<D, 4>(p, num_tokens, num_kv_heads, max_splits, stream);
    case 6: return launch_decode<D, 6>(p, num_tokens, num_kv_heads, max_splits, stream);
    case 8: return launch_decode<D, 8>(p, num_tokens, num_kv_heads, max_splits, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_attention_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_tokens,
                                                int32_t max_blocks_per_seq) {
  if (!pool || num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 1) return 0;
  return ws_layout(pool->cfg, num_tokens, max_blocks_per_seq).total;
}

static pkv_status check_common(pkv_pool* pool, const int32_t* context_lens, const int32_t* qsl, int32_t num_seqs,
                               int32_t num_tokens, int32_t max_blocks, void* workspace, size_t ws_bytes) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (num_seqs < 0 || num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be >= 0");
  if (num_tokens > 0 && num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "tokens without rows");
  if (num_seqs > num_tokens) return fail(PKV_ERR_INVALID_ARG, "every row needs at least one query token");
  if (max_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  if (num_tokens > 0 && (!context_lens || !qsl || !workspace))
    return fail(PKV_ERR_INVALID_ARG, "metadata and workspace pointers must be non-NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const WsLayout w = ws_layout(pool->cfg, num_tokens, max_blocks);
  if (w.max_splits > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many splits per row; raise split_blocks");
  if (ws_bytes < w.total)
    return fail(PKV_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(w.total) + " bytes");
  return PKV_OK;
}

extern "C" pkv_status pkv_attention_plan(pkv_pool* pool, const int32_t* context_lens, const int32_t* query_start_loc,
                                         int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq,
                               workspace, workspace_bytes);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  pool->plan = PlanKey{workspace, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq};
  if (num_tokens == 0) return PKV_OK;
  const WsLayout w = ws_layout(pool->cfg, num_tokens, max_blocks_per_seq);
  char* ws = static_cast<char*>(workspace);
  const int n = num_seqs > num_tokens ? num_seqs : num_tokens;
  int blocks = (n + 255) / 256;
  if (blocks > pool->num_sms * 4) blocks = pool->num_sms * 4;
  cudaError_t e = launch_pdl(plan_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, context_lens,
                             query_start_loc, (int)num_seqs, (int)num_tokens, (int)(max_blocks_per_seq * kBS),
                             reinterpret_cast<int32_t*>(ws + w.tok_row), reinterpret_cast<int32_t*>(ws + w.tok_ctx),
                             pool->dev_error);
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
  pkv_status st = check_common(pool, context_lens, query_start_loc, num_seqs, num_tokens, max_blocks_per_seq,
                               workspace, workspace_bytes);
  if (st != PKV_OK) return st;
  pool->last_launches = 0;
  const pkv_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_tokens == 0) return PKV_OK;
  if (!q || !out || !block_tables) return fail(PKV_ERR_INVALID_ARG, "q, out and block_tables must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (q == out) return fail(PKV_ERR_INVALID_ARG, "out may not alias q");
  const PlanKey& k = pool->plan;
  if (k.workspace != workspace || k.context_lens != context_lens || k.query_start_loc != query_start_loc ||
      k.num_seqs != num_seqs || k.num_tokens != num_tokens || k.max_blocks_per_seq != max_blocks_per_seq)
    return fail(PKV_ERR_INVALID_ARG, "no matching plan: call pkv_attention_plan for this workspace and metadata");

  const WsLayout w = ws_layout(c, num_tokens, max_blocks_per_seq);
  char* ws = static_cast<char*>(workspace);
  DecodeParams p;
  p.q = static_cast<const __half*>(q);
  p.kpool = static_cast<const __half*>(pkv_pool_layer_ptr(pool, layer, 0));
  p.vpool = static_cast<const __half*>(pkv_pool_layer_ptr(pool, layer, 1));
  p.block_tables = block_tables;
  p.tok_row = reinterpret_cast<const int32_t*>(ws + w.tok_row);
  p.tok_ctx = reinterpret_cast<const int32_t*>(ws + w.tok_ctx);
  p.out = static_cast<__half*>(out);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  p.err = pool->dev_error;
  p.max_blocks = max_blocks_per_seq;
  p.num_q_heads = c.num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.num_blocks = c.num_blocks;
  p.split_blocks = c.split_blocks;
  p.max_splits = w.max_splits;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));

  const int group = c.num_q_heads / c.num_kv_heads;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  switch (c.head_dim) {
    case 64: e = launch_decode_g<64>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    case 128: e = launch_decode_g<128>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    case 256: e = launch_decode_g<256>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    default: return fail(PKV_ERR_UNSUPPORTED, "head_dim");
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  pool->last_launches = 1;
  if (w.max_splits > 1) {
    MergeParams m{p.part_o, p.part_ml, p.tok_ctx, p.out, c.num_q_heads, c.split_blocks, w.max_splits};
    switch (c.head_dim) {
      case 64: e = launch_pdl(merge_kernel<64>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
      case 128: e = launch_pdl(merge_kernel<128>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
      default: e = launch_pdl(merge_kernel<256>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    pool->last_launches = 2;
  }
  return PKV_OK;
}

// ---------------------------------------------------------------------------------------------------
// Allocation-free variant of the attention call.
//
// Some callers cannot hand the library a workspace: an engine that has already reserved every byte of
// device memory for its own pools, or a caller that may not issue cudaMalloc (which can synchronise the
// whole device) while a pass is in flight.  For them the split-K scratch -- the per-token row/context
// table and the partial (m, l, o) results -- lives in one fixed array compiled into this library.
// Each device that loads the library holds the array until the process exits.
// ---------------------------------------------------------------------------------------------------
#include <mutex>

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
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  pool->last_launches = 0;
  const pkv_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_seqs < 0 || num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be >= 0");
  if (num_tokens > 0 && num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "tokens without rows");
  if (num_seqs > num_tokens) return fail(PKV_ERR_INVALID_ARG, "every row needs at least one query token");
  if (max_blocks_per_seq < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  if (num_tokens == 0) return PKV_OK;
  if (!q || !out || !block_tables || !context_lens || !query_start_loc)
    return fail(PKV_ERR_INVALID_ARG, "q, out and metadata pointers must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (q == out) return fail(PKV_ERR_INVALID_ARG, "out may not alias q");
  const WsLayout w = ws_layout(c, num_tokens, max_blocks_per_seq);
  if (w.max_splits > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many splits per row; raise split_blocks");
  if (w.total > kNoAllocScratchBytes)
    return fail(PKV_ERR_OUT_OF_RANGE, "pass needs " + std::to_string(w.total) + " bytes of scratch; the built-in "
                "array holds " + std::to_string(kNoAllocScratchBytes) + " (use pkv_attention with a workspace)");
  int device = -1;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (device != pool->device) return fail(PKV_ERR_INVALID_ARG, "the pool's device must be the current device");
  void* scratch = noalloc_scratch_ptr(device, &e);
  if (!scratch) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch array");

  char* ws = static_cast<char*>(scratch);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* tok_row = reinterpret_cast<int32_t*>(ws + w.tok_row);
  int32_t* tok_ctx = reinterpret_cast<int32_t*>(ws + w.tok_ctx);
  // Nothing in the scratch needs to start at zero: the plan rewrites the token table for every token,
  // and every partial the merge reads is written by the decode kernel of the same call.
  const int n = num_seqs > num_tokens ? num_seqs : num_tokens;
  int blocks = (n + 255) / 256;
  if (blocks > pool->num_sms * 4) blocks = pool->num_sms * 4;
  e = launch_pdl(plan_kernel, dim3(blocks), dim3(256), 0, s, context_lens, query_start_loc, (int)num_seqs,
                 (int)num_tokens, (int)(max_blocks_per_seq * kBS), tok_row, tok_ctx, pool->dev_error);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");

  DecodeParams p;
  p.q = static_cast<const __half*>(q);
  p.kpool = static_cast<const __half*>(pkv_pool_layer_ptr(pool, layer, 0));
  p.vpool = static_cast<const __half*>(pkv_pool_layer_ptr(pool, layer, 1));
  p.block_tables = block_tables;
  p.tok_row = tok_row;
  p.tok_ctx = tok_ctx;
  p.out = static_cast<__half*>(out);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  p.err = pool->dev_error;
  p.max_blocks = max_blocks_per_seq;
  p.num_q_heads = c.num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.num_blocks = c.num_blocks;
  p.split_blocks = c.split_blocks;
  p.max_splits = w.max_splits;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  const int group = c.num_q_heads / c.num_kv_heads;
  switch (c.head_dim) {
    case 64: e = launch_decode_g<64>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    case 128: e = launch_decode_g<128>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    case 256: e = launch_decode_g<256>(group, p, num_tokens, c.num_kv_heads, w.max_splits, s); break;
    default: return fail(PKV_ERR_UNSUPPORTED, "head_dim");
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  pool->last_launches = 2;
  if (w.max_splits > 1) {
    MergeParams m{p.part_o, p.part_ml, p.tok_ctx, p.out, c.num_q_heads, c.split_blocks, w.max_splits};
    switch (c.head_dim) {
      case 64: e = launch_pdl(merge_kernel<64>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
      case 128: e = launch_pdl(merge_kernel<128>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
      default: e = launch_pdl(merge_kernel<256>, dim3(num_tokens, c.num_q_heads), dim3(128), 0, s, m); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    pool->last_launches = 3;
  }
  return PKV_OK;
}
