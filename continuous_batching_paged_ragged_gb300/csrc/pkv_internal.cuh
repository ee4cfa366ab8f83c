// Internal helpers shared by libpkv's translation units: host-side error state, the pool handle,
// launch helpers (programmatic dependent launch), and inline-PTX wrappers for mbarriers and the
// bulk (TMA) copy engine on sm_103a.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "pkv.h"

namespace pkv {

// ---- host-side error reporting -----------------------------------------------------------------
void set_error(const std::string& msg);
void clear_error();
pkv_status fail(pkv_status code, const std::string& msg);
pkv_status cuda_fail(cudaError_t e, const char* what);

constexpr size_t kStatusBytes = 256;

struct PlanKey {
  const void* workspace = nullptr;
  const int32_t* context_lens = nullptr;
  const int32_t* query_start_loc = nullptr;
  int32_t num_seqs = -1;
  int32_t num_tokens = -1;
  int32_t max_blocks_per_seq = -1;
  // Under PKV_VALIDATE=1: a hash of the context_lens and query_start_loc contents the plan was built from.
  bool summed = false;
  uint64_t meta_sum = 0;
};

// Plans remembered per pool: one per workspace, the most recently planned last.  A plan on a workspace
// replaces that workspace's earlier plan and nothing else; past kMaxPlans workspaces the oldest is
// forgotten (its next pkv_attention is refused until it is planned again).
constexpr size_t kMaxPlans = 32;

// What PKV_VALIDATE=1 learned about a call's metadata (nothing when the check did not run).
struct MetaCheck {
  bool ran = false;
  uint64_t sum = 0;  // hash of the context_lens and query_start_loc contents
};

}  // namespace pkv

struct pkv_pool {
  // The cache as the TMA engine sees it, 128-byte swizzle: fp16, rows of head_dim values (one per (layer,
  // K/V, block, KV head, slot)); 8-bit, rows of 128 code bytes (a (block, KV head) run is 16*head_dim/128
  // consecutive rows), at head_dim 256 a 3-D map (128 code bytes, the key's half, the key).
  CUtensorMap kv_map;
  // fp16: the same cache as whole (block, KV head) runs of K or V, one box of 16 rows x head_dim values laid
  // out as head_dim / 64 swizzled 2 KB sub-tiles (the 2-D map's boxes side by side): one copy per run
  CUtensorMap run_map;
  pkv_config cfg;
  char* base = nullptr;        // device: cache (8-bit: codes, then scales), then the status area
  size_t cache_bytes = 0;      // bytes before the status area
  size_t scales_off = 0;       // 8-bit cache: offset of the scale bytes
  int32_t* dev_error = nullptr;  // device error word (in the status area)
  int32_t last_launches = 0;
  int num_sms = 0;
  int device = 0;
  std::vector<pkv::PlanKey> plans;  // the plans issued through this pool, one per workspace (most recent last)
  // 8-bit cache: tensor map of the fp16 shadow in the last workspace used for prefill rows (re-encoded when
  // the workspace or its size changes)
  CUtensorMap shadow_map;
  const void* shadow_base = nullptr;
  uint64_t shadow_rows = 0;
};

namespace pkv {
// 2-D TMA map of `rows` rows of head_dim fp16 values at `base`: boxes of 16 rows x 64 values, 128-byte swizzle
// (the layout of an fp16 pool, and of the 8-bit cache's fp16 shadow).
pkv_status encode_f16_rows(CUtensorMap* map, void* base, uint64_t rows, int head_dim);
// 3-D TMA map of the same rows whose box is a whole run: 16 rows x head_dim values, stored as head_dim / 64
// sub-tiles of 16 rows x 64 values (128-byte swizzle), sub-tile h at 2048 h bytes -- the layout of head_dim / 64
// boxes of the 2-D map side by side, in one copy.
pkv_status encode_f16_runs(CUtensorMap* map, void* base, uint64_t rows, int head_dim);
// The PKV_VALIDATE=1 host check of a call's device metadata (a no-op otherwise); null pointers are skipped.
// When `check` is given and the check ran, it receives a hash of the context_lens and query_start_loc contents.
pkv_status validate_metadata(const pkv_pool* pool, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* context_lens, const int32_t* qsl, int32_t num_seqs, int32_t num_tokens,
                             const int64_t* slots, void* stream, MetaCheck* check = nullptr);
}  // namespace pkv

namespace pkv {

// ---- launch with programmatic dependent launch (PDL) ---------------------------------------------
// Every kernel of the library calls griddep_wait() before touching global memory written by earlier
// work, so letting the next grid be scheduled early is always safe and hides launch latency.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv

// ---- device helpers ------------------------------------------------------------------------------
#if defined(__CUDACC__)

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace pkv {
namespace dev {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

#ifndef PKV_WAIT_MODE
#define PKV_WAIT_MODE 0
#endif
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
#if PKV_WAIT_MODE == 1
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
#elif PKV_WAIT_MODE == 2
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(PKV_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

// Non-blocking probe: whether phase `parity` of `bar` has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Limits of every on-chip wait: it gives up only after more than kWaitMinPolls polls AND more than
// kWaitLimitNs of %globaltimer time.
constexpr uint32_t kWaitMinPolls = 1u << 16;
constexpr int64_t kWaitLimitNs = 1000000000ll;

// Bounded wait: gives up (returns false) only after more than `min_polls` polls AND more than `limit_ns`
// of %globaltimer time, measured as a signed difference so that an adjustment of the timer can neither
// wrap the elapsed time nor end the wait early on its own.  Callers record PKV_DEVERR_WAIT_TIMEOUT
// and unwind without touching the barrier again.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int64_t limit_ns = kWaitLimitNs,
                                          uint32_t min_polls = kWaitMinPolls) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t polls = 1;; ++polls) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((polls & 255u) == 0 && polls > min_polls) {
      const int64_t dt = (int64_t)(globaltimer_ns() - t0);
      if (dt > limit_ns) return false;
    }
  }
}

// A pool whose error word records a wait timeout refuses further work until pkv_pool_check clears it.
__device__ __forceinline__ bool pool_poisoned(const int32_t* err) {
  return err && (*reinterpret_cast<const volatile int32_t*>(err) & PKV_DEVERR_WAIT_TIMEOUT) != 0;
}

// 1-D bulk copy global -> shared through the TMA engine, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same without an L2 cache hint.
__device__ __forceinline__ void bulk_g2s_plain(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// 3-D tiled TMA load of a box of `map` at element coordinates (x, y, z) into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_addr(dst_smem)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// 2-D tiled TMA load of a box of `map` at element coordinates (x, y) into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_addr(dst_smem)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// Warp-level matrix helpers (sm_80+ forms, valid on sm_103a).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Brings the 128-byte line holding `addr` into L2 (a hint: no data returned, nothing to wait for).
__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier global accesses (an acquire among them) before its later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Producer side of a named barrier: counts this thread's arrival without waiting.
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- 5th-generation tensor cores (tcgen05) and tensor memory -----------------------------------
// Tensor memory (TMEM) is 128 lanes x 512 columns of 32-bit cells per SM.  An MMA with M = 128 writes
// its fp32 accumulator row m to lane m, column n.  Warp w of a CTA may read or write lanes
// 32*(w % 4) .. 32*(w % 4) + 31 only.  Addresses are (lane << 16) | column.

// Allocate `ncols` TMEM columns (a power of two >= 32); the base address is written to *dst_smem.
// Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Ordering of tcgen05 operations across a thread synchronisation (barrier or mbarrier).
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05.mma: start address, leading- and stride-dimension byte
// offsets (all >> 4), descriptor version 1, 128-byte swizzle.  Operand tiles are stored as rows of 128
// bytes (64 fp16), 8-row atoms of 1024 bytes, the 16-byte chunk c of row r at chunk (c ^ (r % 8)) --
// the layout a TMA copy with 128-byte swizzle writes into a 1024-byte aligned destination.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of a dense kind::f16 MMA with fp16 A and B, fp32 accumulator, M x N.
// a_mn / b_mn: the operand is stored MN-major (its M or N index contiguous) instead of K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                          // accumulator format: fp32
         | (0u << 7) | (0u << 10)           // A, B format: fp16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], issued by one thread.  A (M x 16 per MMA, fp16) sits in TMEM with row m
// in lane m and two consecutive K elements packed per 32-bit column.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// This thread's TMEM lane, 32 consecutive columns from `taddr`, into v[0..31] (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
      "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// 2^x by the hardware's approximate base-2 exponential (denormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// GPU-scope atomic add with release semantics: earlier writes of this thread (and of warp mates ordered
// before it by a warp barrier) are visible to whoever acquires the counter afterwards.
__device__ __forceinline__ int atom_add_release_gpu(int32_t* addr, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// GPU-scope atomic add with acquire and release semantics (returns the old value).
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}
// GPU-scope load with acquire semantics.
__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* addr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* addr) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void set_error(int32_t* err, int32_t bits) {
  if (err) atomicOr(err, bits);
}

// ---- 8-bit cache rows: E4M3 codes with one power-of-two scale per (token, KV head) row ---------------
// Largest magnitude among 8 fp16 values, as fp16 bits with the sign cleared (for finite values the bit
// patterns order like the magnitudes).
__device__ __forceinline__ uint32_t f16x8_amax_bits(const uint4& r) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}
// The same over a row spread across LANES consecutive lanes (a lane-aligned group; every lane of the warp
// takes part).
template <int LANES>
__device__ __forceinline__ uint32_t row_amax_bits(uint32_t m) {
#pragma unroll
  for (int o = 1; o < LANES; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}
// Scale byte e + 127 of a row whose largest magnitude has fp16 bits `amax`: e is the smallest integer with
// amax <= 448 * 2^e (0 for an all-zero row).  With amax = 1.m * 2^k (a normal fp32 for every fp16 value)
// and 448 = 1.75 * 2^8: e = k - 8, plus one when 1.m > 1.75.
__device__ __forceinline__ int e4m3_scale_byte(uint32_t amax) {
  if (amax == 0) return 127;
  const uint32_t b = __float_as_uint(__half2float(__ushort_as_half((unsigned short)amax)));
  const int k = (int)(b >> 23) - 127;
  return k - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0) + 127;
}
// Power of two 2^(sb - 127) as fp32, for scale bytes 1 .. 254.
__device__ __forceinline__ float scale_of_byte(uint32_t sb) { return __uint_as_float(sb << 23); }
// E4M3 codes of 8 fp16 values divided by 2^(sb - 127): the division is an exact power-of-two scaling in
// fp32, then each value is rounded to the nearest E4M3 value, ties to even (saturating, which |x| / 2^e
// <= 448 never reaches).  Byte i of the result is value i.
__device__ __forceinline__ uint2 e4m3_encode8(const uint4& r, int sb) {
  const float inv = __uint_as_float((uint32_t)(254 - sb) << 23);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    c[i] = __nv_cvt_float2_to_fp8x2(make_float2(f.x * inv, f.y * inv), __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}
// Four E4M3 codes (byte i = code i) as two fp16 pairs: lo = (code 0, code 1), hi = (code 2, code 3), low
// half first; exact.  The word's two 16-bit halves feed one conversion each, with no repacking.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

// Eight E4M3 codes with scale byte sb as eight fp16 values code * 2^(sb - 127): exact wherever the value is an
// fp16 number, which it is unless within 3 % of the fp16 maximum (there it saturates to +-65504).
__device__ __forceinline__ uint4 e4m3x8_dequant(const uint2& codes, uint32_t sb) {
  const float sc = scale_of_byte(sb);
  uint32_t h[4];
  e4m3x4_to_f16x2x2(codes.x, h[0], h[1]);
  e4m3x4_to_f16x2x2(codes.y, h[2], h[3]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    const __half2 r = __floats2half2_rn(fminf(fmaxf(f.x * sc, -65504.f), 65504.f),
                                        fminf(fmaxf(f.y * sc, -65504.f), 65504.f));
    h[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Row of packed token t: the largest b with query_start_loc[b] <= t (query_start_loc has num_seqs + 1
// entries).  Binary search; callers validate the row's bounds afterwards.
__device__ __forceinline__ int row_of_token(const int32_t* __restrict__ qsl, int num_seqs, int t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace dev
}  // namespace pkv

#endif  // __CUDACC__
