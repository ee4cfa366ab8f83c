// Pool handle, error reporting, slot mapping and kv_append.
//
// kv_append follows "Continuous Batching Is Not a Bigger Batch" (opening section and "The allocator is
// the other half"): every computed token's key and value are kept, one pair per token per layer, in the
// slot of a 16-token block that was allocated as the token was computed.  For an fp16 cache it is a pure
// bit copy.  For the 8-bit cache (same page, "Checking it on a real system": quantize the cache when it is
// the limit) each (token, KV head) row is stored as E4M3 codes with one power-of-two scale.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "pkv_internal.cuh"

namespace pkv {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }
void clear_error() { g_last_error.clear(); }
pkv_status fail(pkv_status code, const std::string& msg) {
  g_last_error = msg;
  return code;
}
pkv_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return PKV_ERR_CUDA;
}

static bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 6 || g == 8; }

static pkv_status check_config(const pkv_config* c) {
  if (!c) return fail(PKV_ERR_INVALID_ARG, "config is NULL");
  if (c->num_layers < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_blocks < 1)
    return fail(PKV_ERR_INVALID_ARG, "layers, heads and blocks must be positive");
  if (c->num_q_heads % c->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (c->block_size != 16) return fail(PKV_ERR_UNSUPPORTED, "block_size must be 16");
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (!supported_group(c->num_q_heads / c->num_kv_heads))
    return fail(PKV_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4, 6 or 8");
  if (c->split_blocks < 0) return fail(PKV_ERR_INVALID_ARG, "split_blocks must be >= 0");
  if (c->kv_dtype != PKV_KV_F16 && c->kv_dtype != PKV_KV_E4M3)
    return fail(PKV_ERR_UNSUPPORTED, "kv_dtype must be PKV_KV_F16 or PKV_KV_E4M3");
  return PKV_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The cache seen by the TMA engine, 128-byte swizzle throughout.  fp16: rows of head_dim values, one row per
// (layer, K/V, block, KV head, slot), boxes of 16 rows x 64 values (128 bytes), so a (block, KV head) run of
// K or V is head_dim / 64 boxes.  8-bit: the codes as rows of 128 bytes; a run (16 * head_dim bytes) is
// one box of 16 * head_dim / 128 rows -- except at head_dim 256, where each half of a key's 256 code bytes is
// its own box (16 keys x 128 bytes), as fp16 boxes are.
static EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn) encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return encode;
}

pkv_status encode_f16_rows(CUtensorMap* map, void* base, uint64_t rows, int head_dim) {
  EncodeTiledFn encode = tensor_map_encoder();
  if (!encode) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (rows >= (1ull << 31)) return fail(PKV_ERR_UNSUPPORTED, "too many rows for 32-bit TMA row coordinates");
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64u, 16u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
  return PKV_OK;
}

pkv_status encode_f16_runs(CUtensorMap* map, void* base, uint64_t rows, int head_dim) {
  EncodeTiledFn encode = tensor_map_encoder();
  if (!encode) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (rows >= (1ull << 31)) return fail(PKV_ERR_UNSUPPORTED, "too many rows for 32-bit TMA row coordinates");
  // dimensions: 64 values of a 64-value column group, the row, the column group (its stride is 128 bytes,
  // below the row's: the box walks a group's 16 rows before the next group, as the 2-D boxes do)
  cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(head_dim / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128u};
  cuuint32_t box[3] = {64u, 16u, (cuuint32_t)(head_dim / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the run map: " + std::to_string((int)r));
  return PKV_OK;
}

static pkv_status encode_kv_map(pkv_pool* p) {
  const pkv_config& c = p->cfg;
  const uint64_t toks = (uint64_t)c.num_layers * 2 * c.num_blocks * c.num_kv_heads * c.block_size;
  if (c.kv_dtype != PKV_KV_E4M3) {
    const pkv_status st = encode_f16_rows(&p->kv_map, p->base, toks, c.head_dim);
    if (st != PKV_OK) return st;
    return encode_f16_runs(&p->run_map, p->base, toks, c.head_dim);
  }
  EncodeTiledFn encode = tensor_map_encoder();
  if (!encode) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (c.head_dim == 256) {
    // a key's 256 code bytes as two 128-byte halves: one box per half (16 keys x 128 bytes), so that within
    // a box key r is swizzle row r (two 128-byte rows per key would repeat the swizzle every four keys)
    if (toks >= (1ull << 31)) return fail(PKV_ERR_UNSUPPORTED, "pool too large for 32-bit TMA coordinates");
    cuuint64_t dims3[3] = {128u, 2u, (cuuint64_t)toks};
    cuuint64_t strides3[2] = {128u, 256u};
    cuuint32_t box3[3] = {128u, 1u, (cuuint32_t)c.block_size};
    cuuint32_t estr3[3] = {1, 1, 1};
    CUresult r = encode(&p->kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p->base, dims3, strides3, box3, estr3,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return PKV_OK;
  }
  const uint64_t rows = toks * c.head_dim / 128;
  if (rows >= (1ull << 31)) return fail(PKV_ERR_UNSUPPORTED, "pool too large for 32-bit TMA row coordinates");
  cuuint64_t dims[2] = {128u, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128u};
  cuuint32_t box[2] = {128u, (cuuint32_t)(c.block_size * c.head_dim / 128)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&p->kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, p->base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
  return PKV_OK;
}

// Bytes of the K/V values (fp16) or codes (8-bit) of every layer.
static size_t values_bytes_of(const pkv_config* c) {
  return (size_t)2 * c->num_layers * (size_t)c->num_blocks * c->num_kv_heads * c->block_size * c->head_dim *
         (c->kv_dtype == PKV_KV_E4M3 ? 1 : sizeof(__half));
}
// Everything before the status area: values, then (8-bit) one scale byte per cached row, padded to 256.
static size_t cache_bytes_of(const pkv_config* c) {
  if (c->kv_dtype != PKV_KV_E4M3) return values_bytes_of(c);
  const size_t scales = (size_t)2 * c->num_layers * (size_t)c->num_blocks * c->num_kv_heads * c->block_size;
  return (values_bytes_of(c) + scales + 255) / 256 * 256;
}

// PKV_VALIDATE=1 (read at every call): the device metadata of a call are copied to the host and checked
// before anything is launched -- query_start_loc from 0 to num_tokens without decreasing, 1 <= q_len <=
// ctx <= max_blocks * block_size per row, every block id a row's context reaches in [0, num_blocks), every
// slot in [-1, num_slots).  The stream is synchronized first; while it is being captured into a graph nothing
// is checked (a capture cannot synchronize).  Any pointer may be null (not checked).
// FNV-1a over 32-bit words (a plain change detector, not a security measure).
static uint64_t fnv1a_words(uint64_t h, const std::vector<int32_t>& words) {
  for (int32_t w : words) {
    const uint32_t u = static_cast<uint32_t>(w);
    for (int i = 0; i < 4; ++i) {
      h ^= (u >> (8 * i)) & 0xFFu;
      h *= 1099511628211ull;
    }
  }
  return h;
}

pkv_status validate_metadata(const pkv_pool* pool, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* context_lens, const int32_t* qsl, int32_t num_seqs, int32_t num_tokens,
                             const int64_t* slots, void* stream, MetaCheck* check) {
  const char* env = std::getenv("PKV_VALIDATE");
  if (!env || std::strcmp(env, "1") != 0 || num_tokens <= 0) return PKV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE: cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) return PKV_OK;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE: cudaStreamSynchronize");
  auto fetch = [&](const void* src, size_t bytes, void* dst) -> cudaError_t {
    return cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
  };
  const pkv_config& c = pool->cfg;
  std::vector<int32_t> q(qsl ? num_seqs + 1 : 0), ctx(context_lens ? num_seqs : 0);
  if (qsl && (e = fetch(qsl, q.size() * 4, q.data())) != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE: copy");
  if (context_lens && (e = fetch(context_lens, ctx.size() * 4, ctx.data())) != cudaSuccess)
    return cuda_fail(e, "PKV_VALIDATE: copy");
  if (check) {
    check->ran = true;
    check->sum = fnv1a_words(fnv1a_words(14695981039346656037ull, ctx), q);
  }
  if (qsl) {
    if (q[0] != 0 || q[num_seqs] != num_tokens)
      return fail(PKV_ERR_INVALID_ARG, "PKV_VALIDATE: query_start_loc must run from 0 to num_tokens");
    for (int b = 0; b < num_seqs; ++b)
      if (q[b + 1] < q[b]) return fail(PKV_ERR_INVALID_ARG, "PKV_VALIDATE: query_start_loc decreases at row " +
                                                              std::to_string(b));
  }
  if (qsl && context_lens) {
    for (int b = 0; b < num_seqs; ++b) {
      const int ql = q[b + 1] - q[b];
      if (ql < 1 || ctx[b] < ql || (int64_t)ctx[b] > (int64_t)max_blocks * c.block_size)
        return fail(PKV_ERR_INVALID_ARG, "PKV_VALIDATE: row " + std::to_string(b) + " has q_len " + std::to_string(ql) +
                                             " and context " + std::to_string(ctx[b]));
    }
  }
  if (block_tables && context_lens) {
    std::vector<int32_t> bt((size_t)num_seqs * max_blocks);
    if ((e = fetch(block_tables, bt.size() * 4, bt.data())) != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE: copy");
    for (int b = 0; b < num_seqs; ++b) {
      const int64_t nblk = std::min<int64_t>(((int64_t)ctx[b] + c.block_size - 1) / c.block_size, max_blocks);
      for (int64_t j = 0; j < nblk; ++j) {
        const int32_t id = bt[(size_t)b * max_blocks + j];
        if (id < 0 || id >= c.num_blocks)
          return fail(PKV_ERR_OUT_OF_RANGE, "PKV_VALIDATE: row " + std::to_string(b) + " block " + std::to_string(j) +
                                                " is " + std::to_string(id));
      }
    }
  }
  if (slots) {
    std::vector<int64_t> sl(num_tokens);
    if ((e = fetch(slots, sl.size() * 8, sl.data())) != cudaSuccess) return cuda_fail(e, "PKV_VALIDATE: copy");
    const int64_t ns = (int64_t)c.num_blocks * c.block_size;
    for (int t = 0; t < num_tokens; ++t)
      if (sl[t] < -1 || sl[t] >= ns)
        return fail(PKV_ERR_OUT_OF_RANGE, "PKV_VALIDATE: slot of token " + std::to_string(t) + " is " +
                                              std::to_string(sl[t]));
  }
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" const char* pkv_last_error(void) { return g_last_error.c_str(); }

extern "C" size_t pkv_pool_bytes(const pkv_config* cfg) {
  if (check_config(cfg) != PKV_OK) return 0;
  return cache_bytes_of(cfg) + kStatusBytes;
}

extern "C" pkv_status pkv_pool_init(const pkv_config* cfg, void* dev_cache, size_t bytes, pkv_pool** out) {
  clear_error();
  pkv_status st = check_config(cfg);
  if (st != PKV_OK) return st;
  if (!dev_cache || !out) return fail(PKV_ERR_INVALID_ARG, "dev_cache and out must be non-NULL");
  if (reinterpret_cast<uintptr_t>(dev_cache) % 256 != 0)
    return fail(PKV_ERR_INVALID_ARG, "dev_cache must be 256-byte aligned");
  size_t need = cache_bytes_of(cfg) + kStatusBytes;
  if (bytes < need)
    return fail(PKV_ERR_INVALID_ARG, "buffer too small: need " + std::to_string(need) + " bytes");
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, dev_cache);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(PKV_ERR_INVALID_ARG, "dev_cache is not device memory");
  pkv_pool* p = new pkv_pool();
  p->cfg = *cfg;
  if (p->cfg.split_blocks == 0) p->cfg.split_blocks = 32;
  p->base = static_cast<char*>(dev_cache);
  p->cache_bytes = cache_bytes_of(cfg);
  p->scales_off = cfg->kv_dtype == PKV_KV_E4M3 ? values_bytes_of(cfg) : 0;
  p->dev_error = reinterpret_cast<int32_t*>(p->base + p->cache_bytes);
  p->device = attr.device;
  e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  st = encode_kv_map(p);
  if (st != PKV_OK) {
    delete p;
    return st;
  }
  e = cudaMemset(p->dev_error, 0, kStatusBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "clearing the status area");
  }
  *out = p;
  return PKV_OK;
}

extern "C" void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

extern "C" void* pkv_pool_layer_ptr(const pkv_pool* pool, int32_t layer, int32_t kv) {
  if (!pool || layer < 0 || layer >= pool->cfg.num_layers || (kv != 0 && kv != 1)) return nullptr;
  const pkv_config& c = pool->cfg;
  size_t per = (size_t)c.num_blocks * c.num_kv_heads * c.block_size * c.head_dim *
               (c.kv_dtype == PKV_KV_E4M3 ? 1 : sizeof(__half));
  return pool->base + ((size_t)layer * 2 + kv) * per;
}

extern "C" void* pkv_pool_scales_ptr(const pkv_pool* pool, int32_t layer) {
  if (!pool || pool->cfg.kv_dtype != PKV_KV_E4M3 || layer < 0 || layer >= pool->cfg.num_layers) return nullptr;
  const pkv_config& c = pool->cfg;
  return pool->base + pool->scales_off + (size_t)layer * c.num_blocks * c.num_kv_heads * 2 * c.block_size;
}

extern "C" pkv_status pkv_pool_check(pkv_pool* pool, int32_t* bits, int32_t clear) {
  clear_error();
  if (!pool || !bits) return fail(PKV_ERR_INVALID_ARG, "pool and bits must be non-NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(bits, pool->dev_error, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (clear) {
    e = cudaMemset(pool->dev_error, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  }
  return PKV_OK;
}

extern "C" int32_t pkv_last_launch_count(const pkv_pool* pool) { return pool ? pool->last_launches : 0; }

// ---------------------------------------------------------------------------------------------------
// Test hook: a bounded on-chip wait that runs out.  One thread waits, through the same bounded wait the
// attention kernels use, on an mbarrier that nobody arrives at, with the time limit shortened to
// `limit_ns`; when the wait gives up it records PKV_DEVERR_WAIT_TIMEOUT in the pool's error word and the
// kernel returns.  Nothing traps and nothing waits without a limit.
// ---------------------------------------------------------------------------------------------------
namespace pkv {
__global__ void expire_wait_kernel(int32_t* err, int64_t limit_ns) {
  __shared__ uint64_t bar;
  dev::griddep_wait();
  if (threadIdx.x != 0) return;
  dev::mbar_init(&bar, 1);
  dev::fence_mbar_init();
  if (!dev::mbar_wait(&bar, 0, limit_ns, 256)) dev::set_error(err, PKV_DEVERR_WAIT_TIMEOUT);
}
}  // namespace pkv

extern "C" pkv_status pkv_debug_expire_wait(pkv_pool* pool, int64_t limit_ns, void* stream) {
  clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  pool->last_launches = 0;
  const char* env = std::getenv("PKV_TEST_HOOKS");
  if (!env || std::strcmp(env, "1") != 0)
    return fail(PKV_ERR_UNSUPPORTED, "pkv_debug_expire_wait is a test hook: set PKV_TEST_HOOKS=1 to enable it");
  if (limit_ns < 1 || limit_ns > 100000000ll) return fail(PKV_ERR_OUT_OF_RANGE, "limit_ns must be in [1, 1e8]");
  const cudaError_t e = launch_pdl(expire_wait_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream, pool->dev_error,
                                   (int64_t)limit_ns);
  if (e != cudaSuccess) return cuda_fail(e, "expire-wait launch");
  pool->last_launches = 1;
  return PKV_OK;
}

// ---------------------------------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------------------------------
namespace pkv {

// One thread per 16-byte chunk of one token's [Hkv][d] K (and the matching chunk of V).
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slot_mapping, int num_tokens,
                                                        uint4* __restrict__ pool_k, uint4* __restrict__ pool_v,
                                                        int num_kv_heads, int chunks_per_head, int64_t num_slots,
                                                        int32_t* err) {
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int64_t per_token = (int64_t)num_kv_heads * chunks_per_head;
  const int64_t total = (int64_t)num_tokens * per_token;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;
    const int64_t h = rem / chunks_per_head;
    const int64_t c = rem - h * chunks_per_head;
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (c == 0 && h == 0) dev::set_error(err, PKV_DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t blk = slot >> 4, off = slot & 15;
    const int64_t dst = ((blk * num_kv_heads + h) * 16 + off) * chunks_per_head + c;
    pool_k[dst] = __ldg(k + i);
    pool_v[dst] = __ldg(v + i);
  }
}

// 8-bit cache: one thread per 16-byte chunk (8 values) of one token's row of one KV head, CPH = head_dim / 8
// consecutive lanes per row (CPH divides 32, so a row never straddles warps).  The row's largest magnitude
// is reduced across its lanes; every lane then writes its 8 codes and the row's first lane the scale bytes.
// The loop runs warp by warp, so every lane of a warp takes part in the reductions.
template <int CPH>
__global__ void __launch_bounds__(256) kv_append_e4m3_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                             const int64_t* __restrict__ slot_mapping, int num_tokens,
                                                             unsigned char* __restrict__ codes_k,
                                                             unsigned char* __restrict__ codes_v,
                                                             unsigned char* __restrict__ scales, int num_kv_heads,
                                                             int64_t num_slots, int32_t* err) {
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  const int64_t per_token = (int64_t)num_kv_heads * CPH;
  const int64_t total = (int64_t)num_tokens * per_token;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < total;
       base += nwarps * 32) {
    const int64_t i = base + lane;
    const bool in = i < total;
    const int64_t t = in ? i / per_token : 0;
    const int64_t rem = i - t * per_token;
    const int64_t h = rem / CPH, c = rem % CPH;
    const int64_t slot = in ? __ldg(slot_mapping + t) : -1;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 rk = in ? __ldg(k + i) : zero, rv = in ? __ldg(v + i) : zero;
    const uint32_t ak = dev::row_amax_bits<CPH>(dev::f16x8_amax_bits(rk));
    const uint32_t av = dev::row_amax_bits<CPH>(dev::f16x8_amax_bits(rv));
    if (!in || slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      if (c == 0 && h == 0) dev::set_error(err, PKV_DEVERR_SLOT_RANGE);
      continue;
    }
    const int sbk = dev::e4m3_scale_byte(ak), sbv = dev::e4m3_scale_byte(av);
    const int64_t blk = slot >> 4, off = slot & 15;
    const int64_t row = (blk * num_kv_heads + h) * 16 + off;
    reinterpret_cast<uint2*>(codes_k + row * (CPH * 8))[c] = dev::e4m3_encode8(rk, sbk);
    reinterpret_cast<uint2*>(codes_v + row * (CPH * 8))[c] = dev::e4m3_encode8(rv, sbv);
    if (c == 0) {
      unsigned char* rec = scales + (blk * num_kv_heads + h) * 32;  // [K: 16 slots][V: 16 slots]
      rec[off] = (unsigned char)sbk;
      rec[16 + off] = (unsigned char)sbv;
    }
  }
}

__global__ void __launch_bounds__(256) slot_mapping_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                                           const int32_t* __restrict__ context_lens,
                                                           const int32_t* __restrict__ qsl, int num_seqs,
                                                           int num_tokens, int num_blocks,
                                                           int64_t* __restrict__ slot_mapping, int32_t* err) {
  dev::griddep_wait();
  dev::griddep_launch_dependents();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < num_tokens; t += gridDim.x * blockDim.x) {
    const int b = dev::row_of_token(qsl, num_seqs, t);
    const int q0 = __ldg(qsl + b), q1 = __ldg(qsl + b + 1);
    const int q_len = q1 - q0, ctx = __ldg(context_lens + b);
    int64_t slot = -1;
    if (t >= q1 || q_len < 1 || ctx < q_len || ctx > max_blocks * 16) {
      dev::set_error(err, PKV_DEVERR_ROW_META);
    } else {
      const int p = ctx - q_len + (t - q0);
      const int blk = __ldg(block_tables + (int64_t)b * max_blocks + (p >> 4));
      if (blk < 0 || blk >= num_blocks) dev::set_error(err, PKV_DEVERR_BLOCK_RANGE);
      else slot = (int64_t)blk * 16 + (p & 15);
    }
    slot_mapping[t] = slot;
  }
}

}  // namespace pkv

extern "C" pkv_status pkv_append(pkv_pool* pool, int32_t layer, const void* k, const void* v,
                                 const int64_t* slot_mapping, int32_t num_tokens, void* stream) {
  clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  pool->last_launches = 0;
  if (layer < 0 || layer >= pool->cfg.num_layers) return fail(PKV_ERR_OUT_OF_RANGE, "layer out of range");
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens must be >= 0");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 != 0)
    return fail(PKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  pkv_status vst = validate_metadata(pool, nullptr, 0, nullptr, nullptr, 0, num_tokens, slot_mapping, stream);
  if (vst != PKV_OK) return vst;
  const pkv_config& c = pool->cfg;
  const int chunks = c.head_dim / 8;
  const int64_t total = (int64_t)num_tokens * c.num_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)pool->num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (c.kv_dtype == PKV_KV_E4M3) {
    const uint4* k4 = static_cast<const uint4*>(k);
    const uint4* v4 = static_cast<const uint4*>(v);
    unsigned char* ck = static_cast<unsigned char*>(pkv_pool_layer_ptr(pool, layer, 0));
    unsigned char* cv = static_cast<unsigned char*>(pkv_pool_layer_ptr(pool, layer, 1));
    unsigned char* sc = static_cast<unsigned char*>(pkv_pool_scales_ptr(pool, layer));
    const int64_t ns = (int64_t)c.num_blocks * c.block_size;
    cudaError_t e;
    switch (chunks) {
      case 8: e = launch_pdl(kv_append_e4m3_kernel<8>, dim3((unsigned)blocks), dim3(threads), 0, (cudaStream_t)stream, k4,
                             v4, slot_mapping, (int)num_tokens, ck, cv, sc, (int)c.num_kv_heads, ns, pool->dev_error);
        break;
      case 16: e = launch_pdl(kv_append_e4m3_kernel<16>, dim3((unsigned)blocks), dim3(threads), 0, (cudaStream_t)stream, k4,
                              v4, slot_mapping, (int)num_tokens, ck, cv, sc, (int)c.num_kv_heads, ns, pool->dev_error);
        break;
      default: e = launch_pdl(kv_append_e4m3_kernel<32>, dim3((unsigned)blocks), dim3(threads), 0, (cudaStream_t)stream,
                              k4, v4, slot_mapping, (int)num_tokens, ck, cv, sc, (int)c.num_kv_heads, ns, pool->dev_error);
        break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    pool->last_launches = 1;
    return PKV_OK;
  }
  cudaError_t e = launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, (cudaStream_t)stream,
                             static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, (int)num_tokens,
                             static_cast<uint4*>(pkv_pool_layer_ptr(pool, layer, 0)),
                             static_cast<uint4*>(pkv_pool_layer_ptr(pool, layer, 1)), (int)c.num_kv_heads, chunks,
                             (int64_t)c.num_blocks * c.block_size, pool->dev_error);
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  pool->last_launches = 1;
  return PKV_OK;
}

extern "C" pkv_status pkv_slot_mapping(pkv_pool* pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                       int32_t num_tokens, int64_t* slot_mapping, void* stream) {
  clear_error();
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  pool->last_launches = 0;
  if (num_tokens < 0 || num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be >= 0");
  if (num_tokens == 0) return PKV_OK;
  if (num_seqs < 1) return fail(PKV_ERR_INVALID_ARG, "tokens without rows");
  if (max_blocks_per_seq < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  if (!block_tables || !context_lens || !query_start_loc || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "metadata pointers must be non-NULL");
  pkv_status vst = validate_metadata(pool, block_tables, max_blocks_per_seq, context_lens, query_start_loc, num_seqs,
                                     num_tokens, nullptr, stream);
  if (vst != PKV_OK) return vst;
  const int threads = 256;
  int blocks = (num_tokens + threads - 1) / threads;
  if (blocks > pool->num_sms * 8) blocks = pool->num_sms * 8;
  cudaError_t e = launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0, (cudaStream_t)stream, block_tables,
                             (int)max_blocks_per_seq, context_lens, query_start_loc, (int)num_seqs, (int)num_tokens,
                             (int)pool->cfg.num_blocks, slot_mapping, pool->dev_error);
  if (e != cudaSuccess) return cuda_fail(e, "slot_mapping launch");
  pool->last_launches = 1;
  return PKV_OK;
}
