/*
 * pkv.h -- C ABI of libpkv: the per-pass hot path of a continuous-batching engine on one GB300 (sm_103a):
 * append this pass's K/V into a block-paged cache, then run causal grouped-query attention for a ragged
 * batch of decode rows (one new token) and chunked-prefill rows (many new tokens).
 *
 * Sources (web pages, cited by title and section):
 *   [CB]  "Continuous Batching Is Not a Bigger Batch" (deepconcepts.dev)
 *   [SB]  "Static batching" (danielfleming.xyz)
 *   [SC]  "Saturation and Capacity" (doublewordai inference-lab)
 *   [ABL] "An advertised batch limit proves nothing until sampled" (a8q9.cn)
 *
 * Conventions for every call below
 *   - Device pointers are owned by the caller (e.g. torch tensors).  The library never allocates device
 *     memory; where it needs scratch, the caller passes a workspace sized by a *_bytes query.
 *   - GPU work is enqueued asynchronously on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream).  A call returns before its kernels finish.
 *   - Argument and shape errors are detected on the host and returned BEFORE anything is launched;
 *     pkv_last_error() then holds a message (thread-local, valid until the next call on the thread).
 *   - Contents of device metadata (block ids, slots, lengths) cannot be checked on the host without a
 *     sync.  Kernels bounds-check every index they derive from them: an out-of-range value is skipped
 *     (never dereferenced) and recorded in the pool's device error word, read by pkv_pool_check().
 *   - PKV_VALIDATE=1 in the environment (read at every call): the calls below also copy the device metadata
 *     they are given (query_start_loc, context_lens, block tables up to each row's context, slots) to the
 *     host after synchronizing the stream, and refuse a bad pass before launching anything --
 *     PKV_ERR_INVALID_ARG for rows (query_start_loc not running from 0 to num_tokens without decreasing, or
 *     not 1 <= q_len <= ctx <= max_blocks_per_seq * block_size), PKV_ERR_OUT_OF_RANGE for block ids and
 *     slots.  A plan issued under PKV_VALIDATE=1 also remembers a hash of the context_lens and
 *     query_start_loc contents; a pkv_attention / pkv_attention_append on that workspace whose metadata
 *     contents differ (same pointers, rewritten in place without a new plan) is refused with
 *     PKV_ERR_INVALID_ARG.  A debugging aid: it costs a synchronization and copies per call, and is skipped
 *     while the stream is being captured into a graph.
 *   - No call traps the device, and no kernel waits on another grid.
 *   - A pool handle is used by one host thread at a time: it remembers the plan issued on each of its 32
 *     most recently planned workspaces and, on an 8-bit cache, the tensor map of the last workspace's fp16
 *     shadow.  Different pools are independent; pkv_last_error is per thread.
 *   - Supported shapes: fp16 Q and K/V inputs; an fp16 or 8-bit (E4M3) cache; head_dim 64, 128 or 256;
 *     block_size 16; num_q_heads a multiple of num_kv_heads with a group of 1, 2, 4, 6 or 8 query heads
 *     per KV head.  Others: PKV_ERR_UNSUPPORTED.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes, misaligned buffer */
  PKV_ERR_OUT_OF_RANGE = 2,  /* layer, request id or size outside what the object was built for    */
  PKV_ERR_UNSUPPORTED = 3,   /* shape the kernels are not built for                                   */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call failed; pkv_last_error() has cudaGetErrorString  */
  PKV_ERR_NO_BLOCKS = 5,     /* scheduler: pool cannot hold a request even when empty                 */
  PKV_ERR_NOT_FOUND = 6      /* scheduler: unknown request id                                         */
} pkv_status;

/* Device error word bits (pkv_pool_check). */
#define PKV_DEVERR_SLOT_RANGE   0x1  /* pkv_append: slot outside [-1, num_blocks*block_size)        */
#define PKV_DEVERR_BLOCK_RANGE  0x2  /* attention: block id outside [0, num_blocks)                  */
#define PKV_DEVERR_ROW_META     0x4  /* row with q_len < 1, q_len > ctx, or ctx > max_blocks*bs       */
#define PKV_DEVERR_QSL          0x8  /* query_start_loc not monotone / not ending at num_tokens       */
#define PKV_DEVERR_WAIT_TIMEOUT 0x10 /* an on-chip barrier wait gave up (should never happen)          */

/* ------------------------------------------------------------------------------------------------
 * Cache pool
 *
 * [CB] "What the scheduler does on one step" / "Where the batch size actually comes from": every
 * sequence holds one key and one value per token per layer, allocated on demand in 16-token blocks;
 * grouped-query attention keeps num_kv_heads < num_q_heads.  [SB] "Ragged batches": a paged layout
 * stores only real tokens.
 *
 * Layout of the caller's buffer (row-major), kv_dtype = PKV_KV_F16:
 *     cache[num_layers][2 (K, V)][num_blocks][num_kv_heads][block_size][head_dim]   fp16
 * followed by a 256-byte status area (the device error word).  One (block, kv head) is a contiguous
 * run of block_size*head_dim*2 bytes, which the kernels move with single bulk copies.
 * Bytes per token of context = 2 * num_layers * num_kv_heads * head_dim * 2 ([CB], same section).
 *
 * kv_dtype = PKV_KV_E4M3, the 8-bit cache.  [CB] "Checking it on a real system": when the cache is
 * what limits the batch, quantize it; [ABL] "Context math sets the ceiling the fields ignore": 8-bit KV
 * is half the raw bytes of fp16, with scales on top.  Every cached row (one token's head_dim values of
 * one KV head, K and V separately) is stored as E4M3 codes (OCP 8-bit floating point: bias 7, no
 * infinities, largest magnitude 448) and one power-of-two scale 2^e, kept as the byte e + 127; e is the
 * smallest integer with max|x| <= 448 * 2^e (0 for an all-zero row), and each code is x / 2^e rounded to
 * the nearest E4M3 value, ties to even.  Nothing is clipped; attention reads code * 2^e exactly.
 *     codes [num_layers][2 (K, V)][num_blocks][num_kv_heads][block_size][head_dim]   uint8
 *     scales[num_layers][num_blocks][num_kv_heads][2 (K, V)][block_size]              uint8
 * then the status area (at the next 256-byte boundary).  A (block, kv head) run of codes is
 * block_size*head_dim bytes; its K and V scales are one 32-byte record.  Bytes per token of context =
 * 2 * num_layers * num_kv_heads * (head_dim + 1).  K and V inputs must be finite.
 * ---------------------------------------------------------------------------------------------- */
#define PKV_KV_F16  0
#define PKV_KV_E4M3 1

typedef struct {
  int32_t num_layers;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;    /* tokens per block; must be 16 */
  int32_t num_blocks;    /* physical blocks per layer    */
  int32_t split_blocks;  /* blocks per split-K partition of a decode row; 0 = library default (32) */
  int32_t kv_dtype;      /* PKV_KV_F16 (0) or PKV_KV_E4M3 */
} pkv_config;

typedef struct pkv_pool pkv_pool;

/* Bytes the caller must provide to pkv_pool_init for this configuration (cache + status area),
 * or 0 if the configuration is invalid. */
size_t pkv_pool_bytes(const pkv_config* cfg);

/* Wrap caller-owned device memory `dev_cache` (>= pkv_pool_bytes(cfg) bytes, 256-byte aligned) as a
 * pool.  Zeroes the status area (synchronously, on the legacy default stream); the cache contents
 * are left as they are.  *out receives a host handle; free it with pkv_pool_destroy. */
pkv_status pkv_pool_init(const pkv_config* cfg, void* dev_cache, size_t bytes, pkv_pool** out);

/* Frees the host handle only; the device buffer stays the caller's. */
void pkv_pool_destroy(pkv_pool* pool);

/* Device address of layer `layer`'s K (kv = 0) or V (kv = 1) pool [num_blocks][Hkv][bs][d] (fp16 values,
 * or E4M3 codes for an 8-bit cache); NULL on a bad argument. */
void* pkv_pool_layer_ptr(const pkv_pool* pool, int32_t layer, int32_t kv);

/* Device address of layer `layer`'s scale bytes [num_blocks][Hkv][2 (K, V)][bs] of an 8-bit cache; NULL
 * for an fp16 cache or a bad argument. */
void* pkv_pool_scales_ptr(const pkv_pool* pool, int32_t layer);

/* Synchronously read the device error word (PKV_DEVERR_* bits) into *bits, then clear it if `clear`.
 * Waits for all work on the legacy default stream's device.  While PKV_DEVERR_WAIT_TIMEOUT is set,
 * attention launches return without work; after clearing it, issue a new pkv_attention_plan before
 * the next pkv_attention (the interrupted launch may have left split counters mid-count). */
pkv_status pkv_pool_check(pkv_pool* pool, int32_t* bits, int32_t clear);

/* ------------------------------------------------------------------------------------------------
 * Slot mapping (device)
 *
 * [CB] "What the scheduler does on one step": a row's new tokens are the positions from
 * num_computed_tokens up; blocks are allocated as tokens are computed.  Token i of row b sits at
 * absolute position p = context_lens[b] - q_len_b + i and writes slot
 *     block_tables[b][p / block_size] * block_size + p % block_size.
 *
 * block_tables    int32 [num_seqs][max_blocks_per_seq]   device
 * context_lens    int32 [num_seqs]  cached + new tokens   device
 * query_start_loc int32 [num_seqs + 1], [0] = 0, [num_seqs] = num_tokens   device
 * slot_mapping    int64 [num_tokens] output               device
 * Rows whose metadata is out of range get slot -1 and set PKV_DEVERR_ROW_META / _BLOCK_RANGE.
 * ---------------------------------------------------------------------------------------------- */
pkv_status pkv_slot_mapping(pkv_pool* pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, const int32_t* query_start_loc, int32_t num_seqs,
                            int32_t num_tokens, int64_t* slot_mapping, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Append (kv_append)
 *
 * [CB] opening section and "The allocator is the other half": each computed token's key and value
 * are stored in the cache so later passes need not recompute them; storage is the token's slot in a
 * 16-token block.  Copies k[t], v[t] ([num_kv_heads][head_dim] fp16 each) of `layer` into slot
 * slot_mapping[t] for t < num_tokens; a slot of -1 is skipped (padding); any other out-of-range slot
 * is skipped and sets PKV_DEVERR_SLOT_RANGE.  fp16 cache: a bit copy, no arithmetic.  8-bit cache: each
 * (token, KV head) row of K and of V is quantized as the pool section describes (codes and scale byte,
 * bit-exact).  Duplicate slots in one call race (last writer unspecified).
 *
 * k, v          fp16 [num_tokens][num_kv_heads][head_dim]   device, 16-byte aligned
 * slot_mapping  int64 [num_tokens]                          device
 * ---------------------------------------------------------------------------------------------- */
pkv_status pkv_append(pkv_pool* pool, int32_t layer, const void* k, const void* v,
                      const int64_t* slot_mapping, int32_t num_tokens, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Ragged paged attention
 *
 * [CB] "What the scheduler does on one step": one pass mixes decode rows (one new token) and
 * chunked-prefill rows (up to the token budget of new prompt tokens), with no separate prefill phase.
 * Row b owns query tokens query_start_loc[b] .. query_start_loc[b+1]-1 (q_len_b of them) and
 * context_lens[b] keys, this pass's appended tokens included.  Query i of the row is at absolute
 * position ctx_b - q_len_b + i and attends causally to keys 0 .. ctx_b - q_len_b + i.  Query head h
 * reads KV head h / (num_q_heads / num_kv_heads).  Scores are scaled by 1/sqrt(head_dim); softmax
 * and accumulation in fp32; output rounded once to fp16 (round-to-nearest-even).
 *
 * Use: size a workspace with pkv_attention_workspace_bytes, call pkv_attention_plan once per pass
 * (after the metadata is on the device), then pkv_attention once per layer.  A plan stays valid
 * for every pkv_attention call with the same workspace and metadata pointers and sizes until the
 * next pkv_attention_plan on that workspace; changing the metadata CONTENTS requires a new plan.
 * pkv_attention refuses (PKV_ERR_INVALID_ARG) a call whose workspace/metadata pointers or sizes
 * differ from the last plan issued on `workspace` (and, under PKV_VALIDATE=1, one whose metadata
 * contents changed).  Plans live per workspace: planning one workspace leaves the plans of the
 * pool's other workspaces valid (double-buffered passes), up to the 32 most recently planned
 * workspaces per pool.  Plans and calls on one workspace must be ordered on one stream (or
 * synchronised by the caller).
 *
 * The result is independent of the batch: a row's split-K partition depends only on its own
 * context length, so a row gives bit-identical output alone or in any batch, in any row order.
 *
 * 8-bit cache: attention reads the dequantized values code * 2^e exactly (scales applied in fp32).  Rows
 * with 16 or more new tokens first have their blocks dequantized into an fp16 shadow
 * inside the workspace, read by the tensor-core tile kernel; values within 3 % of the fp16 maximum saturate
 * there.  pkv_attention_workspace_bytes then includes room for min(num_blocks, R * max_blocks_per_seq)
 * shadow blocks, R the most rows of 16+ new tokens the pass can hold; prefill rows holding more blocks in
 * total (rows sharing blocks count each time) are refused and reported (PKV_DEVERR_BLOCK_RANGE).
 *
 * q                fp16 [num_tokens][num_q_heads][head_dim]   device, 16-byte aligned
 * block_tables     int32 [num_seqs][max_blocks_per_seq]       device
 * context_lens     int32 [num_seqs]                           device
 * query_start_loc  int32 [num_seqs + 1]                       device
 * out              fp16 [num_tokens][num_q_heads][head_dim]   device (may not alias q)
 * workspace        device, >= pkv_attention_workspace_bytes(...) bytes, 256-byte aligned
 * ---------------------------------------------------------------------------------------------- */
size_t pkv_attention_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_tokens,
                                     int32_t max_blocks_per_seq);

pkv_status pkv_attention_plan(pkv_pool* pool, const int32_t* context_lens, const int32_t* query_start_loc,
                              int32_t num_seqs, int32_t num_tokens, int32_t max_blocks_per_seq,
                              void* workspace, size_t workspace_bytes, void* stream);

pkv_status pkv_attention(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens, void* out,
                         void* workspace, size_t workspace_bytes, void* stream);

/* kv_append and attention of one layer in one call: the same result -- cache contents and output --
 * as pkv_append(pool, layer, k, v, slot_mapping, num_tokens) followed by pkv_attention(...) with the
 * other arguments, under the same plan.  When no row of the pass can take the prefill path (every row
 * has fewer than 16 new tokens; the host checks num_tokens - num_seqs < 15), the append runs inside
 * the decode launch: tiles take this pass's keys and values from k / v directly (on an 8-bit cache,
 * quantized exactly as the append would store them), and each token is written to the cache by the warp
 * whose block holds its position, so no separate append precedes the attention.  Otherwise (and on an
 * 8-bit cache whenever a row may have 16 or more new tokens) this is the append launch followed by the
 * attention launches.  Tokens of rows
 * whose metadata is rejected (PKV_DEVERR_ROW_META) are not appended on the fused path.
 *
 * k, v             fp16 [num_tokens][num_kv_heads][head_dim]   device, 16-byte aligned
 * slot_mapping     int64 [num_tokens]                          device (-1: skip the token)
 * (everything else as pkv_attention) */
pkv_status pkv_attention_append(pkv_pool* pool, int32_t layer, const void* q, const void* k, const void* v,
                                const int64_t* slot_mapping, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                int32_t num_tokens, void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Allocation-free attention.  The pages have no counterpart to this call; it exists for callers that
 * cannot give the library a workspace -- an engine whose device memory is already carved up by its
 * own allocator, or code that must not call cudaMalloc (a device-wide synchronisation) mid-pass.
 *
 * Does what pkv_attention_plan followed by pkv_attention does, with the same arguments minus the
 * workspace, and gives the same result.  The split-K scratch lives in one array of
 * PKV_NOALLOC_SCRATCH_BYTES compiled into libpkv, held on every device that loads the library until
 * the process exits; the library allocates nothing.  A pass whose scratch
 * (pkv_attention_workspace_bytes for the same sizes) exceeds that limit is refused with
 * PKV_ERR_OUT_OF_RANGE before anything is launched.
 *
 * The first call in a device's context looks up the array's device address (cudaGetSymbolAddress) with
 * that device current -- the pool's device must be the current device -- so make that first call
 * before any stream capture: a first call made while `stream` is capturing is refused with
 * PKV_ERR_INVALID_ARG.  The address is cached per (device, context), so a context re-created after
 * cudaDeviceReset looks it up again.  Every call shares the one array and leaves its contents behind;
 * nothing in it has to start at zero, but two calls whose kernels can overlap on the GPU (different
 * streams with no ordering between them) race on it.  Every refusal (sizes, the 8-bit cache's prefill
 * limits, the capture rule) comes before anything is launched. */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
pkv_status pkv_attention_noalloc(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens, void* out,
                                 void* stream);

/* Test hook, off by default: refused with PKV_ERR_UNSUPPORTED unless PKV_TEST_HOOKS=1 is in the environment.
 * The pages have no counterpart; it exercises the failure path of [ABL] "Counting jobs while they run" (a
 * job must not be left holding the device).  Launches one kernel whose thread waits on an on-chip barrier
 * that never completes, through the same bounded wait every attention kernel uses, with the time limit
 * shortened to limit_ns (1 .. 1e8); when the wait gives up it sets PKV_DEVERR_WAIT_TIMEOUT in the pool's
 * error word and returns.  Afterwards attention launches on the pool do no work until pkv_pool_check
 * clears the bit and the pass is planned again. */
pkv_status pkv_debug_expire_wait(pkv_pool* pool, int64_t limit_ns, void* stream);

/* Number of kernel launches the last successful pkv_append / pkv_attention_plan / pkv_attention /
 * pkv_slot_mapping call on `pool` enqueued (for accounting; host-side counter). */
int32_t pkv_last_launch_count(const pkv_pool* pool);

/* Message for the last failed call on this thread ("" if none). */
const char* pkv_last_error(void);

/* ------------------------------------------------------------------------------------------------
 * Host reference scheduler (generates the per-pass batches; never on the timed path)
 *
 * [CB] "What the scheduler does on one step": schedule() runs once per pass.  Phase one walks running
 * requests in arrival order; each wants num_tokens - num_computed_tokens (1 when decoding, the rest of
 * the prompt when prefilling) capped by the token budget (chunked prefill).  Blocks are allocated for
 * them; on failure the newest running request is popped, its blocks freed, its status set PREEMPTED,
 * num_computed_tokens reset to 0 and it is prepended to the waiting queue; retry.  If the popped
 * request is the one being scheduled, phase one stops.  Phase two (only when the pass preempted
 * nobody) admits from the waiting queue's head while the budget lasts and fewer than max_num_seqs
 * run; an unallocatable head stops admission for the pass.  [SC] "Runtime capacity control":
 * max_num_seqs gates admission only and must be >= 1; lowering it drains, never evicts.  [ABL]
 * "Counting jobs while they run": a cancelled request must free its memory (pkv_sched_abort).
 * A pass that computes a request's last known token yields one output token; at max_output outputs
 * the request finishes and frees its blocks in the same pass (freed blocks join the free list's tail).
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
  int32_t max_num_seqs;   /* >= 1                                    */
  int32_t token_budget;   /* new tokens per pass, >= 1               */
  int32_t block_size;     /* tokens per block, >= 1                  */
  int32_t num_blocks;     /* physical blocks in the pool             */
} pkv_sched_config;

typedef struct pkv_sched pkv_sched;

/* One pass's ragged batch.  All arrays are HOST memory owned by the scheduler, valid until the next
 * pkv_sched_step / pkv_sched_destroy.  Rows are in scheduling order (running first, then admitted). */
typedef struct {
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t max_blocks_per_seq;       /* width of block_tables: max blocks held by a scheduled row (>= 1) */
  const int64_t* req_ids;           /* [num_seqs]                                   */
  const int32_t* q_lens;            /* [num_seqs]                                   */
  const int32_t* context_lens;      /* [num_seqs]  num_computed before + q_len       */
  const int32_t* query_start_loc;   /* [num_seqs + 1]                               */
  const int32_t* block_tables;      /* [num_seqs][max_blocks_per_seq], -1 padded     */
  const int64_t* slot_mapping;      /* [num_tokens]                                 */
  int32_t num_preempted;
  const int64_t* preempted;         /* in pop order (newest first)                  */
  int32_t num_admitted;
  const int64_t* admitted;
  int32_t num_finished;
  const int64_t* finished;
} pkv_step;

typedef struct {
  int64_t steps;
  int64_t preemptions;
  int64_t recomputed_tokens;        /* num_computed_tokens discarded by preemption */
  int64_t recomputed_prompt_tokens; /* the prompt part of it                       */
  int64_t max_batch;                /* most rows in one pass                       */
  int64_t batch_sum;                /* sum of rows over passes (mean = /steps)     */
  int64_t tokens_scheduled;
  int32_t running;
  int32_t waiting;
  int32_t free_blocks;
  int64_t live_tokens;              /* summed over passes, after each pass: tokens running requests hold */
  int64_t held_slots;               /* summed over passes: slots of the blocks running requests hold    */
  int64_t prefix_hit_tokens;        /* recompute refunded by prefix caching                            */
} pkv_sched_stats;

/* Block allocation policies and units of scheduling (pkv_sched_set_policy).  [CB] "The allocator is
 * the other half": on demand (the default) allocates a request's blocks as its tokens are computed and
 * preempts when the pool runs out; RESERVE (Orca) admits a request only if its worst case fits --
 * ceil((prompt_len + declared_output) / block_size) free blocks, all taken at admission and returned when
 * it finishes -- so it never preempts, at the price of holding cache for output the client only claimed.
 * [CB] "The boundary: when this is worth nothing": UNIT_PASS re-decides membership every pass (continuous
 * batching, the default); UNIT_REQUEST is static batching: a batch forms when nothing runs, takes members
 * until the first pass in which one of them finishes, and then runs to its slowest member. */
#define PKV_ALLOC_ON_DEMAND 0
#define PKV_ALLOC_RESERVE   1
#define PKV_UNIT_PASS       0
#define PKV_UNIT_REQUEST    1

/* free_order: the initial free list ([num_blocks] distinct ids in [0, num_blocks)), or NULL for
 * 0..num_blocks-1.  Copied. */
pkv_status pkv_sched_create(const pkv_sched_config* cfg, const int32_t* free_order, pkv_sched** out);
void pkv_sched_destroy(pkv_sched* s);
/* Arrival: appended to the waiting queue.  Duplicate live ids: PKV_ERR_INVALID_ARG.  A request that
 * could never fit the pool (ceil((prompt_len + max_output) / block_size) > num_blocks):
 * PKV_ERR_NO_BLOCKS. */
pkv_status pkv_sched_add(pkv_sched* s, int64_t req_id, int32_t prompt_len, int32_t max_output);
/* As pkv_sched_add, with the output the client declares (>= max_output; RESERVE reserves for it).  A
 * request whose reservation could never fit the pool: PKV_ERR_NO_BLOCKS. */
pkv_status pkv_sched_add_declared(pkv_sched* s, int64_t req_id, int32_t prompt_len, int32_t max_output,
                                  int32_t declared_output);
/* Choose the policies; only before the first request is added (PKV_ERR_INVALID_ARG afterwards). */
pkv_status pkv_sched_set_policy(pkv_sched* s, int32_t alloc, int32_t unit);
/* Prefix caching of recompute after preemption ([CB] "What the scheduler does on one step": the recompute
 * "is partly refundable" when the freed blocks were not evicted by the time the request comes back).  A
 * preempted request's full blocks stay registered while they sit in the free list (returned last block
 * first, so its prefix is evicted last); handing a block out evicts it.  On readmission the request takes
 * back the longest still-registered prefix of its blocks, leaving at least one token to compute, and only
 * the rest is recomputed (pkv_step rows then start past the reused blocks).  On demand only (a reserving
 * scheduler never preempts); set before the first request is added. */
pkv_status pkv_sched_set_prefix_caching(pkv_sched* s, int32_t enable);
/* Run one pass; fills *out (num_seqs may be 0 when nothing is left to do). */
pkv_status pkv_sched_step(pkv_sched* s, pkv_step* out);
pkv_status pkv_sched_abort(pkv_sched* s, int64_t req_id);
pkv_status pkv_sched_set_max_num_seqs(pkv_sched* s, int32_t max_num_seqs);
void pkv_sched_get_stats(const pkv_sched* s, pkv_sched_stats* out);
/* 1 when no request is running or waiting. */
int32_t pkv_sched_done(const pkv_sched* s);
/* Current free list (head first) copied into out[0 .. min(n, free)-1]; returns the free count. */
int32_t pkv_sched_free_list(const pkv_sched* s, int32_t* out, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
