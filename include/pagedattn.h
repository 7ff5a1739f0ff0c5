/*
 * pagedattn -- paged grouped-query decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI. Every pointer argument named "device" is CUDA device memory of the
 * pool's device; sizes are element counts unless stated; no call throws.
 * Device work is enqueued on `stream` (a cudaStream_t passed as void*, NULL
 * for the legacy default stream) and is asynchronous: no call synchronises
 * except pa_get_device_error.
 *
 * The operation (sources named by page title and section):
 *  - Paged KV cache: K/V live in fixed-size physical blocks; a per-sequence
 *    block table maps logical block i to a physical block, and token t of a
 *    sequence sits in slot t % block_size of block block_table[t / block_size]
 *    ("十年 C++ 后端 GAP 六个月 ... TFFInfer", section 3.6.4 KVCache:
 *    PageManager, LayerKVContext::get_location; heterogeneous C++ LLM engine
 *    article, sections 2.3 and 4.3).
 *  - KV quantisation: asymmetric per-channel codes, scale = (max-min)/L,
 *    zero_point = round(-min/scale), Q = clamp(round(x/scale)+zp, 0, L),
 *    dequantised as (Q - zp) * scale, with L = 255 (uint8) or 15 (uint4, two
 *    codes per byte) (engine article, sections 2.4, 2.6, 4.4).
 *  - fp8 KV (TFFInfer section 9.3 names FP8 among the formats to add; the
 *    pages fix no scheme): E4M3 codes of the OCP 8-bit floating point format
 *    with one symmetric scale per (block, kv head, channel),
 *    scale = max|x| / 448, code = E4M3(x / scale) rounded to nearest-even and
 *    saturated to +-448, dequantised as value(code) * scale.
 *  - Decode attention: for each sequence b and query head h, with KV head
 *    j = h / (Hq / Hkv) (GQA as in "从零实现 C++ LLM 推理引擎", section
 *    "3. GQA"), out = softmax(q . K^T * softmax_scale) . V over the
 *    sequence's seq_len cached tokens (engine article, section 4.3
 *    paged_attention_kernel; online softmax of the TFFInfer article, section
 *    3.7.2 item 5).
 *
 * Storage format of a pool (library-owned device memory, one allocation):
 * records of pages, [num_blocks][Hkv] records, a page being one block of one
 * kv head, each record contiguous:
 *   bf16 : K bf16 [block_size][head_dim], V bf16 [block_size][head_dim]
 *   uint8: K codes uint8 [block_size][head_dim], V codes likewise, then
 *          K scale float32 [head_dim], K zero point int32 [head_dim],
 *          V scale float32 [head_dim], V zero point int32 [head_dim]
 *   uint4: as uint8 with codes uint8 [block_size][head_dim/2], channel 2i in
 *          the low nibble and 2i+1 in the high nibble
 *   fp8  : K codes (E4M3 bits) uint8 [block_size][head_dim], V codes likewise,
 *          then K scale float32 [head_dim], V scale float32 [head_dim]
 * One (scale, zero point) pair, or one scale for fp8, per (physical block,
 * kv head, channel). Records start on 256-byte boundaries (record bytes:
 * 2 x codes + 4 x 4 x head_dim for uint8 / uint4, 2 x codes + 2 x 4 x
 * head_dim for fp8, 2 x codes for bf16).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_KV_BF16 = 0, PA_KV_UINT8 = 1, PA_KV_UINT4 = 2, PA_KV_FP8 = 3 } pa_kv_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size or count; nothing launched */
  PA_ERR_UNSUPPORTED = 2,   /* head_dim/block_size/group size/dtype not built */
  PA_ERR_OOM = 3,           /* device allocation failed, or workspace too small */
  PA_ERR_CUDA = 4,          /* a CUDA runtime call failed (see pa_last_error) */
  PA_ERR_DEVICE_BOUNDS = 5, /* pa_get_device_error: a kernel met a bad index */
  PA_ERR_TIMEOUT = 6        /* pa_get_device_error: a kernel wait gave up */
} pa_status;

/* Bits of the per-pool device error word (pa_get_device_error). Kernels set
 * them with atomicOr and skip the offending work; they never trap. */
#define PA_DEVERR_BLOCK_TABLE 0x1u /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 0x2u     /* length < 0 or > max_blocks * block_size */
#define PA_DEVERR_APPEND 0x4u      /* cu_new not non-decreasing */
#define PA_DEVERR_TIMEOUT 0x8u     /* a bounded mbarrier wait expired */

typedef struct pa_pool pa_pool; /* opaque, library-owned */

typedef struct {
  int32_t num_blocks;   /* physical blocks, >= 1 */
  int32_t block_size;   /* tokens per block: 16 or 32 */
  int32_t num_kv_heads; /* >= 1 */
  int32_t head_dim;     /* 64 or 128 */
  int32_t kv_dtype;     /* pa_kv_dtype */
  int32_t device;       /* CUDA device ordinal */
} pa_pool_desc;

/* Device addresses of page 0's components (layout above); page n's
 * component lies n * page_stride bytes further. Scale and zero-point pointers
 * are NULL for a bf16 pool, zero-point pointers for an fp8 pool. */
typedef struct {
  void* k;
  void* v;
  float* k_scale;
  int32_t* k_zp;
  float* v_scale;
  int32_t* v_zp;
  size_t page_stride; /* bytes of one page record */
  size_t num_pages;   /* num_blocks * num_kv_heads */
} pa_pool_buffers;

/* pa_create_pool: allocate a pool (one device allocation; contents zero,
 * scales 1.0) on desc->device and return its handle in *out.
 * Errors: PA_ERR_INVALID_ARG (null pointer, counts < 1), PA_ERR_UNSUPPORTED
 * (block_size not 16/32, head_dim not 64/128, unknown dtype), PA_ERR_OOM.
 * The pool owns its memory until pa_destroy. */
PA_API pa_status pa_create_pool(const pa_pool_desc* desc, pa_pool** out);

/* pa_destroy: free the pool (synchronises the device first). NULL is a no-op. */
PA_API pa_status pa_destroy(pa_pool* pool);

/* pa_append_kv: store new tokens' K and V into their blocks (engine article
 * section 2.6 formula for quantised pools; TFFInfer section 3.6.4 addressing).
 *   k_new, v_new   device bf16 [T_new][Hkv][head_dim]; sequence b's new tokens
 *                  are rows cu_new[b] .. cu_new[b+1]-1
 *   cu_new         device int32 [batch+1], non-decreasing, cu_new[0] = 0
 *   ctx_lens       device int32 [batch]: tokens already stored for b; the new
 *                  tokens take logical positions ctx_lens[b], ctx_lens[b]+1, ...
 *   block_table    device int32 [batch][max_blocks] (row stride max_blocks)
 *   max_new_per_seq upper bound on cu_new[b+1]-cu_new[b] (sizes the grid;
 *                  0 = unknown, taken as max_blocks*block_size)
 * bf16 pools get an exact copy of the bits. Quantised pools re-quantise every
 * touched (block, kv head, channel) over the block's valid tokens: stored
 * tokens enter as float(code - zp) * scale, new ones as their bf16 value;
 * scale = (max-min)/L (or |min|/L, or 1.0, for an empty range),
 * zp = rint(-min/scale) (int32, unclamped), code = clamp(rint(x/scale)+zp, 0, L),
 * all in IEEE fp32. fp8 pools likewise re-quantise from float(value(code)) *
 * scale and the new values: scale = max|x| / 448 (1.0 when not > 0),
 * code = E4M3(x / scale), nearest-even, saturated to +-448. A block written by one sequence must not be written by
 * another sequence in the same call. Bad table entries or lengths set the
 * device error word and skip that block or sequence. */
PA_API pa_status pa_append_kv(pa_pool* pool, const void* k_new, const void* v_new, const int32_t* cu_new,
                       const int32_t* ctx_lens, const int32_t* block_table, int32_t batch,
                       int32_t max_blocks, int32_t max_new_per_seq, void* stream);

/* pa_decode: one decode step of grouped-query attention over the paged pool
 * (engine article section 4.3; TFFInfer section 3.7.2 online softmax).
 *   q            device bf16 [batch][num_q_heads][head_dim], 16-byte aligned
 *   block_table  device int32 [batch][max_blocks]
 *   seq_lens     device int32 [batch]: tokens to attend (the step's new token
 *                already appended); 0 gives a zero output row
 *   softmax_scale usually 1/sqrt(head_dim)
 *   out          device float32 [batch][num_q_heads][head_dim], 16-byte aligned
 *   workspace    device scratch of at least pa_decode_workspace_bytes(...)
 *                bytes (256-byte aligned), caller-owned. Zero it once after
 *                allocating it: a small part holds merge tickets tagged with
 *                the call that wrote them; nothing else is read before written
 *   num_splits   number of equal partitions of the (sequence, kv head, block)
 *                work list, one thread block each (0 = one per resident slot
 *                of the device). Sequences cut by a partition boundary are
 *                merged by a log-sum-exp combine kernel.
 * num_q_heads must be a multiple of Hkv with a group size Hq/Hkv <= 8.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OOM (workspace too
 * small), PA_ERR_CUDA. Bad table entries or lengths set the device error
 * word; the affected blocks are skipped. */
PA_API pa_status pa_decode(pa_pool* pool, const void* q, const int32_t* block_table,
                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                    int32_t max_blocks, float softmax_scale, float* out, void* workspace,
                    size_t workspace_bytes, int32_t num_splits, void* stream);

/* pa_decode_step: the decode step in one decode launch (plus the combine):
 * store every sequence's new token (TFFInfer section 3.8: KV cache store,
 * then attention) and attend, as pa_append_kv with one token per sequence
 * (cu_new = 0, 1, ..., batch; ctx_lens = seq_lens - 1) followed by pa_decode
 * would, with the same codes, scales and zero points bit for bit. The thread
 * block that reads a sequence's last page for a kv head stores that head's
 * new token into the block first (re-quantising it for uint8 / uint4 / fp8
 * pools), so the block is written and read once.
 *   k_new, v_new device bf16 [batch][Hkv][head_dim]: row b is sequence b's
 *                new token, at position seq_lens[b] - 1 (ignored when
 *                seq_lens[b] == 0)
 *   the other arguments as pa_decode; seq_lens counts the new token.
 * The blocks receiving new tokens must not be shared with another sequence
 * (copy-on-write first) and must not be written by a kernel still running;
 * with PA_DECODE_EARLY_PLAN the preceding kernel must, as for pa_decode, write
 * neither seq_lens nor block_table. Errors as pa_decode; null k_new / v_new:
 * PA_ERR_INVALID_ARG (nothing launched). */
PA_API pa_status pa_decode_step(pa_pool* pool, const void* k_new, const void* v_new, const void* q,
                                const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                int32_t num_q_heads, int32_t max_blocks, float softmax_scale, float* out,
                                void* workspace, size_t workspace_bytes, int32_t num_splits, void* stream);

/* pa_decode_noalloc: pa_decode for callers that cannot allocate device
 * memory (no allocator on the hot path, memory reserved up front, or no
 * allocator to hand a workspace from). The pages this library follows have no
 * counterpart of it. It computes exactly what pa_decode computes, with the
 * split-KV scratch taken from a fixed 8 MiB array in the library's device
 * image instead of a caller workspace; it calls no allocating routine.
 *   - The array exists on every device that loads the library, until the
 *     process exits. The first call on a device looks up the array's device
 *     address (with the pool's device current); make that first call before
 *     any stream capture.
 *   - Batches whose scratch need (pa_decode_workspace_bytes) exceeds 8 MiB are
 *     rejected with PA_ERR_OOM and a message naming both sizes.
 *   - All calls on a device share the one array and nothing in it must start
 *     at zero: calls whose GPU work overlaps (other streams, other host
 *     threads) race on it; serialise them.
 * Other arguments, errors and semantics as pa_decode. */
PA_API pa_status pa_decode_noalloc(pa_pool* pool, const void* q, const int32_t* block_table,
                                   const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                   int32_t max_blocks, float softmax_scale, float* out,
                                   int32_t num_splits, void* stream);

/* Bytes of workspace pa_decode needs for this batch, head count and split
 * count (0 = the automatic split count); 0 on invalid arguments. */
PA_API size_t pa_decode_workspace_bytes(const pa_pool* pool, int32_t batch, int32_t num_q_heads,
                                 int32_t num_splits);

/* pa_decode_multi: several query tokens per sequence against the paged cache
 * (chunked prefill, and the draft tokens a speculative step verifies; the
 * engine article, sections 2.2 and 4.2, mixes prefill chunks into decode
 * steps, TFFInfer section 9.3 plans speculative decoding).
 *   q    device bf16 [batch][n_q][num_q_heads][head_dim], 16-byte aligned
 *   out  device float32 [batch][n_q][num_q_heads][head_dim], 16-byte aligned
 *   seq_lens counts all n_q new tokens of sequence b (stored before the
 *   call); query token i attends to the tokens t < seq_lens[b] - (n_q-1-i),
 *   a zero row where that is <= 0.
 * Other arguments, errors and the early-plan contract as for pa_decode; the
 * in-kernel merge option does not apply (partials always go through the
 * combine kernel). The query tokens of a kv head's group are processed in
 * column groups of at most 8 (token, head) columns, each reading the
 * sequence's pages once; n_q == 1 is pa_decode. */
PA_API pa_status pa_decode_multi(pa_pool* pool, const void* q, const int32_t* block_table,
                                 const int32_t* seq_lens, int32_t batch, int32_t n_q, int32_t num_q_heads,
                                 int32_t max_blocks, float softmax_scale, float* out, void* workspace,
                                 size_t workspace_bytes, int32_t num_splits, void* stream);

/* Bytes of workspace pa_decode_multi needs; 0 on invalid arguments. */
PA_API size_t pa_decode_multi_workspace_bytes(const pa_pool* pool, int32_t batch, int32_t n_q,
                                              int32_t num_q_heads, int32_t num_splits);

/* Resolve num_splits = 0 to the partition count pa_decode would use. */
PA_API int32_t pa_decode_num_splits(const pa_pool* pool, int32_t num_splits);

/* Decode kernel selection for a pool. AUTO uses the tensor-core kernel where
 * it is built (bf16 pools, and uint8 / uint4 pools of head_dim 128: scores and P.V as
 * mma.m16n8k16 over the GQA group, pages staged by swizzled 2-D TMA) and the
 * CUDA-core kernel otherwise;
 * CUDA_CORE forces the fp32 FMA kernel (kept for comparison). Both compute
 * the same operation. Sequences cut by slice boundaries are merged by a
 * separate log-sum-exp combine kernel; OR-ing PA_DECODE_FUSED_COMBINE merges
 * them inside the decode kernel instead (the last slice to finish a sequence
 * merges its partials, found through call-tagged tickets that it clears once
 * it has merged, so a CUDA graph that replays the call finds them zero again;
 * after a call that reported PA_DEVERR_TIMEOUT, zero the workspace again
 * before the next call with this option). OR-ing
 * PA_DECODE_EARLY_PLAN lets the decode kernel read seq_lens and block_table
 * (and plan its work) while the kernel launched just before it on the stream
 * is still running; it still waits for that kernel before reading any page or
 * writing anything; the split-KV combine kernel likewise reads seq_lens
 * before waiting on the decode kernel. Set it only when that preceding
 * kernel writes neither seq_lens nor block_table (pa_append_kv writes
 * neither).
 * PA_ERR_UNSUPPORTED if TENSOR_CORE is asked for a pool it does not serve. */
typedef enum {
  PA_DECODE_AUTO = 0,
  PA_DECODE_CUDA_CORE = 1,
  PA_DECODE_TENSOR_CORE = 2,
  PA_DECODE_FUSED_COMBINE = 4,
  PA_DECODE_EARLY_PLAN = 8
} pa_decode_path;
PA_API pa_status pa_pool_set_decode_path(pa_pool* pool, int32_t path);

/* Partition of a pool's decode work: the thread blocks take equal shares of
 * a line on which each (sequence, kv head) unit occupies its pages plus
 * `unit_cost_pages` more positions, standing for the fixed work of a unit
 * (loading its query, merging the warps' states, writing its row or
 * partial) in units of page time. A block whose share crosses many unit
 * boundaries thus gets fewer pages. 0 splits the pages evenly; a negative
 * value restores the default of the pool's decode kernel. The results do
 * not depend on it. PA_ERR_INVALID_ARG for a null pool or a value above
 * 4096. */
PA_API pa_status pa_pool_set_unit_cost(pa_pool* pool, int32_t unit_cost_pages);

/* Device addresses of the pool's arrays, for inspection and tests. */
PA_API pa_status pa_pool_view(const pa_pool* pool, pa_pool_buffers* out);

/* Synchronise `stream`, return the pool's device error bits in *flags and
 * clear them. Returns PA_ERR_DEVICE_BOUNDS / PA_ERR_TIMEOUT when bits were
 * set, PA_ERR_CUDA if the synchronisation failed, else PA_OK. */
PA_API pa_status pa_get_device_error(pa_pool* pool, void* stream, uint32_t* flags);

/* Diagnostic of the failure detection: run, on `device`, one bounded device
 * wait that cannot complete (an mbarrier that nothing arrives at, given up
 * after about limit_cycles SM clocks, the way every kernel wait of this
 * library gives up) and return the error bits it recorded in *flags:
 * PA_DEVERR_TIMEOUT when the wait expired and reported. Synchronous; the
 * device stays usable afterwards.
 * Errors: PA_ERR_INVALID_ARG (null flags, device < 0, limit outside
 * [1, 4e9]; nothing launched), PA_ERR_CUDA. */
PA_API pa_status pa_selftest_wait_timeout(int32_t device, int64_t limit_cycles, uint32_t* flags);

/* Bandwidth calibration, not part of the decode path: read `bytes` bytes at
 * `src` with 16-byte streaming loads spread over every SM of the current
 * device, folding them into one 32-bit word that is OR-ed into *sink only in
 * the (practically never taken) case that it equals a fixed constant, so that
 * no load can be dropped and nothing is written otherwise. Timed beside the
 * decode call, it gives the time of the simplest kernel that reads the same
 * number of bytes: the ceiling that one launch of that size can reach.
 *   src    device, 16-byte aligned; bytes a multiple of 16
 *   sink   device uint32_t
 * Asynchronous on `stream` (a cudaStream_t; NULL = the default stream).
 * Errors: PA_ERR_INVALID_ARG (null pointer, misaligned src, bytes not a
 * multiple of 16; nothing launched), PA_ERR_CUDA. */
PA_API pa_status pa_stream_read(const void* src, size_t bytes, uint32_t* sink, void* stream);

/* Static description of a status code. */
PA_API const char* pa_status_string(pa_status s);

/* Message of the last failed call on this thread ("" if none). */
PA_API const char* pa_last_error(void);

/* ---- Host block manager (which physical blocks hold which sequence's tokens)
 *
 * Host-side bookkeeping for a pool's physical blocks (TFFInfer article,
 * section 3.6.4 KVCache: PageManager; heterogeneous engine article, section
 * 2.3 paged KV and its prefix sharing): a free list, each sequence's block
 * table (token t in slot t % block_size of table[t / block_size]), reference
 * counts for blocks that sequences share, and
 *  - a prefix cache: a full block is known by the chained hash of the token
 *    ids of all blocks up to it; a sequence admitted with a prompt whose
 *    leading full blocks are cached shares those blocks, whose KV is already
 *    written (with an unmatched prompt's full blocks entered into the cache
 *    when admitted: the caller writes their KV before any later reader runs
 *    on the same stream);
 *  - fork: a child shares all of its parent's blocks;
 *  - copy-on-write: before a sequence writes into a partly filled block that
 *    another sequence also holds, the block is replaced by a private one and
 *    a (src, dst) pair is returned for the caller to copy (pa_copy_blocks).
 * Blocks no sequence holds that are cached stay cached and are reused least
 * recently released first. Host memory only, no device work; not
 * thread-safe (one manager per scheduling thread). Token ids may be NULL when
 * the prefix cache is off. Calls that fail (PA_ERR_INVALID_ARG, or
 * PA_ERR_OOM when the blocks run out) change nothing. */
typedef struct pa_block_manager pa_block_manager;
PA_API pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_cache,
                              pa_block_manager** out);
PA_API pa_status pa_bm_destroy(pa_block_manager* bm);
/* Admit sequence `seq_id` holding `n_tokens` prompt tokens; *n_cached_tokens
 * (optional) receives how many leading tokens are in shared cached blocks
 * (a multiple of block_size), whose KV need not be written again. */
PA_API pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                                    int32_t n_tokens, int32_t* n_cached_tokens);
PA_API pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);
/* Reserve slots for `n_tokens` more tokens of a sequence (a decode step: 1).
 * At most one copy is returned (the shared partly filled last block); the
 * caller copies it before writing. Blocks this call fills join the cache. */
PA_API pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                                     int32_t n_tokens, int32_t* copy_src, int32_t* copy_dst,
                                     int32_t copy_capacity, int32_t* n_copies);
PA_API pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id);
/* The sequence's block table into table[0 .. max_blocks) (-1 padded), its
 * block count and token count (each optional). PA_ERR_INVALID_ARG when the
 * table does not fit (the counts are still written). */
PA_API pa_status pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* table,
                                   int32_t max_blocks, int32_t* num_blocks, int64_t* seq_len);
/* Blocks that can be handed out: free ones plus cached ones nobody holds. */
PA_API int32_t pa_bm_num_free_blocks(const pa_block_manager* bm);
/* Sequences holding `block` (-1 for a bad id). */
PA_API int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block);

/* CPU swap tier (engine article, section 4.3: the block manager's swap_out
 * moves GPU blocks to a CPU second-level cache, swap_in brings them back).
 * The caller owns a host buffer of num_cpu_blocks slots of
 * pa_pool_block_bytes each and applies each returned copy list with
 * pa_swap_blocks, in call order on one stream.
 *  - pa_bm_set_cpu_blocks: size the host tier (slots 0 .. n-1); refused
 *    while any slot is in use.
 *  - pa_bm_swap_out: every block of a resident sequence is copied to a slot
 *    of its own (gpu_src[i] -> cpu_dst[i], i < *n_copies) and released on
 *    the GPU (blocks other sequences hold stay; an idle cached block stays
 *    cached). The sequence is then swapped out: append, fork and block table
 *    are refused for it until pa_bm_swap_in.
 *  - pa_bm_swap_in: fresh GPU blocks for each slot (cpu_src[i] ->
 *    gpu_dst[i]); the slots are freed.
 *  - pa_bm_swapped_slots: a swapped-out sequence's slots, in token order.
 * Capacities are in entries; PA_ERR_OOM when slots or blocks run out, and
 * failed calls change nothing. Freeing a swapped-out sequence frees its
 * slots. */
PA_API pa_status pa_bm_set_cpu_blocks(pa_block_manager* bm, int32_t num_cpu_blocks);
PA_API int32_t pa_bm_num_free_cpu_blocks(const pa_block_manager* bm);
PA_API pa_status pa_bm_swap_out(pa_block_manager* bm, int64_t seq_id, int32_t* gpu_src, int32_t* cpu_dst,
                                int32_t capacity, int32_t* n_copies);
PA_API pa_status pa_bm_swap_in(pa_block_manager* bm, int64_t seq_id, int32_t* cpu_src, int32_t* gpu_dst,
                               int32_t capacity, int32_t* n_copies);
PA_API pa_status pa_bm_swapped_slots(const pa_block_manager* bm, int64_t seq_id, int32_t* slots,
                                     int32_t capacity, int32_t* n_slots);

/* Device: copy whole blocks (the page records of every kv head) src[i] ->
 * dst[i] in a pool, for copy-on-write. src, dst: host arrays of n block ids,
 * src[i] != dst[i]. Enqueued on `stream`. */
PA_API pa_status pa_copy_blocks(pa_pool* pool, const int32_t* src, const int32_t* dst, int32_t n, void* stream);

/* Bytes of one block's page records (all kv heads): the size of a host slot
 * of the swap tier. 0 for a NULL pool. */
PA_API size_t pa_pool_block_bytes(const pa_pool* pool);

/* Device <-> host: copy whole blocks between the pool and a caller-owned host
 * buffer of num_host_blocks slots of pa_pool_block_bytes each (pinned memory
 * for asynchronous copies). direction PA_SWAP_OUT copies block blocks[i] to
 * slot slots[i], PA_SWAP_IN slot slots[i] to block blocks[i]. blocks, slots:
 * host arrays of n ids. One cudaMemcpyAsync per block, enqueued on `stream`;
 * the caller keeps the buffer alive until they complete.
 * Errors: PA_ERR_INVALID_ARG (null pool or buffer, ids out of range, unknown
 * direction; nothing enqueued), PA_ERR_CUDA. */
#define PA_SWAP_OUT 0
#define PA_SWAP_IN 1
PA_API pa_status pa_swap_blocks(pa_pool* pool, void* host_buffer, int32_t num_host_blocks,
                                const int32_t* blocks, const int32_t* slots, int32_t n, int32_t direction,
                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
