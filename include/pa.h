/*
 * pa.h -- C ABI of libpa.so: paged KV cache decode on one GB300 (sm_103a).
 *
 * Method sources (page title, section):
 *   [PA] "論文解説: PagedAttention — 仮想メモリ着想のKVキャッシュ管理でLLMサービングを高効率化"
 *   [VA] "論文解説: vAttention - PagedAttentionを使わないLLMサービング向け動的メモリ管理"
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every call returns a pa_status; nothing crosses the ABI as an exception.
 *   On a non-OK status pa_last_error() holds a message (per calling thread).
 * - Device calls take device pointers owned by the caller, enqueue work on
 *   `stream` (a cudaStream_t; NULL = the legacy default stream) and return
 *   without synchronising.  They allocate no device memory: scratch space is
 *   a caller-provided workspace.  Pointers must be 16-byte aligned.
 * - Out-of-range arguments that the host can see are rejected, never clamped
 *   (the vAttention explainer's request-offset helper raises on an identifier
 *   outside [0, max_batch); the same rule is applied throughout).
 * - Indices that live in device memory (slots, block-table entries, context
 *   lengths, request ids, copy pairs) are checked by the kernels: an offending
 *   element is skipped, and when `dev_err` is non-NULL the kernel ORs a
 *   PA_DEV_ERR_* bit into *dev_err (a device int the caller zeroes and reads
 *   back).  No kernel traps, and no kernel waits without a time limit: a wait
 *   that exceeds about one second sets PA_DEV_ERR_TIMEOUT and the kernel
 *   returns.
 *
 * Data layout
 * -----------
 * KV pool: [NB][B][2][H_kv][D] elements of `kv_dtype`; index 0 on the third
 * axis is K, 1 is V (the explainer's kv_cache of shape (blocks, B, 2, d),
 * widened to H_kv heads).  Token position t of a sequence lives in logical
 * block t / B at offset t % B; its slot is physical_block * B + t % B.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,     /* bad argument (shape, range, alignment, unknown id) */
    PA_ERR_OOM = 2,         /* the block allocator has too few free blocks; state unchanged */
    PA_ERR_STATE = 3,       /* the allocator's state forbids the operation (e.g. refcount underflow) */
    PA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed; message in pa_last_error() */
    PA_ERR_UNSUPPORTED = 5  /* valid but not built: dtype / head dim / block size / group size */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2 } pa_dtype;

/* Bits a kernel ORs into *dev_err. */
#define PA_DEV_ERR_SLOT 0x1      /* slot_mapping entry >= NB*B */
#define PA_DEV_ERR_BLOCK 0x2     /* block-table entry or copy pair outside [0, NB), or chained copy pairs */
#define PA_DEV_ERR_CTX 0x4       /* context length < 1, > max_ctx or > MB*B */
#define PA_DEV_ERR_REQ 0x8       /* request id outside [0, N_max) */
#define PA_DEV_ERR_TIMEOUT 0x10  /* a bounded wait inside a kernel ran out */

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* pa_last_error(void);

/* Library version string. */
const char* pa_version(void);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t pa_launch_count(void);

/* Time limit, in nanoseconds, of every wait inside the kernels launched from
 * now on by any thread (the watchdog of "no kernel waits without a time
 * limit" above); 0 restores the built-in 1 s.  A wait that runs out sets
 * PA_DEV_ERR_TIMEOUT and the kernel returns, leaving that call's outputs
 * undefined; before returning it still waits, with the built-in limit, for
 * the copies and tensor-core products it has issued, so the next call finds
 * the GPU and the caller's buffers usable.  A very short limit makes the
 * waits run out on purpose, which is how the timeout exit is tested. */
void pa_set_wait_limit_ns(uint64_t ns);

/* ------------------------------------------------------------------------
 * Cache write ([PA] 技術的詳細 / PagedAttentionアルゴリズム: tokens are stored in
 * fixed-size blocks reached through the block table; the slot encoding
 * physical_block * B + offset is this library's).
 * k, v: [T][H_kv][D] of dtype; pool: [NB][B][2][H_kv][D] of dtype;
 * slot_mapping: [T] int64.  Token i's K and V rows are copied bit for bit to
 * pool[slot / B][slot % B][0] and [1].  slot < 0 skips the token (padding);
 * slot >= NB*B is skipped and flagged PA_DEV_ERR_SLOT.  Two tokens with the
 * same slot race (caller error).  T == 0 is a no-op.
 * Supported: dtype F16/BF16, (H_kv * D) a multiple of 8.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(const void* k, const void* v, void* pool, const int64_t* slot_mapping, int T, int NB,
                               int B, int H_kv, int D, pa_dtype dtype, int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Copy-on-write block copy ([PA] 技術的詳細 / Copy-on-Write KVキャッシュ共有:
 * a block shared by several sequences is copied before one of them writes).
 * pairs: [n][2] int64 (src, dst), device memory.  pool[dst] = pool[src] for
 * whole blocks (B * 2 * H_kv * D elements), bit for bit.  The pairs must not
 * chain: destinations are distinct and no destination is also a source in the
 * same call (flagged PA_DEV_ERR_BLOCK if violated; the copies then race).
 * A pair with an index outside [0, NB) is skipped and flagged.  n == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_copy_blocks(void* pool, const int64_t* pairs, int n, int NB, int B, int H_kv, int D, pa_dtype dtype,
                         int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Block swap between two pools ([PA] 実装のポイント: under memory pressure the
 * scheduler preempts a request and either swaps its KV cache to CPU memory
 * or recomputes it later; this is the swap copy, in both directions).
 * dst_pool: [NB_dst][B][2][H_kv][D], src_pool: [NB_src][B][2][H_kv][D]; each
 * is device memory or page-locked host memory (cudaHostAlloc, or pinned with
 * cudaHostRegister; with unified addressing its host pointer is used as is).
 * Pageable host memory is rejected with PA_ERR_INVALID.
 * pairs: [n][2] int64 (src block, dst block), in device or page-locked host
 * memory.  dst_pool[dst] = src_pool[src] for whole blocks, bit for bit, moved
 * by the GPU's own loads and stores (no per-block memcpy calls).  A pair
 * outside [0, NB_src) x [0, NB_dst) is skipped and flagged PA_DEV_ERR_BLOCK;
 * destinations must be distinct.  For copies inside one pool use
 * pa_copy_blocks.  n == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_swap_blocks(void* dst_pool, int NB_dst, const void* src_pool, int NB_src, const int64_t* pairs, int n,
                         int B, int H_kv, int D, pa_dtype dtype, int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Incremental block-table update ([VA] 背景と動機: preparing block tables on
 * the CPU took a large share of a vLLM decode iteration; the tables stay on
 * the device and only changed entries travel).
 * tables: [N][MB] int32 device memory; updates: [n][3] int32 device memory
 * (row, logical block, physical block), as pa_alloc_append_batch emits them.
 * Sets tables[row][logical block] = physical block.  An entry with a negative
 * row is padding and is skipped (so a fixed-size update list can be captured
 * in a CUDA graph); entries with row >= N or logical block outside [0, MB)
 * are skipped and flagged PA_DEV_ERR_BLOCK.  Two updates of the same entry
 * race (the allocator never emits that).  n == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status pa_update_block_tables(int32_t* tables, int N, int MB, const int32_t* updates, int n, int* dev_err,
                                 void* stream);

/* ------------------------------------------------------------------------
 * Workspace for pa_decode / pa_decode_contiguous, in bytes.
 * partition_tokens: 0 = default (512), -1 = one partition per sequence,
 * > 0 = split each context into partitions of that many tokens (a multiple
 * of 32).  max_ctx bounds every context length of the calls that use the
 * workspace.  Returns 0 for invalid arguments.
 * ---------------------------------------------------------------------- */
size_t pa_decode_workspace_bytes(int N, int H_q, int H_kv, int D, int max_ctx, int partition_tokens);

/* ------------------------------------------------------------------------
 * Paged decode attention ([PA] 技術的詳細 / PagedAttentionアルゴリズム, decode
 * equation; アルゴリズムの擬似コード for the block-by-block online softmax).
 * For every sequence s < N and query head h < H_q, with g = h / (H_q / H_kv):
 *     x_t = scale * (q[s][h] . K_t),  t = 0 .. ctx_lens[s]-1,
 *     out[s][h] = sum_t softmax(x)_t * V_t,
 * K_t, V_t = pool[block_tables[s][t / B]][t % B][0 / 1][g].
 *
 * out: [N][H_q][D] of out_dtype (F32, F16 or BF16), in device memory or in
 * pinned host memory (cudaHostAlloc / cudaHostRegister, addressed through the
 * same pointer): the kernels then write each output row across the host link
 * as it completes, which replaces a separate device-to-host copy of the
 * result; q: [N][H_q][D] of kv_dtype;
 * block_tables: [N][MB] int32 (entries past ceil(ctx/B) are not read);
 * ctx_lens: [N] int32 in [1, min(max_ctx, MB*B)];
 * scale: usually 1/sqrt(D).
 * Long contexts are split into partitions of partition_tokens (see
 * pa_decode_workspace_bytes); partitions are merged by the same kernel that
 * pa_partition_reduce runs.  workspace: ws_bytes >= pa_decode_workspace_bytes(...)
 * of device memory, contents need not be initialised, and must not be used by
 * another call that overlaps on the GPU.
 * attend_events: NULL, or a pointer to two cudaEvent_t that are recorded on
 * `stream` immediately before and after the attention kernel (for timing it
 * apart from the scheduling and merge kernels).
 * Supported: kv_dtype F16/BF16, D in {64, 128}, B in {4, 8, 16, 32},
 * 1 <= H_q / H_kv <= 8, NB*B < 2^31.
 * ---------------------------------------------------------------------- */
pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* pool, const int32_t* block_tables,
                    const int32_t* ctx_lens, int N, int H_q, int H_kv, int D, int B, int MB, int NB, int max_ctx,
                    float scale, int partition_tokens, void* workspace, size_t ws_bytes, pa_dtype kv_dtype,
                    int* dev_err, void* const* attend_events, void* stream);

/* ------------------------------------------------------------------------
 * The same attention over contiguous per-request buffers ([VA] 技術的詳細 /
 * リクエスト単位のKVキャッシュインデキシング: request r's cache is the sub-tensor
 * starting at r * S, S = max context * H_kv * D elements).
 * k_buf, v_buf: [N_max][S_max][H_kv][D] of kv_dtype; req_ids: [N] int32 in
 * [0, N_max) (out-of-range ids are flagged PA_DEV_ERR_REQ and their rows are
 * not written); ctx_lens[s] <= S_max.  Other arguments as pa_decode.
 * ---------------------------------------------------------------------- */
pa_status pa_decode_contiguous(void* out, pa_dtype out_dtype, const void* q, const void* k_buf, const void* v_buf,
                               const int32_t* req_ids, const int32_t* ctx_lens, int N, int H_q, int H_kv, int D,
                               int N_max, int S_max, int max_ctx, float scale, int partition_tokens, void* workspace,
                               size_t ws_bytes, pa_dtype kv_dtype, int* dev_err, void* const* attend_events,
                               void* stream);

/* ------------------------------------------------------------------------
 * Causal paged prefill attention ([PA] 実装のポイント: the paged kernel serves
 * the prefill phase as well as decode).  Sequence s holds ctx_lens[s] tokens
 * in the pool, the last q_len_s = q_start[s+1] - q_start[s] of them being the
 * chunk whose queries are rows q_start[s] .. q_start[s+1]-1 of q.  Query i of
 * the chunk sits at position p = ctx - q_len + i and attends causally:
 *     out[row][h] = sum_{t <= p} softmax_t(scale * q[row][h] . K_t) V_t.
 * The chunk's own K/V must already be in the pool (pa_reshape_and_cache).
 * q, out: [T][H_q][D] (out fp32 or the kv dtype); q_start: [N+1] int32 with
 * q_start[0] = 0 and q_start[N] = T; max_q_len >= every chunk length.
 * Runs on the tensor cores (tcgen05, accumulators in TMEM).  A chunk longer
 * than its context is flagged PA_DEV_ERR_CTX and not computed.
 * workspace (nullable), ws_bytes >= pa_prefill_workspace_bytes(N, H_kv, D, B,
 * MB) of device memory: with a bf16 cache a first kernel stages each
 * sequence's V there as fp16, so the value product takes P in fp16, one
 * product per key instead of two (the staging kernel's time is part of the
 * call).  The conversion is exact: a (sequence, KV head) holding a V
 * magnitude >= 65536, or a group of 32 keys with only magnitudes < 2^-10,
 * is computed as without a workspace instead.  Without a
 * workspace a bf16 cache takes P as a high and a low bf16 part (two products,
 * the same precision).  fp16 caches ignore the workspace.  The workspace's
 * contents need not be initialised; calls that overlap on the GPU must not
 * share one.  Rows with an fp16 value product run on a persistent kernel
 * over 256-key tiles (2-CTA clusters), the others on a kernel with two query
 * tiles per CTA; the environment variable PA_PREFILL_KERNEL=narrow puts
 * every row on the second (results differ only by rounding order).
 * Supported: kv_dtype F16/BF16, D in {64, 128}, B in {8, 16, 32},
 * H_q / H_kv <= 128, N <= 65535, scale > 0.  out, q, pool and workspace must
 * be 16-byte aligned, an fp32 out 32-byte aligned (PA_ERR_INVALID otherwise).
 * ---------------------------------------------------------------------- */
size_t pa_prefill_workspace_bytes(int N, int H_kv, int D, int B, int MB);
pa_status pa_prefill(void* out, pa_dtype out_dtype, const void* q, const void* pool, const int32_t* block_tables,
                     const int32_t* ctx_lens, const int32_t* q_start, int N, int T, int H_q, int H_kv, int D, int B,
                     int MB, int NB, int max_q_len, float scale, pa_dtype kv_dtype, void* workspace, size_t ws_bytes,
                     int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * pa_decode without a caller-provided workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory where they decode (a plug-in inside a framework that owns every
 * allocation, a serving loop that must not allocate after start-up, an engine
 * that has already carved up all of HBM).  Arguments and results are those of
 * pa_decode minus `workspace` / `ws_bytes`.
 * - Scratch space: a file-scope device array of PA_STATIC_WORKSPACE_BYTES
 *   (32 MiB) inside libpa.so.  Every GPU that loads the library holds it until
 *   the process exits.  A batch whose pa_decode_workspace_bytes(...) exceeds
 *   it is rejected with PA_ERR_UNSUPPORTED and a message; nothing is launched.
 * - The first call on a device looks up the array's device address for that
 *   device (cudaGetSymbolAddress with the device current) and caches it with
 *   the context's unique ID; the first call after the context is torn down
 *   (cudaDeviceReset) looks it up again.  Make that first call before any
 *   stream capture.  The call allocates nothing.
 * - All calls share the one array and it keeps the last call's contents; the
 *   kernels rewrite every part of it they read, so nothing needs clearing.
 *   Calls that overlap on the GPU (different streams, or threads) race on it:
 *   order them on one stream or use pa_decode with separate workspaces.
 * ---------------------------------------------------------------------- */
#define PA_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)
pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q, const void* pool,
                             const int32_t* block_tables, const int32_t* ctx_lens, int N, int H_q, int H_kv, int D,
                             int B, int MB, int NB, int max_ctx, float scale, int partition_tokens,
                             pa_dtype kv_dtype, int* dev_err, void* const* attend_events, void* stream);

/* ------------------------------------------------------------------------
 * Cache write for the contiguous per-request layout ([VA] リクエスト単位のKV
 * キャッシュインデキシング: request r's cache starts at r * S).
 * k, v: [T][H_kv][D]; k_buf, v_buf: [N_max][S_max][H_kv][D].  Token i's rows go
 * to request req_ids[i] at position positions[i]; req_ids[i] < 0 skips the
 * token; a request id >= N_max is flagged PA_DEV_ERR_REQ and a position
 * outside [0, S_max) PA_DEV_ERR_SLOT (both skipped).  With pa_vkv buffers the
 * position must lie inside the pages pa_vkv_step has mapped.
 * ---------------------------------------------------------------------- */
pa_status pa_write_contiguous(const void* k, const void* v, void* k_buf, void* v_buf, const int32_t* req_ids,
                              const int32_t* positions, int T, int N_max, int S_max, int H_kv, int D, pa_dtype dtype,
                              int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Virtually contiguous KV buffers with physical pages mapped on demand
 * ([VA] 技術的詳細: reserve the virtual range up front with cuMemAddressReserve,
 * back it with physical pages through cuMemCreate + cuMemMap as contexts grow;
 * 実装のポイント: the init / alloc_reqid / step / free_reqid interface; free
 * keeps the pages mapped for the slot's next owner, the explainer's deferred
 * reclamation).  Page size is the driver's minimum granularity (2 MB on this
 * hardware; the explainer's 64 KB pages need a modified driver and are not
 * used).  Buffers of layer l: K and V, each [max_batch][S][H_kv][D] where
 * S = *S_tokens >= max_ctx (a whole number of pages per request); pass
 * N_max = max_batch and S_max = S to pa_decode_contiguous / pa_write_contiguous.
 * Host calls, one device (the device current at create); not thread-safe.
 * - pa_vkv_create reserves 2 * num_layers ranges, maps nothing.
 * - pa_vkv_alloc_reqid picks a free request slot (one that still has pages
 *   first); PA_ERR_OOM when all max_batch are taken.
 * - pa_vkv_step maps pages so request req_ids[i] covers ctx_lens[i] tokens
 *   (rounded up to 32, the decode kernel's read granule) in every buffer; a
 *   request whose pages cannot be created is left as it was and PA_ERR_OOM
 *   returned (requests before it in the list keep their new pages).
 * - pa_vkv_free_reqid releases the slot, not its pages; pa_vkv_reclaim unmaps
 *   the pages of every free slot.
 * ---------------------------------------------------------------------- */
pa_status pa_vkv_create(int num_layers, int max_batch, int max_ctx, int H_kv, int D, pa_dtype dtype, void** out);
void pa_vkv_destroy(void* vkv);
/* k_bufs, v_bufs: [num_layers] device pointers (nullable); S_tokens: request stride in tokens;
 * page_bytes: physical page size. */
pa_status pa_vkv_info(void* vkv, void** k_bufs, void** v_bufs, int64_t* S_tokens, int64_t* page_bytes);
pa_status pa_vkv_alloc_reqid(void* vkv, int* req_id);
pa_status pa_vkv_step(void* vkv, const int32_t* req_ids, const int32_t* ctx_lens, int n);
pa_status pa_vkv_free_reqid(void* vkv, int req_id);
pa_status pa_vkv_reclaim(void* vkv);
pa_status pa_vkv_mapped_pages(void* vkv, int req_id, int* pages);

/* ------------------------------------------------------------------------
 * Merge of split-context partials (the running maximum / exponential sum /
 * unnormalised output the block-by-block online softmax keeps, [PA]
 * アルゴリズムの擬似コード, taken per partition and combined).
 * Row r has nparts[r] in [1, P] partitions; part_m2, part_l: [R][P] fp32,
 * part_acc: [R][P][D] fp32.  m2 is the partition's maximum score in base-2
 * units (max_t x_t * log2 e); l = sum_t 2^(x_t log2 e - m2);
 * acc = sum_t 2^(x_t log2 e - m2) V_t.
 *     M = max_p m2_p,  out[r] = sum_p 2^(m2_p - M) acc_p / sum_p 2^(m2_p - M) l_p.
 * out: [R][D] of out_dtype.  D in {64, 128}.  Rows with nparts outside
 * [1, P] are not written and are flagged PA_DEV_ERR_CTX.
 * ---------------------------------------------------------------------- */
pa_status pa_partition_reduce(void* out, pa_dtype out_dtype, const float* part_m2, const float* part_l,
                              const float* part_acc, const int32_t* nparts, int R, int P, int D, int* dev_err,
                              void* stream);

/* ------------------------------------------------------------------------
 * Host block allocator ([PA] 技術的詳細 / PagedAttentionアルゴリズム and
 * Copy-on-Write KVキャッシュ共有; 実装のポイント: one slab, the library's own
 * allocator).  An opaque handle owned by the library; pa_alloc_destroy frees it.
 * Not thread-safe: one thread per handle at a time.
 * - Free list: a LIFO stack.  initial_free_order (nullable = 0..NB-1) lists
 *   block ids in hand-out order.  Freeing pushes a sequence's blocks in
 *   logical order.
 * - Appending token position pos: if pos % B == 0 a free block is appended to
 *   the table; otherwise, if the last block's reference count is above one, a
 *   free block replaces it, (old, new) is emitted as a copy pair and the old
 *   count drops by one (copy before write).  Slot = block * B + pos % B.
 * - Every call is all-or-nothing: PA_ERR_OOM and PA_ERR_INVALID leave the
 *   state unchanged.
 * ---------------------------------------------------------------------- */
pa_status pa_alloc_create(int NB, int B, const int32_t* initial_free_order, void** out);
void pa_alloc_destroy(void* alloc);
pa_status pa_alloc_add_seq(void* alloc, int seq_id);                 /* new empty sequence, seq_id >= 0 */
/* Append n tokens to seq_id.  slots_out: [n]; cow_pairs_out: [cow_cap][2]
 * (at most one pair per call); *n_cow receives the pair count. */
pa_status pa_alloc_append_slots(void* alloc, int seq_id, int n, int64_t* slots_out, int64_t* cow_pairs_out,
                                int cow_cap, int* n_cow);
/* Append n_tokens[i] tokens to each of n_seqs distinct sequences, in order.
 * slots_out: [sum n_tokens]; cow_pairs_out: [cow_cap][2].
 * table_updates_out (nullable): [upd_cap][3] int32 triples (row i of the
 * batch, logical block, physical block), one per block-table entry the call
 * sets (each new block and each copy-on-write replacement), in order; *n_upd
 * receives their count.  Feeding them to pa_update_block_tables keeps a
 * device copy of the batch's tables ([n_seqs][MB], rows in seq_ids order)
 * current without re-uploading it. */
pa_status pa_alloc_append_batch(void* alloc, int n_seqs, const int32_t* seq_ids, const int32_t* n_tokens,
                                int64_t* slots_out, int64_t* cow_pairs_out, int cow_cap, int* n_cow,
                                int32_t* table_updates_out, int upd_cap, int* n_upd);
pa_status pa_alloc_fork(void* alloc, int parent, int child);          /* child shares all parent blocks */
pa_status pa_alloc_free_seq(void* alloc, int seq_id);                 /* drop references, recycle blocks */
pa_status pa_alloc_block_table(void* alloc, int seq_id, int32_t* out, int cap, int* n);
/* Pack the tables of n_seqs sequences into out[n_seqs][MB] (unused entries
 * -1) and their lengths into ctx_out[n_seqs] (nullable). */
pa_status pa_alloc_block_tables(void* alloc, int n_seqs, const int32_t* seq_ids, int32_t* out, int MB,
                                int32_t* ctx_out);
pa_status pa_alloc_seq_len(void* alloc, int seq_id, int64_t* out);
pa_status pa_alloc_refcount(void* alloc, int block, int* out);
int pa_alloc_num_free(void* alloc);                                   /* -1 for a NULL handle */
pa_status pa_alloc_free_list(void* alloc, int32_t* out, int cap, int* n); /* next block to hand out first */
/* Checkpoint / resume of the whole allocator state as a flat int64 array:
 * {tag, NB, B, nfree, nseq, free stack (bottom first)[nfree], refcounts[NB],
 * then per sequence in increasing id: id, tokens, nblocks, blocks[nblocks]}.
 * pa_alloc_export writes *n words (out NULL: only *n; cap < *n:
 * PA_ERR_INVALID).  pa_alloc_import builds a new handle from such an array
 * after checking it: every block is either free (listed once, count 0) or
 * counted exactly as often as the tables name it, and every table has
 * ceil(tokens / B) blocks; anything else is PA_ERR_INVALID. */
pa_status pa_alloc_export(void* alloc, int64_t* out, size_t cap, size_t* n);
pa_status pa_alloc_import(const int64_t* in, size_t n, void** out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
