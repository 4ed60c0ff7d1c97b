/*
 * pagedkv.h -- C ABI of libpagedkv.so: paged decode attention on GB300 (sm_103a).
 *
 * The operations follow three descriptions of PagedAttention:
 *   [S]  "Efficient Memory Management for Large Language Model Serving with
 *        PagedAttention" (azimuth.plus summary of Kwon et al., SOSP 2023):
 *        sections "Core idea", "The PagedAttention algorithm" (block-wise
 *        attention equation), "vLLM" (block manager), "Memory sharing"
 *        (copy-on-write), "Inside: block-table lookup".
 *   [T]  CSDN tutorial "PagedAttention实战": §2.1 Page / PageTable, §2.2
 *        BlockManager, §3.1 SequenceManager.append_kv, §3.2 PagedAttention.compute,
 *        §5.1 clone_sequence.
 *   [K]  Bidirectional KV-cache transfer for multi-turn prefill/decode-disaggregated
 *        vLLM (spke.com translation of an AWS blog post): sections "Bidirectional
 *        KV transfer" (KV blocks move between the nodes' pools) and "KV recompute
 *        threshold" (default 64 tokens).
 *
 * Conventions shared by every entry point
 *   - All device buffers are allocated and owned by the caller.  The library never
 *     allocates device memory and keeps no per-call state between calls.
 *   - Device work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     an opaque pointer; NULL = the legacy default stream).  Inputs must stay alive
 *     and unmodified until the stream has executed the call.
 *   - Arguments are validated on the host before anything is enqueued: a status
 *     other than PA_OK means nothing was enqueued.  PA_ERR_CUDA reports a failed
 *     launch (the CUDA error is cleared; pa_last_cuda_error returns it).
 *   - No entry point aborts, exits or throws.
 *   - Layouts are dense row-major, all with the innermost dimension contiguous:
 *       q, out                [num_seqs][num_q_heads][head_dim]
 *       k_cache, v_cache      [num_blocks][block_size][num_kv_heads][head_dim]
 *                              ([T] §2.1: a page holds keys/values of shape
 *                               [page_size, num_heads, head_dim])
 *       block_tables          int32 [num_seqs][max_blocks_per_seq]; entry j of row s
 *                             is the physical block of logical block j ([S] "Core
 *                             idea": the block table maps logical to physical blocks);
 *                             entries at j >= ceil(context_len / block_size) are not
 *                             read (pad them with -1, [T] §2.1's unmapped value)
 *       context_lens          int32 [num_seqs]
 *       slot_mapping          int64 [num_tokens]: slot = physical_block * block_size
 *                             + offset ([T] §3.1)
 *       src_dst_pairs         int32 [num_pairs][2]
 *   - Device pointers must be 16-byte aligned (PA_ERR_INVALID otherwise).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* bad pointer, shape, alignment or argument       */
    PA_ERR_UNSUPPORTED = 2,  /* valid but not built (head_dim, block_size, ...)  */
    PA_ERR_CUDA = 3,         /* a CUDA call or launch failed                     */
    PA_ERR_OOM = 4,          /* host allocator: no free block ([T] §2.2)         */
    PA_ERR_TIMEOUT = 5       /* a device-side wait gave up (pa_device_errors)    */
} pa_status;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* Human-readable name of a status; never NULL. */
const char *pa_status_string(pa_status s);

/* The CUDA error code of the last PA_ERR_CUDA returned on this thread (0 if none). */
int pa_last_cuda_error(void);

/* ------------------------------------------------------------------------- *
 * Decode attention.                                                          *
 * ------------------------------------------------------------------------- */

/*
 * pa_decode -- single-query attention of every sequence over its paged KV cache.
 *
 * Defines ([S] "The PagedAttention algorithm", block-wise attention equation; [T]
 * §3.2): for sequence s with T = context_lens[s] tokens and query head h,
 *     kv   = h / (num_q_heads / num_kv_heads)          (contiguous GQA groups)
 *     K_t  = k_cache[block_tables[s][t / B]][t % B][kv][:]   (same for V_t)
 *     s_t  = scale * dot(q[s][h], K_t)
 *     out[s][h] = sum_t exp(s_t - max) V_t / sum_t exp(s_t - max)
 * computed block by block with per-block maxima and exp-sums merged by the
 * log-sum-exp rule the equation states.  Only the first T - (nb-1)*B rows of the
 * last block count; stale rows past T never affect the result.  T = 0 yields a zero
 * row ([T] §3.2 returns zeros for an empty sequence).  Context lengths are clamped
 * to [0, max_blocks_per_seq * block_size].
 *
 * Long contexts are split so that several CTAs share one sequence; their partial
 * (max, exp-sum, weighted V) results are merged with the same rule.
 * partition_size selects the split:
 *   0      balanced split: the K/V of all (sequence, kv head) pairs is cut into
 *          equal shares, one per CTA of a persistent grid, so every CTA streams
 *          about the same number of bytes whatever the length mix; the CTA that
 *          completes a split pair's partials merges them (one kernel launch);
 *   > 0    fixed partitions of partition_size tokens (a multiple of block_size),
 *          merged by a second kernel.
 * Both give the same result up to fp32 rounding order.  The workspace needs no
 * initialisation: the balanced split's merge counters are tagged with a
 * per-call epoch, and a completed call leaves them at zero, so the replays of a
 * captured CUDA graph (which reuse the captured epoch) each start clean.  After a
 * device timeout (pa_device_errors), clear a graph's workspace before replaying.
 *
 * Arguments
 *   out            device, [S][Hq][d], dtype `dtype`, written
 *   q              device, [S][Hq][d], dtype `dtype`
 *   k_cache/v_cache device, [num_blocks][B][Hkv][d], dtype `dtype`; two separate
 *                  buffers or one.  When v_cache lies above k_cache, a multiple of
 *                  16 bytes and less than 2^40 bytes away (for instance both halves
 *                  of one [2][num_blocks][B][Hkv][d] buffer), every block's K and V
 *                  tiles arrive with one copy instead of two, which streams faster;
 *                  the results are the same either way.
 *   block_tables   device int32 [S][max_blocks_per_seq]; referenced entries must be
 *                  in [0, num_blocks) (an entry outside reads zeros, never faults)
 *   context_lens   device int32 [S]
 *   scale          softmax scale (1/sqrt(head_dim) for the pages' definition)
 *   head_dim       64 or 128;  block_size 16 or 32;  num_q_heads % num_kv_heads == 0
 *   workspace      device scratch of at least pa_decode_workspace_size(...) bytes
 *                  (may be NULL when that size is 0); 16-byte aligned.  Its
 *                  contents need no initialisation and are not meaningful after.
 * Errors: PA_ERR_INVALID (null/misaligned pointer, non-positive size, bad
 *   partition size, workspace too small, q/kv head mismatch, num_blocks*block_size
 *   >= 2^31), PA_ERR_UNSUPPORTED (head_dim / block_size / dtype not built),
 *   PA_ERR_CUDA (launch failure).
 */
pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int num_seqs, int num_blocks, float scale,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    pa_dtype dtype, int partition_size, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * pa_decode_append -- append each sequence's newest token and decode, in one launch.
 *
 * Same result as pa_reshape_and_cache of the newest tokens followed by pa_decode
 * ([T] §3.1 append_kv then §3.2 compute, the per-step loop of [T] §4): for every
 * sequence s with T = context_lens[s] >= 1, position T - 1 is the new token; its
 * K and V rows are k_new[s], v_new[s] ([S][Hkv][d], dtype `dtype`).  They are
 * written into the caches at that position's slot (block_tables[s][(T-1)/B] * B +
 * (T-1) % B, which the allocator's pa_alloc_append returned), and the attention
 * over positions 0 .. T-1 uses them.  Copy-on-write pairs of the step must be
 * applied (pa_copy_blocks) before the call.  Sequences with T = 0 write nothing
 * and yield zeros.  Other arguments, workspace and errors as pa_decode;
 * PA_ERR_INVALID also for null or misaligned k_new / v_new.
 */
pa_status pa_decode_append(void *out, const void *q, void *k_cache, void *v_cache,
                           const void *k_new, const void *v_new, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                           int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, pa_dtype dtype, int partition_size,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode_plan / pa_decode_planned -- the balanced-split decode with each CTA's
 * start computed on the host.
 *
 * The pages have no counterpart: this is a way to run pa_decode (balanced split),
 * with or without the fused append of pa_decode_append, for a caller that holds
 * the context lengths and block tables on the host (its block allocator made
 * them).  Unplanned, every CTA of the persistent grid first reads the lengths,
 * sums the stream of (sequence, kv head, head group) units, finds its own range,
 * and reads the block-table row of its first item: two dependent memory round
 * trips before its first K/V copy.  pa_decode_plan does that work on the host,
 * once per step.  It writes, per CTA, the stream total, the CTA's range, its first
 * sequence with that sequence's first position and length, and the first
 * 16 block ids of its first item.  A planned launch reads its entry and issues
 * its first copies at once.  Output, caches and workspace use are bit-identical to
 * the unplanned call's: the walk and the arithmetic are the same.
 *
 * pa_decode_plan_bytes: size of the plan for these arguments on the current
 *   device: 128 bytes per CTA of the persistent grid (about 2 per SM).
 *   (size_t)-1 for invalid arguments.
 * pa_decode_plan: plan (host int32, plan_bytes = pa_decode_plan_bytes) <- the
 *   schedule for block_tables [num_seqs][max_blocks_per_seq] and context_lens
 *   [num_seqs], both HOST arrays with the values the launch will read on the
 *   device.  The plan covers plan_bytes / 128 CTAs, the grid the size was computed
 *   for.  Host only: no CUDA call, no device work, no allocation.  Errors:
 *   PA_ERR_INVALID (null pointer, bad sizes, plan_bytes not a positive multiple of
 *   128).
 * pa_decode_planned: as pa_decode with partition_size 0 (k_new = v_new = NULL) or
 *   pa_decode_append (both set), plus `plan`: a DEVICE copy of the plan (16-byte
 *   aligned, plan_bytes = pa_decode_plan_bytes for the same arguments, made from
 *   the same lengths and tables).  A plan made from other lengths or tables gives
 *   a wrong output but no access outside the arguments, and the appended rows
 *   still go where the block table says; where its positions cannot match the
 *   lengths the launch reads, the walk stops and PA_DEVERR_PLAN is raised
 *   (pa_device_errors).  Errors: as pa_decode_append; PA_ERR_INVALID also for a
 *   null or misaligned plan or a plan_bytes that does not match.
 */
size_t pa_decode_plan_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, pa_dtype dtype);
pa_status pa_decode_plan(int32_t *plan, size_t plan_bytes, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         pa_dtype dtype);
pa_status pa_decode_planned(void *out, const void *q, void *k_cache, void *v_cache,
                            const void *k_new, const void *v_new, const int32_t *block_tables,
                            int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                            int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                            int head_dim, int block_size, pa_dtype dtype, const int32_t *plan,
                            size_t plan_bytes, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * pa_decode_shared -- decode a batch whose sequences share prefix blocks.
 *
 * Same result as pa_decode (or, with k_new/v_new, pa_decode_append), but each
 * block shared by a group of sequences is read once for the whole group ([S]
 * "Memory sharing": parallel samples point at the same physical prompt blocks).
 * The decode runs in two launches: the shared blocks of every group, with the
 * query rows of all its members against each kv head, then every sequence's own
 * blocks; the two partial results are merged by the log-sum-exp rule of [S]'s
 * block-wise attention equation.
 *
 *   share   device int32 [S][2]: share[s][0] = batch index of the first member of
 *           s's group, or -1 when s shares nothing; share[s][1] = number of leading
 *           blocks the group shares.  Preconditions: members are consecutive in the
 *           batch; all have the same share[s][1] = P; their block-table rows agree
 *           on entries 0 .. P-1; and every member's context is longer than
 *           P * block_size (the newest token is never in a shared block: the
 *           allocator copies such a block on write).  The last one is checked on
 *           the device: a member that breaks it raises PA_DEVERR_SHARE and is
 *           decoded as if it shared nothing (its own result stays correct without
 *           k_new/v_new; with them its append writes into a block the group
 *           shares, which the others may read either way).  The others are not
 *           checked.
 *   k_new, v_new   both null (plain decode) or as in pa_decode_append.
 * Requires num_q_heads / num_kv_heads <= 16 (PA_ERR_UNSUPPORTED otherwise).  Always
 * uses the balanced split.  Workspace: pa_decode_shared_workspace_size bytes.
 * Errors as pa_decode; PA_ERR_INVALID also for a null or misaligned share.
 */
pa_status pa_decode_shared(void *out, const void *q, void *k_cache, void *v_cache,
                           const void *k_new, const void *v_new, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens,
                           const int32_t *share, int num_seqs, int num_blocks, float scale,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           pa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of pa_decode_shared: twice pa_decode_workspace_size(..., 0) (the
 * two launches may overlap, each has its own counters and partial rows) plus fp32
 * shared-prefix rows [S][Hq][d + 4] (the row's o, then its log2-sum-exp, then
 * padding; 256-byte aligned end).  (size_t)-1 for invalid arguments. */
size_t pa_decode_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks_per_seq);

/*
 * pa_decode_shared_plan / pa_decode_shared_planned -- pa_decode_shared with each
 * CTA's start in both launches computed on the host.
 *
 * The pages have no counterpart (see pa_decode_plan).  Unplanned, every CTA of
 * each launch first reads all context lengths and group entries (and, for the
 * shared blocks' launch, the member entries after each group's first member),
 * sums the launch's stream, finds its range and reads its first block-table row:
 * several dependent memory round trips before its first copy, in each launch.
 * pa_decode_shared_plan replays both walks on the host and writes one 128-byte
 * entry per CTA per launch: the shared blocks' launch's entries, then the own
 * blocks' launch's.  An entry holds what pa_decode_plan's does, with the first
 * sequence's units as that launch counts them (the group's member count and
 * shared block count; the first own block, and whether the (kv head, sequence)
 * order applies).  Output, caches and workspace use are bit-identical to the
 * unplanned pa_decode_shared's.
 *
 * pa_decode_shared_plan_bytes: size of the plan on the current device: 2 x 128
 *   bytes per CTA of the persistent grid of the launches (both launches run on
 *   the same grid; (size_t)-1 where they would not, or for invalid arguments,
 *   including num_q_heads / num_kv_heads > 16).
 * pa_decode_shared_plan: plan (host int32) <- the schedule for HOST copies of
 *   block_tables, context_lens and share (as pa_decode_shared reads them).  The
 *   plan covers plan_bytes / 256 CTAs per launch.  Host only: no CUDA call, no
 *   device work, no allocation.  Errors: PA_ERR_INVALID (null pointer, bad sizes,
 *   plan_bytes not a positive multiple of 256).
 * pa_decode_shared_planned: as pa_decode_shared, plus `plan`: a DEVICE copy of the
 *   plan (16-byte aligned, plan_bytes = pa_decode_shared_plan_bytes for the same
 *   arguments, made from the same lengths, tables and share entries).  A plan made
 *   from other inputs gives wrong outputs but no access outside the arguments;
 *   appended rows still go where the block table says, and only for a sequence
 *   whose length the launch reads equals the plan's; a walk whose positions cannot
 *   match raises PA_DEVERR_PLAN.  Errors: as pa_decode_shared; PA_ERR_INVALID also
 *   for a null or misaligned plan or a plan_bytes that does not match.
 */
size_t pa_decode_shared_plan_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, pa_dtype dtype);
pa_status pa_decode_shared_plan(int32_t *plan, size_t plan_bytes, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                const int32_t *share, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, pa_dtype dtype);
pa_status pa_decode_shared_planned(void *out, const void *q, void *k_cache, void *v_cache,
                                   const void *k_new, const void *v_new,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, const int32_t *share, int num_seqs,
                                   int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, pa_dtype dtype,
                                   const int32_t *plan, size_t plan_bytes, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Partition size pa_decode uses for these arguments: 0 for the balanced split,
 * else the fixed partition size (capped at the table capacity).  Returns -1 for
 * invalid arguments.
 */
int pa_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq, int partition_size);

/*
 * Bytes of workspace pa_decode needs for these arguments.  Fixed partitions: 0
 * when one partition covers the table, else fp32 partial outputs [S][P][Hq][d]
 * (256-byte aligned end) followed by fp32 log2-sum-exp values [S][P][Hq], P =
 * ceil(max_blocks_per_seq * block_size / partition_size).  Balanced split: C =
 * 4 * (SMs of the current device) 64-bit merge counters (256-byte aligned end),
 * then the same two arrays with 2 * C * 16 rows, whatever the lengths.  Returns
 * (size_t)-1 for invalid arguments.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int partition_size);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a deployment variant of pa_decode, with
 * the same arguments, the same result and the same kernels, minus the workspace.
 * It is for callers that may not allocate device memory on their hot path, such as
 * a plugin of an inference engine that has planned every buffer up front, an
 * embedded runtime with a fixed memory budget, or a C caller with no device
 * allocator (cudaMalloc can synchronise the device).  The split-KV scratch is a
 * fixed device array inside the library, PA_DECODE_NOALLOC_SCRATCH_BYTES long,
 * which every GPU that loads the library keeps until the process exits.
 *
 *   - Sizes whose scratch (pa_decode_workspace_size) exceeds the array are
 *     rejected with PA_ERR_UNSUPPORTED before anything is enqueued; use pa_decode
 *     with a caller workspace (or a larger partition_size) for those.
 *   - The first call on each device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call before
 *     any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero.  Calls whose work overlaps on the GPU
 *     (different streams, or several host threads) race on it: serialise them.
 *   - It never calls cudaMalloc, cudaFree or an allocating library routine.
 * Errors: as pa_decode, plus PA_ERR_UNSUPPORTED for sizes beyond the array.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (64u << 20)
pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int num_blocks,
                            float scale, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, pa_dtype dtype, int partition_size, void *stream);

/* ------------------------------------------------------------------------- *
 * Cache writes.                                                              *
 * ------------------------------------------------------------------------- */

/*
 * pa_reshape_and_cache -- write each new token's K and V rows into its slot.
 *
 * Defines ([T] §3.1 append_kv: logical page pos // page_size, offset
 * pos % page_size; [S] "Core idea": blocks fill one token at a time):
 *     for t in [0, num_tokens): slot = slot_mapping[t];
 *       k_cache[slot / B][slot % B][:][:] = k[t][:][:]   (and v likewise)
 * A negative slot skips the token (padding).  A slot >= num_blocks * B is also
 * skipped: the kernel never writes outside the caches.  Bit-exact copies.
 *
 *   k, v           device [num_tokens][num_kv_heads][head_dim], dtype `dtype`
 *   slot_mapping   device int64 [num_tokens]
 * Duplicate slots within one call: which token's row lands is unspecified.
 * Errors: PA_ERR_INVALID, PA_ERR_UNSUPPORTED (head_dim * elem size not a multiple
 *   of 16 bytes), PA_ERR_CUDA.  num_tokens = 0 is a no-op.
 */
pa_status pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                               void *stream);

/*
 * pa_copy_blocks -- copy-on-write of whole blocks.
 *
 * Defines ([S] "Memory sharing": a sequence about to write into a shared block gets
 * a private copy of that block only, like fork()):
 *     for each pair i: k_cache[dst_i] = k_cache[src_i]; v_cache[dst_i] = v_cache[src_i]
 * where a block is block_bytes contiguous bytes (block_size * num_kv_heads *
 * head_dim * elem size).  Pairs run concurrently: no dst may equal any src or
 * another dst (the allocator only produces fresh destinations).  Pairs with an
 * index outside [0, num_blocks) are skipped.  Bit-exact.
 *
 *   src_dst_pairs  device int32 [num_pairs][2] (src, dst)
 *   block_bytes    multiple of 16
 * Errors: PA_ERR_INVALID, PA_ERR_CUDA.  num_pairs = 0 is a no-op.
 */
pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_dst_pairs,
                         int num_pairs, int num_blocks, size_t block_bytes, void *stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools, e.g. the device pool and a
 * pool in pinned host memory ([S] "vLLM": a preempted request's blocks move to CPU
 * memory and come back when it resumes).
 *
 * Defines, for each pair i (src_i, dst_i) = src_dst_pairs[i]:
 *     dst_k[dst_i] = src_k[src_i];  dst_v[dst_i] = src_v[src_i]
 * with a block = block_bytes contiguous bytes, pools of src_num_blocks and
 * dst_num_blocks blocks.  Each pool pointer may be device memory or pinned host
 * memory mapped into the device's address space (cudaHostAlloc / cudaHostRegister
 * memory under unified addressing); so may src_dst_pairs.  Pairs with an index out
 * of range are skipped; destinations must be distinct and must not overlap a
 * source of the same call.  Bit-exact.  pa_alloc_swap_out / pa_alloc_swap_in emit
 * the pairs.
 * Errors: PA_ERR_INVALID (null or misaligned pointer, bad size, or a pointer the
 *   device cannot reach: pageable host memory, checked with cudaPointerGetAttributes
 *   before the launch), PA_ERR_UNSUPPORTED (block_bytes above 1 GiB), PA_ERR_CUDA.
 *   num_pairs = 0 is a no-op.
 */
pa_status pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                         const int32_t *src_dst_pairs, int num_pairs, int src_num_blocks,
                         int dst_num_blocks, size_t block_bytes, void *stream);

/*
 * pa_gather_blocks / pa_scatter_blocks -- pack blocks of a pool into a contiguous
 * staging buffer and unpack them into (other) blocks of a pool: the two local
 * halves of moving a sequence's KV from one engine's pool to another's ([K]
 * "Bidirectional KV transfer": the receiving side reads the sender's KV blocks and
 * places them in its own blocks).
 *     gather:  staging_k[i] = k_cache[block_ids[i]]   (and v), i < num_ids
 *     scatter: k_cache[block_ids[i]] = staging_k[i]   (and v)
 * staging_k / staging_v: [num_ids][block_bytes] contiguous, device or pinned host
 * memory; block_ids: device-accessible int32 [num_ids].  Ids outside
 * [0, num_blocks) are skipped (their staging block is left as it was).  Scatter ids
 * must be distinct.  Bit-exact.  Errors as pa_swap_blocks.
 */
pa_status pa_gather_blocks(const void *k_cache, const void *v_cache, const int32_t *block_ids,
                           int num_ids, int num_blocks, void *staging_k, void *staging_v,
                           size_t block_bytes, void *stream);
pa_status pa_scatter_blocks(const void *staging_k, const void *staging_v, void *k_cache,
                            void *v_cache, const int32_t *block_ids, int num_ids, int num_blocks,
                            size_t block_bytes, void *stream);

/*
 * Host predicate of [K] "KV recompute threshold": fetching another engine's KV for
 * a prefix pays off only from threshold_tokens reusable tokens up (the article's
 * default is 64); below it the receiver recomputes the prefix.  1 = transfer,
 * 0 = recompute (also for reusable_tokens <= 0).
 */
int pa_kv_transfer_worthwhile(long long reusable_tokens, long long threshold_tokens);
#define PA_KV_RECOMPUTE_THRESHOLD_DEFAULT 64

/*
 * Device-side error flags of the current device (bitwise OR of PA_DEVERR_*), read
 * and cleared with a synchronous copy after `stream` drains.  Every wait inside a
 * decode kernel is bounded: a CTA whose wait runs out (a TMA transfer that never
 * lands, a warp that stopped) sets a flag, stops issuing copies, lets the copies
 * it already issued land, and returns instead of hanging (its other waits end at
 * their own limit at the latest); the launch's output is then incomplete.  The pages have no counterpart: this is
 * the library's own failure detection.
 * Returns PA_ERR_TIMEOUT when a timeout flag was set, else PA_ERR_INVALID when
 * PA_DEVERR_SHARE or PA_DEVERR_PLAN was (*flags holds the flags, now cleared);
 * PA_OK when none was;
 * PA_ERR_CUDA if the stream or the copy failed.
 * After a timeout the split-KV merge counters of an aborted launch may be left
 * non-zero: a later call is unaffected (each call tags its counters anew), but a
 * captured CUDA graph replays its tag, so clear its workspace before replaying it.
 */
#define PA_DEVERR_TIMEOUT_FULL  1u   /* consumer waited too long for a K/V tile   */
#define PA_DEVERR_TIMEOUT_EMPTY 2u   /* producer waited too long for a free stage */
#define PA_DEVERR_SHARE         4u   /* pa_decode_shared: a member's context ends
                                        inside its group's shared blocks          */
#define PA_DEVERR_PLAN          8u   /* pa_decode_planned, pa_decode_shared_planned: the plan does not match
                                        the context lengths the launch read       */
pa_status pa_device_errors(unsigned int *flags, void *stream);

/*
 * Limit, in ns, of the bounded device-side waits of decode launches enqueued after
 * this call, by any thread (0 restores the default, 2 s).  Returns the previous
 * limit.  A shorter limit makes a stalled launch give up sooner; a limit shorter
 * than the launch's own waits for memory (microseconds) makes it give up at once,
 * which the tests use to exercise the timeout path.  The wait for copies already
 * in flight when a CTA stops always takes the default bound.  The pages have no
 * counterpart (failure detection of this library).
 */
#define PA_WAIT_LIMIT_DEFAULT_NS 2000000000ull
unsigned long long pa_set_wait_limit_ns(unsigned long long ns);

/* ------------------------------------------------------------------------- *
 * Host block allocator ([S] "vLLM": free list, reference counts, copy-on-write;  *
 * [T] §2.2 BlockManager, §3.1 append_kv, §5.1 clone_sequence).  Host memory    *
 * only; never touches the GPU.  Not thread-safe: one caller at a time.         *
 * ------------------------------------------------------------------------- */
typedef struct pa_alloc pa_alloc;

/*
 * Create a pool of num_blocks blocks of block_size tokens.  The free list starts as
 * `free_order` (a permutation of 0..num_blocks-1; NULL = 0, 1, ..., num_blocks-1,
 * the tutorial's list(range(total_pages))).  Allocation pops the LAST element.
 */
pa_status pa_alloc_create(pa_alloc **out, int num_blocks, int block_size,
                          const int32_t *free_order);
void pa_alloc_destroy(pa_alloc *a);

/* New empty sequence; ids are 0, 1, 2, ... in creation order (forks included). */
pa_status pa_alloc_new_seq(pa_alloc *a, int *seq_id);

/* New sequence sharing all of `parent`'s blocks (each block's refcount + 1). */
pa_status pa_alloc_fork(pa_alloc *a, int parent, int *child);

/*
 * Reserve the slot of the next token of `seq` (position p = current length):
 *   - logical block p / B not mapped yet: pop a free block (refcount 1);
 *   - mapped but shared (refcount > 1): copy-on-write -- pop a free block, emit
 *     (*cow_src, *cow_dst) = (old, new), old refcount - 1, map the new block;
 *   - otherwise write in place.
 * *slot = block * B + p % B.  *cow_src = *cow_dst = -1 when nothing is copied.
 * PA_ERR_OOM (no free block) leaves every piece of state unchanged.
 */
pa_status pa_alloc_append(pa_alloc *a, int seq, int64_t *slot, int32_t *cow_src,
                          int32_t *cow_dst);

/* Reserve n slots at once (same as n calls of pa_alloc_append); slots[n] and up to
 * n copy pairs (cow_pairs[2*i], cow_pairs[2*i+1]) with *num_cow set.  On PA_ERR_OOM
 * the appends made before the failing one stay (as with separate calls); *done
 * (optional) tells how many succeeded. */
pa_status pa_alloc_append_n(pa_alloc *a, int seq, int n, int64_t *slots, int32_t *cow_pairs,
                            int *num_cow, int *done);

/* Release a sequence: its blocks' refcounts drop in table order; a block reaching 0
 * is appended to the end of the free list. */
pa_status pa_alloc_free_seq(pa_alloc *a, int seq);

/* Copy up to `cap` entries of the sequence's block table; *n = its full length. */
pa_status pa_alloc_block_table(const pa_alloc *a, int seq, int32_t *out, int cap, int *n);
pa_status pa_alloc_seq_len(const pa_alloc *a, int seq, int *len);
int pa_alloc_refcount(const pa_alloc *a, int block);     /* -1 if out of range */
int pa_alloc_num_free(const pa_alloc *a);
/* Copy up to `cap` free-list entries (bottom to top: the next pop is the last). */
pa_status pa_alloc_free_list(const pa_alloc *a, int32_t *out, int cap, int *n);

/*
 * Swap space ([S] "vLLM": when GPU memory runs short, the scheduler pauses a
 * request by moving its blocks to CPU memory, and brings them back later).
 * pa_alloc_set_host_pool gives the allocator num_host_blocks blocks of host memory
 * (ids 0..H-1, free list 0, 1, ..., H-1, popped from the end); allowed while no
 * sequence is swapped out.
 *
 * pa_alloc_swap_out(seqs[0..n)): every distinct device block the sequences
 * reference (met in the given sequence order, then table order) takes the next free
 * host block; each reference moves to the host block (device refcount - 1, host
 * refcount + 1; a device block reaching 0 goes to the end of the device free list,
 * in release order).  pairs[2i], pairs[2i+1] = (device block, host block), in the
 * order the host blocks were taken, *num_pairs = their count: the copies to run with
 * pa_swap_blocks(device pool -> host pool) before the device blocks are reused.  A
 * device block also held by a sequence that stays resident keeps its data and
 * refcount; the swapped sequences get their own host copy.
 * pa_alloc_swap_in is the reverse: (host block, device block) pairs, host blocks
 * reaching 0 return to the end of the host free list.
 * A swapped-out sequence keeps its length; pa_alloc_block_table returns its host
 * block ids; pa_alloc_append / pa_alloc_fork refuse it (PA_ERR_INVALID);
 * pa_alloc_free_seq releases its host blocks.
 * Errors (nothing changes): PA_ERR_INVALID (a sequence not live, in the wrong pool,
 * listed twice, or cap < the number of pairs, *num_pairs telling how many are
 * needed), PA_ERR_OOM (fewer free blocks in the target pool than pairs).
 */
pa_status pa_alloc_set_host_pool(pa_alloc *a, int num_host_blocks);

/*
 * Memory accounting of the device pool ([S] "Results": the remaining waste of paged
 * KV memory is the unfilled tail of each sequence's last block, under B tokens;
 * [S] "Memory sharing": forked samples and beams share blocks).  Over the resident
 * (not swapped-out) sequences:
 *   used_blocks     device blocks with refcount > 0
 *   logical_blocks  table entries summed over the sequences (what unshared
 *                   per-sequence storage would take)
 *   token_slots     used_blocks * block_size
 *   tokens          slots holding a token: per used block, the largest number of
 *                   rows any of its holders has filled
 * Waste fraction = 1 - tokens / token_slots; sharing saving = 1 - used_blocks /
 * logical_blocks.
 */
typedef struct {
    int64_t used_blocks;
    int64_t logical_blocks;
    int64_t token_slots;
    int64_t tokens;
    int64_t resident_seqs;
    int64_t swapped_seqs;
} pa_alloc_usage;
pa_status pa_alloc_usage_stats(const pa_alloc *a, pa_alloc_usage *out);
pa_status pa_alloc_swap_out(pa_alloc *a, const int *seqs, int n, int32_t *pairs, int cap,
                            int *num_pairs);
pa_status pa_alloc_swap_in(pa_alloc *a, const int *seqs, int n, int32_t *pairs, int cap,
                           int *num_pairs);
int pa_alloc_is_swapped(const pa_alloc *a, int seq);       /* 1, 0; -1 if not live */
int pa_alloc_host_refcount(const pa_alloc *a, int block);  /* -1 if out of range */
int pa_alloc_num_free_host(const pa_alloc *a);
pa_status pa_alloc_host_free_list(const pa_alloc *a, int32_t *out, int cap, int *n);

/*
 * Host helper: the share argument of pa_decode_shared, derived from the block
 * tables (host int32 [S][W], -1 padded) and context lengths (host int32 [S]).
 * A group is a maximal run of consecutive rows whose entry 0 is the same physical
 * block (>= 0); its P is the number of leading entries equal in all its rows,
 * capped at floor((T - 1) / block_size) for every member T.  Groups with fewer
 * than two rows or P < min_shared_blocks get {-1, 0}.  share: host int32 [S][2],
 * written for every row.  PA_ERR_INVALID for bad sizes or null pointers.
 */
pa_status pa_share_groups(const int32_t *block_tables, int num_seqs, int max_blocks_per_seq,
                          const int32_t *context_lens, int block_size, int min_shared_blocks,
                          int32_t *share);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
