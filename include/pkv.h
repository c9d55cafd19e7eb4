/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache library.
 *
 * The operation set follows the pages' statement of paged attention:
 *   - the KV cache of a sequence lives in fixed-size blocks placed anywhere in
 *     a pool, and a per-sequence block table keeps the logical order
 *     (x321.org "The serving bottleneck is not just FLOPs", section
 *     "PagedAttention borrows an operating-system trick");
 *   - attention is softmax(Q K^T / sqrt(d_head)) V (same page, section "First
 *     understand what the KV cache is storing"), here evaluated by a kernel
 *     that follows the block mapping;
 *   - blocks of an identical prefix are shared with copy-on-write
 *     (praveentn.live "PagedAttention KV-cache constraint", section "What the
 *     change bought").
 *
 * Conventions for every call
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  Argument errors
 *     are detected on the host before anything is enqueued; nothing is
 *     launched when a call fails.
 *   - Device pointers are owned by the caller.  The kernels allocate no
 *     device memory; scratch space is passed in by the caller.
 *   - Kernels are enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns after the launch, asynchronously.
 *   - `d_status` (optional, may be NULL) is a device int32 that kernels OR
 *     PKV_STATUS_* bits into when they meet an out-of-range index; the access
 *     is skipped (reads as zero) instead of faulting.  The caller zeroes it
 *     and reads it after synchronising.
 *   - bf16 values are passed as their 16-bit patterns (pkv_bf16).  Tensors
 *     are dense, row-major, with the shapes given below; device pointers must
 *     be 16-byte aligned.
 *   - KV cache layout: k_cache and v_cache are each
 *     [num_blocks][num_kv_heads][block_size][head_dim] bf16, so one (block,
 *     KV head) tile of block_size x head_dim values is contiguous.
 *   - Slot encoding: slot = physical_block * block_size + offset_in_block;
 *     a negative slot means "no token, skip".
 *   - Grouped-query attention: query head g reads KV head
 *     g / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;

/* return codes */
#define PKV_OK               0
#define PKV_ERR_ARG         -1  /* null/misaligned pointer, bad size or shape    */
#define PKV_ERR_OOM         -2  /* allocator: not enough free blocks             */
#define PKV_ERR_RANGE       -3  /* index outside its table / pool                */
#define PKV_ERR_UNSUPPORTED -4  /* valid but not compiled (head_dim, block, ...) */
#define PKV_ERR_CUDA        -5  /* a CUDA runtime call failed                    */
#define PKV_ERR_TIMEOUT     -6  /* reserved: a device wait gave up               */
#define PKV_ERR_SHARED      -7  /* allocator: append into a shared partial block */
#define PKV_ERR_WORKSPACE   -8  /* workspace too small                           */

/* bits OR-ed into *d_status by kernels */
#define PKV_STATUS_BAD_SLOT   1  /* pkv_write: slot >= num_blocks * block_size   */
#define PKV_STATUS_BAD_BLOCK  2  /* block id outside [0, num_blocks)             */
#define PKV_STATUS_BAD_LEN    4  /* seq_len < 0 or above the table's capacity    */
#define PKV_STATUS_TIMEOUT    8  /* a bounded on-chip wait gave up               */
#define PKV_STATUS_BAD_QSTART 16 /* prefill: q_start entry out of order or range */
#define PKV_STATUS_BAD_ITEM   32 /* decode work list: item out of range, or built for other lengths / tables */

/* Human-readable name of a return code (static storage). */
const char *pkv_error_string(int code);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *pkv_last_cuda_error(void);

/*
 * pkv_write -- store the keys and values of new tokens into their cache slots.
 *
 * Pages: the cache keeps every past key and value and grows by one token per
 * decode step (x321.org "The serving bottleneck is not just FLOPs", section
 * "First understand what the KV cache is storing"); a request grows by taking
 * more blocks (same page, "PagedAttention borrows an operating-system trick").
 *
 * For every token t < num_tokens with s = slot_mapping[t] >= 0 and every KV
 * head h:  k_cache[s / block_size][h][s % block_size][:] = k[t][h][:]
 *          v_cache[...same...]                          = v[t][h][:]
 *   k, v          device, [num_tokens][num_kv_heads][head_dim] bf16 (read)
 *   slot_mapping  device, [num_tokens] int64 (read)
 *   k_cache/v_cache  device, layout above (written)
 * Slots >= num_blocks*block_size set PKV_STATUS_BAD_SLOT and are skipped.
 * Two tokens with the same slot race (undefined which one lands).
 * head_dim must be a multiple of 8.  num_tokens == 0 is a no-op.
 */
int pkv_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping,
              int num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache, int num_blocks,
              int block_size, int num_kv_heads, int head_dim, int32_t *d_status,
              void *stream);

/*
 * pkv_block_copy -- materialise copy-on-write: copy whole blocks.
 *
 * Pages: shared prefix blocks are referenced by several sequences and copied
 * on write (praveentn.live "PagedAttention KV-cache constraint", section
 * "What the change bought").
 *
 * For each pair i < num_pairs with (src, dst) = (pairs[2i], pairs[2i+1]):
 *   k_cache[dst][:][:][:] = k_cache[src][:][:][:]; the same for v_cache.
 *   src_dst_pairs  device, [num_pairs][2] int32 (read)
 * An id outside [0, num_blocks) sets PKV_STATUS_BAD_BLOCK and skips the pair.
 * The dst ids must be distinct and disjoint from the src ids (the allocator's
 * copy-on-write pairs always are); otherwise the result is undefined.
 */
int pkv_block_copy(pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *src_dst_pairs,
                   int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                   int head_dim, int32_t *d_status, void *stream);

/*
 * Bytes of caller-provided device workspace paged_attention_decode needs for
 * these sizes (0 when no sequence can span more than one partition).
 * partition_size: tokens per split-K partition, a multiple of block_size;
 * 0 selects the default (768).  Returns 0 for invalid sizes as well; check
 * the decode call's return code.
 */
size_t paged_attention_workspace_size(int num_seqs, int q_len, int num_q_heads,
                                      int head_dim, int max_seq_len, int partition_size);

/*
 * paged_attention_decode -- attention of the newest q_len tokens of each
 * sequence over its block-paged KV cache.
 *
 * Pages: Attention(Q,K,V) = softmax(Q K^T / sqrt(d_head)) V (x321.org "The
 * serving bottleneck is not just FLOPs", section "First understand what the KV
 * cache is storing"), evaluated by a kernel that follows the block mapping
 * (same page, "PagedAttention borrows an operating-system trick"; praveentn.live
 * "PagedAttention KV-cache constraint", section "What it cost": an indirection
 * on every attention step that needs a custom kernel).
 *
 * For sequence i with L = seq_lens[i], query row r < q_len and query head g:
 *   keys visible: t < n = L - q_len + 1 + r (q_len = 1: all L keys; a longer
 *   query chunk is causal inside the chunk), key/value row t of KV head
 *   h = g / (num_q_heads/num_kv_heads) read from block
 *   block_tables[i][t / block_size], offset t % block_size;
 *   out[i][r][g][:] = sum_t softmax_t(scale * q[i][r][g].k_t) * v_t, rounded
 *   to bf16 (round to nearest even).  n <= 0 gives zeros.
 *   q, out        device, [num_seqs][q_len][num_q_heads][head_dim] bf16
 *   block_tables  device, [num_seqs][max_blocks_per_seq] int32; entries past
 *                 ceil(L / block_size) are never used (any value; the kernel
 *                 may read up to 32 of them before it knows L)
 *   seq_lens      device, [num_seqs] int32, 0 <= L <= max_seq_len and
 *                 L <= max_blocks_per_seq * block_size (else PKV_STATUS_BAD_LEN,
 *                 and L is clamped)
 *   max_seq_len   host upper bound of seq_lens; sizes the grid and workspace
 *   partition_size tokens per split-K partition (0 = 768), a multiple of
 *                 block_size; sequences longer than one partition are reduced
 *                 across partitions with an exact log-sum-exp merge
 *   workspace     device scratch of at least paged_attention_workspace_size(...)
 *                 bytes (may be NULL when that size is 0); contents are not
 *                 preserved between calls
 * Supported: head_dim in {64, 128}; block_size in {16, 32, 64, 128}; q_len in {1, 16}
 *   with q_len * num_q_heads / num_kv_heads <= 128 and, for q_len = 1,
 *   num_q_heads / num_kv_heads <= 16.  Other sizes return PKV_ERR_UNSUPPORTED.
 * Block ids outside [0, num_blocks) set PKV_STATUS_BAD_BLOCK; the block reads
 * as zeros.
 */
int paged_attention_decode(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                           const pkv_bf16 *v_cache, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                           int max_seq_len, int q_len, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, float scale,
                           int partition_size, pkv_bf16 *out, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, void *stream);

/*
 * paged_attention_decode_ex -- paged_attention_decode that also marks, for
 * measurement, where its main kernel ends.
 *
 * The pages have no counterpart to this call.  A decode is one main kernel
 * (the paged attention itself) followed, when a sequence spans more than one
 * partition, by the cross-partition merge.  main_done_event, when not NULL,
 * is a cudaEvent_t created by the caller; it is recorded on `stream` right
 * after the main kernel is enqueued and before the merge, so that the elapsed
 * time from an event recorded before the call to it is the main kernel's.
 * Everything else is paged_attention_decode's, which is this call with NULL.
 * A failing record returns PKV_ERR_CUDA.
 */
int paged_attention_decode_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                              const pkv_bf16 *v_cache, const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                              int max_seq_len, int q_len, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, int num_blocks, float scale,
                              int partition_size, pkv_bf16 *out, void *workspace,
                              size_t workspace_bytes, int32_t *d_status, void *stream,
                              void *main_done_event);

/*
 * paged_attention_decode_write -- the decode step of single-token sequences
 * with the new token's store folded in: pkv_write of num_seqs tokens followed
 * by paged_attention_decode with q_len = 1, as one call.
 *
 * Pages: each decode step stores the new token's keys and values in their
 * slot and then attends over the sequence's blocks (x321.org "The serving
 * bottleneck is not just FLOPs", "First understand what the KV cache is
 * storing" and "PagedAttention borrows an operating-system trick").
 *   k_new, v_new   device, [num_seqs][num_kv_heads][head_dim] bf16: the newest
 *                  token of each sequence
 *   slot_mapping   device, [num_seqs] int64: slot of sequence i's newest token,
 *                  which must be its table position, i.e. block_tables[i][(L-1)
 *                  / block_size] * block_size + (L-1) % block_size with L =
 *                  seq_lens[i] (the slot the allocator's append returns), or
 *                  negative for no store
 *   everything else as paged_attention_decode (q, out [num_seqs][1][Hq][d]).
 * The CTA that reads the newest token's block stores the token's rows and
 * also places them into its staged copy of that block, so no separate write
 * grid runs and no copy has to wait for the store.  A non-negative slot other
 * than the newest token's table position is undefined: where the check runs
 * it sets PKV_STATUS_BAD_SLOT and the token is not stored.  Where the
 * decode runs on the tensor cores (max_seq_len >= 16384) the store is a
 * separate pkv_write launch before it.  main_done_event as in
 * paged_attention_decode_ex (may be NULL).
 */
int paged_attention_decode_write(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                 const int64_t *slot_mapping, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *seq_lens, int num_seqs, int max_seq_len,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, int partition_size, pkv_bf16 *out,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status,
                                 void *stream, void *main_done_event);

/*
 * pkv_decode_items -- host: the work list of a single-token decode batch, for
 * paged_attention_decode_items.
 *
 * The pages have no counterpart to this call; it moves the decode's schedule
 * to the host, which knows every length when it builds the step (the
 * allocator's append and table fill).  Each sequence's keys are split into
 * partitions of partition_size tokens as paged_attention_decode splits them,
 * and every (partition, KV head) becomes one item:
 *   {sequence, KV head | partition << 16, length, physical block of the
 *    partition's first logical block (-1 if block_tables is NULL or the
 *    partition is empty)}
 * The items are ordered longest partition first (ties in sequence, partition
 * and head order), so the CTAs that start first carry the most keys and the
 * shortest partitions fill the end of the grid.  A sequence of length 0 gets
 * one empty item per KV head (its output rows are zeros).
 * partition_size 0 lets the call choose among 768, 1024, 1536, 2048, 3072 and
 * 4096 tokens (those that are multiples of block_size; 3072 and 4096 only when
 * block_tables is given and no physical block serves two sequences) the one a
 * schedule model of the decode kernel on a GB300 predicts fastest for these
 * lengths: more, shorter partitions balance the grid's end, fewer longer ones
 * save each CTA's start and the merge.  A workspace sized for partition 768
 * (paged_attention_workspace_size with partition_size 0) fits every choice.
 *   seq_lens      host, [num_seqs] int32, each in [0, max_blocks_per_seq *
 *                 block_size] (else PKV_ERR_RANGE)
 *   block_tables  host, [num_seqs][max_blocks_per_seq] int32, or NULL
 *   items_out     host, [1 + max_items][4] int32: row 0 = {count, partition
 *                 size used, m, 1 + count}, rows 1..count the items, then
 *                 the m sequences with more than one partition (those the
 *                 split-K merge combines), four to a row, -1 after the last.
 *                 Pass row 0's partition size to paged_attention_decode_items.
 * *num_items receives the rows after the header, count + ceil(m / 4) (also
 * when they exceed max_items, which returns PKV_ERR_RANGE and writes
 * nothing).  A partition_size that is not a multiple of block_size returns
 * PKV_ERR_ARG.
 */
int pkv_decode_items(const int32_t *seq_lens, const int32_t *block_tables, int max_blocks_per_seq,
                     int num_seqs, int num_kv_heads, int head_dim, int block_size,
                     int partition_size, int32_t *items_out, int max_items, int *num_items);

/*
 * paged_attention_decode_items -- the single-token decode over a work list:
 * paged_attention_decode_write (or, with k_new, v_new and slot_mapping all
 * NULL, paged_attention_decode with q_len = 1), one CTA per item.
 *   items       device, 16-byte aligned, [1 + grid_items][4] int32 (at least
 *               the rows pkv_decode_items wrote for these seq_lens and
 *               block_tables); partition_size must be the size the list was
 *               built for (row 0's second entry).  The split-K merge runs over
 *               the list's merge rows only.
 *   grid_items  CTAs to launch, >= the count in row 0 (CTAs past the count do
 *               nothing; the rows after the header are a valid choice), so a
 *               CUDA graph can be captured for a bound
 * Every other argument and the result are those of paged_attention_decode_write.
 * An item naming a sequence, head or partition out of range, a length other
 * than seq_lens[sequence], or a first block other than the table's sets
 * PKV_STATUS_BAD_ITEM (the item is skipped, or computed with the table's
 * blocks); a list built for other arguments gives undefined output but never
 * reads or writes out of bounds.  Where the decode runs on the tensor cores
 * (max_seq_len >= 16384) the list is not used.
 *   flags       0, or PKV_DECODE_OVERLAP: the caller guarantees that nothing
 *               this call reads (q, k_new, v_new, slot_mapping, the caches,
 *               tables, lengths, items) and nothing it stores into the caches
 *               is written or read by the work queued before it on the stream,
 *               as with the layers of one decode step.  The call then streams
 *               its keys and values at once and waits for that earlier work
 *               only before it writes workspace or out, so consecutive calls
 *               overlap (one workspace may serve them all).  Other bits:
 *               PKV_ERR_ARG.  Ignored on the tensor-core route.
 */
#define PKV_DECODE_OVERLAP 1

int paged_attention_decode_items(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                 const int64_t *slot_mapping, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *seq_lens, int num_seqs, int max_seq_len,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, int partition_size,
                                 const int32_t *items, int grid_items, pkv_bf16 *out,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status,
                                 void *stream, void *main_done_event, int flags);

/*
 * paged_attention_prefill -- attention of a chunk of new tokens per sequence,
 * each sequence with its own chunk length (chunked prefill).
 *
 * Pages: the scheduler splits a long prompt into chunks and runs them in the
 * same step as the decodes of other requests; the prompt side is the
 * compute-heavy phase (x321.org "The serving bottleneck is not just FLOPs",
 * section "Continuous batching is the other half of the story").  The chunk's
 * keys and values are in the cache already (pkv_write before this call), so a
 * chunk attends over the paged cache exactly like paged_attention_decode's
 * causal chunk, and a decode is a chunk of one token.
 *
 * Sequence i owns query rows q_start[i] .. q_start[i+1]-1, its newest
 * c = q_start[i+1] - q_start[i] tokens.  With L = seq_lens[i], row
 * q_start[i] + r (r < c) and query head g see keys t < n = L - c + 1 + r of KV
 * head g / (num_q_heads/num_kv_heads); out = sum_t softmax_t(scale * q.k_t) v_t
 * rounded to bf16; n <= 0 gives zeros.
 *   q, out        device, [total_q][num_q_heads][head_dim] bf16
 *   q_start       device, [num_seqs + 1] int32, never decreasing, within
 *                 [0, total_q] (normally q_start[0] = 0 and q_start[num_seqs] =
 *                 total_q).  A sequence whose pair of entries breaks this sets
 *                 PKV_STATUS_BAD_QSTART and gets no rows; rows of out that no
 *                 sequence owns are not written.
 *   block_tables, seq_lens, k_cache, v_cache, num_blocks, block_size, scale:
 *                 as paged_attention_decode (L <= max_blocks_per_seq *
 *                 block_size, else PKV_STATUS_BAD_LEN and L is clamped)
 * No workspace: every query tile of floor(128 / G) tokens x G heads
 * (G = num_q_heads / num_kv_heads) is one unit of work over all the keys it
 * sees, on the tensor cores.
 * Supported: head_dim in {64, 128}; G from 1 to 16 (a G that does not divide
 * 128 makes tiles of floor(128 / G) tokens, whose last 128 mod G rows are
 * spare); block_size in {16, 32, 64, 128}; num_seqs <= 1024.  Other sizes
 * return PKV_ERR_UNSUPPORTED.
 * total_q == 0 or num_seqs == 0 is a no-op.
 */
int paged_attention_prefill(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *seq_lens, const int32_t *q_start, int num_seqs,
                            int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, pkv_bf16 *out,
                            int32_t *d_status, void *stream);

/*
 * paged_attention_prefill_ex -- paged_attention_prefill with its keys split
 * into partitions (split-K), for batches with fewer query tiles than the GPU
 * has SMs (a short chunk behind a long context).
 *
 * The pages have no counterpart to the split; the result is the same
 * attention (it changes only the fp32 summation order).  With partition_size
 * > 0 (a multiple of 128 tokens), every query tile's keys are cut into
 * partitions of partition_size keys, each computed by its own unit of work
 * into the workspace as (running max, sum, unnormalised output), and a second
 * kernel merges each row's partitions exactly (log-sum-exp).  max_seq_len
 * bounds every seq_lens entry (a larger one sets PKV_STATUS_BAD_LEN and is
 * clamped).  partition_size == 0 is paged_attention_prefill (no workspace).
 *   workspace      device, 16-byte aligned, at least
 *                  paged_attention_prefill_workspace_size(...) bytes
 *                  (PKV_ERR_WORKSPACE otherwise); nothing in it needs clearing
 * Everything else as paged_attention_prefill.
 */
size_t paged_attention_prefill_workspace_size(int total_q, int num_q_heads, int head_dim, int max_seq_len,
                                              int partition_size);

int paged_attention_prefill_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *seq_lens, const int32_t *q_start, int num_seqs,
                               int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, float scale, int max_seq_len,
                               int partition_size, pkv_bf16 *out, void *workspace,
                               size_t workspace_bytes, int32_t *d_status, void *stream);

/*
 * pkv_prefill_items -- host-built work list for the prefill's persistent grid:
 * which of the batch's items (pairs of query tiles, or single tiles, per
 * sequence and KV head, numbered as the kernel numbers them) each of grid
 * CTAs takes.
 *
 * The pages have no counterpart; it balances the tensor-core work of a few
 * long chunks over a grid smaller than the GPU (a continuous-batching step,
 * x321.org "The serving bottleneck is not just FLOPs", section "Continuous
 * batching is the other half of the story"), where CTA c taking items c,
 * c + grid, ... can leave some CTAs one item longer than the rest.  Items are
 * costed by their key tiles (a pair's two query tiles share each key tile)
 * plus a fixed cost per item, then handed out longest first, each to the
 * least-loaded CTA.
 *   seq_lens       host [num_seqs] lengths (negative counts as 0)
 *   q_start        host [num_seqs + 1] first query row of each sequence
 *   total_q        the query rows of the call (as paged_attention_prefill;
 *                  with q_start it decides pairs of query tiles or single ones)
 *   num_q_heads, num_kv_heads  as paged_attention_prefill (group <= 16)
 *   grid           CTAs of the launch (>= 1)
 *   items_out      host [max_ints]: grid, n, the offsets of each CTA's range
 *                  [grid + 1], then the n item indices
 *   *num_ints      3 + grid + n
 * Returns PKV_OK, PKV_ERR_ARG (a null pointer, a count out of range, q_start
 * out of order or outside [0, total_q]), PKV_ERR_UNSUPPORTED (group > 16) or
 * PKV_ERR_RANGE (max_ints too small; *num_ints holds the size needed).
 */
int pkv_prefill_items(const int32_t *seq_lens, const int32_t *q_start, int num_seqs, int total_q,
                      int num_q_heads, int num_kv_heads, int grid, int32_t *items_out, int max_ints,
                      int *num_ints);

/*
 * paged_attention_mixed -- one continuous-batching step: single-token decodes
 * and prompt chunks in one call, the decodes streamed by the decode kernel
 * while the chunks run on the tensor cores.
 *
 * Pages: the scheduler runs chunks of long prompts in the same step as the
 * decodes of other requests; the prompt side is compute-heavy, the decode side
 * memory-bound (x321.org "The serving bottleneck is not just FLOPs", section
 * "Continuous batching is the other half of the story").  The result is that
 * of paged_attention_prefill over the whole batch.
 *   The first num_decodes sequences are single-token decodes whose query rows
 *   are rows 0 .. num_decodes-1 of q (q_start[i] = i for i <= num_decodes);
 *   sequences num_decodes .. num_seqs-1 are chunks (any length, rows from
 *   q_start[num_decodes] on).
 *   decode_items  device, the pkv_decode_items list of the decodes' lengths
 *                 seq_lens[0 .. num_decodes-1] and tables, for
 *                 decode_partition_size; decode_grid as grid_items of
 *                 paged_attention_decode_items
 *   max_decode_len, decode_partition_size, workspace: as max_seq_len,
 *                 partition_size and workspace of paged_attention_decode for
 *                 the num_decodes decodes (paged_attention_workspace_size).
 *                 Beside a long chunk grid the decodes may run unsplit (a
 *                 partition of at least max_decode_len: no merge, no
 *                 workspace), since they only need to end before the chunks.
 *   prefill_ctas  the chunks' persistent grid: at most this many CTAs, one per
 *                 SM (0: every SM); the decodes' CTAs take the other SMs from
 *                 the start and every SM the chunks free later.  Size it to the
 *                 chunks' share of the step's work.
 *   prefill_items device copy of a pkv_prefill_items list built for the chunk
 *                 sequences (seq_lens + num_decodes, q_start + num_decodes,
 *                 the same total_q) and grid = prefill_ctas, or NULL: CTA c
 *                 then takes chunk items c, c + grid, ...  With a list the
 *                 chunks' grid is prefill_ctas even without decodes.  A list of
 *                 another grid size, or entries outside the batch, set
 *                 PKV_STATUS_BAD_ITEM and are skipped (their rows unwritten).
 * Everything else as paged_attention_prefill.  Rows of decodes and chunks must
 * not overlap.  Where the decodes' bound reaches the tensor-core route
 * (max_decode_len >= 16384) the two parts run one after the other.
 */
int paged_attention_mixed(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                          const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
                          const int32_t *q_start, int num_seqs, int total_q, int num_decodes,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, float scale, int max_decode_len, int decode_partition_size,
                          const int32_t *decode_items, int decode_grid, int prefill_ctas,
                          const int32_t *prefill_items, pkv_bf16 *out, void *workspace,
                          size_t workspace_bytes, int32_t *d_status, void *stream);

/*
 * paged_attention_decode_static_scratch -- paged_attention_decode without a
 * caller-provided workspace and without allocating anything.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: an engine that hands all of device memory to
 * its own arena at start-up and allows no allocation afterwards, or a plugin
 * whose host framework owns every allocation.  Arguments and results are those
 * of paged_attention_decode minus workspace / workspace_bytes.
 *
 * The split-K scratch is a fixed array of PKV_STATIC_SCRATCH_BYTES inside the
 * library; every GPU that loads the library keeps it until the process exits.
 * Calls whose scratch need (paged_attention_workspace_size) is larger return
 * PKV_ERR_WORKSPACE and launch nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  The call never invokes
 * cudaMalloc, cudaFree or any other allocating routine.  All calls share the
 * one array: calls whose kernels overlap on the GPU (different streams, or
 * several host threads) race on it and give undefined results; serialise them.
 * Nothing in the array needs to start at zero.
 */
#define PKV_STATIC_SCRATCH_BYTES (8u << 20)  /* 8 MiB */

int paged_attention_decode_static_scratch(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                          const pkv_bf16 *v_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *seq_lens,
                                          int num_seqs, int max_seq_len, int q_len,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, float scale,
                                          int partition_size, pkv_bf16 *out, int32_t *d_status,
                                          void *stream);

/*
 * pkv_swap_out / pkv_swap_in -- move whole blocks between the device caches
 * and page-locked host memory (the data side of pkv_seq_swap_out / _in).
 *
 * Pages: praveentn.live "PagedAttention KV-cache constraint", "What it cost"
 * (swapping blocks when memory runs out).  For i < n, with b = block_ids[i]:
 *   out:  host_k[i][:][:][:] = k_cache[b][:][:][:]   (same for v)
 *   in:   k_cache[b][:][:][:] = host_k[i][:][:][:]   (same for v)
 *   block_ids       device, [n] int32; ids outside [0, num_blocks) set
 *                   PKV_STATUS_BAD_BLOCK and are skipped
 *   host_k, host_v  page-locked host memory (cudaHostAlloc / cudaMallocHost /
 *                   cudaHostRegister), [n][num_kv_heads][block_size][head_dim]
 *                   bf16, 16-byte aligned; the kernel reads or writes it
 *                   directly through unified addressing.  Pageable memory is
 *                   refused (PKV_ERR_ARG).
 * Bit-exact copies; the ids of one call must be distinct for pkv_swap_in.
 */
int pkv_swap_out(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_ids, int n,
                 pkv_bf16 *host_k, pkv_bf16 *host_v, int num_blocks, int block_size, int num_kv_heads,
                 int head_dim, int32_t *d_status, void *stream);
int pkv_swap_in(const pkv_bf16 *host_k, const pkv_bf16 *host_v, const int32_t *block_ids, int n,
                pkv_bf16 *k_cache, pkv_bf16 *v_cache, int num_blocks, int block_size, int num_kv_heads,
                int head_dim, int32_t *d_status, void *stream);

/* ------------------------------------------------------------------------
 * Host block allocator: pool, block tables, refcounts, copy-on-write.
 *
 * Pages: a request grows by allocating more free blocks and returns them to
 * the pool when it ends; every free block is interchangeable (x321.org "The
 * serving bottleneck is not just FLOPs", "PagedAttention borrows an
 * operating-system trick"; praveentn.live "PagedAttention KV-cache
 * constraint", "What the change bought").  Blocks needed for L tokens:
 * ceil(L / block_size) (chenhuiyu.github.io "A complete explanation from first
 * principles", "Calculate a block-allocation example").
 *
 * Policy: free blocks form a LIFO stack that starts as [NB-1, ..., 1, 0]
 * (block 0 is handed out first); blocks whose refcount falls to zero are
 * pushed back in logical order.  Every failing call leaves the state
 * unchanged.  Host memory only; one owner; not thread-safe.
 * ------------------------------------------------------------------------ */
typedef struct pkv_alloc pkv_alloc;

int  pkv_alloc_create(int num_blocks, int block_size, pkv_alloc **out);
void pkv_alloc_destroy(pkv_alloc *a);

/* New empty sequence; PKV_ERR_ARG if seq_id exists. */
int pkv_seq_add(pkv_alloc *a, int64_t seq_id);

/* Append n_tokens >= 0 tokens: take ceil((len+n)/bs) - blocks new blocks and
 * write the n slots (host, int64) of positions len .. len+n-1 to slots_out.
 * PKV_ERR_OOM if too few blocks are free; PKV_ERR_SHARED if the tokens would
 * land in a partially filled block whose refcount is above 1 (call
 * pkv_seq_cow first). */
int pkv_seq_append(pkv_alloc *a, int64_t seq_id, int n_tokens, int64_t *slots_out);

/* Append n_tokens tokens with their ids (prefix caching).  Like pkv_seq_append,
 * except that a whole block of this call whose token prefix (every token from
 * the start of the sequence through the end of the block) matches a
 * registered block exactly is not stored again: the sequence's table points to
 * that block (its refcount + 1), the block's tokens get slot -1 (pkv_write
 * skips them) and count in *cached_out.  Every block this sequence fills is
 * registered under its prefix unless the prefix already names a block.
 * Registered blocks nobody holds stay cached and count as free; a block is
 * taken from the free stack first, else the least recently released cached
 * block is evicted.  Prefix caching follows a sequence while all its tokens
 * come through this call (fork and copy-on-write keep it); pkv_seq_append or a
 * swap-in ends it for that sequence.  Errors as pkv_seq_append; all lookups
 * are made before any block is taken, and a failing call changes nothing. */
int pkv_seq_append_tokens(pkv_alloc *a, int64_t seq_id, const int32_t *token_ids, int n_tokens,
                          int64_t *slots_out, int *cached_out);

/* Registered (content-addressed) blocks, and those of them nobody holds. */
int pkv_prefix_cache_stats(const pkv_alloc *a, int64_t *registered_blocks, int64_t *evictable_blocks);

/* pkv_seq_append for n distinct sequences at once, n_tokens each: the slots of
 * sequence i go to slots_out[i * n_tokens ...].  All or nothing: every check
 * (ids, shared partial blocks, enough free blocks for all) runs before any
 * sequence changes, so a failing call leaves the state unchanged; the blocks
 * are then taken in the order of seq_ids, exactly as n single appends would. */
int pkv_seq_append_batch(pkv_alloc *a, const int64_t *seq_ids, int n, int n_tokens, int64_t *slots_out);

/* child := a new sequence sharing every block of parent (refcount + 1 each). */
int pkv_seq_fork(pkv_alloc *a, int64_t parent, int64_t child);

/* Give seq_id a private copy of logical block `logical_block` (-1: the block the
 * next append writes into, none when the last block is full).  If that block's
 * refcount is above 1: take a free block, lower the old refcount, repoint the
 * table entry, write {src, dst} to pair_out and set *copied = 1; else set
 * *copied = 0.  The caller then runs pkv_block_copy on the pairs. */
int pkv_seq_cow(pkv_alloc *a, int64_t seq_id, int logical_block, int32_t *pair_out,
                int *copied);

/* Drop a sequence; blocks whose refcount reaches 0 return to the pool. */
int pkv_seq_free(pkv_alloc *a, int64_t seq_id);

/* Swap a resident sequence out (praveentn.live "PagedAttention KV-cache
 * constraint", "What it cost": under memory pressure blocks are swapped or
 * recomputed).  Writes its block ids in logical order (ceil(len / block_size)
 * of them; PKV_ERR_RANGE if more than max_blocks) to blocks_out and *n_out,
 * then releases them like pkv_seq_free does.  The caller copies those blocks
 * to host memory with pkv_swap_out, enqueued before anything that writes into
 * them again.  The sequence keeps its id and length but holds no block until
 * pkv_seq_swap_in: append, fork, cow and block_table refuse it (PKV_ERR_ARG);
 * pkv_seq_free drops it.  A shared block stays resident for its other owners;
 * the swapped sequence comes back with private copies. */
int pkv_seq_swap_out(pkv_alloc *a, int64_t seq_id, int32_t *blocks_out, int max_blocks, int *n_out);

/* Bring a swapped-out sequence back: take ceil(len / block_size) free blocks
 * as its new table (logical order), written to blocks_out and *n_out for the
 * caller's pkv_swap_in.  PKV_ERR_OOM, state unchanged, if too few are free. */
int pkv_seq_swap_in(pkv_alloc *a, int64_t seq_id, int32_t *blocks_out, int max_blocks, int *n_out);

/* Current length (tokens) of a sequence, or a negative error code. */
int64_t pkv_seq_len(const pkv_alloc *a, int64_t seq_id);

/* Host [n][max_blocks] table rows (-1 past each sequence's blocks) and int32
 * lengths.  PKV_ERR_RANGE if a sequence has more than max_blocks blocks. */
int pkv_block_table(const pkv_alloc *a, const int64_t *seq_ids, int n, int32_t *table_out,
                    int max_blocks, int32_t *lens_out);

/* Blocks that can be handed out: the free stack plus the cached blocks nobody holds. */
int pkv_num_free(const pkv_alloc *a);
/* Refcount of a block, or PKV_ERR_RANGE. */
int pkv_refcount(const pkv_alloc *a, int block);

/* ------------------------------------------------------------------------
 * Decode step runner: one decode step of a batch through every layer of a
 * model, issued by one host call.
 *
 * Pages: each decode step grows every running sequence by one token, taking a
 * new block when its last one is full, stores the token's keys and values in
 * its slot, and runs attention over the sequence's blocks through its table
 * (x321.org "The serving bottleneck is not just FLOPs", "PagedAttention
 * borrows an operating-system trick").  The runner chains exactly those calls
 * of this library: pkv_seq_append_batch, pkv_block_table, then per layer
 * pkv_write and paged_attention_decode (for single-token steps the pair as
 * paged_attention_decode_items over the pkv_decode_items work list the runner
 * builds from the step's lengths).  The pages have no counterpart to the
 * runner itself; it exists so that a serving loop pays one host call per step
 * instead of one per operation and per layer.
 *
 * Buffers (all owned by the caller, sized by pkv_step_layout_of):
 *   host_stage / dev_stage  page-locked host memory and device memory of
 *       layout.stage_bytes each, 16-byte aligned.  The caller writes each
 *       step's inputs into host_stage; the runner writes the slots, tables and
 *       lengths into it and copies all of it to dev_stage in one copy.
 *       Segments (byte offsets; every segment starts on a 256-byte boundary),
 *       first those every layer reads, then the layers one after the other:
 *         slots               slots_offset, [max_seqs * q_len] int64
 *         block tables        tables_offset, [max_seqs][max_blocks_per_seq] int32
 *         lengths             lens_offset, [max_seqs] int32
 *         work list (q_len 1) items_offset, [1 + max_items][4] int32
 *         queries of layer l  q_offset + l * layer_stride,
 *                             [max_seqs][q_len][num_q_heads][head_dim] bf16
 *                             (q_layer_bytes)
 *         new keys of layer l k_offset + l * layer_stride,
 *         new values          v_offset + l * layer_stride,
 *                             [max_seqs * q_len][num_kv_heads][head_dim] bf16
 *                             (kv_layer_bytes each)
 *       A run over n sequences uses the first n rows of each segment; the
 *       runner writes the work list itself.
 *   dev_out / host_out      device and page-locked host memory of
 *       layout.out_bytes; layer l's output [max_seqs][q_len][num_q_heads]
 *       [head_dim] bf16 at l * out_layer_bytes.  Each run copies all of
 *       dev_out to host_out.
 *   workspace               device, layout.workspace_bytes (split-K scratch
 *       for the longest sequence the tables can hold; may be NULL when 0).
 *   k_caches / v_caches     host arrays of num_layers device pointers, one
 *       pool per layer, each [num_blocks][num_kv_heads][block_size][head_dim].
 *
 * With use_graph != 0 the device part of a run (copy in, the layers' writes
 * and decodes, copy out) is captured once into a CUDA graph for each key
 * (n, number of partitions of the longest sequence, partition size, and for
 * single tokens the work list's item count rounded up to 256: the captured
 * decode grid, whose CTAs past the count return at once) and replayed; the
 * decode's max_seq_len is then that number of partitions times the partition
 * size, an upper bound of the lengths (at most 32 graphs are kept; capture
 * happens on a private stream).  With use_graph == 0 the same copies and kernels are
 * enqueued one by one on every run, with the exact maximum length.  Graphs
 * save host time when a step has many short kernels (many layers); a step of
 * a few long kernels gains nothing from them.
 * ------------------------------------------------------------------------ */
typedef struct {
  int num_layers;          /* >= 1 */
  int max_seqs;            /* largest batch of a run, >= 1 */
  int q_len;               /* new tokens per sequence and step (1 or 16) */
  int num_q_heads, num_kv_heads, head_dim;
  int block_size, num_blocks, max_blocks_per_seq;
  int partition_size;      /* as paged_attention_decode; 0 = its default */
  float scale;
  int use_graph;           /* 0: enqueue calls one by one; else CUDA graphs */
} pkv_step_config;

typedef struct {
  size_t q_offset, q_layer_bytes;
  size_t k_offset, v_offset, kv_layer_bytes;
  size_t slots_offset, tables_offset, lens_offset;
  size_t stage_bytes;      /* host_stage and dev_stage */
  size_t out_layer_bytes, out_bytes;
  size_t workspace_bytes;
  size_t items_offset;     /* q_len 1: the decode's work list (pkv_decode_items), 0 otherwise */
  int max_items;           /* rows of that list after its header */
  size_t layer_stride;     /* bytes from one layer's queries, keys, values to the next layer's */
} pkv_step_layout;

typedef struct pkv_step pkv_step;

/* Buffer layout of a configuration (host only).  PKV_ERR_ARG for sizes below
 * 1 (partition_size below 0) or byte counts that overflow. */
int pkv_step_layout_of(const pkv_step_config *cfg, pkv_step_layout *layout);

/* Create a runner over an allocator and caller-owned buffers (see above).
 * Like the allocator, a runner has one owner and is not thread-safe.
 * PKV_ERR_ARG for a null, misaligned or too small buffer, or a host buffer
 * that is not page-locked; PKV_ERR_CUDA if the runner's event or stream cannot
 * be made.  The allocator, caches and buffers must outlive the runner. */
int pkv_step_create(const pkv_step_config *cfg, pkv_alloc *alloc, pkv_bf16 *const *k_caches,
                    pkv_bf16 *const *v_caches, void *host_stage, void *dev_stage, pkv_bf16 *dev_out,
                    pkv_bf16 *host_out, void *workspace, size_t workspace_bytes, int32_t *d_status,
                    pkv_step **out);

/* Waits for the runner's last run, then releases its graphs, event and stream. */
void pkv_step_destroy(pkv_step *s);

/* One step for the n <= max_seqs distinct sequences seq_ids (host array):
 *   1. wait until the runner's previous run has finished on the GPU;
 *   2. check that every sequence has room for q_len more tokens in
 *      max_blocks_per_seq blocks (PKV_ERR_RANGE, nothing changed, if not);
 *      with use_graph, capture the step's graph if its key (above) has none
 *      yet (a failed capture returns its error, nothing changed);
 *   3. pkv_seq_append_batch of q_len tokens each (its errors are returned and
 *      change nothing), slots into host_stage; pkv_block_table of the n
 *      sequences into host_stage;
 *   4. enqueue: the common segments and layer 0's inputs host_stage ->
 *      dev_stage, then each further layer's inputs, on a copy stream of the
 *      runner's own; on `stream`, for each layer l once its inputs have
 *      landed, the pkv_write of its n * q_len new keys and values and the
 *      paged_attention_decode of its n query rows (q_len = 1: both as one
 *      paged_attention_decode_items over the step's work list); each layer's
 *      output dev_out -> host_out on the copy stream as soon as its kernels
 *      finish.  The copies of one layer overlap the kernels of the others;
 *      `stream` waits for the last output copy, so the step is complete on
 *      `stream` (for events or graphs) as before.
 * Returns after the enqueue.  The caller writes the step's queries, keys and
 * values for rows 0..n-1 into host_stage before the call, and may touch
 * host_stage and host_out again only after pkv_step_wait (or a synchronisation
 * of `stream`).  Every failure except a CUDA error from the enqueue itself
 * leaves the allocator unchanged.  A CUDA error in step 4 returns PKV_ERR_CUDA
 * with the tokens appended but their keys and values not stored: the caller
 * must free those sequences (or store the tokens itself) before decoding them
 * again.  n == 0 only waits. */
int pkv_step_run(pkv_step *s, const int64_t *seq_ids, int n, void *stream);

/* Block until the runner's last run has finished; PKV_ERR_CUDA on failure. */
int pkv_step_wait(pkv_step *s);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
