/*
 * pagedkv.h -- C ABI of libpagedkv: decode-time paged attention on GB300.
 *
 * A sequence's key/value cache is split into fixed-size blocks of B token
 * slots. The blocks live in one shared pool and are reached through the
 * sequence's block table, which maps logical block index to physical block
 * number ("Paged KV Cache Allocation and the Block Table", section "Blocks,
 * tables, and the indirection"; "paged attention deep", section "The block
 * table"). Token t of a sequence lives at
 *
 *     slot = block_table[t / B] * B + (t % B)
 *
 * ("The KV Cache Is an Allocator Problem", the physical-address equation).
 *
 * Conventions shared by every GPU entry point:
 *   - Pool layout: k_cache and v_cache are each [num_blocks, B, Hk, d],
 *     row-major, so a block holds K [B, Hk, d] and V [B, Hk, d] ("paged
 *     attention deep", "Anatomy of a KV block"; the S06 listing's pool shape).
 *   - New-token layout: k, v are [T, Hk, d]; queries and outputs [S, Hq, d].
 *   - Query head h reads KV head h / (Hq / Hk).
 *   - Every pointer argument of a GPU entry point is a DEVICE pointer owned
 *     by the caller and 16-byte aligned. The library allocates no device
 *     memory: split-K scratch is passed in by the caller.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *     enqueued asynchronously; the call returns after the launches.
 *   - Host-side argument checks run before any launch and return a status;
 *     nothing aborts, traps or prints. Launch failures map to PK_ERR_CUDA.
 *   - Device-side bounds checks (slot, block id, pair, context length) never
 *     touch memory out of range: the offending access is skipped and the
 *     first such event is recorded in a device error word, read back with
 *     pk_get_device_error().
 *
 * The host block manager (pk_bm_*) owns only host memory and is not
 * thread-safe: one handle per thread, or external locking.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PK_OK = 0,
    PK_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, bad layout      */
    PK_ERR_UNSUPPORTED = 2,   /* valid but not compiled: dtype, head_dim, B, group size */
    PK_ERR_OUT_OF_BLOCKS = 3, /* the pool cannot supply the blocks; state unchanged     */
    PK_ERR_UNKNOWN_SEQ = 4,   /* no sequence with that id                               */
    PK_ERR_SEQ_EXISTS = 5,    /* a sequence with that id already exists                 */
    PK_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed                   */
    PK_ERR_WORKSPACE = 7,     /* split-K workspace missing or too small                 */
    PK_ERR_INVARIANT = 8,     /* pk_bm_check_invariants found a violation               */
    PK_ERR_NOMEM = 9          /* host allocation failed                                 */
} pk_status;

typedef enum { PK_F32 = 0, PK_BF16 = 1 } pk_dtype;

/* Attention kernel choice. AUTO picks the tensor-core kernel for bf16 when it
 * is compiled for the shape and the CUDA-core kernel otherwise. */
typedef enum { PK_ATTN_AUTO = 0, PK_ATTN_SIMT = 1, PK_ATTN_MMA = 2 } pk_attn_impl;

/* Device error word layout: (kind << 24) | (low 24 bits of the offending index). */
enum {
    PK_DEVERR_NONE = 0,
    PK_DEVERR_SLOT = 1,        /* slot_mapping entry >= num_blocks * B                 */
    PK_DEVERR_BLOCK_ID = 2,    /* block table entry outside [0, num_blocks)            */
    PK_DEVERR_PAIR = 3,        /* copy_blocks pair outside [0, num_blocks)             */
    PK_DEVERR_CONTEXT = 4,     /* context_lens entry < 1 or beyond the table / bound   */
    PK_DEVERR_TIMEOUT = 5,     /* a pipeline wait gave up (never expected)             */
    PK_DEVERR_ORDER = 6        /* seq_order entry outside [0, num_seqs)                */
};

/* Geometry of one layer's KV pool. */
typedef struct {
    int32_t num_blocks;   /* N: physical blocks in the pool          */
    int32_t block_size;   /* B: token slots per block                */
    int32_t num_kv_heads; /* Hk                                      */
    int32_t head_dim;     /* d                                       */
    pk_dtype dtype;       /* element type of caches, q, k, v and out */
} pk_cache_desc;

/* ------------------------------------------------------------------------ */
/* GPU entry points                                                         */
/* ------------------------------------------------------------------------ */

/* Slot scatter: for each new token i with s = slot_mapping[i] >= 0,
 *     k_cache[s / B, s % B, :, :] = k[i, :, :]   and the same for v.
 * Negative slots are skipped. ("Paged KV Cache Allocation and the Block
 * Table", the append_token routine: the token's K/V are written at
 * physical * block_size + slot.)
 *   k, v          [num_tokens, Hk, d] contiguous, dtype of the pool.
 *   slot_mapping  int64 [num_tokens]; duplicate slots in one call race.
 *   num_tokens    >= 0 (0 is a no-op).
 * Out-of-range slots are skipped and recorded (PK_DEVERR_SLOT). */
pk_status pk_reshape_and_cache(const void *k, const void *v, const int64_t *slot_mapping,
                               int32_t num_tokens, void *k_cache, void *v_cache,
                               const pk_cache_desc *desc, void *stream);

/* The slot scatter of one decode step plus its block-table bookkeeping on
 * device-resident tables ("Paged KV Cache Allocation and the Block Table",
 * append_token; "The KV Cache Is an Allocator Problem", the physical-address
 * equation). Token i is the next token of row i: its position is
 * pos = context_lens[i]; its K/V go to slot_mapping[i] as in
 * pk_reshape_and_cache; block_tables[i][pos / B] becomes slot_mapping[i] / B
 * (the block holding the token, whether newly opened or a copy-on-write
 * replacement) and context_lens[i] becomes pos + 1. block_tables is
 * [num_tokens, max_blocks_per_seq] int32 and context_lens [num_tokens] int32,
 * both device memory, updated in place. A row whose pos is outside the table,
 * or whose slot is not at offset pos mod B of its block, is left unchanged
 * and recorded (PK_DEVERR_CONTEXT); its K/V are still written. */
pk_status pk_reshape_and_cache_append(const void *k, const void *v, const int64_t *slot_mapping,
                                      int32_t num_tokens, void *k_cache, void *v_cache,
                                      const pk_cache_desc *desc, int32_t *block_tables,
                                      int32_t max_blocks_per_seq, int32_t *context_lens,
                                      void *stream);

/* Copy-on-write block copy: for each pair p, the whole block src = pairs[2p]
 * is copied to dst = pairs[2p+1] in both k_cache and v_cache (all B slots, all
 * heads). ("paged attention deep", "Copy-on-write for shared prefixes": the
 * writer gets a private copy of the single shared block; "Paged KV Cache
 * Allocation and the Block Table", "Sharing blocks between sequences".)
 *   src_dst_pairs int64 [num_pairs][2]. Precondition: the dst blocks are
 *                 distinct and no dst is also a src in the same call.
 * Must be enqueued before the scatter that writes into dst.
 * Out-of-range ids are skipped and recorded (PK_DEVERR_PAIR). */
pk_status pk_copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                         int32_t num_pairs, const pk_cache_desc *desc, void *stream);

/* Swap copies for preemption ("Paged KV Cache Allocation and the Block
 * Table", "What the design costs": a sequence's blocks swapped to host memory
 * and restored). Copies whole blocks (K and V) between the device pool and a
 * host pool of the same block shape, [num_host_blocks, B, Hk, d]:
 *   direction PK_SWAP_OUT: pairs[p] = (device block, host block);
 *   direction PK_SWAP_IN:  pairs[p] = (host block, device block)
 * -- exactly the pairs pk_bm_swap_out / pk_bm_swap_in return.
 *   k_host, v_host  pinned host memory the device can address (cudaHostAlloc
 *                   or registered); PK_ERR_INVALID_ARG otherwise.
 *   pairs           int64 [num_pairs][2], readable by the device (device
 *                   memory or pinned host memory).
 * A swap-out must be enqueued before anything writes the device blocks it
 * freed; a swap-in before anything reads the sequence's new blocks.
 * Out-of-range ids are skipped and recorded (PK_DEVERR_PAIR). */
enum { PK_SWAP_OUT = 0, PK_SWAP_IN = 1 };
pk_status pk_swap_blocks(void *k_cache, void *v_cache, void *k_host, void *v_host,
                         int32_t num_host_blocks, const int64_t *pairs, int32_t num_pairs,
                         int32_t direction, const pk_cache_desc *desc, void *stream);

/* Decode attention through the block table ("PagedAttention", S06, the
 * paged_attention listing and "Why this needed a custom CUDA kernel": the
 * table lookup happens inside the kernel, no pre-gather). For each sequence
 * s and query head h, with n = context_lens[s] and kvh = h / (Hq / Hk):
 *     x_t = scale * <q[s,h,:], K[table[s][t/B], t%B, kvh, :]>     t < n
 *     out[s,h,:] = sum_t softmax(x)_t * V[table[s][t/B], t%B, kvh, :]
 *   out           [S, Hq, d], dtype of q (fp32 accumulation inside).
 *   q             [S, Hq, d].
 *   block_size    B, the listing's block_size argument: must equal
 *                 desc->block_size (PK_ERR_INVALID_ARG otherwise).
 *   block_tables  int32 [S, max_blocks_per_seq]; entries at or beyond
 *                 ceil(n / B) are never read.
 *   context_lens  int32 [S], each in [1, min(max_context_len, max_blocks*B)];
 *                 the length after the step's token has been scattered.
 *   max_context_len  host-side upper bound on context_lens (sizes the grid).
 *   partition_size   0: one partition per sequence (no split-K);
 *                    -1: automatic; > 0: split each context into partitions
 *                    of this many tokens (a multiple of B), merged with a
 *                    log-sum-exp reduction. With the tensor-core kernel the
 *                    merge is a second launch on `stream`, enqueued as the
 *                    attention launch's programmatic dependent (it starts
 *                    while the attention drains and waits for it to finish
 *                    before reading); it runs only when the call splits.
 *   workspace        device scratch of at least
 *                    pk_paged_attention_workspace_size(...) bytes when the
 *                    chosen partitioning splits; may be NULL otherwise.
 * A context length outside its bounds is clamped and recorded
 * (PK_DEVERR_CONTEXT); a bad table entry is recorded (PK_DEVERR_BLOCK_ID). */
pk_status pk_paged_attention_decode(void *out, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_tables,
                                    const int32_t *context_lens, float scale, int32_t block_size,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    int32_t max_blocks_per_seq, int32_t max_context_len,
                                    int32_t partition_size, void *workspace,
                                    size_t workspace_bytes, const pk_cache_desc *desc,
                                    void *stream);

/* As pk_paged_attention_decode without the block_size argument (B is
 * desc->block_size), plus two scheduling controls:
 *   seq_order  optional device int32 [S], a permutation of 0..S-1: the order in
 *              which sequences' work is launched (NULL = index order). Results
 *              do not depend on it; launching the longest sequences first
 *              (pk_longest_first_order) keeps the longest work from trailing.
 *              An entry outside [0, S) is recorded (PK_DEVERR_ORDER).
 *   impl       the kernel (PK_ERR_UNSUPPORTED if not compiled for the shape). */
pk_status pk_paged_attention_decode_impl(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, float scale,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_blocks_per_seq, int32_t max_context_len,
                                         int32_t partition_size, void *workspace,
                                         size_t workspace_bytes, const pk_cache_desc *desc,
                                         const int32_t *seq_order, pk_attn_impl impl,
                                         void *stream);

/* Host helper for seq_order: order_out[0..n-1] = sequence indices sorted by
 * descending context_lens (host int32 [n]), ties by index. */
pk_status pk_longest_first_order(const int32_t *context_lens, int32_t num_seqs,
                                 int32_t *order_out);

/* As pk_paged_attention_decode_impl, with the work given as a list of items
 * instead of the (sequence, partition) grid: work_items is device int32
 * [num_items][2], item y = (sequence, partition index), and one CTA per
 * (KV head, item) runs. Only the listed items run, so a split whose longest
 * context sets the partition count launches nothing for the shorter
 * sequences' missing partitions. Precondition: the list holds every
 * partition of every sequence exactly once for the resolved partition size
 * (pk_paged_attention_resolve_partition) and the context lengths the kernel
 * reads -- pk_attention_work_items builds it; an item outside the batch or
 * the partition count is skipped and recorded (PK_DEVERR_ORDER). Results do
 * not depend on the item order. 1 <= num_items <= 65535. */
pk_status pk_paged_attention_decode_items(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, float scale,
                                          int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, int32_t max_context_len,
                                          int32_t partition_size, const int32_t *work_items,
                                          int32_t num_items, void *workspace,
                                          size_t workspace_bytes, const pk_cache_desc *desc,
                                          pk_attn_impl impl, void *stream);

/* One decode step's slot scatter fused into its attention: as
 * pk_reshape_and_cache(k_new, v_new, slot_mapping, num_seqs, ...) followed by
 * pk_paged_attention_decode_items, where token i of k_new / v_new
 * ([num_seqs, Hk, d]) is the last token of sequence i (its context length
 * counts it). The tensor-core kernel writes each sequence's new K/V for a KV
 * head in the CTA that then reads that head -- the one whose partition holds
 * the token -- ordering the write before its TMA reads, so the step needs no
 * separate scatter launch; otherwise the scatter runs first as its own
 * kernel. Copy-on-write copies (pk_copy_blocks) must be enqueued before. */
pk_status pk_paged_attention_decode_append(
    void *out, const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
    void *k_cache, void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
    float scale, int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
    int32_t max_context_len, int32_t partition_size, const int32_t *work_items, int32_t num_items,
    void *workspace, size_t workspace_bytes, const pk_cache_desc *desc, void *stream);

/* One decode step on device-resident block tables in one launch: the step's
 * slot scatter, its block-table bookkeeping and the attention ("Paged KV
 * Cache Allocation and the Block Table", append_token; "PagedAttention",
 * S06). The same result as pk_reshape_and_cache_append followed by
 * pk_paged_attention_decode_items over the advanced lengths, with:
 *   context_lens      int32 [S] (device), each sequence's length before the
 *                     step's token; read only;
 *   context_lens_out  int32 [S] (device), receives context_lens + 1; must not
 *                     alias context_lens (alternate two buffers between
 *                     steps). A row whose slot is not at offset
 *                     context_lens[i] mod B of its block receives
 *                     context_lens[i] unchanged and is recorded
 *                     (PK_DEVERR_CONTEXT);
 *   block_tables      updated in place: row i's entry of the block holding
 *                     position context_lens[i] becomes slot_mapping[i] / B
 *                     (a newly opened block or a copy-on-write replacement);
 *   max_context_len, partition_size, work_items: for the advanced lengths.
 * The tensor-core kernel does all of it inside the attention launch: the CTA
 * holding a sequence's new token takes that token's block from its slot
 * instead of the table, writes the token's K/V for its KV head, and for KV
 * head 0 also writes the table entry and the new length. The CUDA-core
 * kernel runs the scatter and bookkeeping as its own kernel first.
 * Copy-on-write copies (pk_copy_blocks) must be enqueued before. */
pk_status pk_paged_attention_decode_advance(
    void *out, const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
    void *k_cache, void *v_cache, int32_t *block_tables, const int32_t *context_lens,
    int32_t *context_lens_out, float scale, int32_t num_seqs, int32_t num_q_heads,
    int32_t max_blocks_per_seq, int32_t max_context_len, int32_t partition_size,
    const int32_t *work_items, int32_t num_items, void *workspace, size_t workspace_bytes,
    const pk_cache_desc *desc, void *stream);

/* Host helper for pk_paged_attention_decode_items: the items of sequences
 * with host context_lens [n] cut into partitions of `partition` tokens (0 = no
 * split; pass the resolved size), longest item first (ties: the longer
 * sequence, then batch order, then the later partition) -- the
 * longest-processing-time-first order. *num_items_out receives the count;
 * PK_ERR_INVALID_ARG if it exceeds cap (items_out untouched). */
pk_status pk_attention_work_items(const int32_t *context_lens, int32_t num_seqs,
                                  int32_t partition, int32_t *items_out, int32_t cap,
                                  int32_t *num_items_out);

/* Host planner for pk_paged_attention_decode_items: the partition size and
 * the work list of a batch whose host context lengths are known.
 * partition_size > 0 or 0 is used as given (0 = no split); -1 chooses from
 * the lengths: with W = (sum of context lengths x Hk) / (SMs x resident CTAs
 * per SM of the kernel that will run), a batch whose longest context is
 * above 2W (and 1024 tokens) is cut into items of about W tokens -- k equal
 * parts of the longest context, k = floor(max / W), multiples of 64 tokens,
 * at least 512 -- else it stays whole. *partition_out receives the size (0 =
 * no split); pass it as partition_size to the attention call and size the
 * workspace with pk_paged_attention_workspace_size for it (any choice of -1
 * is covered by the size for 512). Items as pk_attention_work_items. */
pk_status pk_attention_plan(const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t partition_size, const pk_cache_desc *desc,
                            int32_t *partition_out, int32_t *items_out, int32_t cap,
                            int32_t *num_items_out);

/* Allocation-free decode attention. The pages have no counterpart: this is a
 * library convenience for callers that cannot allocate device memory -- a
 * serving engine whose memory planner already gave nearly all HBM to the KV
 * pool, a host framework's operator hook that supplies only input and output
 * buffers, or a latency-critical loop that cannot pay for cudaMalloc/cudaFree
 * and their implicit synchronisation.
 * Same arguments and result as pk_paged_attention_decode, minus the
 * workspace: the split-K scratch is a static device array of
 * PK_STATIC_WORKSPACE_BYTES that every GPU loading the library holds until
 * the process exits. The call allocates nothing.
 *   - Returns PK_ERR_WORKSPACE, before any launch, when the partitioning
 *     needs more scratch than PK_STATIC_WORKSPACE_BYTES
 *     (see pk_paged_attention_workspace_size).
 *   - The first call on a device looks up the array's device address for
 *     that device (with the device current); make that first call before
 *     any stream capture.
 *   - All calls on a device share the one array, and it keeps the last
 *     call's contents; nothing in it needs to start at zero (every partial
 *     the merge reads is written earlier in the same call). Calls whose work
 *     overlaps on the GPU (e.g. on two streams) race on it.
 *   - The array's address is kept per device ordinal for the life of the
 *     process: it assumes the device's primary context is never reset
 *     (cudaDeviceReset) while the library is loaded. */
#define PK_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)
pk_status pk_paged_attention_decode_static(void *out, const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *block_tables,
                                           const int32_t *context_lens, float scale,
                                           int32_t block_size, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t max_blocks_per_seq,
                                           int32_t max_context_len, int32_t partition_size,
                                           const pk_cache_desc *desc, void *stream);

/* Cascade (shared-prefix) decode attention ("PagedAttention" S06, "In
 * production": the shared prefix batched separately from the divergent
 * suffixes; "Copy-on-write, for free": forked samples share the prefix
 * blocks). Same result as pk_paged_attention_decode, but for each group of
 * sequences that share their first prefix tokens (pk_bm_prefix_groups) the
 * prefix K/V is read once per KV head and scored against every member's
 * queries; each member's remaining tokens are attended on their own, and
 * the parts are merged by log-sum-exp.
 *   group_offsets    device int32 [num_groups + 1] into group_members;
 *   group_members    device int32, batch positions of the members (the first
 *                    member's table supplies the prefix blocks);
 *   group_prefix_len device int32 [num_groups], shared tokens (multiple of B);
 *   seq_prefix_len   device int32 [S], shared tokens of each batch position
 *                    (0 outside groups);
 *   max_group_size   members per group; G * max_group_size <= 16;
 *   max_prefix_len   host bound on group_prefix_len;
 *   partition_size   0: one partition for the prefix and one for the rest;
 *                    > 0: partitions of this many tokens (a multiple of B);
 *                    -1: automatic (one partition when num_groups x Hk covers
 *                    the SMs, else prefix partitions that do, >= 512 tokens);
 *   seq_order        optional launch order of the suffix work (see _impl);
 *   workspace        pk_cascade_workspace_size(...) bytes (required).
 * bf16 only (PK_ERR_UNSUPPORTED otherwise). With num_groups == 0 this is
 * pk_paged_attention_decode_impl with the automatic kernel. */
pk_status pk_cascade_attention_decode(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, float scale, int32_t num_seqs,
    int32_t num_q_heads, int32_t max_blocks_per_seq, int32_t max_context_len,
    int32_t partition_size, const int32_t *group_offsets, const int32_t *group_members,
    const int32_t *group_prefix_len, const int32_t *seq_prefix_len, int32_t num_groups,
    int32_t max_group_size, int32_t max_prefix_len, const int32_t *seq_order, void *workspace,
    size_t workspace_bytes, const pk_cache_desc *desc, void *stream);

/* Workspace bytes of pk_cascade_attention_decode: fp32 partials
 * [S, Hq, Ppre + Psuf, d + 2] (Ppre = ceil(max_prefix_len / partition),
 * Psuf = ceil(max_context_len / partition)); 0 on invalid arguments. Host
 * only. */
size_t pk_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                 int32_t num_groups, int32_t max_prefix_len,
                                 int32_t partition_size, const pk_cache_desc *desc);

/* The partition size (in tokens) that a partition_size argument resolves to
 * for this shape: 0 means no split. Host only, no GPU needed. */
int32_t pk_paged_attention_resolve_partition(int32_t num_seqs, int32_t num_q_heads,
                                             int32_t max_context_len, int32_t partition_size,
                                             const pk_cache_desc *desc);

/* Bytes of split-K workspace pk_paged_attention_decode needs for these
 * arguments (0 when the resolved partitioning does not split). Layout inside:
 * fp32 partial outputs [S, Hq, P, d], then running maxima and sums [S, Hq, P]
 * each, P = ceil(max_context_len / partition). Every partial the merge reads
 * is written earlier in the same call, so the workspace needs no clearing;
 * calls whose work overlaps on the GPU must not share a workspace. Host
 * only. */
size_t pk_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, int32_t partition_size,
                                         const pk_cache_desc *desc);

/* A pure read stream over `bytes` (a multiple of 16; device memory, 16-byte
 * aligned): every 16-byte vector is loaded once and the loads are folded so
 * none can be dropped; *sink (device) is left unchanged in practice. A
 * reference for the read bandwidth the attention kernels can reach, measured
 * by the benchmark beside them. Not part of the decode path. */
pk_status pk_read_stream(const void *buf, size_t bytes, unsigned int *sink, void *stream);

/* Self-test of the bounded pipeline waits: one CTA waits on an mbarrier
 * phase that nothing completes, polling at most `polls` times (0: the limit
 * every pipeline wait of the attention kernels uses), then records
 * PK_DEVERR_TIMEOUT (index 0) in the device error word and returns -- what a
 * stuck pipeline stage does instead of hanging. Touches no caller memory. */
pk_status pk_selftest_wait_timeout(uint32_t polls, void *stream);

/* Reads the device error word of the current device into *code_out (0 = no
 * error; see PK_DEVERR_*) after synchronising `stream`, then clears it. */
pk_status pk_get_device_error(int32_t *code_out, void *stream);

/* A static, NUL-terminated description of a status. */
const char *pk_status_string(pk_status status);

/* ------------------------------------------------------------------------ */
/* Host block manager                                                       */
/* ------------------------------------------------------------------------ */
/* Free list, per-sequence block tables, reference counts, fork and
 * copy-on-write ("Paged KV Cache Allocation and the Block Table", the
 * append_token routine and "Sharing blocks between sequences"; "PagedAttention",
 * S06, the BlockManager listing and "Reference counts must be exact").
 * The free list is a stack: its first pop is alloc_order[0]; a retired
 * sequence's blocks whose count reaches zero are pushed in table order. */
typedef struct pk_bm pk_bm;

/* alloc_order: a permutation of 0..num_blocks-1 (copied), or NULL for
 * 0, 1, 2, ... On success *out owns a new manager. */
pk_status pk_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *alloc_order,
                       pk_bm **out);
void pk_bm_destroy(pk_bm *bm);

pk_status pk_bm_add_seq(pk_bm *bm, int64_t seq_id);

/* Appends n >= 0 tokens to seq_id. slots_out[i] (int64, n entries) receives
 * token i's slot. When the sequence's first new token falls into a partly
 * filled tail block shared with another table, the block is copied first:
 * the (src, dst) pair goes to cow_pairs_out[0..1] and *n_cow_out = 1 (else
 * 0); the caller must run pk_copy_blocks on it before the scatter. All or
 * nothing: PK_ERR_OUT_OF_BLOCKS leaves the manager unchanged. */
pk_status pk_bm_append_slots(pk_bm *bm, int64_t seq_id, int32_t n, int64_t *slots_out,
                             int64_t *cow_pairs_out, int32_t *n_cow_out);

/* One decode step's host side: appends one token to each of seq_ids[0..n-1]
 * in order. slots_out [n] gets the slots; cow_pairs_out [n][2] gets the copy
 * pairs in order and *n_cow_out their count. All or nothing over the batch. */
pk_status pk_bm_append_batch(pk_bm *bm, const int64_t *seq_ids, int32_t n, int64_t *slots_out,
                             int64_t *cow_pairs_out, int32_t *n_cow_out);

/* child gets the parent's table and length; every block's count goes up. */
pk_status pk_bm_fork(pk_bm *bm, int64_t parent, int64_t child);

/* Decrements every block of the table; blocks reaching zero return to the
 * free list. */
pk_status pk_bm_free_seq(pk_bm *bm, int64_t seq_id);

pk_status pk_bm_seq_len(const pk_bm *bm, int64_t seq_id, int64_t *len_out);

/* Copies up to cap entries of the table; *len_out = its full length. */
pk_status pk_bm_block_table(const pk_bm *bm, int64_t seq_id, int32_t *out, int32_t cap,
                            int32_t *len_out);

/* Row i of tables_out [n][max_blocks] = the table of seq_ids[i], padded with
 * -1; lens_out[i] (int32) = its token count. PK_ERR_INVALID_ARG if a table is
 * longer than max_blocks. */
pk_status pk_bm_export_tables(const pk_bm *bm, const int64_t *seq_ids, int32_t n,
                              int32_t max_blocks, int32_t *tables_out, int32_t *lens_out);

int32_t pk_bm_num_free(const pk_bm *bm);
int32_t pk_bm_refcount(const pk_bm *bm, int32_t block); /* -1 if out of range */

/* Recounts every block's references from the tables and checks: counts
 * match, no named block is free, no block is lost or listed twice, each
 * table holds ceil(len / B) blocks, every cached block is found by its own
 * key, and named + free + unreferenced cached blocks make up the pool.
 * PK_ERR_INVARIANT on the first violation. */
pk_status pk_bm_check_invariants(const pk_bm *bm);

/* Swap space for preemption: num_host_blocks host blocks, handed out first
 * to last as host_order[0], host_order[1], ... (NULL: 0, 1, 2, ...). Once. */
pk_status pk_bm_set_swap_space(pk_bm *bm, int32_t num_host_blocks, const int32_t *host_order);

/* Swaps a sequence out: every block of its table, in table order, gets a
 * host block; pairs_out[j] = (device block, host block) for pk_swap_blocks
 * (PK_SWAP_OUT); the device block loses the sequence's reference and returns
 * to the free list when no table names it (a block shared with a fork stays).
 * cap >= table length. All or nothing (PK_ERR_OUT_OF_BLOCKS when the swap
 * space is short). A swapped sequence cannot append, fork or be exported;
 * pk_bm_free_seq returns its host blocks. */
pk_status pk_bm_swap_out(pk_bm *bm, int64_t seq_id, int64_t *pairs_out, int32_t cap,
                         int32_t *n_out);

/* Swaps a sequence back in: fresh private device blocks in table order;
 * pairs_out[j] = (host block, device block) for pk_swap_blocks (PK_SWAP_IN);
 * the host blocks return to the swap space. All or nothing
 * (PK_ERR_OUT_OF_BLOCKS when the device pool is short). */
pk_status pk_bm_swap_in(pk_bm *bm, int64_t seq_id, int64_t *pairs_out, int32_t cap,
                        int32_t *n_out);

int32_t pk_bm_is_swapped(const pk_bm *bm, int64_t seq_id); /* 1, 0, or -1 if unknown */
int32_t pk_bm_host_free(const pk_bm *bm);                 /* free swap-space blocks   */

/* Prefix caching ("PagedAttention" S06, "What's next": block contents are
 * hashed so that any two requests with a common prefix share the same
 * physical blocks). Only full blocks are cached. A block's key is every token
 * id of the prompt up to and including the block: a 64-bit hash chained over
 * the blocks, verified on lookup against the block's depth, its parent's
 * chain hash and its own B token ids (a false hit needs two different
 * prefixes with equal 64-bit chain hashes and equal last blocks). A cached
 * block that loses its last reference stays cached and unreferenced (it still
 * counts in pk_bm_num_free); allocations take the free list first and then
 * evict the unreferenced cached block released longest ago (deepest first
 * among blocks released by one call). Host only: the K/V of a cached block
 * stay where the first request wrote them. */

/* New sequence whose prompt is tokens[0, n): its table starts with every
 * leading full block found in the cache (a hit at block j needs all of
 * tokens[0, (j+1)B) to match; the first miss ends the walk), each named once
 * more. Its length becomes *n_cached_out = hits * B; the caller appends the
 * remaining n - *n_cached_out tokens with pk_bm_append_slots and writes their
 * K/V. A caller that must compute the last prompt token passes n - 1. */
pk_status pk_bm_add_seq_cached(pk_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t n,
                               int32_t *n_cached_out);

/* Registers the full blocks among the first n tokens of a sequence (tokens =
 * its token ids, n <= its length; their K/V written on the stream that later
 * readers use): block j gets the key of tokens[0, (j+1)B) unless it is cached
 * already or another block holds that key (the first stays). */
pk_status pk_bm_commit(pk_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t n);

/* Tokens of tokens[0, n) that pk_bm_add_seq_cached would find cached now. */
pk_status pk_bm_cache_match(const pk_bm *bm, const int32_t *tokens, int32_t n,
                            int32_t *n_cached_out);

/* Cached blocks, of which unreferenced; blocks served from the cache since
 * creation; cached blocks evicted by allocations. NULL outputs are skipped. */
pk_status pk_bm_cache_stats(const pk_bm *bm, int64_t *cached, int64_t *unreferenced,
                            int64_t *hits, int64_t *evictions);
int32_t pk_bm_is_cached(const pk_bm *bm, int32_t block); /* 1, 0, or -1 if out of range */

/* The free list, next block to be handed out first: up to cap ids into out,
 * the list's length into *n_out. Unreferenced cached blocks are not on it. */
pk_status pk_bm_free_blocks(const pk_bm *bm, int32_t *out, int32_t cap, int32_t *n_out);

/* ------------------------------------------------------------------------ */
/* Allocator policy simulator                                               */
/* ------------------------------------------------------------------------ */
/* "The KV Cache Is an Allocator Problem", section "The experiment": one
 * deterministic trace of requests replayed against a cache of `capacity`
 * token slots under one policy. Each step t: (1) every request admitted
 * before t that has generated fewer than `gen` tokens tries to grow by one
 * slot, in trace order; a failure drops it (PK_SIM_DROP: its cache is
 * released) or leaves it to retry next step (PK_SIM_STALL); (2) requests
 * whose completion step is t release their cache; (3) requests arriving at
 * t are admitted, in trace order, if their prompt's cache (for maximum
 * reservation: prompt + max_new slots) can be allocated, else rejected.
 * Contiguous placement is first fit; the paged policy runs this library's
 * block manager on floor(capacity / B) blocks handed out 0, 1, 2, ...
 * Host only; single-threaded; no allocation survives the call. */
typedef struct {
    int32_t arrival;     /* step the request arrives, >= 0                   */
    int32_t prompt;      /* prompt tokens, >= 1                              */
    int32_t max_new;     /* max_new_tokens (what maximum reservation holds)  */
    int32_t gen;         /* tokens it generates, 0 <= gen <= max_new         */
    int32_t completion;  /* step it leaves and releases its cache, > arrival */
} pk_sim_request;

enum {
    PK_POLICY_MAX_RESERVATION = 0,
    PK_POLICY_EXACT_CONTIGUOUS = 1,
    PK_POLICY_PAGED = 2
};
enum { PK_SIM_DROP = 0, PK_SIM_STALL = 1 };

typedef struct {
    int64_t admitted, rejected;
    int64_t rejected_despite_free;         /* free capacity >= what was asked */
    int64_t growth_failures;
    int64_t growth_failures_despite_free;  /* at least one slot was free      */
    int64_t dropped, completed;
    int64_t peak_live, peak_reserved, peak_waste; /* after every allocation    */
    int64_t capacity;                      /* slots the policy can use        */
    int32_t num_steps;                     /* samples the run produces        */
} pk_sim_summary;

/* End-of-step state: live tokens, reserved slots, waste = reserved - live,
 * free = capacity - reserved, and the largest run of contiguous free slots
 * (paged: of free blocks with consecutive ids, times B). */
typedef struct {
    int32_t step, active;
    int64_t live, reserved, waste, free_slots, largest_free;
} pk_sim_sample;

/* Steps a trace spans: 1 + the largest arrival or completion step (-1 on a
 * bad argument). */
int32_t pk_sim_num_steps(const pk_sim_request *trace, int32_t n);

/* Runs the trace; fills *summary and samples[0 .. min(max_samples,
 * num_steps) - 1]. PK_ERR_INVALID_ARG for a malformed trace, policy, rule or
 * a paged capacity below one block. */
pk_status pk_sim_run(const pk_sim_request *trace, int32_t n, int32_t capacity, int32_t policy,
                     int32_t block_size, int32_t rule, pk_sim_summary *summary,
                     pk_sim_sample *samples, int32_t max_samples);

/* Shared-prefix groups for cascade attention. Sequences of seq_ids[0..n-1]
 * whose tables begin with the same physical block (forks of one parent) are
 * grouped in batch order, in chunks of at most max_group_size; a chunk of two
 * or more becomes a group when its members' tables agree on at least
 * min_prefix_blocks leading blocks that every member has filled. Outputs (host
 * arrays, capacity n each, n + 1 for group_offsets):
 *   group_offsets[g] .. group_offsets[g+1]-1 index group_members, which holds
 *     batch positions (indices into seq_ids); the first member's table
 *     supplies the group's prefix blocks;
 *   group_prefix_len[g]: shared tokens (a multiple of B);
 *   seq_prefix_len[i]: shared tokens of batch position i (0 outside groups);
 *   *num_groups_out: number of groups.
 * ("paged attention deep", "Copy-on-write for shared prefixes": forked
 * sequences name the same prefix blocks.) */
pk_status pk_bm_prefix_groups(const pk_bm *bm, const int64_t *seq_ids, int32_t n,
                              int32_t max_group_size, int32_t min_prefix_blocks,
                              int32_t *group_offsets, int32_t *group_members,
                              int32_t *group_prefix_len, int32_t *seq_prefix_len,
                              int32_t *num_groups_out);

/* live_tokens: sum of sequence lengths; reserved_slots: B * (blocks in use);
 * tail_waste: sum over sequences of B*ceil(len/B) - len; shared_blocks:
 * blocks with refcount > 1; cow_copies: copy-on-write copies so far. Any
 * output pointer may be NULL. */
pk_status pk_bm_stats(const pk_bm *bm, int64_t *live_tokens, int64_t *reserved_slots,
                      int64_t *tail_waste, int32_t *shared_blocks, int64_t *cow_copies);

/* ------------------------------------------------------------------------ */
/* One decode step from host buffers                                        */
/* ------------------------------------------------------------------------ */
/* Buffers of pk_decode_step. Host pointers should be pinned (page-locked) so
 * the copies are asynchronous; device pointers are caller-owned, 16-byte
 * aligned. With q_dev, k_dev, v_dev and out_dev all NULL (zero-copy mode) the
 * kernels read q and the new K/V from, and write the output to, the host
 * buffers directly -- the same bytes cross the host link, inside the kernels
 * rather than as separate copies. Where the GPU reads host memory through the
 * host's page tables (a Grace-attached GB300) any host memory serves, at its
 * own address, and nothing is looked up; elsewhere the host buffers (and
 * meta_host) must be pinned, device-mapped memory (else PK_ERR_INVALID_ARG),
 * and the device mapping of each address is looked up once and kept in the
 * library-managed state: a host buffer freed and pinned again at the same
 * address then needs pk_decode_step_release first. */
typedef struct {
    const void *q_host;  /* [S, Hq, d] queries of the step                     */
    const void *k_host;  /* [S, Hk, d] the step's new keys                      */
    const void *v_host;  /* [S, Hk, d] the step's new values                    */
    void *q_dev;         /* device copies of the three above (NULL: zero-copy) */
    void *k_dev;
    void *v_dev;
    void *meta_host;     /* pinned staging of pk_decode_step_meta_bytes bytes  */
    void *meta_dev;      /* device staging of the same size                    */
    size_t meta_bytes;
    void *out_dev;       /* [S, Hq, d] attention output on the device (or NULL) */
    void *out_host;      /* [S, Hq, d] its host copy                            */
    void *workspace;     /* split-K workspace (see pk_paged_attention_decode)   */
    size_t workspace_bytes;
    /* In: nonzero when meta_dev already holds these sequences' block tables
     * and context lengths as left by the previous successful pk_decode_step
     * (or pk_decode_step_launch) with the same seq_ids, max_blocks_per_seq
     * and buffers, and the block manager has not touched them since (no
     * fork, free, swap or append outside the decode step; none at all
     * between a step's prepare and its launch). Out: 1 after a successful
     * launch, 0 after a prepare or a failed call. Set it to 0 whenever that
     * does not hold. */
    int32_t tables_resident;
    /* Library-managed (zero-initialise): the work plan of the resident steps,
     * its partition size and item count (see pk_attention_plan). */
    int32_t plan_partition;
    int32_t plan_items;
    /* Library-managed (NULL-initialise): the prepared step and the captured
     * graphs of the steady resident steps; free it with
     * pk_decode_step_release. */
    void *state;
} pk_step_buffers;

/* Bytes of pk_step_buffers.meta_host / meta_dev (meta_bytes) for S sequences
 * and tables of max_blocks_per_seq entries (0 for non-positive arguments).
 * meta_host holds two staging halves that consecutive steps alternate
 * between, so one step's metadata can be prepared while the previous step's
 * is still being read; meta_dev uses the first half of this size. */
size_t pk_decode_step_meta_bytes(int32_t num_seqs, int32_t max_blocks_per_seq);

/* One decode step of the whole path for the distinct sequences
 * seq_ids[0..S-1] (host):
 *   1. copies host -> device of q, k, v from the caller's host buffers;
 *   2. host: append one token to each sequence (pk_bm_append_batch); unless
 *      buffers->tables_resident, export the padded tables and lengths and
 *      plan the attention's work list (pk_attention_plan with partition_size)
 *      -- into meta_host; a resident step keeps the plan's partition and
 *      rebuilds the list only when a sequence starts a new partition;
 *   3. copy host -> device of the metadata in one transfer (resident mode:
 *      only the slots and copy-on-write pairs, and the work list when it
 *      changed; in zero-copy mode the resident kernel reads the slots from
 *      meta_host itself, so a steady step copies no metadata);
 *   4. device: pk_copy_blocks for the step's pairs, then a full step runs the
 *      slot scatter (pk_reshape_and_cache) and the attention over the work
 *      list (pk_paged_attention_decode_items, automatic kernel); a resident
 *      step runs both and the device-side table and length bookkeeping as
 *      one pk_paged_attention_decode_advance launch, the lengths alternating
 *      between two device buffers;
 *   5. copy device -> host of the output into out_host.
 * All work is enqueued on `stream`; out_host holds the result once the stream
 * is synchronised. The workspace must cover the plan's partition: with
 * partition_size = -1, pk_paged_attention_workspace_size for 512 tokens and
 * the longest context the steps reach. The pages
 * have no counterpart for this packaging; each step it performs is theirs
 * (see the entry points above). On an error after step 2 the block manager
 * keeps the appended tokens and tables_resident is 0.
 *
 * On a stream the caller created (not the legacy or per-thread default
 * stream, and not being captured), a steady resident step -- no
 * copy-on-write pair, the same work list -- runs as one CUDA graph, captured
 * on the first such step of each staging half: the input copies, the slot
 * copy, the scatter, the attention and the output copy. Other host buffers
 * than a graph was captured with are patched into it: the q/k/v copies'
 * sources in copying mode (a new out_host rebuilds the graph instead), in
 * zero-copy mode the host-buffer arguments of the kernels that read or write
 * them (the attention, its merge, and the CUDA-core path's separate
 * scatter). The graphs are rebuilt when the work list changes or after a full
 * step. The per-step host work is then the block-manager append and one graph
 * launch. */
pk_status pk_decode_step(pk_bm *bm, const int64_t *seq_ids, int32_t num_seqs, int32_t num_q_heads,
                         float scale, int32_t max_blocks_per_seq, int32_t partition_size,
                         void *k_cache, void *v_cache, const pk_cache_desc *desc,
                         pk_step_buffers *buffers, void *stream);

/* pk_decode_step in two halves, so that the host half of a step can overlap
 * the device half of the step before -- as a serving loop does when it
 * schedules the next step while the current one runs on the GPU.
 *
 * pk_decode_step_prepare is steps 2 of pk_decode_step (the block-manager
 * append, and the tables, lengths and work plan unless tables_resident) into
 * the staging half of meta_host that the step before the previous one used;
 * it first waits until that step has finished reading it (an event recorded
 * after its work), so at most one step is ever outstanding on a half. It
 * enqueues no device work and reads no q/k/v. It sets tables_resident to 0
 * after the append (the device tables do not yet hold the new token).
 * PK_ERR_INVALID_ARG if a prepared step has not been launched yet, or if
 * tables_resident is set for another shape than the last prepared step's.
 *
 * pk_decode_step_launch is steps 1 and 3-5 for the prepared step (the same
 * num_seqs and max_blocks_per_seq): the input copies, the metadata copy from
 * the prepared half, the kernels and the output copy, or the captured graph of
 * that half; it sets tables_resident to 1 once the work is enqueued. The
 * prepared step is consumed even when the launch fails (tables_resident then
 * stays 0, and the next step is a full one). Inputs are read when the step
 * runs, so q/k/v must not change until the stream has passed the step.
 *
 * pk_decode_step is prepare followed by launch. A pipelined loop is: prepare
 * step 0; then for every step t: fill its inputs, launch it, prepare step
 * t+1 (host work while step t runs), synchronise, read the output. */
pk_status pk_decode_step_prepare(pk_bm *bm, const int64_t *seq_ids, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t max_blocks_per_seq,
                                 int32_t partition_size, const pk_cache_desc *desc,
                                 pk_step_buffers *buffers);
pk_status pk_decode_step_launch(int32_t num_seqs, int32_t num_q_heads, float scale,
                                int32_t max_blocks_per_seq, void *k_cache, void *v_cache,
                                const pk_cache_desc *desc, pk_step_buffers *buffers,
                                void *stream);

/* Captured graphs currently held in buffers->state (0, 1 or 2: one per
 * staging half). Host only. */
int32_t pk_decode_step_graph_count(const pk_step_buffers *buffers);

/* Frees the library-managed state in buffers->state (the captured graphs,
 * events and any prepared step) and sets it to NULL; call before freeing the
 * buffers or destroying the stream, after the last step has finished. */
void pk_decode_step_release(pk_step_buffers *buffers);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
