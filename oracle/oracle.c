/*
 * oracle.c -- the CPU oracle for paged-KV-cache decode.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The product path (libpagedkv) never does,
 * and the two share no code, header, table or helper.
 *
 * Plain, slow, single-threaded C. Floating point is double precision. Every
 * function restates one passage of the pages it follows:
 *
 *   [P1] "Paged KV Cache Allocation and the Block Table" (mercemay.com),
 *        sections "Blocks, tables, and the indirection" (the append_token
 *        routine), "Sharing blocks between sequences" (refcounts, CoW,
 *        reclamation).
 *   [P2] "The KV Cache Is an Allocator Problem" (synapticradio.com), the
 *        physical-address equation  addr = table[floor(t/B)] * B + (t mod B)
 *        and the reserved-slots equation  B * ceil(L/B).
 *   [P3] "PagedAttention" (llminference.xinbetween.com, S06), the BlockManager
 *        listing (free list, tables, append, free_request), "Copy-on-write, for
 *        free", "Reference counts must be exact", and the paged_attention
 *        listing (gather K through the table, softmax, weighted sum of V).
 *   [P4] "paged attention deep" (aicassindra.com), "Anatomy of a KV block"
 *        (a block holds K [B, n_kv_heads, d_head] and an equally shaped V),
 *        "The block table" (logical_block = t // B, offset = t % B) and
 *        "Copy-on-write for shared prefixes" (copy the single shared block,
 *        decrement the original's count).
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - The free list is a stack. Its first pop returns alloc_order[0]; a
 *     retired sequence's blocks are pushed in table order. [P3 listing pops
 *     from the end of a Python list and extends it on free; the P3 widget hands
 *     out ascending ids from a fresh pool.]
 *   - Appending n tokens is all-or-nothing: if the pool cannot supply every
 *     block the n tokens need, nothing changes and OR_ERR_OUT_OF_BLOCKS is
 *     returned. [P3 "return False -> preempt".]
 *   - Copy-on-write copies the whole block (all B slots, all heads, K and V).
 *     It fires only when the first token of an append lands in a partly
 *     filled tail block whose refcount is above one. [P4 "copies that single
 *     block".]
 *   - Query head h reads KV head h / (Hq / Hk).
 *   - Prefix caching ("PagedAttention" S06, "What's next": block contents are
 *     hashed so that requests with a common prefix share physical blocks).
 *     Only full blocks are cached. A block's key is every token of the
 *     prompt up to and including the block, so a hit at block j means the
 *     whole prefix matches. A cached block whose last reference goes away
 *     stays cached (unreferenced, evictable) rather than returning to the
 *     free list; an allocation takes the free list first and, only when it
 *     is empty, evicts the unreferenced cached block released longest ago
 *     (among blocks released by one call, the deepest first).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    OR_OK = 0,
    OR_ERR_ARG = 1,
    OR_ERR_OUT_OF_BLOCKS = 2,
    OR_ERR_UNKNOWN_SEQ = 3,
    OR_ERR_SEQ_EXISTS = 4,
    OR_ERR_NOMEM = 5
};

enum { OR_F32 = 0, OR_BF16 = 1 };

/* ------------------------------------------------------------------------- */
/* Block manager                                                             */
/* ------------------------------------------------------------------------- */

typedef struct {
    long long id;
    long long len;      /* tokens written so far                     */
    int *table;         /* logical block index -> physical block id  */
    int nblk;           /* entries used in table                     */
    int cap;            /* entries allocated in table                */
    int live;
    int swapped;        /* 1: table holds host swap-space block ids  */
} or_seq;

typedef struct {
    int num_blocks;
    int block_size;
    int *free_stack;    /* free_stack[top - 1] is handed out next */
    int top;
    int *refcount;      /* number of tables naming each block     */
    or_seq *seqs;
    int nseq;
    int seq_cap;
    long long cow_copies;
    int num_host_blocks;  /* swap space in host memory (0: none)      */
    int *host_stack;      /* host_stack[host_top - 1] is handed next  */
    int host_top;
    /* prefix cache, per block */
    int *cached;          /* 1: the block holds a committed prefix          */
    int **key;            /* key[b]: tokens 0 .. key_len[b]-1 of that prefix */
    int *key_len;
    long long *released;  /* clock of the call that left it unreferenced    */
    long long clock;
    long long cache_hits; /* blocks served from the cache                    */
    long long evictions;
} or_bm;

static or_seq *find_seq(or_bm *bm, long long id) {
    for (int i = 0; i < bm->nseq; i++)
        if (bm->seqs[i].live && bm->seqs[i].id == id) return &bm->seqs[i];
    return NULL;
}

static int table_push(or_seq *s, int block) {
    if (s->nblk == s->cap) {
        int ncap = s->cap ? 2 * s->cap : 8;
        int *t = (int *)realloc(s->table, sizeof(int) * (size_t)ncap);
        if (!t) return OR_ERR_NOMEM;
        s->table = t;
        s->cap = ncap;
    }
    s->table[s->nblk++] = block;
    return OR_OK;
}

/* Blocks an allocation can take: the free list plus every cached block that
 * no table names. */
static int available(or_bm *bm) {
    int n = bm->top;
    for (int b = 0; b < bm->num_blocks; b++)
        if (bm->cached[b] && bm->refcount[b] == 0) n++;
    return n;
}

static void uncache(or_bm *bm, int b) {
    free(bm->key[b]);
    bm->key[b] = NULL;
    bm->key_len[b] = 0;
    bm->cached[b] = 0;
}

/* One block for a table: the top of the free list, else the unreferenced
 * cached block released longest ago (deepest first on a tie), which leaves
 * the cache. The caller has checked available(bm) > 0. */
static int take_block(or_bm *bm) {
    if (bm->top > 0) return bm->free_stack[--bm->top];
    int best = -1;
    for (int b = 0; b < bm->num_blocks; b++) {
        if (!bm->cached[b] || bm->refcount[b] != 0) continue;
        if (best < 0 || bm->released[b] < bm->released[best] ||
            (bm->released[b] == bm->released[best] && bm->key_len[b] > bm->key_len[best]))
            best = b;
    }
    uncache(bm, best);
    bm->evictions += 1;
    return best;
}

/* A table stops naming block b. At zero references an uncached block goes
 * back on the free list; a cached one stays, stamped with this call's clock. */
static void release(or_bm *bm, int b) {
    bm->refcount[b] -= 1;
    if (bm->refcount[b] == 0) {
        if (bm->cached[b])
            bm->released[b] = bm->clock;
        else
            bm->free_stack[bm->top++] = b;
    }
}

/* The cached block whose key is exactly tokens[0 .. len-1], or -1. */
static int find_cached(or_bm *bm, const int *tokens, int len) {
    for (int b = 0; b < bm->num_blocks; b++)
        if (bm->cached[b] && bm->key_len[b] == len &&
            memcmp(bm->key[b], tokens, sizeof(int) * (size_t)len) == 0)
            return b;
    return -1;
}

static or_seq *new_seq(or_bm *bm, long long id) {
    if (bm->nseq == bm->seq_cap) {
        int ncap = bm->seq_cap ? 2 * bm->seq_cap : 16;
        or_seq *p = (or_seq *)realloc(bm->seqs, sizeof(or_seq) * (size_t)ncap);
        if (!p) return NULL;
        bm->seqs = p;
        bm->seq_cap = ncap;
    }
    or_seq *s = &bm->seqs[bm->nseq++];
    memset(s, 0, sizeof(*s));
    s->id = id;
    s->live = 1;
    return s;
}

/* A pool of num_blocks blocks of block_size slots; alloc_order (a permutation
 * of 0..num_blocks-1, or NULL for 0,1,2,...) is the order of the first pops. */
or_bm *or_bm_new(int num_blocks, int block_size, const int *alloc_order) {
    if (num_blocks <= 0 || block_size <= 0) return NULL;
    or_bm *bm = (or_bm *)calloc(1, sizeof(or_bm));
    if (!bm) return NULL;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->free_stack = (int *)malloc(sizeof(int) * (size_t)num_blocks);
    bm->refcount = (int *)calloc((size_t)num_blocks, sizeof(int));
    bm->cached = (int *)calloc((size_t)num_blocks, sizeof(int));
    bm->key = (int **)calloc((size_t)num_blocks, sizeof(int *));
    bm->key_len = (int *)calloc((size_t)num_blocks, sizeof(int));
    bm->released = (long long *)calloc((size_t)num_blocks, sizeof(long long));
    if (!bm->free_stack || !bm->refcount || !bm->cached || !bm->key || !bm->key_len ||
        !bm->released) {
        free(bm->free_stack);
        free(bm->refcount);
        free(bm->cached);
        free(bm->key);
        free(bm->key_len);
        free(bm->released);
        free(bm);
        return NULL;
    }
    /* Push in reverse so that the first pop returns alloc_order[0]. */
    for (int i = 0; i < num_blocks; i++) {
        int b = alloc_order ? alloc_order[num_blocks - 1 - i] : num_blocks - 1 - i;
        bm->free_stack[i] = b;
    }
    bm->top = num_blocks;
    return bm;
}

void or_bm_delete(or_bm *bm) {
    if (!bm) return;
    for (int i = 0; i < bm->nseq; i++) free(bm->seqs[i].table);
    free(bm->seqs);
    for (int b = 0; b < bm->num_blocks; b++) free(bm->key[b]);
    free(bm->free_stack);
    free(bm->refcount);
    free(bm->cached);
    free(bm->key);
    free(bm->key_len);
    free(bm->released);
    free(bm->host_stack);
    free(bm);
}

int or_bm_add_seq(or_bm *bm, long long id) {
    if (find_seq(bm, id)) return OR_ERR_SEQ_EXISTS;
    return new_seq(bm, id) ? OR_OK : OR_ERR_NOMEM;
}

/* Append n tokens to sequence id. slots_out[i] receives the physical slot of
 * the i-th token. If the first token lands in a shared tail block, its
 * (source, destination) copy-on-write pair goes to cow_out[0..1] and *n_cow
 * becomes 1; otherwise *n_cow is 0. */
int or_bm_append(or_bm *bm, long long id, int n, long long *slots_out,
                 long long *cow_out, int *n_cow) {
    const int B = bm->block_size;
    or_seq *s = find_seq(bm, id);
    if (n_cow) *n_cow = 0;
    if (!s) return OR_ERR_UNKNOWN_SEQ;
    if (n < 0 || s->swapped) return OR_ERR_ARG;

    /* Count the blocks the n tokens need before touching anything. */
    int need = 0;
    long long L = s->len;
    for (int i = 0; i < n; i++, L++) {
        if (L % B == 0)
            need++;                                  /* a fresh block   */
        else if (i == 0 && bm->refcount[s->table[s->nblk - 1]] > 1)
            need++;                                  /* a CoW copy      */
    }
    if (need > available(bm)) return OR_ERR_OUT_OF_BLOCKS;

    for (int i = 0; i < n; i++) {
        long long offset = s->len % B;
        if (offset == 0) {
            /* [P1] the sequence has outgrown its table: one more block. */
            int blk = take_block(bm);
            bm->refcount[blk] = 1;
            if (table_push(s, blk) != OR_OK) return OR_ERR_NOMEM;
        } else {
            int tail = s->table[s->nblk - 1];
            if (bm->refcount[tail] > 1) {
                /* [P1]/[P4] writing into a shared block: take a private copy. */
                int blk = take_block(bm);
                bm->refcount[blk] = 1;
                bm->refcount[tail] -= 1;
                s->table[s->nblk - 1] = blk;
                bm->cow_copies += 1;
                if (cow_out) {
                    cow_out[0] = tail;
                    cow_out[1] = blk;
                }
                if (n_cow) *n_cow = 1;
            }
        }
        /* [P2] physical address = table[floor(t / B)] * B + (t mod B). */
        long long t = s->len;
        long long slot = (long long)s->table[t / B] * B + t % B;
        if (slots_out) slots_out[i] = slot;
        s->len += 1;
    }
    return OR_OK;
}

/* [P1] a forked sequence names the same blocks as its parent; every block's
 * reference count goes up by one. */
int or_bm_fork(or_bm *bm, long long parent, long long child) {
    if (find_seq(bm, child)) return OR_ERR_SEQ_EXISTS;
    if (!find_seq(bm, parent)) return OR_ERR_UNKNOWN_SEQ;
    if (find_seq(bm, parent)->swapped) return OR_ERR_ARG;
    or_seq *c = new_seq(bm, child);
    if (!c) return OR_ERR_NOMEM;
    or_seq *p = find_seq(bm, parent); /* re-find: new_seq may move the array */
    for (int j = 0; j < p->nblk; j++) {
        if (table_push(c, p->table[j]) != OR_OK) return OR_ERR_NOMEM;
        bm->refcount[p->table[j]] += 1;
    }
    c->len = p->len;
    return OR_OK;
}

/* [P1] retiring a sequence decrements every block it names and returns only
 * the blocks whose count reaches zero. */
int or_bm_free_seq(or_bm *bm, long long id) {
    or_seq *s = find_seq(bm, id);
    if (!s) return OR_ERR_UNKNOWN_SEQ;
    bm->clock += 1;
    for (int j = 0; j < s->nblk; j++) {
        int b = s->table[j];
        if (s->swapped) {            /* host blocks go back to the swap space */
            bm->host_stack[bm->host_top++] = b;
            continue;
        }
        release(bm, b);
    }
    free(s->table);
    s->table = NULL;
    s->nblk = s->cap = 0;
    s->live = 0;
    return OR_OK;
}

/* Swap space: num_host_blocks blocks in host memory, handed out first to
 * last as host_order[0], host_order[1], ... (NULL: 0, 1, 2, ...). */
int or_bm_set_swap_space(or_bm *bm, int num_host_blocks, const int *host_order) {
    if (num_host_blocks < 0 || bm->num_host_blocks) return OR_ERR_ARG;
    bm->host_stack = (int *)malloc(sizeof(int) * (size_t)(num_host_blocks > 0 ? num_host_blocks : 1));
    if (!bm->host_stack) return OR_ERR_NOMEM;
    for (int i = 0; i < num_host_blocks; i++)
        bm->host_stack[i] = host_order ? host_order[num_host_blocks - 1 - i] : num_host_blocks - 1 - i;
    bm->num_host_blocks = num_host_blocks;
    bm->host_top = num_host_blocks;
    return OR_OK;
}

/* Preemption by swapping ("Paged KV Cache Allocation and the Block Table",
 * "What the design costs": the server may swap a sequence's blocks to host
 * memory). Every block of the table, in table order, gets a host block:
 * pairs_out[2j] = device block, pairs_out[2j+1] = host block. The device
 * block loses the sequence's reference and returns to the free list when no
 * table names it any more. All or nothing: OR_ERR_OUT_OF_BLOCKS if the swap
 * space is short. The caller copies the pairs device -> host before the
 * freed blocks are written again. */
int or_bm_swap_out(or_bm *bm, long long id, long long *pairs_out, int *n_out) {
    or_seq *s = find_seq(bm, id);
    if (n_out) *n_out = 0;
    if (!s) return OR_ERR_UNKNOWN_SEQ;
    if (s->swapped) return OR_ERR_ARG;
    if (s->nblk > bm->host_top) return OR_ERR_OUT_OF_BLOCKS;
    bm->clock += 1;
    for (int j = 0; j < s->nblk; j++) {
        int d = s->table[j];
        int h = bm->host_stack[--bm->host_top];
        pairs_out[2 * j] = d;
        pairs_out[2 * j + 1] = h;
        release(bm, d);
        s->table[j] = h;
    }
    s->swapped = 1;
    if (n_out) *n_out = s->nblk;
    return OR_OK;
}

/* Brings a swapped sequence back: every host block, in table order, gets a
 * fresh private device block: pairs_out[2j] = host block, pairs_out[2j+1] =
 * device block; the host block returns to the swap space. All or nothing:
 * OR_ERR_OUT_OF_BLOCKS if the device pool is short. */
int or_bm_swap_in(or_bm *bm, long long id, long long *pairs_out, int *n_out) {
    or_seq *s = find_seq(bm, id);
    if (n_out) *n_out = 0;
    if (!s) return OR_ERR_UNKNOWN_SEQ;
    if (!s->swapped) return OR_ERR_ARG;
    if (s->nblk > available(bm)) return OR_ERR_OUT_OF_BLOCKS;
    for (int j = 0; j < s->nblk; j++) {
        int h = s->table[j];
        int d = take_block(bm);
        bm->refcount[d] = 1;
        pairs_out[2 * j] = h;
        pairs_out[2 * j + 1] = d;
        bm->host_stack[bm->host_top++] = h;
        s->table[j] = d;
    }
    s->swapped = 0;
    if (n_out) *n_out = s->nblk;
    return OR_OK;
}

int or_bm_is_swapped(or_bm *bm, long long id) {
    or_seq *s = find_seq(bm, id);
    return s ? s->swapped : -1;
}

int or_bm_host_free(or_bm *bm) { return bm->host_top; }

/* Prefix caching: a new sequence whose prompt is tokens[0 .. n-1] starts
 * with every leading full block already in the cache. Block j is a hit when
 * a cached block's key is exactly tokens[0 .. (j+1)B - 1]; the first miss
 * ends the walk. Each hit is named by the new table (one more reference).
 * The sequence's length becomes hits * B (*n_cached); the caller appends and
 * writes the remaining n - *n_cached tokens as usual. */
int or_bm_add_seq_cached(or_bm *bm, long long id, const int *tokens, int n, int *n_cached) {
    const int B = bm->block_size;
    if (n_cached) *n_cached = 0;
    if (n < 0 || (n > 0 && !tokens)) return OR_ERR_ARG;
    if (find_seq(bm, id)) return OR_ERR_SEQ_EXISTS;
    or_seq *s = new_seq(bm, id);
    if (!s) return OR_ERR_NOMEM;
    for (int j = 0; (long long)(j + 1) * B <= n; j++) {
        int b = find_cached(bm, tokens, (j + 1) * B);
        if (b < 0) break;
        if (table_push(s, b) != OR_OK) return OR_ERR_NOMEM;
        bm->refcount[b] += 1;
        bm->cache_hits += 1;
    }
    s->len = (long long)s->nblk * B;
    if (n_cached) *n_cached = (int)s->len;
    return OR_OK;
}

/* Registers the full blocks among the first n tokens of sequence id (its
 * token ids are tokens[0 .. n-1], n <= its length, their K/V written): block
 * j gets the key tokens[0 .. (j+1)B - 1] unless it is cached already or
 * another block already holds that key (the first one stays). */
int or_bm_commit(or_bm *bm, long long id, const int *tokens, int n) {
    const int B = bm->block_size;
    or_seq *s = find_seq(bm, id);
    if (!s) return OR_ERR_UNKNOWN_SEQ;
    if (s->swapped || n < 0 || n > s->len || (n > 0 && !tokens)) return OR_ERR_ARG;
    for (int j = 0; (long long)(j + 1) * B <= n; j++) {
        int b = s->table[j];
        int len = (j + 1) * B;
        if (bm->cached[b] || find_cached(bm, tokens, len) >= 0) continue;
        bm->key[b] = (int *)malloc(sizeof(int) * (size_t)len);
        if (!bm->key[b]) return OR_ERR_NOMEM;
        memcpy(bm->key[b], tokens, sizeof(int) * (size_t)len);
        bm->key_len[b] = len;
        bm->cached[b] = 1;
    }
    return OR_OK;
}

/* Cached blocks, of which unreferenced; blocks served from the cache;
 * cached blocks evicted by allocations. */
void or_bm_cache_stats(or_bm *bm, long long *cached, long long *unreferenced,
                       long long *hits, long long *evictions) {
    long long c = 0, u = 0;
    for (int b = 0; b < bm->num_blocks; b++) {
        c += bm->cached[b];
        u += bm->cached[b] && bm->refcount[b] == 0;
    }
    *cached = c;
    *unreferenced = u;
    *hits = bm->cache_hits;
    *evictions = bm->evictions;
}

int or_bm_is_cached(or_bm *bm, int block) {
    return (block >= 0 && block < bm->num_blocks) ? bm->cached[block] : -1;
}

/* Whole-block copies between two pools of the same block shape: block
 * pairs[2p] of `from` goes to block pairs[2p+1] of `to` (K and V). */
int or_swap_copy(void *to_k, void *to_v, const void *from_k, const void *from_v,
                 const long long *pairs, int num_pairs, int to_blocks, int from_blocks,
                 int B, int Hk, int d, int esz) {
    const size_t blk_bytes = (size_t)B * (size_t)Hk * (size_t)d * (size_t)esz;
    for (int p = 0; p < num_pairs; p++) {
        long long src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= from_blocks || dst < 0 || dst >= to_blocks) return OR_ERR_ARG;
        memcpy((char *)to_k + (size_t)dst * blk_bytes, (const char *)from_k + (size_t)src * blk_bytes, blk_bytes);
        memcpy((char *)to_v + (size_t)dst * blk_bytes, (const char *)from_v + (size_t)src * blk_bytes, blk_bytes);
    }
    return OR_OK;
}

/* Copies sequence id's table into out[0..cap-1]; returns its length, or a
 * negative error code. */
int or_bm_table(or_bm *bm, long long id, int *out, int cap) {
    or_seq *s = find_seq(bm, id);
    if (!s) return -OR_ERR_UNKNOWN_SEQ;
    for (int j = 0; j < s->nblk && j < cap; j++) out[j] = s->table[j];
    return s->nblk;
}

long long or_bm_seq_len(or_bm *bm, long long id) {
    or_seq *s = find_seq(bm, id);
    return s ? s->len : -1;
}

int or_bm_refcount(or_bm *bm, int block) {
    if (block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[block];
}

int or_bm_num_free(or_bm *bm) { return available(bm); }

long long or_bm_cow_copies(or_bm *bm) { return bm->cow_copies; }

/* Writes the free list, next-handed-out first, into out[0..top-1]. */
int or_bm_free_list(or_bm *bm, int *out, int cap) {
    int n = 0;
    for (int i = bm->top - 1; i >= 0 && n < cap; i--) out[n++] = bm->free_stack[i];
    return bm->top;
}

/* ------------------------------------------------------------------------- */
/* Cache writes                                                              */
/* ------------------------------------------------------------------------- */

/* [P1 append_token] / [P4 block anatomy]: token i's K and V (each Hk * d
 * elements of esz bytes) go to slot slots[i] of the pool, which is laid out
 * [num_blocks, B, Hk, d]. A negative slot means "skip this token". */
int or_reshape_and_cache(void *k_cache, void *v_cache, const void *k, const void *v,
                         const long long *slots, int num_tokens, int num_blocks,
                         int B, int Hk, int d, int esz) {
    const size_t row = (size_t)Hk * (size_t)d * (size_t)esz;
    for (int i = 0; i < num_tokens; i++) {
        long long s = slots[i];
        if (s < 0) continue;
        if (s >= (long long)num_blocks * B) return OR_ERR_ARG;
        long long blk = s / B, off = s % B;
        size_t dst = ((size_t)blk * (size_t)B + (size_t)off) * row;
        memcpy((char *)k_cache + dst, (const char *)k + (size_t)i * row, row);
        memcpy((char *)v_cache + dst, (const char *)v + (size_t)i * row, row);
    }
    return OR_OK;
}

/* [P4 copy-on-write]: copy the whole block src to block dst, K and V. */
int or_copy_blocks(void *k_cache, void *v_cache, const long long *pairs, int num_pairs,
                   int num_blocks, int B, int Hk, int d, int esz) {
    const size_t blk_bytes = (size_t)B * (size_t)Hk * (size_t)d * (size_t)esz;
    for (int p = 0; p < num_pairs; p++) {
        long long src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return OR_ERR_ARG;
        memcpy((char *)k_cache + (size_t)dst * blk_bytes, (char *)k_cache + (size_t)src * blk_bytes, blk_bytes);
        memcpy((char *)v_cache + (size_t)dst * blk_bytes, (char *)v_cache + (size_t)src * blk_bytes, blk_bytes);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Paged attention                                                           */
/* ------------------------------------------------------------------------- */

/* One stored element as a double. bf16 is the upper half of an fp32 word. */
static double element(const void *base, size_t idx, int dtype) {
    if (dtype == OR_F32) return (double)((const float *)base)[idx];
    uint32_t w = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Decode attention of one query head through the block table [P3 listing,
 * P4 "The block table"]:
 *   for t < ctx:  phys = table[t / B], slot offset t % B,
 *                 x_t = scale * <q, K[phys, t % B, kvh, :]>
 *   w = softmax(x)  (largest score subtracted before exp)
 *   out = sum_t w_t * V[phys, t % B, kvh, :]
 * q is [S, Hq, d]; the pools are [num_blocks, B, Hk, d]; tables is
 * [S, max_blocks] int32; out is [S, Hq, d] double. If sel is not NULL, only
 * the nsel (seq, head) pairs sel[2i], sel[2i+1] are computed. */
int or_paged_attention(double *out, const void *q, const void *k_cache, const void *v_cache,
                       int dtype, const int *tables, int max_blocks, const long long *ctx_lens,
                       int S, int Hq, int Hk, int d, int B, int num_blocks, double scale,
                       const int *sel, int nsel) {
    if (Hk <= 0 || Hq % Hk != 0 || d <= 0 || B <= 0) return OR_ERR_ARG;
    const int G = Hq / Hk;
    const int npairs = sel ? nsel : S * Hq;
    for (int i = 0; i < npairs; i++) {
        int s = sel ? sel[2 * i] : i / Hq;
        int h = sel ? sel[2 * i + 1] : i % Hq;
        if (s < 0 || s >= S || h < 0 || h >= Hq) return OR_ERR_ARG;
        const int kvh = h / G;
        const long long n = ctx_lens[s];
        if (n <= 0 || (n + B - 1) / B > max_blocks) return OR_ERR_ARG;
        double *x = (double *)malloc(sizeof(double) * (size_t)n);
        if (!x) return OR_ERR_NOMEM;
        const size_t qbase = ((size_t)s * Hq + h) * (size_t)d;

        for (long long t = 0; t < n; t++) {
            int phys = tables[(size_t)s * max_blocks + (size_t)(t / B)];
            if (phys < 0 || phys >= num_blocks) { free(x); return OR_ERR_ARG; }
            size_t kbase = (((size_t)phys * B + (size_t)(t % B)) * Hk + kvh) * (size_t)d;
            double dot = 0.0;
            for (int e = 0; e < d; e++)
                dot += element(q, qbase + e, dtype) * element(k_cache, kbase + e, dtype);
            x[t] = scale * dot;
        }
        double m = x[0];
        for (long long t = 1; t < n; t++) if (x[t] > m) m = x[t];
        double z = 0.0;
        for (long long t = 0; t < n; t++) { x[t] = exp(x[t] - m); z += x[t]; }

        double *o = out + ((size_t)s * Hq + h) * (size_t)d;
        for (int e = 0; e < d; e++) o[e] = 0.0;
        for (long long t = 0; t < n; t++) {
            int phys = tables[(size_t)s * max_blocks + (size_t)(t / B)];
            size_t vbase = (((size_t)phys * B + (size_t)(t % B)) * Hk + kvh) * (size_t)d;
            double w = x[t] / z;
            for (int e = 0; e < d; e++) o[e] += w * element(v_cache, vbase + e, dtype);
        }
        free(x);
    }
    return OR_OK;
}
