/*
 * libpagedkv -- paged KV cache hot path for NVIDIA GB300 (sm_103a).
 *
 * A C ABI: plain pointers and sizes, no C++ or framework types.  Every function
 * returns an int status (PKV_OK == 0, negative on error) and never lets a C++
 * exception out.  Device work is enqueued asynchronously on the caller's stream
 * (`stream` is a cudaStream_t passed as void*; NULL = the legacy default
 * stream); nothing here synchronises.  The caller owns every buffer.  All
 * device pointers must belong to the current CUDA device.
 *
 * Metadata that can only be checked on the device (block ids read from a block
 * table, slots, context lengths) is checked by the kernels.  A bad entry is
 * skipped -- never trapped -- and the first error code is stored into the
 * caller's device word `dev_err` (int32, set to 0 by the caller before the
 * launch; the first error wins through atomicCAS).  Read it after the stream
 * has been synchronised.
 *
 * Terms (after "P06 BlockManager" and "ans20xx day 31"):
 *   block_size (bs)  tokens per physical KV block (attention: 8, 16, 32 or 64)
 *   block table      int32 [num_seqs, max_blocks_per_seq]: logical block i of a
 *                    sequence is physical block table[s][i]
 *   slot             physical row of a token: table[pos / bs] * bs + pos % bs
 *   KV cache         fp16 [num_blocks, block_size, num_kv_heads, head_dim],
 *                    one tensor for K and one for V per layer
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (host return values) ---------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)   /* null pointer, negative size, misalignment */
#define PKV_ERR_UNSUPPORTED (-2)   /* head_dim, block size or GQA ratio without a kernel */
#define PKV_ERR_CUDA (-3)          /* a CUDA runtime/driver call failed */
#define PKV_ERR_OUT_OF_BLOCKS (-4) /* BlockManager: no capacity; state unchanged */
#define PKV_ERR_BAD_INDEX (-5)     /* unknown sequence, position outside a table */

/* ---- device error codes (stored into *dev_err by the kernels) ------------ */
#define PKV_DEV_OK 0
#define PKV_DEV_BAD_BLOCK_ID 1     /* table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT_LEN 2  /* context_lens[s] < 0 or > max_blocks * bs */
#define PKV_DEV_BAD_SLOT 3         /* slot >= num_blocks * block_size */
#define PKV_DEV_WAIT_TIMEOUT 4     /* a bounded wait on a copy gave up; every
                                      output of that launch is then undefined */
#define PKV_DEV_BAD_POSITION 5     /* position outside its block table */
#define PKV_DEV_BAD_GROUP 6        /* a shared-prefix group whose members do not
                                      share the stated blocks, or too many rows */

/* Human-readable name of a status code (static string). */
const char* pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/* ---- paged decode attention --------------------------------------------- */
/*
 * Single-token decode attention over a paged KV cache.
 * Defined by "qaqbuyan: vLLM PagedAttention" (`paged_attention`: gather each
 * logical block through the block table, then softmax(q K^T * scale) V) and by
 * the slot rule of "P06 BlockManager".  For every sequence s and query head h,
 * with g = h / (num_q_heads / num_kv_heads) and L = context_lens[s]:
 *   out[s, h, :] = sum_t softmax_t(scale * <q[s, h, :], K_s[t, g, :]>) V_s[t, g, :]
 * over exactly the L tokens t = 0 .. L-1, where K_s[t] is row t % bs of
 * physical block block_tables[s][t / bs].  L == 0 gives a zero row.
 *
 *   out        fp16 [num_seqs, num_q_heads, head_dim], written
 *   q          fp16 [num_seqs, num_q_heads, head_dim]
 *   k_cache,
 *   v_cache    fp16 [num_blocks, block_size, num_kv_heads, head_dim]; 16-byte
 *              aligned
 *   block_tables int32 [num_seqs, max_blocks_per_seq] (device)
 *   context_lens int32 [num_seqs] (device); tokens per sequence, the token
 *              written this step included
 *   head_dim must be 128, block_size one of 8, 16, 32, 64 and
 *   num_q_heads / num_kv_heads one of 1, 2, 4, 8; otherwise PKV_ERR_UNSUPPORTED.
 *   q must be 4-byte aligned.
 *   workspace  device scratch of at least
 *              pkv_paged_attention_workspace_bytes(...) bytes (may be NULL when
 *              that is 0); holds per-split partial results of long contexts.
 *              Contents need no initialisation.  Two launches in flight at
 *              once must not share a workspace.
 *   dev_err    device int32 (see above); may be NULL to skip reporting.
 * fp32 accumulation throughout; the result is rounded to fp16 once.  Long
 * contexts are cut into splits of 2048, 1024 or 512 tokens, the longest that
 * still gives num_seqs x num_kv_heads x ceil(max_blocks_per_seq * block_size /
 * split) >= 1024 CTAs; their partials are merged by log-sum-exp.  A
 * sequence's output bits therefore depend on its own length and on those
 * launch sizes only: not on block ids, the order of the batch or the other
 * sequences' lengths.  (In a batch of at most 128 sequences whose last
 * split can be at least half a split long -- by the table width -- the last
 * split of each sequence is visited on the device longest, shortest, second
 * longest, ... by context_lens; that changes which CTA runs a unit, never the
 * arithmetic.)
 */
int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, int max_blocks_per_seq, float scale,
                               void* workspace, size_t workspace_bytes, int32_t* dev_err,
                               void* stream);

/* Workspace bytes pkv_paged_attention_decode (and _fused) need for these
 * sizes (host only): room for the partials of 512-token splits, the shortest
 * a launch uses, so it covers every split length; 0 when no sequence can span
 * more than one 512-token split. */
size_t pkv_paged_attention_workspace_bytes(int num_seqs, int num_q_heads,
                                           int max_blocks_per_seq, int block_size,
                                           int head_dim);

/* Split length in tokens (2048, 1024 or 512) that pkv_paged_attention_decode,
 * _fused and the grouped entry points use for these sizes (host only, no
 * device call): the longest for which num_seqs x num_kv_heads x
 * ceil(max_blocks_per_seq * block_size / split) reaches 1024.  A sequence's
 * output bits are a function of its own data and this split length.
 * PKV_ERR_INVALID_ARG for non-positive sizes or an unsupported block size. */
int pkv_paged_attention_split_tokens(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                                     int block_size);

/*
 * Fused cache write + attention: one launch does what pkv_reshape_and_cache of
 * the step's new tokens followed by pkv_paged_attention_decode does.  The new
 * token of sequence s is its last one, position L - 1 (L = context_lens[s]);
 * its slot is recomputed on the device from the block table
 * (table[(L-1) / bs] * bs + (L-1) % bs, "P06 BlockManager"), k_new[s] / v_new[s]
 * are stored there and used for that row of the attention.  Sequences with
 * L == 0 write nothing.
 *   k_new, v_new  fp16 [num_seqs, num_kv_heads, head_dim], 16-byte aligned
 *   k_cache, v_cache are written (the new rows only)
 * Other arguments, layouts and errors as pkv_paged_attention_decode.
 */
int pkv_paged_attention_decode_fused(void* out, const void* q, const void* k_new,
                                     const void* v_new, void* k_cache, void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks,
                                     int max_blocks_per_seq, float scale, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * Allocation-free variant of pkv_paged_attention_decode.  The pages have no
 * counterpart: it exists for callers that cannot allocate device memory, such
 * as a plugin whose host framework owns the whole device memory pool, or code
 * on a latency-critical path that must not take an allocation's implicit
 * device synchronisation.  Same arguments and result as
 * pkv_paged_attention_decode, minus the workspace: the split partials go to a
 * fixed 16 MiB scratch array in this library's device memory, which every GPU
 * that loads the library holds until the process exits.
 *   - Returns PKV_ERR_UNSUPPORTED when the sizes need more scratch than the
 *     array holds, i.e. when pkv_paged_attention_workspace_bytes(...) for the
 *     same sizes exceeds 16 MiB (16777216 bytes).
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call made outside stream capture looks the scratch array's
 *     device address up again in the current context (cudaGetSymbolAddress,
 *     which allocates nothing), so a context created anew on the device
 *     (after cudaDeviceReset, or another driver context made current) uses
 *     the array's address in that context.  A call on a stream that is being
 *     captured reuses the address the device's last uncaptured call found:
 *     make the first call on a device, with that device current, before any
 *     stream capture.
 *   - Every call shares the one array and leaves its contents behind; nothing
 *     in it needs to start at zero.  Calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race on it: serialise them.
 */
int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int64_t num_blocks,
                                       int max_blocks_per_seq, float scale, int32_t* dev_err,
                                       void* stream);

/*
 * Grouped decode attention for sequences that share a prefix (forked samples
 * of one prompt, "ans20xx day 31" `fork_sequence`; prefix-cache hits, "P06
 * BlockManager").  Same result as pkv_paged_attention_decode on the same
 * arguments; the grouping only changes how the work is done: the prefix a
 * group shares is read from HBM once for all its members instead of once per
 * member.
 *   group_first   int32 [num_groups + 1] (device): group i is the sequences
 *                 group_first[i] .. group_first[i+1] - 1 (contiguous, covering
 *                 0 .. num_seqs - 1 in order)
 *   seq_group     int32 [num_seqs] (device): the group of each sequence
 *   group_shared  int32 [num_groups] (device): tokens every member holds through
 *                 the same physical blocks as the group's first member; a
 *                 multiple of 16 and of block_size, <= every member's context
 *                 length, <= max_shared_tokens; 0 for no sharing.  Members x
 *                 (num_q_heads / num_kv_heads) must be <= 16.  Violations are
 *                 reported as PKV_DEV_BAD_GROUP.
 *   max_own_tokens  the most tokens any sequence holds past its group's shared
 *                 prefix (a sequence with group_shared 0 owns all its tokens);
 *                 sizes the launch, and a sequence beyond it is reported as
 *                 PKV_DEV_BAD_GROUP
 *   workspace     at least pkv_paged_attention_grouped_workspace_bytes(...)
 * The new tokens must already be in the cache (pkv_reshape_and_cache).  One
 * kernel launch streams every shared prefix and every sequence's own tiles
 * (the shared units first), a second merges the partials; both kinds of unit
 * are cut at the split length pkv_paged_attention_decode would use for the
 * same sizes.
 */
int pkv_paged_attention_decode_grouped(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* group_first,
                                       const int32_t* seq_group, const int32_t* group_shared,
                                       int num_groups, int max_shared_tokens,
                                       int max_own_tokens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int64_t num_blocks, int max_blocks_per_seq,
                                       float scale, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_err, void* stream);

/*
 * Fused cache write + grouped attention: what pkv_reshape_and_cache of the
 * step's new tokens followed by pkv_paged_attention_decode_grouped does, in
 * one launch (as pkv_paged_attention_decode_fused is to
 * pkv_paged_attention_decode).  The new token of sequence s (position
 * context_lens[s] - 1, slot from its block table) must lie past its group's
 * shared prefix, in a block of its own (copy-on-write makes it so); otherwise
 * the write is skipped and PKV_DEV_BAD_GROUP reported.
 *   k_new, v_new  fp16 [num_seqs, num_kv_heads, head_dim], 16-byte aligned
 * Other arguments, layouts and errors as pkv_paged_attention_decode_grouped.
 */
int pkv_paged_attention_decode_grouped_fused(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
    void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* group_first, const int32_t* seq_group, const int32_t* group_shared,
    int num_groups, int max_shared_tokens, int max_own_tokens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
    float scale, void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * Copy-on-write folded into the fused launch: what pkv_copy_blocks of the
 * step's copy-on-write pairs followed by pkv_paged_attention_decode_fused
 * (or _grouped_fused) does, in the one attention launch.  "ans20xx day 31"
 * (fork and copy-on-write): before a forked sequence writes into a block it
 * shares, the block is copied into a private one and the write goes there.
 * For each sequence s with cow_block[s] >= 0, logical block cow_block[s] of
 * its table (the private copy, dst) receives a whole-block copy, K and V of
 * every KV head of this layer, of physical block cow_src[s] (the shared
 * source); then the new token is written (into the copy when it falls in
 * that block) and attention reads the copied block's values.  The unit that
 * streams the block reads it from cow_src[s] (the bytes the copy will hold)
 * and stores the staged tile as the copy, so nothing waits for a separate
 * copy kernel.
 *   cow_block  int32 [num_seqs] (device): logical block index, -1 for none;
 *              one per sequence per call (pkv_cow_targets builds it)
 *   cow_src    int32 [num_seqs] (device): the source physical block
 * The block must hold some of the sequence's own tokens (below
 * context_lens[s], past a group's shared prefix), else PKV_DEV_BAD_POSITION;
 * a source or table entry outside [0, num_blocks) gives PKV_DEV_BAD_BLOCK_ID;
 * either way no copy is made for s.  Every block size the attention entry
 * points take (8, 16, 32, 64): a block of 32 or 64 rows is staged by 2 or 4
 * tiles, each storing its rows, and the rows past the context's last tile are
 * copied from the source by the unit holding that tile.
 * The pages' order is copy, then write.  Within one launch a copy takes the
 * source's rows while other sequences of the launch may write new tokens into
 * that source; so no other sequence may write its new token into a copied
 * source block at a row other than the copying sequence's own new-token row
 * (that row the copy replaces with its own token).  The BlockManager's fork
 * gives every sample of a prompt the same length, so their first writes fall
 * on one row.  Other arguments, layouts and errors as
 * pkv_paged_attention_decode_fused / pkv_paged_attention_decode_grouped_fused.
 */
int pkv_paged_attention_decode_fused_cow(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* cow_block,
    const int32_t* cow_src, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream);
int pkv_paged_attention_decode_grouped_fused_cow(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
    void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* group_first, const int32_t* seq_group, const int32_t* group_shared,
    int num_groups, int max_shared_tokens, int max_own_tokens, const int32_t* cow_block,
    const int32_t* cow_src, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * Host helper for the _cow launches (host memory only): for copy-on-write
 * pairs (src, dst) as pkv_bm_take_cow_pairs returns them, find the sequence
 * and logical block whose table entry is dst.  cow_block[s] = that logical
 * block and cow_src[s] = src; -1 / -1 for sequences no pair names.  Returns
 * PKV_OK; PKV_ERR_BAD_INDEX if a dst appears in no table, or in two places;
 * PKV_ERR_UNSUPPORTED if one sequence needs two copies (use pkv_copy_blocks).
 *   pairs int64 [num_pairs, 2], tables int32 [num_seqs, max_blocks] (host)
 */
int pkv_cow_targets(const int64_t* pairs, int num_pairs, const int32_t* tables, int num_seqs,
                    int max_blocks, int32_t* cow_block, int32_t* cow_src);

/* Workspace bytes pkv_paged_attention_decode_grouped needs (host only). */
size_t pkv_paged_attention_grouped_workspace_bytes(int num_seqs, int num_q_heads,
                                                   int max_blocks_per_seq, int block_size,
                                                   int head_dim, int max_shared_tokens);

/*
 * Host planning for pkv_paged_attention_decode_grouped (host memory only).
 * Consecutive sequences whose tables start with the same physical block form a
 * group of at most max_members (16 / (num_q_heads / num_kv_heads) for the
 * kernel); a group shares the longest run of leading blocks that every member
 * has in common with its first member, cut to a multiple of 16 tokens and of
 * block_size and to the shortest member's context length.  Sequences are not
 * reordered: sort them by their first block beforehand to group them all.
 *   tables [num_seqs, max_blocks], context_lens [num_seqs] (host)
 *   outputs (host): group_first [num_seqs + 1], seq_group [num_seqs],
 *   group_shared [num_seqs] (the first *num_groups entries are used),
 *   *max_shared_tokens, *max_own_tokens for the attention call.
 */
int pkv_plan_shared_prefix_groups(const int32_t* tables, const int32_t* context_lens,
                                  int num_seqs, int max_blocks, int block_size, int max_members,
                                  int32_t* group_first, int32_t* seq_group,
                                  int32_t* group_shared, int* num_groups,
                                  int* max_shared_tokens, int* max_own_tokens);

/* ---- cache write --------------------------------------------------------- */
/*
 * reshape_and_cache: store the K/V of new tokens at their slots.
 * "ans20xx day 31": a decoded token is written into the last, not yet full block
 * of its sequence; "P06 BlockManager" gives its slot.  For i < num_tokens:
 *   k_cache[slot / bs, slot % bs, :, :] = k[i, :, :]   (same for v)
 * with slot = slot_mapping[i].  A negative slot skips the token (padding); a slot
 * >= num_blocks * block_size is skipped and reported as PKV_DEV_BAD_SLOT.
 * Two tokens with the same slot in one call race (undefined which lands).
 *   k, v        fp16 [num_tokens, num_kv_heads, head_dim], 16-byte aligned
 *   slot_mapping int64 [num_tokens] (device)
 *   k_cache, v_cache fp16 [num_blocks, block_size, num_kv_heads, head_dim]
 *   num_kv_heads * head_dim must be a multiple of 8.  Bit-exact copy.
 */
int pkv_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int64_t num_blocks, int32_t* dev_err,
                          void* stream);

/*
 * Slot mapping on the device: slot_mapping[s] = table[s][p / bs] * bs + p % bs
 * with p = positions[s] ("P06 BlockManager", problem summary).  p < 0 gives -1
 * (no write).  p >= max_blocks_per_seq * bs or a table entry outside
 * [0, num_blocks) gives -1 and PKV_DEV_BAD_POSITION / PKV_DEV_BAD_BLOCK_ID.
 *   block_tables int32 [num_seqs, max_blocks_per_seq], positions int32
 *   [num_seqs], slot_mapping int64 [num_seqs]; all device.
 */
int pkv_slot_mapping(const int32_t* block_tables, const int32_t* positions, int num_seqs,
                     int max_blocks_per_seq, int block_size, int64_t num_blocks,
                     int64_t* slot_mapping, int32_t* dev_err, void* stream);

/* ---- copy-on-write block copy -------------------------------------------- */
/*
 * copy_blocks: for every pair (src, dst) and every layer,
 *   k_caches[layer][dst] = k_caches[layer][src]   (same for v_caches)
 * copying the whole block.  "ans20xx day 31", toy COW append: when a sequence
 * writes into a block it still shares after a fork, it takes a new block and
 * the old block's KV is copied into it (the page copies the valid bytes; the
 * whole block is copied here, so dst equals src byte for byte).
 *   k_caches, v_caches  HOST arrays of num_layers device pointers (one launch per
 *                64 layers)
 *   block_pairs  int64 [num_pairs, 2] (device), (src, dst) per row; ids outside
 *                [0, num_blocks) are skipped and reported as PKV_DEV_BAD_BLOCK_ID
 *   block_bytes  bytes of one block of one cache (16 * num_kv_heads * head_dim * 2
 *                for fp16); a multiple of 16, pointers 16-byte aligned
 * A dst that is also another pair's src, or two pairs with one dst, race.
 */
int pkv_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                    const int64_t* block_pairs, int num_pairs, int64_t block_bytes,
                    int64_t num_blocks, int32_t* dev_err, void* stream);

/* ---- swap between pools ---------------------------------------------------- */
/*
 * swap_blocks: for every pair (src, dst) and every pool i,
 *   dst_pools[i][dst] = src_pools[i][src]   (block_bytes bytes each)
 * "qaqbuyan: vLLM PagedAttention", `_preempt_request`: a preempted request's KV
 * blocks are copied from GPU memory to CPU memory (swap-out) and its GPU blocks
 * freed; swap-in copies them back into freshly allocated blocks.  One kernel
 * gathers the blocks, so either side may be host memory that the GPU can
 * address: pinned (page-locked) and mapped, e.g. cudaHostAlloc or torch's
 * pin_memory on a unified-address system.  The copy travels over the host link.
 *   src_pools, dst_pools  HOST arrays of num_pools pointers (e.g. K and V of
 *                         each layer), 16-byte aligned
 *   block_pairs  int64 [num_pairs, 2] (src, dst), readable by the GPU; ids
 *                outside [0, src_num_blocks) / [0, dst_num_blocks) are skipped
 *                and reported as PKV_DEV_BAD_BLOCK_ID
 *   block_bytes  bytes of one block of one pool, a multiple of 16
 * Bit-exact.  Overlapping destinations race.
 */
int pkv_swap_blocks(const void* const* src_pools, void* const* dst_pools, int num_pools,
                    const int64_t* block_pairs, int num_pairs, int64_t block_bytes,
                    int64_t src_num_blocks, int64_t dst_num_blocks, int32_t* dev_err,
                    void* stream);

/* ---- diagnostics ------------------------------------------------------------ */
/*
 * Self-test of the bounded waits the kernels use on their TMA barriers (the
 * pages have no counterpart; it exercises this library's failure path).  One
 * thread waits on an mbarrier that nothing arrives on; after limit_ms (1..2000)
 * the wait gives up, stores PKV_DEV_WAIT_TIMEOUT into *dev_err (device int32,
 * zero beforehand) and 0 into *landed (device int32), and the kernel returns:
 * no hang, no trap, the context stays usable.
 */
int pkv_selftest_bounded_wait(int32_t* dev_err, int32_t* landed, int limit_ms, void* stream);

/*
 * Synthetic inputs (benchmarks, the model-less serving driver; not part of the
 * paged-attention method).  Writes n standard-normal fp16 values to dst (device,
 * 16-byte aligned): element i is element offset + i of a stream keyed by seed,
 * so consecutive calls with offsets advancing by n continue one stream.
 * Element j takes output j / 2 of SplitMix64 (Steele, Lea and Flood 2014)
 * started at state seed, and the Box-Muller transform of its bits 40..63
 * (u1 in (0, 1]) and 16..39 (u2 in [0, 1)): cosine for even j, sine for odd,
 * in fp32 with the hardware sine/cosine (within ~1e-5 of the exact transform
 * before the fp16 rounding).
 * Returns INVALID_ARG for n < 0 or a misaligned / NULL dst (n > 0).
 */
int pkv_fill_normal_f16(void* dst, int64_t n, uint64_t seed, uint64_t offset, void* stream);

/* ---- host BlockManager ---------------------------------------------------- */
/*
 * The BlockManager of "P06 BlockManager" (free list taken FIFO, reference
 * counts, chained block hashes with at most (len - 1) / bs matchable blocks, an
 * LRU pool of evictable cached blocks, atomic allocate/append, reverse-order
 * free), plus fork and copy-on-write from "ans20xx day 31".  Host memory only,
 * single-threaded: one handle must not be used from two threads at once.
 * Sequence ids are caller-chosen int64 values.  Operations that fail with
 * PKV_ERR_OUT_OF_BLOCKS leave every piece of state unchanged.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* initial_free_order: NULL for 0..num_blocks-1, or a permutation of it (the
 * order in which free blocks are handed out).  Returns NULL on bad arguments. */
pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size, int enable_prefix_cache,
                                 const int32_t* initial_free_order);
/* Frees the manager (NULL is ignored). */
void pkv_bm_destroy(pkv_block_manager* bm);

/* Allocate a new sequence holding num_tokens prompt tokens.  Writes its block
 * table (up to table_cap entries) and sets *num_table_blocks and
 * *num_cached_tokens (prefix-cache hits x bs).  PKV_ERR_INVALID_ARG if the id
 * is in use or table_cap is too small (state unchanged). */
int pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                    int64_t num_tokens, int32_t* table_out, int64_t table_cap,
                    int64_t* num_table_blocks, int64_t* num_cached_tokens);

/* Append one token; *slot_out receives its slot.  Takes a new block at a block
 * boundary, or -- when the partial last block is shared after a fork -- a
 * private copy whose (old, new) pair is queued for pkv_bm_take_cow_pairs. */
int pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int32_t token, int64_t* slot_out);

/* Append one token to each of n sequences, in order; slots_out[i] receives each
 * slot.  Stops at the first failure and returns its status with
 * *num_done = appends completed (each completed append stays). */
int pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* tokens,
                        int64_t n, int64_t* slots_out, int64_t* num_done);

/* child shares every block of parent (ref + 1 each) and copies its tokens. */
int pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Release a sequence (unknown ids are ignored; never fails). */
int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);

/* Slot of position pos ("P06 BlockManager": table[pos / bs] * bs + pos % bs);
 * PKV_ERR_BAD_INDEX for an unknown id, a negative position or one past its table. */
int pkv_bm_slot(const pkv_block_manager* bm, int64_t seq_id, int64_t pos, int64_t* slot_out);
/* Blocks an allocation may take: free list + evictable pool. */
int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);
/* The coarse check ceil(num_tokens / bs) <= num_free_blocks: 1 or 0. */
int pkv_bm_can_allocate(const pkv_block_manager* bm, int64_t num_tokens);
/* Table length of a sequence (or PKV_ERR_BAD_INDEX); copies up to cap entries. */
int64_t pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out, int64_t cap);
/* Tokens a sequence holds (prompt + appended), or PKV_ERR_BAD_INDEX. */
int64_t pkv_bm_num_tokens(const pkv_block_manager* bm, int64_t seq_id);
/* Prompt tokens its allocate found in the prefix cache, or PKV_ERR_BAD_INDEX. */
int64_t pkv_bm_num_cached_tokens(const pkv_block_manager* bm, int64_t seq_id);
/* Rows [n, max_blocks] of block tables (pad entries past each table) and the
 * token counts of the listed sequences, ready for the attention kernel. */
int pkv_bm_fill_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int64_t n,
                             int32_t* tables_out, int64_t max_blocks, int32_t pad,
                             int32_t* context_lens_out);
/* Pending copy-on-write pairs: returns their count; when cap_pairs is at least
 * that count the pairs are written to out ([count, 2] int64) and drained. */
int64_t pkv_bm_take_cow_pairs(pkv_block_manager* bm, int64_t* out, int64_t cap_pairs);

/* Introspection (tests): free list in hand-out order, evictable pool oldest
 * first, reference counts [num_blocks].  Return the element count. */
int64_t pkv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int64_t cap);
int64_t pkv_bm_evictable_list(const pkv_block_manager* bm, int32_t* out, int64_t cap);
int64_t pkv_bm_ref_counts(const pkv_block_manager* bm, int32_t* out, int64_t cap);
/* 0 when invariants I1..I5 of "P06 BlockManager" hold, else the number of the
 * first one violated (1..5). */
int pkv_bm_check_invariants(const pkv_block_manager* bm);

/* ---- host continuous-batching scheduler ------------------------------------- */
/*
 * The per-step host work of a decode server without a model ("qaqbuyan: vLLM
 * PagedAttention", `ContinuousBatchingScheduler.step` and `_preempt_request`;
 * "ans20xx day 31", scheduling): release finished requests, admit waiting ones
 * first-come first-served while the BlockManager can allocate them (prefix
 * cache hits skip part of the prompt), append one sampled token per running
 * request, and on OutOfBlocks preempt -- of the requests not yet decoded in
 * this step, the one with the most generated tokens -- by recompute (requeue
 * with its tokens; prefilled again later) or swap (its blocks go to host
 * blocks, and come back on re-admission past the prefix-cache hits).  Tokens
 * are drawn from a counter-based generator keyed by (seed, request, position).
 * Host memory only; the BlockManager is borrowed and must outlive the
 * scheduler; single-threaded.
 */
typedef struct pkv_scheduler pkv_scheduler;

/* Caller-owned buffers one step fills, in the order the device must use them:
 * swap-in pairs and prefill slots (admissions), swap-out pairs (preemptions),
 * copy-on-write pairs, then the decode batch. */
typedef struct pkv_sched_step_out {
  int64_t* batch_rids;         /* [max_batch] sequence ids of the decode batch */
  int32_t* positions;          /* [max_batch] position decoded (context length - 1) */
  int32_t* tokens;             /* [max_batch] token appended */
  int64_t* slots;              /* [max_batch] its slot */
  int32_t* block_tables;       /* [max_batch, max_blocks_per_seq], -1 padded */
  int32_t* context_lens;       /* [max_batch] */
  int64_t* prefill_rids;       /* [prefill_cap] rows to write for admissions ... */
  int32_t* prefill_positions;  /* ... their positions ... */
  int64_t* prefill_slots;      /* ... and slots */
  int64_t prefill_cap;         /* >= max_batch * max_blocks_per_seq * block_size */
  int64_t* swap_in_pairs;      /* [swap_cap, 2] (host block, device block) */
  int64_t* swap_out_pairs;     /* [swap_cap, 2] (device block, host block) */
  int64_t swap_cap;            /* >= max_batch * max_blocks_per_seq */
  int64_t* cow_pairs;          /* [cow_cap, 2] (src, dst) */
  int64_t cow_cap;             /* >= max_batch */
  /* Shared-prefix groups of the decode batch (pkv_paged_attention_decode_grouped):
   * with group_limit > 0 the batch is ordered by first physical block and
   * planned as pkv_plan_shared_prefix_groups does; 0 leaves it unplanned. */
  int32_t group_limit;         /* in: at most this many members per group */
  int32_t* group_first;        /* [max_batch + 1] */
  int32_t* seq_group;          /* [max_batch] */
  int32_t* group_shared;       /* [max_batch] */
  int32_t num_groups, max_shared_tokens, max_own_tokens;
  int32_t num_batch, num_prefill, num_swap_in, num_swap_out, num_cow;
  int32_t num_admitted, num_finished, num_preempted;
  int64_t cached_tokens;       /* prompt tokens found in the prefix cache this step */
} pkv_sched_step_out;

/* preemption_swap: 0 = recompute, 1 = swap into host_blocks host blocks
 * (falls back to recompute when they run short).  NULL on bad arguments. */
pkv_scheduler* pkv_sched_create(pkv_block_manager* bm, int max_batch, int max_blocks_per_seq,
                                int block_size, int preemption_swap, int64_t host_blocks,
                                uint64_t seed, int vocab);
/* Frees the scheduler (not its BlockManager; NULL is ignored). */
void pkv_sched_destroy(pkv_scheduler* sched);
/* Queue a request (ids unique; prompt non-empty; prompt + max_new_tokens must
 * fit max_blocks_per_seq blocks). */
int pkv_sched_add_request(pkv_scheduler* sched, int64_t rid, const int32_t* prompt,
                          int64_t num_prompt_tokens, int64_t max_new_tokens);
/* Plan one step into *out (capacities as above, checked before any change). */
int pkv_sched_step(pkv_scheduler* sched, pkv_sched_step_out* out);
/* Device side of a step's decode batch, for pkv_sched_launch_decode. */
typedef struct pkv_decode_launch {
  void* k_cache;               /* fp16 [num_blocks, block_size, num_kv_heads, head_dim] */
  void* v_cache;
  int64_t num_blocks;
  int num_q_heads, num_kv_heads, head_dim;
  const void* q;               /* fp16 [max_batch, num_q_heads, head_dim], rows of the batch */
  const void* k_new;           /* fp16 [max_batch, num_kv_heads, head_dim] */
  const void* v_new;
  void* out;                   /* fp16 [max_batch, num_q_heads, head_dim] */
  void* meta;                  /* device staging for the step's metadata ... */
  size_t meta_bytes;           /* ... of at least pkv_sched_meta_bytes() */
  void* workspace;             /* attention workspace (grouped size when grouping) */
  size_t workspace_bytes;
  float scale;
  int32_t* dev_err;
  int32_t meta_staged;         /* nonzero: pkv_sched_stage_decode already copied this
                                  step's metadata into meta (skip the copy) */
} pkv_decode_launch;

/* Device staging bytes pkv_sched_launch_decode needs. */
size_t pkv_sched_meta_bytes(const pkv_scheduler* sched);

/* Enqueue the decode part of a planned step on `stream`: copy the batch's
 * block tables, context lengths and groups from out's (pinned) arrays to
 * d->meta, then one fused launch writes the new tokens' K/V at their slots
 * (recomputed from the tables; they equal out->slots) and runs paged
 * attention -- grouped when the step planned shared-prefix groups -- plus
 * the merge launch when a context spans several splits.  The caller has
 * filled q / k_new / v_new for rows 0 .. out->num_batch - 1 and enqueued the
 * step's swaps, prefill writes and copies before.  When out's block_tables,
 * context_lens, group_first, seq_group and group_shared lie back to back in
 * that order (max_batch x max_blocks, max_batch, max_batch + 1, max_batch and
 * max_batch int32), the metadata goes to the device in one copy. */
int pkv_sched_launch_decode(const pkv_scheduler* sched, const pkv_sched_step_out* out,
                            const pkv_decode_launch* d, void* stream);

/* The metadata copy of pkv_sched_launch_decode alone, enqueued on `stream`
 * (e.g. a copy stream, so that it overlaps the previous step's kernels): the
 * caller then orders the decode stream after it (an event) and launches with
 * d->meta_staged set.  d->meta must not be in use by an earlier step's kernels
 * still running (double-buffer it), and out's pinned arrays must stay
 * untouched until the copy has completed. */
int pkv_sched_stage_decode(const pkv_scheduler* sched, const pkv_sched_step_out* out,
                           const pkv_decode_launch* d, void* stream);

/* Requests waiting or running. */
int64_t pkv_sched_num_unfinished(const pkv_scheduler* sched);
/* Tokens of a request so far (prompt + generated): the count; copies up to cap. */
int64_t pkv_sched_request_tokens(const pkv_scheduler* sched, int64_t rid, int32_t* out,
                                 int64_t cap);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
