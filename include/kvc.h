/*
 * kvc.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library.
 *
 * What the library computes (sources are web pages, cited by title and section):
 *  - "La caché de claves y valores: cuánto cuesta cada token" (gustavoai.dev),
 *    section "Las claves y los valores de una posición no cambian": a decode
 *    token appends its k_t, v_t to the end of each head's cache and its query
 *    row then attends, unmasked, over every cached row including its own:
 *        o_t = softmax(q_t K^T * scale) V.
 *  - "Tornar a inferência barata: KV cache, batching e quantização"
 *    (neuralialabs.com), PagedAttention paragraph: the cache is stored in
 *    fixed-size blocks with one block table per sequence, logically
 *    contiguous and physically scattered; sequences with a common prefix can
 *    share the blocks that hold it.  Grouped-query attention paragraph: each
 *    KV head is shared by a group of query heads.
 *  - "Aufmerksamkeit" feed (chatgpz.de), PagedAttention article, SECTION 2
 *    (PagePool, PagedRequest: FIFO free list, refcounts, a page claimed at each
 *    page boundary) and SECTION 3 (copy-on-write prefix sharing); xformers
 *    article parts 4-5 (packed varlen batches with block-diagonal (causal)
 *    masks; BMGHK grouped-query layout); FlashAttention article, "Was ist der
 *    mathematische Aspekt von Softmax?" (per-block max and exp-sum, rescaled
 *    by e^(m_block - m_global) when merged).
 *
 * Conventions
 *  - Every function returns kvc_status; nothing throws across the ABI.  On
 *    failure kvc_last_error_string() (thread-local) holds a message.
 *  - Device buffers are allocated by the caller and passed as raw device
 *    pointers; the library never allocates device memory.  The library owns
 *    only the host metadata behind a kvc_handle (free list, refcounts).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Device work is asynchronous on it; argument errors are
 *    returned synchronously before anything is launched.
 *  - Element type: fp16 (IEEE binary16) for q, k, v and the caches; outputs
 *    fp16 or fp32 (kvc_dtype).  Arithmetic accumulates in fp32.
 *  - Cache layout (this library's choice; results do not depend on it): all
 *    layers in one allocation per K and V, element
 *        pool[layer][block][kv_head][offset][dim]
 *    i.e. [L][NB][Hkv][bs][D], so one (block, KV head) tile of bs*D fp16 is
 *    contiguous.  slot = block * bs + offset.
 *  - Query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *  - Kernels never spin without bound and never trap: device-side problems
 *    (an out-of-range id, a bad context length, an expired wait) set bits in a
 *    sticky device error word (kvc_device_error_flags) and the affected rows
 *    are skipped or zero-filled.  Checked mode validates device-side index
 *    arrays on the host first and returns the error synchronously.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVC_OK = 0,
    KVC_ERR_INVALID = 1,     /* bad argument, or a block that is not live */
    KVC_ERR_OOM = 2,         /* the block pool has no free block ("OOM -- no free pages") */
    KVC_ERR_CAPACITY = 3,    /* a position/context beyond the block table or the pool */
    KVC_ERR_CUDA = 4,        /* a CUDA runtime call failed */
    KVC_ERR_UNSUPPORTED = 5  /* a shape the library has no kernel for (head_dim, block_size, group) */
} kvc_status;

typedef enum { KVC_F16 = 0, KVC_F32 = 1 } kvc_dtype;

/* device error word bits (kvc_device_error_flags) */
#define KVC_DEVERR_BLOCK_ID 0x1u   /* a block-table entry outside [0, num_blocks) */
#define KVC_DEVERR_CONTEXT 0x2u    /* a context length < 1 or beyond the table / max_context_len */
#define KVC_DEVERR_SLOT 0x4u       /* an append slot >= num_blocks * block_size */
#define KVC_DEVERR_TIMEOUT 0x8u    /* a bounded wait on a copy expired (the work was skipped) */
#define KVC_DEVERR_SEQLENS 0x10u   /* cu_seqlens not non-decreasing / beyond total_tokens */

typedef struct {
    int num_layers;   /* L */
    int num_blocks;   /* NB, physical blocks per layer */
    int block_size;   /* bs, tokens per block (16) */
    int num_kv_heads; /* Hkv */
    int head_dim;     /* D (64 or 128) */
    int dtype;        /* kvc_dtype of the cache: KVC_F16 */
} kvc_config;

typedef struct kvc_cache* kvc_handle;

/* ---- diagnostics ---------------------------------------------------- */
const char* kvc_last_error_string(void);
int kvc_version(void);
/* Checked mode (process-wide, default off): device index arrays passed to
 * kv_append / paged_decode_attention / prefill_attention are copied to the
 * host (synchronising `stream`) and validated before launch. */
kvc_status kvc_set_checked_mode(int on);
/* Read (and optionally clear) the sticky device error word of the current
 * device.  Synchronous. */
kvc_status kvc_device_error_flags(uint32_t* flags, int clear);

/* ---- cache geometry and the block pool (host) ------------------------
 * Bytes of ONE pool (K or V) for all layers: L*NB*Hkv*bs*D*2.  The K+V total
 * per token is 2*L*Hkv*D*2 bytes (the neuralialabs page's formula). */
kvc_status kv_cache_pool_bytes(const kvc_config* cfg, size_t* bytes);

/* Create a cache over caller-allocated pools (each kv_cache_pool_bytes
 * bytes, 16-byte aligned).  k_pool/v_pool may both be NULL: a host-only
 * cache whose block pool works but whose device operations return
 * KVC_ERR_INVALID.  The free list starts as 0, 1, ..., NB-1. */
kvc_status kv_cache_create(const kvc_config* cfg, void* k_pool, void* v_pool, kvc_handle* out);
kvc_status kv_cache_destroy(kvc_handle h);
/* Device pointers to one layer's K and V slices ([NB][Hkv][bs][D]). */
kvc_status kv_cache_layer(kvc_handle h, int layer, void** k_layer, void** v_layer);

/* PagePool semantics (chatgpz.de PagedAttention article, SECTION 2-3):
 * alloc pops the head of the FIFO free list (refcount 1; empty -> KVC_ERR_OOM);
 * share increments a live block's refcount; release decrements it and at zero
 * appends the block to the tail of the free list.  Sharing or releasing a
 * block that is not live is KVC_ERR_INVALID. */
kvc_status kv_block_alloc(kvc_handle h, int32_t* block);
kvc_status kv_block_share(kvc_handle h, int32_t block);
kvc_status kv_block_release(kvc_handle h, int32_t block);
kvc_status kv_block_refcount(kvc_handle h, int32_t block, int32_t* refcount);
kvc_status kv_block_num_free(kvc_handle h, int32_t* num_free);
/* (NB - free) / NB * 100 */
kvc_status kv_cache_utilisation(kvc_handle h, double* percent);

/* Copy-on-write of one block: if its refcount is > 1, allocate a new block,
 * queue a device copy of the whole block (all layers, K and V) on `stream`,
 * release the old reference and return the new id; otherwise *new_block =
 * block and nothing is copied. */
kvc_status kv_block_cow(kvc_handle h, int32_t block, int32_t* new_block, void* stream);
/* Device copy of whole blocks src[i] -> dst[i] (host arrays of n ids), all
 * layers, K and V, on `stream`.  Bit copy. */
kvc_status kv_copy_blocks(kvc_handle h, const int32_t* src, const int32_t* dst, int n, void* stream);

/* ---- slot arithmetic (host) -----------------------------------------
 * The PagedAttention article of the chatgpz.de feed, SECTION 2 (PagedRequest:
 * token position p lives in page block_table[p / page_size] at offset
 * p % page_size), and the neuralialabs.com PagedAttention paragraph (a block
 * table maps a sequence's logical blocks to physical ones).
 * Slots of positions first_pos[b] .. first_pos[b]+count[b]-1 of every
 * sequence b, packed in order into slots (host, sum(count) entries):
 *     slot = block_table[b][pos / bs] * bs + pos % bs.
 * block_table is a host [B][max_blocks] array.  A position past the table
 * or on a negative entry is KVC_ERR_CAPACITY. */
kvc_status kv_slot_mapping(const int32_t* block_table, int max_blocks, int B, const int32_t* first_pos,
                           const int32_t* count, int block_size, int64_t* slots);

/* One decode step's block management for B sequences (host).  Follows the
 * chatgpz.de PagedAttention article: SECTION 2 (PagedRequest claims a new
 * page from the FIFO pool when a token starts a page) and SECTION 3
 * (copy-on-write: a token written into a page whose refcount is above one
 * first gets a private copy of that page).  For each sequence b in order, the
 * new token goes to position positions[b]; if that position starts a new
 * block (positions[b] == num_blocks[b] * bs) a block is allocated and
 * appended to the table; otherwise, if its block has refcount > 1, a new
 * block is allocated, the pair (old, new) is recorded in copy_src/copy_dst
 * (capacity B), the old reference is released and the table entry replaced.
 * slot_mapping[b] receives the token's slot.  The caller then runs
 * kv_copy_blocks(copy_src, copy_dst, *n_copies) BEFORE kv_append.
 * block_table ([B][max_blocks]) and num_blocks ([B]) are host arrays updated
 * in place.  All-or-nothing: on KVC_ERR_OOM / KVC_ERR_CAPACITY nothing is
 * changed. */
kvc_status kv_step_prepare(kvc_handle h, int32_t* block_table, int max_blocks, int32_t* num_blocks,
                           const int32_t* positions, int B, int64_t* slot_mapping, int32_t* copy_src,
                           int32_t* copy_dst, int* n_copies);

/* ---- device operations ----------------------------------------------
 * kv_append ("La caché de claves y valores", step 2 of a decode token):
 * k_cache[layer][slot] = k_new[t], v_cache[layer][slot] = v_new[t] for every
 * token t < n and KV head, where slot = slot_mapping[t].  k_new/v_new are
 * device [n][Hkv][D] fp16; slot_mapping is device int64 [n]; a negative slot
 * is skipped; a slot >= NB*bs sets KVC_DEVERR_SLOT and is skipped.  Bit copy. */
kvc_status kv_append(kvc_handle h, int layer, const void* k_new, const void* v_new,
                     const int64_t* slot_mapping, int n, void* stream);

/* Split plan of paged_decode_attention for these sizes on the current
 * device: the number of context splits (CTAs along the context, a whole
 * number of thread-block clusters of up to 8), the blocks per split and the
 * workspace bytes it needs (zero unless the longest context needs more than
 * one cluster).  blocks_per_split = 0 picks automatically. */
kvc_status paged_decode_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                             int blocks_per_split, int* num_splits, int* blocks_per_split_out,
                             size_t* workspace_bytes);
/* Zero-fill a workspace (cudaMemsetAsync).  Optional: the decode kernels
 * write every workspace word they read.  Calls that share a workspace must not
 * overlap in time (same stream, or ordered by events). */
kvc_status paged_decode_workspace_init(void* workspace, size_t bytes, void* stream);

/* Paged GQA decode attention for one token per sequence ("La caché de
 * claves y valores", gustavoai.dev, section "Las claves y los valores de una
 * posición no cambian": the new query row attends, unmasked, over every
 * cached row; neuralialabs.com PagedAttention and grouped-query attention
 * paragraphs: the rows come through the sequence's block table and a group of
 * query heads shares one KV head; xformers article part 5: contiguous groups):
 *   out[b][h] = softmax(q[b][h] . K_b^T * scale) V_b
 * over the context_lens[b] tokens of sequence b (the appended token
 * included), K_b/V_b gathered through block_table[b] from KV head
 * h / (Hq / Hkv).
 *   q            device fp16 [B][Hq][D]
 *   k_cache      device fp16 [num_blocks][Hkv][bs][D] (one layer), v_cache same
 *   block_table  device int32 [B][max_blocks]
 *   context_lens device int32 [B], 1 <= ctx <= min(max_blocks*bs, max_context_len)
 *   out          device [B][Hq][D], out_dtype KVC_F16 or KVC_F32
 *   workspace    device, 16-byte aligned, >= paged_decode_plan(...)'s bytes (may be NULL when
 *                that is 0)
 * The context of each sequence is cut into splits of blocks_per_split blocks;
 * each (sequence, KV head, split) is one CTA that keeps the running max and
 * exp-sum per query head; the splits merge with the rescaling rule of the
 * FlashAttention article, on chip within a thread-block cluster and, for
 * contexts longer than one cluster covers, through the workspace.
 * Preconditions: Hq % Hkv == 0, Hq/Hkv <= 64, head_dim in {64, 128},
 * block_size == 16; 16-byte aligned pointers. */
kvc_status paged_decode_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                  const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                  int B, int Hq, int Hkv, int head_dim, int block_size,
                                  int max_context_len, float scale, void* out, int out_dtype,
                                  void* workspace, size_t workspace_bytes, int blocks_per_split,
                                  void* stream);

/* The same step with the append fused in (steps 2 and 3 of a decode token
 * on the gustavoai.dev page in one kernel): for every sequence b the new
 * token's rows k_new[b], v_new[b] (device fp16 [B][Hkv][D]) are written to
 * position context_lens[b]-1 of the cache, i.e. slot
 * block_table[b][(ctx-1)/bs]*bs + (ctx-1)%bs, and take part in the attention
 * of that same call.  Bit-identical cache contents to kv_append with those
 * slots followed by paged_decode_attention. */
kvc_status paged_decode_append_attention(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                         void* v_cache, int num_blocks,
                                         const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                         int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                         float scale, void* out, int out_dtype, void* workspace,
                                         size_t workspace_bytes, int blocks_per_split, void* stream);

/* Cascade (shared-prefix) decode.  Same result as paged_decode_attention on
 * the same arguments; only the way it is computed differs.  Sequences form
 * groups of consecutive indices that share the leading blocks of their block
 * tables (a common prefix whose blocks the pool refcounts: the prefix
 * sharing of the chatgpz.de PagedAttention article, SECTION 3, and the
 * neuralialabs.com PagedAttention paragraph).  Each group's shared blocks are
 * read once and attended by all of its members together; every sequence's
 * remaining blocks are attended as in paged_decode_attention; the two
 * partial states merge with the rescaling rule of the FlashAttention article.
 *   group_start    device int32 [n_groups + 1]: group g is sequences
 *                  group_start[g] .. group_start[g+1]-1; group_start[0] = 0,
 *                  group_start[n_groups] = B, at most 8 sequences per group
 *   shared_blocks  device int32 [B]: the number of leading blocks that every
 *                  member of b's group has in common (the same value for all
 *                  members; 0 = none), with 16 * shared_blocks[b] <
 *                  context_lens[b] (each member keeps at least its newest
 *                  token private)
 *   max_shared_blocks  host upper bound of shared_blocks (sizes the launch)
 *   workspace      device, 16-byte aligned, >= paged_decode_cascade_plan's bytes
 * The members' rows must really begin with the same block ids: the call
 * reads the shared blocks through the first member's row.  Checked mode
 * verifies all of it on the host; unchecked, a bad group sets
 * KVC_DEVERR_CONTEXT and its outputs are undefined.  Three kernel launches
 * (prefix, suffix, merge) on `stream`. */
/* Host helper for the cascade: forms the groups from host copies of the
 * block table [B][max_blocks] and the context lengths [B].  Consecutive
 * sequences whose rows begin with the same block id form a group (split into
 * runs of at most max_group, 1..8); a group's shared block count is the
 * number of leading entries all its members have in common, capped so that
 * every member keeps at least its newest token outside it
 * (16 * shared <= ctx - 1).  A sequence alone, or whose group shares nothing,
 * gets shared 0.  Writes group_start [n_groups + 1] (capacity B + 1),
 * *n_groups, shared_blocks [B] and *max_shared (all host memory). */
kvc_status kv_cascade_groups(const int32_t* block_table, int B, int max_blocks, const int32_t* context_lens,
                             int block_size, int max_group, int32_t* group_start, int* n_groups,
                             int32_t* shared_blocks, int* max_shared);
kvc_status paged_decode_cascade_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                     int n_groups, int max_shared_blocks, size_t* workspace_bytes);
/* Routing of cascade calls (process-wide).  A call saves at most
 * (B - n_groups) * max_shared_blocks block reads per KV head against the
 * plain decode; when that is below `blocks`, it runs paged_decode_attention's
 * kernel on the same arguments (one launch, every block read per sequence)
 * instead of the three cascade launches, which would cost more than they
 * save.  The result definition is the same either way.  Default 36000,
 * measured on GB300 (one call, L2 flushed): 8 groups x 8 sequences sharing
 * 512 blocks (28,672 saved) ran 0.94x the plain decode, 25 x 8 sharing 256
 * (44,800 saved) 1.13x.  0 always runs the cascade.
 * paged_decode_cascade_plan's workspace size covers the route that the
 * setting at plan time picks: plan again after changing it.  KVC_ERR_INVALID
 * for a negative count. */
kvc_status kvc_set_cascade_min_saved_blocks(int blocks);
kvc_status paged_decode_cascade_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                          const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                          const int32_t* group_start, const int32_t* shared_blocks, int n_groups,
                                          int max_shared_blocks, int B, int Hq, int Hkv, int head_dim,
                                          int block_size, int max_context_len, float scale, void* out, int out_dtype,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* Multi-token decode (speculative verification): each sequence appends
 * q_len (1..8) new tokens in one step and all of them attend at once,
 * causally among themselves: token t sits at position ctx - q_len + t and
 * attends to positions 0 .. ctx - q_len + t of its context (speculative
 * decoding paragraph of "Tornar a inferência barata" (neuralialabs.com):
 * verifying gamma proposed tokens is one forward pass over gamma positions).
 *   q        device fp16 [B][q_len][Hq][D]
 *   out      device [B][q_len][Hq][D], out_dtype KVC_F16 or KVC_F32
 *   context_lens  device int32 [B], including the q_len new tokens
 *                 (q_len <= ctx <= min(max_blocks * bs, max_context_len))
 *   workspace     device, 16-byte aligned, >= paged_decode_multi_plan's bytes
 * Other arguments as in paged_decode_attention; the new tokens' K/V must be
 * in the cache already (kv_append with their slots).  Each block is read
 * once for all q_len tokens.  The softmax weights multiply V in fp16 and the
 * row sums add the same rounded weights, so every output row is an exact
 * convex combination of V rows with weights off by at most 2^-11 relative
 * (the prefill's default form); the single-token decode keeps ~fp32 weights.  One kernel launch where a thread-block cluster
 * covers the longest context (the plan's workspace is then 0 bytes), else two
 * (partial states per cluster, then their merge). */
kvc_status paged_decode_multi_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                   int q_len, size_t* workspace_bytes);
/* Process-wide: 1 runs multi-token calls with head_dim 64 and q_len x
 * (Hq / Hkv) <= 64 query rows on a tensor-core (tcgen05) kernel instead of
 * the default mma.sync kernel; 0 (the default) keeps the mma.sync kernel.
 * Both give the same result within the decode tolerance.  The tensor-core
 * kernel puts the 128 keys of a tile on the products' M side, one TMEM lane
 * and softmax thread per key, and the query rows on N.  On GB300 it measured
 * slower for 32 sequences x 2048 tokens, 14 / 2 heads (per layer of a
 * 24-layer graph, q_len 2 / 4 / 8: 13.3 / 15.5 / 21.6 us against 8.4 / 12.1
 * / 18.8 us): a tile's 12 MMA instructions and its softmax stage, handed from
 * warp role to warp role, take longer than the tile's copy.  A plan made under
 * one setting is valid under the other only if the two give the same
 * workspace size: plan again after changing it. */
kvc_status kvc_set_multi_tc(int on);
kvc_status paged_decode_multi_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                        const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                        int q_len, int B, int Hq, int Hkv, int head_dim, int block_size,
                                        int max_context_len, float scale, void* out, int out_dtype, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Quantized (fp8) KV cache — an extension: the pages quantize weights, not
 * the KV cache, and fix no quantized format.  Values are e4m3 codes (1 sign,
 * 4 exponent bits with bias 7, 3 fraction bits; largest 448), one byte each,
 * with one float scale per (slot, KV head) row: a cached value is
 * code value * scale.  Per-row scales mean that appending a token never
 * re-quantizes the rest of its block.  A layer's fp8 cache is one record of
 * kv_fp8_record_bytes(head_dim) = 32 * D + 128 bytes per (block, KV head),
 * [NB][Hkv][record], so that the decode reads a block with one copy:
 *   bytes [0, 16 D)          K codes: 16 token rows of D codes; code x of row
 *                            r sits at r * D + (((x >> 4) ^ p(r)) << 4) +
 *                            (x & 15), p(r) = (r >> 1) & 3 for D = 64, r & 7
 *                            for D = 128 (the 16-byte chunks of a row are
 *                            permuted so the kernel's fragment loads hit
 *                            distinct shared-memory banks)
 *   bytes [16 D, 16 D + 64)  the 16 K scales (float, token order)
 *   then 16 D bytes          V codes: D dim rows of 16 token codes, token
 *                            tau (0..15) at byte 4 * ((tau & 7) >> 1) +
 *                            2 * (tau >> 3) + (tau & 1) of its row (tokens
 *                            2t, 2t+1, 2t+8, 2t+9 are bytes 4t..4t+3: the
 *                            kernel loads its matrix-multiply fragments with
 *                            one 32-bit read per row)
 *   last 64 bytes            the 16 V scales (float, token order).
 * The bytes per token are 53 % of the fp16 cache's (D = 64). */
kvc_status kv_fp8_record_bytes(int head_dim, size_t* bytes);
/* kv_append_fp8: quantize k_new / v_new (device fp16 [n][Hkv][D]) and write
 * them into the records of their slots: scale = absmax / 448 of the row (IEEE
 * division; 1 for an all-zero row), code = e4m3(x / scale) rounded to nearest
 * even.  Slots as in kv_append (negative = skip, >= NB*bs sets
 * KVC_DEVERR_SLOT).  All device pointers 16-byte aligned. */
kvc_status kv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int n, void* kv_fp8,
                         int num_blocks, int Hkv, int head_dim, int block_size, void* stream);
/* paged_decode_attention over an fp8 cache (kv_fp8: the layer's records):
 * the same result definition with every cached value code value * scale;
 * workspace as paged_decode_plan's.  Codes convert to fp16 exactly; the K
 * scale multiplies the scores in fp32; each probability times its V scale
 * multiplies V as one fp16 value, and the softmax sums add each rounded
 * value times the reciprocal of its scale, so every output row is a convex
 * combination of the dequantized V rows with weights within 2^-11 relative
 * of the exact ones. */
kvc_status paged_decode_attention_fp8(const void* q, const void* kv_fp8, int num_blocks, const int32_t* block_table,
                                      int max_blocks, const int32_t* context_lens, int B, int Hq, int Hkv,
                                      int head_dim, int block_size, int max_context_len, float scale, void* out,
                                      int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split,
                                      void* stream);

/* Launch overlap (process-wide, default off).  When on, decode kernels (and
 * kvc_copy_async's copies) are launched as programmatic dependents of the
 * kernel before them on the stream: they read block tables, context lengths
 * and the cached K/V history before that kernel has finished, and q, k_new,
 * v_new, the workspace and out only after.  A decode kernel releases its own
 * dependents once its dependency wait has passed and its warps have taken
 * their first blocks, so in an unbroken run of decode calls on one stream (no
 * other kernel, copy or event between them; kvc_copy_async calls excepted) a
 * call may start before earlier calls of the run have finished.  Contract: no
 * kernel of that run, nor the kernel launched just before the run, writes a
 * call's block table, context lengths or the cache rows it reads (other than
 * through that call's own append); a kvc_copy_async without KVC_COPY_AHEAD
 * may, since it finishes its copy before anything after it starts.  One call
 * per layer, every layer a different cache, meets this; calls on the same
 * layer need something between them (a copy, an event, another kernel). */
kvc_status kvc_set_launch_overlap(int on);

/* Staging copy (no counterpart in the pages: an interface choice of this
 * library, for steps whose inputs arrive in host memory).  Copies `bytes`
 * from src to dst with a kernel on `stream`.  src and dst may each be device
 * memory or pinned host memory (cudaHostAlloc / cudaHostRegister), which the
 * GPU reads and writes directly over the host link; pageable host memory is
 * refused.  Both 16-byte aligned, bytes a multiple of 16 (0: nothing to do),
 * no overlap.  Being a kernel, the copy chains with the decode kernels under
 * launch overlap with no copy-to-kernel dependency to resolve:
 *   flags 0: the copy starts once the kernel before it on the stream has
 *     finished, and the kernel after it may read the copied bytes at once,
 *     even before its dependency wait (so block tables and context lengths
 *     may be staged this way);
 *   KVC_COPY_AHEAD: the copy starts at once, alongside the kernel before it,
 *     which must neither read nor write src or dst; the call still counts as
 *     finished only once that kernel has.  Later kernels may read the bytes
 *     only after their dependency wait (q, k_new, v_new; not block tables,
 *     context lengths or cache rows).
 * The flags-0 promise (a kernel may read the bytes before its dependency
 * wait) rests on the copy making its writes visible device-wide (a fence and
 * a CTA barrier) before it lets the next kernel launch.  CUDA documents the
 * visibility of a preceding kernel's writes only after the dependency wait,
 * so this ordering is established by test (the host-step test poisons every
 * staged input before each run), not by a documented guarantee.
 * With launch overlap off both forms are plain stream-ordered copies.
 * Errors (synchronous): KVC_ERR_INVALID for null, misaligned, overlapping or
 * pageable buffers and unknown flags; KVC_ERR_CUDA if the launch fails. */
#define KVC_COPY_AHEAD 1u
kvc_status kvc_copy_async(void* dst, const void* src, size_t bytes, unsigned flags, void* stream);

/* Per-CTA timeline of decode launches (builds with -DKVC_TRACE=1 only;
 * otherwise KVC_ERR_UNSUPPORTED).  Each 80-byte record holds eight global-timer
 * stamps in ns (CTA start, first K/V copies issued, dependency wait passed,
 * warp 0's main loop done, all warps done, CTA merge done, cluster merge
 * reached (rank 0: every CTA of the cluster arrived), exit; 0 = not reached),
 * then uint32 launch number, SM id, blockIdx.x and (blockIdx.y << 16 | blockIdx.z).  Copies up to `capacity` records into host
 * memory; `clear` resets the device buffer.  Synchronous. */
kvc_status kvc_trace_read(void* records, int capacity, int* count, int clear);

/* Allocation-free decode.  The pages have no counterpart: this is an
 * interface choice of this library.  Same arguments, preconditions and
 * results as paged_decode_attention, but with no workspace argument: when the
 * longest context needs split scratch, it goes to a fixed 16 MiB array that
 * the library declares in device memory (every GPU that loads the library
 * holds those 16 MiB until the process exits).  It serves callers that must
 * not allocate device memory while they run: allocator or memory-pool code
 * that would re-enter itself, plug-ins that are handed only their input and
 * output buffers, and serving loops that forbid cudaMalloc after start-up.
 * The call itself allocates nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: it does not survive cudaDeviceReset (or any other reset of the
 *    device's primary context), after which this call must not be used.
 *  - All calls on a device share the one array: calls that can overlap on
 *    the GPU (other streams, concurrent graphs) race on it.  Nothing in it
 *    needs to start at zero: every word a call reads, the same call writes first.
 *  - Sizes whose scratch exceeds 16 MiB (see paged_decode_plan) return
 *    KVC_ERR_CAPACITY without launching anything.
 *  - Checked mode does not apply to this call. */
kvc_status paged_decode_attention_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                                                   int num_blocks, const int32_t* block_table, int max_blocks,
                                                   const int32_t* context_lens, int B, int Hq, int Hkv, int head_dim,
                                                   int block_size, int max_context_len, float scale, void* out,
                                                   int out_dtype, int blocks_per_split, void* stream);

/* Varlen packed prefill (xformers article parts 4-5): for every segment s
 * (rows cu_seqlens[s] .. cu_seqlens[s+1]-1) and query head h,
 *   out = softmax(Q K^T * scale + mask) V,
 * K/V of KV head h / (Hq/Hkv) from the same segment only; mask allows j <= i
 * when causal, everything in the segment otherwise.
 *   q device fp16 [total_tokens][Hq][D]; k, v device fp16 [total_tokens][Hkv][D]
 *   cu_seqlens device int32 [nseq+1], cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[nseq] = total_tokens; max_seqlen >= every segment length.
 *   out device [total_tokens][Hq][D], out_dtype KVC_F16 or KVC_F32. */
kvc_status prefill_attention(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                             int nseq, int total_tokens, int max_seqlen, int Hq, int Hkv, int head_dim,
                             float scale, int causal, void* out, int out_dtype, void* stream);

/* Precision of P, the softmax weights that multiply V on the tensor cores in prefill_attention_ex.
 *   KVC_PREFILL_P_F16    P rounded to fp16 (its exponent base is the running row max, so P <= 2^8), and
 *                        the normaliser l sums the rounded weights: every output row is an exact convex
 *                        combination of V rows with weights perturbed by at most 2^-11 relative.  Observed
 *                        error vs an fp64 softmax: ~5e-4 max-abs on unit-variance inputs.  The default.
 *   KVC_PREFILL_P_SPLIT  P = fp16 high part + fp16 residual, both multiplied by V (twice the P V products):
 *                        the weights carry ~22 bits, observed error ~5e-6 max-abs. */
#define KVC_PREFILL_P_F16 0
#define KVC_PREFILL_P_SPLIT 1

/* prefill_attention with a choice of P precision (above); prefill_attention is this call with
 * KVC_PREFILL_P_F16.  KVC_ERR_INVALID for any other p_precision; everything else as prefill_attention. */
kvc_status prefill_attention_ex(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                int nseq, int total_tokens, int max_seqlen, int Hq, int Hkv, int head_dim,
                                float scale, int causal, int p_precision, void* out, int out_dtype, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
