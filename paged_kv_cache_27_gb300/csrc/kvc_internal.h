// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvc {

constexpr int kBlockSize = 16;  // tokens per block (the page size used throughout the pages)
// query heads per KV head the decode paths take (the decode kernel in chunks of 8 heads per CTA)
constexpr int kMaxGroupHeads = 64;

// Device address of the sticky error word of the current device.
cudaError_t device_error_word(unsigned** ptr);

// ---- append / block copy (append.cu) ---------------------------------------
cudaError_t launch_append(const __half* k_new, const __half* v_new, const int64_t* slots, int n, __half* k_layer,
                          __half* v_layer, int num_blocks, int Hkv, int D, unsigned* err, cudaStream_t stream);
// quantizing append: e4m3 codes [NB][Hkv][16][D] and one float scale per (slot, KV head) row
// fp8 V code pool: per (block, KV head), D rows (one per dim) of 16 token codes; token tau (0..15) sits at byte
// vt_pos(tau) of its row, so that the mma.sync fragment of lane t (tokens 2t, 2t+1, 2t+8, 2t+9) is the 4 bytes at 4t
__host__ __device__ constexpr int vt_pos(int tau) { return 4 * ((tau & 7) >> 1) + 2 * (tau >> 3) + (tau & 1); }
// fp8 cache record of one (block, KV head): K codes (16 x D bytes), K scales (16 floats), V codes (D x 16
// bytes), V scales (16 floats)
__host__ __device__ constexpr int fp8_record_bytes(int D) { return 2 * (kBlockSize * D + kBlockSize * 4); }
// byte offset of K code x of token row r inside a record: the row's 16-byte chunks are permuted (by (r >> 1) & 3
// at D = 64, r & 7 at D = 128) so that the decode kernel's fragment loads of 8 rows x 4 lanes hit 32 banks
__host__ __device__ constexpr int fp8_kswz(int D, int r, int x) {
    return r * D + ((((x >> 4) ^ (D == 64 ? ((r >> 1) & 3) : (r & 7))) << 4) | (x & 15));
}
cudaError_t launch_append_fp8(const __half* k_new, const __half* v_new, const int64_t* slots, int n,
                              uint8_t* kv_fp8, int num_blocks, int Hkv, int D, unsigned* err, cudaStream_t stream);
// copies whole blocks src[i] -> dst[i] for every layer (pools [L][NB][block_elems])
cudaError_t launch_copy_blocks(const int32_t* src, const int32_t* dst, int n, __half* k_pool, __half* v_pool,
                               int L, int num_blocks, int64_t block_elems, cudaStream_t stream);

// ---- decode (decode.cu) ------------------------------------------------------
struct DecodePlan {
    int num_splits;        // grid.x = num_parts * cluster
    int blocks_per_split;  // blocks of 16 tokens one cluster covers
    int cluster;           // CTAs per thread-block cluster (they share the cluster's blocks)
    int num_parts;         // clusters along the longest context; > 1 needs the workspace + combine kernel
    size_t workspace_bytes;
};
cudaError_t decode_plan(int B, int Hq, int Hkv, int D, int max_context_len, int blocks_per_split,
                        DecodePlan* plan);
struct DecodeArgs {
    const __half* q;
    const __half* k_new;  // null: attention only; else the step's new K/V rows [B][Hkv][D]
    const __half* v_new;
    const __half* k_cache;
    const __half* v_cache;
    int num_blocks;
    const int32_t* block_table;
    int max_blocks;
    const int32_t* context_lens;
    int B, Hq, Hkv, D;
    int max_context_len;
    float scale;
    void* out;
    int out_f32;
    void* workspace;
    size_t workspace_bytes;
    int blocks_per_split;  // blocks per cluster, 0 = automatic
    unsigned* err;
    // fp8 cache instead of k_cache / v_cache when set: one record per (block, KV head), [NB][Hkv][record]
    const uint8_t* kv_fp8 = nullptr;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Partial states of query rows (m, l, acc) merged into the output by the combine kernel (decode.cu).
struct CombineParams {
    const float* part_ml;
    const float* part_acc;
    const int32_t* context_lens;
    const int32_t* blk_off;  // null, or per sequence: blocks of its row covered by the prefix parts
    void* out;
    unsigned* err;
    int Hq, part_stride, part_base, bpc, max_blocks, max_ctx, out_f32;
    int prefix_chunk;  // blocks per prefix part (cascade), 0 = no prefix parts
    int cascade;       // 1: only partials were written; this kernel writes every output row
    int q_len;         // query rows per sequence (multi-token decode; 1 otherwise): row y is sequence y / q_len
    int early_release; // 1: the next kernel may launch as soon as this one starts (see the combine kernel)
};
// grid (Hq, rows): one CTA per (query head, query row)
cudaError_t launch_combine(const CombineParams& c, int D, int rows, cudaStream_t stream);
// the decode kernel over every sequence past its first blk_off[b] blocks, partial states only (cascade suffix)
cudaError_t launch_decode_suffix(const DecodeArgs& a, const DecodePlan& plan, const int32_t* blk_off, int part_base,
                                 int part_stride, float* part_ml, float* part_acc, cudaStream_t stream);

// Cascade decode: groups of at most 8 consecutive sequences whose block-table rows begin with the same
// shared blocks. The group kernel (group.cu) reads those blocks once per group for all its sequences; the
// decode kernel covers each sequence's remaining blocks; the combine kernel merges both.
constexpr int kMaxGroupSize = 8;
struct CascadePlan {
    DecodePlan suffix;  // the decode kernel over every sequence's blocks past its shared prefix
    int chunk;          // shared blocks per prefix CTA
    int cluster;        // prefix CTAs per cluster (one prefix part per cluster)
    int nchunks;        // prefix parts per (sequence, head): clusters over the longest shared prefix
    int part_stride;    // partial rows per (sequence, head): nchunks + suffix.num_parts
    bool plain;         // shared prefixes too short to pay for the extra launches: run the plain decode
    size_t workspace_bytes;
};
cudaError_t cascade_plan(int B, int Hq, int Hkv, int D, int max_context_len, int n_groups, int max_shared_blocks,
                         CascadePlan* plan);
// process-wide: cascade calls saving fewer block reads per KV head than this run the plain decode
void set_cascade_min_saved_blocks(int blocks);
// process-wide: multi-token calls at head dim 64 on the tensor-core kernel (multi_tc.cu) instead of mma.sync
void set_multi_tc(int on);
// group_start: device [n_groups + 1]; shared_blocks: device [B], the shared blocks of each sequence's group
cudaError_t launch_cascade(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                           int n_groups, int max_shared_blocks, cudaStream_t stream);

// Multi-token decode (group.cu): q_len (1..8) new tokens per sequence, causal among them (token t at
// position ctx - q_len + t); q and out are [B][q_len][Hq][D]. A CTA's warps split a chunk of a sequence's
// blocks and each carries all the tokens' query rows of its KV head, so every block is read once for all
// tokens; the CTAs of a cluster merge in distributed shared memory, and the combine kernel merges the
// clusters where a context needs more than one.
constexpr int kMaxQueryTokens = 8;
struct MultiPlan {
    int chunk;    // blocks per CTA
    int cluster;  // CTAs per cluster
    int nclus;    // clusters per context (of the longest); > 1: partial states and the combine kernel
    int stages;   // blocks in flight per warp
    size_t workspace_bytes;
};
cudaError_t multi_plan(int B, int Hq, int Hkv, int D, int max_context_len, int q_len, MultiPlan* plan);
cudaError_t launch_multi(const DecodeArgs& a, int q_len, cudaStream_t stream);
// process-wide: launch decode kernels as programmatic dependents of the previous kernel
void set_launch_overlap(int on);
// copies up to `cap` trace records (80 bytes each) of the decode kernel; cudaErrorNotSupported
// unless the library was built with -DKVC_TRACE=1
cudaError_t trace_read(void* host, int cap, int* n, int clear);
int launch_overlap();

// Records `msg` as the calling thread's last error (kvc_last_error_string) and returns `status`.
int set_last_error(int status, const char* msg);

// ---- prefill (prefill.cu) ----------------------------------------------------
struct PrefillArgs {
    const __half* q;
    const __half* k;
    const __half* v;
    const int32_t* cu_seqlens;
    int nseq, total_tokens, max_seqlen;
    int Hq, Hkv, D;
    float scale;
    int causal;
    void* out;
    int out_f32;
    int split_p;  // P as fp16 high part + fp16 residual (else one fp16 value)
    unsigned* err;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// head dim 64: one 128-row query tile per CTA, S double-buffered in TMEM (prefill_1t.cu)
cudaError_t launch_prefill_1t(const PrefillArgs& a, cudaStream_t stream);

}  // namespace kvc
