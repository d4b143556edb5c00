// Multi-token decode on the tensor cores (tcgen05), head dim 64 (multi_tc.cu): parameters and launcher, used by
// the multi-token host code in group.cu.
#pragma once
#include "decode_common.cuh"

namespace kvc {
namespace mtc {

constexpr int D = 64;
constexpr int kTileBlocks = 8;   // paged blocks per 128-key tile
constexpr int kMaxRows = 64;     // query rows (q_len x G) of one (sequence, KV head)
constexpr int kMaxChunk = 2048;  // blocks per CTA at most (their ids are in shared memory)

struct Params {
    const __half* q;              // [B][q_len][Hq][D]
    const int32_t* block_table;   // [B][max_blocks]
    const int32_t* context_lens;  // [B], the q_len new tokens included
    void* out;                    // [B][q_len][Hq][D], written here when one cluster covers a context
    float* part_ml;               // otherwise partial states: part `cluster index` of each row, rows part_stride apart
    float* part_acc;
    unsigned* err;
    int B, max_blocks, num_blocks, Hq, Hkv, G, q_len, max_ctx, out_f32;
    int chunk;        // blocks per CTA, a multiple of kTileBlocks
    int cs;           // CTAs per cluster (consecutive blockIdx.x)
    int nclus;        // clusters per (sequence, KV head)
    int part_stride;  // partial rows per query row
    float scale_log2;
};

// whether the tensor-core kernel takes q_len x G query rows per (sequence, KV head) at head dim D
inline bool supported(int D_, int rows) { return D_ == D && rows >= 1 && rows <= kMaxRows; }

// chunking: about one CTA per SM over the B x Hkv (sequence, KV head) units, whole 128-key tiles; the chunks of a
// unit form one cluster where they fit one (at most max_cluster(rows) CTAs), else clusters of that size
void plan(int B, int Hkv, int rows, int max_ctx, int sms, int* chunk, int* cluster, int* nclus);

// grid (nclus * cluster, Hkv, B), clusters of `cluster` CTAs along x
cudaError_t launch(const CUtensorMap& tmK, const CUtensorMap& tmV, const Params& p, int rows, bool pdl,
                   cudaStream_t stream);

}  // namespace mtc
}  // namespace kvc
