// The cascade's shared-prefix pass on the tensor cores (tcgen05), head dim 64 (group_tc.cu): parameters and
// launcher, used by the cascade host code in group.cu.
#pragma once
#include "decode_common.cuh"

namespace kvc {
namespace gtc {

constexpr int D = 64;
constexpr int kMaxChunk = 2048;  // blocks per CTA at most (their ids are in shared memory)
constexpr int kChunkAlign = 8;   // chunks are whole 128-key tiles

struct Params {
    const __half* q;              // [B][Hq][D]
    const int32_t* block_table;   // [B][max_blocks]
    const int32_t* group_start;   // [n_groups + 1]: group g is sequences group_start[g] .. group_start[g+1]-1
    const int32_t* blk_off;       // [B] shared blocks of each sequence's group
    float* part_ml;               // partial states: part `chunk` of each row, rows part_stride apart
    float* part_acc;
    unsigned* err;
    int max_blocks, num_blocks, Hq, Hkv, G;
    int chunk;        // shared blocks per CTA (a multiple of 8)
    int nchunks;      // chunks per group (grid.x)
    int part_stride;  // partial rows per query row
    float scale_log2;
};

// grid (nchunks, Hkv, n_groups); every CTA writes the partial states of its chunk (part `chunk` of each of its
// group's rows), which the combine kernel merges with the suffix parts
cudaError_t launch(const CUtensorMap& tmK, const CUtensorMap& tmV, const Params& p, dim3 grid, bool pdl,
                   cudaStream_t stream);

}  // namespace gtc
}  // namespace kvc
