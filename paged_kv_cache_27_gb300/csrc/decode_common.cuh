// Pieces shared by the decode-side translation units (decode.cu: the decode and combine kernels;
// group.cu: the kernel for query groups that share their key blocks): build knobs, the per-head-dim tile
// configuration, the shared-memory swizzle of a K/V tile, output stores, and host launch helpers.
#pragma once
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

// ---- build knobs (defaults are the measured best on GB300) ---------------------------------------
#ifndef KVC_DEC_WARPS64
#define KVC_DEC_WARPS64 8
#endif
#ifndef KVC_DEC_STAGES64
#define KVC_DEC_STAGES64 2
#endif
// fp8 cache: 1 = the P V products take each weight times its V scale as one fp16 operand, and the row sums add
// each rounded weight times the reciprocal of its scale (so every output row stays a convex combination of the
// dequantized V rows, weights within 2^-11 relative); 0 = an fp16 high part plus residual, two products per tile.
// Measured (two A/B pairs, one call with L2 flushed): B = 16 x 65536 67.6 -> 65.5 us, B = 4 x 131072 41.0 ->
// 38.9-39.6 us; the 24-layer 32 x 2048 graph unchanged (6.61 -> 6.59 us per layer).
#ifndef KVC_DEC_FP8_ONE_P
#define KVC_DEC_FP8_ONE_P 1
#endif
#ifndef KVC_DEC_STAGES64_FP8  // stages per warp with an fp8 cache (a stage is half the bytes)
#define KVC_DEC_STAGES64_FP8 2
#endif
#ifndef KVC_DEC_STAGES128_FP8
#define KVC_DEC_STAGES128_FP8 2
#endif
#ifndef KVC_DEC_WARPS128
#define KVC_DEC_WARPS128 4
#endif
#ifndef KVC_DEC_STAGES128
#define KVC_DEC_STAGES128 2
#endif
#ifndef KVC_DEC_MAX_CLUSTER
#define KVC_DEC_MAX_CLUSTER 8
#endif
// Where a decode kernel lets the next kernel on the stream launch (programmatic dependent launch): 0 at its
// start, 1 after its own dependency wait, 2 when a warp refills its first stage (its first block is consumed),
// 3 when a warp has issued its last copy, 4 after the block loop, 5 after the CTA merge, 6 not at all (at exit).
// A 24-layer decode step (32 x 2048) measured 4388 / 4410 / 4555 / 4545 / 4472 / 4317 / 3932 GB/s: a trigger
// before the dependency wait lets every queued layer launch at once (their CTAs hold SM slots while they wait);
// one well after the first block leaves the next layer's first copies too late.
#ifndef KVC_DEC_TRIGGER
#define KVC_DEC_TRIGGER 2
#endif
#ifndef KVC_COMBINE_EARLY_TRIGGER  // the split combine kernel lets the next kernel launch as soon as it starts
#define KVC_COMBINE_EARLY_TRIGGER 1
#endif
// 1: the split combine merges the parts in one pass with online rescaling (one round trip to the partials);
// 0: the maximum over every part first, then the weighted sums (two).  Per layer of a 24-layer graph, two A/B
// pairs: B = 1 x 16384 6.50 -> 6.16 us, B = 4 x 16384 10.1 -> 9.6, B = 1 x 131072 16.6 -> 16.4, B = 4 x 65536
// 26.2 -> 25.7.
#ifndef KVC_COMBINE_ONE_PASS
#define KVC_COMBINE_ONE_PASS 1
#endif
#ifndef KVC_COMBINE_EARLY_ALWAYS  // 1: the combine releases the next launch at its start whatever the grid's size
#define KVC_COMBINE_EARLY_ALWAYS 0
#endif
#ifndef KVC_GROUP_EARLY_TRIGGER  // the group kernel lets the next kernel launch as soon as it starts
#define KVC_GROUP_EARLY_TRIGGER 1
#endif
#ifndef KVC_DEC_EARLY_REFILL  // 1: refill a stage once its K and V are in registers, before the softmax
#define KVC_DEC_EARLY_REFILL 1
#endif
#ifndef KVC_DEC_MIN_CTAS  // resident CTAs per SM the register allocation must allow
#define KVC_DEC_MIN_CTAS 1
#endif
#ifndef KVC_DEC_PLAN_CTAS  // CTAs per SM one launch is sized for; the rest lets the next launch start early
#define KVC_DEC_PLAN_CTAS 2
#endif
// Fewest blocks per warp the split planner aims for: with two stages per warp, four blocks are two copy round
// trips.  Below KVC_DEC_SMALL_BYTES of K/V per call a plan that needs the combine launch keeps to half the
// resident clusters, so that the combine can release the next launch (the next layer) at its start and the two
// run side by side; above it the halved copy rate costs more than the overlap gains.  Measured per layer of a
// 24-layer graph (L2 flushed per replay), against plans that filled the GPU with one or two blocks per warp:
// B = 1 x 4096 5.5 -> 4.7 us, B = 4 x 4096 8.3 -> 5.0, B = 1 x 16384 8.9 -> 7.0-7.2, B = 1 x 65536 12.3 -> 11.1,
// B = 4 x 16384 11.8 -> 11.2; at 64 MiB and above the full wave stays ahead (B = 4 x 65536 26.5 us against 28.5
// on half of it).  The 32 x 2048 step keeps its four blocks per warp in one cluster per (sequence, KV head).
#ifndef KVC_DEC_MIN_BLOCKS_PER_WARP
#define KVC_DEC_MIN_BLOCKS_PER_WARP 4
#endif
#ifndef KVC_DEC_SMALL_BYTES
#define KVC_DEC_SMALL_BYTES (int64_t(64) << 20)
#endif
// Largest cluster of a plan with several clusters per (sequence, KV head) (the combine merges their parts).
// Measured against 8 (two A/B pairs; one call with L2 flushed / per layer of a 24-layer graph): B = 1 x 16384
// 13.4 -> 12.3 / 6.93 -> 6.64 us, B = 1 x 131072 22.0 -> 20.7 / 17.2 -> 16.7, B = 4 x 16384 18.4 -> 16.5 /
// 10.8 -> 9.9, B = 4 x 131072 55.9 -> 53.3 / 46.0 -> 45.2; plans of one cluster per unit keep clusters of 8.
#ifndef KVC_DEC_SPLIT_MAX_CLUSTER
#define KVC_DEC_SPLIT_MAX_CLUSTER 4
#endif
// 1: the CTAs of a cluster hand their merged states to rank 0 with st.async, whose bytes complete on an mbarrier
// in rank 0 (senders leave at once); 0: remote stores, then a cluster barrier (release / acquire)
#ifndef KVC_DEC_ASYNC_PUSH
#define KVC_DEC_ASYNC_PUSH 1
#endif
// 1: the decode kernel waits for its cluster's prologue phase right after its dependency wait; 0: just before
// its first push into rank 0's inbox
#ifndef KVC_DEC_EARLY_CLUSTER_WAIT
#define KVC_DEC_EARLY_CLUSTER_WAIT 1
#endif
// Lazy running maximum in the decode kernel's online softmax: a block's scores are weighted against the running
// maximum m as they are, 2^(x - m) <= 2^KVC_DEC_LAZY_MAX, unless one of them exceeds m by more than that; only
// then is the block's maximum reduced across the lanes and the state rescaled.  0: every block moves the maximum.
#ifndef KVC_DEC_LAZY_MAX
#define KVC_DEC_LAZY_MAX 8
#endif

// Plans of several waves (more CTAs than can be resident): the CTAs at position z along the sequences take the
// z-th longest context, so that the long contexts start in the first wave and the short ones fill the tail
// (longest-processing-time-first list scheduling; CTAs are dispatched in the order of their linear index).
// B = 200 sequences of 16..4096 tokens, 14 q / 2 KV heads: 41.5 -> 36.9 us per call with the batch itself
// sorted.  0: sequence z.
#ifndef KVC_DEC_LEN_ORDER
#define KVC_DEC_LEN_ORDER 1
#endif
constexpr int kLenOrderMaxB = 1024;  // batches up to this size (the order costs two warp passes over B lengths)

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCluster = KVC_DEC_MAX_CLUSTER;
// blocks one cluster covers at most: its slice of the block table sits in shared memory (16 KiB at 4096 blocks,
// which keeps two 8-warp CTAs per SM)
constexpr int kMaxClusterBlocks = 4096;

// Tile configuration per head dim. With kFp8 the cache holds one record per (block, KV head) (fp8_record_bytes):
// the block's K codes (16 token rows of D bytes, each row's 16-byte chunks permuted by fp8_kswz), its 16 K
// scales, its V codes (D dim rows of 16 token bytes in the order vt_pos gives) and its 16 V scales.  A stage is
// one record, brought in by one bulk copy; the codes go from shared memory straight into the mma.sync fragments
// (one 32-bit load per fragment row).
template <int D, bool kFp8 = false>
struct DecodeCfg {
    static constexpr int kWarps = D == 64 ? KVC_DEC_WARPS64 : KVC_DEC_WARPS128;
    static constexpr int kStages = kFp8 ? (D == 64 ? KVC_DEC_STAGES64_FP8 : KVC_DEC_STAGES128_FP8)
                                        : (D == 64 ? KVC_DEC_STAGES64 : KVC_DEC_STAGES128);
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kTileBytes = kBlockSize * D * 2;    // one 16 x D fp16 tile
    static constexpr int kCodeTileBytes = kBlockSize * D;    // one 16 x D e4m3 tile
    static constexpr int kScaleBytes = kBlockSize * 4;       // 16 float scales
    static constexpr int kStageBytes = kFp8 ? fp8_record_bytes(D)  // one record: K codes, K scales, V codes, V scales
                                            : 2 * kTileBytes;     // K tile + V tile
    // a warp's ring starts on a 1024-byte boundary (the fp16 tiles' TMA swizzle repeats every 1024 bytes)
    static constexpr int kWarpRingBytes = (kStages * kStageBytes + 1023) / 1024 * 1024;
    static constexpr int kRingBytes = kWarps * kWarpRingBytes;
    // the warps' stage barriers, then rank 0's inbox barrier (padded to keep what follows 16-byte aligned)
    static constexpr int kBarBytes = kWarps * kStages * 8 + 16;
    static constexpr int kStateBytes = 8 * (D + 2) * 4;  // merged (m[8], l[8], acc[8][D]) of this CTA
    // + the inbox of cluster rank 0 (one slot per other CTA of the cluster) and the cluster's slice of the block
    // table (bpc entries), both sized at launch, + alignment slack
    static constexpr int kBaseSmemBytes = kRingBytes + kBarBytes + kStateBytes + 1024;
    static int smem_bytes(int cluster, int G, int bpc) {
        return kBaseSmemBytes + (cluster - 1) * (16 + G * D) * 4 + (bpc * 4 + 15) / 16 * 16;
    }
    static constexpr int kMergeStride = D + 4;  // floats per parked row
    static_assert(16 * 4 + 8 * kMergeStride * 4 <= kWarpRingBytes, "warp state must fit a warp ring");
};

// byte offset of 16-byte chunk `chunk` (8 fp16 columns) of row `row` inside a tile loaded as boxes of 16
// rows x 64 columns with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(((chunk >> 3) << 11) + (row << 7) + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void store_out(void* out, int out_f32, int64_t idx, float v) {
    if (out_f32)
        static_cast<float*>(out)[idx] = v;
    else
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
}
// four consecutive outputs starting at idx (a multiple of 4)
__device__ __forceinline__ void store_out4(void* out, int out_f32, int64_t idx, float4 v) {
    if (out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
    } else {
        uint2 h;
        h.x = pack_half2(v.x, v.y);
        h.y = pack_half2(v.z, v.w);
        *reinterpret_cast<uint2*>(static_cast<__half*>(out) + idx) = h;
    }
}
__device__ __forceinline__ float4 fma4(float w, float4 a, float4 acc) {
    return make_float4(fmaf(w, a.x, acc.x), fmaf(w, a.y, acc.y), fmaf(w, a.z, acc.z), fmaf(w, a.w, acc.w));
}
__device__ __forceinline__ float4 scale4(float4 a, float s) { return make_float4(a.x * s, a.y * s, a.z * s, a.w * s); }

// The sequence at position z (0 <= z < B <= kLenOrderMaxB) of the order "longer length class first, then lower
// index", over 32 classes of about max_ctx / 32 tokens (longest: class 31).  Every thread of the CTA calls it
// (it holds two CTA barriers); the answer depends on the lengths alone, so every CTA computes the same order and
// z -> sequence is a permutation of [0, B) whatever the lengths hold (out-of-range lengths are clamped into a
// class; the kernel reports them as before).  Shared scratch: hist 32 ints, cls B bytes, one int for the answer.
__device__ inline int seq_by_length(const int32_t* __restrict__ lens, int B, int max_ctx, int z, int* hist,
                                    uint8_t* cls, int* answer) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    // class = floor(len * 32 / (max_ctx + 1)) in float: monotone in len and the same in every CTA
    const float per_token = 32.f / (static_cast<float>(max_ctx) + 1.f);
    if (threadIdx.x < 32) hist[threadIdx.x] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < B; j += blockDim.x) {
        const int len = min(max(lens[j], 0), max_ctx);
        const int c = min(31, static_cast<int>(static_cast<float>(len) * per_token));
        cls[j] = static_cast<uint8_t>(c);
        atomicAdd(&hist[c], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // lane i counts class 31 - i: the inclusive scan over the lanes ends at each class's last position + 1
        const int c = hist[31 - lane];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned hit = __ballot_sync(full, z >= incl - c && z < incl);
        int seq = min(max(z, 0), B - 1);  // z outside [0, B): not a launch this kernel makes
        if (hit != 0) {
            const int src = __ffs(hit) - 1;
            const int want = 31 - src;
            int r = z - __shfl_sync(full, incl - c, src);  // rank within the class, by index
            for (int j0 = 0; j0 < B; j0 += 32) {
                const int j = j0 + lane;
                unsigned m = __ballot_sync(full, j < B && cls[j] == want);
                const int n = __popc(m);
                if (r < n) {
                    for (int k = 0; k < r; ++k) m &= m - 1;
                    seq = j0 + __ffs(m) - 1;
                    break;
                }
                r -= n;
            }
        }
        if (lane == 0) *answer = seq;
    }
    __syncthreads();
    return *answer;
}

// ---- host helpers ------------------------------------------------------------------------------------
inline int sm_count() {
    static std::atomic<int> cached[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128 && cached[dev].load()) return cached[dev].load();
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128) cached[dev].store(n);
    return n;
}

// partial rows in a workspace: (m, l) pairs padded to a multiple of 4 floats, then the acc rows (16-byte aligned)
inline size_t partials_bytes(size_t nrow, int D) {
    return (((nrow * 2 + 3) & ~static_cast<size_t>(3)) + nrow * D) * sizeof(float);
}
inline float* partials_acc(float* part_ml, size_t nrow) {
    return part_ml + ((nrow * 2 + 3) & ~static_cast<size_t>(3));
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D view of one layer's pool: rows of D fp16 (a (block, KV head, offset) row each),
// boxes of 16 rows x 64 columns, 128-byte swizzle.
inline cudaError_t make_tile_map(CUtensorMap* map, const void* base, int D, int64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


template <typename Kern, typename... Args>
inline cudaError_t launch(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace kvc
