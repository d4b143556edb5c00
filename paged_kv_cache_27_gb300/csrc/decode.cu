// Paged grouped-query decode attention for sm_103a.
//
// What it computes ("La caché de claves y valores", gustavoai.dev, section
// "Las claves y los valores de una posición no cambian"): for each sequence
// b and query head h, the unmasked row
//     out[b][h] = softmax(q[b][h] . K_b^T * scale) V_b
// over the context_lens[b] cached tokens (the token appended in this step
// included).  K_b, V_b are found through the sequence's block table
// (PagedAttention, chatgpz.de SECTION 2 and neuralialabs.com); query head h
// reads KV head h / G, G = Hq / Hkv (xformers article part 5, BMGHK).
//
// Design (GB300):
//  * one CTA per (context split, KV head, sequence); the G <= 8 query heads of
//    a KV head are the rows of one m16n8k16 tile, so every K/V tile fetched
//    from HBM is used by the whole group;
//  * each warp owns a private ring of kStages stages; one lane issues the two
//    TMA tile loads (K and V, 16 tokens x D fp16 each, 128-byte swizzled so the
//    ldmatrix reads below are bank-conflict free) and the warp waits on the
//    stage's mbarrier (bounded wait, error flag on expiry);
//  * S = Q K^T and O += P V on the tensor cores (mma.sync, fp16 in, fp32
//    accumulate); P is split into an fp16 high part and an fp16 residual so the
//    P V product keeps ~fp32 accuracy;
//  * online softmax in fp32, base 2 (scale * log2 e folded into the scores),
//    row max by quad shuffles;
//  * warps of a CTA merge through shared memory, splits of a sequence through
//    a workspace and a small combine kernel, both with the rescaling rule of
//    the FlashAttention article ("Was ist der mathematische Aspekt von
//    Softmax?"): partial (m, l, acc) are rescaled by 2^(m - M), M the global max.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

constexpr int kWarps = 4;   // warps per CTA
constexpr int kStages = 4;  // ring stages per warp
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecodeGeom {
    static constexpr int kTileBytes = kBlockSize * D * 2;  // one 16 x D fp16 tile
    static constexpr int kStageBytes = 2 * kTileBytes;     // K tile + V tile
    static constexpr int kWarpRingBytes = kStages * kStageBytes;
    static constexpr int kRingBytes = kWarps * kWarpRingBytes;
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static constexpr int kSmemBytes = kRingBytes + kBarBytes + 1024;  // + alignment slack
    static constexpr int kMergeStride = D + 4;                        // floats per merged row
    static_assert(8 * 2 * 4 + 8 * kMergeStride * 4 <= kWarpRingBytes, "merge area must fit a warp ring");
};

struct DecodeKernelParams {
    const __half* q;
    const int32_t* block_table;
    const int32_t* context_lens;
    void* out;
    float* part_ml;   // [B][Hq][nsplit][2] (m, l) in base-2 units
    float* part_acc;  // [B][Hq][nsplit][D]
    unsigned* err;
    int max_blocks, num_blocks, B, Hq, Hkv, G, max_ctx, bps, nsplit, out_f32;
    float scale_log2;
};

// byte offset of 16-byte chunk `chunk` (8 fp16 columns) of row `row` inside a
// tile loaded as boxes of 16 rows x 64 columns with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(((chunk >> 3) << 11) + (row << 7) + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void store_out(const DecodeKernelParams& p, int64_t idx, float v) {
    if (p.out_f32)
        static_cast<float*>(p.out)[idx] = v;
    else
        static_cast<__half*>(p.out)[idx] = __float2half_rn(v);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   const DecodeKernelParams p) {
    using Geo = DecodeGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kRingBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

    const int ctx = p.context_lens[b];
    if (ctx < 1 || ctx > p.max_blocks * kBlockSize || ctx > p.max_ctx) {
        if (split == 0) {
            if (threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            for (int e = threadIdx.x; e < p.G * D; e += blockDim.x)
                store_out<D>(p, (static_cast<int64_t>(b) * p.Hq + kvh * p.G + e / D) * D + e % D, 0.f);
        }
        return;
    }
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    const int nsplit = (nblk + p.bps - 1) / p.bps;
    if (split >= nsplit) return;
    const int j0 = split * p.bps;
    const int nb_split = min(j0 + p.bps, nblk) - j0;
    const int nb_w = warp < nb_split ? (nb_split - warp + kWarps - 1) / kWarps : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kStages; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();

    uint64_t* wbars = bars + warp * kStages;
    uint8_t* wring = smem + warp * Geo::kWarpRingBytes;
    const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks;

    // lane 0: issue the K and V tiles of this warp's i-th block into stage i % kStages
    auto issue = [&](int i) {
        const int jj = j0 + warp + i * kWarps;
        const int phys = table[jj];
        uint64_t* bar = &wbars[i % kStages];
        if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, KVC_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // complete the phase without data; the block is skipped
            return;
        }
        const uint64_t policy = l2_policy_evict_first();
        uint8_t* st = wring + (i % kStages) * Geo::kStageBytes;
        mbar_arrive_expect_tx(bar, Geo::kStageBytes);
        const int y = (phys * p.Hkv + kvh) * kBlockSize;
#pragma unroll
        for (int x = 0; x < D; x += 64) {
            tma_load_2d(st + (x / 64) * 2048, &tmK, bar, x, y, policy);
            tma_load_2d(st + Geo::kTileBytes + (x / 64) * 2048, &tmV, bar, x, y, policy);
        }
    };
    if (lane == 0) {
        const int n0 = min(nb_w, kStages);
        for (int i = 0; i < n0; ++i) issue(i);
    }

    // query fragments (A operand, rows = the G heads of this KV head; rows >= G are zero)
    uint32_t qa[D / 16][2];
    {
        const bool row_ok = g < p.G;
        const __half* qrow = p.q + (static_cast<int64_t>(b) * p.Hq + kvh * p.G + (row_ok ? g : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * t4) : 0u;
            qa[ks][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * t4) : 0u;
        }
    }

    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const float sl2 = p.scale_log2;

    int i = 0;
    bool timed_out = false;
    for (; i < nb_w; ++i) {
        const int stage = i % kStages;
        const uint32_t parity = (i / kStages) & 1;
        const int jj = j0 + warp + i * kWarps;
        const int phys = table[jj];
        const bool ok = mbar_wait_bounded(&wbars[stage], parity, kWaitLimitNs);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        if (phys >= 0 && phys < p.num_blocks) {
            const uint32_t kbase = smem_u32(wring + stage * Geo::kStageBytes);
            const uint32_t vbase = kbase + Geo::kTileBytes;
            // ---- S = Q K^T for the 16 tokens of this block (two n-tiles of 8) ----
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kc = 0; kc < D / 32; ++kc) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + swz(nt * 8 + (lane & 7), kc * 4 + (lane >> 3)), b0, b1, b2, b3);
                    mma_f16_16816(sc[nt], qa[2 * kc][0], 0u, qa[2 * kc][1], 0u, b0, b1);
                    mma_f16_16816(sc[nt], qa[2 * kc + 1][0], 0u, qa[2 * kc + 1][1], 0u, b2, b3);
                }
            }
            // ---- online softmax (row g; columns 2*t4, 2*t4+1 of each n-tile) ----
            const int rem = ctx - jj * kBlockSize;  // valid tokens in this block (>= 1)
            float x[2][2];
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = nt * 8 + 2 * t4 + e;
                    x[nt][e] = tok < rem ? sc[nt][e] * sl2 : -INFINITY;
                    mx = fmaxf(mx, x[nt][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = ex2(m_run - m_new);
            m_run = m_new;
            uint32_t phi[2], plo[2];
            float ps = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float p0 = ex2(x[nt][0] - m_new), p1 = ex2(x[nt][1] - m_new);
                ps += p0 + p1;
                phi[nt] = pack_half2(p0, p1);
                const float2 h = unpack_half2(phi[nt]);
                plo[nt] = pack_half2(p0 - h.x, p1 - h.y);
            }
            l_run = l_run * alpha + ps;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                o[nd][0] *= alpha;
                o[nd][1] *= alpha;
            }
            // rows of V past the context may hold any bits (even NaN): zero them in registers
            uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
            if (rem < kBlockSize) {
                keep0 = (2 * t4 < rem ? 0x0000ffffu : 0u) | (2 * t4 + 1 < rem ? 0xffff0000u : 0u);
                keep1 = (8 + 2 * t4 < rem ? 0x0000ffffu : 0u) | (9 + 2 * t4 < rem ? 0xffff0000u : 0u);
            }
            // ---- O += P V (P = hi + lo) ----
#pragma unroll
            for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                const int mi = lane >> 3;
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vbase + swz((mi & 1) * 8 + (lane & 7), nd2 * 2 + (mi >> 1)), v0, v1, v2, v3);
                v0 &= keep0;
                v2 &= keep0;
                v1 &= keep1;
                v3 &= keep1;
                mma_f16_16816(o[2 * nd2], phi[0], 0u, phi[1], 0u, v0, v1);
                mma_f16_16816(o[2 * nd2], plo[0], 0u, plo[1], 0u, v0, v1);
                mma_f16_16816(o[2 * nd2 + 1], phi[0], 0u, phi[1], 0u, v2, v3);
                mma_f16_16816(o[2 * nd2 + 1], plo[0], 0u, plo[1], 0u, v2, v3);
            }
        }
        __syncwarp();
        if (lane == 0 && i + kStages < nb_w) issue(i + kStages);
    }
    if (timed_out) {
        if (lane == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        // let copies still in flight land before the shared memory is reused
        for (int k = i; k < min(nb_w, i + kStages); ++k)
            mbar_wait_bounded(&wbars[k % kStages], (k / kStages) & 1, kWaitLimitNs / 8);
        m_run = -INFINITY;
        l_run = 0.f;
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

    // ---- merge the warps of this CTA (each warp parks its state in its own ring) ----
    __syncwarp();
    float* wm = reinterpret_cast<float*>(wring);  // [8] m, [8] l, then [8][D+4] acc
    if (t4 == 0) {
        wm[g] = m_run;
        wm[8 + g] = l_run;
    }
    float* wo = wm + 16;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd)
        *reinterpret_cast<float2*>(wo + g * Geo::kMergeStride + nd * 8 + 2 * t4) = make_float2(o[nd][0], o[nd][1]);
    __syncthreads();

    const bool direct = nsplit == 1;
    for (int e = threadIdx.x; e < p.G * D; e += blockDim.x) {
        const int gg = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * Geo::kWarpRingBytes)[gg]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float* r = reinterpret_cast<const float*>(smem + w * Geo::kWarpRingBytes);
            const float wgt = ex2(r[gg] - M);  // an empty warp has m = -inf -> weight 0
            L += r[8 + gg] * wgt;
            O += r[16 + gg * Geo::kMergeStride + d] * wgt;
        }
        const int h = kvh * p.G + gg;
        if (direct) {
            store_out<D>(p, (static_cast<int64_t>(b) * p.Hq + h) * D + d, L > 0.f ? O / L : 0.f);
        } else {
            const int64_t row = (static_cast<int64_t>(b) * p.Hq + h) * p.nsplit + split;
            if (d == 0) {
                p.part_ml[row * 2 + 0] = M;
                p.part_ml[row * 2 + 1] = L;
            }
            p.part_acc[row * D + d] = O;
        }
    }
}

// Merge the split partials of every (sequence, query head): 8 groups of 32
// lanes walk the splits with a running (M, L, acc), then the groups merge.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_combine_kernel(const float* __restrict__ part_ml,
                                                                    const float* __restrict__ part_acc,
                                                                    const int32_t* __restrict__ context_lens,
                                                                    void* out, int Hq, int nsplit_grid, int bps,
                                                                    int max_blocks, int max_ctx, int out_f32) {
    constexpr int V = D / 32;  // dims per lane
    __shared__ float sM[8], sL[8], sO[8][D];
    const int h = blockIdx.x, b = blockIdx.y;
    const int grp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ctx = context_lens[b];
    if (ctx < 1 || ctx > max_blocks * kBlockSize || ctx > max_ctx) return;
    const int nsplit = ((ctx + kBlockSize - 1) / kBlockSize + bps - 1) / bps;
    if (nsplit <= 1) return;
    const int64_t row0 = (static_cast<int64_t>(b) * Hq + h) * nsplit_grid;
    float M = -INFINITY, L = 0.f, O[V];
#pragma unroll
    for (int v = 0; v < V; ++v) O[v] = 0.f;
    for (int s = grp; s < nsplit; s += 8) {
        const float m = part_ml[(row0 + s) * 2], l = part_ml[(row0 + s) * 2 + 1];
        const float Mn = fmaxf(M, m);
        const float a = ex2(M - Mn), w = ex2(m - Mn);
        L = L * a + l * w;
#pragma unroll
        for (int v = 0; v < V; ++v) O[v] = O[v] * a + part_acc[(row0 + s) * D + lane * V + v] * w;
        M = Mn;
    }
    if (lane == 0) {
        sM[grp] = M;
        sL[grp] = L;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) sO[grp][lane * V + v] = O[v];
    __syncthreads();
    if (threadIdx.x < D) {
        const int d = threadIdx.x;
        float Mx = -INFINITY;
        for (int k = 0; k < 8; ++k) Mx = fmaxf(Mx, sM[k]);
        float Lt = 0.f, Ot = 0.f;
        for (int k = 0; k < 8; ++k) {
            const float w = ex2(sM[k] - Mx);  // groups that saw no split have M = -inf
            Lt += sL[k] * w;
            Ot += sO[k][d] * w;
        }
        const float r = Lt > 0.f ? Ot / Lt : 0.f;
        const int64_t idx = (static_cast<int64_t>(b) * Hq + h) * D + d;
        if (out_f32)
            static_cast<float*>(out)[idx] = r;
        else
            static_cast<__half*>(out)[idx] = __float2half_rn(r);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int sm_count() {
    static std::atomic<int> cached[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128 && cached[dev].load()) return cached[dev].load();
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128) cached[dev].store(n);
    return n;
}

cudaError_t decode_plan(int B, int Hq, int Hkv, int D, int max_ctx, int bps_req, DecodePlan* plan) {
    const int nblk = (max_ctx + kBlockSize - 1) / kBlockSize;
    int bps = bps_req;
    if (bps <= 0) {
        const int sms = sm_count();
        if (sms <= 0) return cudaErrorNoDevice;
        // aim for about two waves of 3 resident CTAs per SM, at least one block per warp
        const int64_t work = static_cast<int64_t>(B) * Hkv * nblk;
        const int64_t target = static_cast<int64_t>(sms) * 6;
        int64_t want = (work + target - 1) / target;
        want = std::max<int64_t>(want, kWarps);
        want = (want + kWarps - 1) / kWarps * kWarps;
        bps = static_cast<int>(std::min<int64_t>(want, nblk));
    }
    const int nsplit = (nblk + bps - 1) / bps;
    plan->blocks_per_split = bps;
    plan->num_splits = nsplit;
    plan->workspace_bytes = nsplit > 1 ? static_cast<size_t>(B) * Hq * nsplit * (2 + D) * sizeof(float) : 0;
    return cudaSuccess;
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view of one layer's pool: rows of D fp16 (a (block, KV head, offset) row each),
// boxes of 16 rows x 64 columns, 128-byte swizzle.
static cudaError_t make_tile_map(CUtensorMap* map, const void* base, int D, int64_t rows) {
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

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    using Geo = DecodeGeom<D>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(paged_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Geo::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    CUtensorMap tmK, tmV;
    cudaError_t e = make_tile_map(&tmK, a.k_cache, D, rows);
    if (e != cudaSuccess) return e;
    e = make_tile_map(&tmV, a.v_cache, D, rows);
    if (e != cudaSuccess) return e;

    DecodeKernelParams p;
    p.q = a.q;
    p.block_table = a.block_table;
    p.context_lens = a.context_lens;
    p.out = a.out;
    p.part_ml = static_cast<float*>(a.workspace);
    p.part_acc = plan.num_splits > 1
                     ? static_cast<float*>(a.workspace) + static_cast<size_t>(a.B) * a.Hq * plan.num_splits * 2
                     : nullptr;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.max_ctx = a.max_context_len;
    p.bps = plan.blocks_per_split;
    p.nsplit = plan.num_splits;
    p.out_f32 = a.out_f32;
    p.scale_log2 = a.scale * kLog2e;

    dim3 grid(plan.num_splits, a.Hkv, a.B);
    paged_decode_kernel<D><<<grid, kWarps * 32, Geo::kSmemBytes, stream>>>(tmK, tmV, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (plan.num_splits > 1) {
        dim3 cgrid(a.Hq, a.B);
        paged_decode_combine_kernel<D><<<cgrid, 256, 0, stream>>>(p.part_ml, p.part_acc, a.context_lens, a.out,
                                                                  a.Hq, plan.num_splits, plan.blocks_per_split,
                                                                  a.max_blocks, a.max_context_len, a.out_f32);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    DecodePlan plan;
    cudaError_t e = decode_plan(a.B, a.Hq, a.Hkv, a.D, a.max_context_len, a.blocks_per_split, &plan);
    if (e != cudaSuccess) return e;
    if (plan.workspace_bytes > a.workspace_bytes) return cudaErrorInvalidValue;
    switch (a.D) {
        case 64: return launch_decode_d<64>(a, plan, stream);
        case 128: return launch_decode_d<128>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
