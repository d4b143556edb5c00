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
// With k_new/v_new the kernel also performs the step's append: the new
// token's K/V go to position ctx-1 of the cache (step 2 of a decode token on
// the gustavoai.dev page) and enter the attention directly.
//
// Design (GB300):
//  * one CTA per (context split, KV head, sequence), the grid sized from the
//    measured occupancy so that every CTA is resident at once; the splits of
//    one (sequence, KV head) form a thread-block cluster (up to 8 CTAs);
//  * the G <= 8 query heads of a KV head are the rows of one m16n8k16 tile, so
//    every K/V tile fetched from HBM serves the whole group;
//  * each warp owns a ring of stages; lane 0 issues the K and V tile loads
//    (16 tokens x D fp16 each) with 2-D TMA and the 128-byte swizzle so that
//    the ldmatrix reads are bank-conflict free; the warp waits on the stage's
//    mbarrier (bounded wait, error flag on expiry) and refills it;
//  * the block-table entries are fetched in one coalesced load (one entry per
//    lane) together with the context length, and passed by shuffles;
//  * S = Q K^T and O += P V on the tensor cores (mma.sync, fp16 in, fp32
//    accumulate); P is split into an fp16 high part and an fp16 residual so
//    the P V product keeps ~fp32 accuracy; online softmax in fp32, base 2;
//  * merging follows the FlashAttention article ("Was ist der mathematische
//    Aspekt von Softmax?"): partial (m, l, acc) are rescaled by 2^(m - M), M
//    the global maximum.  Warps merge through shared memory, the CTAs of a
//    cluster through distributed shared memory (no global round trip); only
//    contexts longer than a cluster's reach write per-cluster partials, which
//    a small combine kernel merges;
//  * with launch overlap on, the kernel is a programmatic dependent of the
//    previous kernel: it fetches block tables, context lengths and cached K/V
//    before waiting for that kernel, and reads q, k_new, v_new (and writes
//    anything) only after.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

// Tuning knobs (compile-time; the defaults are the measured best on GB300).
#ifndef KVC_DEC_WARPS64
#define KVC_DEC_WARPS64 8
#endif
#ifndef KVC_DEC_STAGES64
#define KVC_DEC_STAGES64 2
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
#ifndef KVC_DEC_EARLY_TRIGGER  // let the next kernel launch as soon as every CTA of this one has started
#define KVC_DEC_EARLY_TRIGGER 1
#endif

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWarpBlocks = 32;  // blocks per warp per split (one table entry per lane)
constexpr int kMaxCluster = KVC_DEC_MAX_CLUSTER;

std::atomic<int> g_launch_overlap{0};

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = D == 64 ? KVC_DEC_WARPS64 : KVC_DEC_WARPS128;
    static constexpr int kStages = D == 64 ? KVC_DEC_STAGES64 : KVC_DEC_STAGES128;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kTileBytes = kBlockSize * D * 2;  // one 16 x D fp16 tile
    static constexpr int kStageBytes = 2 * kTileBytes;     // K tile + V tile
    static constexpr int kWarpRingBytes = kStages * kStageBytes;
    static constexpr int kRingBytes = kWarps * kWarpRingBytes;
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static constexpr int kStateBytes = 8 * (D + 2) * 4;  // the CTA's merged (m, l, acc) for 8 rows
    static constexpr int kSmemBytes = kRingBytes + kBarBytes + kStateBytes + 1024;  // + alignment slack
    static constexpr int kMergeStride = D + 4;                                       // floats per parked row
    static constexpr int kMaxBps = kWarps * kMaxWarpBlocks;
    static_assert(16 * 4 + 8 * kMergeStride * 4 <= kWarpRingBytes, "warp state must fit a warp ring");
};

struct DecodeKernelParams {
    const __half* q;
    const __half* k_new;  // null: no append
    const __half* v_new;
    __half* k_cache;      // generic pointers to the same layer as the tensor maps (append target)
    __half* v_cache;
    const int32_t* block_table;
    const int32_t* context_lens;
    void* out;
    float* part_ml;   // [B][Hq][nparts][2] (m, l) in base-2 units, one part per cluster
    float* part_acc;  // [B][Hq][nparts][D]
    unsigned* err;
    int max_blocks, num_blocks, B, Hq, Hkv, G, max_ctx, bps, csize, nparts, out_f32;
    float scale_log2;
    unsigned trace_seq;  // launch counter, used by the optional trace only
};

// ---- optional per-CTA timeline trace (build with -DKVC_TRACE=1) -----------------------------
// Each CTA records the global timer at: start, TMA issued, dependency wait passed, main loop done,
// exit; plus its SM and coordinates.  kvc_trace_read() copies the records out.
#ifndef KVC_TRACE
#define KVC_TRACE 0
#endif
#if KVC_TRACE
struct TraceRec {
    unsigned long long t[5];
    unsigned seq, smid, x, yz;
};
constexpr int kTraceCap = 1 << 16;
__device__ TraceRec g_trace[kTraceCap];
__device__ unsigned g_trace_n;
#define KVC_TRACE_MARK(i) \
    if (threadIdx.x == 0) tr_t[i] = global_timer_ns()
#define KVC_TRACE_END()                                                    \
    do {                                                                   \
        if (threadIdx.x == 0) {                                            \
            tr_t[4] = global_timer_ns();                                   \
            const unsigned k = atomicAdd(&g_trace_n, 1u);                  \
            if (k < kTraceCap) {                                           \
                TraceRec& r = g_trace[k];                                  \
                for (int q_ = 0; q_ < 5; ++q_) r.t[q_] = tr_t[q_];         \
                unsigned sm_;                                              \
                asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));           \
                r.seq = p.trace_seq;                                       \
                r.smid = sm_;                                              \
                r.x = blockIdx.x;                                          \
                r.yz = (blockIdx.y << 16) | blockIdx.z;                    \
            }                                                              \
        }                                                                  \
    } while (0)
#else
#define KVC_TRACE_MARK(i) \
    do {                  \
    } while (0)
#define KVC_TRACE_END() \
    do {                \
    } while (0)
#endif

// byte offset of 16-byte chunk `chunk` (8 fp16 columns) of row `row` inside a
// tile loaded as boxes of 16 rows x 64 columns with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(((chunk >> 3) << 11) + (row << 7) + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void store_out(void* out, int out_f32, int64_t idx, float v) {
    if (out_f32)
        static_cast<float*>(out)[idx] = v;
    else
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// ---- thread-block cluster helpers ------------------------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeKernelParams p) {
    using C = DecodeCfg<D>;
    constexpr int NW = C::kWarps, ST = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
    // the CTA's merged state: m[8], l[8], acc[8][D]
    float* s_m = reinterpret_cast<float*>(smem + C::kRingBytes + C::kBarBytes);
    float* s_l = s_m + 8;
    float* s_acc = s_m + 16;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
#if KVC_TRACE
    unsigned long long tr_t[5] = {0, 0, 0, 0, 0};
#endif
#if KVC_DEC_EARLY_TRIGGER
    grid_dependents_launch();
#endif
    KVC_TRACE_MARK(0);

    // The block-table entries this lane would own if the split were full are fetched together with the
    // context length (one round trip instead of two); indices stay inside the table row.
    const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
    const int j0 = split * p.bps;
    const int jl = j0 + warp + lane * NW;
    const int spec_blk = (warp + lane * NW < p.bps && jl < p.max_blocks) ? table[jl] : -1;
    const int ctx = p.context_lens[b];
    // every CTA of a cluster sees the same (b, kvh): these exits are uniform over the cluster
    if (ctx < 1 || ctx > p.max_blocks * kBlockSize || ctx > p.max_ctx) {
        grid_dependency_wait();
        if (split == 0) {
            if (threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            for (int e = threadIdx.x; e < p.G * D; e += blockDim.x)
                store_out(p.out, p.out_f32, (static_cast<int64_t>(b) * p.Hq + kvh * p.G + e / D) * D + e % D, 0.f);
        }
        return;
    }
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    const int nsplit = (nblk + p.bps - 1) / p.bps;
    const int cs = p.csize;
    const int cidx = split / cs;                       // this CTA's cluster along the context
    const int nclus = (nsplit + cs - 1) / cs;          // clusters this sequence needs
    if (cidx >= nclus) return;                         // the whole cluster is past the context
    const bool active = split < nsplit;                // an inactive CTA only joins the cluster merge
    const int nb_split = active ? min(j0 + p.bps, nblk) - j0 : 0;
    const int nb_w = warp < nb_split ? (nb_split - warp + NW - 1) / NW : 0;  // <= kMaxWarpBlocks
    const int my_blk = lane < nb_w ? spec_blk : -1;  // this warp's block-table entries, one per lane

    if (threadIdx.x == 0) {
        for (int i = 0; i < NW * ST; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();

    uint64_t* wbars = bars + warp * ST;
    uint8_t* wring = smem + warp * C::kWarpRingBytes;
    const uint64_t policy = l2_policy_evict_first();

    // lane 0: the K and V tiles of this warp's i-th block into stage i % ST
    auto issue = [&](int i, int phys) {
        uint64_t* bar = &wbars[i % ST];
        if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, KVC_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // complete the phase without data; the block is skipped
            return;
        }
        uint8_t* st = wring + (i % ST) * C::kStageBytes;
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int y = (phys * p.Hkv + kvh) * kBlockSize;
#pragma unroll
        for (int x = 0; x < D; x += 64) {
            tma_load_2d(st + (x / 64) * 2048, &tmK, bar, x, y, policy);
            tma_load_2d(st + C::kTileBytes + (x / 64) * 2048, &tmV, bar, x, y, policy);
        }
    };
#pragma unroll
    for (int i = 0; i < ST; ++i) {
        const int phys = __shfl_sync(0xffffffffu, my_blk, i);
        if (lane == 0 && i < nb_w) issue(i, phys);
    }
    KVC_TRACE_MARK(1);

    // ---- everything below may read what the previous kernel wrote ----
    grid_dependency_wait();
    KVC_TRACE_MARK(2);

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

    // fused append: the warp holding the block of position ctx-1 writes the new row to the cache
    // and patches it into its shared-memory tile before use
    int app_iter = -1;
    const int app_row = (ctx - 1) % kBlockSize;
    uint4 app_val = make_uint4(0, 0, 0, 0);
    if (p.k_new != nullptr && split == nsplit - 1 && ((nblk - 1 - j0) % NW) == warp) {
        app_iter = (nblk - 1 - j0) / NW;
        const int phys = __shfl_sync(0xffffffffu, my_blk, app_iter);
        const int c = lane & 15;
        const bool is_v = lane >= 16;
        if (c < D / 8) {
            const __half* src = (is_v ? p.v_new : p.k_new) + (static_cast<int64_t>(b) * p.Hkv + kvh) * D + c * 8;
            app_val = *reinterpret_cast<const uint4*>(src);
            if (phys >= 0 && phys < p.num_blocks) {
                __half* dst = (is_v ? p.v_cache : p.k_cache) +
                              ((static_cast<int64_t>(phys) * p.Hkv + kvh) * kBlockSize + app_row) * D + c * 8;
                *reinterpret_cast<uint4*>(dst) = app_val;
            }
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
        const int stage = i % ST;
        const uint32_t parity = (i / ST) & 1;
        const int jj = j0 + warp + i * NW;
        const int phys = __shfl_sync(0xffffffffu, my_blk, i);
        const bool ok = mbar_wait_bounded(&wbars[stage], parity, kWaitLimitNs);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        if (phys >= 0 && phys < p.num_blocks) {
            const uint32_t kbase = smem_u32(wring + stage * C::kStageBytes);
            const uint32_t vbase = kbase + C::kTileBytes;
            if (i == app_iter) {
                const int c = lane & 15;
                if (c < D / 8) {
                    const uint32_t a = (lane >= 16 ? vbase : kbase) + swz(app_row, c);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(app_val.x), "r"(app_val.y),
                                 "r"(app_val.z), "r"(app_val.w)
                                 : "memory");
                }
                __syncwarp();
            }
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
        const int nxt = __shfl_sync(0xffffffffu, my_blk, (i + ST) & 31);
        if (lane == 0 && i + ST < nb_w) issue(i + ST, nxt);
    }
#if !KVC_DEC_EARLY_TRIGGER
    grid_dependents_launch();  // the next kernel may start its prologue while this one finishes
#endif
    KVC_TRACE_MARK(3);
    if (timed_out) {
        if (lane == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        // let copies still in flight land before the shared memory is reused
        for (int k = i; k < min(nb_w, i + ST); ++k) mbar_wait_bounded(&wbars[k % ST], (k / ST) & 1, kWaitLimitNs / 8);
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = 0.f;
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
        *reinterpret_cast<float2*>(wo + g * C::kMergeStride + nd * 8 + 2 * t4) = make_float2(o[nd][0], o[nd][1]);
    __syncthreads();

    const bool direct = nclus == 1 && cs == 1;  // a single CTA holds the whole context
    for (int e = threadIdx.x; e < p.G * D; e += blockDim.x) {
        const int gg = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float*>(smem + w * C::kWarpRingBytes)[gg]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float* r = reinterpret_cast<const float*>(smem + w * C::kWarpRingBytes);
                const float wgt = ex2(r[gg] - M);  // an empty warp has m = -inf -> weight 0
                L += r[8 + gg] * wgt;
                O += r[16 + gg * C::kMergeStride + d] * wgt;
            }
        }
        if (direct) {
            store_out(p.out, p.out_f32, (static_cast<int64_t>(b) * p.Hq + kvh * p.G + gg) * D + d,
                      L > 0.f ? O / L : 0.f);
        } else {
            if (d == 0) {
                s_m[gg] = M;
                s_l[gg] = L;
            }
            s_acc[gg * D + d] = O;
        }
    }
    if (direct) {
        KVC_TRACE_END();
        return;
    }

    // ---- merge the CTAs of this cluster through distributed shared memory ----
    if (cs > 1)
        cluster_sync_all();  // every CTA's state is in its shared memory
    else
        __syncthreads();
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int nthreads = cs * C::kThreads;
    for (int e = rank * C::kThreads + threadIdx.x; e < p.G * D; e += nthreads) {
        const int gg = e / D, d = e % D;
        float mc[kMaxCluster], lc[kMaxCluster];
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            if (c < cs) {
                mc[c] = ld_cluster_f32(map_to_rank(s_m + gg, c));
                lc[c] = ld_cluster_f32(map_to_rank(s_l + gg, c));
                M = fmaxf(M, mc[c]);
            }
        }
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            if (c < cs && lc[c] > 0.f) {  // an inactive or empty CTA contributes nothing
                const float w = ex2(mc[c] - M);
                L += lc[c] * w;
                O += ld_cluster_f32(map_to_rank(s_acc + gg * D + d, c)) * w;
            }
        }
        const int h = kvh * p.G + gg;
        if (nclus == 1) {
            store_out(p.out, p.out_f32, (static_cast<int64_t>(b) * p.Hq + h) * D + d, L > 0.f ? O / L : 0.f);
        } else {
            const int64_t row = (static_cast<int64_t>(b) * p.Hq + h) * p.nparts + cidx;
            if (d == 0) {
                p.part_ml[row * 2 + 0] = M;
                p.part_ml[row * 2 + 1] = L;
            }
            p.part_acc[row * D + d] = O;
        }
    }
    if (cs > 1) cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    KVC_TRACE_END();
}

// Merge the per-cluster partials of every (sequence, query head) for contexts
// longer than one cluster covers: 8 groups of 32 lanes walk the parts with a
// running (M, L, acc), then the groups merge.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_combine_kernel(const float* __restrict__ part_ml,
                                                                    const float* __restrict__ part_acc,
                                                                    const int32_t* __restrict__ context_lens,
                                                                    void* out, int Hq, int nparts_grid, int bps,
                                                                    int csize, int max_blocks, int max_ctx,
                                                                    int out_f32) {
    constexpr int V = D / 32;  // dims per lane
    __shared__ float sM[8], sL[8], sO[8][D];
    grid_dependency_wait();
    const int h = blockIdx.x, b = blockIdx.y;
    const int grp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ctx = context_lens[b];
    if (ctx < 1 || ctx > max_blocks * kBlockSize || ctx > max_ctx) return;
    const int nsplit = ((ctx + kBlockSize - 1) / kBlockSize + bps - 1) / bps;
    const int nparts = (nsplit + csize - 1) / csize;
    if (nparts <= 1) return;  // the cluster wrote the output itself
    const int64_t row0 = (static_cast<int64_t>(b) * Hq + h) * nparts_grid;
    float M = -INFINITY, L = 0.f, O[V];
#pragma unroll
    for (int v = 0; v < V; ++v) O[v] = 0.f;
    for (int s = grp; s < nparts; s += 8) {
        const float m = part_ml[(row0 + s) * 2], l = part_ml[(row0 + s) * 2 + 1];
        if (!(l > 0.f)) continue;
        const float Mn = fmaxf(M, m);
        const float a = M == -INFINITY ? 0.f : ex2(M - Mn);
        const float w = ex2(m - Mn);
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
            if (!(sL[k] > 0.f)) continue;  // groups that saw no part
            const float w = ex2(sM[k] - Mx);
            Lt += sL[k] * w;
            Ot += sO[k][d] * w;
        }
        store_out(out, out_f32, (static_cast<int64_t>(b) * Hq + h) * D + d, Lt > 0.f ? Ot / Lt : 0.f);
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

// one-time kernel attributes and the resident CTAs per SM of the decode kernel
template <int D>
static cudaError_t decode_setup(int* ctas_per_sm) {
    using C = DecodeCfg<D>;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    static int occ = 0;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(paged_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (err == cudaSuccess && kMaxCluster > 8)
            err = cudaFuncSetAttribute(paged_decode_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err == cudaSuccess)
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, paged_decode_kernel<D>, C::kThreads,
                                                                C::kSmemBytes);
        if (err == cudaSuccess && occ < 1) err = cudaErrorInvalidConfiguration;
    });
    if (ctas_per_sm) *ctas_per_sm = occ;
    return err;
}

template <int D>
static cudaError_t plan_d(int B, int Hq, int Hkv, int max_ctx, int bps_req, DecodePlan* plan) {
    using C = DecodeCfg<D>;
    const int nblk = std::max((max_ctx + kBlockSize - 1) / kBlockSize, 1);
    int bps = bps_req;
    if (bps <= 0) {
        const int sms = sm_count();
        if (sms <= 0) return cudaErrorNoDevice;
        int occ = 0;
        cudaError_t e = decode_setup<D>(&occ);
        if (e != cudaSuccess) return e;
        // one wave: every CTA resident at once; at least one block per warp
        const int64_t work = static_cast<int64_t>(B) * Hkv * nblk;
        const int64_t slots = static_cast<int64_t>(sms) * occ;
        int64_t want = (work + slots - 1) / slots;
        want = std::max<int64_t>(want, C::kWarps);
        want = (want + C::kWarps - 1) / C::kWarps * C::kWarps;
        bps = static_cast<int>(std::min<int64_t>(std::min<int64_t>(want, C::kMaxBps), nblk));
    }
    if (bps > C::kMaxBps) bps = C::kMaxBps;
    const int nsplit = (nblk + bps - 1) / bps;
    const int cs = std::min(nsplit, kMaxCluster);
    const int nparts = (nsplit + cs - 1) / cs;
    plan->blocks_per_split = bps;
    plan->cluster = cs;
    plan->num_splits = nparts * cs;  // grid.x, a whole number of clusters
    plan->num_parts = nparts;
    plan->workspace_bytes = nparts > 1 ? static_cast<size_t>(B) * Hq * nparts * (2 + D) * sizeof(float) : 0;
    return cudaSuccess;
}

cudaError_t decode_plan(int B, int Hq, int Hkv, int D, int max_ctx, int bps_req, DecodePlan* plan) {
    switch (D) {
        case 64: return plan_d<64>(B, Hq, Hkv, max_ctx, bps_req, plan);
        case 128: return plan_d<128>(B, Hq, Hkv, max_ctx, bps_req, plan);
        default: return cudaErrorInvalidValue;
    }
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFn encode_fn() {
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

template <typename Kern, typename... Args>
static cudaError_t launch(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
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

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    cudaError_t e = decode_setup<D>(nullptr);
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    CUtensorMap tmK, tmV;
    e = make_tile_map(&tmK, a.k_cache, D, rows);
    if (e != cudaSuccess) return e;
    e = make_tile_map(&tmV, a.v_cache, D, rows);
    if (e != cudaSuccess) return e;

    DecodeKernelParams p;
    p.q = a.q;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_cache = const_cast<__half*>(a.k_cache);
    p.v_cache = const_cast<__half*>(a.v_cache);
    p.block_table = a.block_table;
    p.context_lens = a.context_lens;
    p.out = a.out;
    const size_t nrow = static_cast<size_t>(a.B) * a.Hq * plan.num_parts;
    p.part_ml = plan.num_parts > 1 ? static_cast<float*>(a.workspace) : nullptr;
    p.part_acc = plan.num_parts > 1 ? p.part_ml + nrow * 2 : nullptr;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.max_ctx = a.max_context_len;
    p.bps = plan.blocks_per_split;
    p.csize = plan.cluster;
    p.nparts = plan.num_parts;
    p.out_f32 = a.out_f32;
    p.scale_log2 = a.scale * kLog2e;
    static std::atomic<unsigned> launch_seq{0};
    p.trace_seq = launch_seq.fetch_add(1);

    const bool pdl = g_launch_overlap.load(std::memory_order_relaxed) != 0;
    dim3 grid(plan.num_splits, a.Hkv, a.B);
    e = launch(paged_decode_kernel<D>, grid, dim3(C::kThreads), C::kSmemBytes, stream, pdl,
               static_cast<unsigned>(plan.cluster), tmK, tmV, p);
    if (e != cudaSuccess) return e;
    if (plan.num_parts > 1) {
        dim3 cgrid(a.Hq, a.B);
        e = launch(paged_decode_combine_kernel<D>, cgrid, dim3(256), 0, stream, true, 1u,
                   static_cast<const float*>(p.part_ml), static_cast<const float*>(p.part_acc), a.context_lens,
                   a.out, a.Hq, plan.num_parts, plan.blocks_per_split, plan.cluster, a.max_blocks,
                   a.max_context_len, a.out_f32);
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

cudaError_t trace_read(void* host, int cap, int* n, int clear) {
#if KVC_TRACE
    unsigned cnt = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&cnt, g_trace_n, sizeof(cnt));
    if (e != cudaSuccess) return e;
    const int m = static_cast<int>(std::min<unsigned>(std::min<unsigned>(cnt, kTraceCap), static_cast<unsigned>(cap)));
    if (m > 0) e = cudaMemcpyFromSymbol(host, g_trace, sizeof(TraceRec) * m);
    if (e != cudaSuccess) return e;
    *n = m;
    if (clear) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_trace_n, &z, sizeof(z));
    }
    return e;
#else
    (void)host;
    (void)cap;
    (void)clear;
    *n = 0;
    return cudaErrorNotSupported;
#endif
}

void set_launch_overlap(int on) { g_launch_overlap.store(on ? 1 : 0); }
int launch_overlap() { return g_launch_overlap.load(); }

}  // namespace kvc
