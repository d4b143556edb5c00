// Decode over query rows that share their key blocks, on sm_103a: the multi-token decode (the q_len new tokens of
// one sequence) and the cascade decode's shared-prefix pass (the sequences of one group; with head dim 64 and
// groups of 17 or more query rows that pass runs on the tensor cores instead, group_tc.cu).
//
// Multi-token decode: q_len new tokens per sequence attend over the paged cache at once, causally among
// themselves (token t sits at position ctx - q_len + t and sees keys 0 .. ctx - q_len + t).  Speculative
// decoding paragraph of "Tornar a inferência barata" (neuralialabs.com): the proposed tokens are verified in
// one pass over their positions.  Cascade prefix: the sequences of a group whose block-table rows begin with the
// same blocks (the shared prefix blocks of the PagedAttention paragraph of the same page) attend over those
// blocks once for the whole group; the decode kernel covers each sequence's remaining blocks and the combine
// kernel merges both.
//
// Work split: a CTA takes one (unit, KV head, chunk of blocks, row group); a unit is a sequence (multi-token)
// or a group (cascade prefix).  The query rows of a unit and KV head are its members x G heads (member = new
// token, or sequence of the group), row r = member * G + h; a row group is up to 8 * NT of them, and each warp
// carries the whole row group as NT mma.sync n-tiles of 8 rows.  The CTA's warps take the chunk's blocks
// round-robin, each through its own ring of TMA stages, so a block's K and V tiles are read from shared memory
// once for every member.  Per block (the decode kernel's math): S^T = K Q^T, causal mask per row (multi-token),
// online softmax in base 2, O^T += V^T (P_hi + P_lo)^T.  The warps' states are merged in shared memory, then the
// CTAs of a thread-block cluster (consecutive chunks) merge in rank 0 through distributed shared memory.  A
// multi-token cluster that covers the whole context writes the output; otherwise each cluster writes a partial
// state and the combine kernel (decode.cu) merges them.
#include "decode_common.cuh"
#include "group_tc.h"
#include "multi_tc.h"

namespace kvc {

#ifndef KVC_MULTI_WARPS  // warps per CTA
#define KVC_MULTI_WARPS 8
#endif
#ifndef KVC_MULTI_STAGES64  // blocks in flight per warp, head_dim 64, two CTAs per SM (up to 16 query rows)
#define KVC_MULTI_STAGES64 2
#endif
#ifndef KVC_MULTI_STAGES64_WIDE  // the same with one CTA per SM (17 to 32 query rows)
#define KVC_MULTI_STAGES64_WIDE 4
#endif
#ifndef KVC_MULTI_STAGES128
#define KVC_MULTI_STAGES128 2
#endif
#ifndef KVC_MULTI_MAX_TILES64  // n-tiles per warp at most, head_dim 64 (more rows make more row groups)
#define KVC_MULTI_MAX_TILES64 2
#endif
#ifndef KVC_MULTI_TWO_CTA_TILES  // head_dim 64: n-tiles per warp up to which a CTA is sized for two CTAs per SM
#define KVC_MULTI_TWO_CTA_TILES 2
#endif
#ifndef KVC_MULTI_EARLY_REFILL  // 1: refill a stage once its V fragments are in registers, before the softmax
#define KVC_MULTI_EARLY_REFILL 1
#endif
// Multi-token calls: 1 = the P V products take P as an fp16 high part plus an fp16 residual (~fp32 weights, twice
// the products); 0 = P in fp16 with the sums over the rounded weights (the prefill's default form), measured on the
// 24-layer graph at 32 x 2048: T = 2 / 4 / 8 8.43 / 12.0 / 18.7 -> 7.94 / 11.1 / 16.9 us per layer.  The cascade's
// prefix pass always splits P: it re-associates the plain decode's sum, and stays within 1e-5 of it.
#ifndef KVC_MULTI_P_SPLIT
#define KVC_MULTI_P_SPLIT 0
#endif
#ifndef KVC_MULTI_CTAS  // CTAs per SM the chunking aims for (one where a CTA needs the SM's registers)
#define KVC_MULTI_CTAS 2
#endif
// A cascade call runs the cascade kernels only when the block reads it saves per KV head, at most
// (B - n_groups) x max_shared_blocks, reach this many; otherwise the plain decode (one launch) is faster.  Measured
// on GB300 (one call, L2 flushed; groups x members x shared blocks, 1..200 private tokens each): 8 x 8 x 512
// (28,672 saved) 0.94x, 25 x 8 x 128 (22,400) 0.89x, 8 x 8 x 768 (43,008) 1.11x, 25 x 8 x 256 (44,800) 1.13x.
#ifndef KVC_CASCADE_MIN_SAVED_BLOCKS
#define KVC_CASCADE_MIN_SAVED_BLOCKS 36000
#endif
static std::atomic<int> g_cascade_min_saved{KVC_CASCADE_MIN_SAVED_BLOCKS};
void set_cascade_min_saved_blocks(int blocks) { g_cascade_min_saved.store(blocks); }
// multi-token decode at head dim 64 with up to 64 query rows on the tensor cores (multi_tc.cu) when set; off by
// default (measured slower than the mma.sync kernel on the listed shapes)
static std::atomic<int> g_multi_tc{0};
void set_multi_tc(int on) { g_multi_tc.store(on ? 1 : 0); }
#ifndef KVC_PREFIX_TC_MIN_ROWS  // cascade prefix, head dim 64: groups of this many query rows run on the tensor cores
#define KVC_PREFIX_TC_MIN_ROWS 17
#endif

constexpr int kMultiMaxChunk = 2048;  // blocks per CTA at most (their ids are in shared memory)
constexpr int kMultiMaxCluster = 8;   // CTAs per cluster at most

template <int D, int NT>
struct GroupCfg {
    static constexpr int kWarps = KVC_MULTI_WARPS;
    static constexpr int kThreads = kWarps * 32;
    // resident CTAs per SM the register allocation must allow
    static constexpr int kMinCtas = D == 64 && NT <= KVC_MULTI_TWO_CTA_TILES ? 2 : 1;
    // (two CTAs per SM with 4 n-tiles: 3 stages, so that the parked state fits a warp's ring)
    static constexpr int kStages =
        D == 64 ? (kMinCtas == 2 ? (NT == 4 && KVC_MULTI_STAGES64 < 3 ? 3 : KVC_MULTI_STAGES64)
                                 : KVC_MULTI_STAGES64_WIDE)
                : KVC_MULTI_STAGES128;
    static constexpr int RG = 8 * NT;  // query rows of a CTA
    static constexpr int kTileBytes = kBlockSize * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
    static constexpr int kWarpRingBytes = kStages * kStageBytes;
    static constexpr int kRingBytes = kWarps * kWarpRingBytes;
    // after its blocks a warp parks its state in its own ring: m[RG], l[RG], then acc rows at a stride of
    // D + 4 floats
    static constexpr int kRowStride = D + 4;
    static_assert(RG * (2 + kRowStride) * 4 <= kWarpRingBytes, "a warp's state must fit its ring");
    // the inbox after the rings (read in a cluster's rank 0): one slot per CTA of the cluster with that
    // CTA's merged state m[RG], l[RG], acc[RG][D]
    static constexpr int kSlotFloats = RG * (2 + D);
    static constexpr int kBarBytes = kWarps * kStages * 8;
    static size_t smem_bytes(int chunk, int cluster) {
        return kRingBytes + static_cast<size_t>(cluster) * kSlotFloats * 4 + kBarBytes + 16 +
               4 * static_cast<size_t>(chunk) + 1024;
    }
};

struct GroupKernelParams {
    const __half* q;              // [B][q_len][Hq][D] (multi-token) or [B][Hq][D] (cascade prefix)
    const int32_t* block_table;   // [B][max_blocks]
    const int32_t* context_lens;  // multi-token: [B], including the q_len new tokens
    const int32_t* group_start;   // cascade prefix: [n_groups + 1], group u is sequences group_start[u] ..
    const int32_t* blk_off;       // cascade prefix: [B], the shared blocks of each sequence's group
    void* out;                    // [B][q_len][Hq][D] (multi-token, written here when one cluster covers a context)
    float* part_ml;               // partial states: part `cluster index` of each row, rows part_stride apart
    float* part_acc;
    unsigned* err;
    int max_blocks, num_blocks, Hq, Hkv, G, q_len, max_ctx, out_f32;
    int chunk;        // blocks per CTA
    int cs;           // CTAs per cluster (consecutive blockIdx.x)
    int nclus;        // clusters per (unit, KV head, row group)
    int part_stride;  // partial rows per query row
    float scale_log2;
};

// kPrefix: the cascade's shared-prefix pass (unit = group, no mask, partial states only); else multi-token
template <int D, int NT, bool kPrefix>
__global__ void __launch_bounds__(GroupCfg<D, NT>::kThreads, GroupCfg<D, NT>::kMinCtas)
    paged_decode_group_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const GroupKernelParams p) {
    using C = GroupCfg<D, NT>;
    constexpr int NW = C::kWarps, ST = C::kStages, RG = C::RG;
    constexpr bool kSplitP = kPrefix || KVC_MULTI_P_SPLIT;  // P as high part + residual (see KVC_MULTI_P_SPLIT)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int cs = p.cs;
    float* s_inbox = reinterpret_cast<float*>(smem + C::kRingBytes);                      // [cs][kSlotFloats]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_inbox + static_cast<size_t>(cs) * C::kSlotFloats);  // [NW][ST]
    int* s_ids = reinterpret_cast<int*>(bars + NW * ST) + 4;  // the chunk's physical block ids

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;  // == blockIdx.x % cs
    const int cidx = (blockIdx.x / cs) % p.nclus, rg = blockIdx.x / (cs * p.nclus);
    const int kvh = blockIdx.y, u = blockIdx.z;  // u: the sequence (multi-token) or the group (cascade prefix)
    const int r0 = rg * RG;
    // the unit: its members (T new tokens of sequence u, or the sequences s0 .. s0 + T - 1 of group u), the
    // table row its blocks come from, its keys [0, ctx) and its blocks; every CTA of a cluster has the same
    // (unit, KV head, row group), so the exits below are uniform over the cluster
    int T, s0, ctx;
    if constexpr (kPrefix) {
        s0 = p.group_start[u];
        T = p.group_start[u + 1] - s0;
        if (T < 1 || r0 >= T * p.G) {  // an empty group, or no rows in this row group
            leave_before_dependency_wait();
            return;
        }
        const int nsh = p.blk_off[s0];
        if (T > kMaxGroupSize || nsh < 0 || nsh > p.max_blocks) {
            if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            leave_before_dependency_wait();
            return;  // the combine kernel writes these sequences' rows
        }
        ctx = nsh * kBlockSize;  // the shared blocks lie inside every member's context: no key is masked
    } else {
        s0 = u;
        T = p.q_len;
        ctx = p.context_lens[u];
        if (ctx < T || ctx > p.max_blocks * kBlockSize || ctx > p.max_ctx) {
            grid_dependency_wait();
            if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            // with several clusters per context the combine kernel writes the zeros
            if (p.nclus == 1 && rank == 0)
                for (int e = threadIdx.x; e < min(RG, T * p.G - r0) * D; e += blockDim.x) {
                    const int r = r0 + e / D, t = r / p.G, h = r % p.G;
                    store_out(p.out, p.out_f32,
                              ((static_cast<int64_t>(u) * T + t) * p.Hq + kvh * p.G + h) * D + e % D, 0.f);
                }
            return;
        }
    }
    const int R = T * p.G;
    const int rows = min(RG, R - r0);  // >= 1: the row groups tile the R rows
    // row r of the unit as a row of q (and of the output and the partials) of Hq heads: member r / G, head r % G
    auto q_row = [&](int r) -> int64_t {
        const int64_t seq_row = kPrefix ? static_cast<int64_t>(s0) + r / p.G : static_cast<int64_t>(u) * T + r / p.G;
        return seq_row * p.Hq + kvh * p.G + r % p.G;
    };
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    if (cidx * cs * p.chunk >= nblk) {  // the whole cluster is past this context (or no block is shared)
        leave_before_dependency_wait();
        return;
    }
    // this CTA's blocks [j0, j0 + n); a CTA of a live cluster may have none and still takes part in its merge
    const int j0 = (cidx * cs + rank) * p.chunk;
    const int n = max(0, min(nblk, j0 + p.chunk) - j0);
    const int32_t* table = p.block_table + static_cast<int64_t>(s0) * p.max_blocks + j0;
    // this warp's blocks: j0 + warp + k * NW for k < nmine
    const int nmine = warp < n ? (n - warp + NW - 1) / NW : 0;

    uint64_t* wbars = bars + warp * ST;
    uint8_t* wring = smem + warp * C::kWarpRingBytes;
    const uint64_t policy = l2_policy_evict_first();
    // lane 0: the K and V tiles of physical block phys into stage s
    auto issue = [&](int s, int phys) {
        uint64_t* bar = &wbars[s];
        if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, KVC_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // completes the phase without data: the block is skipped
            return;
        }
        uint8_t* st = wring + s * C::kStageBytes;
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int y = (phys * p.Hkv + kvh) * kBlockSize;
#pragma unroll
        for (int x = 0; x < D; x += 64) {
            tma_load_2d(st + (x / 64) * 2048, &tmK, bar, x, y, policy);
            tma_load_2d(st + C::kTileBytes + (x / 64) * 2048, &tmV, bar, x, y, policy);
        }
    };
    // each warp's lane 0 sets up its barriers and issues its first blocks straight from the table; the
    // chunk's ids go to shared memory meanwhile, for the refills
    // rank 0's inbox barrier (in the padding after the stage barriers): completes when the other CTAs' merged
    // states have arrived by asynchronous pushes of push_bytes each
    uint64_t* inbox_bar = bars + NW * ST;
    const uint32_t push_bytes = static_cast<uint32_t>(rows * D * 4 + rows * 8);
    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&wbars[s], 1);
        if (KVC_DEC_ASYNC_PUSH && warp == 0 && cs > 1) mbar_init(inbox_bar, 1);
        fence_barrier_init();
        if (KVC_DEC_ASYNC_PUSH && warp == 0 && cs > 1 && rank == 0)
            mbar_arrive_expect_tx(inbox_bar, static_cast<uint32_t>(cs - 1) * push_bytes);
        if (warp == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        int first[ST];
#pragma unroll
        for (int s = 0; s < ST; ++s) first[s] = s < nmine ? table[warp + s * NW] : -1;
#pragma unroll
        for (int s = 0; s < ST; ++s)
            if (s < nmine) issue(s, first[s]);
    }
    for (int k = threadIdx.x; k < n; k += blockDim.x) s_ids[k] = table[k];
    __syncthreads();
    // announces that this CTA has started; the matching wait comes before the first remote store into
    // rank 0's inbox.  Nothing is published here, so the arrive needs no fence.
    if (cs > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    grid_dependency_wait();  // q and out may belong to the previous kernel
    if (n == 0) grid_dependents_launch();  // a CTA without blocks; the others release at their first refill
    // every CTA of the cluster has passed its prologue (rank 0's inbox barrier is initialised): the pushes after
    // the block loop need no further check (the decode kernel measured this wait at the end of a launch)
    if (KVC_DEC_EARLY_CLUSTER_WAIT && cs > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    // query fragments (B operand of S^T = K Q^T): column g of tile nt is row r0 + 8 nt + g (zero past R)
    uint32_t qa[NT][D / 16][2];
    // the last key position each of this lane's score columns (rows r0 + 8 nt + 2 t4 + e) may see
    int lastk[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int r = r0 + nt * 8 + g;
        const bool row_ok = r < R;
        const __half* qp = p.q + q_row(row_ok ? r : 0) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[nt][ks][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 2 * t4) : 0u;
            qa[nt][ks][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 8 + 2 * t4) : 0u;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int rc = r0 + nt * 8 + 2 * t4 + e;
            lastk[nt][e] = rc < R && !kPrefix ? ctx - T + rc / p.G : ctx - 1;
        }
    }
    // O^T accumulators: o[nt][mt] = dims mt*16 + g (+8) x rows 2*t4, 2*t4+1 of tile nt
    float o[NT][D / 16][4];
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
    }
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3;
    int k = 0;
    bool timed_out = false;
#pragma unroll 1
    for (; k < nmine; ++k) {
        const int s = k % ST;
        const bool ok = mbar_wait_bounded(&wbars[s], (k / ST) & 1, kWaitLimitNs);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            break;
        }
        const int jl = warp + k * NW;  // block index within the chunk
        const int phys = s_ids[jl];
        bool refilled = false;
        // the warp has read stage s: lane 0 refills it with the warp's block ST further on
        auto refill = [&](int kk, int ss) {
            __syncwarp();
            if (lane == 0 && kk + ST < nmine) issue(ss, s_ids[warp + (kk + ST) * NW]);
            if (kk == 0) grid_dependents_launch();  // the next kernel may start once every warp is under way
            refilled = true;
        };
        if (phys >= 0 && phys < p.num_blocks) {
            const uint32_t kbase = smem_u32(wring + s * C::kStageBytes);
            const uint32_t vbase = kbase + C::kTileBytes;
            const int k0 = (j0 + jl) * kBlockSize;  // key position of the block's first row
            const int rem = ctx - k0;               // rows of the block inside the context (>= 1)
            float sc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kbase + swz((mi & 1) * 8 + (lane & 7), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816(sc[nt], a0, a1, a2, a3, qa[nt][ks][0], qa[nt][ks][1]);
            }
            // rows of V past the context may hold any bits (even NaN): zero them in registers
            uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
            if (rem < kBlockSize) {
                keep0 = (2 * t4 < rem ? 0x0000ffffu : 0u) | (2 * t4 + 1 < rem ? 0xffff0000u : 0u);
                keep1 = (8 + 2 * t4 < rem ? 0x0000ffffu : 0u) | (9 + 2 * t4 < rem ? 0xffff0000u : 0u);
            }
#if KVC_MULTI_EARLY_REFILL
            // V^T fragments into registers, then the stage goes back to the copy engine before the softmax
            uint32_t va[D / 16][4];
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
                ldsm_x4_t(vbase + swz((mi >> 1) * 8 + (lane & 7), 2 * mt + (mi & 1)), va[mt][0], va[mt][1], va[mt][2],
                          va[mt][3]);
            if (rem < kBlockSize) {  // the context's last block (warp-uniform)
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    va[mt][0] &= keep0;
                    va[mt][1] &= keep0;
                    va[mt][2] &= keep1;
                    va[mt][3] &= keep1;
                }
            }
            // the copy may overwrite the stage only once the warp's reads of it have returned: one register of each
            // ldmatrix folded (a warp issues in order, and an ldmatrix's four registers arrive together), so the
            // refill cannot issue before every read is back (the K fragments were consumed by the S products above)
            uint32_t dep = 0;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) asm volatile("xor.b32 %0, %0, %1;" : "+r"(dep) : "r"(va[mt][0]));
            refill(k, s);
#endif
            uint32_t bh[NT][2], bl[NT][2];
            // every row sees every key of this block (warp-uniform): no mask, and every running maximum is finite
            // once the first update below has run
            const bool all_vis = k0 + kBlockSize - 1 <= (kPrefix ? ctx - 1 : ctx - T);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // keys k0 + g and k0 + g + 8 against rows 2 t4 (+1): visible up to each row's last key
                float x0, x1, x2, x3;
                if (all_vis) {
                    x0 = sc[nt][0] * sl2;
                    x1 = sc[nt][1] * sl2;
                    x2 = sc[nt][2] * sl2;
                    x3 = sc[nt][3] * sl2;
                } else {
                    x0 = k0 + g <= lastk[nt][0] ? sc[nt][0] * sl2 : -INFINITY;
                    x1 = k0 + g <= lastk[nt][1] ? sc[nt][1] * sl2 : -INFINITY;
                    x2 = k0 + g + 8 <= lastk[nt][0] ? sc[nt][2] * sl2 : -INFINITY;
                    x3 = k0 + g + 8 <= lastk[nt][1] ? sc[nt][3] * sl2 : -INFINITY;
                }
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
                // lazy running maxima (as in the decode kernel): they move only when a visible score exceeds them
                // by more than 2^KVC_DEC_LAZY_MAX, so the weights stay <= 2^KVC_DEC_LAZY_MAX
                if (KVC_DEC_LAZY_MAX == 0 || __any_sync(0xffffffffu, mx0 > m_run[nt][0] + KVC_DEC_LAZY_MAX ||
                                                                      mx1 > m_run[nt][1] + KVC_DEC_LAZY_MAX)) {
#pragma unroll
                    for (int sh = 4; sh < 32; sh <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
                    }
                    const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
                    // a row with no visible key so far (m stays -inf) keeps a zero state
                    const float al0 = mn0 == -INFINITY ? 1.f : ex2(m_run[nt][0] - mn0);
                    const float al1 = mn1 == -INFINITY ? 1.f : ex2(m_run[nt][1] - mn1);
                    m_run[nt][0] = mn0;
                    m_run[nt][1] = mn1;
                    l_run[nt][0] *= al0;
                    l_run[nt][1] *= al1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        o[nt][mt][0] *= al0;
                        o[nt][mt][1] *= al1;
                        o[nt][mt][2] *= al0;
                        o[nt][mt][3] *= al1;
                    }
                }
                const float mn0 = m_run[nt][0], mn1 = m_run[nt][1];
                float p0, p1, p2, p3;
                if (all_vis) {
                    p0 = ex2(x0 - mn0);
                    p2 = ex2(x2 - mn0);
                    p1 = ex2(x1 - mn1);
                    p3 = ex2(x3 - mn1);
                } else {
                    p0 = mn0 == -INFINITY ? 0.f : ex2(x0 - mn0);
                    p2 = mn0 == -INFINITY ? 0.f : ex2(x2 - mn0);
                    p1 = mn1 == -INFINITY ? 0.f : ex2(x1 - mn1);
                    p3 = mn1 == -INFINITY ? 0.f : ex2(x3 - mn1);
                }
                // P^T as the B operand in fp16 (split: plus the fp16 residual as a second operand)
                const uint32_t h01 = pack_half2(p0, p1), h23 = pack_half2(p2, p3);
                const float2 f01 = unpack_half2(h01), f23 = unpack_half2(h23);
                bh[nt][0] = movmatrix_trans(h01);
                bh[nt][1] = movmatrix_trans(h23);
                if constexpr (kSplitP) {
                    l_run[nt][0] += p0 + p2;
                    l_run[nt][1] += p1 + p3;
                    bl[nt][0] = movmatrix_trans(pack_half2(p0 - f01.x, p1 - f01.y));
                    bl[nt][1] = movmatrix_trans(pack_half2(p2 - f23.x, p3 - f23.y));
                } else {
                    // the sums take the rounded weights that multiply V, so each output row stays an exact convex
                    // combination of V rows (weights off by at most 2^-11 relative)
                    l_run[nt][0] += f01.x + f23.x;
                    l_run[nt][1] += f01.y + f23.y;
                }
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
#if KVC_MULTI_EARLY_REFILL
                const uint32_t a0 = va[mt][0], a1 = va[mt][1], a2 = va[mt][2], a3 = va[mt][3];
#else
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vbase + swz((mi >> 1) * 8 + (lane & 7), 2 * mt + (mi & 1)), a0, a1, a2, a3);
                a0 &= keep0;
                a1 &= keep0;
                a2 &= keep1;
                a3 &= keep1;
#endif
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_f16_16816(o[nt][mt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                    if constexpr (kSplitP) mma_f16_16816(o[nt][mt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                }
            }
        }
        if (!refilled) refill(k, s);
    }
    if (timed_out) {
        if (lane == 0) {
            atomicOr(p.err, KVC_DEVERR_TIMEOUT);
            // let the copies still in flight land before the ring's memory is reused
            for (int kk = k; kk < min(nmine, k + ST); ++kk)
                mbar_wait_bounded(&wbars[kk % ST], (kk / ST) & 1, kWaitLimitNs / 8);
        }
        // the warp contributes nothing; the rest of the CTA and the cluster go on to the merges
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
        }
    }
    // sums over the 8 lanes that share a row (their keys)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l_run[nt][0] += __shfl_xor_sync(0xffffffffu, l_run[nt][0], sh);
            l_run[nt][1] += __shfl_xor_sync(0xffffffffu, l_run[nt][1], sh);
        }
    // the warp parks its state in its own ring (every copy into it has landed)
    __syncwarp();
    {
        float* wpark = reinterpret_cast<float*>(wring);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = nt * 8 + 2 * t4 + e;
                if (g == 0) {
                    wpark[c] = m_run[nt][e];
                    wpark[RG + c] = l_run[nt][e];
                }
                float* row = wpark + 2 * RG + c * C::kRowStride;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    row[mt * 16 + g] = o[nt][mt][e];
                    row[mt * 16 + g + 8] = o[nt][mt][2 + e];
                }
            }
    }
    __syncthreads();
    // in a cluster every CTA pushes its merged state into its slot of rank 0's inbox with remote stores, once
    // every CTA of the cluster has started (the arrive after the prologue), so rank 0's shared memory is live
    uint32_t slot = 0, remote_bar = 0;
    if (cs > 1) {
        if (!KVC_DEC_EARLY_CLUSTER_WAIT) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        slot = map_to_rank(s_inbox + rank * C::kSlotFloats, 0);
        remote_bar = map_to_rank(inbox_bar, 0);
    }
    const bool push_async = KVC_DEC_ASYNC_PUSH && cs > 1 && rank != 0;
    // the output (or partial) row of query row c of this CTA
    auto out_row = [&](int c) -> int64_t { return q_row(r0 + c); };
    const bool final_out = !kPrefix && p.nclus == 1;  // this cluster's result is the output
    // one thread per (row, 4 dims): the CTA's merged (m, l, acc) from its warps' parked states
    for (int idx = threadIdx.x; idx < rows * (D / 4); idx += blockDim.x) {
        const int c = idx / (D / 4), d = (idx % (D / 4)) * 4;
        constexpr int kRingF = C::kWarpRingBytes / 4;
        const float* park = reinterpret_cast<const float*>(smem);  // warp w's parked state at w * kRingF
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, park[w * kRingF + c]);
        float L = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float* wp = park + w * kRingF;
                if (wp[c] == -INFINITY) continue;  // the warp saw no visible key of this row
                const float f = ex2(wp[c] - M);
                L = fmaf(wp[RG + c], f, L);
                A = fma4(f, *reinterpret_cast<const float4*>(wp + 2 * RG + c * C::kRowStride + d), A);
            }
        }
        if (push_async) {
            st_async_f32x4(slot + 4u * (2 * RG + c * D + d), A, remote_bar);
            if (d == 0) {
                st_async_f32(slot + 4u * c, M, remote_bar);
                st_async_f32(slot + 4u * (RG + c), L, remote_bar);
            }
        } else if (cs > 1) {
            st_cluster_f32x4(slot + 4u * (2 * RG + c * D + d), A);
            if (d == 0) {
                st_cluster_f32(slot + 4u * c, M);
                st_cluster_f32(slot + 4u * (RG + c), L);
            }
        } else if (final_out) {
            store_out4(p.out, p.out_f32, out_row(c) * D + d, scale4(A, L > 0.f ? 1.f / L : 0.f));
        } else {
            const int64_t prow = out_row(c) * p.part_stride + cidx;
            *reinterpret_cast<float4*>(p.part_acc + prow * D + d) = A;
            if (d == 0) {
                p.part_ml[prow * 2 + 0] = M;
                p.part_ml[prow * 2 + 1] = L;
            }
        }
    }
    if (cs == 1) return;
#if KVC_DEC_ASYNC_PUSH
    // the other CTAs have issued their asynchronous pushes and leave; rank 0 waits until their bytes have landed
    // on its inbox barrier and its own slot is written, then merges the slots
    if (rank != 0) return;
    __syncthreads();
    if (!mbar_wait_cluster_bounded(inbox_bar, 0, 4 * kWaitLimitNs)) {
        if (threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
    }
#else
    // rank 0 merges the slots once every CTA has pushed its state (release / acquire); the others leave
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (rank != 0) return;
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
#endif
    for (int idx = threadIdx.x; idx < rows * (D / 4); idx += blockDim.x) {
        const int c = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float M = -INFINITY;
        for (int q = 0; q < cs; ++q)
            if (s_inbox[q * C::kSlotFloats + RG + c] > 0.f) M = fmaxf(M, s_inbox[q * C::kSlotFloats + c]);
        float L = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < cs; ++q) {
            const float* sl = s_inbox + q * C::kSlotFloats;
            const float l = sl[RG + c];
            if (!(l > 0.f)) continue;  // a CTA without visible keys of this row takes no part
            const float f = ex2(sl[c] - M);
            L = fmaf(l, f, L);
            A = fma4(f, *reinterpret_cast<const float4*>(sl + 2 * RG + c * D + d), A);
        }
        if (final_out) {
            store_out4(p.out, p.out_f32, out_row(c) * D + d, scale4(A, L > 0.f ? 1.f / L : 0.f));
        } else {
            const int64_t prow = out_row(c) * p.part_stride + cidx;
            *reinterpret_cast<float4*>(p.part_acc + prow * D + d) = A;
            if (d == 0) {
                p.part_ml[prow * 2 + 0] = M;
                p.part_ml[prow * 2 + 1] = L;
            }
        }
    }
}

// ---- host side ---------------------------------------------------------------------------------------
// n-tiles per warp and row groups for R query rows per unit
static void group_tiles(int D, int R, int* nt, int* nrg) {
    const int maxt = D == 64 ? KVC_MULTI_MAX_TILES64 : 2;  // accumulators: NT * D / 2 floats a lane
    *nt = std::min(maxt, std::max(1, (R + 7) / 8));
    *nrg = (std::max(R, 1) + 8 * *nt - 1) / (8 * *nt);
}

// chunking of nblk blocks per unit for `units` (unit, KV head, row group) triples: about KVC_MULTI_CTAS CTAs per SM
// (one when a CTA needs the SM's registers), chunks a multiple of the warps so that every warp gets the same
// number of blocks; the chunks of a unit form one cluster where they fit one, else clusters of the largest size
static void group_chunks(int D, int nt, int64_t units, int64_t nblk, int sms, int* chunk, int* cluster, int* nclus) {
    const int nw = KVC_MULTI_WARPS;
    const int per_sm = D == 64 && nt <= KVC_MULTI_TWO_CTA_TILES ? KVC_MULTI_CTAS : 1;
    const int64_t per_unit = std::max<int64_t>(1, static_cast<int64_t>(per_sm) * sms / std::max<int64_t>(1, units));
    int64_t c = (std::max<int64_t>(1, nblk) + per_unit - 1) / per_unit;
    c = (c + nw - 1) / nw * nw;
    *chunk = static_cast<int>(std::min<int64_t>(kMultiMaxChunk, c));
    const int nch = static_cast<int>((std::max<int64_t>(1, nblk) + *chunk - 1) / *chunk);
    *cluster = std::min(nch, kMultiMaxCluster);
    *nclus = (nch + *cluster - 1) / *cluster;
}

template <int D, int NT, bool kPrefix>
static cudaError_t launch_group_kernel(const CUtensorMap& tmK, const CUtensorMap& tmV, const GroupKernelParams& p,
                                       dim3 grid, bool pdl, cudaStream_t stream) {
    using C = GroupCfg<D, NT>;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(paged_decode_group_kernel<D, NT, kPrefix>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(C::smem_bytes(kMultiMaxChunk, kMultiMaxCluster)));
    });
    if (err != cudaSuccess) return err;
    return launch(paged_decode_group_kernel<D, NT, kPrefix>, grid, dim3(C::kThreads), C::smem_bytes(p.chunk, p.cs),
                  stream, pdl, static_cast<unsigned>(p.cs), tmK, tmV, p);
}

// the group kernel for head dim D with nt n-tiles per warp
template <int D, bool kPrefix>
static cudaError_t launch_group_nt(int nt, const CUtensorMap& tmK, const CUtensorMap& tmV, const GroupKernelParams& p,
                                   dim3 grid, bool pdl, cudaStream_t stream) {
    if constexpr (D == 64) {
        switch (nt) {
            case 1: return launch_group_kernel<64, 1, kPrefix>(tmK, tmV, p, grid, pdl, stream);
            case 2: return launch_group_kernel<64, 2, kPrefix>(tmK, tmV, p, grid, pdl, stream);
            case 3: return launch_group_kernel<64, 3, kPrefix>(tmK, tmV, p, grid, pdl, stream);
            default: return launch_group_kernel<64, 4, kPrefix>(tmK, tmV, p, grid, pdl, stream);
        }
    } else {
        return nt == 1 ? launch_group_kernel<128, 1, kPrefix>(tmK, tmV, p, grid, pdl, stream)
                       : launch_group_kernel<128, 2, kPrefix>(tmK, tmV, p, grid, pdl, stream);
    }
}

static GroupKernelParams group_params(const DecodeArgs& a, float* part_ml, float* part_acc) {
    GroupKernelParams p;
    p.q = a.q;
    p.block_table = a.block_table;
    p.context_lens = a.context_lens;
    p.group_start = nullptr;
    p.blk_off = nullptr;
    p.out = a.out;
    p.part_ml = part_ml;
    p.part_acc = part_acc;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.q_len = 1;
    p.max_ctx = a.max_context_len;
    p.out_f32 = a.out_f32;
    p.scale_log2 = a.scale * kLog2e;
    return p;
}

// the cascade prefix on the tensor cores (group_tc.cu): head dim 64, groups of up to `rows` query rows
// the tensor-core prefix kernel takes at most 64 query rows (a group's sequences x its G heads)
static bool use_tc_prefix(int D, int rows) { return D == gtc::D && rows >= KVC_PREFIX_TC_MIN_ROWS && rows <= 64; }

// chunking for the tensor-core prefix pass: one CTA per SM over all (group, KV head) pairs, whole 128-key tiles
static void tc_chunks(int64_t units, int64_t nblk, int sms, int* chunk, int* nchunks) {
    const int64_t per_unit = std::max<int64_t>(1, sms / std::max<int64_t>(1, units));
    int64_t c = (std::max<int64_t>(1, nblk) + per_unit - 1) / per_unit;
    c = (c + gtc::kChunkAlign - 1) / gtc::kChunkAlign * gtc::kChunkAlign;
    *chunk = static_cast<int>(std::min<int64_t>(gtc::kMaxChunk, c));
    *nchunks = static_cast<int>((std::max<int64_t>(1, nblk) + *chunk - 1) / *chunk);
}

static gtc::Params tc_params(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                             float* part_ml, float* part_acc, int chunk, int nchunks, int part_stride) {
    gtc::Params p;
    p.q = a.q;
    p.block_table = a.block_table;
    p.group_start = group_start;
    p.blk_off = shared_blocks;
    p.part_ml = part_ml;
    p.part_acc = part_acc;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.chunk = chunk;
    p.nchunks = nchunks;
    p.part_stride = part_stride;
    p.scale_log2 = a.scale * kLog2e;
    return p;
}

// ---- multi-token decode ------------------------------------------------------------------------------
// q_len >= 2 tokens of q_len x G query rows on the tensor-core kernel (multi_tc.cu)
static bool use_multi_tc(int D, int q_len, int G) {
    return g_multi_tc.load(std::memory_order_relaxed) != 0 && q_len >= 2 && mtc::supported(D, q_len * G);
}

cudaError_t multi_plan(int B, int Hq, int Hkv, int D, int max_ctx, int q_len, MultiPlan* plan) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    if (D != 64 && D != 128) return cudaErrorInvalidValue;
    if (use_multi_tc(D, q_len, Hq / Hkv)) {
        mtc::plan(B, Hkv, q_len * (Hq / Hkv), max_ctx, sms, &plan->chunk, &plan->cluster, &plan->nclus);
        plan->stages = 3;
        plan->workspace_bytes =
            plan->nclus > 1 ? partials_bytes(static_cast<size_t>(B) * q_len * Hq * plan->nclus, D) : 0;
        return cudaSuccess;
    }
    int nt, nrg;
    group_tiles(D, q_len * (Hq / Hkv), &nt, &nrg);
    const int64_t nblk = std::max((max_ctx + kBlockSize - 1) / kBlockSize, 1);
    group_chunks(D, nt, static_cast<int64_t>(B) * Hkv * nrg, nblk, sms, &plan->chunk, &plan->cluster, &plan->nclus);
    plan->stages = D != 64 ? KVC_MULTI_STAGES128
                   : nt > KVC_MULTI_TWO_CTA_TILES ? KVC_MULTI_STAGES64_WIDE
                   : nt == 4 && KVC_MULTI_STAGES64 < 3 ? 3 : KVC_MULTI_STAGES64;
    plan->workspace_bytes =
        plan->nclus > 1 ? partials_bytes(static_cast<size_t>(B) * q_len * Hq * plan->nclus, D) : 0;
    if (q_len == 1) {  // a single new token is the plain decode
        DecodePlan dp;
        cudaError_t e = decode_plan(B, Hq, Hkv, D, max_ctx, 0, &dp);
        if (e != cudaSuccess) return e;
        plan->workspace_bytes = dp.workspace_bytes;
    }
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_multi_d(const DecodeArgs& a, int q_len, const MultiPlan& mp, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    CUtensorMap tmK, tmV;
    cudaError_t e = make_tile_map(&tmK, a.k_cache, D, rows);
    if (e != cudaSuccess) return e;
    e = make_tile_map(&tmV, a.v_cache, D, rows);
    if (e != cudaSuccess) return e;
    const size_t nrow = static_cast<size_t>(a.B) * q_len * a.Hq * mp.nclus;
    float* part_ml = static_cast<float*>(a.workspace);
    const bool parts = mp.nclus > 1;  // partial states and the combine kernel
    float* part_acc = parts ? partials_acc(part_ml, nrow) : nullptr;
    const int G = a.Hq / a.Hkv;
    if (use_multi_tc(D, q_len, G)) {
        mtc::Params tp;
        tp.q = a.q;
        tp.block_table = a.block_table;
        tp.context_lens = a.context_lens;
        tp.out = a.out;
        tp.part_ml = parts ? part_ml : nullptr;
        tp.part_acc = part_acc;
        tp.err = a.err;
        tp.B = a.B;
        tp.max_blocks = a.max_blocks;
        tp.num_blocks = a.num_blocks;
        tp.Hq = a.Hq;
        tp.Hkv = a.Hkv;
        tp.G = G;
        tp.q_len = q_len;
        tp.max_ctx = a.max_context_len;
        tp.out_f32 = a.out_f32;
        tp.chunk = mp.chunk;
        tp.cs = mp.cluster;
        tp.nclus = mp.nclus;
        tp.part_stride = mp.nclus;
        tp.scale_log2 = a.scale * kLog2e;
        e = mtc::launch(tmK, tmV, tp, q_len * G, launch_overlap() != 0, stream);
    } else {
        GroupKernelParams p = group_params(a, parts ? part_ml : nullptr, part_acc);
        p.q_len = q_len;
        p.chunk = mp.chunk;
        p.cs = mp.cluster;
        p.nclus = mp.nclus;
        p.part_stride = mp.nclus;
        int nt, nrg;
        group_tiles(D, q_len * p.G, &nt, &nrg);
        e = launch_group_nt<D, false>(nt, tmK, tmV, p, dim3(nrg * mp.nclus * mp.cluster, a.Hkv, a.B),
                                      launch_overlap() != 0, stream);
    }
    if (e != cudaSuccess || !parts) return e;
    // several clusters per context: merge their partial states
    CombineParams c;
    c.part_ml = part_ml;
    c.part_acc = part_acc;
    c.context_lens = a.context_lens;
    c.blk_off = nullptr;
    c.out = a.out;
    c.err = a.err;
    c.Hq = a.Hq;
    c.part_stride = mp.nclus;
    c.part_base = 0;
    c.bpc = mp.cluster * mp.chunk;
    c.max_blocks = a.max_blocks;
    c.max_ctx = a.max_context_len;
    c.out_f32 = a.out_f32;
    c.prefix_chunk = 0;
    c.cascade = 1;  // every output row comes from the parts
    c.q_len = q_len;
    c.early_release = 0;
    return launch_combine(c, D, a.B * q_len, stream);
}

cudaError_t launch_multi(const DecodeArgs& a, int q_len, cudaStream_t stream) {
    MultiPlan mp;
    cudaError_t e = multi_plan(a.B, a.Hq, a.Hkv, a.D, a.max_context_len, q_len, &mp);
    if (e != cudaSuccess) return e;
    if (mp.workspace_bytes > a.workspace_bytes) return cudaErrorInvalidValue;
    if (q_len == 1) return launch_decode(a, stream);  // q [B][1][Hq][D] is the plain decode's q
    switch (a.D) {
        case 64: return launch_multi_d<64>(a, q_len, mp, stream);
        case 128: return launch_multi_d<128>(a, q_len, mp, stream);
        default: return cudaErrorInvalidValue;
    }
}

// ---- cascade ----------------------------------------------------------------------------------------
cudaError_t cascade_plan(int B, int Hq, int Hkv, int D, int max_ctx, int n_groups, int max_shared_blocks,
                         CascadePlan* plan) {
    cudaError_t e = decode_plan(B, Hq, Hkv, D, max_ctx, 0, &plan->suffix);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    // prefix rows: up to kMaxGroupSize sequences x G heads per (group, KV head)
    int nt, nrg;
    group_tiles(D, kMaxGroupSize * (Hq / Hkv), &nt, &nrg);
    if (use_tc_prefix(D, kMaxGroupSize * (Hq / Hkv))) {
        tc_chunks(static_cast<int64_t>(std::max(n_groups, 1)) * Hkv, max_shared_blocks, sms, &plan->chunk,
                  &plan->nchunks);
        plan->cluster = 1;
    } else {
        group_chunks(D, nt, static_cast<int64_t>(std::max(n_groups, 1)) * Hkv * nrg, max_shared_blocks, sms,
                     &plan->chunk, &plan->cluster, &plan->nchunks);
    }
    if (max_shared_blocks <= 0) plan->nchunks = 0;
    plan->part_stride = plan->nchunks + plan->suffix.num_parts;
    const int64_t saved = static_cast<int64_t>(std::max(B - n_groups, 0)) * std::max(max_shared_blocks, 0);
    plan->plain = saved < g_cascade_min_saved.load(std::memory_order_relaxed);
    // the plain decode over the full contexts is the suffix plan without block offsets: its workspace
    // (plan->suffix.workspace_bytes) never exceeds the cascade's, so one size serves both routes
    plan->workspace_bytes = plan->plain ? plan->suffix.workspace_bytes
                                        : partials_bytes(static_cast<size_t>(B) * Hq * plan->part_stride, D);
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_cascade_d(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                                    int n_groups, const CascadePlan& cp, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    const size_t nrow = static_cast<size_t>(a.B) * a.Hq * cp.part_stride;
    float* part_ml = static_cast<float*>(a.workspace);
    float* part_acc = partials_acc(part_ml, nrow);
    cudaError_t e = cudaSuccess;
    // 1. the shared prefixes, each read once per group: prefix parts 0 .. nchunks-1 (one per cluster)
    if (cp.nchunks > 0 && n_groups > 0) {
        CUtensorMap tmK, tmV;
        e = make_tile_map(&tmK, a.k_cache, D, rows);
        if (e != cudaSuccess) return e;
        e = make_tile_map(&tmV, a.v_cache, D, rows);
        if (e != cudaSuccess) return e;
        if (use_tc_prefix(D, kMaxGroupSize * (a.Hq / a.Hkv))) {  // as cascade_plan chose
            const gtc::Params tp = tc_params(a, group_start, shared_blocks, part_ml, part_acc, cp.chunk, cp.nchunks,
                                             cp.part_stride);
            e = gtc::launch(tmK, tmV, tp, dim3(cp.nchunks, a.Hkv, n_groups), launch_overlap() != 0, stream);
        } else {
            GroupKernelParams p = group_params(a, part_ml, part_acc);
            p.group_start = group_start;
            p.blk_off = shared_blocks;
            p.chunk = cp.chunk;
            p.cs = cp.cluster;
            p.nclus = cp.nchunks;
            p.part_stride = cp.part_stride;
            int nt, nrg;
            group_tiles(D, kMaxGroupSize * p.G, &nt, &nrg);
            e = launch_group_nt<D, true>(nt, tmK, tmV, p, dim3(nrg * cp.nchunks * cp.cluster, a.Hkv, n_groups),
                                         launch_overlap() != 0, stream);
        }
        if (e != cudaSuccess) return e;
    }
    // 2. every sequence past its shared blocks: suffix parts from nchunks on
    e = launch_decode_suffix(a, cp.suffix, shared_blocks, cp.nchunks, cp.part_stride, part_ml, part_acc, stream);
    if (e != cudaSuccess) return e;
    // 3. merge both into the output
    CombineParams c;
    c.part_ml = part_ml;
    c.part_acc = part_acc;
    c.context_lens = a.context_lens;
    c.blk_off = shared_blocks;
    c.out = a.out;
    c.err = a.err;
    c.Hq = a.Hq;
    c.part_stride = cp.part_stride;
    c.part_base = cp.nchunks;
    c.bpc = cp.suffix.blocks_per_split;
    c.max_blocks = a.max_blocks;
    c.max_ctx = a.max_context_len;
    c.out_f32 = a.out_f32;
    c.prefix_chunk = cp.cluster * cp.chunk;  // shared blocks per prefix part
    c.cascade = 1;
    c.q_len = 1;
    c.early_release = 0;
    return launch_combine(c, D, a.B, stream);
}

cudaError_t launch_cascade(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                           int n_groups, int max_shared_blocks, cudaStream_t stream) {
    CascadePlan cp;
    cudaError_t e = cascade_plan(a.B, a.Hq, a.Hkv, a.D, a.max_context_len, n_groups, max_shared_blocks, &cp);
    if (e != cudaSuccess) return e;
    if (cp.workspace_bytes > a.workspace_bytes) return cudaErrorInvalidValue;
    if (cp.plain) return launch_decode(a, stream);  // the same result, every block read per sequence
    switch (a.D) {
        case 64: return launch_cascade_d<64>(a, group_start, shared_blocks, n_groups, cp, stream);
        case 128: return launch_cascade_d<128>(a, group_start, shared_blocks, n_groups, cp, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
