// Multi-token decode on the 5th-generation tensor cores of sm_103a, head dim 64: the q_len new tokens of a sequence
// attend over its paged cache at once, causally among themselves (token t sits at position ctx - q_len + t and sees
// keys 0 .. ctx - q_len + t).  Speculative-decoding paragraph of "Tornar a inferência barata" (neuralialabs.com):
// the drafted tokens are verified in one pass over their positions; the result definition is the plain decode's
// ("La caché de claves y valores", gustavoai.dev) row by row, and the chunk merge is the FlashAttention article's
// rescaling rule ("Was ist der mathematische Aspekt von Softmax?").
//
// Orientation: the keys are the M = 128 side of both products, so that every key of a 128-key tile (8 paged blocks)
// has a TMEM lane and a softmax thread of its own, and the R = q_len x G query rows of a (sequence, KV head), at
// most 64, are the N side:
//   S^T(j) = K(j) Q^T     M = 128 keys x N = NR rows (R rounded up to 16, 32 or 64), K = 64 dims; K and Q K-major
//                         in shared memory (128-byte swizzle), fp32 in TMEM buffer j % 2
//   softmax               thread = key: its NR scores, the causal limit of each row, a lazy running maximum per row
//                         kept in shared memory (it moves only when a score exceeds it by 2^8; then O^T is
//                         rescaled in TMEM), P^T written to shared memory as one 128-byte row per key: the fp16 high
//                         parts of the rows' weights, then their fp16 residuals
//   O^T += V(j)^T P^T(j)  M = 128 x N = 2 NR, K = 128 keys; A = V^T MN-major (dims 0-63 from the V tile, and a
//                         constant tile whose row 64 is all ones, so that row 64 of O^T accumulates the weight sums
//                         with the same rescaling), B = P^T MN-major; columns [0, NR) take the high parts, [NR, 2 NR)
//                         the residuals, summed at the end (~fp32 weights, as the mma.sync decode paths keep)
// Warps 0-3 run the softmax (warp w holds TMEM lane quarter w), lane 0 of warp 4 issues the products, warp 5 the TMA
// copies (8 paged blocks of K and 8 of V per tile, three tiles in flight).  A CTA takes a chunk of the context; the
// CTAs of a thread-block cluster (consecutive chunks of one (sequence, KV head)) push their (m, l, acc) into rank 0's
// shared memory with st.async, and rank 0 writes the output, or a partial state where a context needs several
// clusters (merged by the combine kernel).  Every wait is bounded: a timeout sets an error bit and drains the CTA.
#include "multi_tc.h"
#include "tcgen05.cuh"

namespace kvc {
namespace mtc {

constexpr int kKeys = 128;                   // keys per tile: the products' M, one TMEM lane each
constexpr int kSoftWarps = 16;               // 4 per TMEM lane quarter, each on a quarter of the query rows
constexpr int kMmaWarp = kSoftWarps;
constexpr int kLoadKWarp = kSoftWarps + 1;  // copies the K tiles
constexpr int kLoadVWarp = kSoftWarps + 2;  // copies the V tiles
constexpr int kThreads = (kSoftWarps + 3) * 32;
constexpr int kMaxStages = 4;
constexpr int kTileBytes = kKeys * 128;      // 128 keys x 64 fp16: one K or V tile, 16 KiB
constexpr int kBoxBytes = kBlockSize * 128;  // the rows of one paged block, 2 KiB
constexpr float kRescaleLog2 = 8.f;          // weights stay below 2^8, far inside fp16
constexpr uint32_t kTmemCols = 256;          // S^T buffers at columns 0 and 64, O^T from column 128 (2 NR columns)
constexpr int kTmemS = 64;
constexpr int kTmemO = 128;
constexpr int kSmemLimit = 227 * 1024;

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

template <int NR>
struct Geom {
    // K and V rings: a K tile is free once its S^T product is done, a V tile once its P V product is
    static constexpr int KS = 4;
    static constexpr int VS = NR == 64 ? 3 : 4;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = KS * kTileBytes;
    static constexpr int kPBytes = NR == 64 ? 2 * kTileBytes : kTileBytes;  // P^T (high parts, then residuals)
    static constexpr int kPOff = kVOff + VS * kTileBytes;                  // two P^T buffers (tile parity)
    static constexpr int kOnesOff = kPOff + 2 * kPBytes;
    static constexpr int kQOff = kOnesOff + kTileBytes;
    static constexpr int kBarOff = kQOff + NR * 128;
    static constexpr int kMiscOff = kBarOff + 256;  // m[64], l[64], wmax[4][64], flags[2][16]
    static constexpr int kIdsOff = kMiscOff + (2 * 64 + 4 * 64 + 32) * 4;
    static constexpr int kSlotFloats = NR * (2 + D);  // a pushed state: m[NR], l[NR], acc[NR][D]
    static constexpr size_t smem_bytes(int chunk, int cs) {
        return static_cast<size_t>(kIdsOff) + align16(4 * chunk) + static_cast<size_t>(cs - 1) * kSlotFloats * 4 +
               1024;
    }
    static_assert(kBarOff % 1024 == 0, "the query tile is 1024-byte aligned");
    static_assert(NR * D * 4 <= kPBytes, "the epilogue's acc rows fit the P^T region");
};

__host__ __device__ constexpr int nr_of(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : 64; }

// byte offset of 16-byte chunk c (0..7) of row `row` in a 1024-byte aligned tile of 128-byte rows, 128-byte
// swizzle (the layout TMA writes and the MMA reads)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

// Wait for a phase; gives up when another thread of the CTA has given up (abort flag) or after the limit, in which
// case it raises the flag itself.  The waits of this kernel sit on its per-tile chain (each hands a tile from one
// warp role to the next), so the thread polls instead of sleeping.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// N consecutive columns of this lane's TMEM row (N = 4, 8 or 16), loaded and stored
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&x)[N]) {
    if constexpr (N == 4) {
        tmem_ld4(taddr, x);
    } else if constexpr (N == 8) {
        tmem_ld8(taddr, x);
    } else {
        tmem_ld16(taddr, x);
    }
}
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&x)[N]) {
    if constexpr (N == 4) {
        tmem_st4(taddr, x);
    } else if constexpr (N == 8) {
        tmem_st8(taddr, x);
    } else {
        tmem_st16f(taddr, x);
    }
}
// N / 2 words of packed fp16 pairs (columns col .. col + N - 1, col a multiple of N) into row `row` of a swizzled
// tile of 128-byte rows
template <int N>
__device__ __forceinline__ void st_half_cols(uint8_t* tile, int row, int col, const uint32_t (&w)[N / 2]) {
    if constexpr (N == 4) {
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(smem_u32(tile + sw128(row, col >> 3) + (col & 7) * 2)),
                     "r"(w[0]), "r"(w[1])
                     : "memory");
    } else {
#pragma unroll
        for (int c = 0; c < N / 8; ++c)
            *reinterpret_cast<uint4*>(tile + sw128(row, (col >> 3) + c)) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
    multi_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const Params p) {
    using Gm = Geom<NR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int KS = Gm::KS, VS = Gm::VS;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::kBarOff);
    uint64_t* k_full = bars;                     // [KS] the K tile landed
    uint64_t* k_empty = k_full + kMaxStages;     // [KS] S^T of the stage's tile done: the stage may be refilled
    uint64_t* v_full = k_empty + kMaxStages;     // [VS] the V tile landed
    uint64_t* v_empty = v_full + kMaxStages;     // [VS] P V of the stage's tile done
    uint64_t* s_full = v_empty + kMaxStages;     // [2] S^T of the buffer's current tile in TMEM
    uint64_t* p_full = s_full + 2;    // [2] P^T of the buffer's current tile written (one arrival per softmax warp)
    uint64_t* o_full = p_full + 2;    // [2] P V of the buffer's current tile done (P^T buffer j % 2 free again)
    uint64_t* o_last = o_full + 2;    // P V of the last tile done
    uint64_t* fin = o_last + 1;       // every product issued done
    uint64_t* inbox_bar = fin + 1;    // rank 0: the other CTAs' states have landed
    uint64_t* xsync = inbox_bar + 1;  // [2] the softmax warps' exchanges within a tile (one arrival per warp)
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(xsync + 2);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    float* m_s = reinterpret_cast<float*>(smem + Gm::kMiscOff);  // running maximum per row (epilogue)
    float* l_s = m_s + 64;                                        // weight sum per row (epilogue)
    float* wmax = l_s + 64;                                       // [lane quarter][row] tile maxima (slow path)
    int* flags = reinterpret_cast<int*>(wmax + 4 * 64);           // [tile parity][softmax warp]
    int* s_ids = reinterpret_cast<int*>(smem + Gm::kIdsOff);      // the chunk's physical block ids
    float* s_inbox = reinterpret_cast<float*>(smem + Gm::kIdsOff + align16(4 * p.chunk));
    uint8_t* ps = smem + Gm::kPOff;  // P^T buffers at ps and ps + kPBytes
    uint8_t* ones = smem + Gm::kOnesOff;
    uint8_t* qs = smem + Gm::kQOff;
    float* E = reinterpret_cast<float*>(ps);  // epilogue: this CTA's acc rows [R][D] (P^T is no longer read)
    auto kst = [&](int s) { return smem + Gm::kKOff + s * kTileBytes; };
    auto vst = [&](int s) { return smem + Gm::kVOff + s * kTileBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cs = p.cs;
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;  // == blockIdx.x % cs
    const int cidx = blockIdx.x / cs;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int T = p.q_len, G = p.G, R = T * G;
    // every CTA of a cluster sees the same (sequence, KV head): the exits below are uniform over the cluster
    const int ctx = p.context_lens[b];
    if (ctx < T || ctx > p.max_blocks * kBlockSize || ctx > p.max_ctx) {
        grid_dependency_wait();
        if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
        // with several clusters per context the combine kernel writes the zeros
        if (p.nclus == 1 && rank == 0)
            for (int e = threadIdx.x; e < R * D; e += kThreads) {
                const int r = e / D;
                store_out(p.out, p.out_f32,
                          ((static_cast<int64_t>(b) * T + r / G) * p.Hq + kvh * G + r % G) * D + e % D, 0.f);
            }
        return;
    }
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    if (cidx * cs * p.chunk >= nblk) {  // the whole cluster is past this context
        leave_before_dependency_wait();
        return;
    }
    // this CTA's blocks [j0, j0 + n); a CTA of a live cluster may have none and still takes part in its merge
    const int j0 = blockIdx.x * p.chunk;
    const int n = max(0, min(nblk, j0 + p.chunk) - j0);
    const int nt = (n + kTileBlocks - 1) / kTileBlocks;
    const uint32_t push_bytes = static_cast<uint32_t>(R * D * 4 + R * 8);

    // ---- prologue: barriers, tensor memory, the chunk's block ids, the ones tile ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kSoftWarps);
        }
        mbar_init(&o_full[0], 1);
        mbar_init(&o_full[1], 1);
        mbar_init(o_last, 1);
        mbar_init(fin, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&xsync[i], kSoftWarps);
        if (cs > 1) mbar_init(inbox_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
        // the one arrival of the inbox phase, with the bytes it waits for (they may land before or after it)
        if (cs > 1 && rank == 0) mbar_arrive_expect_tx(inbox_bar, static_cast<uint32_t>(cs - 1) * push_bytes);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks + j0;
    for (int k = threadIdx.x; k < n; k += kThreads) s_ids[k] = table[k];
    // the ones tile: row (key) k holds 1.0 at element 0 of its 64-element row, i.e. row 64 of the V^T operand
    // (element 0 sits in 16-byte chunk 0 ^ (k & 7) after the swizzle); everything else is zero
    for (int i = threadIdx.x; i < kTileBytes / 16; i += kThreads) {
        const int k = i >> 3, c = i & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c == (k & 7)) v.x = 0x3C00u;  // fp16 1.0 in the low half
        reinterpret_cast<uint4*>(ones)[i] = v;
    }
    fence_proxy_async_smem();  // the ones tile is read by the tensor cores (async proxy)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    // announces that this CTA has started; the matching wait comes before the first push into rank 0
    if (cs > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // the K (or V) copies of key tile t (the whole load warp): lane i < 8 copies block i of the tile, if its id is in
    // range, as a 16-row box into its slot of the tile; lane 0 first announces the bytes on the stage's barrier
    const uint64_t policy = l2_policy_evict_first();
    auto load_tile = [&](int t, bool v) {
        const int s = v ? t % VS : t % KS;
        uint64_t* bar = v ? &v_full[s] : &k_full[s];
        const int bi = t * kTileBlocks + lane;
        const int phys = lane < kTileBlocks && bi < n ? s_ids[bi] : -1;
        const bool in = phys >= 0 && phys < p.num_blocks;
        if (!v && lane < kTileBlocks && bi < n && !in) atomicOr(p.err, KVC_DEVERR_BLOCK_ID);  // its keys are masked
        const uint32_t bytes = static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, in))) * kBoxBytes;
        if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
        __syncwarp();
        if (in)
            tma_load_2d((v ? vst(s) : kst(s)) + lane * kBoxBytes, v ? &tmV : &tmK, bar, 0,
                        (phys * p.Hkv + kvh) * kBlockSize, policy);
    };
    // the first tiles go out before the dependency wait: the cached history does not depend on the previous kernel
    if (warp == kLoadKWarp || warp == kLoadVWarp) {
        const bool v = warp == kLoadVWarp;
        if (lane == 0) prefetch_tensormap(v ? &tmV : &tmK);
        for (int t = 0; t < min(nt, v ? VS : KS); ++t) load_tile(t, v);
    }
    grid_dependency_wait();  // q and out may belong to the previous kernel
    grid_dependents_launch();
    // every CTA of the cluster has passed its prologue (rank 0's inbox barrier is initialised)
    if (cs > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    // the query tile: row r < R is token r / G, head r % G of this KV head; rows R .. NR - 1 zero
    for (int i = threadIdx.x; i < NR * 8; i += kThreads) {
        const int r = i >> 3, c = i & 7;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < R)
            val = *reinterpret_cast<const uint4*>(
                p.q + ((static_cast<int64_t>(b) * T + r / G) * p.Hq + kvh * G + r % G) * D + c * 8);
        *reinterpret_cast<uint4*>(qs + sw128(r, c)) = val;
    }
    fence_proxy_async_smem();  // visible to the tensor cores
    __syncthreads();

    bool ok = true;
    if (warp == kLoadKWarp || warp == kLoadVWarp) {
        // ================= loads: the remaining K (or V) tiles =================
        const bool v = warp == kLoadVWarp;
        const int NS = v ? VS : KS;
        uint64_t* emp = v ? v_empty : k_empty;
        uint64_t* ful = v ? v_full : k_full;
        int issued = min(nt, NS);
        for (int t = NS; t < nt; ++t) {
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&emp[t % NS], ((t - NS) / NS) & 1, s_abort)))) break;
            load_tile(t, v);
            issued = t + 1;
        }
        // copies still in flight land before the shared memory is released (immediate unless aborted)
        if (lane == 0)
            for (int t = max(0, issued - NS); t < issued; ++t)
                mbar_wait_bounded(&ful[t % NS], (t / NS) & 1, kWaitLimitNs / 8);
    } else if (warp == kMmaWarp) {
        // ================= tensor-core products (one thread) =================
        if (lane == 0 && nt > 0) {
            constexpr uint32_t idS = umma_idesc_f16(kKeys, NR, 0, 0);
            constexpr uint32_t idPV = umma_idesc_f16(kKeys, 2 * NR, 1, 1);
            // descriptors: only the 14-bit start-address field moves (every shared-memory address is below 2^18)
            const uint64_t dQ = umma_smem_desc(smem_u32(qs), 16, 1024);
            // P^T as the MN-major B operand: 8-key groups 1024 bytes apart; with NR = 64 the residual half is the
            // second 64-row atom, one tile further; buffer j % 2 one P^T region further
            const uint64_t dP = umma_smem_desc(smem_u32(ps), kTileBytes, 1024);
            // S^T(j) = K(j) Q^T into buffer j % 2 over 4 steps of 16 dims; the K stage is free once it is done
            auto mma_s = [&](int j) {
                const uint64_t dK = umma_smem_desc(smem_u32(kst(j % KS)), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16_ss(tmem + (j & 1) * kTmemS, dK + ((ks * 32) >> 4), dQ + ((ks * 32) >> 4), idS, ks > 0);
                umma_commit(&s_full[j & 1]);
                umma_commit(&k_empty[j % KS]);
            };
            // O^T += V(j)^T P^T(j) over 8 steps of 16 keys (one paged block each); V^T as the MN-major A operand:
            // dims 0-63 from the V tile, dims 64-127 from the ones tile (the leading byte offset between the two)
            auto mma_pv = [&](int j) {
                const uint32_t va = smem_u32(vst(j % VS));
                const uint64_t dV = umma_smem_desc(va, smem_u32(ones) - va, 1024);
                const uint64_t dPj = dP + static_cast<uint64_t>(((j & 1) * Gm::kPBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk)
                    umma_f16_ss(tmem + kTmemO, dV + ((kk * 2048) >> 4), dPj + ((kk * 2048) >> 4), idPV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&o_full[j & 1]);
                umma_commit(&v_empty[j % VS]);
            };
            // issue each product as soon as it may go: S^T(sj) once K(sj) has landed and buffer sj % 2 is free (the
            // softmax of tile sj - 2 is done, i.e. its P V has been issued); P V(pj) once P^T(pj) is written and V(pj)
            // has landed.  Neither waits for the other.
            int sj = 0, pj = 0;
            uint64_t t_last = global_timer_ns();
            for (uint32_t spin = 1; pj < nt; ++spin) {
                bool progress = false;
                if (sj < nt && sj < pj + 2 && mbar_test(&k_full[sj % KS], (sj / KS) & 1)) {
                    tc_fence_after();
                    mma_s(sj);
                    ++sj;
                    progress = true;
                }
                if (pj < sj && mbar_test(&p_full[pj & 1], (pj >> 1) & 1) &&
                    mbar_test(&v_full[pj % VS], (pj / VS) & 1)) {
                    tc_fence_after();
                    mma_pv(pj);
                    if (pj == nt - 1) umma_commit(o_last);
                    ++pj;
                    progress = true;
                }
                if (progress) {
                    t_last = global_timer_ns();
                } else if ((spin & 63u) == 0u) {
                    if (*s_abort) {
                        ok = false;
                        break;
                    }
                    if (global_timer_ns() - t_last > kWaitLimitNs) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                }
            }
            // every product issued is complete before the tensor memory is released
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, kWaitLimitNs);
            if (!ok) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        }
    } else {
        // ================= softmax: thread = key of the tile (TMEM lane) x a quarter of the rows ===========
        constexpr int NRQ = NR / 4;  // query rows of this warp
        const int qd = warp & 3;     // TMEM lane quarter: keys 32 qd .. 32 qd + 31 of the tile
        const int kq = qd * 32 + lane;
        const int r0 = (warp >> 2) * NRQ;  // rows r0 .. r0 + NRQ - 1
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const float sl2 = p.scale_log2;
        const int last0 = ctx - T;  // the first new token's last visible key
        // running maxima of this warp's rows (base-2 units), the same in every lane and in the 4 warps of the rows;
        // they move only when a score exceeds them by more than 2^8 (always from -inf)
        float m[NRQ];
#pragma unroll
        for (int i = 0; i < NRQ; ++i) m[i] = -INFINITY;
        uint32_t xuse = 0;  // uses of the exchange barriers so far (their phases)
        // the softmax warps meet on exchange barrier i (bounded wait)
        auto exchange = [&](int i) -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(&xsync[i]);
            const bool r = __all_sync(0xffffffffu, wait_or_abort(&xsync[i], (xuse >> i) & 1u, s_abort));
            xuse ^= 1u << i;
            return r;
        };
        for (int j = 0; j < nt; ++j) {
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[j & 1], (j >> 1) & 1, s_abort)))) break;
            tc_fence_after();
            float x[NRQ];
            ld_cols<NRQ>(tmem + (j & 1) * kTmemS + r0 + lane_base, x);
            // this thread's key: row kq & 15 of block kq >> 4 of the tile
            const int blk = j * kTileBlocks + (kq >> 4);
            const int kpos = (j0 + blk) * kBlockSize + (kq & 15);
            const bool valid = blk < n && kpos < ctx && s_ids[blk] >= 0 && s_ids[blk] < p.num_blocks;
            // rows that see the key: token r / G sees keys up to last0 + r / G
            int rmin = valid ? 0 : R;
            if (valid && kpos > last0) rmin = (kpos - last0) * G;
            bool need = false;
#pragma unroll
            for (int i = 0; i < NRQ; ++i) {
                const int r = r0 + i;
                x[i] = r >= rmin && r < R ? x[i] * sl2 : -INFINITY;
                need |= x[i] > m[i] + kRescaleLog2;  // rows >= R keep m = -inf and x = -inf
            }
            // a V row of a key outside the context (past its end, or in a skipped block) may hold any bits; its
            // weight is 0, and 0 times NaN would poison O: zero the row
            if (warp < 4 && __any_sync(0xffffffffu, !valid)) {
                // the V tile must have landed before its rows are overwritten
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&v_full[j % VS], (j / VS) & 1, s_abort)))) break;
                if (!valid) {
                    uint4* vr = reinterpret_cast<uint4*>(vst(j % VS) + kq * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) vr[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            const int wneed = __any_sync(0xffffffffu, need);
            if (lane == 0) flags[(j & 1) * kSoftWarps + warp] = wneed;
            if (!(ok = exchange(0))) break;
            int any_need = 0;
#pragma unroll
            for (int w = 0; w < kSoftWarps; ++w) any_need |= flags[(j & 1) * kSoftWarps + w];
            if (any_need) {
                // (rare) some score exceeds its row's running maximum by more than 2^8: the tile's row maxima, each
                // warp over its 32 keys, then over the 4 lane quarters
#pragma unroll
                for (int i = 0; i < NRQ; ++i) {
                    float v = x[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) wmax[qd * 64 + r0 + i] = v;
                }
                if (!(ok = exchange(1))) break;
                float al[NRQ];
                bool any_alpha = false;
#pragma unroll
                for (int i = 0; i < NRQ; ++i) {
                    const int r = r0 + i;
                    const float mt = fmaxf(fmaxf(wmax[r], wmax[64 + r]), fmaxf(wmax[128 + r], wmax[192 + r]));
                    al[i] = 1.f;
                    if (mt > m[i] + kRescaleLog2) {
                        al[i] = m[i] == -INFINITY ? 0.f : ex2(m[i] - mt);
                        m[i] = mt;
                    }
                    any_alpha |= al[i] != 1.f;
                }
                // rescale this warp's columns of O^T (lanes 0-63: dims, lane 64: the weight sums; quarter 3 holds
                // only zero rows); warp-uniform, since the factors depend on the rows only
                if (j > 0 && any_alpha && qd < 3) {
                    // O^T is idle: P V of tile j - 1 (and so of every earlier tile) complete, that of tile j not
                    // issued before this warp's arrival
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&o_full[(j - 1) & 1], ((j - 1) >> 1) & 1,
                                                                     s_abort))))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // high parts, then residuals
                        const uint32_t ta = tmem + kTmemO + h * NR + r0 + lane_base;
                        float o[NRQ];
                        ld_cols<NRQ>(ta, o);
#pragma unroll
                        for (int i = 0; i < NRQ; ++i) o[i] *= al[i];
                        st_cols<NRQ>(ta, o);
                    }
                    tmem_wait_st();
                }
            }
            // P^T(j) overwrites P^T(j - 2) in buffer j % 2: P V of tile j - 2 must be done reading it
            if (j > 1 && !(ok = __all_sync(0xffffffffu, wait_or_abort(&o_full[j & 1], ((j - 2) >> 1) & 1, s_abort))))
                break;
            uint8_t* pj = ps + (j & 1) * Gm::kPBytes;
            // the weights of this warp's rows: fp16 high parts in columns r0 .., residuals in columns NR + r0 ..
            // (with NR = 64 the residuals are the second 64-column atom)
            uint32_t hv[NRQ / 2], lv[NRQ / 2];
#pragma unroll
            for (int e = 0; e < NRQ / 2; ++e) {
                const float p0 = x[2 * e] == -INFINITY ? 0.f : ex2(x[2 * e] - m[2 * e]);
                const float p1 = x[2 * e + 1] == -INFINITY ? 0.f : ex2(x[2 * e + 1] - m[2 * e + 1]);
                hv[e] = pack_half2(p0, p1);
                const float2 f = unpack_half2(hv[e]);
                lv[e] = pack_half2(p0 - f.x, p1 - f.y);
            }
            st_half_cols<NRQ>(pj, kq, r0, hv);
            if constexpr (NR == 64)
                st_half_cols<NRQ>(pj + kTileBytes, kq, r0, lv);
            else
                st_half_cols<NRQ>(pj, kq, NR + r0, lv);
            fence_proxy_async_smem();  // P^T and any zeroed V row are read by the tensor cores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[j & 1]);
        }
        // ---- this CTA's state: acc rows (O^T lanes 0-63, high part + residual), weight sums (lane 64), maxima ----
        if (qd == 0 && lane == 0)
#pragma unroll
            for (int i = 0; i < NRQ; ++i) m_s[r0 + i] = m[i];
        if (ok && nt > 0) ok = __all_sync(0xffffffffu, wait_or_abort(o_last, 0, s_abort));
        if (ok && nt > 0 && qd < 3) {
            tc_fence_after();
            float hi[NRQ], lo[NRQ];
            ld_cols<NRQ>(tmem + kTmemO + r0 + lane_base, hi);
            ld_cols<NRQ>(tmem + kTmemO + NR + r0 + lane_base, lo);
#pragma unroll
            for (int i = 0; i < NRQ; ++i) {
                const int r = r0 + i;
                if (r < R) {
                    const float v = hi[i] + lo[i];
                    if (kq < D) E[r * D + kq] = v;
                    else if (kq == D) l_s[r] = v;
                }
            }
        } else if (qd < 3) {
            // no tile (or aborted): an empty state
#pragma unroll
            for (int i = 0; i < NRQ; ++i) {
                const int r = r0 + i;
                if (r < R) {
                    if (kq < D) E[r * D + kq] = 0.f;
                    else if (kq == D) l_s[r] = 0.f;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
    }
    // every TMEM access of the CTA is complete; the allocating warp frees it
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

    // ---- merge: the CTA's state is (m_s, l_s, E); one thread per (row, 4 dims) ----
    auto out_row = [&](int r) -> int64_t { return (static_cast<int64_t>(b) * T + r / G) * p.Hq + kvh * G + r % G; };
    const bool final_out = p.nclus == 1;
    auto emit = [&](int r, int d, float M, float L, float4 A) {
        if (final_out) {
            store_out4(p.out, p.out_f32, out_row(r) * D + d, scale4(A, L > 0.f ? 1.f / L : 0.f));
        } else {
            const int64_t prow = out_row(r) * p.part_stride + cidx;
            *reinterpret_cast<float4*>(p.part_acc + prow * D + d) = A;
            if (d == 0) {
                p.part_ml[prow * 2 + 0] = M;
                p.part_ml[prow * 2 + 1] = L;
            }
        }
    };
    if (cs == 1) {
        for (int idx = threadIdx.x; idx < R * (D / 4); idx += kThreads) {
            const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
            emit(r, d, m_s[r], l_s[r], *reinterpret_cast<const float4*>(E + r * D + d));
        }
        return;
    }
    if (rank != 0) {
        // push the state into slot rank - 1 of rank 0's inbox: m[NR], l[NR], acc[NR][D]; the bytes complete on rank
        // 0's inbox barrier, so nothing else is needed before leaving
        const uint32_t slot = map_to_rank(s_inbox + (rank - 1) * Gm::kSlotFloats, 0);
        const uint32_t rbar = map_to_rank(inbox_bar, 0);
        for (int idx = threadIdx.x; idx < R * (D / 4); idx += kThreads) {
            const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
            st_async_f32x4(slot + 4u * (2 * NR + r * D + d), *reinterpret_cast<const float4*>(E + r * D + d), rbar);
            if (d == 0) {
                st_async_f32(slot + 4u * r, m_s[r], rbar);
                st_async_f32(slot + 4u * (NR + r), l_s[r], rbar);
            }
        }
        return;
    }
    // rank 0: the other CTAs' states (acquire at cluster scope), then the merge with its own
    if (!mbar_wait_cluster_bounded(inbox_bar, 0, 4 * kWaitLimitNs) && threadIdx.x == 0)
        atomicOr(p.err, KVC_DEVERR_TIMEOUT);
    for (int idx = threadIdx.x; idx < R * (D / 4); idx += kThreads) {
        const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
        float M = l_s[r] > 0.f ? m_s[r] : -INFINITY;
        for (int c = 0; c < cs - 1; ++c) {
            const float* sl = s_inbox + c * Gm::kSlotFloats;
            if (sl[NR + r] > 0.f) M = fmaxf(M, sl[r]);
        }
        float L = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        if (l_s[r] > 0.f) {
            const float w = ex2(m_s[r] - M);
            L = l_s[r] * w;
            A = fma4(w, *reinterpret_cast<const float4*>(E + r * D + d), A);
        }
        for (int c = 0; c < cs - 1; ++c) {
            const float* sl = s_inbox + c * Gm::kSlotFloats;
            const float l = sl[NR + r];
            if (!(l > 0.f)) continue;  // a CTA without visible keys of this row takes no part
            const float w = ex2(sl[r] - M);
            L = fmaf(l, w, L);
            A = fma4(w, *reinterpret_cast<const float4*>(sl + 2 * NR + r * D + d), A);
        }
        emit(r, d, M, L, A);
    }
}

// ---- host side ---------------------------------------------------------------------------------------
template <int NR>
static int max_cluster_nr(int chunk) {
    int cs = 8;
    while (cs > 1 && Geom<NR>::smem_bytes(chunk, cs) > static_cast<size_t>(kSmemLimit)) --cs;
    return cs;
}
static int max_cluster(int rows, int chunk) {
    switch (nr_of(rows)) {
        case 16: return max_cluster_nr<16>(chunk);
        case 32: return max_cluster_nr<32>(chunk);
        default: return max_cluster_nr<64>(chunk);
    }
}

void plan(int B, int Hkv, int rows, int max_ctx, int sms, int* chunk, int* cluster, int* nclus) {
    const int64_t nblk = std::max((max_ctx + kBlockSize - 1) / kBlockSize, 1);
    const int64_t units = std::max<int64_t>(1, static_cast<int64_t>(B) * Hkv);
    const int64_t per_unit = std::max<int64_t>(1, sms / units);  // about one CTA per SM
    int64_t c = (nblk + per_unit - 1) / per_unit;
    c = (c + kTileBlocks - 1) / kTileBlocks * kTileBlocks;
    *chunk = static_cast<int>(std::min<int64_t>(kMaxChunk, c));
    const int nch = static_cast<int>((nblk + *chunk - 1) / *chunk);
    *cluster = std::min(nch, max_cluster(rows, *chunk));
    *nclus = (nch + *cluster - 1) / *cluster;
}

template <int NR>
static cudaError_t launch_nr(const CUtensorMap& tmK, const CUtensorMap& tmV, const Params& p, bool pdl,
                             cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(multi_tc_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    });
    if (err != cudaSuccess) return err;
    const size_t smem = Geom<NR>::smem_bytes(p.chunk, p.cs);
    if (smem > static_cast<size_t>(kSmemLimit)) return cudaErrorInvalidValue;
    return kvc::launch(multi_tc_kernel<NR>, dim3(p.nclus * p.cs, p.Hkv, p.B), dim3(kThreads), smem, stream, pdl,
                       static_cast<unsigned>(p.cs), tmK, tmV, p);
}

cudaError_t launch(const CUtensorMap& tmK, const CUtensorMap& tmV, const Params& p, int rows, bool pdl,
                   cudaStream_t stream) {
    if (!supported(D, rows) || p.chunk <= 0 || p.chunk > kMaxChunk || p.chunk % kTileBlocks || p.cs < 1 || p.cs > 8)
        return cudaErrorInvalidValue;
    switch (nr_of(rows)) {
        case 16: return launch_nr<16>(tmK, tmV, p, pdl, stream);
        case 32: return launch_nr<32>(tmK, tmV, p, pdl, stream);
        default: return launch_nr<64>(tmK, tmV, p, pdl, stream);
    }
}

}  // namespace mtc
}  // namespace kvc
