// The cascade decode's shared-prefix pass on the 5th-generation tensor cores of sm_103a, head dim 64: the
// sequences of a group attend over the blocks their block-table rows share (the group kernel's prefix work,
// group.cu, with the products on tcgen05 instead of mma.sync).
//
// A CTA takes one (group, KV head, chunk of the shared blocks); the group's query rows (sequences x G heads, at
// most 64) are the M = 128 rows of the products, the rest zero.  Eighteen warps, as in the one-tile prefill kernel
// (prefill_1t.cu): lane 0 of warp 17 issues the copies, lane 0 of warp 16 the products, warps 0-15 run the
// softmax, four threads per query row (TMEM lane), each on 32 keys of a 128-key tile.  A key tile is 8 paged
// blocks, each a 16-row TMA box into its slot of the tile (the 128-byte swizzle repeats every 8 rows, so the
// boxes compose into the layout of one 128-row tile).  Per tile j:
//   S(j) = Q K(j)^T  M = 128 x N = 128, fp32 in TMEM buffer j % 2
//   softmax          keys in a block whose id is out of range are masked; the running max moves only when it has grown by 2^8 (then O
//                    is rescaled in TMEM); P is written over S as an fp16 high part and residual
//   O += P(j) V(j)   M = 128 x N = 64, P from TMEM, V MN-major in shared memory
// Row quarters that hold no query row only keep the barrier protocol.  Each CTA writes its rows' (m, l, O) as
// one partial state; the combine kernel (decode.cu) merges the chunks.  Every wait is bounded; a timeout sets
// an error bit and drains the CTA.
#include "group_tc.h"
#include "tcgen05.cuh"

namespace kvc {
namespace gtc {

constexpr int kRows = 128;                          // the products' M: one TMEM lane per query row
constexpr int kKeys = 128;                          // keys per tile: N of S, K of P V
constexpr int kTileBlocks = kKeys / kBlockSize;     // 8 paged blocks per key tile
constexpr int kKeyParts = 4;                        // a row's keys of a tile are split over 4 threads
constexpr int kPartKeys = kKeys / kKeyParts;        // 32 keys each
constexpr int kRowWarps = 4 * kKeyParts;            // 4 TMEM lane quarters x 4 key parts
constexpr int kMmaWarp = kRowWarps;
constexpr int kLoadWarp = kRowWarps + 1;
constexpr int kThreads = (kRowWarps + 2) * 32;
constexpr int KS = 4, VS = 4;                       // K and V ring depths
static_assert(KS == VS, "the loads issue K and V of a tile together");
constexpr int kTileBytes = kKeys * 128;             // one K or V tile: 128 rows of 64 fp16, 16 KiB
constexpr int kBoxBytes = kBlockSize * 128;         // one block's rows, 2 KiB
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kRows * 128;
constexpr int kVOff = kKOff + KS * kTileBytes;
constexpr int kBarOff = kVOff + VS * kTileBytes;
constexpr int kXOff = kBarOff + 512;                // row max / row sum exchange: [parity][key part][row]
constexpr int kIdsOff = kXOff + 2 * kKeyParts * kRows * 4;
constexpr int kTmemO = 2 * kKeys;                   // TMEM: S buffers [0, 128) and [128, 256), O [256, 320)
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;                 // P stays below 2^8, far inside fp16
constexpr size_t smem_bytes(int chunk) { return kIdsOff + 4 * static_cast<size_t>(chunk) + 1024; }
static_assert(smem_bytes(kMaxChunk) <= 227 * 1024, "shared memory of one CTA");


// byte offset of 16-byte chunk c (0..7) of row `row` in a 1024-byte aligned tile of 128-byte rows, 128-byte
// swizzle (the layout TMA writes and the MMA reads)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

// Wait for a phase; gives up when another thread of the CTA has given up (abort flag) or after the limit, in
// which case it raises the flag itself.  The waiting thread sleeps in the hardware until the phase completes
// or 20 us pass.
__device__ __forceinline__ bool try_wait_sleep(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) prefix_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* k_full = bars;            // [KS] K tile landed
    uint64_t* k_empty = k_full + KS;    // [KS] S product of the stage's tile done
    uint64_t* v_full = k_empty + KS;    // [VS] V tile landed
    uint64_t* v_empty = v_full + VS;    // [VS] P V product of the stage's tile done
    uint64_t* s_full = v_empty + VS;    // [2] S of the buffer's current tile in TMEM
    uint64_t* p_full = s_full + 2;      // [2] P of the buffer's current tile in TMEM (16 arrivals)
    uint64_t* o_full = s_full + 4;      // P V of the latest tile done
    uint64_t* o_last = s_full + 5;      // P V of the last tile done
    uint64_t* xchg = s_full + 6;        // [4] the 4 warps of a lane quarter have posted (4 arrivals)
    uint64_t* fin = s_full + 10;        // every product issued so far done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_full + 11);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_full + 11) + 1;
    float* xbuf = reinterpret_cast<float*>(smem + kXOff);
    int* s_ids = reinterpret_cast<int*>(smem + kIdsOff);  // the chunk's physical block ids
    uint8_t* qs = smem + kQOff;
    auto kst = [&](int st) { return smem + kKOff + st * kTileBytes; };
    auto vst = [&](int st) { return smem + kVOff + st * kTileBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, kvh = blockIdx.y, u = blockIdx.z;
    // the group: sequences s0 .. s0 + T - 1, whose rows begin with the same nsh blocks (read through the first
    // member's row), every key of them inside every member's context; the exits below are uniform over the CTA
    const int s0 = p.group_start[u];
    const int T = p.group_start[u + 1] - s0;
    if (T < 1) {
        leave_before_dependency_wait();
        return;
    }
    const int nsh = p.blk_off[s0];
    if (T > kMaxGroupSize || nsh < 0 || nsh > p.max_blocks) {
        if (chunk == 0 && kvh == 0 && threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
        leave_before_dependency_wait();
        return;  // the combine kernel writes these sequences' rows
    }
    const int ctx = nsh * kBlockSize, nblk = nsh;  // keys and blocks of the shared prefix
    const int R = T * p.G;                          // query rows, at most kMaxGroupSize x 8 = 64
    const int j0 = chunk * p.chunk;                 // this CTA's blocks [j0, j0 + n) of the shared blocks
    if (j0 >= nblk) {  // the group shares fewer blocks
        leave_before_dependency_wait();
        return;
    }
    const int n = min(nblk, j0 + p.chunk) - j0;
    const int nt = (n + kTileBlocks - 1) / kTileBlocks;  // key tiles
    const int32_t* table = p.block_table + static_cast<int64_t>(s0) * p.max_blocks + j0;
    // row r of the group as a row of q (and of the partials) of Hq heads: sequence s0 + r / G, head r % G
    auto q_row = [&](int r) -> int64_t { return (static_cast<int64_t>(s0) + r / p.G) * p.Hq + kvh * p.G + r % p.G; };

    // ---- prologue: barriers, tensor memory, the chunk's block ids, a zeroed V ring (a V slot no copy fills
    // holds zeros or an earlier tile's rows, never stale bits that a zero weight could turn into NaN) ----
    if (threadIdx.x == 0) {
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], kRowWarps);
        }
        mbar_init(o_full, 1);
        mbar_init(o_last, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&xchg[i], kKeyParts);
        mbar_init(fin, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    for (int k = threadIdx.x; k < n; k += kThreads) s_ids[k] = table[k];
    for (int i = threadIdx.x; i < VS * kTileBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kVOff)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the zeros are ordered before the copies (async proxy) into the ring
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // the copies of key tile t (the whole load warp): lane i < 8 copies block i of the tile, if its id is in
    // range, as a 16-row box into its slot; lane 0 first announces the bytes on the tile's barrier
    const uint64_t policy = l2_policy_evict_first();
    auto load_tile = [&](int t, bool v) {
        uint64_t* bar = v ? &v_full[t % VS] : &k_full[t % KS];
        const int b = t * kTileBlocks + lane;
        const int phys = lane < kTileBlocks && b < n ? s_ids[b] : -1;
        const bool in = phys >= 0 && phys < p.num_blocks;
        if (!v && lane < kTileBlocks && b < n && !in) atomicOr(p.err, KVC_DEVERR_BLOCK_ID);  // its keys are masked
        const uint32_t bytes = static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, in))) * kBoxBytes;
        if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
        __syncwarp();
        if (in)
            tma_load_2d((v ? vst(t % VS) : kst(t % KS)) + lane * kBoxBytes, v ? &tmV : &tmK, bar, 0,
                        (phys * p.Hkv + kvh) * kBlockSize, policy);
    };
    // the first tiles go out before the dependency wait: the cached history does not depend on the previous kernel
    if (warp == kLoadWarp) {
        if (lane == 0) {
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
        for (int t = 0; t < min(nt, KS); ++t) {
            load_tile(t, false);
            load_tile(t, true);
        }
    }
    grid_dependency_wait();  // q may come from the previous kernel
    grid_dependents_launch();
    // the query tile: rows r < R from q, the others zero (row r: 64 fp16 = 8 chunks of 16 bytes, swizzled)
    for (int i = threadIdx.x; i < kRows * 8; i += kThreads) {
        const int r = i >> 3, c = i & 7;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) val = *reinterpret_cast<const uint4*>(p.q + q_row(r) * D + c * 8);
        *reinterpret_cast<uint4*>(qs + sw128(r, c)) = val;
    }
    fence_proxy_async_smem();  // visible to the tensor cores
    __syncthreads();

    if (warp == kLoadWarp) {
        // ================= loads: the remaining key tiles (the whole warp) =================
        int k_issued = min(nt, KS), v_issued = min(nt, VS);
        bool ok = true;
        for (int t = min(nt, KS); ok && t < nt; ++t) {
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&k_empty[t % KS], ((t - KS) / KS) & 1, s_abort)))) break;
            load_tile(t, false);
            k_issued = t + 1;
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(&v_empty[t % VS], ((t - VS) / VS) & 1, s_abort)))) break;
            load_tile(t, true);
            v_issued = t + 1;
        }
        // copies still in flight land before the shared memory is released (immediate unless aborted)
        if (lane == 0) {
            for (int t = max(0, k_issued - KS); t < k_issued; ++t)
                mbar_wait_bounded(&k_full[t % KS], (t / KS) & 1, kWaitLimitNs / 8);
            for (int t = max(0, v_issued - VS); t < v_issued; ++t)
                mbar_wait_bounded(&v_full[t % VS], (t / VS) & 1, kWaitLimitNs / 8);
        }
    } else if (warp == kMmaWarp) {
        // ================= tensor-core products (one thread) =================
        if (lane == 0) {
            constexpr uint32_t idS = umma_idesc_f16(kRows, kKeys, 0, 0);
            constexpr uint32_t idPV = umma_idesc_f16(kRows, D, 0, 1);
            // descriptors built once per operand; only the 14-bit start-address field moves (every shared-memory
            // address is below 2^18, so (address >> 4) never carries into the next field)
            const uint64_t dQ = umma_smem_desc(smem_u32(qs), 16, 1024);
            const uint64_t dK = umma_smem_desc(smem_u32(kst(0)), 16, 1024);
            // V as the MN-major B operand: 8-key groups 1024 bytes apart
            const uint64_t dV = umma_smem_desc(smem_u32(vst(0)), kTileBytes, 1024);
            const uint32_t tO = tmem + kTmemO;
            // S(j) = Q K(j)^T into buffer j % 2 over 4 steps of 16 dims: M = 128 rows, N = 128 keys
            auto mma_s = [&](int j) {
                const uint64_t b0 = dK + static_cast<uint64_t>((j % KS) * (kTileBytes >> 4));
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16_ss(tmem + (j & 1) * kKeys, dQ + ((ks * 32) >> 4), b0 + ((ks * 32) >> 4), idS, ks > 0);
                umma_commit(&s_full[j & 1]);
                umma_commit(&k_empty[j % KS]);
            };
            // O += P(j) V(j): 8 steps of 16 keys, P (high part, then residual) read from TMEM buffer j % 2
            auto mma_pv = [&](int j) {
                const uint64_t v0 = dV + static_cast<uint64_t>((j % VS) * (kTileBytes >> 4));
                const uint32_t tP = tmem + (j & 1) * kKeys;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    const uint64_t b = v0 + ((kk * 2048) >> 4);
                    const uint32_t tPk = tP + (kk >> 1) * kPartKeys + (kk & 1) * 8;
                    umma_f16_ts(tO, tPk, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_f16_ts(tO, tPk + 16, b, idPV, 1u);
                }
                umma_commit(o_full);
                umma_commit(&v_empty[j % VS]);
            };
            bool ok = true;
            for (int j = 0; ok && j < min(nt, 2); ++j) {
                if (!(ok = wait_or_abort(&k_full[j % KS], (j / KS) & 1, s_abort))) break;
                tc_fence_after();
                mma_s(j);
            }
            for (int j = 0; ok && j < nt; ++j) {
                // P(j) V(j) once P(j) is in TMEM and V(j) has landed
                if (!(ok = wait_or_abort(&v_full[j % VS], (j / VS) & 1, s_abort))) break;
                if (!(ok = wait_or_abort(&p_full[j & 1], (j >> 1) & 1, s_abort))) break;
                tc_fence_after();
                mma_pv(j);
                if (j == nt - 1) umma_commit(o_last);
                // S(j + 2) into buffer j % 2 once P(j) V(j) has read P(j) there
                if (j + 2 < nt) {
                    if (!(ok = wait_or_abort(&k_full[(j + 2) % KS], ((j + 2) / KS) & 1, s_abort))) break;
                    if (!(ok = wait_or_abort(o_full, j & 1, s_abort))) break;
                    tc_fence_after();
                    mma_s(j + 2);
                }
            }
            // every product issued is complete before the tensor memory is released
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, kWaitLimitNs);
            if (!ok) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        }
    } else {
        // ================= row warps: softmax and the partial state =================
        // Thread = query row (TMEM lane) x one 32-key part of every tile; the 4 threads of a row (warps wq,
        // wq + 4, wq + 8, wq + 12) agree on the running max through shared memory; O is split over the parts by
        // 32-column chunks (parts 0 and 1).
        const int kp = warp >> 2, wq = warp & 3;
        const int row = wq * 32 + lane;
        if (wq * 32 >= R) {
            // a quarter without query rows: only the barrier protocol (P's 16 arrivals per tile)
            for (int j = 0; j < nt; ++j) {
                if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[j & 1], (j >> 1) & 1, s_abort))) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[j & 1]);
            }
        } else {
            const int lastk = ctx - 1;  // every shared key is inside every member's context
            const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
            const uint32_t tSp = tmem + kp * kPartKeys + lane_base;  // this part's columns of S / P (buffer 0)
            const bool owns_o = kp * 32 < D;                         // O columns [32 kp, 32 kp + 32)
            const uint32_t tOp = tmem + kTmemO + kp * 32 + lane_base;
            uint64_t* xq = &xchg[wq];
            const float sl2 = p.scale_log2;
            const bool neg_scale = sl2 < 0.f;  // then the largest scaled score comes from the smallest raw one
            const float fill = neg_scale ? INFINITY : -INFINITY;
            float m_used = -INFINITY, l = 0.f;  // l: this part's share of the row sum
            bool ok = true;
            for (int j = 0; j < nt; ++j) {
                ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[j & 1], (j >> 1) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                const uint32_t tS = tSp + (j & 1) * kKeys;
                float s[kPartKeys];
                tmem_ld32(tS, s);
                // this part's 32 keys are blocks jb and jb + 1 of the chunk
                const int jb = j * kTileBlocks + 2 * kp;
                const int k0 = (j0 + jb) * kBlockSize;  // its first key position
                const bool b0ok = jb < n && s_ids[jb] >= 0 && s_ids[jb] < p.num_blocks;
                const bool b1ok = jb + 1 < n && s_ids[jb + 1] >= 0 && s_ids[jb + 1] < p.num_blocks;
                const bool masked = k0 + kPartKeys - 1 > lastk || !b0ok || !b1ok;
                float ext = fill;
                if (masked) {
#pragma unroll
                    for (int c = 0; c < kPartKeys; ++c) {
                        const bool valid = k0 + c <= lastk && (c < kBlockSize ? b0ok : b1ok);
                        s[c] = valid ? s[c] : fill;
                        ext = neg_scale ? fminf(ext, s[c]) : fmaxf(ext, s[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kPartKeys; ++c) ext = neg_scale ? fminf(ext, s[c]) : fmaxf(ext, s[c]);
                }
                // exchange with the row's other parts (double-buffered by tile parity)
                float* xb = xbuf + (j & 1) * kKeyParts * kRows;
                xb[kp * kRows + row] = ext;
                __syncwarp();
                if (lane == 0) mbar_arrive(xq);
                ok = __all_sync(0xffffffffu, wait_or_abort(xq, j & 1, s_abort));
                if (!ok) break;
#pragma unroll
                for (int q = 0; q < kKeyParts; ++q) {
                    const float other = xb[q * kRows + row];
                    ext = neg_scale ? fminf(ext, other) : fmaxf(ext, other);
                }
                // the tile's largest scaled score (-inf when every key is masked); the running max moves only
                // when it has grown by 2^8 (or from -inf): then l and O are rescaled
                const float mx = ext == fill ? -INFINITY : ext * sl2;
                float alpha = 1.f;
                if (mx > m_used + kRescaleLog2) {  // includes the first finite max (m_used = -inf)
                    alpha = m_used == -INFINITY ? 0.f : ex2(m_used - mx);
                    m_used = mx;
                }
                const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
                // P = 2^(s * scale * log2 e - m) over this part's S columns: high part of keys (2i, 2i + 1) in
                // column i, the residual in column 16 + i; masked keys (s = fill) give 0
#pragma unroll
                for (int c = 0; c < kPartKeys; ++c) s[c] = s[c] == fill ? 0.f : ex2(fmaf(s[c], sl2, neg_m));
                float ls = 0.f;
                uint32_t hv[16], lv[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    const int c = 2 * e2;
                    hv[e2] = pack_half2(s[c], s[c + 1]);
                    const float2 f = unpack_half2(hv[e2]);
                    lv[e2] = pack_half2(s[c] - f.x, s[c + 1] - f.y);
                    ls += s[c] + s[c + 1];
                }
                tmem_st16(tS, hv);
                tmem_st16(tS + 16, lv);
                l = l * alpha + ls;
                // rescale O (rare: the running max moved): it must be idle, i.e. P(j-1) V(j-1) complete; P(j) V(j)
                // is not issued before this thread's arrival below
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f) && owns_o) {
                    ok = __all_sync(0xffffffffu, wait_or_abort(o_full, (j - 1) & 1, s_abort));
                    if (!ok) break;
                    tc_fence_after();
                    float o[32];
                    tmem_ld32(tOp, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tOp, o);
                }
                // a key tile past the shared blocks' end (its unfilled slots): the rows past the end are zeroed, so
                // that whatever they hold cannot turn a zero weight into NaN
                const int vrem = ctx - (j0 + j * kTileBlocks) * kBlockSize;
                if (vrem < kKeys && warp == 0) {
                    ok = __all_sync(0xffffffffu, wait_or_abort(&v_full[j % VS], (j / VS) & 1, s_abort));
                    if (!ok) break;
                    uint8_t* vt = vst(j % VS);
                    for (int e3 = lane; e3 < (kKeys - vrem) * 8; e3 += 32)
                        *reinterpret_cast<uint4*>(vt + sw128(vrem + e3 / 8, e3 % 8)) = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();  // visible to the tensor cores (async proxy)
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[j & 1]);
            }
            // the row sum: this part's share plus the other parts'
            if (ok) {
                float* xb = xbuf + (nt & 1) * kKeyParts * kRows;
                xb[kp * kRows + row] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(xq);
                ok = __all_sync(0xffffffffu, wait_or_abort(xq, nt & 1, s_abort));
                if (ok) {
                    l = 0.f;
#pragma unroll
                    for (int q = 0; q < kKeyParts; ++q) l += xb[q * kRows + row];
                }
            }
            if (ok && owns_o) ok = __all_sync(0xffffffffu, wait_or_abort(o_last, 0, s_abort));
            if (ok && owns_o) {
                tc_fence_after();
                float o[32];
                tmem_ld32(tOp, o);
                if (row < R) {
                    // this chunk's partial state of the row: running max (log2 units), sum, unnormalised O
                    const int64_t prow = q_row(row) * p.part_stride + chunk;
                    float4* dst = reinterpret_cast<float4*>(p.part_acc + prow * D + kp * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    if (kp == 0) {
                        p.part_ml[prow * 2 + 0] = m_used;
                        p.part_ml[prow * 2 + 1] = l;
                    }
                }
            }
        }
    }
    // every TMEM access of the CTA is complete; the allocating warp frees it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t launch(const CUtensorMap& tmK, const CUtensorMap& tmV, const Params& p, dim3 grid, bool pdl,
                   cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(prefix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem_bytes(kMaxChunk)));
    });
    if (err != cudaSuccess) return err;
    if (p.chunk <= 0 || p.chunk > kMaxChunk || p.chunk % kChunkAlign) return cudaErrorInvalidValue;
    return kvc::launch(prefix_tc_kernel, grid, dim3(kThreads), smem_bytes(p.chunk), stream, pdl, 1u, tmK, tmV, p);
}

}  // namespace gtc
}  // namespace kvc
