// Varlen packed prefill attention for sm_103a on the 5th-generation tensor cores, head dim 64: one CTA per
// 128-row query tile.  Same result definition as prefill.cu (xformers article of the "Aufmerksamkeit" feed,
// chatgpz.de, parts 4 and 5; the running-max / exp-sum rule of the FlashAttention article over key tiles).
//
// Design: one CTA per (128-row query tile of a segment, query head); eighteen warps.  Lane 0 of warp 17
// issues every TMA copy, lane 0 of warp 16 every tcgen05.mma; warps 0-15 run the softmax, four threads
// per query row (TMEM lane), each on 32 of the tile's 128 keys.  Per 128-key tile j:
//   S(j) = Q K^T   tcgen05.mma M=128 x N=128, Q and K K-major in shared memory (128-byte swizzle, as TMA
//                  writes them), fp32 accumulator in TMEM buffer j % 2
//   softmax        the row threads read S(j), mask only the parts that cross the causal diagonal or the
//                  segment end, agree on the row max through shared memory, keep the running max until it
//                  has grown by 2^8 (then rescale O in TMEM), and write P(j) over S(j) in fp16 (or as an fp16
//                  high part and residual, so the product keeps ~fp32 weights)
//   O += P(j) V    tcgen05.mma M=128 x N=D with P read from TMEM (the A operand) and V MN-major in shared
//                  memory; O stays in TMEM
// With two S buffers, S(j+1) is computed while the softmax of tile j runs, and S(j+2) is issued into
// buffer j % 2 as soon as P(j) V has read P(j) there.  K and V have rings of their own.  With D = 64 this
// beats two query tiles per CTA (more CTAs, shorter chains); with D = 128 two query tiles sharing each K/V
// tile win (prefill.cu).  Every wait is bounded; a timeout sets an error bit and drains the CTA.
#include <algorithm>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace kvc {
namespace pf1 {

// 1: the softmax's scale-and-shift of unmasked scores in packed fp32x2 multiply-adds (the same rounding per
// lane); 0: one fmaf per score.  Two A/B pairs: seqlens 592/1920/128/3200 x 8 heads causal 49.1 -> 47.2 us,
// non-causal 86.0 -> 83.2; B = 2 x 256, 8 / 2 heads 12.0 -> 11.5.
#ifndef KVC_PREFILL_1T_FMA2
#define KVC_PREFILL_1T_FMA2 1
#endif


constexpr int kPfRows = 128;   // query rows per CTA: the MMA's M, one TMEM lane each
constexpr int kPfCtaRows = kPfRows;
constexpr int kPfKeys = 128;   // keys per K/V tile: N of S, K of P V
constexpr int kPfKeyParts = 4;                        // a row's keys of a tile are split over 4 threads
constexpr int kPfPartKeys = kPfKeys / kPfKeyParts;    // 32 keys each
constexpr int kPfRowWarps = 4 * kPfKeyParts;          // 4 TMEM lane quarters x 4 key parts
constexpr int kPfMmaWarp = kPfRowWarps;       // issues the tensor-core products
constexpr int kPfLoadWarp = kPfRowWarps + 1;  // issues the TMA copies
constexpr int kPfThreads = (kPfRowWarps + 2) * 32;
constexpr uint64_t kPfWaitNs = 1000000000ull;
constexpr float kPfLog2e = 1.4426950408889634f;
constexpr float kPfRescaleLog2 = 8.f;  // P stays below 2^8, far inside fp16

template <int D>
struct PfGeom {
    static constexpr int kChunks = D / 64;                    // 64-dim (128-byte) column chunks
    static constexpr int kKStages = D == 64 ? 4 : 3;          // K ring depth
    static constexpr int kVStages = D == 64 ? 4 : 2;          // V ring depth
    static constexpr int kQChunk = kPfRows * 128;             // 16 KiB
    static constexpr int kKVChunk = kPfKeys * 128;            // 16 KiB
    static constexpr int kQBytes = kChunks * kQChunk;         // the query tile
    static constexpr int kKVBytes = kChunks * kKVChunk;       // one K or V tile
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKVBytes;
    static constexpr int kBarOff = kVOff + kVStages * kKVBytes;
    static constexpr int kXOff = kBarOff + 512;  // row-max / row-sum exchange: [parity][key part][row] floats
    static constexpr int kSmemBytes = kXOff + 2 * kPfKeyParts * kPfRows * 4 + 1024;  // + alignment
    static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
    // TMEM columns: two S buffers [0, 128) and [128, 256) (key tile j in buffer j % 2), O [256, 256 + D).
    // P(j) is written over S(j) once the row warps have read it: key part q's P (fp16, or its high part) in
    // columns [32q, 32q + 16) of the buffer, the residuals of the split form in [32q + 16, 32q + 32).
    static constexpr int kTmemO = 2 * kPfKeys;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kTmemO + D <= 512, "tensor memory");
};

struct PrefillKernelParams {
    const int32_t* cu_seqlens;
    void* out;
    unsigned* err;
    int nseq, total_tokens, tiles_per_seq, Hq, Hkv, G, causal, out_f32;
    float scale_log2;
};

// byte offset of 16-byte chunk c (0..7) of row `row` in a 1024-byte aligned tile of 128-byte rows, 128-byte
// swizzle (the layout TMA writes and the MMA reads)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// acc + the two fp16 halves of h (each converted exactly), as two rounded fp32 additions
__device__ __forceinline__ float add_f16x2_to_f32(uint32_t h, float acc) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %0, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(h));
    return acc;
}

// Wait for a phase; gives up when another thread of the CTA has given up (abort flag) or after the limit,
// in which case it raises the flag itself.  The waiting thread sleeps in the hardware until the phase
// completes or 20 us pass, so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool pf_try_wait_sleep(uint64_t* bar, uint32_t parity) {
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
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (pf_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kPfWaitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

template <int D, bool kSplitP>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV,
                                                                const PrefillKernelParams p) {
    using Geo = PfGeom<D>;
    constexpr int KS = Geo::kKStages, VS = Geo::kVStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kBarOff);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;                    // [KS] K tile landed
    uint64_t* k_empty = k_full + KS;                // [KS] S product of the stage's tile done
    uint64_t* v_full = k_empty + KS;                // [VS] V tile landed
    uint64_t* v_empty = v_full + VS;                // [VS] P V product of the stage's tile done
    uint64_t* s_full = v_empty + VS;                // [2] S of the buffer's current tile in TMEM
    uint64_t* p_full = s_full + 2;                  // [2] P of the buffer's current tile in TMEM (16 arrivals)
    uint64_t* o_full = s_full + 4;                  // P V of the latest tile done
    uint64_t* o_last = s_full + 5;                  // P V of the last tile done
    uint64_t* xchg = s_full + 6;                    // [4] the 4 warps of a lane quarter have posted (4 arrivals)
    uint64_t* fin = s_full + 10;                    // every product issued so far done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_full + 11);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_full + 11) + 1;
    float* xbuf = reinterpret_cast<float*>(smem + Geo::kXOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // heaviest causal row blocks first: block index = ((last row block - row block) * nseq + segment) * Hq + head
    const int per_block = p.nseq * p.Hq;
    const int tile = p.tiles_per_seq - 1 - static_cast<int>(blockIdx.x / per_block);
    const int seg = static_cast<int>(blockIdx.x % per_block) / p.Hq, h = static_cast<int>(blockIdx.x % per_block) % p.Hq;
    const int hk = h / p.G;

    const int beg = p.cu_seqlens[seg], end = p.cu_seqlens[seg + 1];
    const int len = end - beg;
    if (beg < 0 || len < 0 || end > p.total_tokens) {
        if (threadIdx.x == 0 && tile == 0 && h == 0) atomicOr(p.err, KVC_DEVERR_SEQLENS);
        return;
    }
    if (tile == 0 && h == 0 && threadIdx.x == 0 && len > p.tiles_per_seq * kPfCtaRows)
        atomicOr(p.err, KVC_DEVERR_SEQLENS);  // rows past max_seqlen are not computed
    const int r0 = tile * kPfCtaRows;
    if (r0 >= len) return;
    const int nt = ((p.causal ? min(len, r0 + kPfRows) : len) + kPfKeys - 1) / kPfKeys;  // key tiles

    uint8_t* qs = smem + Geo::kQOff;
    auto kst = [&](int st) { return smem + Geo::kKOff + st * Geo::kKVBytes; };
    auto vst = [&](int st) { return smem + Geo::kVOff + st * Geo::kKVBytes; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
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
            mbar_init(&p_full[b], kPfRowWarps);
        }
        mbar_init(o_full, 1);
        mbar_init(o_last, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&xchg[i], kPfKeyParts);
        mbar_init(fin, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, Geo::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == kPfLoadWarp) {
        // ================= loads: every TMA copy (one thread) =================
        if (lane == 0) {
            auto load_k = [&](int t) {
                uint64_t* bar = &k_full[t % KS];
                mbar_arrive_expect_tx(bar, Geo::kKVBytes);
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
                    tma_load_3d(kst(t % KS) + c * Geo::kKVChunk, &tmK, bar, c * 64, hk, beg + t * kPfKeys);
            };
            auto load_v = [&](int t) {
                uint64_t* bar = &v_full[t % VS];
                mbar_arrive_expect_tx(bar, Geo::kKVBytes);
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
                    tma_load_3d(vst(t % VS) + c * Geo::kKVChunk, &tmV, bar, c * 64, hk, beg + t * kPfKeys);
            };
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            mbar_arrive_expect_tx(q_full, Geo::kQBytes);
#pragma unroll
            for (int c = 0; c < Geo::kChunks; ++c) tma_load_3d(qs + c * Geo::kQChunk, &tmQ, q_full, c * 64, h, beg + r0);
            // tile t goes into the stage of tile t - stages once that tile's product is done
            int k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int t = 0; ok && t < nt; ++t) {
                if (t >= KS && !(ok = pf_wait(&k_empty[t % KS], ((t - KS) / KS) & 1, s_abort))) break;
                load_k(t);
                k_issued = t + 1;
                if (t >= VS && !(ok = pf_wait(&v_empty[t % VS], ((t - VS) / VS) & 1, s_abort))) break;
                load_v(t);
                v_issued = t + 1;
            }
            // copies still in flight land before the shared memory is released (immediate unless aborted:
            // the products consumed every tile)
            mbar_wait_bounded(q_full, 0, kPfWaitNs / 8);
            for (int t = max(0, k_issued - KS); t < k_issued; ++t)
                mbar_wait_bounded(&k_full[t % KS], (t / KS) & 1, kPfWaitNs / 8);
            for (int t = max(0, v_issued - VS); t < v_issued; ++t)
                mbar_wait_bounded(&v_full[t % VS], (t / VS) & 1, kPfWaitNs / 8);
        }
    } else if (warp == kPfMmaWarp) {
        // ================= tensor-core products (one thread) =================
        if (lane == 0) {
            constexpr uint32_t idS = umma_idesc_f16(kPfRows, kPfKeys, 0, 0);
            constexpr uint32_t idPV = umma_idesc_f16(kPfRows, D, 0, 1);
            // Descriptors are built once per operand; within a tile only the start-address field moves, by
            // compile-time offsets (every shared-memory address is below 2^18, so the 14-bit field
            // (address >> 4) never carries into the next field).
            const uint64_t dQ = umma_smem_desc(smem_u32(qs), 16, 1024);
            const uint64_t dK = umma_smem_desc(smem_u32(kst(0)), 16, 1024);
            // V as the MN-major B operand: 8-key groups 1024 bytes apart, 64-dim atoms one chunk apart
            const uint64_t dV = umma_smem_desc(smem_u32(vst(0)), Geo::kKVChunk, 1024);
            const uint32_t tO = tmem + Geo::kTmemO;
            // S(j) = Q K(j)^T into buffer j % 2 over D / 16 steps of 16 dims: M = 128 rows, N = 128 keys
            auto mma_s = [&](int j) {
                const uint64_t b0 = dK + static_cast<uint64_t>((j % KS) * (Geo::kKVBytes >> 4));
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks >> 2, kk = ks & 3;
                    umma_f16_ss(tmem + (j & 1) * kPfKeys, dQ + ((c * Geo::kQChunk + kk * 32) >> 4),
                                b0 + ((c * Geo::kKVChunk + kk * 32) >> 4), idS, ks > 0);
                }
                umma_commit(&s_full[j & 1]);
                umma_commit(&k_empty[j % KS]);
            };
            // O += P(j) V(j): 8 steps of 16 keys, P read from TMEM buffer j % 2 (fp16, or high and residual
            // parts), N = D
            auto mma_pv = [&](int j) {
                const uint64_t v0 = dV + static_cast<uint64_t>((j % VS) * (Geo::kKVBytes >> 4));
                const uint32_t tP = tmem + (j & 1) * kPfKeys;
#pragma unroll
                for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                    const uint64_t b = v0 + ((kk * 2048) >> 4);
                    const uint32_t tPk = tP + (kk >> 1) * kPfPartKeys + (kk & 1) * 8;  // hi; lo 16 columns on
                    umma_f16_ts(tO, tPk, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                    if constexpr (kSplitP) umma_f16_ts(tO, tPk + 16, b, idPV, 1u);
                }
                umma_commit(o_full);
                umma_commit(&v_empty[j % VS]);
            };

            bool ok = pf_wait(q_full, 0, s_abort);
            for (int j = 0; ok && j < min(nt, 2); ++j) {
                if (!(ok = pf_wait(&k_full[j % KS], (j / KS) & 1, s_abort))) break;
                tc_fence_after();
                mma_s(j);
            }
            for (int j = 0; ok && j < nt; ++j) {
                // P(j) V(j) once P(j) is in TMEM and V(j) has landed
                if (!(ok = pf_wait(&v_full[j % VS], (j / VS) & 1, s_abort))) break;
                if (!(ok = pf_wait(&p_full[j & 1], (j >> 1) & 1, s_abort))) break;
                tc_fence_after();
                mma_pv(j);
                if (j == nt - 1) umma_commit(o_last);
                // S(j + 2) into buffer j % 2 once P(j) V(j) has read P(j) there
                if (j + 2 < nt) {
                    if (!(ok = pf_wait(&k_full[(j + 2) % KS], ((j + 2) / KS) & 1, s_abort))) break;
                    if (!(ok = pf_wait(o_full, j & 1, s_abort))) break;
                    tc_fence_after();
                    mma_s(j + 2);
                }
            }
            // every product issued is complete before the tensor memory is released
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, kPfWaitNs);
            if (!ok) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        }
    } else {
        // ================= row warps: softmax and output =================
        // Thread = query row (TMEM lane) x one 32-key part of every key tile.  The 4 threads of a row (warps
        // wq, wq + 4, wq + 8, wq + 12) post their part's extreme score to each other through shared memory,
        // so all take the same running max; each writes P for its part, and O (rescales, output) is split over
        // the parts by 32-column chunks.
        const int kp = warp >> 2, wq = warp & 3;
        const int row = wq * 32 + lane;
        const int qi = r0 + row;  // row of the segment
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tSp = tmem + kp * kPfPartKeys + lane_base;  // this part's columns of S / P (buffer 0)
        const bool owns_o = kp * 32 < D;                           // O columns [32 kp, 32 kp + 32)
        const uint32_t tOp = tmem + Geo::kTmemO + kp * 32 + lane_base;
        uint64_t* xq = &xchg[wq];
        const float sl2 = p.scale_log2;
        const bool neg_scale = sl2 < 0.f;  // then the largest scaled score comes from the smallest raw one
        const float fill = neg_scale ? INFINITY : -INFINITY;
        float m_used = -INFINITY, l = 0.f;  // l: this part's share of the row sum
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, pf_wait(&s_full[j & 1], (j >> 1) & 1, s_abort));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tSp + (j & 1) * kPfKeys;
            float s[kPfPartKeys];
            tmem_ld32(tS, s);
            const int k0 = j * kPfKeys + kp * kPfPartKeys;  // first key of this part
            // a part that crosses the causal diagonal or the segment end needs the mask; the others do not
            const bool masked = k0 + kPfPartKeys > len || (p.causal && k0 + kPfPartKeys - 1 > r0);
            float e[4];
            if (masked) {
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = fill;
#pragma unroll
                for (int c = 0; c < kPfPartKeys; ++c) {
                    const int kj = k0 + c;
                    const bool valid = kj < len && (!p.causal || kj <= qi);
                    const float v = valid ? s[c] : fill;
                    e[c & 3] = neg_scale ? fminf(e[c & 3], v) : fmaxf(e[c & 3], v);
                }
            } else if (!neg_scale) {
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = max3f(s[i], s[4 + i], s[8 + i]);
#pragma unroll
                for (int c = 12; c + 8 <= kPfPartKeys; c += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = max3f(e[i], s[c + i], s[c + 4 + i]);
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = fmaxf(e[i], s[kPfPartKeys - 4 + i]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = min3f(s[i], s[4 + i], s[8 + i]);
#pragma unroll
                for (int c = 12; c + 8 <= kPfPartKeys; c += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = min3f(e[i], s[c + i], s[c + 4 + i]);
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = fminf(e[i], s[kPfPartKeys - 4 + i]);
            }
            float ext = neg_scale ? fminf(fminf(e[0], e[1]), fminf(e[2], e[3]))
                                  : fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]));
            // exchange with the row's other parts (double-buffered by tile parity)
            float* xb = xbuf + (j & 1) * kPfKeyParts * kPfRows;
            xb[kp * kPfRows + row] = ext;
            __syncwarp();
            if (lane == 0) mbar_arrive(xq);
            ok = __all_sync(0xffffffffu, pf_wait(xq, j & 1, s_abort));
            if (!ok) break;
#pragma unroll
            for (int q = 0; q < kPfKeyParts; ++q) {
                const float other = xb[q * kPfRows + row];
                ext = neg_scale ? fminf(ext, other) : fmaxf(ext, other);
            }
            // the tile's largest scaled score (-inf when every key is masked); the running max moves only when
            // it has grown by 2^8 (or from -inf): then l and O are rescaled
            const float mx = ext == fill ? -INFINITY : ext * sl2;
            float alpha = 1.f;
            if (mx > m_used + kPfRescaleLog2) {  // includes the first finite max (m_used = -inf)
                alpha = m_used == -INFINITY ? 0.f : ex2(m_used - mx);
                m_used = mx;
            }
            const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
            // P = 2^(s * scale * log2 e - m) written over this part's S columns in fp16, keys (2i, 2i + 1) in
            // column i (split form: the high part there, the residual in column 16 + i).  l sums the fp16
            // weights written (split form: P in fp32).
            if (masked) {
#pragma unroll
                for (int c = 0; c < kPfPartKeys; ++c) {
                    const int kj = k0 + c;
                    const bool valid = kj < len && (!p.causal || kj <= qi);
                    s[c] = valid ? ex2(fmaf(s[c], sl2, neg_m)) : 0.f;
                }
            } else {
#if KVC_PREFILL_1T_FMA2
                // two scores per packed fp32x2 multiply-add (each lane rounds as fmaf does), then 2^x each
                const uint64_t sc2 = pack_f32x2(sl2, sl2), nm2 = pack_f32x2(neg_m, neg_m);
#pragma unroll
                for (int c = 0; c < kPfPartKeys; c += 2) {
                    float x0, x1;
                    unpack_f32x2(fma_f32x2(pack_f32x2(s[c], s[c + 1]), sc2, nm2), x0, x1);
                    s[c] = ex2(x0);
                    s[c + 1] = ex2(x1);
                }
#else
#pragma unroll
                for (int c = 0; c < kPfPartKeys; ++c) s[c] = ex2(fmaf(s[c], sl2, neg_m));
#endif
            }
            float ls4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t hv[16], lv[16];
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                const int c = 2 * e2;
                hv[e2] = pack_half2(s[c], s[c + 1]);
                if constexpr (kSplitP) {
                    const float2 f = unpack_half2(hv[e2]);
                    lv[e2] = pack_half2(s[c] - f.x, s[c + 1] - f.y);
                    ls4[e2 & 3] += s[c] + s[c + 1];
                } else {
                    ls4[e2 & 3] = add_f16x2_to_f32(hv[e2], ls4[e2 & 3]);
                }
            }
            tmem_st16(tS, hv);
            if constexpr (kSplitP) tmem_st16(tS + 16, lv);
            l = l * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
            // rescale O (rare: the running max moved): it must be idle, i.e. P(j-1) V(j-1) complete; P(j) V(j)
            // is not issued before this thread's arrival below
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f) && owns_o) {
                ok = __all_sync(0xffffffffu, pf_wait(o_full, (j - 1) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                float o[32];
                tmem_ld32(tOp, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= alpha;
                tmem_st32(tOp, o);
            }
            // the segment's last key tile: V rows past its end (the next segment's tokens) are zeroed, so that
            // whatever they hold cannot reach this segment's output through a zero weight
            const int vrem = len - j * kPfKeys;
            if (vrem < kPfKeys && warp == 0) {
                ok = __all_sync(0xffffffffu, pf_wait(&v_full[j % VS], (j / VS) & 1, s_abort));
                if (!ok) break;
                uint8_t* vt = vst(j % VS);
                for (int e3 = lane; e3 < (kPfKeys - vrem) * 8 * Geo::kChunks; e3 += 32) {
                    const int r = vrem + e3 / (8 * Geo::kChunks), rest = e3 % (8 * Geo::kChunks);
                    *reinterpret_cast<uint4*>(vt + (rest / 8) * Geo::kKVChunk + sw128(r, rest % 8)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();  // visible to the tensor cores (async proxy)
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[j & 1]);
        }
        // the row sum: this part's share plus the other parts'
        if (ok) {
            float* xb = xbuf + (nt & 1) * kPfKeyParts * kPfRows;
            xb[kp * kPfRows + row] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(xq);
            ok = __all_sync(0xffffffffu, pf_wait(xq, nt & 1, s_abort));
            if (ok) {
                l = 0.f;
#pragma unroll
                for (int q = 0; q < kPfKeyParts; ++q) l += xb[q * kPfRows + row];
            }
        }
        if (ok && owns_o) ok = __all_sync(0xffffffffu, pf_wait(o_last, 0, s_abort));
        if (ok && owns_o) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t base = (static_cast<int64_t>(beg + qi) * p.Hq + h) * D + kp * 32;
            float o[32];
            tmem_ld32(tOp, o);
            if (qi < len) {
                if (p.out_f32) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                             o[4 * i + 3] * inv);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + base);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_half2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                            pack_half2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                            pack_half2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                            pack_half2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
                }
            }
        }
    }
    // every TMEM access of the CTA is complete; the allocating warp frees it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Geo::kTmemCols);
    }
}

using EncodeTiledFnP = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiledFnP encode_fn_p() {
    static EncodeTiledFnP fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnP>(ptr);
    });
    return fn;
}

// [T][H][D] fp16 viewed as (dim, head, token); boxes of 64 dims x 1 head x 128 tokens, 128-byte swizzle
static cudaError_t make_packed_map(CUtensorMap* map, const void* base, int D, int H, int T) {
    EncodeTiledFnP fn = encode_fn_p();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t gdim[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t gstride[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool kSplitP>
static cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t stream) {
    using Geo = PfGeom<D>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prefill_kernel<D, kSplitP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Geo::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tq, tk, tv;
    cudaError_t e = make_packed_map(&tq, a.q, D, a.Hq, a.total_tokens);
    if (e == cudaSuccess) e = make_packed_map(&tk, a.k, D, a.Hkv, a.total_tokens);
    if (e == cudaSuccess) e = make_packed_map(&tv, a.v, D, a.Hkv, a.total_tokens);
    if (e != cudaSuccess) return e;
    PrefillKernelParams p;
    p.cu_seqlens = a.cu_seqlens;
    p.out = a.out;
    p.err = a.err;
    p.nseq = a.nseq;
    p.total_tokens = a.total_tokens;
    p.tiles_per_seq = (a.max_seqlen + kPfCtaRows - 1) / kPfCtaRows;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.causal = a.causal;
    p.out_f32 = a.out_f32;
    p.scale_log2 = a.scale * kPfLog2e;
    const int64_t nblocks = static_cast<int64_t>(p.tiles_per_seq) * a.nseq * a.Hq;
    if (nblocks > 2147483647LL) return cudaErrorInvalidConfiguration;
    prefill_kernel<D, kSplitP><<<static_cast<unsigned>(nblocks), kPfThreads, Geo::kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace pf1

cudaError_t launch_prefill_1t(const PrefillArgs& a, cudaStream_t stream) {
    using namespace pf1;
    if (a.nseq <= 0 || a.total_tokens <= 0 || a.max_seqlen <= 0) return cudaSuccess;
    if (a.D != 64) return cudaErrorInvalidValue;
    return a.split_p ? launch_prefill_d<64, true>(a, stream) : launch_prefill_d<64, false>(a, stream);
}

}  // namespace kvc
