// Varlen packed prefill attention for sm_103a on the 5th-generation tensor cores.
//
// What it computes (xformers article of the "Aufmerksamkeit" feed,
// chatgpz.de, parts 4 and 5): sequences of different lengths are packed
// back to back without padding (cu_seqlens); each segment attends only to
// itself (block-diagonal mask), causally (j <= i) or not; query head h reads
// KV head h / (Hq / Hkv).  Per row: softmax(q K^T * scale) V, with the
// running-max / exp-sum rule of the FlashAttention article over key tiles.
//
// Design (head dim 128, and head dim 64 on batches of 65,536 (token, query head) pairs or more; smaller head
// dim 64 batches run prefill_1t.cu): one CTA per (256 query rows of a segment, query
// head) = two 128-row query tiles A and B that share every K/V tile; ten warps.  Warps 0-3 own tile A's rows
// and warps 4-7 tile B's (thread = row = TMEM lane) and run the softmax; lane 0 of warp 8 issues every
// tcgen05.mma, lane 0 of warp 9 every TMA copy.  Per 128-key tile j and query tile X:
//   S_X = Q_X K^T   tcgen05.mma M=128 x N=128, Q and K K-major in shared memory (128-byte swizzle, as TMA
//                   writes them), fp32 accumulator in TMEM
//   softmax         the row threads read S_X from TMEM one 64-key half at a time, mask only on tiles that
//                   cross the causal diagonal or the segment end, keep the running max until it has grown by
//                   2^8 (then rescale O_X in TMEM), and write P_X over S_X in fp16 (or as an fp16 high part and
//                   residual, so the product keeps ~fp32 weights)
//   O_X += P_X V    tcgen05.mma M=128 x N=D with P read from TMEM (the A operand) and V MN-major in shared
//                   memory; O_X stays in TMEM
// The products go out in the order P_A V(j), S_A(j+1), P_B V(j), S_B(j+1): S_X(j+1) reuses P_X(j)'s columns,
// so it waits for the commit of P_X V(j); while one group of row warps runs its softmax, the tensor cores work
// on the other group's products.  K and V have rings of their own.  Every wait is bounded; a timeout sets an
// error bit and drains the CTA.
#include <algorithm>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace kvc {

constexpr int kPfRows = 128;   // rows of one query tile: the MMA's M, one TMEM lane each
constexpr int kPfQTiles = 2;   // query tiles per CTA, A and B
constexpr int kPfCtaRows = kPfRows * kPfQTiles;
constexpr int kPfKeys = 128;   // keys per K/V tile: N of S, K of P V
constexpr int kPfRowWarps = 4 * kPfQTiles;
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
    static constexpr int kQBytes = kChunks * kQChunk;         // one query tile
    static constexpr int kKVBytes = kChunks * kKVChunk;       // one K or V tile
    static constexpr int kQOff = 0;                           // Q_A, Q_B
    static constexpr int kKOff = kQOff + kPfQTiles * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKVBytes;
    static constexpr int kBarOff = kVOff + kVStages * kKVBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers, TMEM address, abort flag; alignment
    static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
    // TMEM columns: S_A / P_A [0, 128), S_B / P_B [128, 256), O_A [256, 256 + D), O_B [256 + D, 256 + 2D).
    // P_X is written over S_X once the row warps have read S_X: per 64-key half h, P in fp16 (or its high
    // fp16 part) in columns [64h, 64h + 32), the residuals of the split form in [64h + 32, 64h + 64), two keys
    // per column.
    static constexpr int kTmemO = kPfQTiles * kPfKeys;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kTmemO + kPfQTiles * D <= 512, "tensor memory");
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

// 1: the softmax's scale-and-shift of unmasked scores in packed fp32x2 multiply-adds (half the instructions,
// the same rounding per lane); 0: one fmaf per score.  The softmax is bound by its instruction stream: two A/B
// pairs, 4 x 4096 tokens, 32 / 8 heads: head dim 128 causal 596.1 -> 583.8 us, non-causal 994 -> 968, head dim
// 64 causal 534 -> 522.
#ifndef KVC_PREFILL_FMA2
#define KVC_PREFILL_FMA2 1
#endif

// acc + the two fp16 halves of h (each converted exactly), as two rounded fp32 additions
__device__ __forceinline__ float add_f16x2_to_f32(uint32_t h, float acc) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %0, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(h));
    return acc;
}

// Wait for a phase; gives up when another thread of the CTA has given up (abort flag) or after the limit,
// in which case it raises the flag itself.
// The waiting thread sleeps in the hardware until the phase completes or 20 us pass, so waiting warps do not
// take issue slots from working ones.
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

// number of key tiles query tile X (first row rx) reads; 0 when it has no row in the segment
__device__ __forceinline__ int pf_key_tiles(int rx, int len, int causal) {
    if (rx >= len) return 0;
    const int kv_len = causal ? min(len, rx + kPfRows) : len;
    return (kv_len + kPfKeys - 1) / kPfKeys;
}

// 1: the fp16 weights of a 64-key half go to TMEM in one 32-column store; 0: two 16-column stores.  Two A/B
// pairs, 4 x 4096 tokens, 32 / 8 heads: head dim 128 causal 601.3 -> 598.5 us, non-causal 1005.7 -> 994.7, head
// dim 64 causal 537.1 -> 534.7.  (Eight 8-column stores per half, interleaved with the weights: 1001 us; half of
// the weights' 2^x on the FMA pipe by a cubic instead of the multi-function unit: 818 us.)
#ifndef KVC_PREFILL_SOFTMAX_ST32
#define KVC_PREFILL_SOFTMAX_ST32 1
#endif

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
    uint64_t* k_full = bars + 1;        // [KS] K tile landed
    uint64_t* k_empty = bars + 1 + KS;  // [KS] S products of the stage's tile done
    uint64_t* v_full = bars + 1 + 2 * KS;        // [VS] V tile landed
    uint64_t* v_empty = bars + 1 + 2 * KS + VS;  // [VS] P V products of the stage's tile done
    uint64_t* s_full = bars + 1 + 2 * KS + 2 * VS;  // [2] S_X of the current key tile in TMEM
    uint64_t* p_full = s_full + 2;                  // [2] P_X of the current key tile in TMEM (4 arrivals)
    uint64_t* o_full = s_full + 4;                  // [2] P_X V of the current key tile done
    uint64_t* fin = s_full + 6;                     // every MMA issued so far done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_full + 7);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_full + 7) + 1;

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
    const int nt0 = pf_key_tiles(r0, len, p.causal), nt1 = pf_key_tiles(r0 + kPfRows, len, p.causal);
    const int nq = nt1 > 0 ? 2 : 1;       // query tiles with rows in the segment
    const int ntiles = max(nt0, nt1);     // key tiles of the CTA (tile B reads at least as many as A)

    auto qs = [&](int x) { return smem + Geo::kQOff + x * Geo::kQBytes; };
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
        for (int x = 0; x < kPfQTiles; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_full[x], 1);
        }
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
            mbar_arrive_expect_tx(q_full, nq * Geo::kQBytes);
            for (int x = 0; x < nq; ++x)
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
                    tma_load_3d(qs(x) + c * Geo::kQChunk, &tmQ, q_full, c * 64, h, beg + r0 + x * kPfRows);
            // tile t goes into the stage of tile t - stages once that tile's products are done
            int k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int t = 0; ok && t < ntiles; ++t) {
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
            const uint64_t dQ = umma_smem_desc(smem_u32(qs(0)), 16, 1024);
            const uint64_t dK = umma_smem_desc(smem_u32(kst(0)), 16, 1024);
            // V as the MN-major B operand: 8-key groups 1024 bytes apart, 64-dim atoms one chunk apart
            const uint64_t dV = umma_smem_desc(smem_u32(vst(0)), Geo::kKVChunk, 1024);
            // S_X(j) = Q_X K(j)^T over D / 16 steps of 16 dims: M = 128 rows, N = 128 keys
            auto mma_s = [&](int x, int st) {
                const uint64_t a0 = dQ + static_cast<uint64_t>(x * (Geo::kQBytes >> 4));
                const uint64_t b0 = dK + static_cast<uint64_t>(st * (Geo::kKVBytes >> 4));
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks >> 2, kk = ks & 3;
                    umma_f16_ss(tmem + x * kPfKeys, a0 + ((c * Geo::kQChunk + kk * 32) >> 4),
                                b0 + ((c * Geo::kKVChunk + kk * 32) >> 4), idS, ks > 0);
                }
                umma_commit(&s_full[x]);
            };
            // O_X += P_X(j) V(j): 8 steps of 16 keys, P read from TMEM (fp16, or high and residual parts), N = D
            auto mma_pv = [&](int x, int st, bool first) {
                const uint64_t v0 = dV + static_cast<uint64_t>(st * (Geo::kKVBytes >> 4));
                const uint32_t tP = tmem + x * kPfKeys, tO = tmem + Geo::kTmemO + x * D;
#pragma unroll
                for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                    const uint64_t b = v0 + ((kk * 2048) >> 4);
                    const uint32_t tPk = tP + (kk >> 2) * 64 + (kk & 3) * 8;  // hi; lo 32 columns on
                    umma_f16_ts(tO, tPk, b, idPV, (!first || kk > 0) ? 1u : 0u);
                    if constexpr (kSplitP) umma_f16_ts(tO, tPk + 32, b, idPV, 1u);
                }
                umma_commit(&o_full[x]);
            };

            bool ok = pf_wait(q_full, 0, s_abort) && pf_wait(&k_full[0], 0, s_abort);
            if (ok) {
                tc_fence_after();
                for (int x = 0; x < nq; ++x) mma_s(x, 0);
                umma_commit(&k_empty[0]);
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                if (!(ok = pf_wait(&v_full[j % VS], (j / VS) & 1, s_abort))) break;
                bool k_next = false;
                // per query tile: P_X(j) V(j) once P_X(j) is in TMEM; then S_X(j + 1) into the same columns
                // once that product has read P_X(j)
                for (int x = 0; ok && x < nq; ++x) {
                    const int ntx = x == 0 ? nt0 : nt1;
                    if (j >= ntx) continue;
                    if (!(ok = pf_wait(&p_full[x], j & 1, s_abort))) break;
                    tc_fence_after();
                    mma_pv(x, j % VS, j == 0);
                    if (j + 1 < ntx) {
                        if (!k_next) {
                            if (!(ok = pf_wait(&k_full[(j + 1) % KS], ((j + 1) / KS) & 1, s_abort))) break;
                            k_next = true;
                        }
                        if (!(ok = pf_wait(&o_full[x], j & 1, s_abort))) break;
                        tc_fence_after();
                        mma_s(x, (j + 1) % KS);
                    }
                }
                if (!ok) break;
                umma_commit(&v_empty[j % VS]);
                if (j + 1 < ntiles) umma_commit(&k_empty[(j + 1) % KS]);
            }
            // every product issued is complete before the tensor memory is released
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, kPfWaitNs);
            if (!ok) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        }
    } else if (warp / 4 < nq) {
        // ================= row warps: softmax and output; thread = query row = TMEM lane =================
        const int x = warp / 4, wq = warp & 3;
        const int rx = r0 + x * kPfRows;        // first row of this query tile
        const int row = wq * 32 + lane;
        const int qi = rx + row;                // row of the segment
        const int nt = x == 0 ? nt0 : nt1;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + x * kPfKeys + lane_base, tO = tmem + Geo::kTmemO + x * D + lane_base;
        const float sl2 = p.scale_log2;
        const bool neg_scale = sl2 < 0.f;  // then the largest scaled score comes from the smallest raw one
        const float fill = neg_scale ? INFINITY : -INFINITY;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            // S_X(j) complete also means P_X(j-1) V(j-1) complete: it was issued before S_X(j)
            ok = __all_sync(0xffffffffu, pf_wait(&s_full[x], j & 1, s_abort));
            if (!ok) break;
            tc_fence_after();
            const int k0 = j * kPfKeys;
            // a tile that crosses the causal diagonal or the segment end needs the mask; the others do not
            const bool masked = k0 + kPfKeys > len || (p.causal && k0 + kPfKeys - 1 > rx);
            float alpha = 1.f;       // rescale of O and of the l of earlier tiles
            float lsum[2] = {0.f, 0.f};  // per 64-key half: sum of the weights written
            // One pass per 64-key half: the half's extreme score, the lazy running max (it moves only when the
            // max has grown by 2^8, or from -inf), then P = 2^(s * scale * log2 e - m) written over the half's
            // own S columns in fp16, keys (2i, 2i + 1) in column i (split form: the high part there, the
            // residual in column 32 + i).  l sums the fp16 weights written (split form: P in fp32).
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float s[64];
                tmem_ld64(tS + hh * 64, s);
                float e[4];
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = fill;
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int kj = k0 + hh * 64 + c;
                        const bool valid = kj < len && (!p.causal || kj <= qi);
                        const float v = valid ? s[c] : fill;
                        e[c & 3] = neg_scale ? fminf(e[c & 3], v) : fmaxf(e[c & 3], v);
                    }
                } else if (!neg_scale) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = max3f(s[i], s[4 + i], s[8 + i]);
#pragma unroll
                    for (int c = 12; c + 8 <= 64; c += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i) e[i] = max3f(e[i], s[c + i], s[c + 4 + i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = fmaxf(e[i], s[60 + i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = min3f(s[i], s[4 + i], s[8 + i]);
#pragma unroll
                    for (int c = 12; c + 8 <= 64; c += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i) e[i] = min3f(e[i], s[c + i], s[c + 4 + i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = fminf(e[i], s[60 + i]);
                }
                const float ext = neg_scale ? fminf(fminf(e[0], e[1]), fminf(e[2], e[3]))
                                            : fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]));
                const float mx = ext == fill ? -INFINITY : ext * sl2;  // -inf when every key is masked
                float a_h = 1.f;
                if (mx > m_used + kPfRescaleLog2) {  // includes the first finite max (m_used = -inf)
                    a_h = m_used == -INFINITY ? 0.f : ex2(m_used - mx);
                    m_used = mx;
                }
                if (hh == 1 && __any_sync(0xffffffffu, a_h != 1.f)) {
                    // the max moved inside the tile: the first half's weights, already written, are scaled to
                    // the new base and re-rounded (l takes their new sum); then this half's scores are read again
                    float w[32], r[32];
                    tmem_ld32(tS, w);
                    if constexpr (kSplitP) tmem_ld32(tS + 32, r);
                    float s0 = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 f = unpack_half2(__float_as_uint(w[i]));
                        if constexpr (kSplitP) {
                            const float2 g = unpack_half2(__float_as_uint(r[i]));
                            const float p0 = (f.x + g.x) * a_h, p1 = (f.y + g.y) * a_h;
                            const uint32_t hi = pack_half2(p0, p1);
                            const float2 hf = unpack_half2(hi);
                            w[i] = __uint_as_float(hi);
                            r[i] = __uint_as_float(pack_half2(p0 - hf.x, p1 - hf.y));
                            s0 += p0 + p1;
                        } else {
                            const uint32_t hi = pack_half2(f.x * a_h, f.y * a_h);
                            w[i] = __uint_as_float(hi);
                            s0 = add_f16x2_to_f32(hi, s0);
                        }
                    }
                    tmem_st32(tS, w);
                    if constexpr (kSplitP) tmem_st32(tS + 32, r);
                    if (a_h != 1.f) lsum[0] = s0;
                    tmem_ld64(tS + 64, s);
                }
                alpha *= a_h;
                const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
                if (masked) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int kj = k0 + hh * 64 + c;
                        const bool valid = kj < len && (!p.causal || kj <= qi);
                        s[c] = valid ? ex2(fmaf(s[c], sl2, neg_m)) : 0.f;
                    }
                } else {
#if KVC_PREFILL_FMA2
                    // two scores per packed fp32x2 multiply-add (each lane rounds as fmaf does), then 2^x each
                    const uint64_t sc2 = pack_f32x2(sl2, sl2), nm2 = pack_f32x2(neg_m, neg_m);
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float x0, x1;
                        unpack_f32x2(fma_f32x2(pack_f32x2(s[c], s[c + 1]), sc2, nm2), x0, x1);
                        s[c] = ex2(x0);
                        s[c + 1] = ex2(x1);
                    }
#else
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = ex2(fmaf(s[c], sl2, neg_m));
#endif
                }
#if KVC_PREFILL_SOFTMAX_ST32
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (kSplitP) {
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        uint32_t hv[16], lv[16];
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2) {
                            const int c = qq * 32 + 2 * e2;
                            hv[e2] = pack_half2(s[c], s[c + 1]);
                            const float2 f = unpack_half2(hv[e2]);
                            lv[e2] = pack_half2(s[c] - f.x, s[c + 1] - f.y);
                            ls4[e2 & 3] += s[c] + s[c + 1];
                        }
                        tmem_st16(tS + hh * 64 + qq * 16, hv);
                        tmem_st16(tS + hh * 64 + 32 + qq * 16, lv);
                    }
                } else {
                    // the half's 32 fp16 pairs in one store
                    float hv[32];
#pragma unroll
                    for (int e2 = 0; e2 < 32; ++e2) {
                        const uint32_t h2 = pack_half2(s[2 * e2], s[2 * e2 + 1]);
                        hv[e2] = __uint_as_float(h2);
                        ls4[e2 & 3] = add_f16x2_to_f32(h2, ls4[e2 & 3]);
                    }
                    tmem_st32(tS + hh * 64, hv);
                }
#else
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    uint32_t hv[16], lv[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const int c = qq * 32 + 2 * e2;
                        hv[e2] = pack_half2(s[c], s[c + 1]);
                        if constexpr (kSplitP) {
                            const float2 f = unpack_half2(hv[e2]);
                            lv[e2] = pack_half2(s[c] - f.x, s[c + 1] - f.y);
                            ls4[e2 & 3] += s[c] + s[c + 1];
                        } else {
                            ls4[e2 & 3] = add_f16x2_to_f32(hv[e2], ls4[e2 & 3]);
                        }
                    }
                    tmem_st16(tS + hh * 64 + qq * 16, hv);
                    if constexpr (kSplitP) tmem_st16(tS + hh * 64 + 32 + qq * 16, lv);
                }
#endif
                lsum[hh] = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
            }
            l = l * alpha + (lsum[0] + lsum[1]);
            // O_X is idle here (P_X(j-1) V(j-1) is complete, P_X(j) V(j) not issued): rescale it in place
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    float o[32];
                    tmem_ld32(tO + c, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tO + c, o);
                }
            }
            // the segment's last key tile: V rows past its end (the next segment's tokens) are zeroed, so that
            // whatever they hold cannot reach this segment's output through a zero weight.  The first query
            // tile that reads this key tile does it; its P V products are issued before the other tile's.
            const int vrem = len - k0;
            if (vrem < kPfKeys && wq == 0 && (x == 0 || j >= nt0)) {
                ok = __all_sync(0xffffffffu, pf_wait(&v_full[j % VS], (j / VS) & 1, s_abort));
                if (!ok) break;
                uint8_t* vt = vst(j % VS);
                for (int e = lane; e < (kPfKeys - vrem) * 8 * Geo::kChunks; e += 32) {
                    const int r = vrem + e / (8 * Geo::kChunks), rest = e % (8 * Geo::kChunks);
                    *reinterpret_cast<uint4*>(vt + (rest / 8) * Geo::kKVChunk + sw128(r, rest % 8)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();  // visible to the tensor cores (async proxy)
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
        }
        if (ok) ok = __all_sync(0xffffffffu, pf_wait(&o_full[x], (nt - 1) & 1, s_abort));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t base = (static_cast<int64_t>(beg + qi) * p.Hq + h) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                float o[32];
                tmem_ld32(tO + c, o);
                if (qi < len) {
                    if (p.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base + c);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                 o[4 * i + 3] * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + base + c);
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

// Head dim 64: batches of at least this many (token, query head) pairs take this file's kernel (two query tiles
// sharing each K/V tile); smaller ones the one-tile kernel (prefill_1t.cu), whose twice as many CTAs shorten the
// critical path of a small or skewed batch.  Measured (causal unless noted, us per call, one-tile vs two-tile):
// seqlens 37/120/8/200 x 8 heads (2,920 pairs) 12.1 vs 16.4; 592/1920/128/3200 x 8 (46,720) 49.2 vs 57.3,
// non-causal 86.0 vs 87.6; 2 x 4096 x 8 (65,536) 81.9 vs 76.4; 4 x 4096 x 8 157.7 vs 141.9; 16 x 1024 x 16 135.4
// vs 125.1; 4 x 4096 x 32 604.4 vs 536.5, non-causal 1018 vs 877.
#ifndef KVC_PREFILL_D64_TWO_TILE_WORK
#define KVC_PREFILL_D64_TWO_TILE_WORK 65536
#endif

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    if (a.nseq <= 0 || a.total_tokens <= 0 || a.max_seqlen <= 0) return cudaSuccess;
    if (a.D == 64) {
        if (static_cast<int64_t>(a.total_tokens) * a.Hq < KVC_PREFILL_D64_TWO_TILE_WORK)
            return launch_prefill_1t(a, stream);  // one query tile per CTA (prefill_1t.cu)
        return a.split_p ? launch_prefill_d<64, true>(a, stream) : launch_prefill_d<64, false>(a, stream);
    }
    switch (a.D * 2 + (a.split_p ? 1 : 0)) {
        case 256: return launch_prefill_d<128, false>(a, stream);
        case 257: return launch_prefill_d<128, true>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
