// Varlen packed prefill attention for sm_103a on the 5th-generation tensor cores.
//
// What it computes (xformers article of the "Aufmerksamkeit" feed,
// chatgpz.de, parts 4 and 5): sequences of different lengths are packed
// back to back without padding (cu_seqlens); each segment attends only to
// itself (block-diagonal mask), causally (j <= i) or not; query head h reads
// KV head h / (Hq / Hkv).  Per row: softmax(q K^T * scale) V, with the
// running-max / exp-sum rule of the FlashAttention article over key tiles.
//
// Design: one CTA per (128-row query tile of a segment, query head), five
// warps.  Lane 0 of warp 4 issues every TMA copy and every tcgen05.mma;
// warps 0-3 own the 128 query rows (thread = row = TMEM lane) and run the
// softmax.  Per 64-key tile j:
//   S = Q K^T   tcgen05.mma M=128 x N=64, Q and K K-major in shared memory
//               (128-byte swizzle, as TMA writes them), fp32 accumulator in TMEM
//   softmax     the row threads read S from TMEM, mask (segment end, causal),
//               keep the running max until it has grown by 2^8 (then rescale
//               O in TMEM), and write P = hi + lo (two fp16 parts, so the
//               product keeps ~fp32 accuracy) to shared memory, K-major
//   O += P V    tcgen05.mma M=128 x N=64 per 64-dim chunk, V MN-major; O stays
//               in TMEM across tiles
// K and V have two-stage rings of their own; S(j+1) is issued as soon as the
// row threads have read S(j), so the tensor cores work on it during softmax(j).
// Every wait is bounded; a timeout sets an error bit and drains the CTA.
#include <algorithm>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace kvc {

constexpr int kPfRows = 128;  // query rows per CTA: the MMA's M, one TMEM lane each
constexpr int kPfKeys = 64;   // keys per K/V tile: N of S, K of P V
constexpr int kPfRowWarps = 4;
constexpr int kPfThreads = (kPfRowWarps + 1) * 32;
constexpr uint64_t kPfWaitNs = 1000000000ull;
constexpr float kPfLog2e = 1.4426950408889634f;
constexpr float kPfRescaleLog2 = 8.f;  // P stays below 2^8, far inside fp16

template <int D>
struct PfGeom {
    static constexpr int kChunks = D / 64;                    // 64-dim (128-byte) column chunks
    static constexpr int kQChunk = kPfRows * 128;             // 16 KiB
    static constexpr int kKVChunk = kPfKeys * 128;            // 8 KiB
    static constexpr int kQBytes = kChunks * kQChunk;
    static constexpr int kKVBytes = kChunks * kKVChunk;       // one K or V tile
    static constexpr int kPBytes = kPfRows * kPfKeys * 2;     // 16 KiB
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;             // 2 stages
    static constexpr int kVOff = kKOff + 2 * kKVBytes;        // 2 stages
    static constexpr int kPhiOff = kVOff + 2 * kKVBytes;
    static constexpr int kPloOff = kPhiOff + kPBytes;
    static constexpr int kBarOff = kPloOff + kPBytes;
    static constexpr int kSmemBytes = kBarOff + 128 + 1024;  // barriers, TMEM address, abort flag; alignment
    static constexpr int kTmemS = 0;                          // S: columns [0, 64)
    static constexpr int kTmemO = kPfKeys;                    // O: columns [64, 64 + D)
    static constexpr uint32_t kTmemCols = kPfKeys + D <= 128 ? 128 : 256;
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

// Wait for a phase; gives up when another thread of the CTA has given up (abort flag) or after the limit,
// in which case it raises the flag itself.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 63u) == 63u && global_timer_ns() - t0 > kPfWaitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads) prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                             const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV,
                                                             const PrefillKernelParams p) {
    using Geo = PfGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kBarOff);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;   // [2] K tile landed
    uint64_t* v_full = bars + 3;   // [2] V tile landed
    uint64_t* k_empty = bars + 5;  // [2] S products of the stage's tile done
    uint64_t* v_empty = bars + 7;  // [2] P V products of the stage's tile done
    uint64_t* s_full = bars + 9;   // S of the current tile in TMEM
    uint64_t* s_free = bars + 10;  // the row warps have read S (4 arrivals)
    uint64_t* p_full = bars + 11;  // P of the current tile in shared memory (4 arrivals)
    uint64_t* o_full = bars + 12;  // P V of the current tile done
    uint64_t* fin = bars + 13;     // every MMA issued so far done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 14);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 14) + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x / p.tiles_per_seq, tile = blockIdx.x % p.tiles_per_seq;
    const int h = blockIdx.y, hk = h / p.G;

    const int beg = p.cu_seqlens[seg], end = p.cu_seqlens[seg + 1];
    const int len = end - beg;
    if (beg < 0 || len < 0 || end > p.total_tokens) {
        if (threadIdx.x == 0 && tile == 0 && h == 0) atomicOr(p.err, KVC_DEVERR_SEQLENS);
        return;
    }
    if (tile == 0 && h == 0 && threadIdx.x == 0 && len > p.tiles_per_seq * kPfRows)
        atomicOr(p.err, KVC_DEVERR_SEQLENS);  // rows past max_seqlen are not computed
    const int r0 = tile * kPfRows;
    if (r0 >= len) return;
    const int kv_len = p.causal ? min(len, r0 + kPfRows) : len;
    const int ntiles = (kv_len + kPfKeys - 1) / kPfKeys;

    uint8_t* qs = smem + Geo::kQOff;
    uint8_t* phi = smem + Geo::kPhiOff;
    uint8_t* plo = smem + Geo::kPloOff;
    auto kst = [&](int st) { return smem + Geo::kKOff + st * Geo::kKVBytes; };
    auto vst = [&](int st) { return smem + Geo::kVOff + st * Geo::kKVBytes; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, kPfRowWarps);
        mbar_init(p_full, kPfRowWarps);
        mbar_init(o_full, 1);
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
    const uint32_t tS = tmem + Geo::kTmemS, tO = tmem + Geo::kTmemO;

    if (warp == kPfRowWarps) {
        // ================= producer: TMA copies and tensor-core products (one thread) =================
        if (lane == 0) {
            auto load_k = [&](int t) {
                uint64_t* bar = &k_full[t & 1];
                mbar_arrive_expect_tx(bar, Geo::kKVBytes);
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
                    tma_load_3d(kst(t & 1) + c * Geo::kKVChunk, &tmK, bar, c * 64, hk, beg + t * kPfKeys);
            };
            auto load_v = [&](int t) {
                uint64_t* bar = &v_full[t & 1];
                mbar_arrive_expect_tx(bar, Geo::kKVBytes);
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
                    tma_load_3d(vst(t & 1) + c * Geo::kKVChunk, &tmV, bar, c * 64, hk, beg + t * kPfKeys);
            };
            prefetch_tensormap(&tmQ);
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
            mbar_arrive_expect_tx(q_full, Geo::kQBytes);
#pragma unroll
            for (int c = 0; c < Geo::kChunks; ++c)
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(qs + c * Geo::kQChunk + half * 64 * 128, &tmQ, q_full, c * 64, h, beg + r0 + half * 64);
            int k_issued = 0, v_issued = 0;  // tiles whose copies were issued
            for (; k_issued < min(ntiles, 2); ++k_issued) load_k(k_issued);
            for (; v_issued < min(ntiles, 2); ++v_issued) load_v(v_issued);
            int k_done = 0, v_done = 0;  // tiles whose copies were waited for
            bool q_done = false;

            constexpr uint32_t idS = umma_idesc_f16(kPfRows, kPfKeys, 0, 0);
            constexpr uint32_t idPV = umma_idesc_f16(kPfRows, 64, 0, 1);
            const uint32_t q_addr = smem_u32(qs);
            // S(j) = Q K(j)^T over D / 16 steps of 16 dims
            auto mma_s = [&](int j) {
                const uint32_t k_addr = smem_u32(kst(j & 1));
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks >> 2, kk = ks & 3;
                    const uint64_t a = umma_smem_desc(q_addr + c * Geo::kQChunk + kk * 32, 16, 1024);
                    const uint64_t b = umma_smem_desc(k_addr + c * Geo::kKVChunk + kk * 32, 16, 1024);
                    umma_f16_ss(tS, a, b, idS, ks > 0);
                }
                umma_commit(s_full);
                umma_commit(&k_empty[j & 1]);
            };
            // O += P(j) V(j): per 64-dim chunk, 4 steps of 16 keys, high and residual parts of P
            auto mma_pv = [&](int j) {
                const uint32_t v_addr = smem_u32(vst(j & 1));
#pragma unroll
                for (int c = 0; c < Geo::kChunks; ++c)
#pragma unroll
                    for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                        // V MN-major: 16 keys = two 8-row groups of 1024 bytes (one 64-dim atom wide)
                        const uint64_t b = umma_smem_desc(v_addr + c * Geo::kKVChunk + kk * 2048, 1024, 1024);
                        const uint64_t ah = umma_smem_desc(smem_u32(phi) + kk * 32, 16, 1024);
                        const uint64_t al = umma_smem_desc(smem_u32(plo) + kk * 32, 16, 1024);
                        umma_f16_ss(tO + c * 64, ah, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                        umma_f16_ss(tO + c * 64, al, b, idPV, 1u);
                    }
                umma_commit(o_full);
                umma_commit(&v_empty[j & 1]);
            };

            bool ok = pf_wait(q_full, 0, s_abort);
            q_done = ok;
            ok = ok && pf_wait(&k_full[0], 0, s_abort);
            if (ok) {
                k_done = 1;
                tc_fence_after();
                mma_s(0);
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                // the K stage of tile j is free once S(j) is done: refill it with tile j + 2
                if (j + 2 < ntiles) {
                    if (!(ok = pf_wait(&k_empty[j & 1], (j >> 1) & 1, s_abort))) break;
                    load_k(j + 2);
                    k_issued = j + 3;
                }
                // S(j + 1) once its K tile has landed and the row warps have read S(j)
                if (j + 1 < ntiles) {
                    if (!(ok = pf_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, s_abort))) break;
                    k_done = j + 2;
                    if (!(ok = pf_wait(s_free, j & 1, s_abort))) break;
                    tc_fence_after();
                    mma_s(j + 1);
                }
                // P(j) V(j) once P(j) is written and V(j) has landed
                if (!(ok = pf_wait(&v_full[j & 1], (j >> 1) & 1, s_abort))) break;
                v_done = j + 1;
                if (!(ok = pf_wait(p_full, j & 1, s_abort))) break;
                tc_fence_after();
                mma_pv(j);
                if (j + 2 < ntiles) {
                    if (!(ok = pf_wait(&v_empty[j & 1], (j >> 1) & 1, s_abort))) break;
                    load_v(j + 2);
                    v_issued = j + 3;
                }
            }
            // every product issued is complete before the tensor memory is released
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, kPfWaitNs);
            if (!ok) {
                atomicOr(p.err, KVC_DEVERR_TIMEOUT);
                // copies still in flight land before the shared memory is released
                if (!q_done) mbar_wait_bounded(q_full, 0, kPfWaitNs / 8);
                for (int t = k_done; t < k_issued; ++t) mbar_wait_bounded(&k_full[t & 1], (t >> 1) & 1, kPfWaitNs / 8);
                for (int t = v_done; t < v_issued; ++t) mbar_wait_bounded(&v_full[t & 1], (t >> 1) & 1, kPfWaitNs / 8);
            }
        }
    } else {
        // ================= row warps: softmax and output; thread = query row = TMEM lane =================
        const int row = threadIdx.x;
        const int qi = r0 + row;  // row of the segment
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = __all_sync(0xffffffffu, pf_wait(s_full, j & 1, s_abort));
            if (!ok) break;
            tc_fence_after();
            float s[2][32];  // keys c = 32 * (c >> 5) + (c & 31)
            tmem_ld32(tS + lane_base, s[0]);
            tmem_ld32(tS + lane_base + 32, s[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);

            const int k0 = j * kPfKeys;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kPfKeys; ++c) {
                const int kj = k0 + c;
                const bool valid = kj < len && (!p.causal || kj <= qi);
                float& x = s[c >> 5][c & 31];
                x = valid ? x * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x);
            }
            // the running max moves only when it has grown by 2^8 (or from -inf): then l and O are rescaled
            float alpha = 1.f;
            if (mx > m_used + kPfRescaleLog2) {  // includes the first finite max (m_used = -inf)
                alpha = m_used == -INFINITY ? 0.f : ex2(m_used - mx);
                m_used = mx;
            }
            float ls = 0.f;
#pragma unroll
            for (int c = 0; c < kPfKeys; ++c) {
                float& x = s[c >> 5][c & 31];
                x = m_used == -INFINITY ? 0.f : ex2(x - m_used);
                ls += x;
            }
            l = l * alpha + ls;
            // P(j-1) V(j-1) must be done before O is rescaled and P is overwritten
            if (j > 0) {
                ok = __all_sync(0xffffffffu, pf_wait(o_full, (j - 1) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        tmem_ld32(tO + lane_base + c, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tO + lane_base + c, o);
                    }
                    tmem_wait_st();
                }
            }
            // the last tile of a segment: V rows past its end (the next segment's tokens) are zeroed, so
            // that whatever they hold cannot reach this segment's output through a zero weight
            const int vrem = len - k0;
            if (vrem < kPfKeys && warp == 0) {
                ok = __all_sync(0xffffffffu, pf_wait(&v_full[j & 1], (j >> 1) & 1, s_abort));
                if (!ok) break;
                uint8_t* vt = vst(j & 1);
                for (int e = lane; e < (kPfKeys - vrem) * 8 * Geo::kChunks; e += 32) {
                    const int r = vrem + e / (8 * Geo::kChunks), rest = e % (8 * Geo::kChunks);
                    *reinterpret_cast<uint4*>(vt + (rest / 8) * Geo::kKVChunk + sw128(r, rest % 8)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // P = hi + lo in fp16, row `row`, 64 keys = 8 chunks of 16 bytes, 128-byte swizzle
#pragma unroll
            for (int cc = 0; cc < kPfKeys / 8; ++cc) {
                uint32_t hv[4], lv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = cc * 8 + 2 * e;
                    const float p0 = s[c >> 5][c & 31], p1 = s[(c + 1) >> 5][(c + 1) & 31];
                    hv[e] = pack_half2(p0, p1);
                    const float2 f = unpack_half2(hv[e]);
                    lv[e] = pack_half2(p0 - f.x, p1 - f.y);
                }
                *reinterpret_cast<uint4*>(phi + sw128(row, cc)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<uint4*>(plo + sw128(row, cc)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
            }
            fence_proxy_async_smem();  // visible to the tensor cores (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, pf_wait(o_full, (ntiles - 1) & 1, s_abort));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t base = (static_cast<int64_t>(beg + qi) * p.Hq + h) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                float o[32];
                tmem_ld32(tO + lane_base + c, o);
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

// [T][H][D] fp16 viewed as (dim, head, token); boxes of 64 dims x 1 head x 64 tokens, 128-byte swizzle
static cudaError_t make_packed_map(CUtensorMap* map, const void* base, int D, int H, int T) {
    EncodeTiledFnP fn = encode_fn_p();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t gdim[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t gstride[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), gdim, gstride, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t stream) {
    using Geo = PfGeom<D>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    p.tiles_per_seq = (a.max_seqlen + kPfRows - 1) / kPfRows;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.causal = a.causal;
    p.out_f32 = a.out_f32;
    p.scale_log2 = a.scale * kPfLog2e;
    dim3 grid(a.nseq * p.tiles_per_seq, a.Hq);
    prefill_kernel<D><<<grid, kPfThreads, Geo::kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    if (a.nseq <= 0 || a.total_tokens <= 0 || a.max_seqlen <= 0) return cudaSuccess;
    switch (a.D) {
        case 64: return launch_prefill_d<64>(a, stream);
        case 128: return launch_prefill_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
