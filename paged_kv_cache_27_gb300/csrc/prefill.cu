// Varlen packed prefill attention for sm_103a.
//
// What it computes (xformers article of the "Aufmerksamkeit" feed,
// chatgpz.de, parts 4 and 5): sequences of different lengths are packed
// back to back without padding (cu_seqlens); each segment attends only to
// itself (block-diagonal mask), causally (j <= i) or not; query head h reads
// KV head h / (Hq / Hkv).  Per row: softmax(q K^T * scale) V.
//
// Design: one CTA per (64-row query tile of a segment, query head); 4 warps
// of 16 query rows.  Q, K and V tiles of 64 tokens x 64 columns are fetched by
// 3-D TMA (token, head, dim) with the 128-byte swizzle into a two-stage ring;
// S = Q K^T and O += P V run on the tensor cores (mma.sync, fp16 in, fp32
// accumulate, P split into fp16 high + residual); online softmax in fp32
// base 2 (the FlashAttention article's running max / exp-sum rule).
#include <algorithm>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

constexpr int kPfRows = 64;   // query rows per CTA
constexpr int kPfKeys = 64;   // keys per KV tile
constexpr int kPfWarps = 4;
constexpr uint64_t kPfWaitNs = 1000000000ull;
constexpr float kPfLog2e = 1.4426950408889634f;

template <int D>
struct PrefillGeom {
    static constexpr int kHalf = 64 * 128;                // one 64-row x 64-col swizzled box: 8 KiB
    static constexpr int kTileBytes = (D / 64) * kHalf;   // 64 rows x D
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kTileBytes;             // 2 stages x (K, V)
    static constexpr int kBarOff = kKVOff + 4 * kTileBytes;
    static constexpr int kSmemBytes = kBarOff + 64 + 1024;
};

struct PrefillKernelParams {
    const int32_t* cu_seqlens;
    void* out;
    unsigned* err;
    int nseq, total_tokens, tiles_per_seq, Hq, Hkv, G, causal, out_f32;
    float scale_log2;
};

// 64-row tile, 128-byte swizzle, boxes of 64 columns stacked at 8 KiB
__device__ __forceinline__ uint32_t pswz(int row, int chunk) {
    return static_cast<uint32_t>(((chunk >> 3) << 13) + (row << 7) + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kPfWarps * 32) prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV,
                                                                const PrefillKernelParams p) {
    using Geo = PrefillGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kBarOff);  // [0] Q, [1..2] KV stages

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
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
    auto kv_stage = [&](int st) { return smem + Geo::kKVOff + st * 2 * Geo::kTileBytes; };

    auto issue_kv = [&](int kt) {
        uint64_t* bar = &bars[1 + (kt & 1)];
        uint8_t* st = kv_stage(kt & 1);
        mbar_arrive_expect_tx(bar, 2 * Geo::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64) {
            tma_load_3d(st + (x / 64) * Geo::kHalf, &tmK, bar, x, hk, beg + kt * kPfKeys);
            tma_load_3d(st + Geo::kTileBytes + (x / 64) * Geo::kHalf, &tmV, bar, x, hk, beg + kt * kPfKeys);
        }
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bars[0], Geo::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64) tma_load_3d(qs + (x / 64) * Geo::kHalf, &tmQ, &bars[0], x, h, beg + r0);
        issue_kv(0);
        if (ntiles > 1) issue_kv(1);
    }
    __syncthreads();

    const bool q_ok = __syncthreads_and(mbar_wait_bounded(&bars[0], 0, kPfWaitNs) ? 1 : 0) != 0;
    // query fragments of this warp's 16 rows
    uint32_t qa[D / 16][4];
    if (q_ok) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            ldsm_x4(smem_u32(qs) + pswz(row, ks * 2 + (lane >> 4)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
    }

    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int qi0 = r0 + warp * 16 + g;  // rows qi0 and qi0 + 8 of the segment

    int fail_kt = q_ok ? -1 : 0;
    for (int kt = 0; kt < ntiles && fail_kt < 0; ++kt) {
        const bool good = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[1 + (kt & 1)], (kt >> 1) & 1, kPfWaitNs));
        if (good) {
            const uint32_t kbase = smem_u32(kv_stage(kt & 1));
            const uint32_t vbase = kbase + Geo::kTileBytes;
            float sc[kPfKeys / 8][4];
#pragma unroll
            for (int nt = 0; nt < kPfKeys / 8; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int kc = 0; kc < D / 32; ++kc) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + pswz(nt * 8 + (lane & 7), kc * 4 + (lane >> 3)), b0, b1, b2, b3);
                    mma_f16_16816(sc[nt], qa[2 * kc][0], qa[2 * kc][1], qa[2 * kc][2], qa[2 * kc][3], b0, b1);
                    mma_f16_16816(sc[nt], qa[2 * kc + 1][0], qa[2 * kc + 1][1], qa[2 * kc + 1][2],
                                  qa[2 * kc + 1][3], b2, b3);
                }
            }
            const int k0 = kt * kPfKeys;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < kPfKeys / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kj = k0 + nt * 8 + 2 * t4 + (e & 1);
                    const int qi = qi0 + (e >> 1) * 8;
                    const bool valid = kj < len && (!p.causal || kj <= qi);
                    sc[nt][e] = valid ? sc[nt][e] * p.scale_log2 : -INFINITY;
                    mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
                }
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float m_new = fmaxf(m_run[r], mx[r]);
                // a row may see no valid key in this tile yet (m stays -inf): keep it at zero weight
                alpha[r] = m_new == -INFINITY ? 1.f : ex2(m_run[r] - m_new);
                m_run[r] = m_new;
            }
            float ps[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < kPfKeys / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mr = m_run[e >> 1];
                    const float pv = mr == -INFINITY ? 0.f : ex2(sc[nt][e] - mr);
                    sc[nt][e] = pv;
                    ps[e >> 1] += pv;
                }
#pragma unroll
            for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + ps[r];
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) {
                o[nd][0] *= alpha[0];
                o[nd][1] *= alpha[0];
                o[nd][2] *= alpha[1];
                o[nd][3] *= alpha[1];
            }
            const int vrem = len - k0;  // keys of this tile inside the segment
#pragma unroll
            for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                uint32_t ah[4], al[4];
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float p0 = sc[2 * kk + half][2 * r], p1 = sc[2 * kk + half][2 * r + 1];
                        const uint32_t hi = pack_half2(p0, p1);
                        const float2 hf = unpack_half2(hi);
                        ah[half * 2 + r] = hi;
                        al[half * 2 + r] = pack_half2(p0 - hf.x, p1 - hf.y);
                    }
                uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
                const int tb = kk * 16;
                if (vrem < tb + 16) {
                    keep0 = (tb + 2 * t4 < vrem ? 0x0000ffffu : 0u) | (tb + 2 * t4 + 1 < vrem ? 0xffff0000u : 0u);
                    keep1 = (tb + 8 + 2 * t4 < vrem ? 0x0000ffffu : 0u) | (tb + 9 + 2 * t4 < vrem ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                    const int mi = lane >> 3;
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(vbase + pswz(tb + (mi & 1) * 8 + (lane & 7), nd2 * 2 + (mi >> 1)), v0, v1, v2, v3);
                    v0 &= keep0;
                    v2 &= keep0;
                    v1 &= keep1;
                    v3 &= keep1;
                    mma_f16_16816(o[2 * nd2], ah[0], ah[1], ah[2], ah[3], v0, v1);
                    mma_f16_16816(o[2 * nd2], al[0], al[1], al[2], al[3], v0, v1);
                    mma_f16_16816(o[2 * nd2 + 1], ah[0], ah[1], ah[2], ah[3], v2, v3);
                    mma_f16_16816(o[2 * nd2 + 1], al[0], al[1], al[2], al[3], v2, v3);
                }
            }
        }
        // every warp is done with this stage before it is refilled
        if (!__syncthreads_and(good ? 1 : 0)) {
            fail_kt = kt;
            break;
        }
        if (threadIdx.x == 0 && kt + 2 < ntiles) issue_kv(kt + 2);
    }
    if (fail_kt >= 0) {
        if (threadIdx.x == 0) {
            atomicOr(p.err, KVC_DEVERR_TIMEOUT);
            // let the copies still in flight land before the shared memory is released
            if (!q_ok) mbar_wait_bounded(&bars[0], 0, kPfWaitNs / 8);
            for (int kt = fail_kt; kt < min(ntiles, fail_kt + 2); ++kt)
                mbar_wait_bounded(&bars[1 + (kt & 1)], (kt >> 1) & 1, kPfWaitNs / 8);
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int qi = qi0 + r * 8;
        if (qi >= len) continue;
        const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
        const int64_t base = (static_cast<int64_t>(beg + qi) * p.Hq + h) * D;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
            const float a = o[nd][2 * r] * inv, c = o[nd][2 * r + 1] * inv;
            const int d = nd * 8 + 2 * t4;
            if (p.out_f32)
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + base + d) = make_float2(a, c);
            else
                *reinterpret_cast<__half2*>(static_cast<__half*>(p.out) + base + d) = __floats2half2_rn(a, c);
        }
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

// [T][H][D] fp16 viewed as (dim, head, token); boxes of 64 dims x 1 head x 64 tokens
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
    using Geo = PrefillGeom<D>;
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
    prefill_kernel<D><<<grid, kPfWarps * 32, Geo::kSmemBytes, stream>>>(tq, tk, tv, p);
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
