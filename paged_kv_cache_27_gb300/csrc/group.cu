// The cascade (shared-prefix) decode on sm_103a: one CTA streams a range of a group's shared K/V blocks once
// through a ring in shared memory and several warps, one per sequence of the group, attend over it; partial
// states are merged by the decode side's combine kernel (decode.cu).  What it computes, and its citations,
// is stated at the kernel and in include/kvc.h.
#include "decode_common.cuh"

namespace kvc {

// ---- groups of sequences that share their first blocks ----------------------------------------------
//
// One CTA streams a range of K/V blocks once through a ring in shared memory (thread 0 issues the copies).
// The group is sequences g0 .. g1-1 (at most 8) whose block-table rows begin with the same `nsh` blocks;
// warp w is sequence g0 + w and attends its query rows (the G heads of the sequence's KV head) over every
// block of the range with the decode kernel's block math (S^T = K Q^T, online softmax in base 2,
// O^T += V^T (P_hi + P_lo)^T), then writes its partial state (m, l, acc) as part `chunk` of its rows; the
// combine kernel merges the parts.  The range is a chunk of the shared blocks, all of them inside every
// member's context, so nothing is masked.
#ifndef KVC_PREFIX_STAGES  // blocks in flight per group CTA
#define KVC_PREFIX_STAGES 12
#endif
#ifndef KVC_PREFIX_CTAS  // group CTAs per SM the chunking aims for
#define KVC_PREFIX_CTAS 4
#endif
constexpr int kGroupStages = KVC_PREFIX_STAGES;  // the deepest ring; a launch may use fewer stages
constexpr int kGroupMaxChunk = 4096;              // blocks per CTA at most (their ids are in shared memory)
constexpr int kGroupMaxSmem = 200 * 1024;         // the dynamic shared memory a group launch may use

// dynamic shared memory of the group kernel with a ring of `stages` blocks and chunks of `chunk` blocks: the
// ring, its full/empty barriers, the abort flag, the chunk's block ids, alignment
template <int D>
constexpr size_t group_smem_bytes(int stages, int chunk) {
    return stages * DecodeCfg<D>::kStageBytes + 2 * stages * 8 + 16 + 4 * static_cast<size_t>(chunk) + 1024;
}

struct GroupKernelParams {
    const __half* q;             // [B][Hq][D]
    const int32_t* block_table;
    const int32_t* group_start;  // [n_groups + 1]
    const int32_t* blk_off;      // per sequence, its group's shared blocks
    float* part_ml;
    float* part_acc;
    unsigned* err;
    int max_blocks, num_blocks, Hq, Hkv, G, chunk, nchunks, part_stride;
    int stages;  // ring depth of this launch, 1 .. kGroupStages
    float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(256) paged_decode_group_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const GroupKernelParams p) {
    using C = DecodeCfg<D>;
    const int ST = p.stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * C::kStageBytes);
    uint64_t* empty = full + ST;
    volatile int* s_abort = reinterpret_cast<volatile int*>(empty + ST);
    int* s_ids = reinterpret_cast<int*>(empty + ST) + 4;  // the chunk's physical block ids

    const int NW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int grp = blockIdx.x / p.nchunks, chunk = blockIdx.x % p.nchunks, kvh = blockIdx.y;
#if KVC_GROUP_EARLY_TRIGGER
    grid_dependents_launch();
#endif
    // the group: its members (warps), the table row they share blocks through, and the block range [j0, j1)
    const int g0 = p.group_start[grp];
    const int nmem = p.group_start[grp + 1] - g0;
    if (nmem < 1) return;
    const int nblk = p.blk_off[g0];
    if (nmem > NW || nblk < 0 || nblk > p.max_blocks) {
        if (threadIdx.x == 0 && chunk == 0 && kvh == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
        return;
    }
    const int32_t* table = p.block_table + static_cast<int64_t>(g0) * p.max_blocks;  // the first member's row
    const int j0 = chunk * p.chunk, j1 = min(nblk, j0 + p.chunk);
    if (j0 >= j1) return;  // the range is shorter
    const int n = j1 - j0;

    auto issue = [&](int i) {  // thread 0: block j0 + i into stage i % ST
        uint64_t* bar = &full[i % ST];
        const int phys = s_ids[i];
        if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, KVC_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // completes the phase without data: the block is skipped
            return;
        }
        uint8_t* st = smem + (i % ST) * C::kStageBytes;
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int y = (phys * p.Hkv + kvh) * kBlockSize;
        const uint64_t policy = l2_policy_evict_first();
#pragma unroll
        for (int x = 0; x < D; x += 64) {
            tma_load_2d(st + (x / 64) * 2048, &tmK, bar, x, y, policy);
            tma_load_2d(st + C::kTileBytes + (x / 64) * 2048, &tmV, bar, x, y, policy);
        }
    };
    // the chunk's block ids, all at once (one round trip instead of one per copy)
    for (int k = threadIdx.x; k < n; k += blockDim.x) s_ids[k] = table[j0 + k];
    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *s_abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int i = 0; i < min(n, ST); ++i) issue(i);
    grid_dependency_wait();  // q may come from the previous kernel

    const bool member = warp < nmem;
    const int64_t qrow = static_cast<int64_t>(g0) + (member ? warp : 0);
    uint32_t qa[D / 16][2];
    {
        const bool row_ok = member && g < p.G;
        const __half* qp = p.q + (qrow * p.Hq + kvh * p.G + (row_ok ? g : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 2 * t4) : 0u;
            qa[ks][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 8 + 2 * t4) : 0u;
        }
    }
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3;
    int issued = min(n, ST), i = 0;
    bool ok = true;
    // bounded wait that also gives up once another warp has
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = global_timer_ns();
        for (uint32_t k = 0;; ++k) {
            if (mbar_try_wait(bar, parity)) return true;
            if (*s_abort) return false;
            if ((k & 63u) == 63u && global_timer_ns() - t0 > kWaitLimitNs) {
                *s_abort = 1;
                return false;
            }
        }
    };
#pragma unroll 1
    for (; i < n; ++i) {
        const int s = i % ST;
        ok = __all_sync(0xffffffffu, wait(&full[s], (i / ST) & 1));
        if (!ok) break;
        if (member) {
            const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
            const uint32_t vbase = kbase + C::kTileBytes;
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kbase + swz((mi & 1) * 8 + (lane & 7), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                mma_f16_16816(sc, a0, a1, a2, a3, qa[ks][0], qa[ks][1]);
            }
            // every key of a shared block is inside every member's context
            const float x0 = sc[0] * sl2, x1 = sc[1] * sl2, x2 = sc[2] * sl2, x3 = sc[3] * sl2;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
            }
            const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
            const float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);  // 0 on the first block
            m_run[0] = mn0;
            m_run[1] = mn1;
            const float p0 = ex2(x0 - mn0), p2 = ex2(x2 - mn0), p1 = ex2(x1 - mn1), p3 = ex2(x3 - mn1);
            l_run[0] = l_run[0] * al0 + p0 + p2;
            l_run[1] = l_run[1] * al1 + p1 + p3;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            const uint32_t h01 = pack_half2(p0, p1), h23 = pack_half2(p2, p3);
            const float2 f01 = unpack_half2(h01), f23 = unpack_half2(h23);
            const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
            const uint32_t bl0 = movmatrix_trans(pack_half2(p0 - f01.x, p1 - f01.y));
            const uint32_t bl1 = movmatrix_trans(pack_half2(p2 - f23.x, p3 - f23.y));
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vbase + swz((mi >> 1) * 8 + (lane & 7), 2 * mt + (mi & 1)), a0, a1, a2, a3);
                mma_f16_16816(o[mt], a0, a1, a2, a3, bh0, bh1);
                mma_f16_16816(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        // thread 0 refills the stage once every warp has read it
        if (threadIdx.x == 0 && issued < n) {
            if (!wait(&empty[s], (i / ST) & 1)) {
                ok = false;
            } else {
                issue(issued);
                ++issued;
            }
        }
        if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (!ok || *s_abort) {
        // thread 0 lets copies still in flight land; the CTA's shared memory stays allocated until it exits
        if (threadIdx.x == 0) {
            atomicOr(p.err, KVC_DEVERR_TIMEOUT);
            for (int k = i; k < issued; ++k) mbar_wait_bounded(&full[k % ST], (k / ST) & 1, kWaitLimitNs / 8);
        }
        return;
    }
    if (!member) return;
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], sh);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], sh);
    }
    // this warp's partial for heads 2*t4, 2*t4+1 (those < G): part `chunk` of its query rows
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int gg = 2 * t4 + hh;
        if (gg >= p.G) continue;
        const int64_t row = (qrow * p.Hq + kvh * p.G + gg) * p.part_stride + chunk;
        if (g == 0) {
            p.part_ml[row * 2 + 0] = m_run[hh];
            p.part_ml[row * 2 + 1] = l_run[hh];
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            p.part_acc[row * D + mt * 16 + g] = o[mt][hh];
            p.part_acc[row * D + mt * 16 + g + 8] = o[mt][2 + hh];
        }
    }
}

// one-time kernel attributes (the ring exceeds the default dynamic shared-memory limit)
template <int D>
static cudaError_t group_setup() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(paged_decode_group_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupMaxSmem);
    });
    return err;
}

// ---- cascade ----------------------------------------------------------------------------------------
cudaError_t cascade_plan(int B, int Hq, int Hkv, int D, int max_ctx, int n_groups, int max_shared_blocks,
                         CascadePlan* plan) {
    cudaError_t e = decode_plan(B, Hq, Hkv, D, max_ctx, 0, &plan->suffix);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    // prefix CTAs: about KVC_PREFIX_CTAS per SM over all (group, KV head) pairs, at least 4 blocks each
    const int64_t pairs = std::max<int64_t>(1, static_cast<int64_t>(n_groups) * Hkv);
    const int64_t per_pair = std::max<int64_t>(1, KVC_PREFIX_CTAS * static_cast<int64_t>(sms) / pairs);
    plan->chunk = static_cast<int>(
        std::min<int64_t>(kGroupMaxChunk, std::max<int64_t>(4, (max_shared_blocks + per_pair - 1) / per_pair)));
    plan->nchunks = max_shared_blocks > 0 ? (max_shared_blocks + plan->chunk - 1) / plan->chunk : 0;
    plan->part_stride = plan->nchunks + plan->suffix.num_parts;
    plan->workspace_bytes = partials_bytes(static_cast<size_t>(B) * Hq * plan->part_stride, D);
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_cascade_d(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                                    int n_groups, const CascadePlan& cp, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    cudaError_t e = group_setup<D>();
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    CUtensorMap tmK, tmV;
    e = make_tile_map(&tmK, a.k_cache, D, rows);
    if (e != cudaSuccess) return e;
    e = make_tile_map(&tmV, a.v_cache, D, rows);
    if (e != cudaSuccess) return e;
    const size_t nrow = static_cast<size_t>(a.B) * a.Hq * cp.part_stride;
    float* part_ml = static_cast<float*>(a.workspace);
    float* part_acc = partials_acc(part_ml, nrow);
    const bool pdl = launch_overlap() != 0;
    const int G = a.Hq / a.Hkv;

    // 1. the shared prefixes: prefix parts 0 .. nchunks-1
    if (cp.nchunks > 0) {
        GroupKernelParams pp;
        pp.q = a.q;
        pp.block_table = a.block_table;
        pp.group_start = group_start;
        pp.blk_off = shared_blocks;
        pp.part_ml = part_ml;
        pp.part_acc = part_acc;
        pp.err = a.err;
        pp.max_blocks = a.max_blocks;
        pp.num_blocks = a.num_blocks;
        pp.Hq = a.Hq;
        pp.Hkv = a.Hkv;
        pp.G = G;
        pp.chunk = cp.chunk;
        pp.nchunks = cp.nchunks;
        pp.part_stride = cp.part_stride;
        pp.scale_log2 = a.scale * kLog2e;
        pp.stages = kGroupStages;
        e = launch(paged_decode_group_kernel<D>, dim3(n_groups * cp.nchunks, a.Hkv),
                   dim3(32 * kMaxGroupSize), group_smem_bytes<D>(kGroupStages, cp.chunk), stream, pdl,
                   1u, tmK, tmV, pp);
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
    c.prefix_chunk = cp.chunk;
    c.cascade = 1;
    c.q_len = 1;
    return launch_combine(c, D, a.B, stream);
}

cudaError_t launch_cascade(const DecodeArgs& a, const int32_t* group_start, const int32_t* shared_blocks,
                           int n_groups, int max_shared_blocks, cudaStream_t stream) {
    CascadePlan cp;
    cudaError_t e = cascade_plan(a.B, a.Hq, a.Hkv, a.D, a.max_context_len, n_groups, max_shared_blocks, &cp);
    if (e != cudaSuccess) return e;
    if (cp.workspace_bytes > a.workspace_bytes) return cudaErrorInvalidValue;
    switch (a.D) {
        case 64: return launch_cascade_d<64>(a, group_start, shared_blocks, n_groups, cp, stream);
        case 128: return launch_cascade_d<128>(a, group_start, shared_blocks, n_groups, cp, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
