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
//  * a thread-block cluster of up to 8 CTAs per (range of the context, KV
//    head, sequence), the grid sized from the measured occupancy so that every
//    CTA is resident at once; a cluster usually covers a whole context;
//  * inside a cluster the blocks go to the cluster's warps round-robin;
//  * the G <= 8 query heads of a KV head are the 8 columns of the m16n8k16
//    tiles (S^T = K Q^T with the 16 tokens of a block as rows, then
//    O^T += V^T P^T with 16 head dims as rows, P^T transposed in registers by
//    movmatrix), so every K/V tile fetched from HBM serves the whole group and
//    no tensor-core row is padding;
//  * each warp owns a ring of stages; lane 0 issues the K and V tile loads
//    (16 tokens x D fp16 each) with 2-D TMA and the 128-byte swizzle so that
//    the ldmatrix reads are bank-conflict free; the warp waits on the stage's
//    mbarrier (bounded wait, error flag on expiry) and refills it;
//  * the cluster's slice of the block table is copied to shared memory in one
//    coalesced pass, in parallel with the context-length load;
//  * the products run on the tensor cores (mma.sync, fp16 in, fp32
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
#include "decode_common.cuh"

namespace kvc {

std::atomic<int> g_launch_overlap{0};

struct DecodeKernelParams {
    const __half* q;
    const __half* k_new;  // null: no append
    const __half* v_new;
    __half* k_cache;      // generic pointers to the same layer as the tensor maps (append target)
    __half* v_cache;
    const uint8_t* kv_fp8;   // fp8: the layer's records, one per (block, KV head) (fp8_record_bytes each)
    const int32_t* block_table;
    const int32_t* context_lens;
    void* out;
    float* part_ml;   // [B][Hq][nparts][2] (m, l) in base-2 units, one part per cluster
    float* part_acc;  // [B][Hq][nparts][D]
    unsigned* err;
    int max_blocks, num_blocks, B, Hq, Hkv, G, max_ctx;
    int hchunks;  // chunks of at most 8 query heads per KV head: grid.y = Hkv * hchunks
    int bpc;     // blocks per cluster: a cluster covers context blocks [c * bpc, (c + 1) * bpc)
    int csize;   // CTAs per cluster
    // partial state of cluster c of (sequence b, query head h) goes to row (b * Hq + h) * part_stride +
    // part_base + c of part_ml / part_acc
    int part_base, part_stride;
    const int32_t* blk_off;  // suffix pass: per sequence, the leading blocks of its table row attended elsewhere
    int out_f32;
    int len_order;  // 1: the CTAs at position z along the sequences take the z-th longest context
    float scale_log2;
    unsigned trace_seq;  // launch counter, used by the optional trace only
};

// ---- optional per-CTA timeline trace (build with -DKVC_TRACE=1) -----------------------------
// Each CTA records the global timer at: start, first copies issued, dependency wait passed, warp 0's
// main loop done, all warps done, CTA merge done, cluster merge passed (rank 0: all CTAs arrived),
// exit; plus its SM and coordinates.  kvc_trace_read() copies the records out.
#ifndef KVC_TRACE
#define KVC_TRACE 0
#endif
#if KVC_TRACE
constexpr int kTraceStamps = 8;
struct TraceRec {
    unsigned long long t[kTraceStamps];
    unsigned seq, smid, x, yz;
};
constexpr int kTraceCap = 1 << 16;
__device__ TraceRec g_trace[kTraceCap];
__device__ unsigned g_trace_n;
#define KVC_TRACE_MARK(i) \
    if (threadIdx.x == 0) s_trace_t[i] = global_timer_ns()
#define KVC_TRACE_END()                                                    \
    do {                                                                   \
        if (threadIdx.x == 0) {                                            \
            s_trace_t[kTraceStamps - 1] = global_timer_ns();               \
            const unsigned k = atomicAdd(&g_trace_n, 1u);                  \
            if (k < kTraceCap) {                                           \
                TraceRec& r = g_trace[k];                                  \
                for (int q_ = 0; q_ < kTraceStamps; ++q_) r.t[q_] = s_trace_t[q_]; \
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

// kSuffix: the cascade's suffix pass (per-sequence block offset, partial states only); the plain decode
// is compiled without either
// kFp8: the cache holds e4m3 codes with per-row scales (tmK / tmV map the codes; V codes are stored per dim,
// 16 token bytes in the order vt_pos gives).  The mma.sync fragments are read from the code tiles with one
// 32-bit load per fragment row and converted to fp16 (exact) in registers: for K, the MMA's k index runs over
// the head dims permuted within each group of 16 so that lane t's four dims are bytes 4t..4t+3 (q's fragments
// follow the same permutation, which leaves the dot products unchanged); for V the token order of the rows
// does the same.  The K scale multiplies the scores and the V scale the probabilities before the P V product,
// so the arithmetic is the fp16 path's
template <int D, bool kSuffix, bool kFp8 = false>
__global__ void __launch_bounds__(DecodeCfg<D, kFp8>::kThreads, KVC_DEC_MIN_CTAS)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeKernelParams p) {
    using C = DecodeCfg<D, kFp8>;
    constexpr int NW = C::kWarps, ST = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
    // the CTA's merged state: m[8], l[8], acc[8][D]
    // this CTA's merged state when it is cluster rank 0: m[8], l[8], acc[G][D] (the layout of an inbox slot)
    float* s_m = reinterpret_cast<float*>(smem + C::kRingBytes + C::kBarBytes);
    // rank 0's inbox: slot c - 1 holds rank c's merged state, laid out like the state at s_m
    float* s_inbox = reinterpret_cast<float*>(smem + C::kRingBytes + C::kBarBytes + C::kStateBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    // a KV head's G query heads go in chunks of at most 8 (the mma tiles' 8 columns) to consecutive CTAs along y,
    // which read the same K/V blocks at about the same time (the second read is mostly an L2 hit)
    __shared__ int s_len_hist[33];
    __shared__ uint8_t s_len_cls[kLenOrderMaxB];
    const int kvh = blockIdx.y / p.hchunks, hc = blockIdx.y - kvh * p.hchunks;
    const int b = p.len_order ? seq_by_length(p.context_lens, p.B, p.max_ctx, static_cast<int>(blockIdx.z),
                                              s_len_hist, s_len_cls, s_len_hist + 32)
                              : static_cast<int>(blockIdx.z);
    const int Gc = min(8, p.G - hc * 8);  // query heads of this CTA
    const int h0 = kvh * p.G + hc * 8;    // its first query head
    // the cluster's slice of the block table (bpc entries), after the inbox's cluster - 1 slots
    int* s_table = reinterpret_cast<int*>(s_inbox + (p.csize - 1) * (16 + Gc * D));
    const int cs = p.csize;
    const int cidx = blockIdx.x / cs;                                    // this CTA's cluster along the context
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;   // == blockIdx.x % cs
#if KVC_TRACE
    __shared__ unsigned long long s_trace_t[8];
    if (threadIdx.x == 0)
        for (int q_ = 0; q_ < 8; ++q_) s_trace_t[q_] = 0;
#endif
#if KVC_DEC_TRIGGER == 0
    grid_dependents_launch();
#endif
    KVC_TRACE_MARK(0);

    // each warp owns its barriers; lane 0 initialises them before it has any load outstanding, so
    // the release fence that publishes the initialisation has nothing to wait for
    uint64_t* wbars = bars + warp * ST;
    // rank 0's inbox barrier: completes when the other CTAs' merged states have arrived (asynchronous pushes)
    uint64_t* inbox_bar = bars + NW * ST;
    // bytes one CTA pushes into an inbox slot: acc[G][D], and m and l of its G heads
    const uint32_t push_bytes = static_cast<uint32_t>(Gc * D * 4 + Gc * 8);
    if (lane == 0) {
        for (int s = 0; s < ST; ++s) mbar_init(&wbars[s], 1);
        if (KVC_DEC_ASYNC_PUSH && warp == 0 && cs > 1) mbar_init(inbox_bar, 1);
        fence_barrier_init();
        // the one arrival of the inbox phase, with the bytes it waits for (they may land before or after it)
        if (KVC_DEC_ASYNC_PUSH && warp == 0 && cs > 1 && rank == 0)
            mbar_arrive_expect_tx(inbox_bar, static_cast<uint32_t>(cs - 1) * push_bytes);
    }

    // One round trip before the first copies: each warp's lane 0 fetches the table entries of its
    // static first round and the context length together; the cluster's whole slice of the table
    // (entries [cb0, cb0 + bpc), clipped to the row) goes to shared memory meanwhile, for the refills.
    // the first blk_off[b] blocks of the row (a shared prefix attended elsewhere) are skipped: this call
    // covers the rest of the context, in block coordinates relative to that offset
    const int off_raw = kSuffix ? p.blk_off[b] : 0;
    const bool off_ok = off_raw >= 0 && off_raw < p.max_blocks;
    const int off = off_ok ? off_raw : 0;
    const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.max_blocks + off;
    const int cb0 = cidx * p.bpc;
    const int nwarps_cl = cs * NW;
    const int gw = rank * NW + warp;  // warp index within the cluster
    const int row_end = min(cb0 + p.bpc, p.max_blocks - off);
    int first_phys[ST];
#pragma unroll
    for (int s = 0; s < ST; ++s) {
        const int j = cb0 + gw + s * nwarps_cl;
        first_phys[s] = (lane == 0 && j < row_end) ? table[j] : -1;
    }
    const int nload = max(0, row_end - cb0);
    for (int t = threadIdx.x; t < nload; t += C::kThreads) s_table[t] = table[cb0 + t];
    const int ctx_full = p.context_lens[b];
    const int ctx = ctx_full - off * kBlockSize;  // tokens this call covers (all of them without an offset)
    // every CTA of a cluster sees the same (b, kvh): these exits are uniform over the cluster
    if (!off_ok || ctx_full < 1 || ctx_full > p.max_blocks * kBlockSize || ctx_full > p.max_ctx || ctx < 1) {
        grid_dependency_wait();
        // with forced partials the combine kernel checks the same and writes the zeros
        if (blockIdx.x == 0 && !kSuffix) {
            if (threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            for (int e = threadIdx.x; e < Gc * D; e += blockDim.x)
                store_out(p.out, p.out_f32, (static_cast<int64_t>(b) * p.Hq + h0 + e / D) * D + e % D, 0.f);
        }
        return;
    }
    const int nblk = (ctx + kBlockSize - 1) / kBlockSize;
    const int nclus = (nblk + p.bpc - 1) / p.bpc;  // clusters this sequence needs
    if (cidx >= nclus) return;                     // the whole cluster is past the context
    const int cb1 = min(cb0 + p.bpc, nblk);        // this cluster covers blocks [cb0, cb1)

    uint8_t* wring = smem + warp * C::kWarpRingBytes;
    const uint64_t policy = l2_policy_evict_first();

    // lane 0: the K and V tiles of physical block phys into stage s
    auto issue = [&](int s, int phys) {
        uint64_t* bar = &wbars[s];
        if (phys < 0 || phys >= p.num_blocks) {
            atomicOr(p.err, KVC_DEVERR_BLOCK_ID);
            mbar_arrive(bar);  // complete the phase without data; the block is skipped
            return;
        }
        uint8_t* st = wring + s * C::kStageBytes;
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int y = (phys * p.Hkv + kvh) * kBlockSize;
        if constexpr (kFp8) {  // the block's record: K codes and scales, V codes and scales, in one copy
            bulk_load(st, p.kv_fp8 + static_cast<int64_t>(phys * p.Hkv + kvh) * C::kStageBytes, C::kStageBytes, bar);
        } else {
#pragma unroll
            for (int x = 0; x < D; x += 64) {
                tma_load_2d(st + (x / 64) * 2048, &tmK, bar, x, y, policy);
                tma_load_2d(st + C::kTileBytes + (x / 64) * 2048, &tmV, bar, x, y, policy);
            }
        }
    };
    // lane 0 issues the warp's static first round (stage s gets block cb0 + gw + s * warps-in-the-
    // cluster) without waiting for the rest of the CTA
    int blk[ST];
#pragma unroll
    for (int s = 0; s < ST; ++s) {
        const int j = cb0 + gw + s * nwarps_cl;
        blk[s] = j < cb1 ? j : -1;
    }
    if (lane == 0) {
        if (!kFp8 && warp == 0) {  // the fp8 records come by bulk copies (the maps are unused)
            prefetch_tensormap(&tmK);
            prefetch_tensormap(&tmV);
        }
#pragma unroll
        for (int s = 0; s < ST; ++s)
            if (blk[s] >= 0) issue(s, first_phys[s]);
    }
    __syncwarp();
    KVC_TRACE_MARK(1);

    __syncthreads();  // the table slice is in shared memory
    // announces that this CTA has started; the matching wait comes before the first remote store
    // into rank 0's shared memory. Nothing is published here, so the arrive needs no fence.
    if (cs > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- everything below may read what the previous kernel wrote ----
    grid_dependency_wait();
    KVC_TRACE_MARK(2);
    // every CTA of the cluster has started and passed its prologue (rank 0's inbox barrier is initialised), so
    // the pushes into rank 0 after the block loop need no further check.  Waiting here, where the CTA usually
    // waits for the previous kernel anyway, keeps this cluster-wide wait off the end of the launch (right before
    // the pushes it measured 0.4 us at the median).
    if (KVC_DEC_EARLY_CLUSTER_WAIT && cs > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
#if KVC_DEC_TRIGGER == 1
    grid_dependents_launch();
#endif

    // query fragments (A operand, rows = the G heads of this KV head; rows >= G are zero)
    uint32_t qa[D / 16][2];
    {
        const bool row_ok = g < Gc;
        const __half* qrow = p.q + (static_cast<int64_t>(b) * p.Hq + h0 + (row_ok ? g : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            // fp8: k indices 2t, 2t+1 / 2t+8, 2t+9 of the group are dims 4t, 4t+1 / 4t+2, 4t+3 (see above)
            const int c0 = kFp8 ? 4 * t4 : 2 * t4, c1 = kFp8 ? 4 * t4 + 2 : 8 + 2 * t4;
            qa[ks][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + c0) : 0u;
            qa[ks][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + c1) : 0u;
        }
    }
    // fused append: any warp of the last cluster may get the block of position ctx-1; each holds the
    // new row (lanes 0-15: K chunks, 16-31: V chunks) to write it to the cache and patch its tile
    const int app_blk = !kFp8 && p.k_new != nullptr && cidx == nclus - 1 ? nblk - 1 : -1;
    const int app_row = (ctx - 1) % kBlockSize;
    uint4 app_val = make_uint4(0, 0, 0, 0);
    if (app_blk >= 0 && (lane & 15) < D / 8) {
        const __half* src = (lane >= 16 ? p.v_new : p.k_new) + (static_cast<int64_t>(b) * p.Hkv + kvh) * D +
                            (lane & 15) * 8;
        app_val = *reinterpret_cast<const uint4*>(src);
    }

    int next_j = cb0 + gw + ST * nwarps_cl;  // fixed round-robin: this warp's blocks are gw mod (warps)
    // fp8: byte offsets in a K code tile of lane (g, t)'s 4 codes per 16-dim group, row g (row g + 8 is 8 * D
    // further: its swizzle term is the same)
    uint32_t koff[D / 16];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) koff[ks] = fp8_kswz(D, g, 16 * ks + 4 * t4);

    // O^T accumulators: o[mt] = dims mt*16 + g (+8) x heads 2*t4, 2*t4+1; running max / sum per head pair
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const float sl2 = p.scale_log2;
    uint32_t phase = 0;  // bit s: parity of stage s's next completion
    bool timed_out = false;

    // refill stage s with the next block of the cluster's range, if any is left (after the warp has read it)
    auto refill = [&](int s) {
        __syncwarp();
        const int nj = next_j;
        next_j += nwarps_cl;
        if (nj < cb1 && lane == 0) issue(s, s_table[nj - cb0]);
#if KVC_DEC_TRIGGER == 3
        if (nj >= cb1 && nj < cb1 + nwarps_cl) grid_dependents_launch();  // this warp's last copy is out
#elif KVC_DEC_TRIGGER == 2
        if (nj == cb0 + gw + ST * nwarps_cl) grid_dependents_launch();  // this warp's first refill
#endif
#pragma unroll
        for (int k = 0; k < ST; ++k)
            if (k == s) blk[k] = nj < cb1 ? nj : -1;
    };

#pragma unroll 1
    for (int i = 0;; ++i) {
        const int s = i % ST;
        bool refilled = false;
        int jj = -1;
#pragma unroll
        for (int k = 0; k < ST; ++k)
            if (k == s) jj = blk[k];  // register select, no local memory
        if (jj < 0) break;            // blocks only grow: the first empty stage ends the warp's work
        {
            const bool ok = mbar_wait_bounded(&wbars[s], (phase >> s) & 1u, kWaitLimitNs);
            phase ^= 1u << s;
            if (__any_sync(0xffffffffu, !ok)) {
                timed_out = true;
                break;
            }
            const int phys = s_table[jj - cb0];
            if (phys >= 0 && phys < p.num_blocks) {
                const int rem = ctx - jj * kBlockSize;  // valid tokens in this block (>= 1)
                // scores of tokens g and g+8 carry sl2 (times their K scales with an fp8 cache); the V scales
                // of tokens g and g+8 (0 past the context) multiply their probabilities before P V
                float sl2g = sl2, sl2g8 = sl2, vsg = 1.f, vsg8 = 1.f;
                // rows of V past the context may hold any bits (even NaN): zero them in registers
                uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
                if (rem < kBlockSize) {
                    keep0 = (2 * t4 < rem ? 0x0000ffffu : 0u) | (2 * t4 + 1 < rem ? 0xffff0000u : 0u);
                    keep1 = (8 + 2 * t4 < rem ? 0x0000ffffu : 0u) | (9 + 2 * t4 < rem ? 0xffff0000u : 0u);
                }
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t va[D / 16][4];
                uint32_t vbase = 0;
                const int mi = lane >> 3;
                if constexpr (kFp8) {
                    // the record: K codes (a row per token, chunks permuted), K scales, V codes (a row of 16
                    // tokens per dim), V scales
                    const uint8_t* kt = wring + s * C::kStageBytes;
                    const float* sk = reinterpret_cast<const float*>(kt + C::kCodeTileBytes);
                    const uint8_t* vt = kt + C::kCodeTileBytes + C::kScaleBytes;
                    const float* sv = reinterpret_cast<const float*>(vt + C::kCodeTileBytes);
                    sl2g = sl2 * sk[g];
                    sl2g8 = sl2 * sk[g + 8];
                    vsg = g < rem ? sv[g] : 0.f;
                    vsg8 = g + 8 < rem ? sv[g + 8] : 0.f;
                    // ---- S^T = K Q^T: rows = the 16 tokens, columns = the 8 head slots; lane (g, t) reads
                    // dims 4t..4t+3 of the group for tokens g and g+8 ----
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(kt + koff[ks]);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kt + koff[ks] + 8 * D);
                        mma_f16_16816(sc, e4m3x2_to_half2(w0), e4m3x2_to_half2(w1), e4m3x2_to_half2(w0 >> 16),
                                      e4m3x2_to_half2(w1 >> 16), qa[ks][0], qa[ks][1]);
                    }
                    // V^T fragments: dims g, g+8 of each group of 16, tokens 2t, 2t+1 | 2t+8, 2t+9 (bytes 4t..4t+3)
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vt + (16 * mt + g) * kBlockSize + 4 * t4);
                        const uint32_t w1 =
                            *reinterpret_cast<const uint32_t*>(vt + (16 * mt + g + 8) * kBlockSize + 4 * t4);
                        va[mt][0] = e4m3x2_to_half2(w0);
                        va[mt][1] = e4m3x2_to_half2(w1);
                        va[mt][2] = e4m3x2_to_half2(w0 >> 16);
                        va[mt][3] = e4m3x2_to_half2(w1 >> 16);
                    }
                    if (rem < kBlockSize) {
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            va[mt][0] &= keep0;
                            va[mt][1] &= keep0;
                            va[mt][2] &= keep1;
                            va[mt][3] &= keep1;
                        }
                    }
                    {
                        // the stage may be refilled once its codes and scales are in registers
                        uint32_t dep = 0;
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(dep) : "r"(va[mt][0]), "r"(va[mt][1]));
                            asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(dep) : "r"(va[mt][2]), "r"(va[mt][3]));
                        }
                        asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(dep)
                                     : "r"(__float_as_uint(sl2g)), "r"(__float_as_uint(sl2g8)));
                        asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(dep)
                                     : "r"(__float_as_uint(vsg)), "r"(__float_as_uint(vsg8)));
                    }
                    refill(s);
                    refilled = true;
                } else {
                    const uint32_t kbase = smem_u32(wring + s * C::kStageBytes);
                    vbase = kbase + C::kTileBytes;
                    if (jj == app_blk) {
                        const int c = lane & 15;
                        if (c < D / 8) {
                            const uint32_t a = (lane >= 16 ? vbase : kbase) + swz(app_row, c);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(app_val.x),
                                         "r"(app_val.y), "r"(app_val.z), "r"(app_val.w)
                                         : "memory");
                            __half* dst = (lane >= 16 ? p.v_cache : p.k_cache) +
                                          ((static_cast<int64_t>(phys) * p.Hkv + kvh) * kBlockSize + app_row) * D +
                                          c * 8;
                            if (hc == 0) *reinterpret_cast<uint4*>(dst) = app_val;  // one head chunk writes
                        }
                        __syncwarp();
                    }
                    // ---- S^T = K Q^T: rows = the 16 tokens, columns = the 8 head slots; the head-dim steps go to
                    // two accumulators in turn (two independent product chains), summed at the end ----
                    float sc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kbase + swz((mi & 1) * 8 + (lane & 7), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                        if (ks & 1)
                            mma_f16_16816(sc2, a0, a1, a2, a3, qa[ks][0], qa[ks][1]);
                        else
                            mma_f16_16816(sc, a0, a1, a2, a3, qa[ks][0], qa[ks][1]);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) sc[k] += sc2[k];
#if KVC_DEC_EARLY_REFILL
                    // V^T fragments now; the stage is then free and its refill goes out before the softmax
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt)
                        ldsm_x4_t(vbase + swz((mi >> 1) * 8 + (lane & 7), 2 * mt + (mi & 1)), va[mt][0], va[mt][1],
                                  va[mt][2], va[mt][3]);
                    if (rem < kBlockSize) {  // the context's last block (warp-uniform)
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            va[mt][0] &= keep0;
                            va[mt][1] &= keep0;
                            va[mt][2] &= keep1;
                            va[mt][3] &= keep1;
                        }
                    }
                    // the copy may overwrite the stage only once the warp's reads of it have returned: one register
                    // of each ldmatrix folded (a warp issues in order, and an ldmatrix's four registers arrive
                    // together), so the refill below cannot issue before every read is back (the K fragments were
                    // consumed by the S products above)
                    uint32_t dep = 0;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) asm volatile("xor.b32 %0, %0, %1;" : "+r"(dep) : "r"(va[mt][0]));
                    refill(s);
                    refilled = true;
#endif
                }
                // ---- online softmax per head (column): this lane holds tokens g, g+8 of heads 2*t4, 2*t4+1 ----
                float x[4];
                x[0] = g < rem ? sc[0] * sl2g : -INFINITY;
                x[1] = g < rem ? sc[1] * sl2g : -INFINITY;
                x[2] = g + 8 < rem ? sc[2] * sl2g8 : -INFINITY;
                x[3] = g + 8 < rem ? sc[3] * sl2g8 : -INFINITY;
                float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
                // the running maxima move only when a score exceeds them by more than 2^KVC_DEC_LAZY_MAX (always
                // in the first block, where they are -inf); the weights below stay <= 2^KVC_DEC_LAZY_MAX
                if (KVC_DEC_LAZY_MAX == 0 || __any_sync(0xffffffffu, mx0 > m_run[0] + KVC_DEC_LAZY_MAX ||
                                                                      mx1 > m_run[1] + KVC_DEC_LAZY_MAX)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                    const float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);
                    m_run[0] = mn0;
                    m_run[1] = mn1;
                    l_run[0] *= al0;
                    l_run[1] *= al1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        o[mt][0] *= al0;
                        o[mt][1] *= al1;
                        o[mt][2] *= al0;
                        o[mt][3] *= al1;
                    }
                }
                const float p0 = ex2(x[0] - m_run[0]), p1 = ex2(x[1] - m_run[1]), p2 = ex2(x[2] - m_run[0]),
                            p3 = ex2(x[3] - m_run[1]);
                // P^T as the B operand (k = tokens, n = heads): transpose the two 8x8 halves in registers;
                // P = hi + lo, both fp16, so the P V product keeps ~fp32 accuracy
                const float q0 = p0 * vsg, q1 = p1 * vsg, q2 = p2 * vsg8, q3 = p3 * vsg8;
                const uint32_t h01 = pack_half2(q0, q1), h23 = pack_half2(q2, q3);
                const float2 f01 = unpack_half2(h01), f23 = unpack_half2(h23);
                const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
                constexpr bool kOneP = kFp8 && KVC_DEC_FP8_ONE_P;
                uint32_t bl0 = 0, bl1 = 0;
                if constexpr (kOneP) {
                    // one fp16 operand q = p x scale: the sums take each rounded q back over its scale (a key with
                    // a zero scale, an all-zero row, still counts its weight p)
                    const float r = rcp_approx(vsg), r8 = rcp_approx(vsg8);
                    l_run[0] += (vsg > 0.f ? f01.x * r : p0) + (vsg8 > 0.f ? f23.x * r8 : p2);
                    l_run[1] += (vsg > 0.f ? f01.y * r : p1) + (vsg8 > 0.f ? f23.y * r8 : p3);
                } else {
                    l_run[0] += p0 + p2;
                    l_run[1] += p1 + p3;
                    bl0 = movmatrix_trans(pack_half2(q0 - f01.x, q1 - f01.y));
                    bl1 = movmatrix_trans(pack_half2(q2 - f23.x, q3 - f23.y));
                }
                // ---- O^T += V^T P^T, one m-tile per 16 dims ----
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    uint32_t a0 = va[mt][0], a1 = va[mt][1], a2 = va[mt][2], a3 = va[mt][3];
#if !KVC_DEC_EARLY_REFILL
                    if constexpr (!kFp8) {
                        ldsm_x4_t(vbase + swz((mi >> 1) * 8 + (lane & 7), 2 * mt + (mi & 1)), a0, a1, a2, a3);
                        a0 &= keep0;
                        a1 &= keep0;
                        a2 &= keep1;
                        a3 &= keep1;
                    }
#endif
                    mma_f16_16816(o[mt], a0, a1, a2, a3, bh0, bh1);
                    if constexpr (!kOneP) mma_f16_16816(o[mt], a0, a1, a2, a3, bl0, bl1);
                }
            }
            if (!refilled) refill(s);
        }
    }
#if KVC_DEC_TRIGGER == 4
    grid_dependents_launch();  // the next kernel may start its prologue while this one finishes
#endif
    KVC_TRACE_MARK(3);
    if (timed_out) {
        if (lane == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
        // let copies still in flight land before the shared memory is reused
#pragma unroll
        for (int s = 0; s < ST; ++s)
            if (blk[s] >= 0) mbar_wait_bounded(&wbars[s], (phase >> s) & 1u, kWaitLimitNs / 8);
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {  // per-lane partial sums over the lanes of a head pair
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }

    // ---- merge the warps of this CTA (each warp parks its state in its own ring) ----
    __syncwarp();
    float* wm = reinterpret_cast<float*>(wring);  // [8] m, [8] l, then [8 heads][D+4] acc
    if (g == 0) {
        wm[2 * t4] = m_run[0];
        wm[2 * t4 + 1] = m_run[1];
        wm[8 + 2 * t4] = l_run[0];
        wm[8 + 2 * t4 + 1] = l_run[1];
    }
    float* wo = wm + 16;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int d = mt * 16 + g;
        wo[(2 * t4) * C::kMergeStride + d] = o[mt][0];
        wo[(2 * t4 + 1) * C::kMergeStride + d] = o[mt][1];
        wo[(2 * t4) * C::kMergeStride + d + 8] = o[mt][2];
        wo[(2 * t4 + 1) * C::kMergeStride + d + 8] = o[mt][3];
    }
    __syncthreads();
    KVC_TRACE_MARK(4);
#if KVC_DEC_TRIGGER == 5
    grid_dependents_launch();
#endif

    const bool final_here = nclus == 1 && !kSuffix;  // this cluster's result is the output
    const bool direct = final_here && cs == 1;                  // a single CTA holds the whole range
    const int stride = 16 + Gc * D;  // floats per cluster merge slot: m[8], l[8], acc[Gc][D]
    // in a cluster this CTA's merged state goes to its slot in rank 0: rank 0's own state at s_m, or
    // inbox slot rank - 1 (same layout)
    uint32_t slot = 0, remote_bar = 0;
    if (cs > 1) {
        // every CTA of the cluster has started (the prologue arrive), so rank 0's shared memory is live
        if (!KVC_DEC_EARLY_CLUSTER_WAIT) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        slot = map_to_rank(rank == 0 ? s_m : s_inbox + (rank - 1) * stride, 0);
        remote_bar = map_to_rank(inbox_bar, 0);
    }
    const bool push_async = KVC_DEC_ASYNC_PUSH && cs > 1 && rank != 0;
    // every thread merges the warps of this CTA for four consecutive outputs (head gg, dims d..d+3): it
    // takes the CTA maximum M of its head and the warp weights 2^(m_w - M) itself, so no further barrier
    // is needed
    {
        constexpr int kRingF = C::kWarpRingBytes / 4;
        const float* wst = reinterpret_cast<const float*>(smem);  // warp w's parked state at w * kRingF
        for (int e = 4 * threadIdx.x; e < Gc * D; e += 4 * C::kThreads) {
            const int gg = e / D, d = e % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, wst[w * kRingF + gg]);
            float L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float* r = wst + w * kRingF;
                const float wgt = M == -INFINITY ? 0.f : ex2(r[gg] - M);  // an empty warp has m = -inf: weight 0
                L += r[8 + gg] * wgt;
                O = fma4(wgt, *reinterpret_cast<const float4*>(r + 16 + gg * C::kMergeStride + d), O);
            }
            const int64_t h = static_cast<int64_t>(b) * p.Hq + h0 + gg;
            if (direct) {
                store_out4(p.out, p.out_f32, h * D + d, scale4(O, L > 0.f ? 1.f / L : 0.f));
            } else if (cs == 1) {  // one CTA per cluster: its state is the cluster's partial
                const int64_t row = h * p.part_stride + (kSuffix ? p.part_base : 0) + cidx;
                *reinterpret_cast<float4*>(p.part_acc + row * D + d) = O;
                if (d == 0) {
                    p.part_ml[row * 2 + 0] = M;
                    p.part_ml[row * 2 + 1] = L;
                }
            } else if (push_async) {
                st_async_f32x4(slot + 4u * (16 + e), O, remote_bar);
                if (d == 0) {
                    st_async_f32(slot + 4u * gg, M, remote_bar);
                    st_async_f32(slot + 4u * (8 + gg), L, remote_bar);
                }
            } else {
                asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(slot + 4u * (16 + e)),
                             "f"(O.x), "f"(O.y), "f"(O.z), "f"(O.w)
                             : "memory");
                if (d == 0) {
                    st_cluster_f32(slot + 4u * gg, M);
                    st_cluster_f32(slot + 4u * (8 + gg), L);
                }
            }
        }
    }
    if (cs == 1) {
        KVC_TRACE_END();
        return;
    }
    KVC_TRACE_MARK(5);

    // ---- merge the CTAs of this cluster in rank 0 ----
#if KVC_DEC_ASYNC_PUSH
    // every other CTA has issued its asynchronous pushes and leaves (nothing of it is read by others); rank 0
    // waits until all their bytes have landed on its inbox barrier (acquire at cluster scope makes them visible)
    // and its own state is in place, and merges locally
    if (rank != 0) {
        KVC_TRACE_MARK(6);
        KVC_TRACE_END();
        return;
    }
    __syncthreads();  // rank 0's own merged state (written by all its threads) is complete
    if (!mbar_wait_cluster_bounded(inbox_bar, 0, 4 * kWaitLimitNs)) {
        if (threadIdx.x == 0) atomicOr(p.err, KVC_DEVERR_TIMEOUT);
    }
#else
    // every CTA has pushed its state into its slot (remote stores, no round trip); it arrives on the cluster
    // barrier (release) and leaves. Rank 0 waits for all arrivals (acquire), which makes every slot visible to
    // it, and merges locally
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (rank != 0) {
        KVC_TRACE_MARK(6);
        KVC_TRACE_END();
        return;  // nothing of this CTA is read by others
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
#endif
    KVC_TRACE_MARK(6);
    // slot c of the merge: c == 0 is this CTA's own state, c >= 1 the inbox slot of rank c; a CTA without
    // blocks has l = 0 and takes no part
    auto src = [&](int c) -> const float* { return c == 0 ? s_m : s_inbox + (c - 1) * stride; };
    for (int e = 4 * threadIdx.x; e < Gc * D; e += 4 * C::kThreads) {
        const int gg = e / D, d = e % D;
        float M = -INFINITY;
        for (int c = 0; c < cs; ++c)
            if (src(c)[8 + gg] > 0.f) M = fmaxf(M, src(c)[gg]);
        float L = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < cs; ++c) {
            const float* r = src(c);
            const float l = r[8 + gg];
            const float w = l > 0.f ? ex2(r[gg] - M) : 0.f;
            L += l * w;
            O = fma4(w, *reinterpret_cast<const float4*>(r + 16 + e), O);
        }
        const int64_t h = static_cast<int64_t>(b) * p.Hq + h0 + gg;
        if (final_here) {
            store_out4(p.out, p.out_f32, h * D + d, scale4(O, L > 0.f ? 1.f / L : 0.f));
        } else {
            const int64_t row = h * p.part_stride + (kSuffix ? p.part_base : 0) + cidx;
            *reinterpret_cast<float4*>(p.part_acc + row * D + d) = O;
            if (d == 0) {
                p.part_ml[row * 2 + 0] = M;
                p.part_ml[row * 2 + 1] = L;
            }
        }
    }
    KVC_TRACE_END();
}



// Merge the partial states of every (sequence, query head): the clusters along a context longer than
// one cluster covers, and in a cascade also the parts of the shared prefix.  The merge rule is the
// FlashAttention article's ("Was ist der mathematische Aspekt von Softmax?"): with M the largest part
// maximum, out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s over the parts that saw a token (l > 0).
// Written for latency, since the parts sit in L2 and there are few of them: every thread loads the (m, l)
// of its parts at once for M, then for L, then each thread accumulates one float4 of dims over a strided
// subset of the parts (independent loads, no running-maximum chain), and the subsets are summed in shared
// memory.  An earlier form walked the parts with a running (M, L, acc) per warp, one dependent L2 round
// trip per part.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_combine_kernel(const CombineParams p) {
    constexpr int NT = 256, Q = D / 4, NPG = NT / Q;  // float4 columns of a row; part subsets
    __shared__ float4 s_o[NPG][Q];
    const int h = blockIdx.x, y = blockIdx.y, b = y / p.q_len;  // y: the query row (a sequence's token)
    const int tid = threadIdx.x;
    // With early_release the next kernel (the next layer's decode) may launch and fetch its tables and first K/V
    // tiles while this one waits; its own dependency wait still covers this grid, whose completion covers the
    // decode before it.  The host asks for it only where a decode grid of this shape takes at most half the
    // resident CTA slots, so the next one fits beside the current one: on grids that fill the GPU the early
    // launch made the next grid's clusters land piecemeal in the slots the current one frees, and the layer of a
    // 24-layer step slowed (B = 1 x 131072: 17.1 -> 20.2 us; B = 1 x 4096: 6.0 -> 4.9 us, where it fits).
    if (KVC_COMBINE_EARLY_TRIGGER && p.early_release) grid_dependents_launch();
    // context lengths and prefix offsets are never written by the kernel before (the launch-overlap contract):
    // they are read before the dependency wait, the parts and the output only after it
    const int ctx_full = p.context_lens[b];
    const int off = p.blk_off != nullptr ? p.blk_off[b] : 0;
    const int ctx = ctx_full - off * kBlockSize;  // tokens of the suffix parts
    const bool bad = off < 0 || off >= p.max_blocks || ctx_full < p.q_len || ctx_full > p.max_blocks * kBlockSize ||
                     ctx_full > p.max_ctx || ctx < 1;
    const int nsuf = bad ? 0 : ((ctx + kBlockSize - 1) / kBlockSize + p.bpc - 1) / p.bpc;
    const int npre = off > 0 && p.prefix_chunk > 0 ? (off + p.prefix_chunk - 1) / p.prefix_chunk : 0;
    if (!bad && !p.cascade && nsuf <= 1) {  // the cluster wrote the output itself
        leave_before_dependency_wait();
        return;
    }
    grid_dependency_wait();
    if (bad) {
        if (p.cascade) {  // the attention kernels left this row to us
            if (h == 0 && tid == 0) atomicOr(p.err, KVC_DEVERR_CONTEXT);
            if (tid < D) store_out(p.out, p.out_f32, (static_cast<int64_t>(y) * p.Hq + h) * D + tid, 0.f);
        }
        return;
    }
    const int n = npre + nsuf;
    const int64_t row0 = (static_cast<int64_t>(y) * p.Hq + h) * p.part_stride;
    auto part_row = [&](int s) -> int64_t { return row0 + (s < npre ? s : p.part_base + s - npre); };
    auto ml_of = [&](int s) { return *reinterpret_cast<const float2*>(p.part_ml + part_row(s) * 2); };

#if KVC_COMBINE_ONE_PASS
    // One pass over the parts: thread (pg, q) keeps a running maximum, sum and float4 column q of the
    // accumulator over parts pg, pg + NPG, ... (online rescaling, so every load can be in flight at once); the
    // NPG part subsets are then merged in shared memory by the threads of the first subset.
    __shared__ float s_mg[NPG], s_lg[NPG];
    const int q = tid % Q, pg = tid / Q;
    float mt = -INFINITY, lt = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = pg; s < n; s += NPG) {
        const int64_t r = part_row(s);
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + r * 2);
        const float4 a = *reinterpret_cast<const float4*>(p.part_acc + r * D + 4 * q);
        if (ml.y > 0.f) {  // a part that saw no token adds nothing
            const float mn = fmaxf(mt, ml.x);
            const float c_old = mt == -INFINITY ? 0.f : ex2(mt - mn), c_new = ex2(ml.x - mn);
            O = fma4(c_new, a, scale4(O, c_old));
            lt = lt * c_old + ml.y * c_new;
            mt = mn;
        }
    }
    s_o[pg][q] = O;
    if (q == 0) {  // every thread of a subset saw the same parts: one (m, l) per subset
        s_mg[pg] = mt;
        s_lg[pg] = lt;
    }
    __syncthreads();
    if (tid < Q) {
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < NPG; ++k) M = fmaxf(M, s_mg[k]);
        float L = 0.f;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NPG; ++k) {
            const float w = s_mg[k] == -INFINITY ? 0.f : ex2(s_mg[k] - M);
            L += s_lg[k] * w;
            t = fma4(w, s_o[k][tid], t);
        }
        store_out4(p.out, p.out_f32, (static_cast<int64_t>(y) * p.Hq + h) * D + 4 * tid,
                   scale4(t, L > 0.f ? 1.f / L : 0.f));
    }
#else
    // two passes: the maximum over every part first, then the weighted sums
    __shared__ float s_red[NT / 32];
    // M: the largest maximum among the parts that saw a token
    float mx = -INFINITY;
    for (int s = tid; s < n; s += NT) {
        const float2 ml = ml_of(s);
        if (ml.y > 0.f) mx = fmaxf(mx, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) s_red[tid >> 5] = mx;
    __syncthreads();
    float M = s_red[0];
#pragma unroll
    for (int k = 1; k < NT / 32; ++k) M = fmaxf(M, s_red[k]);
    __syncthreads();  // s_red is reused below
    // L = sum_s 2^(m_s - M) l_s
    float ls = 0.f;
    for (int s = tid; s < n; s += NT) {
        const float2 ml = ml_of(s);
        if (ml.y > 0.f) ls += ml.y * ex2(ml.x - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if ((tid & 31) == 0) s_red[tid >> 5] = ls;
    // acc: thread (pg, q) sums float4 column q over parts pg, pg + NPG, ...
    const int q = tid % Q, pg = tid / Q;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = pg; s < n; s += NPG) {
        const int64_t r = part_row(s);
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + r * 2);
        const float4 a = *reinterpret_cast<const float4*>(p.part_acc + r * D + 4 * q);
        O = fma4(ml.y > 0.f ? ex2(ml.x - M) : 0.f, a, O);
    }
    s_o[pg][q] = O;
    __syncthreads();
    if (tid < Q) {
        float L = 0.f;
#pragma unroll
        for (int k = 0; k < NT / 32; ++k) L += s_red[k];
        float4 t = s_o[0][tid];
#pragma unroll
        for (int k = 1; k < NPG; ++k) {
            const float4 u = s_o[k][tid];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        store_out4(p.out, p.out_f32, (static_cast<int64_t>(y) * p.Hq + h) * D + 4 * tid,
                   scale4(t, L > 0.f ? 1.f / L : 0.f));
    }
#endif
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// one-time kernel attributes (largest shared-memory size this kernel can be launched with)
template <int D>
static cudaError_t decode_setup() {
    using C = DecodeCfg<D>;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        for (auto kern : {paged_decode_kernel<D, false>, paged_decode_kernel<D, true>}) {
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::smem_bytes(kMaxCluster, 8, kMaxClusterBlocks));
            if (err == cudaSuccess && kMaxCluster > 8)
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(paged_decode_kernel<D, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecodeCfg<D, true>::smem_bytes(kMaxCluster, 8, kMaxClusterBlocks));
        if (err == cudaSuccess && kMaxCluster > 8)
            err = cudaFuncSetAttribute(paged_decode_kernel<D, false, true>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    return err;
}

// resident CTAs per SM of the decode kernel with `smem` bytes of dynamic shared memory (cached)
template <int D>
static cudaError_t decode_occupancy(int smem, int* ctas) {
    using C = DecodeCfg<D>;
    static std::mutex mu;
    static int cached_smem[64] = {0}, cached_occ[64] = {0};
    cudaError_t e = decode_setup<D>();
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < 64; ++i)
        if (cached_smem[i] == smem) {
            *ctas = cached_occ[i];
            return cudaSuccess;
        }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, paged_decode_kernel<D, false>, C::kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    for (int i = 0; i < 64; ++i)
        if (cached_smem[i] == 0) {
            cached_smem[i] = smem;
            cached_occ[i] = occ;
            break;
        }
    *ctas = occ;
    return cudaSuccess;
}

// thread-block clusters of cs CTAs (smem bytes of dynamic shared memory each) that can be resident at once: the
// clusters of one launch are placed within a GPC each, so this is below SMs x CTAs-per-SM / cs for larger clusters
// (cached per (cs, smem))
template <int D>
static cudaError_t decode_resident_clusters(int cs, int smem, int* clusters) {
    using C = DecodeCfg<D>;
    static std::mutex mu;
    static int cached_key[256] = {0}, cached_val[256] = {0};
    cudaError_t e = decode_setup<D>();
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int key = ((dev * 32 + cs) << 20) + smem + 1;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < 256; ++i)
        if (cached_key[i] == key) {
            *clusters = cached_val[i];
            return cudaSuccess;
        }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(cs);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, paged_decode_kernel<D, false>, &cfg);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < 256; ++i)
        if (cached_key[i] == 0) {
            cached_key[i] = key;
            cached_val[i] = n;
            break;
        }
    *clusters = n;
    return cudaSuccess;
}

template <int D>
static cudaError_t plan_d(int B, int Hq, int Hkv, int max_ctx, int bpc_req, DecodePlan* plan) {
    using C = DecodeCfg<D>;
    const int nblk = std::max((max_ctx + kBlockSize - 1) / kBlockSize, 1);
    const int Gfull = std::max(1, Hq / std::max(Hkv, 1));
    const int G = std::min(Gfull, 8);            // query heads of one CTA
    const int hchunks = (Gfull + 7) / 8;          // CTAs per (sequence, KV head) along the heads
    int cs = 1, bpc = nblk;
    if (bpc_req > 0) {
        bpc = std::min(bpc_req, kMaxClusterBlocks);
        cs = std::max(1, std::min(kMaxCluster, (bpc + C::kWarps - 1) / C::kWarps));
    } else {
        // One wave, few parts.  For cluster sizes from the largest down, the clusters that can be resident
        // (KVC_DEC_PLAN_CTAS of the CTAs an SM holds, the rest left for the next launch) are shared out over the
        // (sequence, KV head, head chunk) units; a unit takes one cluster per cs x warps x
        // KVC_DEC_MIN_BLOCKS_PER_WARP blocks of its context, up to its share.  A plan with several clusters per
        // unit needs the combine launch; below KVC_DEC_SMALL_BYTES of K/V such a plan keeps to half the resident
        // clusters, so that the combine can let the next launch (the next layer) start beside it.  The largest
        // cluster size that gives every unit its clusters wins; where none does, each unit gets one CTA (several
        // waves).
        const int smem_est = C::smem_bytes(kMaxCluster, G, std::min(nblk, kMaxClusterBlocks));
        int occ = 0;
        cudaError_t e = decode_occupancy<D>(smem_est, &occ);
        if (e != cudaSuccess) return e;
        const int64_t segs = std::max<int64_t>(1, static_cast<int64_t>(B) * Hkv * hchunks);
        const int64_t min_ncl = (nblk + kMaxClusterBlocks - 1) / kMaxClusterBlocks;
        const int64_t kv_bytes = static_cast<int64_t>(B) * Hkv * nblk * (2 * kBlockSize * D * 2);
        int64_t ncl = min_ncl;
        cs = 1;
        for (int c = kMaxCluster; c >= 1; --c) {
            if (c > 1 && (static_cast<int64_t>(c - 1) * C::kWarps >= nblk)) continue;  // a CTA would have no block
            int resident = 0;
            e = decode_resident_clusters<D>(c, C::smem_bytes(c, G, std::min(nblk, kMaxClusterBlocks)), &resident);
            if (e != cudaSuccess) return e;
            const int64_t usable = static_cast<int64_t>(resident) * std::min(occ, KVC_DEC_PLAN_CTAS) / occ;
            const int64_t per_seg = usable / segs;
            if (per_seg < min_ncl) continue;  // (the table-slice bound) clusters would spill into a second wave
            const int64_t span = static_cast<int64_t>(c) * C::kWarps * KVC_DEC_MIN_BLOCKS_PER_WARP;
            const int64_t want = (nblk + span - 1) / span;
            int64_t n = std::max(min_ncl, std::min(per_seg, want));
            if (n > 1 && kv_bytes < KVC_DEC_SMALL_BYTES) n = std::max(min_ncl, std::min((usable / 2) / segs, want));
            if (n > 1 && c > KVC_DEC_SPLIT_MAX_CLUSTER) continue;  // a plan with the combine: smaller clusters
            ncl = n;
            cs = c;
            break;
        }
        bpc = static_cast<int>((nblk + ncl - 1) / ncl);
    }
    const int nparts = (nblk + bpc - 1) / bpc;
    plan->blocks_per_split = bpc;
    plan->cluster = cs;
    plan->num_parts = nparts;
    plan->num_splits = nparts * cs;  // grid.x: whole clusters
    plan->workspace_bytes = nparts > 1 ? partials_bytes(static_cast<size_t>(B) * Hq * nparts, D) : 0;
    return cudaSuccess;
}

cudaError_t decode_plan(int B, int Hq, int Hkv, int D, int max_ctx, int bpc_req, DecodePlan* plan) {
    switch (D) {
        case 64: return plan_d<64>(B, Hq, Hkv, max_ctx, bpc_req, plan);
        case 128: return plan_d<128>(B, Hq, Hkv, max_ctx, bpc_req, plan);
        default: return cudaErrorInvalidValue;
    }
}

// kernel parameters of a plain decode call (one part per cluster, final output where one cluster covers
// the context); the cascade launch adjusts the partial layout and the block offset
static DecodeKernelParams decode_params(const DecodeArgs& a, const DecodePlan& plan, float* part_ml, float* part_acc) {
    DecodeKernelParams p;
    p.q = a.q;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_cache = const_cast<__half*>(a.k_cache);
    p.v_cache = const_cast<__half*>(a.v_cache);
    p.block_table = a.block_table;
    p.context_lens = a.context_lens;
    p.out = a.out;
    p.part_ml = part_ml;
    p.part_acc = part_acc;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.hchunks = (p.G + 7) / 8;
    p.max_ctx = a.max_context_len;
    p.bpc = plan.blocks_per_split;
    p.csize = plan.cluster;
    p.part_base = 0;
    p.part_stride = plan.num_parts;
    p.blk_off = nullptr;
    p.kv_fp8 = a.kv_fp8;
    p.out_f32 = a.out_f32;
    p.len_order = 0;
    p.scale_log2 = a.scale * kLog2e;
    static std::atomic<unsigned> launch_seq{0};
    p.trace_seq = launch_seq.fetch_add(1);
    return p;
}

// 1 where the grid has more CTAs than can be resident at once (several waves): the kernel then dispatches the
// longest contexts first
template <int D>
static int len_order_for(const DecodeArgs& a, const DecodePlan& plan, int hchunks, int smem) {
    if (!KVC_DEC_LEN_ORDER || a.B < 2 || a.B > kLenOrderMaxB) return 0;
    int occ = 0;
    if (decode_occupancy<D>(smem, &occ) != cudaSuccess) return 0;
    const int64_t ctas = static_cast<int64_t>(plan.num_splits) * a.Hkv * hchunks * a.B;
    return ctas > static_cast<int64_t>(occ) * sm_count() ? 1 : 0;
}

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    cudaError_t e = decode_setup<D>();
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    const bool fp8 = a.kv_fp8 != nullptr;
    CUtensorMap tmK, tmV;  // fp8: the records come by bulk copies and the maps are unused
    if (fp8) {
        memset(&tmK, 0, sizeof(tmK));
        memset(&tmV, 0, sizeof(tmV));
    } else {
        e = make_tile_map(&tmK, a.k_cache, D, rows);
        if (e == cudaSuccess) e = make_tile_map(&tmV, a.v_cache, D, rows);
        if (e != cudaSuccess) return e;
    }

    const size_t nrow = static_cast<size_t>(a.B) * a.Hq * plan.num_parts;
    float* part_ml = plan.num_parts > 1 ? static_cast<float*>(a.workspace) : nullptr;
    DecodeKernelParams p = decode_params(a, plan, part_ml, part_ml ? partials_acc(part_ml, nrow) : nullptr);
    const bool pdl = g_launch_overlap.load(std::memory_order_relaxed) != 0;
    dim3 grid(plan.num_splits, a.Hkv * p.hchunks, a.B);
    p.len_order = len_order_for<D>(a, plan, p.hchunks,
                                   fp8 ? DecodeCfg<D, true>::smem_bytes(plan.cluster, std::min(p.G, 8),
                                                                        plan.blocks_per_split)
                                       : C::smem_bytes(plan.cluster, std::min(p.G, 8), plan.blocks_per_split));
    if (fp8)
        e = launch(paged_decode_kernel<D, false, true>, grid, dim3(DecodeCfg<D, true>::kThreads),
                   DecodeCfg<D, true>::smem_bytes(plan.cluster, std::min(p.G, 8), plan.blocks_per_split), stream, pdl,
                   static_cast<unsigned>(plan.cluster),
                   tmK, tmV, p);
    else
        e = launch(paged_decode_kernel<D, false>, grid, dim3(C::kThreads),
                   C::smem_bytes(plan.cluster, std::min(p.G, 8), plan.blocks_per_split), stream,
                   pdl, static_cast<unsigned>(plan.cluster), tmK, tmV, p);
    if (e != cudaSuccess) return e;
    if (plan.num_parts > 1) {
        CombineParams c;
        c.part_ml = p.part_ml;
        c.part_acc = p.part_acc;
        c.context_lens = a.context_lens;
        c.blk_off = nullptr;
        c.out = a.out;
        c.err = a.err;
        c.Hq = a.Hq;
        c.part_stride = plan.num_parts;
        c.part_base = 0;
        c.bpc = plan.blocks_per_split;
        c.max_blocks = a.max_blocks;
        c.max_ctx = a.max_context_len;
        c.out_f32 = a.out_f32;
        c.prefix_chunk = 0;
        c.cascade = 0;
        c.q_len = 1;
        // release the next kernel at the combine's start when two decode grids of this shape fit at once
        int occ = 0;
        const int smem = C::smem_bytes(plan.cluster, std::min(p.G, 8), plan.blocks_per_split);
        c.early_release = 0;
        if (!fp8 && decode_occupancy<D>(smem, &occ) == cudaSuccess)
            c.early_release = KVC_COMBINE_EARLY_ALWAYS ||
                              2 * static_cast<int64_t>(grid.x) * grid.y * grid.z <= static_cast<int64_t>(occ) * sm_count();
        e = launch(paged_decode_combine_kernel<D>, dim3(a.Hq, a.B), dim3(256), 0, stream, true, 1u, c);
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

cudaError_t launch_combine(const CombineParams& c, int D, int rows, cudaStream_t stream) {
    switch (D) {
        case 64: return launch(paged_decode_combine_kernel<64>, dim3(c.Hq, rows), dim3(256), 0, stream, true, 1u, c);
        case 128: return launch(paged_decode_combine_kernel<128>, dim3(c.Hq, rows), dim3(256), 0, stream, true, 1u, c);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
static cudaError_t launch_suffix_d(const DecodeArgs& a, const DecodePlan& plan, const int32_t* blk_off, int part_base,
                                   int part_stride, float* part_ml, float* part_acc, cudaStream_t stream) {
    using C = DecodeCfg<D>;
    cudaError_t e = decode_setup<D>();
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.Hkv * kBlockSize;
    CUtensorMap tmK, tmV;
    e = make_tile_map(&tmK, a.k_cache, D, rows);
    if (e != cudaSuccess) return e;
    e = make_tile_map(&tmV, a.v_cache, D, rows);
    if (e != cudaSuccess) return e;
    DecodeKernelParams p = decode_params(a, plan, part_ml, part_acc);
    p.blk_off = blk_off;
    p.part_base = part_base;
    p.part_stride = part_stride;
    p.len_order = len_order_for<D>(a, plan, p.hchunks, C::smem_bytes(plan.cluster, std::min(p.G, 8),
                                                                     plan.blocks_per_split));
    const bool pdl = g_launch_overlap.load(std::memory_order_relaxed) != 0;
    return launch(paged_decode_kernel<D, true>, dim3(plan.num_splits, a.Hkv * p.hchunks, a.B), dim3(C::kThreads),
                  C::smem_bytes(plan.cluster, std::min(p.G, 8), plan.blocks_per_split), stream, pdl,
                  static_cast<unsigned>(plan.cluster), tmK, tmV, p);
}

cudaError_t launch_decode_suffix(const DecodeArgs& a, const DecodePlan& plan, const int32_t* blk_off, int part_base,
                                 int part_stride, float* part_ml, float* part_acc, cudaStream_t stream) {
    switch (a.D) {
        case 64: return launch_suffix_d<64>(a, plan, blk_off, part_base, part_stride, part_ml, part_acc, stream);
        case 128: return launch_suffix_d<128>(a, plan, blk_off, part_base, part_stride, part_ml, part_acc, stream);
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

// ---------------------------------------------------------------------------
// Allocation-free decode: the split partials live in a fixed array that the
// library holds in device memory instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB on every device that loads the library
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace on the current device, looked up once per device (host code
// cannot use the symbol itself: on the host it only names a stand-in, not device memory).
static cudaError_t static_workspace_address(void** out) {
    static std::atomic<void*> cache[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    void* p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return e;
        cache[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace kvc

extern "C" kvc_status paged_decode_attention_static_workspace(
    const void* q, const void* k_cache, const void* v_cache, int num_blocks, const int32_t* block_table,
    int max_blocks, const int32_t* context_lens, int B, int Hq, int Hkv, int head_dim, int block_size,
    int max_context_len, float scale, void* out, int out_dtype, int blocks_per_split, void* stream) {
    using kvc::set_last_error;
    auto fail = [](kvc_status s, const char* m) { return static_cast<kvc_status>(set_last_error(s, m)); };
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (B < 0 || Hq < 1 || Hkv < 1 || max_context_len < 1 || num_blocks < 1 || max_blocks < 1 || blocks_per_split < 0)
        return fail(KVC_ERR_INVALID, "bad sizes");
    if (Hq % Hkv) return fail(KVC_ERR_INVALID, "Hq must be a multiple of Hkv");
    if (head_dim != 64 && head_dim != 128) return fail(KVC_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (block_size != kvc::kBlockSize) return fail(KVC_ERR_UNSUPPORTED, "block_size must be 16");
    if (B > 65535 || Hkv > 65535) return fail(KVC_ERR_UNSUPPORTED, "B and Hkv must be <= 65535");
    if (static_cast<int64_t>(num_blocks) * Hkv * block_size >= (int64_t(1) << 31))
        return fail(KVC_ERR_UNSUPPORTED, "num_blocks * Hkv * block_size must be < 2^31");
    if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks) * block_size)
        return fail(KVC_ERR_CAPACITY, "max_context_len beyond max_blocks * block_size");
    if (out_dtype != KVC_F16 && out_dtype != KVC_F32) return fail(KVC_ERR_INVALID, "bad out_dtype");
    if (B == 0) return KVC_OK;
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out) return fail(KVC_ERR_INVALID, "null pointer");
    if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al16(out))
        return fail(KVC_ERR_INVALID, "q, caches and out must be 16-byte aligned");
    kvc::DecodePlan plan;
    cudaError_t e = kvc::decode_plan(B, Hq, Hkv, head_dim, max_context_len, blocks_per_split, &plan);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, cudaGetErrorString(e));
    if (plan.workspace_bytes > kvc::kStaticWorkspaceBytes)
        return fail(KVC_ERR_CAPACITY,
                    "these sizes need more split scratch than the 16 MiB static workspace holds "
                    "(use paged_decode_attention with a caller workspace, or fewer splits)");
    kvc::DecodeArgs a;
    a.q = static_cast<const __half*>(q);
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.k_cache = static_cast<const __half*>(k_cache);
    a.v_cache = static_cast<const __half*>(v_cache);
    a.num_blocks = num_blocks;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.context_lens = context_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = head_dim;
    a.max_context_len = max_context_len;
    a.scale = scale;
    a.out = out;
    a.out_f32 = out_dtype == KVC_F32;
    a.blocks_per_split = blocks_per_split;
    a.workspace_bytes = kvc::kStaticWorkspaceBytes;
    e = kvc::static_workspace_address(&a.workspace);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, cudaGetErrorString(e));
    e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, cudaGetErrorString(e));
    e = kvc::launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KVC_ERR_CUDA, cudaGetErrorString(e));
    return KVC_OK;
}
