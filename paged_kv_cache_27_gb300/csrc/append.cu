// Append (slot-mapped scatter of new K/V rows into the paged cache) and
// whole-block copy (the device half of copy-on-write).
//
// Append is step 2 of a decode token in "La caché de claves y valores"
// (gustavoai.dev, section "Las claves y los valores de una posición no
// cambian"): k_t, v_t go to the end of each head's cache before attention.
// The slot of a token is block_table[pos / bs] * bs + pos % bs (PagedAttention
// article, chatgpz.de, SECTION 2); here the caller passes the slots.
// Copy-on-write (same article, SECTION 3): a sequence about to write into a
// shared block first gets a private copy of the whole block.
//
// Both kernels are pure bandwidth: 16-byte vector loads/stores, consecutive
// threads on consecutive 16-byte chunks of a row.  So is the staging copy at
// the end of this file, which moves a decode step's inputs in from pinned host
// memory (and its output back) inside the stream's kernel sequence.
#include <atomic>

#include "../../include/kvc.h"
#include "decode_common.cuh"
#include "kvc_internal.h"
#include "ptx.cuh"
#include "stage_copy.h"

namespace kvc {

__device__ unsigned g_error_word;

cudaError_t device_error_word(unsigned** ptr) {
    static std::atomic<unsigned*> cache[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) {
        unsigned* p = cache[dev].load(std::memory_order_acquire);
        if (p) {
            *ptr = p;
            return cudaSuccess;
        }
    }
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_error_word);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) cache[dev].store(static_cast<unsigned*>(addr), std::memory_order_release);
    *ptr = static_cast<unsigned*>(addr);
    return cudaSuccess;
}

// One thread per 16-byte chunk of a (token, KV head) row; rows of D fp16.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                         const uint4* __restrict__ v_new,
                                                         const int64_t* __restrict__ slots, int n,
                                                         uint4* __restrict__ k_layer, uint4* __restrict__ v_layer,
                                                         int num_blocks, int Hkv, int chunks_per_row,
                                                         unsigned* err) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t total = static_cast<int64_t>(n) * Hkv * chunks_per_row;
    if (idx >= total) return;
    const int c = static_cast<int>(idx % chunks_per_row);
    const int64_t row = idx / chunks_per_row;  // t * Hkv + h
    const int h = static_cast<int>(row % Hkv);
    const int64_t t = row / Hkv;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= static_cast<int64_t>(num_blocks) * kBlockSize) {
        if (c == 0) atomicOr(err, KVC_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
    const int64_t dst = ((blk * Hkv + h) * kBlockSize + off) * chunks_per_row + c;
    k_layer[dst] = k_new[idx];
    v_layer[dst] = v_new[idx];
}

cudaError_t launch_append(const __half* k_new, const __half* v_new, const int64_t* slots, int n, __half* k_layer,
                          __half* v_layer, int num_blocks, int Hkv, int D, unsigned* err, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int cpr = D / 8;
    const int64_t total = static_cast<int64_t>(n) * Hkv * cpr;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    kv_append_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new), slots, n,
        reinterpret_cast<uint4*>(k_layer), reinterpret_cast<uint4*>(v_layer), num_blocks, Hkv, cpr, err);
    return cudaGetLastError();
}

// Quantized cache (an extension; the pages fix no quantized format): rows of D fp16 values become e4m3 codes
// with one float scale per (token, KV head) row, so that appending a token never re-quantizes the rest of its
// block. One warp per (token, KV head, K or V) row: scale = absmax / 448 with IEEE division (1 for an all-zero
// row), code_i = e4m3(x_i / scale) rounded to nearest even, saturating at 448. Codes and scale go into the
// record of the slot's (block, KV head), [NB][Hkv][fp8_record_bytes(D)]: K codes at fp8_kswz(D, row, i), the
// K scale after the K codes, V codes in the block's dim rows at the token's position vt_pos, the V scale last.
template <int D>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const __half* __restrict__ k_new,
                                                            const __half* __restrict__ v_new,
                                                            const int64_t* __restrict__ slots, int n,
                                                            uint8_t* __restrict__ kv_fp8, int num_blocks, int Hkv,
                                                            unsigned* err) {
    constexpr int PER = D / 32;  // values per lane
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= static_cast<int64_t>(n) * Hkv * 2) return;  // whole warps
    const int kv = static_cast<int>(w & 1);
    const int64_t row = w >> 1;  // t * Hkv + h
    const int h = static_cast<int>(row % Hkv);
    const int64_t slot = slots[row / Hkv];
    if (slot < 0) return;
    if (slot >= static_cast<int64_t>(num_blocks) * kBlockSize) {
        if (lane == 0 && kv == 0) atomicOr(err, KVC_DEVERR_SLOT);
        return;
    }
    const __half* src = (kv ? v_new : k_new) + row * D + lane * PER;
    float x[PER];
    if constexpr (PER == 2) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(src));
        x[0] = f.x;
        x[1] = f.y;
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        x[0] = a.x;
        x[1] = a.y;
        x[2] = c.x;
        x[3] = c.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const int tok = static_cast<int>(slot % kBlockSize);
    uint8_t* rec = kv_fp8 + ((slot / kBlockSize) * Hkv + h) * static_cast<int64_t>(fp8_record_bytes(D));
    uint32_t codes = float2_to_e4m3x2(__fdiv_rn(x[0], sc), __fdiv_rn(x[1], sc));
    if constexpr (PER == 4) codes |= static_cast<uint32_t>(float2_to_e4m3x2(__fdiv_rn(x[2], sc), __fdiv_rn(x[3], sc))) << 16;
    if (kv == 0) {  // K: the token's row of D codes (its lane's PER codes stay inside one 16-byte chunk)
        uint8_t* dst = rec + fp8_kswz(D, tok, lane * PER);
        if constexpr (PER == 2)
            *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
        else
            *reinterpret_cast<uint32_t*>(dst) = codes;
        if (lane == 0) reinterpret_cast<float*>(rec + kBlockSize * D)[tok] = sc;
    } else {  // V: one byte in each of the block's D dim rows of 16 tokens, at the token's position
        uint8_t* vrec = rec + kBlockSize * D + kBlockSize * 4;
        uint8_t* dst = vrec + vt_pos(tok);
#pragma unroll
        for (int i = 0; i < PER; ++i) dst[(lane * PER + i) * kBlockSize] = static_cast<uint8_t>(codes >> (8 * i));
        if (lane == 0) reinterpret_cast<float*>(vrec + kBlockSize * D)[tok] = sc;
    }
}

cudaError_t launch_append_fp8(const __half* k_new, const __half* v_new, const int64_t* slots, int n,
                              uint8_t* kv_fp8, int num_blocks, int Hkv, int D, unsigned* err, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t warps = static_cast<int64_t>(n) * Hkv * 2;
    const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
    if (D == 64)
        kv_append_fp8_kernel<64><<<blocks, 256, 0, stream>>>(k_new, v_new, slots, n, kv_fp8, num_blocks, Hkv, err);
    else if (D == 128)
        kv_append_fp8_kernel<128><<<blocks, 256, 0, stream>>>(k_new, v_new, slots, n, kv_fp8, num_blocks, Hkv, err);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

constexpr int kMaxCopyPairs = 128;
struct CopyPairs {
    int32_t src[kMaxCopyPairs];
    int32_t dst[kMaxCopyPairs];
};

// grid (pair, layer, K|V); each CTA copies one block of one layer of one pool.
__global__ void __launch_bounds__(256) kv_copy_blocks_kernel(const CopyPairs pairs, uint4* __restrict__ k_pool,
                                                              uint4* __restrict__ v_pool, int64_t layer_u4,
                                                              int64_t block_u4) {
    uint4* pool = blockIdx.z ? v_pool : k_pool;
    const int64_t base = static_cast<int64_t>(blockIdx.y) * layer_u4;
    const uint4* s = pool + base + static_cast<int64_t>(pairs.src[blockIdx.x]) * block_u4;
    uint4* d = pool + base + static_cast<int64_t>(pairs.dst[blockIdx.x]) * block_u4;
    for (int64_t c = threadIdx.x; c < block_u4; c += blockDim.x) d[c] = s[c];
}

cudaError_t launch_copy_blocks(const int32_t* src, const int32_t* dst, int n, __half* k_pool, __half* v_pool,
                               int L, int num_blocks, int64_t block_elems, cudaStream_t stream) {
    const int64_t block_u4 = block_elems / 8;
    const int64_t layer_u4 = block_u4 * num_blocks;
    for (int i0 = 0; i0 < n; i0 += kMaxCopyPairs) {
        const int m = (n - i0 < kMaxCopyPairs) ? n - i0 : kMaxCopyPairs;
        CopyPairs p;
        for (int i = 0; i < m; ++i) {
            p.src[i] = src[i0 + i];
            p.dst[i] = dst[i0 + i];
        }
        dim3 grid(m, L, 2);
        kv_copy_blocks_kernel<<<grid, 256, 0, stream>>>(p, reinterpret_cast<uint4*>(k_pool),
                                                        reinterpret_cast<uint4*>(v_pool), layer_u4, block_u4);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Copy of n16 16-byte vectors between device-accessible buffers (device memory, or pinned host memory that
// the GPU reaches directly over the C2C link).  Four vectors in flight per thread: the loads of a host source
// cross the link, so many requests must be outstanding to cover its latency.
// ahead = 0: wait for the kernel before on the stream, copy, make the copy visible device-wide, then let the
//   next kernel launch; that kernel may read the bytes even before its own dependency wait.
// ahead = 1: let the next kernel launch and copy at once, then wait for the kernel before, so that this grid
//   completes only after that one has; the next kernel may read the bytes after its dependency wait.
// Without launch overlap both forms are plain stream-ordered copies (the waits return at once).
constexpr int kCopyThreads = 128;
constexpr int kCopyVec = 4;

__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(const uint4* __restrict__ src,
                                                                  uint4* __restrict__ dst, int64_t n16,
                                                                  int ahead) {
    if (ahead)
        grid_dependents_launch();
    else
        grid_dependency_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads * kCopyVec;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kCopyThreads * kCopyVec + threadIdx.x; base < n16;
         base += stride) {
        uint4 v[kCopyVec];
#pragma unroll
        for (int k = 0; k < kCopyVec; ++k) {
            const int64_t i = base + static_cast<int64_t>(k) * kCopyThreads;
            if (i < n16) v[k] = src[i];
        }
#pragma unroll
        for (int k = 0; k < kCopyVec; ++k) {
            const int64_t i = base + static_cast<int64_t>(k) * kCopyThreads;
            if (i < n16) dst[i] = v[k];
        }
    }
    if (ahead) {
        grid_dependency_wait();
    } else {
        __threadfence();
        __syncthreads();
        grid_dependents_launch();
    }
}

cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, bool ahead, cudaStream_t stream) {
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    const int64_t per_cta = static_cast<int64_t>(kCopyThreads) * kCopyVec;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t want = (n16 + per_cta - 1) / per_cta;
    const unsigned grid = static_cast<unsigned>(want < 2 * sms ? want : 2 * sms);
    return launch(stage_copy_kernel, dim3(grid), dim3(kCopyThreads), 0, stream, launch_overlap() != 0, 1u,
                  static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16, ahead ? 1 : 0);
}

}  // namespace kvc
