// C-ABI layer: argument validation, checked mode, the cache handle and the
// host-side block management; device work is forwarded to the launchers.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/kvc.h"
#include "block_pool.h"
#include "kvc_internal.h"
#include "stage_copy.h"

struct kvc_cache {
    kvc_config cfg;
    void* k_pool;
    void* v_pool;
    kvc::BlockPool pool;
    kvc_cache(const kvc_config& c, void* k, void* v) : cfg(c), k_pool(k), v_pool(v), pool(c.num_blocks) {}
};

namespace {

thread_local std::string g_last_error;
std::atomic<int> g_checked{0};

kvc_status fail(kvc_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kvc_status cuda_fail(cudaError_t e, const char* where) {
    return fail(KVC_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

kvc_status check_config(const kvc_config* c) {
    if (!c) return fail(KVC_ERR_INVALID, "null config");
    if (c->num_layers < 1 || c->num_blocks < 1 || c->num_kv_heads < 1 || c->head_dim < 1)
        return fail(KVC_ERR_INVALID, "config sizes must be positive");
    if (c->block_size != kvc::kBlockSize)
        return fail(KVC_ERR_UNSUPPORTED, "block_size %d not supported (16 only)", c->block_size);
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(KVC_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128)", c->head_dim);
    if (c->dtype != KVC_F16) return fail(KVC_ERR_UNSUPPORTED, "cache dtype must be KVC_F16");
    if (static_cast<int64_t>(c->num_blocks) * c->num_kv_heads * c->block_size >= (int64_t(1) << 31))
        return fail(KVC_ERR_UNSUPPORTED, "num_blocks * num_kv_heads * block_size must be < 2^31");
    return KVC_OK;
}

template <typename T>
kvc_status copy_to_host(std::vector<T>& dst, const T* src, size_t n, cudaStream_t s) {
    dst.resize(n);
    if (n == 0) return KVC_OK;
    cudaError_t e = cudaMemcpyAsync(dst.data(), src, n * sizeof(T), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "checked mode copy");
    return KVC_OK;
}

}  // namespace

int kvc::set_last_error(int status, const char* msg) {
    g_last_error = msg;
    return status;
}

extern "C" {

const char* kvc_last_error_string(void) { return g_last_error.c_str(); }

int kvc_version(void) { return 100; }

kvc_status kvc_set_checked_mode(int on) {
    g_checked.store(on ? 1 : 0);
    return KVC_OK;
}

kvc_status kvc_device_error_flags(uint32_t* flags, int clear) {
    if (!flags) return fail(KVC_ERR_INVALID, "null flags");
    unsigned* w = nullptr;
    cudaError_t e = kvc::device_error_word(&w);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    unsigned v = 0;
    e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (clear) {
        e = cudaMemset(w, 0, sizeof(unsigned));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    }
    *flags = v;
    return KVC_OK;
}

kvc_status kv_cache_pool_bytes(const kvc_config* cfg, size_t* bytes) {
    kvc_status s = check_config(cfg);
    if (s != KVC_OK) return s;
    if (!bytes) return fail(KVC_ERR_INVALID, "null output");
    *bytes = static_cast<size_t>(cfg->num_layers) * cfg->num_blocks * cfg->num_kv_heads * cfg->block_size *
             cfg->head_dim * 2;
    return KVC_OK;
}

kvc_status kv_cache_create(const kvc_config* cfg, void* k_pool, void* v_pool, kvc_handle* out) {
    kvc_status s = check_config(cfg);
    if (s != KVC_OK) return s;
    if (!out) return fail(KVC_ERR_INVALID, "null handle output");
    if ((k_pool == nullptr) != (v_pool == nullptr)) return fail(KVC_ERR_INVALID, "k_pool and v_pool: both or neither");
    if (k_pool && (!aligned16(k_pool) || !aligned16(v_pool))) return fail(KVC_ERR_INVALID, "pools must be 16-byte aligned");
    kvc_cache* h = new (std::nothrow) kvc_cache(*cfg, k_pool, v_pool);
    if (!h) return fail(KVC_ERR_OOM, "host allocation failed");
    *out = h;
    return KVC_OK;
}

kvc_status kv_cache_destroy(kvc_handle h) {
    delete h;
    return KVC_OK;
}

kvc_status kv_cache_layer(kvc_handle h, int layer, void** k_layer, void** v_layer) {
    if (!h || !k_layer || !v_layer) return fail(KVC_ERR_INVALID, "null argument");
    if (!h->k_pool) return fail(KVC_ERR_INVALID, "host-only cache has no device pools");
    if (layer < 0 || layer >= h->cfg.num_layers) return fail(KVC_ERR_INVALID, "layer %d out of range", layer);
    const size_t per = static_cast<size_t>(h->cfg.num_blocks) * h->cfg.num_kv_heads * h->cfg.block_size *
                       h->cfg.head_dim * 2;
    *k_layer = static_cast<char*>(h->k_pool) + per * layer;
    *v_layer = static_cast<char*>(h->v_pool) + per * layer;
    return KVC_OK;
}

kvc_status kv_block_alloc(kvc_handle h, int32_t* block) {
    if (!h || !block) return fail(KVC_ERR_INVALID, "null argument");
    auto lk = h->pool.lock();
    const int32_t b = h->pool.alloc();
    if (b < 0) return fail(KVC_ERR_OOM, "OOM -- no free blocks");
    *block = b;
    return KVC_OK;
}

kvc_status kv_block_share(kvc_handle h, int32_t block) {
    if (!h) return fail(KVC_ERR_INVALID, "null handle");
    auto lk = h->pool.lock();
    if (!h->pool.live(block)) return fail(KVC_ERR_INVALID, "block %d is not live", block);
    h->pool.share(block);
    return KVC_OK;
}

kvc_status kv_block_release(kvc_handle h, int32_t block) {
    if (!h) return fail(KVC_ERR_INVALID, "null handle");
    auto lk = h->pool.lock();
    if (!h->pool.live(block)) return fail(KVC_ERR_INVALID, "block %d is not live", block);
    h->pool.release(block);
    return KVC_OK;
}

kvc_status kv_block_refcount(kvc_handle h, int32_t block, int32_t* refcount) {
    if (!h || !refcount) return fail(KVC_ERR_INVALID, "null argument");
    if (block < 0 || block >= h->cfg.num_blocks) return fail(KVC_ERR_INVALID, "block %d out of range", block);
    auto lk = h->pool.lock();
    *refcount = h->pool.refcount(block);
    return KVC_OK;
}

kvc_status kv_block_num_free(kvc_handle h, int32_t* num_free) {
    if (!h || !num_free) return fail(KVC_ERR_INVALID, "null argument");
    auto lk = h->pool.lock();
    *num_free = h->pool.num_free();
    return KVC_OK;
}

kvc_status kv_cache_utilisation(kvc_handle h, double* percent) {
    if (!h || !percent) return fail(KVC_ERR_INVALID, "null argument");
    auto lk = h->pool.lock();
    *percent = static_cast<double>(h->pool.total() - h->pool.num_free()) / h->pool.total() * 100.0;
    return KVC_OK;
}

static kvc_status copy_blocks_device(kvc_handle h, const int32_t* src, const int32_t* dst, int n, void* stream) {
    const int64_t block_elems = static_cast<int64_t>(h->cfg.num_kv_heads) * h->cfg.block_size * h->cfg.head_dim;
    cudaError_t e = kvc::launch_copy_blocks(src, dst, n, static_cast<__half*>(h->k_pool), static_cast<__half*>(h->v_pool),
                                            h->cfg.num_layers, h->cfg.num_blocks, block_elems, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
    return KVC_OK;
}

kvc_status kv_copy_blocks(kvc_handle h, const int32_t* src, const int32_t* dst, int n, void* stream) {
    if (!h) return fail(KVC_ERR_INVALID, "null handle");
    if (n < 0 || (n > 0 && (!src || !dst))) return fail(KVC_ERR_INVALID, "bad copy list");
    if (n == 0) return KVC_OK;
    if (!h->k_pool) return fail(KVC_ERR_INVALID, "host-only cache has no device pools");
    for (int i = 0; i < n; ++i)
        if (src[i] < 0 || src[i] >= h->cfg.num_blocks || dst[i] < 0 || dst[i] >= h->cfg.num_blocks)
            return fail(KVC_ERR_INVALID, "copy pair %d (%d -> %d) out of range", i, src[i], dst[i]);
    return copy_blocks_device(h, src, dst, n, stream);
}

kvc_status kv_block_cow(kvc_handle h, int32_t block, int32_t* new_block, void* stream) {
    if (!h || !new_block) return fail(KVC_ERR_INVALID, "null argument");
    int32_t nb;
    {
        auto lk = h->pool.lock();
        if (!h->pool.live(block)) return fail(KVC_ERR_INVALID, "block %d is not live", block);
        if (h->pool.refcount(block) <= 1) {
            *new_block = block;
            return KVC_OK;
        }
        if (!h->k_pool) return fail(KVC_ERR_INVALID, "host-only cache has no device pools");
        nb = h->pool.alloc();
        if (nb < 0) return fail(KVC_ERR_OOM, "OOM -- no free blocks for copy-on-write");
        h->pool.release(block);
    }
    kvc_status s = copy_blocks_device(h, &block, &nb, 1, stream);
    if (s != KVC_OK) return s;
    *new_block = nb;
    return KVC_OK;
}

kvc_status kv_slot_mapping(const int32_t* block_table, int max_blocks, int B, const int32_t* first_pos,
                           const int32_t* count, int block_size, int64_t* slots) {
    if (B < 0 || max_blocks < 1 || block_size < 1) return fail(KVC_ERR_INVALID, "bad sizes");
    if (B > 0 && (!block_table || !first_pos || !count || !slots)) return fail(KVC_ERR_INVALID, "null argument");
    int64_t o = 0;
    for (int b = 0; b < B; ++b) {
        if (first_pos[b] < 0 || count[b] < 0) return fail(KVC_ERR_INVALID, "sequence %d: negative position/count", b);
        for (int32_t k = 0; k < count[b]; ++k) {
            const int64_t pos = static_cast<int64_t>(first_pos[b]) + k;
            const int64_t j = pos / block_size;
            if (j >= max_blocks) return fail(KVC_ERR_CAPACITY, "sequence %d: position %lld beyond its block table", b, (long long)pos);
            const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + j];
            if (blk < 0) return fail(KVC_ERR_CAPACITY, "sequence %d: no block for position %lld", b, (long long)pos);
            slots[o++] = static_cast<int64_t>(blk) * block_size + pos % block_size;
        }
    }
    return KVC_OK;
}

kvc_status kv_step_prepare(kvc_handle h, int32_t* block_table, int max_blocks, int32_t* num_blocks,
                           const int32_t* positions, int B, int64_t* slot_mapping, int32_t* copy_src,
                           int32_t* copy_dst, int* n_copies) {
    if (!h || B < 0 || max_blocks < 1) return fail(KVC_ERR_INVALID, "bad arguments");
    if (!n_copies || (B > 0 && (!block_table || !num_blocks || !positions || !slot_mapping || !copy_src || !copy_dst)))
        return fail(KVC_ERR_INVALID, "null argument");
    const int bs = h->cfg.block_size;
    auto lk = h->pool.lock();
    // dry run: validate and count the blocks this step needs
    std::unordered_map<int32_t, int32_t> taken;  // references dropped by earlier copies in this step
    int32_t need = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t pos = positions[b], nb = num_blocks[b];
        if (pos < 0 || nb < 0 || nb > max_blocks) return fail(KVC_ERR_INVALID, "sequence %d: bad position/num_blocks", b);
        const int32_t j = pos / bs;
        if (j == nb) {
            if (nb == max_blocks) return fail(KVC_ERR_CAPACITY, "sequence %d: block table full", b);
            ++need;
        } else if (j < nb) {
            const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + j];
            if (!h->pool.live(blk)) return fail(KVC_ERR_INVALID, "sequence %d: block %d is not live", b, blk);
            const int32_t rc = h->pool.refcount(blk) - taken[blk];
            if (rc > 1) {
                ++need;
                ++taken[blk];
            }
        } else {
            return fail(KVC_ERR_CAPACITY, "sequence %d: position %d skips past its last block", b, pos);
        }
    }
    if (need > h->pool.num_free()) return fail(KVC_ERR_OOM, "OOM -- step needs %d blocks, %d free", need, h->pool.num_free());
    int nc = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t pos = positions[b];
        const int32_t j = pos / bs;
        int32_t* row = block_table + static_cast<int64_t>(b) * max_blocks;
        if (j == num_blocks[b]) {
            row[j] = h->pool.alloc();
            ++num_blocks[b];
        } else {
            const int32_t blk = row[j];
            if (h->pool.refcount(blk) > 1) {
                const int32_t nb = h->pool.alloc();
                h->pool.release(blk);
                copy_src[nc] = blk;
                copy_dst[nc] = nb;
                ++nc;
                row[j] = nb;
            }
        }
        slot_mapping[b] = static_cast<int64_t>(row[j]) * bs + pos % bs;
    }
    *n_copies = nc;
    return KVC_OK;
}

kvc_status kv_append(kvc_handle h, int layer, const void* k_new, const void* v_new, const int64_t* slot_mapping, int n,
                     void* stream) {
    if (!h) return fail(KVC_ERR_INVALID, "null handle");
    if (!h->k_pool) return fail(KVC_ERR_INVALID, "host-only cache has no device pools");
    if (layer < 0 || layer >= h->cfg.num_layers) return fail(KVC_ERR_INVALID, "layer %d out of range", layer);
    if (n < 0) return fail(KVC_ERR_INVALID, "negative n");
    if (n == 0) return KVC_OK;
    if (!k_new || !v_new || !slot_mapping) return fail(KVC_ERR_INVALID, "null pointer");
    if (!aligned16(k_new) || !aligned16(v_new)) return fail(KVC_ERR_INVALID, "k_new/v_new must be 16-byte aligned");
    if (g_checked.load()) {
        std::vector<int64_t> s;
        kvc_status st = copy_to_host(s, slot_mapping, static_cast<size_t>(n), as_stream(stream));
        if (st != KVC_OK) return st;
        const int64_t cap = static_cast<int64_t>(h->cfg.num_blocks) * h->cfg.block_size;
        for (int t = 0; t < n; ++t)
            if (s[t] >= cap) return fail(KVC_ERR_CAPACITY, "slot %lld of token %d beyond the pool (%lld slots)", (long long)s[t], t, (long long)cap);
    }
    void *kl, *vl;
    kv_cache_layer(h, layer, &kl, &vl);
    unsigned* err = nullptr;
    cudaError_t e = kvc::device_error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_append(static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), slot_mapping, n,
                           static_cast<__half*>(kl), static_cast<__half*>(vl), h->cfg.num_blocks, h->cfg.num_kv_heads,
                           h->cfg.head_dim, err, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return KVC_OK;
}

static kvc_status check_decode_shape(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len) {
    if (B < 0 || Hq < 1 || Hkv < 1 || max_context_len < 1) return fail(KVC_ERR_INVALID, "bad sizes");
    if (Hq % Hkv) return fail(KVC_ERR_INVALID, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (Hq / Hkv > kvc::kMaxGroupHeads)
        return fail(KVC_ERR_UNSUPPORTED, "group size %d > %d not supported", Hq / Hkv, kvc::kMaxGroupHeads);
    if (head_dim != 64 && head_dim != 128) return fail(KVC_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
    if (block_size != kvc::kBlockSize) return fail(KVC_ERR_UNSUPPORTED, "block_size %d not supported", block_size);
    if (B > 65535 || Hkv > 65535) return fail(KVC_ERR_UNSUPPORTED, "B and Hkv must be <= 65535");
    return KVC_OK;
}

kvc_status paged_decode_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                             int blocks_per_split, int* num_splits, int* blocks_per_split_out, size_t* workspace_bytes) {
    kvc_status s = check_decode_shape(B, Hq, Hkv, head_dim, block_size, max_context_len);
    if (s != KVC_OK) return s;
    kvc::DecodePlan plan;
    cudaError_t e = kvc::decode_plan(B, Hq, Hkv, head_dim, max_context_len, blocks_per_split, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "decode plan");
    if (num_splits) *num_splits = plan.num_splits;
    if (blocks_per_split_out) *blocks_per_split_out = plan.blocks_per_split;
    if (workspace_bytes) *workspace_bytes = plan.workspace_bytes;
    return KVC_OK;
}

kvc_status paged_decode_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (bytes == 0) return KVC_OK;
    if (!workspace) return fail(KVC_ERR_INVALID, "null workspace");
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "workspace init");
    return KVC_OK;
}

kvc_status kvc_trace_read(void* records, int capacity, int* count, int clear) {
    if (!count || capacity < 0 || (capacity > 0 && !records)) return fail(KVC_ERR_INVALID, "bad arguments");
    cudaError_t e = kvc::trace_read(records, capacity, count, clear);
    if (e == cudaErrorNotSupported) return fail(KVC_ERR_UNSUPPORTED, "library built without -DKVC_TRACE=1");
    if (e != cudaSuccess) return cuda_fail(e, "trace read");
    return KVC_OK;
}

kvc_status kvc_set_launch_overlap(int on) {
    kvc::set_launch_overlap(on);
    return KVC_OK;
}

kvc_status kvc_set_multi_tc(int on) {
    kvc::set_multi_tc(on);
    return KVC_OK;
}

kvc_status kvc_set_cascade_min_saved_blocks(int blocks) {
    if (blocks < 0) return fail(KVC_ERR_INVALID, "negative block count %d", blocks);
    kvc::set_cascade_min_saved_blocks(blocks);
    return KVC_OK;
}

// The address the current device uses for p: device and managed memory as they are, pinned host memory
// through its mapping.  False for pageable host memory and unknown pointers.
static bool device_address(const void* p, void** out) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged && a.type != cudaMemoryTypeHost)
        return false;
    if (!a.devicePointer) return false;
    *out = a.devicePointer;
    return true;
}

kvc_status kvc_copy_async(void* dst, const void* src, size_t bytes, unsigned flags, void* stream) {
    if (flags & ~KVC_COPY_AHEAD) return fail(KVC_ERR_INVALID, "unknown flags 0x%x", flags);
    if (bytes == 0) return KVC_OK;
    if (!dst || !src) return fail(KVC_ERR_INVALID, "null buffer");
    if ((bytes & 15u) || !aligned16(dst) || !aligned16(src))
        return fail(KVC_ERR_INVALID, "both buffers 16-byte aligned and bytes a multiple of 16 (got %zu)", bytes);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
    if (d0 < s0 + bytes && s0 < d0 + bytes) return fail(KVC_ERR_INVALID, "source and destination overlap");
    void *ddev = nullptr, *sdev = nullptr;
    if (!device_address(dst, &ddev)) return fail(KVC_ERR_INVALID, "dst is neither device nor pinned host memory");
    if (!device_address(src, &sdev)) return fail(KVC_ERR_INVALID, "src is neither device nor pinned host memory");
    cudaError_t e = kvc::launch_stage_copy(ddev, sdev, bytes, (flags & KVC_COPY_AHEAD) != 0,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "staging copy launch");
    return KVC_OK;
}

static kvc_status decode_common(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                const void* v_cache, int num_blocks,
                                const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B, int Hq,
                                int Hkv, int head_dim, int block_size, int max_context_len, float scale, void* out,
                                int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split,
                                void* stream);

kvc_status paged_decode_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                  const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B, int Hq,
                                  int Hkv, int head_dim, int block_size, int max_context_len, float scale, void* out,
                                  int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split,
                                  void* stream) {
    return decode_common(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_table, max_blocks,
                         context_lens, B, Hq, Hkv, head_dim, block_size, max_context_len, scale, out, out_dtype,
                         workspace, workspace_bytes, blocks_per_split, stream);
}

kvc_status paged_decode_append_attention(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                         void* v_cache, int num_blocks,
                                         const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                         int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                         float scale, void* out, int out_dtype, void* workspace,
                                         size_t workspace_bytes, int blocks_per_split, void* stream) {
    if (B > 0 && (!k_new || !v_new)) return fail(KVC_ERR_INVALID, "null k_new/v_new");
    if (!aligned16(k_new) || !aligned16(v_new)) return fail(KVC_ERR_INVALID, "k_new/v_new must be 16-byte aligned");
    return decode_common(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks,
                         context_lens, B, Hq, Hkv, head_dim, block_size, max_context_len, scale, out, out_dtype,
                         workspace, workspace_bytes, blocks_per_split, stream);
}

// Every argument check of a decode call; in checked mode also the context lengths and the block-table
// entries, on host copies that are returned through ctx / table (left empty otherwise).
static kvc_status decode_validate(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                  const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B,
                                  int Hq, int Hkv, int head_dim, int block_size, int max_context_len, void* out,
                                  int out_dtype, int blocks_per_split, void* stream, std::vector<int32_t>& ctx,
                                  std::vector<int32_t>& table) {
    kvc_status s = check_decode_shape(B, Hq, Hkv, head_dim, block_size, max_context_len);
    if (s != KVC_OK) return s;
    if (B == 0) return KVC_OK;
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out) return fail(KVC_ERR_INVALID, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(KVC_ERR_INVALID, "q, caches and out must be 16-byte aligned");
    if (num_blocks < 1 || max_blocks < 1) return fail(KVC_ERR_INVALID, "num_blocks and max_blocks must be positive");
    if (static_cast<int64_t>(num_blocks) * Hkv * block_size >= (int64_t(1) << 31))
        return fail(KVC_ERR_UNSUPPORTED, "num_blocks * Hkv * block_size must be < 2^31");
    if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks) * block_size)
        return fail(KVC_ERR_CAPACITY, "max_context_len %d beyond max_blocks * block_size", max_context_len);
    if (out_dtype != KVC_F16 && out_dtype != KVC_F32) return fail(KVC_ERR_INVALID, "bad out_dtype");
    if (blocks_per_split < 0) return fail(KVC_ERR_INVALID, "negative blocks_per_split");
    if (g_checked.load()) {
        kvc_status st = copy_to_host(ctx, context_lens, static_cast<size_t>(B), as_stream(stream));
        if (st == KVC_OK) st = copy_to_host(table, block_table, static_cast<size_t>(B) * max_blocks, as_stream(stream));
        if (st != KVC_OK) return st;
        for (int b = 0; b < B; ++b) {
            if (ctx[b] < 1 || ctx[b] > max_context_len)
                return fail(KVC_ERR_CAPACITY, "sequence %d: context length %d outside [1, %d]", b, ctx[b], max_context_len);
            for (int j = 0; j < (ctx[b] + block_size - 1) / block_size; ++j) {
                const int32_t blk = table[static_cast<size_t>(b) * max_blocks + j];
                if (blk < 0 || blk >= num_blocks)
                    return fail(KVC_ERR_INVALID, "sequence %d: block-table entry %d = %d outside [0, %d)", b, j, blk, num_blocks);
            }
        }
    }
    return KVC_OK;
}

static kvc::DecodeArgs decode_args(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                   const void* v_cache, int num_blocks,
                                   const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B,
                                   int Hq, int Hkv, int head_dim, int max_context_len, float scale, void* out,
                                   int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split) {
    kvc::DecodeArgs a;
    a.q = static_cast<const __half*>(q);
    a.k_new = static_cast<const __half*>(k_new);
    a.v_new = static_cast<const __half*>(v_new);
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
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.blocks_per_split = blocks_per_split;
    a.err = nullptr;
    return a;
}

static kvc_status check_workspace(size_t need, const void* workspace, size_t workspace_bytes) {
    if (need > workspace_bytes || (need && !workspace))
        return fail(KVC_ERR_INVALID, "workspace too small: need %zu bytes", need);
    if (need && !aligned16(workspace)) return fail(KVC_ERR_INVALID, "workspace must be 16-byte aligned");
    return KVC_OK;
}

static kvc_status decode_common(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                const void* v_cache, int num_blocks,
                                const int32_t* block_table, int max_blocks, const int32_t* context_lens, int B, int Hq,
                                int Hkv, int head_dim, int block_size, int max_context_len, float scale, void* out,
                                int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split,
                                void* stream) {
    std::vector<int32_t> ctx, table;
    kvc_status s = decode_validate(q, k_cache, v_cache, num_blocks, block_table, max_blocks, context_lens, B, Hq, Hkv,
                                   head_dim, block_size, max_context_len, out, out_dtype, blocks_per_split, stream, ctx,
                                   table);
    if (s != KVC_OK || B == 0) return s;
    kvc::DecodeArgs a = decode_args(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table,
                                    max_blocks, context_lens, B, Hq, Hkv, head_dim, max_context_len, scale, out,
                                    out_dtype, workspace, workspace_bytes, blocks_per_split);
    kvc::DecodePlan plan;
    cudaError_t e = kvc::decode_plan(B, Hq, Hkv, head_dim, max_context_len, blocks_per_split, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "decode plan");
    s = check_workspace(plan.workspace_bytes, workspace, workspace_bytes);
    if (s != KVC_OK) return s;
    e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_decode(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, k_new ? "paged_decode_append_attention launch" : "paged_decode_attention launch");
    return KVC_OK;
}

kvc_status kv_cascade_groups(const int32_t* block_table, int B, int max_blocks, const int32_t* context_lens,
                             int block_size, int max_group, int32_t* group_start, int* n_groups,
                             int32_t* shared_blocks, int* max_shared) {
    if (B < 0 || max_blocks < 1 || block_size < 1) return fail(KVC_ERR_INVALID, "bad sizes");
    if (max_group < 1 || max_group > kvc::kMaxGroupSize)
        return fail(KVC_ERR_INVALID, "max_group %d outside [1, %d]", max_group, kvc::kMaxGroupSize);
    if (B > 0 && (!block_table || !context_lens || !group_start || !n_groups || !shared_blocks || !max_shared))
        return fail(KVC_ERR_INVALID, "null pointer");
    int ng = 0, mx = 0;
    group_start[0] = 0;
    for (int g0 = 0; g0 < B;) {
        const int32_t* r0 = block_table + static_cast<size_t>(g0) * max_blocks;
        int g1 = g0 + 1;  // members: consecutive rows that start with the same block, at most max_group
        while (g1 < B && g1 - g0 < max_group && block_table[static_cast<size_t>(g1) * max_blocks] == r0[0]) ++g1;
        int shared = 0;
        if (g1 - g0 > 1) {
            int cap = max_blocks;
            for (int b = g0; b < g1; ++b) {
                if (context_lens[b] < 1) return fail(KVC_ERR_INVALID, "sequence %d: context length %d", b, context_lens[b]);
                cap = std::min(cap, (context_lens[b] - 1) / block_size);
            }
            while (shared < cap) {
                bool same = true;
                for (int b = g0 + 1; b < g1 && same; ++b)
                    same = block_table[static_cast<size_t>(b) * max_blocks + shared] == r0[shared];
                if (!same) break;
                ++shared;
            }
        }
        for (int b = g0; b < g1; ++b) shared_blocks[b] = shared;
        mx = std::max(mx, shared);
        group_start[++ng] = g1;
        g0 = g1;
    }
    *n_groups = ng;
    *max_shared = mx;
    return KVC_OK;
}

kvc_status paged_decode_cascade_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                     int n_groups, int max_shared_blocks, size_t* workspace_bytes) {
    kvc_status s = check_decode_shape(B, Hq, Hkv, head_dim, block_size, max_context_len);
    if (s != KVC_OK) return s;
    if (n_groups < 0 || max_shared_blocks < 0) return fail(KVC_ERR_INVALID, "bad group sizes");
    kvc::CascadePlan plan;
    cudaError_t e = kvc::cascade_plan(B, Hq, Hkv, head_dim, max_context_len, std::max(n_groups, 1),
                                      max_shared_blocks, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "cascade plan");
    if (workspace_bytes) *workspace_bytes = plan.workspace_bytes;
    return KVC_OK;
}

kvc_status paged_decode_cascade_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                          const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                          const int32_t* group_start, const int32_t* shared_blocks, int n_groups,
                                          int max_shared_blocks, int B, int Hq, int Hkv, int head_dim,
                                          int block_size, int max_context_len, float scale, void* out, int out_dtype,
                                          void* workspace, size_t workspace_bytes, void* stream) {
    std::vector<int32_t> ctx, table;
    kvc_status s = decode_validate(q, k_cache, v_cache, num_blocks, block_table, max_blocks, context_lens, B, Hq, Hkv,
                                   head_dim, block_size, max_context_len, out, out_dtype, 0, stream, ctx, table);
    if (s != KVC_OK || B == 0) return s;
    if (!group_start || !shared_blocks) return fail(KVC_ERR_INVALID, "null group_start / shared_blocks");
    if (n_groups < 1 || n_groups > B) return fail(KVC_ERR_INVALID, "n_groups %d outside [1, B = %d]", n_groups, B);
    if (max_shared_blocks < 0 || max_shared_blocks >= max_blocks)
        return fail(KVC_ERR_INVALID, "max_shared_blocks %d outside [0, max_blocks)", max_shared_blocks);
    if (g_checked.load()) {
        std::vector<int32_t> gs, sh;
        s = copy_to_host(gs, group_start, static_cast<size_t>(n_groups) + 1, as_stream(stream));
        if (s == KVC_OK) s = copy_to_host(sh, shared_blocks, static_cast<size_t>(B), as_stream(stream));
        if (s != KVC_OK) return s;
        if (gs[0] != 0 || gs[n_groups] != B) return fail(KVC_ERR_INVALID, "group_start must run from 0 to B");
        for (int g = 0; g < n_groups; ++g) {
            const int g0 = gs[g], g1 = gs[g + 1];
            if (g1 <= g0 || g1 - g0 > kvc::kMaxGroupSize)
                return fail(KVC_ERR_INVALID, "group %d: %d members (1..%d)", g, g1 - g0, kvc::kMaxGroupSize);
            for (int b = g0; b < g1; ++b) {
                if (sh[b] != sh[g0]) return fail(KVC_ERR_INVALID, "group %d: members share different block counts", g);
                if (sh[b] < 0 || sh[b] > max_shared_blocks || static_cast<int64_t>(sh[b]) * block_size >= ctx[b])
                    return fail(KVC_ERR_INVALID, "sequence %d: %d shared blocks do not fit its context %d (or the bound %d)",
                                b, sh[b], ctx[b], max_shared_blocks);
                for (int j = 0; j < sh[b]; ++j)
                    if (table[static_cast<size_t>(b) * max_blocks + j] != table[static_cast<size_t>(g0) * max_blocks + j])
                        return fail(KVC_ERR_INVALID, "sequence %d: block %d is not the group's shared block", b, j);
            }
        }
    }
    kvc::DecodeArgs a = decode_args(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_table,
                                    max_blocks, context_lens, B, Hq, Hkv, head_dim, max_context_len, scale, out,
                                    out_dtype, workspace, workspace_bytes, 0);
    kvc::CascadePlan plan;
    cudaError_t e = kvc::cascade_plan(B, Hq, Hkv, head_dim, max_context_len, n_groups, max_shared_blocks, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "cascade plan");
    s = check_workspace(plan.workspace_bytes, workspace, workspace_bytes);
    if (s != KVC_OK) return s;
    e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_cascade(a, group_start, shared_blocks, n_groups, max_shared_blocks, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_cascade_attention launch");
    return KVC_OK;
}

kvc_status kv_fp8_record_bytes(int head_dim, size_t* bytes) {
    if (head_dim != 64 && head_dim != 128) return fail(KVC_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
    if (!bytes) return fail(KVC_ERR_INVALID, "null pointer");
    *bytes = static_cast<size_t>(kvc::fp8_record_bytes(head_dim));
    return KVC_OK;
}

kvc_status kv_append_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping, int n, void* kv_fp8,
                         int num_blocks, int Hkv, int head_dim, int block_size, void* stream) {
    if (n < 0 || num_blocks < 1 || Hkv < 1) return fail(KVC_ERR_INVALID, "bad sizes");
    if (head_dim != 64 && head_dim != 128) return fail(KVC_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
    if (block_size != kvc::kBlockSize) return fail(KVC_ERR_UNSUPPORTED, "block_size %d not supported", block_size);
    if (n == 0) return KVC_OK;
    if (!k_new || !v_new || !slot_mapping || !kv_fp8) return fail(KVC_ERR_INVALID, "null pointer");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_fp8))
        return fail(KVC_ERR_INVALID, "device buffers must be 16-byte aligned");
    if (g_checked.load()) {
        std::vector<int64_t> sl;
        kvc_status st = copy_to_host(sl, slot_mapping, static_cast<size_t>(n), as_stream(stream));
        if (st != KVC_OK) return st;
        for (int t = 0; t < n; ++t)
            if (sl[t] >= static_cast<int64_t>(num_blocks) * block_size)
                return fail(KVC_ERR_CAPACITY, "token %d: slot %lld beyond the pool", t, static_cast<long long>(sl[t]));
    }
    unsigned* err = nullptr;
    cudaError_t e = kvc::device_error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_append_fp8(static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), slot_mapping, n,
                               static_cast<uint8_t*>(kv_fp8), num_blocks, Hkv, head_dim, err, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append_fp8 launch");
    return KVC_OK;
}

kvc_status paged_decode_attention_fp8(const void* q, const void* kv_fp8, int num_blocks, const int32_t* block_table,
                                      int max_blocks, const int32_t* context_lens, int B, int Hq, int Hkv,
                                      int head_dim, int block_size, int max_context_len, float scale, void* out,
                                      int out_dtype, void* workspace, size_t workspace_bytes, int blocks_per_split,
                                      void* stream) {
    std::vector<int32_t> ctx, table;
    kvc_status s = decode_validate(q, kv_fp8, kv_fp8, num_blocks, block_table, max_blocks, context_lens, B, Hq, Hkv,
                                   head_dim, block_size, max_context_len, out, out_dtype, blocks_per_split, stream, ctx,
                                   table);
    if (s != KVC_OK || B == 0) return s;
    kvc::DecodeArgs a = decode_args(q, nullptr, nullptr, nullptr, nullptr, num_blocks, block_table,
                                    max_blocks, context_lens, B, Hq, Hkv, head_dim, max_context_len, scale, out,
                                    out_dtype, workspace, workspace_bytes, blocks_per_split);
    a.kv_fp8 = static_cast<const uint8_t*>(kv_fp8);
    kvc::DecodePlan plan;
    cudaError_t e = kvc::decode_plan(B, Hq, Hkv, head_dim, max_context_len, blocks_per_split, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "decode plan");
    s = check_workspace(plan.workspace_bytes, workspace, workspace_bytes);
    if (s != KVC_OK) return s;
    e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_decode(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_attention_fp8 launch");
    return KVC_OK;
}

kvc_status paged_decode_multi_plan(int B, int Hq, int Hkv, int head_dim, int block_size, int max_context_len,
                                   int q_len, size_t* workspace_bytes) {
    kvc_status s = check_decode_shape(B, Hq, Hkv, head_dim, block_size, max_context_len);
    if (s != KVC_OK) return s;
    if (q_len < 1 || q_len > kvc::kMaxQueryTokens)
        return fail(KVC_ERR_UNSUPPORTED, "q_len %d outside [1, %d]", q_len, kvc::kMaxQueryTokens);
    kvc::MultiPlan plan;
    cudaError_t e = kvc::multi_plan(B, Hq, Hkv, head_dim, max_context_len, q_len, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "multi-token plan");
    if (workspace_bytes) *workspace_bytes = plan.workspace_bytes;
    return KVC_OK;
}

kvc_status paged_decode_multi_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                        const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                        int q_len, int B, int Hq, int Hkv, int head_dim, int block_size,
                                        int max_context_len, float scale, void* out, int out_dtype, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (q_len < 1 || q_len > kvc::kMaxQueryTokens)
        return fail(KVC_ERR_UNSUPPORTED, "q_len %d outside [1, %d]", q_len, kvc::kMaxQueryTokens);
    std::vector<int32_t> ctx, table;
    kvc_status s = decode_validate(q, k_cache, v_cache, num_blocks, block_table, max_blocks, context_lens, B, Hq, Hkv,
                                   head_dim, block_size, max_context_len, out, out_dtype, 0, stream, ctx, table);
    if (s != KVC_OK || B == 0) return s;
    if (g_checked.load())
        for (int b = 0; b < B; ++b)
            if (ctx[b] < q_len)
                return fail(KVC_ERR_CAPACITY, "sequence %d: context length %d below q_len %d", b, ctx[b], q_len);
    kvc::DecodeArgs a = decode_args(q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_table,
                                    max_blocks, context_lens, B, Hq, Hkv, head_dim, max_context_len, scale, out,
                                    out_dtype, workspace, workspace_bytes, 0);
    kvc::MultiPlan plan;
    cudaError_t e = kvc::multi_plan(B, Hq, Hkv, head_dim, max_context_len, q_len, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "multi-token plan");
    s = check_workspace(plan.workspace_bytes, workspace, workspace_bytes);
    if (s != KVC_OK) return s;
    e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_multi(a, q_len, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_multi_attention launch");
    return KVC_OK;
}

kvc_status prefill_attention_ex(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int nseq,
                                int total_tokens, int max_seqlen, int Hq, int Hkv, int head_dim, float scale,
                                int causal, int p_precision, void* out, int out_dtype, void* stream) {
    if (p_precision != KVC_PREFILL_P_F16 && p_precision != KVC_PREFILL_P_SPLIT)
        return fail(KVC_ERR_INVALID, "bad p_precision %d", p_precision);
    if (nseq < 0 || total_tokens < 0 || max_seqlen < 0 || Hq < 1 || Hkv < 1) return fail(KVC_ERR_INVALID, "bad sizes");
    if (Hq % Hkv) return fail(KVC_ERR_INVALID, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (head_dim != 64 && head_dim != 128) return fail(KVC_ERR_UNSUPPORTED, "head_dim %d not supported", head_dim);
    if (out_dtype != KVC_F16 && out_dtype != KVC_F32) return fail(KVC_ERR_INVALID, "bad out_dtype");
    if (nseq == 0 || total_tokens == 0) return KVC_OK;
    if (!q || !k || !v || !cu_seqlens || !out) return fail(KVC_ERR_INVALID, "null pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(KVC_ERR_INVALID, "q, k, v and out must be 16-byte aligned");
    if (static_cast<int64_t>(nseq) * ((max_seqlen + 127) / 128) * Hq > 2147483647LL)
        return fail(KVC_ERR_UNSUPPORTED, "grid too large");
    if (g_checked.load()) {
        std::vector<int32_t> cu;
        kvc_status st = copy_to_host(cu, cu_seqlens, static_cast<size_t>(nseq) + 1, as_stream(stream));
        if (st != KVC_OK) return st;
        if (cu[0] != 0 || cu[nseq] != total_tokens) return fail(KVC_ERR_INVALID, "cu_seqlens must run from 0 to total_tokens");
        for (int s = 0; s < nseq; ++s)
            if (cu[s + 1] < cu[s] || cu[s + 1] - cu[s] > max_seqlen)
                return fail(KVC_ERR_INVALID, "segment %d: length %d outside [0, max_seqlen]", s, cu[s + 1] - cu[s]);
    }
    kvc::PrefillArgs a;
    a.q = static_cast<const __half*>(q);
    a.k = static_cast<const __half*>(k);
    a.v = static_cast<const __half*>(v);
    a.cu_seqlens = cu_seqlens;
    a.nseq = nseq;
    a.total_tokens = total_tokens;
    a.max_seqlen = max_seqlen;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = head_dim;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.out = out;
    a.out_f32 = out_dtype == KVC_F32;
    a.split_p = p_precision == KVC_PREFILL_P_SPLIT;
    cudaError_t e = kvc::device_error_word(&a.err);
    if (e != cudaSuccess) return cuda_fail(e, "device error word");
    e = kvc::launch_prefill(a, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill_attention launch");
    return KVC_OK;
}

kvc_status prefill_attention(const void* q, const void* k, const void* v, const int32_t* cu_seqlens, int nseq,
                             int total_tokens, int max_seqlen, int Hq, int Hkv, int head_dim, float scale, int causal,
                             void* out, int out_dtype, void* stream) {
    return prefill_attention_ex(q, k, v, cu_seqlens, nseq, total_tokens, max_seqlen, Hq, Hkv, head_dim, scale, causal,
                                KVC_PREFILL_P_F16, out, out_dtype, stream);
}

}  // extern "C"
