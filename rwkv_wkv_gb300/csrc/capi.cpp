// C-ABI of libwkv7: the pool, the host-side slot table, argument checks and
// dispatch to the kernels.  The public contract is documented in wkv7.h.
#include "wkv7.h"

#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "wkv7_internal.h"

namespace {

constexpr size_t kHeaderBytes = 256;  // device status word lives here

std::atomic<uint64_t> g_launches{0};
thread_local char g_last_error[512] = "";
std::atomic<int> g_test_wait_timeout{0};  // wkv7_test_force_wait_timeout

void set_error(const char *what, cudaError_t e) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what,
                  cudaGetErrorString(e), static_cast<int>(e));
}

wkv7_status cuda_status(const char *what, cudaError_t e, int launches) {
    g_launches.fetch_add(static_cast<uint64_t>(launches), std::memory_order_relaxed);
    if (e != cudaSuccess) {
        set_error(what, e);
        return WKV7_ERR_CUDA;
    }
    return WKV7_OK;
}

// Host-side id table: a LIFO free list plus an "in use" flag per id.
struct IdTable {
    std::vector<int32_t> free_list;
    std::vector<uint8_t> used;

    void init(int32_t n) {
        used.assign(static_cast<size_t>(n), 0);
        free_list.resize(static_cast<size_t>(n));
        for (int32_t i = 0; i < n; ++i) free_list[static_cast<size_t>(i)] = n - 1 - i;
    }
    int32_t size() const { return static_cast<int32_t>(used.size()); }
    int32_t n_free() const { return static_cast<int32_t>(free_list.size()); }

    wkv7_status alloc(int32_t n, int32_t *out) {
        if (n < 0 || (n > 0 && !out)) return WKV7_ERR_INVALID_ARG;
        if (n > n_free()) return WKV7_ERR_POOL_FULL;
        for (int32_t i = 0; i < n; ++i) {
            int32_t id = free_list.back();
            free_list.pop_back();
            used[static_cast<size_t>(id)] = 1;
            out[i] = id;
        }
        return WKV7_OK;
    }

    wkv7_status release(int32_t n, const int32_t *ids) {
        if (n < 0 || (n > 0 && !ids)) return WKV7_ERR_INVALID_ARG;
        std::vector<uint8_t> seen(used.size(), 0);
        for (int32_t i = 0; i < n; ++i) {  // validate everything first
            int32_t id = ids[i];
            if (id < 0 || id >= size() || !used[static_cast<size_t>(id)]) return WKV7_ERR_BAD_SLOT;
            if (seen[static_cast<size_t>(id)]) return WKV7_ERR_DUP_SLOT;
            seen[static_cast<size_t>(id)] = 1;
        }
        for (int32_t i = 0; i < n; ++i) {
            used[static_cast<size_t>(ids[i])] = 0;
            free_list.push_back(ids[i]);
        }
        return WKV7_OK;
    }
};

bool desc_valid(const wkv7_pool_desc *d) {
    return d && d->n_layers >= 1 && d->n_heads >= 1 && d->head_size >= 1 && d->n_slots >= 1 &&
           d->n_snapshots >= 0 && (d->state_dtype == WKV7_F32 || d->state_dtype == WKV7_BF16) &&
           (d->out_dtype == WKV7_F32 || d->out_dtype == WKV7_BF16);
}

size_t state_elem_bytes(const wkv7_pool_desc *d) { return d->state_dtype == WKV7_BF16 ? 2 : 4; }

size_t slot_bytes_of(const wkv7_pool_desc *d) {
    return static_cast<size_t>(d->n_layers) * static_cast<size_t>(d->n_heads) *
           static_cast<size_t>(d->head_size) * static_cast<size_t>(d->head_size) * state_elem_bytes(d);
}

// The id-validation bitmap after the snapshot store: one bit per id of the
// larger table, rounded up to 256 bytes.
size_t marks_bytes_of(const wkv7_pool_desc *d) {
    const size_t ids = static_cast<size_t>(d->n_slots > d->n_snapshots ? d->n_slots : d->n_snapshots);
    const size_t words = (ids + 31) / 32;
    return (words * 4 + 255) / 256 * 256;
}

}  // namespace

namespace wkv7 {
// For entry points defined outside this file: count their launches and record
// their CUDA errors like every other call does.
void note_launches(int launches) {
    g_launches.fetch_add(static_cast<uint64_t>(launches), std::memory_order_relaxed);
}
void note_cuda_error(const char *what, cudaError_t e) { set_error(what, e); }
}  // namespace wkv7

struct wkv7_pool {
    wkv7_pool_desc desc{};
    char *base = nullptr;
    bool owns = false;
    int32_t *status = nullptr;
    float *states = nullptr;
    float *snaps = nullptr;
    uint32_t *marks = nullptr;  // id-validation bitmap (scratch of wkv7_validate_ids)
    long long slot_floats = 0;  // slot bytes / 4: the unit of the byte-copy verbs
    bool state_bf16 = false;
    bool out_bf16 = false;  // o written in bf16
    std::mutex mu;
    IdTable slots;
    IdTable snapshots;
};

namespace {

wkv7::LayerView layer_view(wkv7_pool *p, int32_t layer) {
    wkv7::LayerView lv;
    lv.states = p->states;  // strides below count state elements (float32 or bf16)
    lv.slot_stride = p->state_bf16 ? 2 * p->slot_floats : p->slot_floats;
    lv.layer_off = static_cast<long long>(layer) * p->desc.n_heads * wkv7::kHeadFloats;
    lv.n_slots = p->desc.n_slots;
    lv.n_heads = p->desc.n_heads;
    lv.status = p->status;
    return lv;
}

bool dtype_valid(wkv7_dtype d) { return d == WKV7_F32 || d == WKV7_BF16; }

bool inputs_present(const void *r, const void *w, const void *k, const void *v, const void *a,
                    const void *b, const void *o) {
    return r && w && k && v && a && b && o;
}

// The recurrence kernels read inputs and write o with 8- to 32-byte vector
// accesses (the chunked prefill's tensor maps also need 16-byte bases); every
// access offset is a multiple of 16 bytes from its base.
bool inputs_aligned(const void *r, const void *w, const void *k, const void *v, const void *a,
                    const void *b, const void *o) {
    const void *x[7] = {r, w, k, v, a, b, o};
    for (const void *p : x)
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return false;
    return true;
}

}  // namespace

extern "C" {

size_t wkv7_pool_required_bytes(const wkv7_pool_desc *desc) {
    if (!desc_valid(desc)) return 0;
    size_t sb = slot_bytes_of(desc);
    return kHeaderBytes + sb * (static_cast<size_t>(desc->n_slots) +
                                static_cast<size_t>(desc->n_snapshots)) +
           marks_bytes_of(desc);
}

wkv7_status wkv7_pool_create(const wkv7_pool_desc *desc, wkv7_pool **out) {
    if (!out) return WKV7_ERR_INVALID_ARG;
    *out = nullptr;
    if (!desc_valid(desc)) return WKV7_ERR_INVALID_ARG;
    if (desc->head_size != wkv7::kHeadSize) return WKV7_ERR_UNSUPPORTED;
    size_t need = wkv7_pool_required_bytes(desc);
    if (desc->device_buffer) {
        if (desc->buffer_bytes < need) return WKV7_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(desc->device_buffer) % 256 != 0) return WKV7_ERR_INVALID_ARG;
    }
    wkv7_pool *p = new (std::nothrow) wkv7_pool();
    if (!p) return WKV7_ERR_NO_MEMORY;
    p->desc = *desc;
    if (desc->device_buffer) {
        p->base = static_cast<char *>(desc->device_buffer);
        p->owns = false;
    } else {
        void *mem = nullptr;
        cudaError_t e = cudaMalloc(&mem, need);
        if (e != cudaSuccess) {
            set_error("cudaMalloc(pool)", e);
            delete p;
            return e == cudaErrorMemoryAllocation ? WKV7_ERR_NO_MEMORY : WKV7_ERR_CUDA;
        }
        e = cudaMemset(mem, 0, kHeaderBytes);
        if (e != cudaSuccess) {
            set_error("cudaMemset(status)", e);
            cudaFree(mem);
            delete p;
            return WKV7_ERR_CUDA;
        }
        p->base = static_cast<char *>(mem);
        p->owns = true;
        p->desc.buffer_bytes = need;
    }
    p->desc.device_buffer = p->base;
    p->status = reinterpret_cast<int32_t *>(p->base);
    p->states = reinterpret_cast<float *>(p->base + kHeaderBytes);
    p->slot_floats = static_cast<long long>(slot_bytes_of(desc) / sizeof(float));
    p->state_bf16 = desc->state_dtype == WKV7_BF16;
    p->out_bf16 = desc->out_dtype == WKV7_BF16;
    p->snaps = p->states + static_cast<size_t>(p->slot_floats) * static_cast<size_t>(desc->n_slots);
    p->marks = reinterpret_cast<uint32_t *>(
        p->base + kHeaderBytes +
        slot_bytes_of(desc) * (static_cast<size_t>(desc->n_slots) + static_cast<size_t>(desc->n_snapshots)));
    try {
        p->slots.init(desc->n_slots);
        p->snapshots.init(desc->n_snapshots);
    } catch (...) {
        if (p->owns) cudaFree(p->base);
        delete p;
        return WKV7_ERR_NO_MEMORY;
    }
    *out = p;
    return WKV7_OK;
}

wkv7_status wkv7_pool_destroy(wkv7_pool *pool) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    wkv7_status st = WKV7_OK;
    if (pool->owns) {
        cudaError_t e = cudaFree(pool->base);
        if (e != cudaSuccess) {
            set_error("cudaFree(pool)", e);
            st = WKV7_ERR_CUDA;
        }
    }
    delete pool;
    return st;
}

wkv7_status wkv7_pool_get_desc(const wkv7_pool *pool, wkv7_pool_desc *out) {
    if (!pool || !out) return WKV7_ERR_INVALID_ARG;
    *out = pool->desc;
    return WKV7_OK;
}

size_t wkv7_slot_bytes(const wkv7_pool *pool) {
    return pool ? static_cast<size_t>(pool->slot_floats) * sizeof(float) : 0;
}

wkv7_status wkv7_pool_state_ptr(wkv7_pool *pool, int32_t slot, int32_t layer, float **dev_ptr) {
    if (!pool || !dev_ptr) return WKV7_ERR_INVALID_ARG;
    if (layer < 0 || layer >= pool->desc.n_layers) return WKV7_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->desc.n_slots) return WKV7_ERR_BAD_SLOT;
    *dev_ptr = reinterpret_cast<float *>(
        reinterpret_cast<char *>(pool->states + static_cast<size_t>(slot) * static_cast<size_t>(pool->slot_floats)) +
        static_cast<size_t>(layer) * pool->desc.n_heads * wkv7::kHeadFloats * state_elem_bytes(&pool->desc));
    return WKV7_OK;
}

wkv7_status wkv7_pool_snapshot_ptr(wkv7_pool *pool, int32_t snap, int32_t layer, float **dev_ptr) {
    if (!pool || !dev_ptr) return WKV7_ERR_INVALID_ARG;
    if (layer < 0 || layer >= pool->desc.n_layers) return WKV7_ERR_INVALID_ARG;
    if (snap < 0 || snap >= pool->desc.n_snapshots) return WKV7_ERR_BAD_SLOT;
    *dev_ptr = reinterpret_cast<float *>(
        reinterpret_cast<char *>(pool->snaps + static_cast<size_t>(snap) * static_cast<size_t>(pool->slot_floats)) +
        static_cast<size_t>(layer) * pool->desc.n_heads * wkv7::kHeadFloats * state_elem_bytes(&pool->desc));
    return WKV7_OK;
}

// ------------------------------------------------------------- slot table --

wkv7_status wkv7_slot_alloc(wkv7_pool *pool, int32_t n, int32_t *ids_out) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(pool->mu);
    return pool->slots.alloc(n, ids_out);
}

wkv7_status wkv7_slot_free(wkv7_pool *pool, int32_t n, const int32_t *ids) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(pool->mu);
    return pool->slots.release(n, ids);
}

wkv7_status wkv7_snapshot_alloc(wkv7_pool *pool, int32_t n, int32_t *ids_out) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(pool->mu);
    return pool->snapshots.alloc(n, ids_out);
}

wkv7_status wkv7_snapshot_free(wkv7_pool *pool, int32_t n, const int32_t *ids) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(pool->mu);
    return pool->snapshots.release(n, ids);
}

int32_t wkv7_slot_count_free(const wkv7_pool *pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> g(const_cast<wkv7_pool *>(pool)->mu);
    return pool->slots.n_free();
}

int32_t wkv7_snapshot_count_free(const wkv7_pool *pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> g(const_cast<wkv7_pool *>(pool)->mu);
    return pool->snapshots.n_free();
}

wkv7_status wkv7_slot_is_allocated(const wkv7_pool *pool, int32_t slot, int32_t *out) {
    if (!pool || !out) return WKV7_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->desc.n_slots) return WKV7_ERR_BAD_SLOT;
    std::lock_guard<std::mutex> g(const_cast<wkv7_pool *>(pool)->mu);
    *out = pool->slots.used[static_cast<size_t>(slot)] ? 1 : 0;
    return WKV7_OK;
}

// ------------------------------------------------------------------ verbs --

wkv7_status wkv7_slot_create(wkv7_pool *pool, int32_t n, int32_t *ids_out, cudaStream_t stream) {
    if (!pool || n < 0 || (n > 0 && !ids_out)) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    wkv7_status st = wkv7_slot_alloc(pool, n, ids_out);
    if (st != WKV7_OK) return st;
    int launches = 0;
    cudaError_t e = wkv7::launch_slot_zero_host(pool->states, pool->desc.n_slots, pool->slot_floats,
                                                ids_out, n, pool->status, stream, &launches);
    st = cuda_status("slot_create", e, launches);
    if (st != WKV7_OK) wkv7_slot_free(pool, n, ids_out);
    return st;
}

wkv7_status wkv7_slot_reset(wkv7_pool *pool, const int32_t *slot_ids_dev, int32_t n,
                            cudaStream_t stream) {
    if (!pool || n < 0 || (n > 0 && !slot_ids_dev)) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    int launches = 0;
    cudaError_t e = wkv7::launch_slot_zero_dev(pool->states, pool->desc.n_slots, pool->slot_floats,
                                               slot_ids_dev, n, pool->status, stream, &launches);
    return cuda_status("slot_reset", e, launches);
}

static wkv7_status copy_verb(wkv7_pool *pool, float *dst, int n_dst, const int32_t *dst_ids,
                             const float *src, int n_src, const int32_t *src_ids, int32_t n,
                             cudaStream_t stream, const char *what) {
    if (!pool || n < 0) return WKV7_ERR_INVALID_ARG;  // null ids: checked by the callers
    if (n == 0) return WKV7_OK;
    if (n_dst == 0 || n_src == 0) return WKV7_ERR_INVALID_ARG;  // no snapshot store
    if (n > n_dst) return WKV7_ERR_INVALID_ARG;  // destinations must be distinct
    wkv7::CopyArgs a;
    a.dst = dst;
    a.src = src;
    a.dst_ids = dst_ids;
    a.src_ids = src_ids;
    a.n = n;
    a.n_dst = n_dst;
    a.n_src = n_src;
    a.slot_floats = pool->slot_floats;
    a.status = pool->status;
    int launches = 0;
    cudaError_t e = wkv7::launch_slot_copy(a, stream, &launches);
    return cuda_status(what, e, launches);
}

wkv7_status wkv7_slot_snapshot(wkv7_pool *pool, const int32_t *slot_ids_dev,
                               const int32_t *snap_ids_dev, int32_t n, cudaStream_t stream) {
    if (!pool || (n > 0 && (!slot_ids_dev || !snap_ids_dev))) return WKV7_ERR_INVALID_ARG;
    return copy_verb(pool, pool->snaps, pool->desc.n_snapshots, snap_ids_dev, pool->states,
                     pool->desc.n_slots, slot_ids_dev, n, stream, "slot_snapshot");
}

wkv7_status wkv7_slot_restore(wkv7_pool *pool, const int32_t *snap_ids_dev,
                              const int32_t *slot_ids_dev, int32_t n, cudaStream_t stream) {
    if (!pool || (n > 0 && (!slot_ids_dev || !snap_ids_dev))) return WKV7_ERR_INVALID_ARG;
    return copy_verb(pool, pool->states, pool->desc.n_slots, slot_ids_dev, pool->snaps,
                     pool->desc.n_snapshots, snap_ids_dev, n, stream, "slot_restore");
}

wkv7_status wkv7_slot_fork(wkv7_pool *pool, const int32_t *src_ids_dev, const int32_t *dst_ids_dev,
                           int32_t n, cudaStream_t stream) {
    if (!pool || (n > 0 && (!src_ids_dev || !dst_ids_dev))) return WKV7_ERR_INVALID_ARG;
    return copy_verb(pool, pool->states, pool->desc.n_slots, dst_ids_dev, pool->states,
                     pool->desc.n_slots, src_ids_dev, n, stream, "slot_fork");
}

// Device address of a caller's pinned (page-locked, mapped) host buffer, or
// nullptr when the pointer is not such memory or is not 16-byte aligned.
static void *pinned_host_device_ptr(const void *host) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error state of this query
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return nullptr;
    if (reinterpret_cast<uintptr_t>(attr.devicePointer) % 16 != 0) return nullptr;
    return attr.devicePointer;
}

wkv7_status wkv7_slot_hibernate(wkv7_pool *pool, const int32_t *slot_ids_dev, int32_t n,
                                void *host_dst, size_t host_bytes, cudaStream_t stream) {
    if (!pool || n < 0 || (n > 0 && (!slot_ids_dev || !host_dst))) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    const size_t slot_bytes = static_cast<size_t>(pool->slot_floats) * sizeof(float);
    if (host_bytes / slot_bytes < static_cast<size_t>(n)) return WKV7_ERR_INVALID_ARG;
    void *dev = pinned_host_device_ptr(host_dst);
    if (!dev) return WKV7_ERR_INVALID_ARG;
    return copy_verb(pool, static_cast<float *>(dev), n, nullptr, pool->states, pool->desc.n_slots,
                     slot_ids_dev, n, stream, "slot_hibernate");
}

wkv7_status wkv7_slot_resume(wkv7_pool *pool, const void *host_src, size_t host_bytes,
                             const int32_t *slot_ids_dev, int32_t n, cudaStream_t stream) {
    if (!pool || n < 0 || (n > 0 && (!slot_ids_dev || !host_src))) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    const size_t slot_bytes = static_cast<size_t>(pool->slot_floats) * sizeof(float);
    if (host_bytes / slot_bytes < static_cast<size_t>(n)) return WKV7_ERR_INVALID_ARG;
    const void *dev = pinned_host_device_ptr(host_src);
    if (!dev) return WKV7_ERR_INVALID_ARG;
    return copy_verb(pool, pool->states, pool->desc.n_slots, slot_ids_dev,
                     static_cast<const float *>(dev), n, nullptr, n, stream, "slot_resume");
}

// ------------------------------------------------------------- recurrence --

wkv7_status wkv7_decode_step(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                             int32_t n, wkv7_dtype in_dtype, const void *r, const void *w,
                             const void *k, const void *v, const void *a, const void *b,
                             void *o, cudaStream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.n_layers || n < 0) return WKV7_ERR_INVALID_ARG;
    if (!dtype_valid(in_dtype)) return WKV7_ERR_INVALID_ARG;
    if (n > pool->desc.n_slots) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    if (!slot_ids_dev || !inputs_present(r, w, k, v, a, b, o)) return WKV7_ERR_INVALID_ARG;
    if (!inputs_aligned(r, w, k, v, a, b, o)) return WKV7_ERR_UNSUPPORTED;
    wkv7::DecodeArgs da;
    da.lv = layer_view(pool, layer);
    da.slot_ids = slot_ids_dev;
    da.n = n;
    da.in = {r, w, k, v, a, b, in_dtype == WKV7_BF16, o, pool->out_bf16};
    da.state_bf16 = pool->state_bf16;
    int launches = 0;
    cudaError_t e = wkv7::launch_decode(da, stream, &launches);
    return cuda_status("decode_step", e, launches);
}

wkv7_status wkv7_decode_multi(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                              int32_t n, int32_t n_tokens, wkv7_dtype in_dtype, const void *r,
                              const void *w, const void *k, const void *v, const void *a,
                              const void *b, void *o, const int32_t *step_snap_ids_dev,
                              cudaStream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.n_layers || n < 0 || n_tokens < 1)
        return WKV7_ERR_INVALID_ARG;
    if (!dtype_valid(in_dtype)) return WKV7_ERR_INVALID_ARG;
    if (n > pool->desc.n_slots) return WKV7_ERR_INVALID_ARG;
    if (n == 0) return WKV7_OK;
    if (!slot_ids_dev || !inputs_present(r, w, k, v, a, b, o)) return WKV7_ERR_INVALID_ARG;
    if (!inputs_aligned(r, w, k, v, a, b, o)) return WKV7_ERR_UNSUPPORTED;
    if (step_snap_ids_dev && pool->desc.n_snapshots == 0) return WKV7_ERR_INVALID_ARG;
    if (static_cast<long long>(n) * n_tokens > 0x7fffffffLL) return WKV7_ERR_INVALID_ARG;
    wkv7::DecodeMultiArgs da;
    da.lv = layer_view(pool, layer);
    da.slot_ids = slot_ids_dev;
    da.n = n;
    da.n_tok = n_tokens;
    da.in = {r, w, k, v, a, b, in_dtype == WKV7_BF16, o, pool->out_bf16};
    da.snaps = pool->snaps;
    da.n_snaps = pool->desc.n_snapshots;
    da.step_snap_ids = step_snap_ids_dev;
    da.state_bf16 = pool->state_bf16;
    int launches = 0;
    cudaError_t e = wkv7::launch_decode_multi(da, stream, &launches);
    return cuda_status("decode_multi", e, launches);
}

static wkv7_status prefill_common(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                                  const int32_t *cu_seqlens_dev, int32_t n_seqs,
                                  int32_t total_tokens, int32_t max_seqlen, wkv7_dtype in_dtype,
                                  const void *r, const void *w, const void *k, const void *v,
                                  const void *a, const void *b, void *o, cudaStream_t stream,
                                  bool chunked, const int32_t *cu_ckpt_dev = nullptr,
                                  const int32_t *ckpt_snap_ids_dev = nullptr) {
    if (!pool || layer < 0 || layer >= pool->desc.n_layers) return WKV7_ERR_INVALID_ARG;
    if (n_seqs < 0 || total_tokens < 0 || max_seqlen < 0) return WKV7_ERR_INVALID_ARG;
    if (!dtype_valid(in_dtype)) return WKV7_ERR_INVALID_ARG;
    if (n_seqs > pool->desc.n_slots) return WKV7_ERR_INVALID_ARG;
    if (max_seqlen > total_tokens) return WKV7_ERR_BAD_SEQLENS;
    if (n_seqs == 0) return WKV7_OK;
    if (!slot_ids_dev || !cu_seqlens_dev) return WKV7_ERR_INVALID_ARG;
    if (total_tokens > 0 && !inputs_present(r, w, k, v, a, b, o)) return WKV7_ERR_INVALID_ARG;
    if (chunked && in_dtype != WKV7_BF16) return WKV7_ERR_UNSUPPORTED;
    if (total_tokens > 0 && !inputs_aligned(r, w, k, v, a, b, o)) return WKV7_ERR_UNSUPPORTED;
    wkv7::PrefillArgs pa;
    pa.lv = layer_view(pool, layer);
    pa.slot_ids = slot_ids_dev;
    pa.cu_seqlens = cu_seqlens_dev;
    pa.n_seqs = n_seqs;
    pa.total_tokens = total_tokens;
    pa.max_seqlen = max_seqlen;
    pa.in = {r, w, k, v, a, b, in_dtype == WKV7_BF16, o, pool->out_bf16};
    pa.ck = {pool->snaps, pool->desc.n_snapshots, cu_ckpt_dev, ckpt_snap_ids_dev};
    pa.state_bf16 = pool->state_bf16;
    const bool force_timeout = g_test_wait_timeout.load(std::memory_order_relaxed) != 0;
    pa.wait_cycles = force_timeout ? wkv7::kTestWaitCycles : wkv7::kWaitCycles;
    pa.test_skip_first_load = force_timeout;
    int launches = 0;
    cudaError_t e = chunked ? wkv7::launch_prefill_chunked(pa, stream, &launches)
                            : wkv7::launch_prefill_sequential(pa, stream, &launches);
    return cuda_status(chunked ? "prefill" : "prefill_sequential", e, launches);
}

wkv7_status wkv7_prefill(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                         const int32_t *cu_seqlens_dev, int32_t n_seqs, int32_t total_tokens,
                         int32_t max_seqlen, wkv7_dtype in_dtype, const void *r, const void *w,
                         const void *k, const void *v, const void *a, const void *b, void *o,
                         cudaStream_t stream) {
    return prefill_common(pool, layer, slot_ids_dev, cu_seqlens_dev, n_seqs, total_tokens,
                          max_seqlen, in_dtype, r, w, k, v, a, b, o, stream, true);
}

wkv7_status wkv7_prefill_sequential(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                                    const int32_t *cu_seqlens_dev, int32_t n_seqs,
                                    int32_t total_tokens, int32_t max_seqlen,
                                    wkv7_dtype in_dtype, const void *r, const void *w,
                                    const void *k, const void *v, const void *a, const void *b,
                                    void *o, cudaStream_t stream) {
    return prefill_common(pool, layer, slot_ids_dev, cu_seqlens_dev, n_seqs, total_tokens,
                          max_seqlen, in_dtype, r, w, k, v, a, b, o, stream, false);
}

wkv7_status wkv7_prefill_checkpointed(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                                      const int32_t *cu_seqlens_dev, int32_t n_seqs,
                                      int32_t total_tokens, int32_t max_seqlen,
                                      wkv7_dtype in_dtype, const void *r, const void *w,
                                      const void *k, const void *v, const void *a, const void *b,
                                      void *o, const int32_t *cu_ckpt_dev,
                                      const int32_t *ckpt_snap_ids_dev, int32_t sequential,
                                      cudaStream_t stream) {
    if (!pool) return WKV7_ERR_INVALID_ARG;
    if (n_seqs > 0 && (!cu_ckpt_dev || !ckpt_snap_ids_dev)) return WKV7_ERR_INVALID_ARG;
    if (n_seqs > 0 && pool->desc.n_snapshots == 0) return WKV7_ERR_INVALID_ARG;  // nowhere to write
    return prefill_common(pool, layer, slot_ids_dev, cu_seqlens_dev, n_seqs, total_tokens,
                          max_seqlen, in_dtype, r, w, k, v, a, b, o, stream, sequential == 0,
                          cu_ckpt_dev, ckpt_snap_ids_dev);
}

// ------------------------------------------------------------- validation --

wkv7_status wkv7_validate_ids(wkv7_pool *pool, int32_t table, const int32_t *ids_a_dev, int32_t n_a,
                              const int32_t *ids_b_dev, int32_t n_b, cudaStream_t stream) {
    if (!pool || n_a < 0 || n_b < 0) return WKV7_ERR_INVALID_ARG;
    if (table != WKV7_TABLE_SLOTS && table != WKV7_TABLE_SNAPSHOTS) return WKV7_ERR_INVALID_ARG;
    if ((n_a > 0 && !ids_a_dev) || (n_b > 0 && !ids_b_dev)) return WKV7_ERR_INVALID_ARG;
    if (n_a == 0 && n_b == 0) return WKV7_OK;
    wkv7::ValidateArgs va;
    va.marks = pool->marks;
    va.n_table = table == WKV7_TABLE_SLOTS ? pool->desc.n_slots : pool->desc.n_snapshots;
    va.ids_a = ids_a_dev;
    va.n_a = n_a;
    va.ids_b = ids_b_dev;
    va.n_b = n_b;
    va.status = pool->status;
    int launches = 0;
    cudaError_t e = wkv7::launch_validate_ids(va, stream, &launches);
    return cuda_status("validate_ids", e, launches);
}

// ----------------------------------------------------------------- status --

wkv7_status wkv7_get_device_status(wkv7_pool *pool, cudaStream_t stream, int32_t timeout_ms,
                                   int32_t *code_out) {
    if (!pool || !code_out) return WKV7_ERR_INVALID_ARG;
    *code_out = WKV7_DEV_OK;
    if (timeout_ms <= 0) timeout_ms = 10000;
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_status("status:event", e, 0);
    e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) {
        cudaEventDestroy(ev);
        return cuda_status("status:record", e, 0);
    }
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        e = cudaEventQuery(ev);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) {
            cudaEventDestroy(ev);
            return cuda_status("status:query", e, 0);
        }
        auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                      std::chrono::steady_clock::now() - t0)
                      .count();
        if (ms > timeout_ms) {
            cudaEventDestroy(ev);
            return WKV7_ERR_TIMEOUT;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    cudaEventDestroy(ev);
    int32_t code = 0;
    e = cudaMemcpy(&code, pool->status, sizeof(code), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status("status:read", e, 0);
    if (code != 0) {
        e = cudaMemset(pool->status, 0, sizeof(int32_t));
        if (e != cudaSuccess) return cuda_status("status:clear", e, 0);
    }
    *code_out = code;
    if (code == WKV7_DEV_DUP_SLOT) return WKV7_ERR_DUP_SLOT;
    return code != 0 ? WKV7_ERR_DEVICE_STATUS : WKV7_OK;
}

const char *wkv7_status_string(wkv7_status s) {
    switch (s) {
        case WKV7_OK: return "ok";
        case WKV7_ERR_INVALID_ARG: return "invalid argument";
        case WKV7_ERR_BAD_SLOT: return "slot id out of range or not allocated";
        case WKV7_ERR_DUP_SLOT: return "duplicate slot id";
        case WKV7_ERR_POOL_FULL: return "not enough free slots";
        case WKV7_ERR_BAD_SEQLENS: return "inconsistent sequence lengths";
        case WKV7_ERR_CUDA: return "CUDA error";
        case WKV7_ERR_UNSUPPORTED: return "unsupported configuration";
        case WKV7_ERR_DEVICE_STATUS: return "a kernel reported a device-side fault";
        case WKV7_ERR_TIMEOUT: return "timed out waiting for the stream";
        case WKV7_ERR_NO_MEMORY: return "out of memory";
    }
    return "unknown status";
}

const char *wkv7_last_error(void) { return g_last_error; }

uint64_t wkv7_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

wkv7_status wkv7_test_force_wait_timeout(int32_t on) {
    g_test_wait_timeout.store(on != 0, std::memory_order_relaxed);
    return WKV7_OK;
}

int32_t wkv7_version(void) { return WKV7_VERSION; }

}  // extern "C"
