// Debug validation of device id arrays: every id in range, no id twice.
//
// The fast paths assume that the slot ids of one call are distinct and that the
// slots a mixed serving step decodes do not overlap the slots it prefills (two
// CTAs updating one state would race).  Checking that on every call would cost
// a pass over the ids and a scratch bitmap per call, so it is a separate pass a
// caller runs when debugging: the state-slot engine's hard-error discipline
// (the rvLLM README: no silent fallback, a wrong request is an error) applied
// to ids that only the device holds.
//
// Two launches on the caller's stream: clear a bitmap of one bit per table id,
// then set each listed id's bit with an atomic OR; an id whose bit was already
// set is a repeat (WKV7_DEV_DUP_SLOT), an id outside the table is
// WKV7_DEV_BAD_SLOT.  Nothing but the bitmap and the status word is written.
#include <mutex>

#include "device_common.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocks = 152 * 8;

__global__ void __launch_bounds__(kThreads) ids_clear_kernel(uint32_t *marks, int n_words) {
    pdl_prologue();
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_words; i += gridDim.x * kThreads) marks[i] = 0u;
}

__global__ void __launch_bounds__(kThreads) ids_mark_kernel(uint32_t *marks, int n_table, const int *ids_a,
                                                            int n_a, const int *ids_b, int n_b, int *status) {
    pdl_prologue();
    const long long n = static_cast<long long>(n_a) + n_b;
    for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * kThreads) {
        const int id = i < n_a ? __ldg(ids_a + i) : __ldg(ids_b + (i - n_a));
        if (id < 0 || id >= n_table) {
            flag_status(status, WKV7_DEV_BAD_SLOT);
            continue;
        }
        const uint32_t bit = 1u << (id & 31);
        if (atomicOr(marks + (id >> 5), bit) & bit) flag_status(status, WKV7_DEV_DUP_SLOT);
    }
}

unsigned blocks_for(long long n) {
    const long long b = (n + kThreads - 1) / kThreads;
    return static_cast<unsigned>(b < 1 ? 1 : (b > kMaxBlocks ? kMaxBlocks : b));
}

}  // namespace

cudaError_t launch_validate_ids(const ValidateArgs &a, cudaStream_t s, int *launches) {
    const int n_words = (a.n_table + 31) / 32;
    cudaError_t e = launch_pdl(ids_clear_kernel, dim3(blocks_for(n_words)), dim3(kThreads), 0, s, a.marks,
                               n_words);
    ++*launches;
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_pdl(ids_mark_kernel, dim3(blocks_for(static_cast<long long>(a.n_a) + a.n_b)), dim3(kThreads), 0,
                   s, a.marks, a.n_table, a.ids_a, a.n_a, a.ids_b, a.n_b, a.status);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ----------------------------------------------- the allocation-free variant
// wkv7_validate_ids_noalloc runs the same check without a pool: its bitmap is
// the file-scope array below instead of the pool's scratch region, and its
// verdict goes to a caller-owned word.  The array is part of the library's
// device image, so every GPU that loads the library holds its 128 KiB until
// the process exits; every call on a device shares it.
constexpr int kNoAllocMaxIds = 1 << 20;
static __device__ __align__(256) uint32_t g_noalloc_marks[kNoAllocMaxIds / 32];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
uint32_t *g_noalloc_ptr[kMaxDevices] = {};  // device address of the array, per device

// Zero the first n_words words of the array and the caller's result word.
__global__ void __launch_bounds__(kThreads) ids_clear_noalloc_kernel(uint32_t *marks, int n_words,
                                                                     int *result) {
    pdl_prologue();
    if (blockIdx.x == 0 && threadIdx.x == 0) *result = 0;
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_words; i += gridDim.x * kThreads) marks[i] = 0u;
}

}  // namespace

}  // namespace wkv7

extern "C" wkv7_status wkv7_validate_ids_noalloc(int32_t n_table, const int32_t *ids_a_dev, int32_t n_a,
                                                 const int32_t *ids_b_dev, int32_t n_b, int32_t *result_dev,
                                                 cudaStream_t stream) {
    using namespace wkv7;
    if (n_table < 0 || n_a < 0 || n_b < 0 || !result_dev) return WKV7_ERR_INVALID_ARG;
    if ((n_a > 0 && !ids_a_dev) || (n_b > 0 && !ids_b_dev)) return WKV7_ERR_INVALID_ARG;
    if (n_table > kNoAllocMaxIds) return WKV7_ERR_UNSUPPORTED;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        note_cuda_error("validate_ids_noalloc:device", e != cudaSuccess ? e : cudaErrorInvalidDevice);
        return WKV7_ERR_CUDA;
    }
    uint32_t *marks = nullptr;
    {  // set-up, once per device, with that device current: the array's device address
        std::lock_guard<std::mutex> g(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_marks);
            if (e != cudaSuccess || !ptr) {
                note_cuda_error("validate_ids_noalloc:cudaGetSymbolAddress",
                                e != cudaSuccess ? e : cudaErrorInvalidSymbol);
                return WKV7_ERR_CUDA;
            }
            g_noalloc_ptr[dev] = static_cast<uint32_t *>(ptr);
        }
        marks = g_noalloc_ptr[dev];
    }
    const int n_words = (n_table + 31) / 32;
    int launches = 0;
    e = launch_pdl(ids_clear_noalloc_kernel, dim3(blocks_for(n_words)), dim3(kThreads), 0, stream, marks,
                   n_words, reinterpret_cast<int *>(result_dev));
    ++launches;
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess && static_cast<long long>(n_a) + n_b > 0) {
        e = launch_pdl(ids_mark_kernel, dim3(blocks_for(static_cast<long long>(n_a) + n_b)), dim3(kThreads), 0,
                       stream, marks, static_cast<int>(n_table), reinterpret_cast<const int *>(ids_a_dev), n_a,
                       reinterpret_cast<const int *>(ids_b_dev), n_b, reinterpret_cast<int *>(result_dev));
        ++launches;
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    note_launches(launches);
    if (e != cudaSuccess) {
        note_cuda_error("validate_ids_noalloc", e);
        return WKV7_ERR_CUDA;
    }
    return WKV7_OK;
}
