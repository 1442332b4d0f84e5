// Slot verbs as device copies ("wkvm: state-slot inference for RWKV, GDN and
// Mamba hybrids", "The allocation unit wkvm changes": create, snapshot, fork,
// hibernate, resume; hibernate and resume move slots to and from a pinned host
// buffer that the kernel reaches through its mapped device address).  A slot is
// one contiguous range of states (every layer and head; float32 or bf16, moved
// here as 16-byte words, so the verbs are bit-exact for either), so every verb
// is a whole-range copy or fill.  Each CTA moves 32 KiB of one slot with
// 128-bit streaming loads/stores; grid.y walks the slot pairs.  HBM-bound:
// 2 x slot_bytes per copied slot, 1 x per zeroed slot.
#include "device_common.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 8;                       // float4 per thread
constexpr long long kVecPerCta = kThreads * kVecPerThread;
constexpr int kMaxGridY = 65535;

__global__ void __launch_bounds__(kThreads) slot_copy_kernel(CopyArgs a, int pair0) {
    pdl_prologue();
    const int pair = pair0 + blockIdx.y;
    const int d = a.dst_ids ? __ldg(a.dst_ids + pair) : pair;  // no id array: the i-th slot of a packed buffer
    const int s = a.src_ids ? __ldg(a.src_ids + pair) : pair;
    if (d < 0 || d >= a.n_dst || s < 0 || s >= a.n_src) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(a.status, WKV7_DEV_BAD_SLOT);
        return;
    }
    const float4 *src = reinterpret_cast<const float4 *>(a.src + static_cast<size_t>(s) * a.slot_floats);
    float4 *dst = reinterpret_cast<float4 *>(a.dst + static_cast<size_t>(d) * a.slot_floats);
    const long long n4 = a.slot_floats / 4;
    const long long base = static_cast<long long>(blockIdx.x) * kVecPerCta + threadIdx.x;
    float4 v[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        long long idx = base + static_cast<long long>(u) * kThreads;
        if (idx < n4) v[u] = __ldcs(src + idx);
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        long long idx = base + static_cast<long long>(u) * kThreads;
        if (idx < n4) __stcs(dst + idx, v[u]);
    }
}

__device__ __forceinline__ void zero_range(float *states, long long slot_floats, int slot) {
    float4 *dst = reinterpret_cast<float4 *>(states + static_cast<size_t>(slot) * slot_floats);
    const long long n4 = slot_floats / 4;
    const long long base = static_cast<long long>(blockIdx.x) * kVecPerCta + threadIdx.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        long long idx = base + static_cast<long long>(u) * kThreads;
        if (idx < n4) __stcs(dst + idx, z);
    }
}

__global__ void __launch_bounds__(kThreads) slot_zero_dev_kernel(float *states, int n_slots,
                                                                 long long slot_floats,
                                                                 const int *ids, int pair0,
                                                                 int *status) {
    pdl_prologue();
    const int slot = __ldg(ids + pair0 + blockIdx.y);
    if (slot < 0 || slot >= n_slots) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(status, WKV7_DEV_BAD_SLOT);
        return;
    }
    zero_range(states, slot_floats, slot);
}

__global__ void __launch_bounds__(kThreads) slot_zero_val_kernel(float *states, int n_slots,
                                                                 long long slot_floats, ZeroIds ids,
                                                                 int *status) {
    pdl_prologue();
    const int slot = ids.ids[blockIdx.y];
    if (slot < 0 || slot >= n_slots) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(status, WKV7_DEV_BAD_SLOT);
        return;
    }
    zero_range(states, slot_floats, slot);
}

unsigned blocks_per_slot(long long slot_floats) {
    const long long n4 = slot_floats / 4;
    return static_cast<unsigned>((n4 + kVecPerCta - 1) / kVecPerCta);
}

}  // namespace

cudaError_t launch_slot_copy(const CopyArgs &a, cudaStream_t s, int *launches) {
    const unsigned gx = blocks_per_slot(a.slot_floats);
    for (int p0 = 0; p0 < a.n; p0 += kMaxGridY) {
        const int cnt = a.n - p0 < kMaxGridY ? a.n - p0 : kMaxGridY;
        cudaError_t e = launch_pdl(slot_copy_kernel, dim3(gx, static_cast<unsigned>(cnt)), dim3(kThreads), 0, s,
                                   a, p0);
        ++*launches;
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_slot_zero_dev(float *states, int n_slots, long long slot_floats,
                                 const int *ids_dev, int n, int *status, cudaStream_t s,
                                 int *launches) {
    const unsigned gx = blocks_per_slot(slot_floats);
    for (int p0 = 0; p0 < n; p0 += kMaxGridY) {
        const int cnt = n - p0 < kMaxGridY ? n - p0 : kMaxGridY;
        cudaError_t e = launch_pdl(slot_zero_dev_kernel, dim3(gx, static_cast<unsigned>(cnt)), dim3(kThreads), 0,
                                   s, states, n_slots, slot_floats, ids_dev, p0, status);
        ++*launches;
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_slot_zero_host(float *states, int n_slots, long long slot_floats,
                                  const int *ids_host, int n, int *status, cudaStream_t s,
                                  int *launches) {
    const unsigned gx = blocks_per_slot(slot_floats);
    for (int p0 = 0; p0 < n; p0 += kZeroIdsPerLaunch) {
        const int cnt = n - p0 < kZeroIdsPerLaunch ? n - p0 : kZeroIdsPerLaunch;
        ZeroIds ids;
        for (int i = 0; i < cnt; ++i) ids.ids[i] = ids_host[p0 + i];
        cudaError_t e = launch_pdl(slot_zero_val_kernel, dim3(gx, static_cast<unsigned>(cnt)), dim3(kThreads), 0,
                                   s, states, n_slots, slot_floats, ids, status);
        ++*launches;
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace wkv7
