// Small device helpers shared by the WKV-7 kernels.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "wkv7.h"

namespace wkv7 {

// Record a device fault in the sticky status word; the first fault wins.
__device__ __forceinline__ void flag_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

// Two floats -> a bf16 pair (low, high), each rounded to nearest even.
__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// Load 4 consecutive input values at element offset `off` as floats.
template <bool BF16>
__device__ __forceinline__ float4 load4(const void *p, size_t off) {
    if constexpr (BF16) {
        uint2 u = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p) + off));
        return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    } else {
        return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + off));
    }
}

// Load one input value at element offset `off` as float.
template <bool BF16>
__device__ __forceinline__ float load1(const void *p, size_t off) {
    if constexpr (BF16) {
        uint16_t u = __ldg(static_cast<const unsigned short *>(p) + off);
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    } else {
        return __ldg(static_cast<const float *>(p) + off);
    }
}

// Load 8 consecutive input values at element offset `off` (16-byte aligned for
// bf16, 32-byte for float) as floats.
template <bool BF16>
__device__ __forceinline__ void load8(const void *p, size_t off, float *x) {
    if constexpr (BF16) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + off));
        x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
        x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
    } else {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + off);
        float4 a = __ldg(q), b = __ldg(q + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
}

// x rounded to the nearest bf16 value (ties to even), as a float.
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Four consecutive state entries at element offset `off` of a float32 state
// array or, with SBF16, a bf16 one (16- or 8-byte aligned).
template <bool SBF16>
__device__ __forceinline__ float4 load_state4(const float *states, size_t off) {
    if constexpr (SBF16) {
        const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(states) + off);
        return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    } else {
        return *reinterpret_cast<const float4 *>(states + off);
    }
}

// The store counterpart: with SBF16 each entry is rounded to bf16 (nearest even).
template <bool SBF16>
__device__ __forceinline__ void store_state4(float *states, size_t off, float4 x) {
    if constexpr (SBF16) {
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(states) + off) =
            make_uint2(pack_bf16_rn(x.x, x.y), pack_bf16_rn(x.z, x.w));
    } else {
        *reinterpret_cast<float4 *>(states + off) = x;
    }
}

// Eight floats to global memory in one 32-byte store (sm_100 and later); p must
// be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float *p, const float *v) {
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
                 "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// Eight 32-bit words to global memory in one 32-byte store; p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8_b32(uint32_t *p, const uint32_t *v) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// One output element o[idx]: float32, or rounded to bf16 (nearest even) when the
// pool's out_dtype is bf16.
__device__ __forceinline__ void store_out(void *o, bool o_bf16, size_t idx, float v) {
    if (o_bf16)
        reinterpret_cast<__nv_bfloat16 *>(o)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(o)[idx] = v;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl lets the next
// kernel in its stream start launching once all of its CTAs have begun
// (launch_dependents), and itself waits for everything before it in the stream
// to complete and become visible (wait) before it reads or writes anything that
// earlier work may produce, so only the launch latency, CTA dispatch and (in the
// decode kernels) a slot-id read and an L2 prefetch overlap the previous kernel's
// tail.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_prologue() {
    pdl_launch_dependents();
    pdl_wait();
}

// Warm L2 with the 128-byte line at p (no visible effect: safe before pdl_wait).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

}  // namespace wkv7
