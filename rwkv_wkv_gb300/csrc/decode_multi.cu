// Multi-token WKV-7 decode over indirected state slots.
//
// RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)": per head and
// token, h = S a; S <- S diag(w) + h b^T + v k^T; o = S r, applied here K
// times in a row to the same state.  The thread mapping is the single-token
// decode's: 256 threads per (row, head), thread t holding the float4 at byte
// offset 16*t + 4096*m of the 16 KiB state, row reductions as xor shuffles
// inside a half-warp.
#include <type_traits>

#include "device_common.cuh"
#include "row_sums.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

// K consecutive tokens per (row, head) with the state held in registers
// throughout: the state is read and written once per call instead of once per
// token, and only the inputs and readouts scale with K.  The inputs of up to
// kGroup tokens are staged in shared memory (as they come, bf16 or float32) by
// the whole CTA at once, so their loads overlap each other and the state load
// instead of sitting on the token chain.  With per-token snapshots the state
// after every token is also
// streamed to its snapshot (the rollback points of a speculative verify: the
// rvLLM README, "Speculative decoding", verifies K+1 tokens in one pass; wkvm's
// fork/restore verbs then keep or drop them).  On a bf16-state pool (SBF16) the
// call is K decode steps: the state is rounded to bf16 after every token, as a
// single-token step stores it, and carried on rounded; the readout of each token
// uses its unrounded state, and the rollback snapshots hold the rounded states.
constexpr int kGroup = 8;  // tokens staged per pass
enum { kR = 0, kW, kK, kV, kA, kB, kInputs };

// Staged inputs of one group of tokens: bf16 inputs stay bf16 in shared memory
// (half the bytes each token's broadcast reads move), float32 ones float32.
template <bool BF16>
struct Staged {
    using Elem = typename std::conditional<BF16, uint16_t, float>::type;
    Elem x[kGroup][kInputs][kHeadSize];
    __device__ __forceinline__ float4 vec4(int t, int i, int c) const {  // elements c..c+3
        if constexpr (BF16) {
            const uint2 u = *reinterpret_cast<const uint2 *>(&x[t][i][c]);
            return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
        } else {
            return *reinterpret_cast<const float4 *>(&x[t][i][c]);
        }
    }
    __device__ __forceinline__ float one(int t, int i, int e) const {
        if constexpr (BF16)
            return __uint_as_float(static_cast<uint32_t>(x[t][i][e]) << 16);
        else
            return x[t][i][e];
    }
    // four consecutive input elements from global memory, as they are stored here
    __device__ __forceinline__ void stage4(int t, int i, int c, const void *src, size_t off) {
        if constexpr (BF16)
            *reinterpret_cast<uint2 *>(&x[t][i][c]) =
                __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(src) + off));
        else
            *reinterpret_cast<float4 *>(&x[t][i][c]) =
                __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(src) + off));
    }
};

template <bool BF16, bool SNAPS, bool SBF16>
__global__ void __launch_bounds__(256, (SNAPS && SBF16) ? 4 : 5) decode_multi_kernel(DecodeMultiArgs p) {
    __shared__ __align__(16) Staged<BF16> xs;
    pdl_prologue();
    const int H = p.lv.n_heads;
    const int unit = blockIdx.x;
    const int bi = unit / H;
    const int h = unit - bi * H;
    const int slot = __ldg(p.slot_ids + bi);
    if (slot < 0 || slot >= p.lv.n_slots) {
        if (threadIdx.x == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }
    // element offset of this (slot, layer, head) state; elements are bf16 with SBF16
    const size_t s_off = static_cast<size_t>(slot) * p.lv.slot_stride + p.lv.layer_off +
                         static_cast<size_t>(h) * kHeadFloats;
    float *S = p.lv.states + s_off;  // float32 states only
    const int tid = threadIdx.x;
    const int c = (tid & 15) * 4;
    const int row0 = tid >> 4;
    const int K = p.n_tok;

    float4 s[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if constexpr (SBF16)
            s[m] = load_state4<true>(p.lv.states, s_off + (row0 + 16 * m) * kHeadSize + c);
        else
            s[m] = __ldcs(reinterpret_cast<const float4 *>(S + (row0 + 16 * m) * kHeadSize + c));
    }

    // token k of row bi, head h: [(bi*K + k)*H + h][64]
    auto io_of = [&](int k) { return (static_cast<size_t>(bi) * K + k) * H * kHeadSize + h * kHeadSize; };
#pragma unroll 1
    for (int g0 = 0; g0 < K; g0 += kGroup) {
        const int ng = min(kGroup, K - g0);
        if (g0 > 0) __syncthreads();  // the previous group is consumed
        // stage: ng tokens x 6 inputs x 16 float4 (one float4 per thread per item)
        for (int e = tid; e < ng * kInputs * 16; e += 256) {
            const int t = e / (kInputs * 16);
            const int rem = e - t * (kInputs * 16);
            const int x = rem >> 4, q = rem & 15;
            const void *src = x == kR ? p.in.r : x == kW ? p.in.w : x == kK ? p.in.k
                            : x == kV ? p.in.v : x == kA ? p.in.a : p.in.b;
            xs.stage4(t, x, 4 * q, src, io_of(g0 + t) + 4 * q);
        }
        __syncthreads();
#pragma unroll 1
        for (int t = 0; t < ng; ++t) {
            const int k = g0 + t;
            const float4 a4 = xs.vec4(t, kA, c);
            float hs[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) hs[m] = dot4(s[m], a4);
            row_sums4(hs, tid & 31);  // every lane needs all four sums
            const float4 w4 = xs.vec4(t, kW, c);
            const float4 b4 = xs.vec4(t, kB, c);
            const float4 k4 = xs.vec4(t, kK, c);
            const float4 r4 = xs.vec4(t, kR, c);
            float os[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float vm = xs.one(t, kV, row0 + 16 * m);
                s[m].x = fmaf(s[m].x, w4.x, fmaf(hs[m], b4.x, vm * k4.x));
                s[m].y = fmaf(s[m].y, w4.y, fmaf(hs[m], b4.y, vm * k4.y));
                s[m].z = fmaf(s[m].z, w4.z, fmaf(hs[m], b4.z, vm * k4.z));
                s[m].w = fmaf(s[m].w, w4.w, fmaf(hs[m], b4.w, vm * k4.w));
                os[m] = dot4(s[m], r4);
                if constexpr (SBF16)
                    s[m] = make_float4(round_bf16(s[m].x), round_bf16(s[m].y), round_bf16(s[m].z),
                                       round_bf16(s[m].w));
            }
            if (SNAPS) {
                const int id = __ldg(p.step_snap_ids + static_cast<size_t>(bi) * K + k);
                if (id >= 0 && id < p.n_snaps) {
                    const size_t d_off = static_cast<size_t>(id) * p.lv.slot_stride + p.lv.layer_off +
                                         static_cast<size_t>(h) * kHeadFloats;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        if constexpr (SBF16)
                            store_state4<true>(p.snaps, d_off + (row0 + 16 * m) * kHeadSize + c, s[m]);
                        else
                            __stcs(reinterpret_cast<float4 *>(p.snaps + d_off + (row0 + 16 * m) * kHeadSize + c),
                                   s[m]);
                    }
                } else if (tid == 0) {
                    flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
                }
            }
            const float ou = reduce_scatter4(os, tid & 15);  // row ((tid >> 2) & 3)'s readout
            if ((tid & 3) == 0) store_out(p.in.o, p.in.o_bf16, io_of(k) + row0 + 16 * ((tid >> 2) & 3), ou);
        }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if constexpr (SBF16)
            store_state4<true>(p.lv.states, s_off + (row0 + 16 * m) * kHeadSize + c, s[m]);
        else
            __stcs(reinterpret_cast<float4 *>(S + (row0 + 16 * m) * kHeadSize + c), s[m]);
    }
}

}  // namespace


cudaError_t launch_decode_multi(const DecodeMultiArgs &a, cudaStream_t s, int *launches) {
    const long long units = static_cast<long long>(a.n) * a.lv.n_heads;
    if (units <= 0 || a.n_tok <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(units));
    const bool snaps = a.step_snap_ids != nullptr;
    const int variant = (a.in.bf16 ? 4 : 0) | (snaps ? 2 : 0) | (a.state_bf16 ? 1 : 0);
    void (*const kernels[8])(DecodeMultiArgs) = {
        decode_multi_kernel<false, false, false>, decode_multi_kernel<false, false, true>,
        decode_multi_kernel<false, true, false>,  decode_multi_kernel<false, true, true>,
        decode_multi_kernel<true, false, false>,  decode_multi_kernel<true, false, true>,
        decode_multi_kernel<true, true, false>,   decode_multi_kernel<true, true, true>};
    const cudaError_t e = launch_pdl(kernels[variant], grid, dim3(256), 0, s, a);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace wkv7
