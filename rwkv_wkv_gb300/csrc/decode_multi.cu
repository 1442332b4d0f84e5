// Multi-token WKV-7 decode over indirected state slots.
//
// RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)": per head and
// token, h = S a; S <- S diag(w) + h b^T + v k^T; o = S r, applied here K
// times in a row to the same state.  The thread mapping is the single-token
// decode's: 256 threads per (row, head), thread t holding the float4 at byte
// offset 16*t + 4096*m of the 16 KiB state, row reductions as xor shuffles
// inside a half-warp.
#include "device_common.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

// K consecutive tokens per (row, head) with the state held in registers
// throughout: the state is read and written once per call instead of once per
// token, and only the inputs and readouts scale with K.  The inputs of token
// k+1 are loaded while token k computes.  With per-token snapshots the state
// after every token is also streamed to its snapshot (the rollback points of a
// speculative verify: the rvLLM README, "Speculative decoding", verifies K+1
// tokens in one pass; wkvm's fork/restore verbs then keep or drop them).
struct TokIn {
    float4 a, w, b, k, r;
    float v[4];
};

template <bool BF16>
__device__ __forceinline__ void load_tok(const TokenInputs &in, size_t io, int c, int row0, TokIn &t) {
    t.a = load4<BF16>(in.a, io + c);
    t.w = load4<BF16>(in.w, io + c);
    t.b = load4<BF16>(in.b, io + c);
    t.k = load4<BF16>(in.k, io + c);
    t.r = load4<BF16>(in.r, io + c);
#pragma unroll
    for (int m = 0; m < 4; ++m) t.v[m] = load1<BF16>(in.v, io + row0 + 16 * m);
}

template <bool BF16, bool SNAPS>
__global__ void __launch_bounds__(256) decode_multi_kernel(DecodeMultiArgs p) {
    const int H = p.lv.n_heads;
    const int unit = blockIdx.x;
    const int bi = unit / H;
    const int h = unit - bi * H;
    const int slot = __ldg(p.slot_ids + bi);
    if (slot < 0 || slot >= p.lv.n_slots) {
        if (threadIdx.x == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }
    float *S = p.lv.states + static_cast<size_t>(slot) * p.lv.slot_stride + p.lv.layer_off +
               static_cast<size_t>(h) * kHeadFloats;
    const int tid = threadIdx.x;
    const int c = (tid & 15) * 4;
    const int row0 = tid >> 4;
    const int K = p.n_tok;

    float4 s[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4 *>(S + (row0 + 16 * m) * kHeadSize + c));

    // token k of row bi, head h: [(bi*K + k)*H + h][64]
    auto io_of = [&](int k) { return (static_cast<size_t>(bi) * K + k) * H * kHeadSize + h * kHeadSize; };
    TokIn cur, nxt;
    load_tok<BF16>(p.in, io_of(0), c, row0, cur);
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
        if (k + 1 < K) load_tok<BF16>(p.in, io_of(k + 1), c, row0, nxt);
        float hs[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) hs[m] = dot4(s[m], cur.a);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
            for (int m = 0; m < 4; ++m) hs[m] += __shfl_xor_sync(0xffffffffu, hs[m], off);
        float os[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            s[m].x = fmaf(s[m].x, cur.w.x, fmaf(hs[m], cur.b.x, cur.v[m] * cur.k.x));
            s[m].y = fmaf(s[m].y, cur.w.y, fmaf(hs[m], cur.b.y, cur.v[m] * cur.k.y));
            s[m].z = fmaf(s[m].z, cur.w.z, fmaf(hs[m], cur.b.z, cur.v[m] * cur.k.z));
            s[m].w = fmaf(s[m].w, cur.w.w, fmaf(hs[m], cur.b.w, cur.v[m] * cur.k.w));
            os[m] = dot4(s[m], cur.r);
        }
        if (SNAPS) {
            const int id = __ldg(p.step_snap_ids + static_cast<size_t>(bi) * K + k);
            if (id >= 0 && id < p.n_snaps) {
                float *D = p.snaps + static_cast<size_t>(id) * p.lv.slot_stride + p.lv.layer_off +
                           static_cast<size_t>(h) * kHeadFloats;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    __stcs(reinterpret_cast<float4 *>(D + (row0 + 16 * m) * kHeadSize + c), s[m]);
            } else if (tid == 0) {
                flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
            }
        }
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
            for (int m = 0; m < 4; ++m) os[m] += __shfl_xor_sync(0xffffffffu, os[m], off);
        if ((tid & 15) == 0) {
            const size_t io = io_of(k);
#pragma unroll
            for (int m = 0; m < 4; ++m) p.in.o[io + row0 + 16 * m] = os[m];
        }
        cur = nxt;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
        __stcs(reinterpret_cast<float4 *>(S + (row0 + 16 * m) * kHeadSize + c), s[m]);
}

}  // namespace


cudaError_t launch_decode_multi(const DecodeMultiArgs &a, cudaStream_t s, int *launches) {
    const long long units = static_cast<long long>(a.n) * a.lv.n_heads;
    if (units <= 0 || a.n_tok <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(units));
    const bool snaps = a.step_snap_ids != nullptr;
    if (a.in.bf16) {
        if (snaps) decode_multi_kernel<true, true><<<grid, 256, 0, s>>>(a);
        else decode_multi_kernel<true, false><<<grid, 256, 0, s>>>(a);
    } else {
        if (snaps) decode_multi_kernel<false, true><<<grid, 256, 0, s>>>(a);
        else decode_multi_kernel<false, false><<<grid, 256, 0, s>>>(a);
    }
    ++*launches;
    return cudaGetLastError();
}

}  // namespace wkv7
