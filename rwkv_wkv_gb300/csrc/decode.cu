// Batched single-token WKV-7 decode over indirected state slots.
//
// RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)": per head and
// token, h = S a; S <- S diag(w) + h b^T + v k^T; o = S r.  One CTA advances
// one (batch row, head) unit: it streams that head's 64x64 float32 state
// (16 KiB) from HBM into registers once, applies the step, streams it back and
// writes the 64 readouts.  The kernel is bound by HBM bandwidth: per unit it
// moves 32 KiB of state against ~37 kFLOP.
//
// Thread mapping (256 threads): thread t holds the float4 at byte offset
// 16*t + 4096*m (m = 0..3) of the state, i.e. key columns 4*(t%16)..+3 of
// value rows t/16 + 16*m.  Each load/store instruction of the CTA covers 4 KiB
// of contiguous memory.  A row's 64 columns sit in one half-warp, so both
// row reductions (S a before the update, S' r after it) stay inside the
// half-warp (row_sums.cuh), and the state never touches shared memory.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "row_sums.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

// CTAs that can be resident when a kernel starts launching before its
// predecessor ends (152 SMs, up to 8 of these CTAs each); only they prefetch.
constexpr int kFirstWaveCtas = 152 * 8;

template <bool BF16>
__global__ void __launch_bounds__(256) decode_kernel(DecodeArgs p) {
    pdl_launch_dependents();
    const int H = p.lv.n_heads;
    const int unit = blockIdx.x;
    const int bi = unit / H;
    const int h = unit - bi * H;
    const int tid = threadIdx.x;
    const int c = (tid & 15) * 4;  // first key column held by this thread
    const int row0 = tid >> 4;     // value rows row0 + 16*m
    // Before waiting for the previous kernel: the slot id (no kernel of the library
    // writes an id array) and, in the CTAs that can be resident while the previous
    // kernel drains, an L2 prefetch of the unit's state rows (it only warms L2), so
    // that the first wave's loads after the wait hit L2.
    const int slot = __ldg(p.slot_ids + bi);
    const bool ok = slot >= 0 && slot < p.lv.n_slots;
    float *S = p.lv.states + static_cast<size_t>(ok ? slot : 0) * p.lv.slot_stride + p.lv.layer_off +
               static_cast<size_t>(h) * kHeadFloats;
    if (ok && unit < kFirstWaveCtas && (tid & 7) == 0) {  // one prefetch per 128-byte line
#pragma unroll
        for (int m = 0; m < 4; ++m) prefetch_l2(S + (row0 + 16 * m) * kHeadSize + c);
    }
    pdl_wait();
    if (!ok) {
        if (tid == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }

    float4 s[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4 *>(S + (row0 + 16 * m) * kHeadSize + c));

    const size_t io = static_cast<size_t>(unit) * kHeadSize;
    const float4 a4 = load4<BF16>(p.in.a, io + c);
    const float4 w4 = load4<BF16>(p.in.w, io + c);
    const float4 b4 = load4<BF16>(p.in.b, io + c);
    const float4 k4 = load4<BF16>(p.in.k, io + c);
    const float4 r4 = load4<BF16>(p.in.r, io + c);
    float vv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) vv[m] = load1<BF16>(p.in.v, io + row0 + 16 * m);

    // delta read on the old state: h_i = sum_j S_ij a_j
    float hs[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) hs[m] = dot4(s[m], a4);
    row_sums4(hs, tid & 31);

    // decay, delta write, kv write; then the readout on the new state
    float os[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        s[m].x = fmaf(s[m].x, w4.x, fmaf(hs[m], b4.x, vv[m] * k4.x));
        s[m].y = fmaf(s[m].y, w4.y, fmaf(hs[m], b4.y, vv[m] * k4.y));
        s[m].z = fmaf(s[m].z, w4.z, fmaf(hs[m], b4.z, vv[m] * k4.z));
        s[m].w = fmaf(s[m].w, w4.w, fmaf(hs[m], b4.w, vv[m] * k4.w));
        os[m] = dot4(s[m], r4);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
        __stcs(reinterpret_cast<float4 *>(S + (row0 + 16 * m) * kHeadSize + c), s[m]);
    const float ou = reduce_scatter4(os, tid & 15);  // row ((tid >> 2) & 3)'s readout
    if ((tid & 3) == 0) store_out(p.in.o, p.in.o_bf16, io + row0 + 16 * ((tid >> 2) & 3), ou);
}

// Decode over a pool whose states are stored in bf16 (half the bytes of the
// float32 kernel's traffic): the step is computed in float32 from the widened
// state and the new state is rounded to bf16 (nearest even) on the way back;
// the readout o = S' r is taken from the unrounded float32 S'.  One CTA of
// 512 / kBf16Rows threads advances one (batch row, head) unit: thread t holds
// key columns 8*(t%8)..+7 (16 bytes) of value rows t/8 + (64/kBf16Rows)*m,
// m < kBf16Rows, and issues all its loads first.  Every CTA load/store
// instruction covers contiguous memory, and a row's 64 columns sit in 8
// consecutive lanes, so both row reductions are 3-level xor shuffles.
constexpr int kBf16Rows = 4;  // value rows per thread (4: 128-thread CTAs, best measured of 2, 4, 8)
constexpr int kBf16Threads = 8 * kHeadSize / kBf16Rows;
constexpr int kBf16RowStep = kHeadSize / kBf16Rows;

template <bool BF16>
__global__ void __launch_bounds__(kBf16Threads) decode_bf16state_kernel(DecodeArgs p) {
    pdl_launch_dependents();
    const int H = p.lv.n_heads;
    const int unit = blockIdx.x;
    const int bi = unit / H;
    const int h = unit - bi * H;
    const int tid = threadIdx.x;
    const int c = (tid & 7) * 8;  // first key column held by this thread
    const int row0 = tid >> 3;    // value rows row0 + kBf16RowStep*m
    // the slot id and an L2 prefetch of the state rows before the wait, as in decode_kernel
    const int slot = __ldg(p.slot_ids + bi);
    const bool ok = slot >= 0 && slot < p.lv.n_slots;
    uint16_t *S = reinterpret_cast<uint16_t *>(p.lv.states) +
                  static_cast<size_t>(ok ? slot : 0) * p.lv.slot_stride + p.lv.layer_off +
                  static_cast<size_t>(h) * kHeadFloats;
    if (ok && unit < kFirstWaveCtas && (tid & 7) == 0) {  // one 128-byte row per prefetch
#pragma unroll
        for (int m = 0; m < kBf16Rows; ++m) prefetch_l2(S + (row0 + kBf16RowStep * m) * kHeadSize);
    }
    pdl_wait();
    if (!ok) {
        if (tid == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }

    uint4 raw[kBf16Rows];
#pragma unroll
    for (int m = 0; m < kBf16Rows; ++m)
        raw[m] = __ldcs(reinterpret_cast<const uint4 *>(S + (row0 + kBf16RowStep * m) * kHeadSize + c));

    const size_t io = static_cast<size_t>(unit) * kHeadSize;
    float a8[8], w8[8], b8[8], k8[8], r8[8];
    load8<BF16>(p.in.a, io + c, a8);
    load8<BF16>(p.in.w, io + c, w8);
    load8<BF16>(p.in.b, io + c, b8);
    load8<BF16>(p.in.k, io + c, k8);
    load8<BF16>(p.in.r, io + c, r8);

    float hs[kBf16Rows], vv[kBf16Rows];
#pragma unroll
    for (int m = 0; m < kBf16Rows; ++m) {  // delta read on the old state: h_i = sum_j S_ij a_j
        vv[m] = load1<BF16>(p.in.v, io + row0 + kBf16RowStep * m);
        const uint32_t q[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(bf16_lo(q[e]), a8[2 * e], acc);
            acc = fmaf(bf16_hi(q[e]), a8[2 * e + 1], acc);
        }
        hs[m] = acc;
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1)
#pragma unroll
        for (int m = 0; m < kBf16Rows; ++m) hs[m] += __shfl_xor_sync(0xffffffffu, hs[m], off);

    // decay, delta write, kv write; the readout on the unrounded new state
    float os[kBf16Rows];
#pragma unroll
    for (int m = 0; m < kBf16Rows; ++m) {
        const uint32_t q[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
        uint32_t outw[4];
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = fmaf(bf16_lo(q[e]), w8[2 * e], fmaf(hs[m], b8[2 * e], vv[m] * k8[2 * e]));
            const float x1 =
                fmaf(bf16_hi(q[e]), w8[2 * e + 1], fmaf(hs[m], b8[2 * e + 1], vv[m] * k8[2 * e + 1]));
            acc = fmaf(x0, r8[2 * e], acc);
            acc = fmaf(x1, r8[2 * e + 1], acc);
            outw[e] = pack_bf16_rn(x0, x1);
        }
        os[m] = acc;
        __stcs(reinterpret_cast<uint4 *>(S + (row0 + kBf16RowStep * m) * kHeadSize + c),
               make_uint4(outw[0], outw[1], outw[2], outw[3]));
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1)
#pragma unroll
        for (int m = 0; m < kBf16Rows; ++m) os[m] += __shfl_xor_sync(0xffffffffu, os[m], off);
    if ((tid & 7) == 0) {
#pragma unroll
        for (int m = 0; m < kBf16Rows; ++m) store_out(p.in.o, p.in.o_bf16, io + row0 + kBf16RowStep * m, os[m]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s, int *launches) {
    const long long units = static_cast<long long>(a.n) * a.lv.n_heads;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(units));
    cudaError_t e;
    if (a.state_bf16)
        e = launch_pdl(a.in.bf16 ? decode_bf16state_kernel<true> : decode_bf16state_kernel<false>, grid,
                       dim3(kBf16Threads), 0, s, a);
    else
        e = launch_pdl(a.in.bf16 ? decode_kernel<true> : decode_kernel<false>, grid, dim3(256), 0, s, a);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace wkv7
