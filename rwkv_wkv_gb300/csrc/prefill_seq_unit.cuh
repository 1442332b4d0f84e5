// The token-by-token WKV-7 recurrence of one (sequence, head) unit on 256
// threads, in float32: the body of the sequential prefill kernel, and the
// chunked kernel's path for a unit whose decay leaves the range of its chunk
// factorisation.
//
// RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)": per head and
// token, h = S a; S <- S diag(w) + h b^T + v k^T; o = S r.  Every value row i
// of S evolves on its own (h_i, S_i. and o_i only read row i), so 256 threads
// run one unit with 4 threads per row, each holding 16 key columns of that row
// in registers for the whole sequence.  Inputs are staged 16 tokens at a time
// in shared memory (key-side vectors are shared by all 64 rows); the two row
// reductions per token are 2-level xor shuffles.  With SBF16 (a bf16-state
// pool) the start state is read as bf16 and every stored state is rounded to
// bf16; at a checkpoint boundary the carry continues from the rounded
// checkpoint.
#pragma once

#include "device_common.cuh"
#include "wkv7_internal.h"

namespace wkv7 {

constexpr int kSeqTile = 16;  // tokens staged per pass
constexpr int kSeqQS = 20;    // floats per 16-column group (padded: conflict-free float4 reads)
constexpr int kSeqKeyInputs = 5;
// Shared-memory staging of one pass: the five key-side inputs and v.
struct SeqStage {
    float key[kSeqTile][kSeqKeyInputs][4][kSeqQS];
    float v[kSeqTile][kHeadSize];
};

// Barrier of the 256 threads that run a unit (named barrier 3: a kernel that
// calls prefill_seq_unit may have other warps that do not take part).
__device__ __forceinline__ void unit_barrier() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// Runs tokens t0..t1-1 of sequence `seq` (checkpoint ids from ck0) for head h
// from the state at element offset s_off, and stores the final state there.
// Called by threads 0-255 of the CTA; `st` is 16-byte aligned shared memory.
template <bool BF16, bool SBF16>
__device__ __forceinline__ void prefill_seq_unit(const PrefillArgs &p, int h, int t0, int t1, int ck0,
                                                 size_t s_off, SeqStage *st) {
    enum { kA = 0, kW = 1, kB = 2, kK = 3, kR = 4 };
    const int H = p.lv.n_heads;
    const int tid = threadIdx.x;
    const int i = tid >> 2;  // value row
    const int q = tid & 3;   // key columns 16q .. 16q+15

    float s[16];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 x = load_state4<SBF16>(p.lv.states, s_off + i * kHeadSize + 16 * q + 4 * m);
        s[4 * m + 0] = x.x; s[4 * m + 1] = x.y; s[4 * m + 2] = x.z; s[4 * m + 3] = x.w;
    }

    for (int tb = t0; tb < t1; tb += kSeqTile) {
        const int n_tok = t1 - tb < kSeqTile ? t1 - tb : kSeqTile;
        unit_barrier();  // previous tile fully consumed
        // stage: n_tok tokens x 6 inputs x 8 chunks of 8 channels
        for (int e = tid; e < n_tok * 48; e += 256) {
            const int tau = e / 48;
            const int rem = e - tau * 48;
            const int x = rem >> 3;
            const int cc = rem & 7;
            const size_t off = (static_cast<size_t>(tb + tau) * H + h) * kHeadSize + 8 * cc;
            float vals[8];
            const void *src = x == kA ? p.in.a : x == kW ? p.in.w : x == kB ? p.in.b
                            : x == kK ? p.in.k : x == kR ? p.in.r : p.in.v;
            load8<BF16>(src, off, vals);
            float *dst = (x == 5) ? &st->v[tau][8 * cc] : &st->key[tau][x][cc >> 1][(cc & 1) * 8];
            reinterpret_cast<float4 *>(dst)[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
            reinterpret_cast<float4 *>(dst)[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
        }
        unit_barrier();
        for (int tau = 0; tau < n_tok; ++tau) {
            const float4 *ka = reinterpret_cast<const float4 *>(st->key[tau][kA][q]);
            const float4 *kw = reinterpret_cast<const float4 *>(st->key[tau][kW][q]);
            const float4 *kbv = reinterpret_cast<const float4 *>(st->key[tau][kB][q]);
            const float4 *kk = reinterpret_cast<const float4 *>(st->key[tau][kK][q]);
            const float4 *kr = reinterpret_cast<const float4 *>(st->key[tau][kR][q]);
            // h_i = sum_j S_ij a_j on the old state
            float hp[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float4 a4 = ka[m];
                hp[m] = fmaf(s[4 * m], a4.x, fmaf(s[4 * m + 1], a4.y,
                        fmaf(s[4 * m + 2], a4.z, s[4 * m + 3] * a4.w)));
            }
            float hsum = (hp[0] + hp[1]) + (hp[2] + hp[3]);
            hsum += __shfl_xor_sync(0xffffffffu, hsum, 1);
            hsum += __shfl_xor_sync(0xffffffffu, hsum, 2);
            const float vi = st->v[tau][i];
            float op[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float4 w4 = kw[m], b4 = kbv[m], k4 = kk[m], r4 = kr[m];
                s[4 * m + 0] = fmaf(s[4 * m + 0], w4.x, fmaf(hsum, b4.x, vi * k4.x));
                s[4 * m + 1] = fmaf(s[4 * m + 1], w4.y, fmaf(hsum, b4.y, vi * k4.y));
                s[4 * m + 2] = fmaf(s[4 * m + 2], w4.z, fmaf(hsum, b4.z, vi * k4.z));
                s[4 * m + 3] = fmaf(s[4 * m + 3], w4.w, fmaf(hsum, b4.w, vi * k4.w));
                op[m] = fmaf(s[4 * m], r4.x, fmaf(s[4 * m + 1], r4.y,
                        fmaf(s[4 * m + 2], r4.z, s[4 * m + 3] * r4.w)));
            }
            float osum = (op[0] + op[1]) + (op[2] + op[3]);
            osum += __shfl_xor_sync(0xffffffffu, osum, 1);
            osum += __shfl_xor_sync(0xffffffffu, osum, 2);
            if (q == 0) store_out(p.in.o, p.in.o_bf16, (static_cast<size_t>(tb + tau) * H + h) * kHeadSize + i, osum);
        }
        const int done = tb + n_tok - t0;  // tokens of the sequence consumed so far
        if (p.ck.cu_ckpt && n_tok == kSeqTile && (done & 63) == 0) {  // a 64-token boundary
            const int id = __ldg(p.ck.ckpt_ids + ck0 + done / 64 - 1);
            if (id >= 0 && id < p.ck.n_snaps) {
                const size_t c_off = static_cast<size_t>(id) * p.lv.slot_stride + p.lv.layer_off +
                                     static_cast<size_t>(h) * kHeadFloats + i * kHeadSize + 16 * q;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    store_state4<SBF16>(p.ck.snaps, c_off + 4 * m,
                                        make_float4(s[4 * m], s[4 * m + 1], s[4 * m + 2], s[4 * m + 3]));
            } else if (tid == 0) {
                flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
            }
            if constexpr (SBF16) {  // carry on from the state as the checkpoint holds it
#pragma unroll
                for (int e = 0; e < 16; ++e) s[e] = round_bf16(s[e]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
        store_state4<SBF16>(p.lv.states, s_off + i * kHeadSize + 16 * q + 4 * m,
                            make_float4(s[4 * m], s[4 * m + 1], s[4 * m + 2], s[4 * m + 3]));
}

}  // namespace wkv7
