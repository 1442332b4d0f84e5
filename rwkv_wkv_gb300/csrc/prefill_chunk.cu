// Chunked WKV-7 prefill on the tcgen05 tensor cores (sm_103a).
//
// The recurrence (RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta
// Rule)"), per head with S[i][j] (i value, j key):
//     h_t = S a_t;  S <- S diag(w_t) + h_t b_t^T + v_t k_t^T;  o_t = S r_t.
// Over a chunk of L = 64 tokens from start state S0, with the relative decay
// D(s,t] = prod_{s<u<=t} w_u (per key channel), unrolling gives
//     H (I - Mab) = S0 A0^T + V Mak          (H = [h_1..h_L], V = [v_1..v_L])
// with Mab[s][t] = <b_s D(s,t-1], a_t>, Mak likewise with k (s < t), so with
// the unit-triangular inverse T = (I - Mab)^-1 and Z = T [Bhat | Qb]:
//     S_L = S0 Phi + Psi,     Phi = diag(D(0,L]) + A0^T Z_B,   Psi = V Y_B
//     O   = S0 R' + O0,       R'  = R0^T + A0^T Z_Q,           O0  = V Y_Q
//     Y   = Mak Z + [Khat | Qk]
// where A0[t] = a_t D(0,t-1], R0[t] = r_t D(0,t], Bhat[s] = b_s D(s,L],
// Khat[s] = k_s D(s,L], Qb[s][t] = <b_s D(s,t], r_t> and Qk likewise (s <= t).
// Everything except the final "S0 [R' | Phi]" product is independent of S0.
//
// One CTA (4 warps) owns one (sequence, head) and walks its chunks in order,
// anchored at the sequence's first token; the last chunk is padded with
// identity tokens (w = 1, other inputs 0).  Per chunk:
//   E   TMA-loaded bf16 inputs -> log2-decay prefix sums (one warp per 16
//       tokens, two channels per lane) -> scaled bf16 operands in 128-byte
//       swizzled K-major tiles.  Decays inside the Gram products are taken
//       relative to the chunk midpoint (token 31), so no factor exceeds
//       2^(half-chunk decay); factors that meet S0 are relative to the start.
//   G1  [Bbar;Kbar] x Am^T  -> Mab, Mak rows        (M=128, N=64,  K=64)
//   G1' [Am;Rm] x [Bbar;Kbar]^T -> Qb^T, Qk^T rows  (M=128, N=128, K=64)
//   T   (I - Mab)^-1 in float32 on the CUDA cores (16x16 blocked substitution)
//   G2  [Bhat^T; Qb^T] x T^T -> Z^T                  (M=128, N=64)
//   G34 Z^T x [A0^T; Mak]^T -> Phi'^T, R''^T, Y'^T   (M=128, N=128)
//   G5  [Y_Q^T; Y_B^T] x V -> O0^T, Psi^T; then += [R'^T; Phi^T] x S0^T with
//       S0 split into bf16 hi + lo (two MMAs)        (M=128, N=64)
// Accumulators live in tensor memory (256 columns); the float32 state leaves
// the accumulator each chunk, is written back as the next chunk's bf16 hi/lo
// operand pair and, after the last chunk, to the slot in float32.
// All waits are bounded; a timeout flags WKV7_DEV_WAIT_TIMEOUT and the CTA
// releases its tensor memory and exits.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "sm100_ptx.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

using namespace sm100;

constexpr int kL = 64;
constexpr int kThreads = 128;
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz
constexpr float kMaxLog2Range = 120.0f;           // |G - Gm| limit (float exponent range)
constexpr int kMS = 68;                           // float stride of the 64x64 fp32 scratch

// Shared-memory map (bytes from a 1024-aligned base).
constexpr uint32_t kTile64 = 8192;    // 64 rows x 128 B (bf16, K = 64)
constexpr uint32_t kTile128 = 16384;  // 128 rows
constexpr uint32_t OFF_IN = 0;        // six TMA tiles: r, w, k, v, a, b (plain [t][j] bf16)
constexpr uint32_t OFF_R1 = OFF_IN + 6 * kTile64;   // G1A | G1B, later OPZ, later OPY | OPA2
constexpr uint32_t OFF_G1A = OFF_R1;
constexpr uint32_t OFF_G1B = OFF_R1 + kTile128;
constexpr uint32_t OFF_OPZ = OFF_R1;
constexpr uint32_t OFF_OPY = OFF_R1;
constexpr uint32_t OFF_OPA2 = OFF_R1 + kTile128;
constexpr uint32_t OFF_G2A = OFF_R1 + 2 * kTile128;  // [Bhat^T; Qb^T]
constexpr uint32_t OFF_G2B = OFF_G2A + kTile128;     // T (rows s, K = t)
constexpr uint32_t OFF_G34B = OFF_G2B + kTile64;     // [A0^T; Mak]
constexpr uint32_t OFF_V = OFF_G34B + kTile128;      // V^T (rows i, K = s)
constexpr uint32_t OFF_KHT = OFF_V + kTile64;        // Khat^T (rows j, K = s)
constexpr uint32_t OFF_R0 = OFF_KHT + kTile64;       // R0 (rows t, K = j)
constexpr uint32_t OFF_SHI = OFF_R0 + kTile64;       // S0 hi (rows i, K = j)
constexpr uint32_t OFF_SLO = OFF_SHI + kTile64;      // S0 lo
constexpr uint32_t OFF_MT = OFF_SLO + kTile64;       // Mab fp32 [64][kMS]; lower blocks: temps
constexpr uint32_t OFF_TT = OFF_MT + 64 * kMS * 4;   // T fp32 [64][kMS]
constexpr uint32_t OFF_TOT = OFF_TT + 64 * kMS * 4;  // per-warp log2-decay totals [4][64]
constexpr uint32_t OFF_GAM = OFF_TOT + 4 * 64 * 4;   // D(0,L] per channel [64]
constexpr uint32_t OFF_BAR = OFF_GAM + 64 * 4;       // two mbarriers
constexpr uint32_t OFF_HOLD = OFF_BAR + 16;          // tensor-memory base
constexpr uint32_t OFF_FLAG = OFF_HOLD + 4;          // abort flag
constexpr uint32_t kSmemUsed = OFF_FLAG + 4;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;    // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
constexpr uint32_t kTmemCols = 256;

enum { IN_R = 0, IN_W = 1, IN_K = 2, IN_V = 3, IN_A = 4, IN_B = 5 };

struct InputMaps {
    CUtensorMap m[6];  // r, w, k, v, a, b
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ float bf16_to_f(uint16_t u) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// Write 32 floats as bf16 into columns col0..col0+31 of `row` of a swizzled tile.
__device__ __forceinline__ void store_row32(uint8_t *tile, int row, int col0, const float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
        u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
        u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
        u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_off(row, col0 + 8 * q)) = u;
    }
}

// Read 32 bf16 of `row` (columns col0..) of a swizzled tile as floats.
__device__ __forceinline__ void load_row32(const uint8_t *tile, int row, int col0, float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u = *reinterpret_cast<const uint4 *>(tile + sw128_off(row, col0 + 8 * q));
        v[8 * q + 0] = bf16_lo(u.x); v[8 * q + 1] = bf16_hi(u.x);
        v[8 * q + 2] = bf16_lo(u.y); v[8 * q + 3] = bf16_hi(u.y);
        v[8 * q + 4] = bf16_lo(u.z); v[8 * q + 5] = bf16_hi(u.z);
        v[8 * q + 6] = bf16_lo(u.w); v[8 * q + 7] = bf16_hi(u.w);
    }
}

// C (2x4 micro-tile at rows r0, r0+1, cols c0..c0+3) += A[rows][k] * B[k][cols]
// over k = 0..15, A and B 16x16 blocks of kMS-strided float matrices.
__device__ __forceinline__ void micro_2x4(const float *A, const float *B, int r0, int c0,
                                          float (&acc)[2][4]) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float a0 = A[r0 * kMS + kk];
        const float a1 = A[(r0 + 1) * kMS + kk];
        const float4 b = *reinterpret_cast<const float4 *>(B + kk * kMS + c0);
        acc[0][0] = fmaf(a0, b.x, acc[0][0]); acc[0][1] = fmaf(a0, b.y, acc[0][1]);
        acc[0][2] = fmaf(a0, b.z, acc[0][2]); acc[0][3] = fmaf(a0, b.w, acc[0][3]);
        acc[1][0] = fmaf(a1, b.x, acc[1][0]); acc[1][1] = fmaf(a1, b.y, acc[1][1]);
        acc[1][2] = fmaf(a1, b.z, acc[1][2]); acc[1][3] = fmaf(a1, b.w, acc[1][3]);
    }
}

// T = (I - M)^-1 for the strictly upper triangular 64x64 M in MT (fp32),
// result in TT (upper triangle and 16x16 diagonal blocks), blocked by 16:
// diagonal blocks by substitution, then T_pq = T_pp sum_{p<u<=q} M_pu T_uq
// level by level (q - p = 1, 2, 3).  The lower 16x16 blocks of MT hold the
// sums.  All 128 threads take part; ends with the block synchronised.
__device__ __forceinline__ void invert_unit_upper(float *MT, float *TT, int tid) {
    if (tid < 64) {
        const int p = tid >> 4, c = tid & 15;
        const float *M = MT + (16 * p) * kMS + 16 * p;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 14; r >= 0; --r) {
            if (r < c) {
                float acc = 0.f;
#pragma unroll
                for (int u = r + 1; u < 16; ++u) acc = fmaf(M[r * kMS + u], x[u], acc);
                x[r] = acc;
            }
        }
        float *Tb = TT + (16 * p) * kMS + 16 * p;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * kMS + c] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d <= 3; ++d) {
        const int nblk = 4 - d;  // blocks (p, p+d), p = 0..nblk-1
        const int mt = tid & 31, blk = tid >> 5;
        const int r0 = 2 * (mt >> 2), c0 = 4 * (mt & 3);
        if (blk < nblk) {  // X_pq = sum_{u=p+1..q} M_pu T_uq -> lower block (q, p) of MT
            const int p = blk, q = blk + d;
            float acc[2][4] = {};
            for (int u = p + 1; u <= q; ++u)
                micro_2x4(MT + (16 * p) * kMS + 16 * u, TT + (16 * u) * kMS + 16 * q, r0, c0, acc);
            float *X = MT + (16 * q) * kMS + 16 * p;
#pragma unroll
            for (int i = 0; i < 2; ++i)
                *reinterpret_cast<float4 *>(X + (r0 + i) * kMS + c0) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        __syncthreads();
        if (blk < nblk) {  // T_pq = T_pp X_pq
            const int p = blk, q = blk + d;
            float acc[2][4] = {};
            micro_2x4(TT + (16 * p) * kMS + 16 * p, MT + (16 * q) * kMS + 16 * p, r0, c0, acc);
            float *Tq = TT + (16 * p) * kMS + 16 * q;
#pragma unroll
            for (int i = 0; i < 2; ++i)
                *reinterpret_cast<float4 *>(Tq + (r0 + i) * kMS + c0) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        __syncthreads();
    }
}

// All threads wait on the barrier; returns false (uniformly) if any gave up.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int *flag) {
    if (!mbar_wait_bounded(bar, parity, kWaitCycles)) *flag = 1;
    __syncthreads();
    return *flag == 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunk_kernel(const PrefillArgs p, const __grid_constant__ InputMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    const int seq = blockIdx.x;
    const int h = blockIdx.y;
    const int H = p.lv.n_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int slot = __ldg(p.slot_ids + seq);
    const int t0 = __ldg(p.cu_seqlens + seq);
    const int t1 = __ldg(p.cu_seqlens + seq + 1);
    if (slot < 0 || slot >= p.lv.n_slots) {
        if (tid == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }
    if (t0 < 0 || t1 < t0 || t1 > p.total_tokens || t1 - t0 > p.max_seqlen) {
        if (tid == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SEQLENS);
        return;
    }
    const int len = t1 - t0;
    if (len == 0) return;

    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t bar_tma = smem_addr(base + OFF_BAR);
    const uint32_t bar_mma = bar_tma + 8;
    uint32_t *holder = reinterpret_cast<uint32_t *>(base + OFF_HOLD);
    volatile int *flag = reinterpret_cast<volatile int *>(base + OFF_FLAG);
    float *MT = reinterpret_cast<float *>(base + OFF_MT);
    float *TT = reinterpret_cast<float *>(base + OFF_TT);
    float *tot = reinterpret_cast<float *>(base + OFF_TOT);
    float *gam = reinterpret_cast<float *>(base + OFF_GAM);
    const uint8_t *in = base + OFF_IN;

    if (warp == 0) tmem_alloc(smem_addr(holder), kTmemCols);
    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *flag = 0;
#pragma unroll
        for (int x = 0; x < 6; ++x) prefetch_tensormap(&maps.m[x]);
    }

    float *S = p.lv.states + static_cast<size_t>(slot) * p.lv.slot_stride + p.lv.layer_off +
               static_cast<size_t>(h) * kHeadFloats;
    {  // start state -> bf16 hi/lo operand tiles (rows i, K = j)
        const int i = tid >> 1, c0 = 32 * (tid & 1);
        float hi[32], lo[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float4 x = *reinterpret_cast<const float4 *>(S + i * kHeadSize + c0 + 4 * q);
            float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                hi[4 * q + e] = __bfloat162float(__float2bfloat16_rn(xs[e]));
                lo[4 * q + e] = xs[e] - hi[4 * q + e];
            }
        }
        store_row32(base + OFF_SHI, i, c0, hi);
        store_row32(base + OFF_SLO, i, c0, lo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;

    const int n_chunks = (len + kL - 1) / kL;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_tma, 6 * kTile64);
#pragma unroll
        for (int x = 0; x < 6; ++x)
            tma_load_3d(smem_addr(base + OFF_IN + x * kTile64), &maps.m[x], 0, h, t0, bar_tma);
    }
    uint32_t ph_tma = 0, ph_mma = 0;
    bool range_bad = false;

    for (int c = 0; c < n_chunks; ++c) {
        const int tc0 = t0 + c * kL;
        const int Lc = min(kL, t1 - tc0);
        const bool last = (c + 1 == n_chunks);
        if (!wait_all(bar_tma, ph_tma, flag)) break;
        ph_tma ^= 1;

        // ---------------------------------------------------------- E phase
        {
            const int tb = 16 * warp;  // this warp's 16 tokens; lane: channels 2l, 2l+1
            const int ch = 2 * lane;
            auto ld2 = [&](int x, int t) -> float2 {
                const uint32_t u = *reinterpret_cast<const uint32_t *>(in + x * kTile64 + t * 128 + 4 * lane);
                return make_float2(bf16_lo(u), bf16_hi(u));
            };
            float pre0[16], pre1[16];
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = tb + i;
                if (t < Lc) {
                    const float2 wv = ld2(IN_W, t);
                    s0 += __log2f(wv.x);
                    s1 += __log2f(wv.y);
                }
                pre0[i] = s0;
                pre1[i] = s1;
            }
            tot[warp * 64 + ch] = s0;
            tot[warp * 64 + ch + 1] = s1;
            __syncthreads();
            float off0 = 0.f, off1 = 0.f;
            for (int w2 = 0; w2 < warp; ++w2) {
                off0 += tot[w2 * 64 + ch];
                off1 += tot[w2 * 64 + ch + 1];
            }
            const float Gm0 = tot[ch] + tot[64 + ch], Gm1 = tot[ch + 1] + tot[64 + ch + 1];
            const float G630 = Gm0 + tot[128 + ch] + tot[192 + ch];
            const float G631 = Gm1 + tot[128 + ch + 1] + tot[192 + ch + 1];
            if (warp == 0) {
                gam[ch] = exp2f(G630);
                gam[ch + 1] = exp2f(G631);
            }
            if (!(fabsf(off0 - Gm0) <= kMaxLog2Range && fabsf(off1 - Gm1) <= kMaxLog2Range))
                range_bad = true;  // G[tb-1] (G[-1] = 0 for the first warp)
            const float EL0 = exp2f(G630 - Gm0), EL1 = exp2f(G631 - Gm1);
            float ep0 = exp2f(off0 - Gm0), ep1 = exp2f(off1 - Gm1);  // e_prev at i = 0
            float dp0 = exp2f(off0), dp1 = exp2f(off1);              // d_prev at i = 0
            uint32_t cb[4][2][4];  // CT operands: [Bhat, Khat, A0, V][channel][token pair]
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = tb + i;
                const bool valid = t < Lc;
                const float G0 = off0 + pre0[i], G1 = off1 + pre1[i];
                if (valid && !(fabsf(G0 - Gm0) <= kMaxLog2Range && fabsf(G1 - Gm1) <= kMaxLog2Range))
                    range_bad = true;
                const float ec0 = exp2f(G0 - Gm0), ec1 = exp2f(G1 - Gm1);
                const float iv0 = exp2f(Gm0 - G0), iv1 = exp2f(Gm1 - G1);
                const float dc0 = exp2f(G0), dc1 = exp2f(G1);
                const float dl0 = EL0 * iv0, dl1 = EL1 * iv1;
                float2 a = make_float2(0.f, 0.f), b = a, k = a, r = a, v = a;
                if (valid) {
                    a = ld2(IN_A, t); b = ld2(IN_B, t); k = ld2(IN_K, t);
                    r = ld2(IN_R, t); v = ld2(IN_V, t);
                }
                uint8_t *g1a = base + OFF_G1A, *g1b = base + OFF_G1B;
                *reinterpret_cast<uint32_t *>(g1a + sw128_off(t, ch)) = pack_bf16(b.x * iv0, b.y * iv1);
                *reinterpret_cast<uint32_t *>(g1a + sw128_off(64 + t, ch)) = pack_bf16(k.x * iv0, k.y * iv1);
                *reinterpret_cast<uint32_t *>(g1b + sw128_off(t, ch)) = pack_bf16(a.x * ep0, a.y * ep1);
                *reinterpret_cast<uint32_t *>(g1b + sw128_off(64 + t, ch)) = pack_bf16(r.x * ec0, r.y * ec1);
                *reinterpret_cast<uint32_t *>(base + OFF_R0 + sw128_off(t, ch)) = pack_bf16(r.x * dc0, r.y * dc1);
                // channel-major operands, two tokens per 32-bit word
                const float cv[4][2] = {{b.x * dl0, b.y * dl1}, {k.x * dl0, k.y * dl1},
                                        {a.x * dp0, a.y * dp1}, {v.x, v.y}};
#pragma unroll
                for (int o = 0; o < 4; ++o)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t hv = __bfloat16_as_ushort(__float2bfloat16_rn(cv[o][e]));
                        if ((i & 1) == 0)
                            cb[o][e][(i >> 1) & 3] = hv;
                        else
                            cb[o][e][(i >> 1) & 3] |= hv << 16;
                    }
                if ((i & 7) == 7) {  // flush 8 tokens of each channel-major row
                    const int col = tb + (i & 8);
                    uint8_t *dst[4] = {base + OFF_G2A, base + OFF_KHT, base + OFF_G34B, base + OFF_V};
#pragma unroll
                    for (int o = 0; o < 4; ++o)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            *reinterpret_cast<uint4 *>(dst[o] + sw128_off(ch + e, col)) =
                                make_uint4(cb[o][e][0], cb[o][e][1], cb[o][e][2], cb[o][e][3]);
                }
                ep0 = ec0; ep1 = ec1;
                dp0 = dc0; dp1 = dc1;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && !last) {  // the input tiles are free: fetch the next chunk
            mbar_arrive_expect_tx(bar_tma, 6 * kTile64);
#pragma unroll
            for (int x = 0; x < 6; ++x)
                tma_load_3d(smem_addr(base + OFF_IN + x * kTile64), &maps.m[x], 0, h, tc0 + kL, bar_tma);
        }

        // --------------------------------------------------- G1 and G1'
        if (tid == 0) {
            tc_fence_after();
            umma_128xNx64(tmem + 0, smem_addr(base + OFF_G1A), smem_addr(base + OFF_G1B), 64, false);
            umma_128xNx64(tmem + 128, smem_addr(base + OFF_G1B), smem_addr(base + OFF_G1A), 128, false);
            umma_commit(bar_mma);
        }
        if (!wait_all(bar_mma, ph_mma, flag)) break;
        ph_mma ^= 1;
        tc_fence_after();
        {
            float v0[32], v1[32];
            const int row = 32 * warp + lane;  // TMEM lane
            tmem_ld32(tmem + lane_base + 0, v0);
            tmem_ld32(tmem + lane_base + 32, v1);
            tmem_ld_wait();
            if (warp < 2) {  // Mab row s: keep t > s, float32 for the inverse
                const int s = row;
                float *dst = MT + s * kMS;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 x = make_float4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]);
                    const int t = 4 * q;
                    x.x = (t + 0 > s) ? x.x : 0.f; x.y = (t + 1 > s) ? x.y : 0.f;
                    x.z = (t + 2 > s) ? x.z : 0.f; x.w = (t + 3 > s) ? x.w : 0.f;
                    *reinterpret_cast<float4 *>(dst + t) = x;
                    float4 y = make_float4(v1[4 * q], v1[4 * q + 1], v1[4 * q + 2], v1[4 * q + 3]);
                    const int u = 32 + 4 * q;
                    y.x = (u + 0 > s) ? y.x : 0.f; y.y = (u + 1 > s) ? y.y : 0.f;
                    y.z = (u + 2 > s) ? y.z : 0.f; y.w = (u + 3 > s) ? y.w : 0.f;
                    *reinterpret_cast<float4 *>(dst + u) = y;
                }
            } else {  // Mak row s' (keep s > s'), and Qb^T row t' (keep s <= t')
                const int s = row - 64;
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    v0[q] = (q > s) ? v0[q] : 0.f;
                    v1[q] = (32 + q > s) ? v1[q] : 0.f;
                }
                store_row32(base + OFF_G34B, 64 + s, 0, v0);
                store_row32(base + OFF_G34B, 64 + s, 32, v1);
                tmem_ld32(tmem + lane_base + 128, v0);
                tmem_ld32(tmem + lane_base + 160, v1);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    v0[q] = (q <= s) ? v0[q] : 0.f;
                    v1[q] = (32 + q <= s) ? v1[q] : 0.f;
                }
                store_row32(base + OFF_G2A, 64 + s, 0, v0);
                store_row32(base + OFF_G2A, 64 + s, 32, v1);
            }
        }
        tc_fence_before();
        __syncthreads();

        // ------------------------------------------------ T = (I - Mab)^-1
        invert_unit_upper(MT, TT, tid);
        {
            const int s = tid >> 1, c0 = 32 * (tid & 1);
            float x[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 y = *reinterpret_cast<const float4 *>(TT + s * kMS + c0 + 4 * q);
                x[4 * q] = y.x; x[4 * q + 1] = y.y; x[4 * q + 2] = y.z; x[4 * q + 3] = y.w;
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) x[q] = (c0 + q >= s) ? x[q] : 0.f;
            store_row32(base + OFF_G2B, s, c0, x);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ------------------------------------------------------------- G2
        if (tid == 0) {
            tc_fence_after();
            umma_128xNx64(tmem + 0, smem_addr(base + OFF_G2A), smem_addr(base + OFF_G2B), 64, false);
            umma_commit(bar_mma);
        }
        if (!wait_all(bar_mma, ph_mma, flag)) break;
        ph_mma ^= 1;
        tc_fence_after();
        {
            float v0[32], v1[32];
            tmem_ld32(tmem + lane_base + 0, v0);
            tmem_ld32(tmem + lane_base + 32, v1);
            tmem_ld_wait();
            store_row32(base + OFF_OPZ, 32 * warp + lane, 0, v0);
            store_row32(base + OFF_OPZ, 32 * warp + lane, 32, v1);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();

        // ------------------------------------------------------------ G34
        if (tid == 0) {
            tc_fence_after();
            umma_128xNx64(tmem + 0, smem_addr(base + OFF_OPZ), smem_addr(base + OFF_G34B), 128, false);
            umma_commit(bar_mma);
        }
        if (!wait_all(bar_mma, ph_mma, flag)) break;
        ph_mma ^= 1;
        tc_fence_after();
        {
            float v[32], add[32];
            if (warp < 2) {  // row j: Phi^T = Phi'^T + diag(gamma); Y_B^T = Y'^T + Khat^T
                const int j = 32 * warp + lane;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_base + 32 * half, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (32 * half + q == j) v[q] += gam[j];
                    store_row32(base + OFF_OPA2, 64 + j, 32 * half, v);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_base + 64 + 32 * half, v);
                    tmem_ld_wait();
                    load_row32(base + OFF_KHT, j, 32 * half, add);
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] += add[q];
                    store_row32(base + OFF_OPY, 64 + j, 32 * half, v);
                }
            } else {  // row t': R'^T = R''^T + R0; Y_Q^T = Y'^T + Qk^T
                const int tq = 32 * warp + lane - 64;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_base + 32 * half, v);
                    tmem_ld_wait();
                    load_row32(base + OFF_R0, tq, 32 * half, add);
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] += add[q];
                    store_row32(base + OFF_OPA2, tq, 32 * half, v);
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_base + 64 + 32 * half, v);
                    tmem_ld32(tmem + lane_base + 192 + 32 * half, add);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q)  // Qk^T[t'][s] is causal: s <= t'
                        v[q] += (32 * half + q <= tq) ? add[q] : 0.f;
                    store_row32(base + OFF_OPY, tq, 32 * half, v);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------- G5 and the state product S0 [R'|Phi]
        if (tid == 0) {
            tc_fence_after();
            umma_128xNx64(tmem + 128, smem_addr(base + OFF_OPY), smem_addr(base + OFF_V), 64, false);
            umma_128xNx64(tmem + 128, smem_addr(base + OFF_OPA2), smem_addr(base + OFF_SHI), 64, true);
            umma_128xNx64(tmem + 128, smem_addr(base + OFF_OPA2), smem_addr(base + OFF_SLO), 64, true);
            umma_commit(bar_mma);
        }
        if (!wait_all(bar_mma, ph_mma, flag)) break;
        ph_mma ^= 1;
        tc_fence_after();
        {
            float v0[32], v1[32];
            tmem_ld32(tmem + lane_base + 128, v0);
            tmem_ld32(tmem + lane_base + 160, v1);
            tmem_ld_wait();
            if (warp < 2) {  // O row t' -> o[tc0 + t'][h][:]
                const int tq = 32 * warp + lane;
                if (tq < Lc) {
                    float *dst = p.in.o + (static_cast<size_t>(tc0 + tq) * H + h) * kHeadSize;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        reinterpret_cast<float4 *>(dst)[q] =
                            make_float4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]);
                        reinterpret_cast<float4 *>(dst)[8 + q] =
                            make_float4(v1[4 * q], v1[4 * q + 1], v1[4 * q + 2], v1[4 * q + 3]);
                    }
                }
            } else {  // S_L column j (rows i) -> next chunk's hi/lo operand; last chunk -> slot
                const int j = 32 * warp + lane - 64;
                uint8_t *shi = base + OFF_SHI, *slo = base + OFF_SLO;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float x = i < 32 ? v0[i] : v1[i - 32];
                    const __nv_bfloat16 hb = __float2bfloat16_rn(x);
                    const float lo = x - __bfloat162float(hb);
                    *reinterpret_cast<__nv_bfloat16 *>(shi + sw128_off(i, j)) = hb;
                    *reinterpret_cast<__nv_bfloat16 *>(slo + sw128_off(i, j)) = __float2bfloat16_rn(lo);
                    if (last) S[i * kHeadSize + j] = x;
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
    }

    if (*flag) {  // a wait gave up: give in-flight copies a last chance, then leave
        if (tid == 0) flag_status(p.lv.status, WKV7_DEV_WAIT_TIMEOUT);
        mbar_wait_bounded(bar_tma, ph_tma, kWaitCycles);
        mbar_wait_bounded(bar_mma, ph_mma, kWaitCycles);
    }
    if (range_bad) flag_status(p.lv.status, WKV7_DEV_DECAY_RANGE);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// [total_tokens][H][64] bf16 viewed as a 3-D tensor (channel, head, token);
// one box = 64 tokens x 1 head x 64 channels, zero-filled past the end.
bool encode_input_map(CUtensorMap *map, const void *ptr, int H, int total_tokens) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadSize), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(total_tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadSize) * 2,
                             static_cast<cuuint64_t>(H) * kHeadSize * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadSize), 1, static_cast<cuuint32_t>(kL)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s, int *launches) {
    if (a.n_seqs <= 0) return cudaSuccess;
    if (a.total_tokens == 0)  // only empty sequences: nothing to load, only metadata to check
        return launch_prefill_sequential(a, s, launches);
    if (a.lv.n_heads > 65535) return cudaErrorInvalidValue;
    InputMaps maps;
    const void *src[6] = {a.in.r, a.in.w, a.in.k, a.in.v, a.in.a, a.in.b};
    for (int x = 0; x < 6; ++x)
        if (!encode_input_map(&maps.m[x], src[x], a.lv.n_heads, a.total_tokens))
            return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(a.n_seqs), static_cast<unsigned>(a.lv.n_heads));
    prefill_chunk_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, maps);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace wkv7
