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
// One CTA (8 warps) owns one (sequence, head) and walks its chunks in order,
// anchored at the sequence's first token; the last chunk is padded with
// identity tokens (w = 1, other inputs 0).  Two CTAs share an SM (about 106 KB
// of shared memory and 256 tensor-memory columns each), so one CTA's MMA
// waits and load latencies are covered by the other's CUDA-core phases.
// Per chunk:
//   E   bf16 inputs, TMA-loaded into shared memory as soon as the previous
//       chunk's G2 completes (early enough that an L2 prefetch would only
//       compete with the loads for the TMA unit) -> log2-decay prefix sums (one
//       warp per 8 tokens, two channels per lane) -> operands scaled in packed
//       bf16 pairs, stored to 128-byte swizzled tiles.  Decays inside the Gram
//       products are taken relative to the chunk midpoint (token 31), so no
//       factor exceeds 2^(half-chunk decay); factors that meet S0 are relative
//       to the start.  A (sequence, head) with a chunk whose half-chunk decay
//       exceeds 2^120 in some channel (beyond the float range of these factors)
//       keeps its start state: after the chunk loop the same CTA runs it token
//       by token in float32 (prefill_seq_unit.cuh) and rewrites its outputs.
// Tensor-memory readbacks give warps w and w+4 the same 32 lanes (rows) and
// split the columns between them.
//   G1  [Bbar;Kbar] x Am^T -> Mab rows s              (M=128, N=64, K=64)
//   G1' [Am;Rm] x [Bbar;Kbar]^T -> rows t: Mak^T; rows t': Qb^T, Qk^T
//                                                    (M=128, N=128, K=64)
//   T   (I - Mab)^-1 by 16x16 blocks: the four diagonal blocks
//       T_ii = (I - M_ii)^-1 in fp32 by back substitution (two warps), then
//       N_ij = T_ii M_ij and the off-diagonal blocks from products of pairs of
//       those blocks (three steps of warp-level TF32 block products); T goes
//       to shared memory in bf16
//   G2  [Bhat^T; Qb^T] x T^T -> Z^T                  (M=128, N=64)
//   G34 Z^T (in tensor memory) x [A0 | Mak^T] (MN-major), accumulated onto
//       [diag(gamma) | Khat^T; R0 | Qk^T] (written into the accumulator during
//       the inverse by warps that are idle then) -> Phi^T, Y_B^T, R'^T, Y_Q^T
//                                                    (M=128, N=128)
//   G5  [Phi^T; R'^T] x (S0_hi + S0_lo)^T + [Y_B^T; Y_Q^T] x V -> [S_L^T; O^T],
//       both A operands in tensor memory, S0 split into bf16 hi + lo (B read
//       MN-major)                                    (M=128, N=64)
//       It runs while the warps build the next chunk's elementwise operands; its
//       completion is awaited just before the next G1 is issued (G1' writes the
//       columns of its A operands).
// One thread (lane 0 of warp 7) issues every copy and MMA.  A thread that issues
// tcgen05.mma is held for about the time the tensor core takes to accept them
// (some 60 cycles per K=16 instruction here), so the issuer is a warp whose work
// right after each issue has slack: not warps 0 and 1, which run the diagonal
// inverse after G1.
// The A operands of G34 and G5 go from the readback registers straight back
// into tensor memory as bf16; they never touch shared memory.
// Accumulators live in tensor memory (256 columns); the float32 state leaves
// the accumulator each chunk, is written back as the next chunk's bf16 hi/lo
// operand pair and, after the last chunk, to the slot (float32, or rounded to
// bf16 on a bf16-state pool; checkpoints likewise).  Each thread's 128-byte
// output row leaves in 32-byte stores when o allows them.
// All waits are bounded (by an argument: about 2 s, or about 50 ms under the
// test hook); a timeout flags WKV7_DEV_WAIT_TIMEOUT and the CTA releases its
// tensor memory and exits.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "prefill_seq_unit.cuh"
#include "sm100_ptx.cuh"
#include "wkv7_internal.h"

namespace wkv7 {
namespace {

using namespace sm100;

constexpr int kL = 64;
constexpr int kThreads = 256;  // 8 warps; two CTAs per SM
constexpr int kIssuer = 224;   // lane 0 of warp 7 issues the copies and MMAs
constexpr float kMaxLog2Range = 120.0f;           // |G - Gm| limit (float exponent range)
constexpr float kMinDecayRel = 0x1p-120f, kMaxDecayRel = 0x1p120f;  // the same limit on 2^(G - Gm)

// Shared-memory map.  Small items first (from the raw base), then the tiles
// from the next 1024-byte boundary.  Region R1 is reused through the chunk:
// G1A | G1B (E -> G1)  ->  fp32 blocks of the inverse | WT (T in bf16 for G2)
// ->  OPZ (-> G34)  ->  OPY | OPA2 (-> G5).
constexpr uint32_t kTile64 = 8192;    // 64 rows x 128 B (bf16, K = 64)
constexpr uint32_t kTile128 = 16384;  // 128 rows
constexpr uint32_t SOFF_TOT = 0;                    // per-warp log2-decay totals [8][64] fp32
constexpr uint32_t SOFF_GAM = SOFF_TOT + 8 * 64 * 4;  // D(0,L] per channel [64]
constexpr uint32_t SOFF_BAR = SOFF_GAM + 64 * 4;    // mbarrier: MMA completion
constexpr uint32_t SOFF_HOLD = SOFF_BAR + 24;       // tensor-memory base (after 3 mbarriers)
constexpr uint32_t SOFF_FLAG = SOFF_HOLD + 4;       // abort flag
constexpr uint32_t kSmallBytes = SOFF_FLAG + 4;
constexpr uint32_t OFF_R1 = 0;                      // tile offsets from the aligned base
constexpr uint32_t OFF_G1A = OFF_R1;
constexpr uint32_t OFF_G1B = OFF_R1 + kTile128;
// fp32 16x16 blocks of the inverse, 80-byte rows (conflict-free float4 rows):
// slots 0-3 M_ii then T_ii, 4-9 M_ij (i < j; later T_23, R_02, R_03, R_13),
// 10-15 N_ij = T_ii M_ij
constexpr int kSlotRow = 20;                          // floats per block row
constexpr uint32_t kSlotBytes = 16 * kSlotRow * 4;
constexpr int kSlotM = 4, kSlotN = 10;
constexpr int kSlotT23 = 0, kSlotR02 = 1, kSlotR03 = 2, kSlotR13 = 3;  // from kSlotM, after N
constexpr uint32_t OFF_WT = OFF_R1 + 3 * kTile64;   // T in bf16 (rows s, K = t)
static_assert(16 * kSlotBytes <= OFF_WT - OFF_R1, "inverse blocks overlap T");
constexpr uint32_t OFF_G2B = OFF_WT;
constexpr uint32_t OFF_G2A = OFF_R1 + 2 * kTile128;  // [Bhat^T; Qb^T]
constexpr uint32_t OFF_G34B = OFF_G2A + kTile128;    // B of G34, MN-major: [A0 | Mak^T] (rows u)
constexpr uint32_t OFF_A0 = OFF_G34B;                // A0 (rows u, 64 key channels j')
constexpr uint32_t OFF_MAKT = OFF_G34B + kTile64;    // Mak^T (rows u, 64 tokens s)
constexpr uint32_t OFF_V = OFF_G34B + kTile128;      // V^T (rows i, K = s)
constexpr uint32_t OFF_KHT = OFF_V + kTile64;        // Khat^T (rows j, K = s)
constexpr uint32_t OFF_R0 = OFF_KHT + kTile64;       // R0 (rows t, K = j)
constexpr uint32_t OFF_SHI = OFF_R0 + kTile64;       // S0^T hi (rows j, 64 values i; MN-major B)
constexpr uint32_t OFF_SLO = OFF_SHI + kTile64;      // S0^T lo
constexpr uint32_t kTileBytes = OFF_SLO + kTile64;
// Staging of the next chunk's six inputs ([64 tokens][64 channels] bf16, 8 KB
// each), TMA-loaded as soon as G2 completes: from then on the current chunk
// needs neither G2A nor region R1 (G34 and G5 take their A operands from
// tensor memory).  r, w go to G2A, k, v, a, b to R1.  The elementwise phase
// reads them all before its first barrier and writes these tiles only after
// it.
__host__ __device__ constexpr uint32_t stage_off(int x) {  // r, w, k, v, a, b
    return x < 2 ? OFF_G2A + x * kTile64 : OFF_R1 + (x - 2) * kTile64;
}
// One column of a bf16 state array (32 entries, element stride 64 from element
// `off`), each rounded to bf16 (nearest even).
__device__ __forceinline__ void store_state_column32_bf16(float *states, size_t off, const float *v) {
    __nv_bfloat16 *d = reinterpret_cast<__nv_bfloat16 *>(states) + off;
#pragma unroll
    for (int q = 0; q < 32; ++q) d[q * kHeadSize] = __float2bfloat16_rn(v[q]);
}

// Index of the strictly-upper 16x16 block (i, j), i < j < 4, in 0..5.
__device__ __forceinline__ int up_idx(int i, int j) { return i * (7 - i) / 2 + (j - i - 1); }
constexpr uint32_t kSmemBytes = kSmallBytes + 1024 + kTileBytes;  // + worst-case alignment
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(sizeof(SeqStage) <= kTileBytes, "the token-by-token path stages in the tiles");
constexpr uint32_t kTmemCols = 256;
// Tensor-memory columns: G1 64-127 and G1' 128-255 (Q_k^T at 192-255 until it
// is moved into G34's accumulator); G34's accumulator 0-127, loaded with its
// additive terms during the inverse; G2 128-191; Z^T, the bf16 A operand of
// G34, 192-223; the bf16 A operands of G5, [Phi^T; R'^T] 128-159 and Y^T
// 160-191; G5 0-63, read back while the next chunk's G1 and G1' run.
// A bf16 A operand in tensor memory holds row m in lane m with K elements 2c,
// 2c+1 packed in column c.
constexpr uint32_t kColG1 = 64, kColG1p = 128, kColG2 = 128, kColZA = 192, kColA2 = 128, kColYA = 160,
                   kColQk = 192;

struct InputMaps {
    CUtensorMap m[6];  // r, w, k, v, a, b
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Product of two bf16 pairs, each lane rounded once to bf16 (nearest even).
__device__ __forceinline__ uint32_t bmul2(uint32_t x, uint32_t y) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
    return d;
}


// Hardware base-2 exponential, logarithm and reciprocal (MUFU, a few ulp,
// denormals flushed); the decay factors they produce are rounded to bf16 right
// after.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Write 16 floats as bf16 into columns col0..col0+15 of `row` of a swizzled tile.
__device__ __forceinline__ void store_row16(uint8_t *tile, int row, int col0, const float *v) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint4 u;
        u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
        u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
        u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
        u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_off(row, col0 + 8 * q)) = u;
    }
}

// Read 16 bf16 of `row` (columns col0..) of a swizzled tile as floats.
__device__ __forceinline__ void load_row16(const uint8_t *tile, int row, int col0, float *v) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint4 u = *reinterpret_cast<const uint4 *>(tile + sw128_off(row, col0 + 8 * q));
        v[8 * q + 0] = bf16_lo(u.x); v[8 * q + 1] = bf16_hi(u.x);
        v[8 * q + 2] = bf16_lo(u.y); v[8 * q + 3] = bf16_hi(u.y);
        v[8 * q + 4] = bf16_lo(u.z); v[8 * q + 5] = bf16_hi(u.z);
        v[8 * q + 6] = bf16_lo(u.w); v[8 * q + 7] = bf16_hi(u.w);
    }
}

// ------------------------------------------- 16x16 fp32 block products (TF32)
// Warp-level D (+)= A B for 16x16 fp32 blocks in shared memory (row pitch
// kSlotRow floats), on the tensor cores with TF32 operands (truncated)
// and fp32 accumulation: two K=8 steps x two 8-column halves of
// mma.sync.m16n8k8.  Fragment layout of m16n8k8 (g = lane / 4, q = lane % 4):
// A a0 (g, q), a1 (g+8, q), a2 (g, q+4), a3 (g+8, q+4); B b0 (q, g), b1 (q+4, g);
// C/D c0 (g, 2q), c1 (g, 2q+1), c2 (g+8, 2q), c3 (g+8, 2q+1) -- per 8-column half.
// A TF32 operand: the float's own bits; the tensor core reads their upper 19 bits
// (truncation).  T leaves the inverse rounded to bf16 (8 bits) anyway, and a
// conversion instruction per operand element cost 3% of the kernel's time.
__device__ __forceinline__ uint32_t tf32_rn(float x) { return __float_as_uint(x); }

__device__ __forceinline__ void mma_tf32_m16n8k8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc[h] (8-column half h of the 16x16 result, C-fragment layout) += A B.
__device__ __forceinline__ void block_mma_acc(const float *A, const float *B, float (&acc)[2][4],
                                              int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint32_t a[4] = {tf32_rn(A[g * 20 + 8 * kk + q]), tf32_rn(A[(g + 8) * 20 + 8 * kk + q]),
                               tf32_rn(A[g * 20 + 8 * kk + q + 4]),
                               tf32_rn(A[(g + 8) * 20 + 8 * kk + q + 4])};
#pragma unroll
        for (int h = 0; h < 2; ++h)
            mma_tf32_m16n8k8(acc[h], a, tf32_rn(B[(8 * kk + q) * 20 + 8 * h + g]),
                             tf32_rn(B[(8 * kk + q + 4) * 20 + 8 * h + g]));
    }
}

// Load a 16x16 block into the C-fragment layout (or zero it).
__device__ __forceinline__ void block_frag_load(const float *C, float (&acc)[2][4], int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float2 x0 = *reinterpret_cast<const float2 *>(C + g * 20 + 8 * h + 2 * q);
        const float2 x1 = *reinterpret_cast<const float2 *>(C + (g + 8) * 20 + 8 * h + 2 * q);
        acc[h][0] = x0.x; acc[h][1] = x0.y; acc[h][2] = x1.x; acc[h][3] = x1.y;
    }
}

__device__ __forceinline__ void block_frag_store(float *D, const float (&acc)[2][4], int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        *reinterpret_cast<float2 *>(D + g * 20 + 8 * h + 2 * q) = make_float2(acc[h][0], acc[h][1]);
        *reinterpret_cast<float2 *>(D + (g + 8) * 20 + 8 * h + 2 * q) = make_float2(acc[h][2], acc[h][3]);
    }
}

// Longest-first order of the sequences (by chunk count, capped at 255; ties in
// index order), so that the CTAs of the longest sequences start first and the
// ragged tail of the grid is short.  The grid is (head, rank) with the rank
// split over y and z.
// Every CTA derives the same order from cu_seqlens; `work` is 1.1 KB of shared
// memory.  Returns the sequence of the given rank.  Up to 256 sequences, one
// thread per sequence counts those ordered before it (a few hundred cycles);
// beyond, a histogram of the keys and two CTA-wide scans.
constexpr int kMaxRankedSeqs = 4096;
constexpr unsigned kGridY = 65535;

__device__ __forceinline__ int chunk_key(const int *cu, int q) {
    const int n = (__ldg(cu + q + 1) - __ldg(cu + q) + kL - 1) / kL;
    return 255 - min(max(n, 0), 255);  // bin 0 holds the longest sequences
}

// Exclusive prefix sum over the CTA of one value per thread; `sums` holds 8 ints.
__device__ __forceinline__ int cta_exclusive_scan(int x, int *sums, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int y = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int z = __shfl_up_sync(0xffffffffu, y, d);
        if (lane >= d) y += z;
    }
    if (lane == 31) sums[warp] = y;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int t = sums[w];
        before += (w < warp) ? t : 0;
        total += t;
    }
    __syncthreads();  // sums may be reused
    return before + y - x;
}

__device__ __noinline__ int seq_of_rank(const int *cu, int n, int rank, int *work) {
    if (n == 1) return 0;
    int *hist = work, *sums = work + 256, *found = work + 264;
    const int tid = threadIdx.x;
    if (n <= kThreads) {  // one thread per sequence: its rank is the number ordered before it
        int *key = work;
        const int mine = tid < n ? chunk_key(cu, tid) : 0;
        if (tid < n) key[tid] = mine;
        __syncthreads();
        if (tid < n) {
            int r = 0;
            for (int q = 0; q < n; ++q) {
                const int kq = key[q];
                r += (kq < mine) | ((kq == mine) & (q < tid));
            }
            if (r == rank) found[0] = tid;
        }
        __syncthreads();
        const int seq = found[0];
        __syncthreads();  // the work area is reused by the caller
        return seq;
    }
    hist[tid] = 0;
    __syncthreads();
    for (int q = tid; q < n; q += kThreads) atomicAdd(&hist[chunk_key(cu, q)], 1);
    __syncthreads();
    int total;
    const int cnt = hist[tid];
    const int start = cta_exclusive_scan(cnt, sums, total);
    if (start <= rank && rank < start + cnt) { found[0] = tid; found[1] = rank - start; }
    __syncthreads();
    const int bin = found[0], want = found[1];
    const int per = (n + kThreads - 1) / kThreads;
    const int q0 = min(n, tid * per), q1 = min(n, q0 + per);
    int mine = 0;
    for (int q = q0; q < q1; ++q) mine += chunk_key(cu, q) == bin;
    const int before = cta_exclusive_scan(mine, sums, total);
    if (before <= want && want < before + mine) {
        int k = before;
        for (int q = q0; q < q1; ++q)
            if (chunk_key(cu, q) == bin) {
                if (k == want) found[2] = q;
                ++k;
            }
    }
    __syncthreads();
    const int seq = found[2];
    __syncthreads();  // the work area is reused by the caller
    return seq;
}

// Every thread waits on the MMA barrier itself.  A thread that gives up sets
// the CTA's abort flag; the flag is read (uniformly) after the phase's closing
// barrier, so a timed-out phase runs to that barrier on garbage and then the
// CTA leaves.
__device__ __forceinline__ bool mma_wait(uint32_t bar, uint32_t parity, volatile int *flag, long long limit) {
    if (mbar_wait_bounded(bar, parity, limit)) return true;
    *flag = 1;
    return false;
}

// The token-by-token route of a unit whose decay leaves the chunk
// factorisation's range; kept out of line so that the chunked path's register
// allocation and instruction stream do not carry it.
template <bool SBF16>
__device__ __noinline__ void prefill_unit_token_by_token(const PrefillArgs &p, int h, int t0, int t1, int ck0,
                                                         size_t s_off, SeqStage *st) {
    prefill_seq_unit<true, SBF16>(p, h, t0, t1, ck0, s_off, st);
}

// SBF16: the pool stores its states in bf16 (see the store paths of the readback);
// OBF16: o is written in bf16 (p.in.o_bf16).
template <bool SBF16, bool OBF16>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_chunk_kernel(const PrefillArgs p, const __grid_constant__ InputMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    pdl_prologue();
    const int H = p.lv.n_heads;
    const int h = blockIdx.x;
    const int rank = static_cast<int>(blockIdx.z * kGridY + blockIdx.y);
    if (rank >= p.n_seqs) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seq = p.n_seqs <= kMaxRankedSeqs
                        ? seq_of_rank(p.cu_seqlens, p.n_seqs, rank, reinterpret_cast<int *>(smem_raw))
                        : rank;

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
    int ck0 = 0;  // this sequence's first checkpoint id index
    if (p.ck.cu_ckpt) {
        ck0 = __ldg(p.ck.cu_ckpt + seq);
        if (ck0 < 0 || __ldg(p.ck.cu_ckpt + seq + 1) - ck0 != len / kL) {
            if (tid == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SEQLENS);
            return;
        }
    }
    if (len == 0) return;

    uint8_t *small = smem_raw;
    // Tiles from the next 1024-byte boundary; offsetting smem_raw (rather than
    // rounding an integer address) keeps the pointers in the shared address space,
    // so every tile access compiles to a shared-memory instruction.
    uint8_t *base = smem_raw + kSmallBytes + ((1024u - ((smem_addr(smem_raw) + kSmallBytes) & 1023u)) & 1023u);
    const uint32_t bar_mma = smem_addr(small + SOFF_BAR);
    uint32_t *holder = reinterpret_cast<uint32_t *>(small + SOFF_HOLD);
    volatile int *flag = reinterpret_cast<volatile int *>(small + SOFF_FLAG);
    float *tot = reinterpret_cast<float *>(small + SOFF_TOT);
    float *gam = reinterpret_cast<float *>(small + SOFF_GAM);
    auto blk = [base](int b) { return reinterpret_cast<float *>(base + OFF_R1 + b * kSlotBytes); };

    if (warp == 0) tmem_alloc(smem_addr(holder), kTmemCols);
    if (tid == kIssuer) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_mma + 8, 1);  // the input barrier
        mbar_init(bar_mma + 16, 1);  // the state product G5
        fence_mbar_init();
        *flag = 0;
#pragma unroll
        for (int x = 0; x < 6; ++x) prefetch_tensormap(&maps.m[x]);
    }

    // TMA loads of inputs x0..x1 (0..5 = r, w, k, v, a, b) of the chunk at token
    // tcn into their staging tiles, completing on the input barrier (whose
    // expected byte count, one chunk's six boxes, is set by the first call of
    // each phase).  Boxes past the last token are zero-filled; the elementwise
    // phase turns those rows into identity tokens.  Issued by the issuer thread.
    const uint32_t bar_in = bar_mma + 8;
    const uint32_t bar_g5 = bar_mma + 16;
    auto stage_inputs = [&](int x0, int x1, int tcn, bool first) {
        if (first) mbar_arrive_expect_tx(bar_in, 6 * kTile64);
        for (int x = x0; x <= x1; ++x)
            tma_load_3d(smem_addr(base + stage_off(x)), &maps.m[x], 0, h, tcn, bar_in);
    };
    // A load the issuer has issued and not yet seen land (on the input barrier's
    // phase in_parity), for the drain after a wait that gave up.  (The MMA
    // barrier needs no such record: every commit is followed by its wait before
    // the loop can stop, so the last commit's phase is the one before ph_mma.)
    bool in_flight = false;
    uint32_t in_parity = 0;
    if (tid == kIssuer && !p.test_skip_first_load) {
        stage_inputs(0, 5, t0, true);
        in_flight = true;
    }

    // element offset of this (slot, layer, head) state; elements are bf16 on a
    // bf16-state pool (read exactly here; stored states are rounded to bf16)
    const size_t s_off = static_cast<size_t>(slot) * p.lv.slot_stride + p.lv.layer_off +
                         static_cast<size_t>(h) * kHeadFloats;
    float *S = p.lv.states + s_off;  // float32 states only
    {  // start state -> bf16 hi/lo tiles of S^T (rows j = key, 64 value entries i per row):
       // the MN-major B operand of the state product
        const int j = tid & 63, i0 = 16 * (tid >> 6);
        float xs[16];  // all loads issued before any shared-memory store
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            if constexpr (SBF16)
                xs[q] = __uint_as_float(static_cast<uint32_t>(__ldcg(reinterpret_cast<const unsigned short *>(
                                            p.lv.states) + s_off + (i0 + q) * kHeadSize + j)) << 16);
            else
                xs[q] = __ldcg(S + (i0 + q) * kHeadSize + j);
        }
        uint32_t hw[8], lw[8];  // values i0 + 2e, i0 + 2e + 1: bf16 hi and the bf16 of the remainder
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            hw[e] = pack_bf16(xs[2 * e], xs[2 * e + 1]);
            lw[e] = pack_bf16(xs[2 * e] - bf16_lo(hw[e]), xs[2 * e + 1] - bf16_hi(hw[e]));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t off = sw128_off(j, i0 + 8 * h);
            *reinterpret_cast<uint4 *>(base + OFF_SHI + off) =
                make_uint4(hw[4 * h], hw[4 * h + 1], hw[4 * h + 2], hw[4 * h + 3]);
            *reinterpret_cast<uint4 *>(base + OFF_SLO + off) =
                make_uint4(lw[4 * h], lw[4 * h + 1], lw[4 * h + 2], lw[4 * h + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int row = 32 * (warp & 3) + lane;  // tensor-memory lane (accumulator row) of this thread
    const int cpart = 32 * (warp >> 2);      // this thread's 32-column part of each 64-column group

    const int n_chunks = (len + kL - 1) / kL;
    // Every output row starts a multiple of 128 bytes (64 for bf16 o) past o, which
    // the host checks is 16-byte aligned, so o's own alignment decides the store width.
    const bool o_v8 = (reinterpret_cast<uintptr_t>(p.in.o) & 31u) == 0;
    uint32_t ph_mma = 0, ph_in = 0, ph_g5 = 0;
    bool g5_pending = false;
    bool range_bad = false;  // a chunk's decay left the factorisation's range (this thread saw it)
    int prev_c = 0, prev_tc0 = 0, prev_Lc = 0;  // chunk whose state product awaits its readback

    // Readback of the state product [S_L^T; O^T] (tensor-memory columns 0-63): O rows to the output, S_L^T rows to the bf16 hi/lo
    // operand tiles of the next chunk, after the last chunk the float32 state to
    // the slot, and after a full chunk the float32 state to its checkpoint
    // snapshot when checkpoints are asked for.
    auto readback_state_product = [&](int occ, int otc0, int oLc, bool final) {
        float v[32];
        tmem_ld32(tmem + lane_base + cpart, v);
        tmem_ld_wait();
        if (row >= 64) {  // O row t' -> o[otc0 + t'][h][cpart ..]
            const int tq = row - 64;
            const size_t oi = (static_cast<size_t>(otc0 + tq) * H + h) * kHeadSize + cpart;
            if (tq < oLc && !OBF16) {  // 128 bytes per thread: 32-byte stores when o allows them
                float *dst = static_cast<float *>(p.in.o) + oi;
                if (o_v8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_global_v8(dst + 8 * q, v + 8 * q);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        reinterpret_cast<float4 *>(dst)[q] =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            } else if (OBF16 && tq < oLc) {  // bf16 o: 64 bytes per thread, rounded to nearest even
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                uint32_t *dst = reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(p.in.o) + oi);
                if (o_v8) {
                    st_global_v8_b32(dst, pk);
                    st_global_v8_b32(dst + 8, pk + 8);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<uint4 *>(dst)[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        } else {  // S_L^T row j (values i of this thread's part)
            const int j = row;
            const bool round_carry = SBF16 && p.ck.cu_ckpt && oLc == kL;
            if (p.ck.cu_ckpt && oLc == kL) {  // the state at token 64 (occ + 1) of the sequence
                const int id = __ldg(p.ck.ckpt_ids + ck0 + occ);
                if (id >= 0 && id < p.ck.n_snaps) {
                    if constexpr (SBF16) {
                        store_state_column32_bf16(p.ck.snaps,
                                                  static_cast<size_t>(id) * p.lv.slot_stride + p.lv.layer_off +
                                                      static_cast<size_t>(h) * kHeadFloats + cpart * kHeadSize + j,
                                                  v);
                    } else {
                        float *cp = p.ck.snaps + static_cast<size_t>(id) * p.lv.slot_stride + p.lv.layer_off +
                                    static_cast<size_t>(h) * kHeadFloats + cpart * kHeadSize + j;
#pragma unroll
                        for (int q = 0; q < 32; ++q) cp[q * kHeadSize] = v[q];
                    }
                } else if (j == 0) {
                    flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
                }
            }
            if (final) {  // column j of S, rows cpart..
                if constexpr (SBF16) {
                    store_state_column32_bf16(p.lv.states, s_off + cpart * kHeadSize + j, v);
                } else {
                    float *sp = S + cpart * kHeadSize + j;
#pragma unroll
                    for (int q = 0; q < 32; ++q) sp[q * kHeadSize] = v[q];
                }
            } else {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {  // 8 values: bf16 hi and the bf16 of the remainder
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x0 = v[8 * q8 + 2 * e], x1 = v[8 * q8 + 2 * e + 1];
                        hw[e] = pack_bf16(x0, x1);
                        // on a bf16-state pool a checkpointed state carries on as stored
                        lw[e] = round_carry ? 0u : pack_bf16(x0 - bf16_lo(hw[e]), x1 - bf16_hi(hw[e]));
                    }
                    const uint32_t off = sw128_off(j, cpart + 8 * q8);
                    *reinterpret_cast<uint4 *>(base + OFF_SHI + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(base + OFF_SLO + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
                fence_proxy_async_smem();  // the hi/lo tiles feed the next state product
            }
        }
    };

    // G34's additive terms, written into its accumulator (columns 0-127) before
    // it runs, so that G34 accumulates onto them: rows j (warps 4, 5) get
    // diag(gamma) and Khat^T, rows t' (warps 6, 7) R0 and the causal part of
    // Q_k^T (s <= t'), taken from G1'.
    auto preload_g34_rows_j = [&]() {
        const int j = row;
        const float gj = gam[j];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t r[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(16 * g + q == j ? gj : 0.f);
            tmem_st16(tmem + lane_base + 16 * g, r);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float add[16];
            uint32_t r[16];
            load_row16(base + OFF_KHT, j, 16 * g, add);
#pragma unroll
            for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(add[q]);
            tmem_st16(tmem + lane_base + 64 + 16 * g, r);
        }
        tmem_st_wait();
    };
    auto preload_g34_rows_t = [&]() {
        const int tq = row - 64;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float add[16];
            uint32_t r[16];
            load_row16(base + OFF_R0, tq, 16 * g, add);
#pragma unroll
            for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(add[q]);
            tmem_st16(tmem + lane_base + 16 * g, r);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float qk[32];
            tmem_ld32(tmem + lane_base + kColQk + 32 * hh, qk);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t r[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    r[q] = __float_as_uint(32 * hh + 16 * g + q <= tq ? qk[16 * g + q] : 0.f);
                tmem_st16(tmem + lane_base + 64 + 32 * hh + 16 * g, r);
            }
        }
        tmem_st_wait();
    };

    for (int c = 0; c < n_chunks; ++c) {
        const int tc0 = t0 + c * kL;
        const int Lc = min(kL, t1 - tc0);
        const bool last = (c + 1 == n_chunks);

        // ---------------------------------------------------------- E phase
        // E1 builds the Gram operands of G1 and G1'; E2 (below, while those MMAs
        // run) the remaining operands from the same registers.
        const int tb = 8 * warp;  // this warp's 8 tokens; lane: channels 2l, 2l+1
        const int ch = 2 * lane;
        const uint32_t xl = static_cast<uint32_t>(lane) >> 2;  // swizzled offset of (row tb + i, column ch):
        const uint32_t rowbase = 1024u * warp + 4u * (lane & 3);  // rowbase + i * 128 + ((xl ^ i) << 4)
        uint32_t in_r[8], in_w[8], in_k[8], in_v[8], in_a[8], in_b[8];
        float e0s, e1s, eGm0, eGm1, EL0, EL1;  // 2^(G_{tb-1} - Gm), 2^Gm, 2^(G_L - Gm) per channel
        {
            if (mma_wait(bar_in, ph_in, flag, p.wait_cycles) && tid == kIssuer) in_flight = false;  // inputs landed
            ph_in ^= 1;
            {
                auto st = [&](int x, int t) -> uint32_t {
                    return *reinterpret_cast<const uint32_t *>(base + stage_off(x) + t * 128 + 4 * lane);
                };
#pragma unroll
                for (int i = 0; i < 8; ++i) {  // tokens past Lc: identity (w = 1, the rest 0)
                    const int t = tb + i;
                    const bool valid = t < Lc;
                    in_r[i] = valid ? st(0, t) : 0u;
                    in_w[i] = valid ? st(1, t) : 0x3F803F80u;  // 1.0, 1.0
                    in_k[i] = valid ? st(2, t) : 0u;
                    in_v[i] = valid ? st(3, t) : 0u;
                    in_a[i] = valid ? st(4, t) : 0u;
                    in_b[i] = valid ? st(5, t) : 0u;
                }
            }
            float p0 = 1.f, p1 = 1.f;  // this warp's decay products
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                p0 *= bf16_lo(in_w[i]);
                p1 *= bf16_hi(in_w[i]);
            }
            const float s0 = lg2_approx(p0), s1 = lg2_approx(p1);  // this warp's log2-decay totals
            *reinterpret_cast<float2 *>(tot + warp * 64 + ch) = make_float2(s0, s1);
            __syncthreads();
            float G0 = 0.f, G1 = 0.f, Gm0 = 0.f, Gm1 = 0.f, G630 = 0.f, G631 = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < 8; ++w2) {
                const float2 x = *reinterpret_cast<const float2 *>(tot + w2 * 64 + ch);
                if (w2 < warp) { G0 += x.x; G1 += x.y; }
                if (w2 < 4) { Gm0 += x.x; Gm1 += x.y; }
                G630 += x.x; G631 += x.y;
            }
            if (warp == 0) *reinterpret_cast<float2 *>(gam + ch) = make_float2(ex2_approx(G630), ex2_approx(G631));
            if (!(fabsf(G0 - Gm0) <= kMaxLog2Range && fabsf(G1 - Gm1) <= kMaxLog2Range))
                range_bad = true;  // G[tb-1] (G[-1] = 0 for the first warp)
            EL0 = ex2_approx(G630 - Gm0);
            EL1 = ex2_approx(G631 - Gm1);
            // 2^Gm is a normal float whenever the range check passes (|Gm| <= 120), so
            // the decays from the chunk start are 2^(G - Gm) * 2^Gm.
            eGm0 = ex2_approx(Gm0);
            eGm1 = ex2_approx(Gm1);
            // e = 2^(G_t - Gm) runs as a product: e_t = e_{t-1} w_t (each e_t lies in
            // [2^-120, 2^120] when the range check passes, so nothing under- or overflows);
            // its reciprocal gives 2^(Gm - G_t).
            e0s = ex2_approx(G0 - Gm0);
            e1s = ex2_approx(G1 - Gm1);
            float e0 = e0s, e1 = e1s;
            uint32_t ep2 = pack_bf16(e0, e1);  // 2^(G_{t-1} - Gm)
            uint8_t *g1a = base + OFF_G1A, *g1b = base + OFF_G1B;
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                e0 *= bf16_lo(in_w[ii]);  // padding tokens have w = 1
                e1 *= bf16_hi(in_w[ii]);
                const uint32_t ec2 = pack_bf16(e0, e1);                              // 2^(G_t - Gm)
                const uint32_t iv2 = pack_bf16(rcp_approx(e0), rcp_approx(e1));    // 2^(Gm - G_t)
                const uint32_t off = rowbase + ii * 128 + ((xl ^ ii) << 4);
                *reinterpret_cast<uint32_t *>(g1a + off) = bmul2(in_b[ii], iv2);
                *reinterpret_cast<uint32_t *>(g1a + 8192 + off) = bmul2(in_k[ii], iv2);
                *reinterpret_cast<uint32_t *>(g1b + off) = bmul2(in_a[ii], ep2);
                *reinterpret_cast<uint32_t *>(g1b + 8192 + off) = bmul2(in_r[ii], ec2);
                ep2 = ec2;
            }
            // With every w in (0, 1] the factors fall from 2^(G_{tb-1} - Gm) (checked above)
            // to the last token's: that one decides whether all lie within 2^+-120 (a NaN or
            // an overflow anywhere reaches it too).
            if (!(e0 >= kMinDecayRel && e0 <= kMaxDecayRel && e1 >= kMinDecayRel && e1 <= kMaxDecayRel))
                range_bad = true;
        }
        fence_proxy_async_smem();
        __syncthreads();

        // --------------------------------------------------- G1 and G1'
        if (g5_pending) {  // the previous chunk's state product ran during the elementwise phase;
                           // G1' writes the tensor-memory columns of its A operands
            mma_wait(bar_g5, ph_g5, flag, p.wait_cycles);
            ph_g5 ^= 1;
            g5_pending = false;
            tc_fence_after();
        }
        if (tid == kIssuer) {
            tc_fence_after();
            umma_128xNx64(tmem + kColG1, smem_addr(base + OFF_G1A), smem_addr(base + OFF_G1B), 64, false);
            umma_128xNx64(tmem + kColG1p, smem_addr(base + OFF_G1B), smem_addr(base + OFF_G1A), 128, false);
            umma_commit(bar_mma);
        }
        {  // E2, while G1 and G1' run: R0, A0 (row-major), Bhat^T, Khat^T, V^T (channel-major)
            float e0 = e0s, e1 = e1s;
            uint32_t dp2 = pack_bf16(e0 * eGm0, e1 * eGm1);  // D(0, t-1]
            uint8_t *r0t = base + OFF_R0;
            uint32_t cb[3][2][4];  // channel-major operands [Bhat, Khat, V][channel ch + (e ^ sw)][token pair]
            uint32_t prv[3];
            // lanes 4-7 of each group of 8 take channel ch + 1 first, so that the eight
            // 16-byte stores of a quarter-warp fall in eight different bank groups
            const uint32_t sw = (static_cast<uint32_t>(lane) >> 2) & 1u;
            const uint32_t sel0 = sw ? 0x7632u : 0x5410u, sel1 = sel0 ^ 0x2222u;
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                e0 *= bf16_lo(in_w[ii]);
                e1 *= bf16_hi(in_w[ii]);
                const uint32_t dc2 = pack_bf16(e0 * eGm0, e1 * eGm1);                           // D(0, t]
                const uint32_t dl2 = pack_bf16(EL0 * rcp_approx(e0), EL1 * rcp_approx(e1));  // D(t, L]
                const uint32_t off = rowbase + ii * 128 + ((xl ^ ii) << 4);
                *reinterpret_cast<uint32_t *>(r0t + off) = bmul2(in_r[ii], dc2);
                *reinterpret_cast<uint32_t *>(base + OFF_A0 + off) = bmul2(in_a[ii], dp2);
                const uint32_t cur[3] = {bmul2(in_b[ii], dl2), bmul2(in_k[ii], dl2), in_v[ii]};
#pragma unroll
                for (int o = 0; o < 3; ++o) {
                    if ((ii & 1) == 0) {
                        prv[o] = cur[o];
                    } else {  // tokens (ii-1, ii) of channel ch, then of channel ch+1
                        cb[o][0][ii >> 1] = __byte_perm(prv[o], cur[o], sel0);
                        cb[o][1][ii >> 1] = __byte_perm(prv[o], cur[o], sel1);
                    }
                }
                dp2 = dc2;
            }
            uint8_t *dst[3] = {base + OFF_G2A, base + OFF_KHT, base + OFF_V};
#pragma unroll
            for (int o = 0; o < 3; ++o)
#pragma unroll
                for (int e = 0; e < 2; ++e)  // 8 tokens of channel-major row ch + (e ^ sw)
                    *reinterpret_cast<uint4 *>(dst[o] + sw128_off(ch + (e ^ sw), tb)) =
                        make_uint4(cb[o][e][0], cb[o][e][1], cb[o][e][2], cb[o][e][3]);
        }
        if (c > 0) {  // the previous chunk's state product, read back while G1 and G1' run
            tc_fence_after();
            readback_state_product(prev_c, prev_tc0, prev_Lc, false);
        }
        mma_wait(bar_mma, ph_mma, flag, p.wait_cycles);
        ph_mma ^= 1;
        tc_fence_after();
        {
            float v[32];
            if (row < 64) {  // G1 row s: Mab -> fp32 block slots (strictly upper part);
                             // then G1' row t: Mak^T (s < t) -> the MN-major half of G34's B
                const int s0 = row, ps = s0 >> 4, r = s0 & 15;
                tmem_ld32(tmem + lane_base + kColG1 + cpart, v);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const int c00 = cpart + 16 * g;
                    const int pc = c00 >> 4;
                    if (pc >= ps) {
                        float *dst = blk(pc == ps ? ps : kSlotM + up_idx(ps, pc)) + r * kSlotRow;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int c = c00 + 4 * q;
                            const float *x = v + 16 * g + 4 * q;
                            reinterpret_cast<float4 *>(dst)[q] =
                                make_float4(c > s0 ? x[0] : 0.f, c + 1 > s0 ? x[1] : 0.f,
                                            c + 2 > s0 ? x[2] : 0.f, c + 3 > s0 ? x[3] : 0.f);
                        }
                    }
                }
                bar_sync_named(1, 128);  // warps 0, 1, 4, 5: Mab is in shared memory
                if (warp < 2) {
                    // T_pp = (I - M_pp)^-1 for the 16x16 diagonal block p, column c, in fp32.
                    // With M_pp = [A B; 0 C] (8x8 blocks), T_pp = [A' A'BC'; 0 C'],
                    // A' = (I - A)^-1 and C' = (I - C)^-1 by back substitution
                    // (x_r = sum_{u > r} M[r][u] x_u above the diagonal), then A'(B C').
                    const int pb = tid >> 4, c = tid & 15, cl = c & 7;
                    const bool right = c >= 8;  // column of C' (rows 8-15) and of A'BC'
                    const int o = right ? 8 : 0;
                    float *md = blk(pb);
                    float x[8];
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) x[rr] = (rr == cl) ? 1.f : 0.f;
#pragma unroll
                    for (int rr = 6; rr >= 0; --rr) {
                        const float4 y0 = reinterpret_cast<const float4 *>(md + (o + rr) * kSlotRow + o)[0];
                        const float4 y1 = reinterpret_cast<const float4 *>(md + (o + rr) * kSlotRow + o)[1];
                        const float mrow[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
                        float acc = 0.f;
#pragma unroll
                        for (int u = rr + 1; u < 8; ++u) acc = fmaf(mrow[u], x[u], acc);
                        if (rr < cl) x[rr] = acc;
                    }
                    float y[8];  // right: y = B x
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) y[rr] = 0.f;
                    if (right) {
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) {
                            const float4 b0 = reinterpret_cast<const float4 *>(md + rr * kSlotRow + 8)[0];
                            const float4 b1 = reinterpret_cast<const float4 *>(md + rr * kSlotRow + 8)[1];
                            y[rr] = b0.x * x[0] + b0.y * x[1] + b0.z * x[2] + b0.w * x[3] +
                                    b1.x * x[4] + b1.y * x[5] + b1.z * x[6] + b1.w * x[7];
                        }
                    }
                    __syncwarp();  // A, B, C of this warp's two blocks are read
                    if (!right) {
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) md[rr * kSlotRow + c] = x[rr];  // A'
                    }
                    __syncwarp();
                    float z[8];  // right: A' y (A' is upper triangular)
                    if (right) {
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) {
                            const float4 a0 = reinterpret_cast<const float4 *>(md + rr * kSlotRow)[0];
                            const float4 a1 = reinterpret_cast<const float4 *>(md + rr * kSlotRow)[1];
                            z[rr] = a0.x * y[0] + a0.y * y[1] + a0.z * y[2] + a0.w * y[3] +
                                    a1.x * y[4] + a1.y * y[5] + a1.z * y[6] + a1.w * y[7];
                        }
                    }
                    __syncwarp();  // A' is read
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const float top = right ? z[rr] : x[rr], bot = right ? x[rr] : 0.f;
                        md[rr * kSlotRow + c] = top;
                        md[(8 + rr) * kSlotRow + c] = bot;
                        *reinterpret_cast<__nv_bfloat16 *>(base + OFF_WT + sw128_off(16 * pb + rr, 16 * pb + c)) =
                            __float2bfloat16_rn(top);
                        *reinterpret_cast<__nv_bfloat16 *>(base + OFF_WT + sw128_off(16 * pb + 8 + rr, 16 * pb + c)) =
                            __float2bfloat16_rn(bot);
                    }
                } else {  // warps 4, 5: T is zero below its diagonal blocks
                    const int s2 = tid - 128;
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    for (int q = 0; q < 2 * (s2 >> 4); ++q)
                        *reinterpret_cast<uint4 *>(base + OFF_WT + sw128_off(s2, 8 * q)) = z;
                }
                // G1' row t: Mak^T (s < t), read after the diagonal blocks are under way
                tmem_ld32(tmem + lane_base + kColG1p + 64 + cpart, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = cpart + q < row ? v[q] : 0.f;
                store_row16(base + OFF_MAKT, row, cpart, v);
                store_row16(base + OFF_MAKT, row, cpart + 16, v + 16);
            } else {  // Qb^T row t' (keep s <= t') -> lower half of G2's A
                const int tq = row - 64;
                tmem_ld32(tmem + lane_base + kColG1p + cpart, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = (cpart + q <= tq) ? v[q] : 0.f;
                store_row16(base + OFF_G2A, 64 + tq, cpart, v);
                store_row16(base + OFF_G2A, 64 + tq, cpart + 16, v + 16);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (*flag) break;

        // ------------------------------------------------ T = (I - Mab)^-1
        // Off-diagonal 16x16 blocks, one warp-level TF32 block product each, in
        // three steps over warps 0-5.  With N_ij = T_ii M_ij (i < j),
        // T_ij = sum_{i<k<=j} N_ik T_kj; grouping the products in pairs,
        //   T_i,i+1 = N_i,i+1 T_i+1,i+1,  T_02 = R_02 T_22,  T_13 = R_13 T_33,
        //   T_03 = R_02 T_23 + R_03 T_33,
        // R_02 = N_02 + N_01 N_12, R_03 = N_03 + N_01 N_13, R_13 = N_13 + N_12 N_23.
        if (warp < 6) {
            // step 1: N_ij for the six pairs (i, j), i < j, one per warp
            const int i = warp < 3 ? 0 : (warp < 5 ? 1 : 2);
            const int j = warp < 3 ? warp + 1 : (warp < 5 ? warp - 1 : 3);
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            block_mma_acc(blk(i), blk(kSlotM + up_idx(i, j)), acc, lane);
            block_frag_store(blk(kSlotN + up_idx(i, j)), acc, lane);
            bar_sync_named(2, 192);
            // step 2: T_01, T_12, T_23 (also kept in fp32), R_02, R_03, R_13 (over the dead M_ij)
            float acc2[2][4];
            const int g = lane >> 2, q = lane & 3;
            if (warp < 3) {
                for (int h = 0; h < 2; ++h)
                    for (int e = 0; e < 4; ++e) acc2[h][e] = 0.f;
                block_mma_acc(blk(kSlotN + up_idx(warp, warp + 1)), blk(warp + 1), acc2, lane);
                if (warp == 2) block_frag_store(blk(kSlotM + kSlotT23), acc2, lane);
            } else {  // R_02 = N_02 + N_01 N_12, R_03 = N_03 + N_01 N_13, R_13 = N_13 + N_12 N_23
                const int c0 = warp == 3 ? up_idx(0, 2) : warp == 4 ? up_idx(0, 3) : up_idx(1, 3);
                const int fa = warp == 5 ? up_idx(1, 2) : up_idx(0, 1);
                const int fb = warp == 3 ? up_idx(1, 2) : warp == 4 ? up_idx(1, 3) : up_idx(2, 3);
                block_frag_load(blk(kSlotN + c0), acc2, lane);
                block_mma_acc(blk(kSlotN + fa), blk(kSlotN + fb), acc2, lane);
                block_frag_store(blk(kSlotM + (warp == 3 ? kSlotR02 : warp == 4 ? kSlotR03 : kSlotR13)), acc2, lane);
            }
            if (warp < 3) {  // T_i,i+1 -> bf16 T (rows 16i + g, +8; columns 16(i+1) + 8h + 2q)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    *reinterpret_cast<uint32_t *>(base + OFF_WT + sw128_off(16 * warp + g, 16 * (warp + 1) + 8 * h + 2 * q)) =
                        pack_bf16(acc2[h][0], acc2[h][1]);
                    *reinterpret_cast<uint32_t *>(base + OFF_WT + sw128_off(16 * warp + g + 8, 16 * (warp + 1) + 8 * h + 2 * q)) =
                        pack_bf16(acc2[h][2], acc2[h][3]);
                }
            }
            bar_sync_named(2, 192);
            // step 3: T_02 = R_02 T_22, T_13 = R_13 T_33, T_03 = R_02 T_23 + R_03 T_33
            if (warp >= 4) preload_g34_rows_j();  // idle in this step
            if (warp < 3) {
                float acc3[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if (warp == 0) {
                    block_mma_acc(blk(kSlotM + kSlotR02), blk(2), acc3, lane);
                } else if (warp == 1) {
                    block_mma_acc(blk(kSlotM + kSlotR13), blk(3), acc3, lane);
                } else {
                    block_mma_acc(blk(kSlotM + kSlotR02), blk(kSlotM + kSlotT23), acc3, lane);
                    block_mma_acc(blk(kSlotM + kSlotR03), blk(3), acc3, lane);
                }
                const int bi = warp == 1 ? 1 : 0, bj = warp == 0 ? 2 : 3;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    *reinterpret_cast<uint32_t *>(base + OFF_WT + sw128_off(16 * bi + g, 16 * bj + 8 * h + 2 * q)) =
                        pack_bf16(acc3[h][0], acc3[h][1]);
                    *reinterpret_cast<uint32_t *>(base + OFF_WT + sw128_off(16 * bi + g + 8, 16 * bj + 8 * h + 2 * q)) =
                        pack_bf16(acc3[h][2], acc3[h][3]);
                }
            }
        } else {
            preload_g34_rows_t();  // warps 6, 7 take no part in the inverse
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();

        // ------------------------------------------------------------- G2
        if (tid == kIssuer) {
            tc_fence_after();
            umma_128xNx64(tmem + kColG2, smem_addr(base + OFF_G2A), smem_addr(base + OFF_G2B), 64, false);
            umma_commit(bar_mma);
        }
        mma_wait(bar_mma, ph_mma, flag, p.wait_cycles);
        ph_mma ^= 1;
        if (tid == kIssuer && !last && !*flag) {  // G2A and R1 are dead
            in_parity = ph_in;
            stage_inputs(0, 5, tc0 + kL, true);
            in_flight = true;
        }
        tc_fence_after();
        {  // Z^T row (this thread's 32 columns) -> bf16 A operand of G34 in tensor memory
            float v[32];
            tmem_ld32(tmem + lane_base + kColG2 + cpart, v);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
            tmem_st16(tmem + lane_base + kColZA + cpart / 2, pk);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        if (*flag) break;

        // ------------------------------------------------------------ G34
        if (tid == kIssuer) {
            tc_fence_after();
            // accumulates onto the additive terms loaded during the inverse
            umma_ta_128xNx64(tmem + 0, tmem + kColZA, smem_addr(base + OFF_G34B), 128, true, true);
            umma_commit(bar_mma);
        }
        mma_wait(bar_mma, ph_mma, flag, p.wait_cycles);
        ph_mma ^= 1;
        tc_fence_after();
        {  // [Phi^T; R'^T] and [Y_B^T; Y_Q^T] rows -> the bf16 A operands of G5 in tensor memory
            float v[32], y[32];
            tmem_ld32(tmem + lane_base + cpart, v);
            tmem_ld32(tmem + lane_base + 64 + cpart, y);
            tmem_ld_wait();
            uint32_t pa[16], py[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                pa[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                py[e] = pack_bf16(y[2 * e], y[2 * e + 1]);
            }
            tmem_st16(tmem + lane_base + kColA2 + cpart / 2, pa);
            tmem_st16(tmem + lane_base + kColYA + cpart / 2, py);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        if (*flag) break;

        // ------------------- G5: [S_L^T; O^T] = [Phi^T; R'^T] [S0_hi | S0_lo]^T + Y^T V^T
        if (tid == kIssuer) {
            tc_fence_after();
            umma_ta_128xNx64(tmem + 0, tmem + kColA2, smem_addr(base + OFF_SHI), 64, false, true);
            umma_ta_128xNx64(tmem + 0, tmem + kColA2, smem_addr(base + OFF_SLO), 64, true, true);
            umma_ta_128xNx64(tmem + 0, tmem + kColYA, smem_addr(base + OFF_V), 64, true, false);
            umma_commit(bar_g5);
        }
        g5_pending = true;  // awaited once the next chunk's elementwise phase is done (or after the loop)
        prev_c = c;
        prev_tc0 = tc0;
        prev_Lc = Lc;
        // The readback of this product waits for the next chunk's first MMA (or the loop end);
        // R1 and the operand tiles are free for the next chunk's elementwise phase now.
    }
    // every thread sees the same abort flag; a unit with a chunk out of range is
    // run token by token below instead, so its chunked final state is not stored
    if (g5_pending && !*flag) {
        mma_wait(bar_g5, ph_g5, flag, p.wait_cycles);
        ph_g5 ^= 1;
        g5_pending = false;
    }
    const bool fallback = __syncthreads_or(range_bad) != 0;
    if (!*flag && !fallback) {
        tc_fence_after();
        readback_state_product(prev_c, prev_tc0, prev_Lc, true);
    }

    if (*flag && tid == kIssuer) {  // a wait gave up: let what the issuer issued land (bounded), then leave
        flag_status(p.lv.status, WKV7_DEV_WAIT_TIMEOUT);
        mbar_wait_bounded(bar_mma, ph_mma ^ 1u, p.wait_cycles);  // the last commit
        // the last state product: not yet waited for, or its wait gave up (a phase
        // before any commit counts as complete, so this returns at once then)
        mbar_wait_bounded(bar_g5, g5_pending ? ph_g5 : ph_g5 ^ 1u, p.wait_cycles);
        if (in_flight) mbar_wait_bounded(bar_in, in_parity, p.wait_cycles);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (fallback && !*flag) {
        // Token by token in float32 from the slot's start state, which the chunked
        // pass has left untouched (its final state is stored only after the last
        // chunk); outputs and checkpoints are rewritten.  The tiles are free: no
        // copy or MMA is in flight.
        __syncthreads();
        prefill_unit_token_by_token<SBF16>(p, h, t0, t1, ck0, s_off, reinterpret_cast<SeqStage *>(base));
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
    if (a.lv.n_heads > 0x7fffffff / 2) return cudaErrorInvalidValue;
    InputMaps maps;
    const void *src[6] = {a.in.r, a.in.w, a.in.k, a.in.v, a.in.a, a.in.b};
    for (int x = 0; x < 6; ++x)
        if (!encode_input_map(&maps.m[x], src[x], a.lv.n_heads, a.total_tokens))
            return cudaErrorInvalidValue;
    void (*const kernels[4])(const PrefillArgs, const InputMaps) = {
        prefill_chunk_kernel<false, false>, prefill_chunk_kernel<false, true>,
        prefill_chunk_kernel<true, false>, prefill_chunk_kernel<true, true>};
    auto kernel = kernels[(a.state_bf16 ? 2 : 0) | (a.in.o_bf16 ? 1 : 0)];
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned ny = static_cast<unsigned>(a.n_seqs) < kGridY ? static_cast<unsigned>(a.n_seqs) : kGridY;
    const dim3 grid(static_cast<unsigned>(a.lv.n_heads), ny, (static_cast<unsigned>(a.n_seqs) + kGridY - 1) / kGridY);
    e = launch_pdl(kernel, grid, dim3(kThreads), kSmemBytes, s, a, maps);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace wkv7
