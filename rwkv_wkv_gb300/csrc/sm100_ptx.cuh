// Thin inline-PTX wrappers for the Blackwell (sm_100 family, built for
// sm_103a) features the chunked prefill uses: mbarriers with bounded waits,
// TMA tensor loads, tcgen05 tensor-memory allocation, UMMA issue/commit and
// tensor-memory loads.  Written from the PTX ISA descriptions of these
// instructions; no library code.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace wkv7 {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may be suspended in hardware for up to
// `suspend_ns` nanoseconds while the phase is incomplete (no issue slots used).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t suspend_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after about
// `limit_cycles` SM clock cycles.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
        if (clock64() - t0 > limit_cycles) return false;
    }
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// Prefetch one tensor-map box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// Named CTA barrier `id` (1..15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void bar_sync_named(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------- tensor memory
// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `holder`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
                 : "memory");
}

// 32 consecutive 32-bit columns of this warp's 32 lanes: lane l of the warp
// receives row (lane base + l), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 16 consecutive 32-bit columns of this warp's 32 lanes (lane l of the
// warp writes row lane base + l).  Complete with tmem_st_wait.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// -------------------------------------------------------------------- UMMA
// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row atoms of 1024
// bytes stacked contiguously (stride-dimension byte offset 1024), atoms
// 1024-byte aligned.  Fields: start address >> 4 in bits 0-13, leading byte
// offset >> 4 in 16-29 (unused for this layout, set to 1), stride byte offset
// >> 4 in 32-45, descriptor version 1 in bits 46-47, layout type 2 (128-byte
// swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Descriptor for an MN-major operand with the 128-byte swizzle: each 128-byte
// row holds 64 consecutive M (or N) elements of one K index, 8-row atoms of
// 1024 bytes stacked along K (stride byte offset 1024); atoms along M/N are
// `mn_stride` bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t mn_stride) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (format 1 in bits 7-9 and
// 10-12), f32 accumulator (format 1 in bits 4-5), both operands K-major
// (bits 15, 16 clear), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn = 0) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K=16 slice; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As umma_bf16 with A (M rows x 16 bf16 of K) in tensor memory at a_tmem: row m
// in lane m, K elements 2c and 2c+1 packed (low, high) in column c, so one K=16
// slice spans 8 columns.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// D (M=128 rows) = A (128 x 64, SW128 K-major at a_saddr) * B^T (B: N x 64,
// SW128 K-major at b_saddr): four K=16 slices, the descriptors' start address
// advanced by 32 bytes per slice.
__device__ __forceinline__ void umma_128xNx64(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                              uint32_t N, bool accumulate) {
    const uint32_t idesc = idesc_bf16_f32(128, N);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        umma_bf16(d_tmem, desc_sw128(a_saddr + 32 * k), desc_sw128(b_saddr + 32 * k), idesc,
                  (accumulate || k > 0) ? 1u : 0u);
    }
}

// As above with B stored MN-major: rows of 64 N-elements per K index, 64-wide
// N atoms `b_atom_stride` bytes apart (N = 128 uses two); the K=16 slices
// advance 2048 bytes (two 8-row atoms) through B.
__device__ __forceinline__ void umma_128xNx64_bmn(uint32_t d_tmem, uint32_t a_saddr,
                                                  uint32_t b_saddr, uint32_t N, bool accumulate,
                                                  uint32_t b_atom_stride = 8192) {
    const uint32_t idesc = idesc_bf16_f32(128, N, 1);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        umma_bf16(d_tmem, desc_sw128(a_saddr + 32 * k),
                  desc_sw128_mn(b_saddr + 2048 * k, b_atom_stride), idesc,
                  (accumulate || k > 0) ? 1u : 0u);
    }
}

// D (M=128) (+)= A (128 x 64 bf16 in tensor memory from column a_tmem, 32
// columns) * B^T, B N x 64 in shared memory: K-major (b_mn = false) or MN-major
// with 64-wide N atoms `b_atom_stride` bytes apart (b_mn = true).
__device__ __forceinline__ void umma_ta_128xNx64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_saddr,
                                                 uint32_t N, bool accumulate, bool b_mn,
                                                 uint32_t b_atom_stride = 8192) {
    const uint32_t idesc = idesc_bf16_f32(128, N, b_mn ? 1u : 0u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t bd = b_mn ? desc_sw128_mn(b_saddr + 2048 * k, b_atom_stride)
                                 : desc_sw128(b_saddr + 32 * k);
        umma_bf16_ta(d_tmem, a_tmem + 8 * k, bd, idesc, (accumulate || k > 0) ? 1u : 0u);
    }
}

// Byte offset of bf16 element (row, col), col < 64, in a K-major tile with
// the 128-byte swizzle (16-byte chunk index XOR row % 8).
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t col) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) +
           (col & 7u) * 2u;
}

}  // namespace sm100
}  // namespace wkv7
