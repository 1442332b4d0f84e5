// Token-by-token WKV-7 prefill on the CUDA cores, in float32 (the recurrence
// of RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)").  One CTA of
// 256 threads runs one (sequence, head): prefill_seq_unit.cuh holds the body.
//
// This is the exact-to-float32 path (wkv7_prefill_sequential); the chunked
// tensor-core path is wkv7_prefill.
#include "prefill_seq_unit.cuh"

namespace wkv7 {
namespace {

template <bool BF16, bool SBF16>
__global__ void __launch_bounds__(256) prefill_seq_kernel(PrefillArgs p) {
    __shared__ __align__(16) SeqStage stage;
    pdl_prologue();

    const int seq = blockIdx.x;
    const int h = blockIdx.y;
    const int slot = __ldg(p.slot_ids + seq);
    const int t0 = __ldg(p.cu_seqlens + seq);
    const int t1 = __ldg(p.cu_seqlens + seq + 1);
    if (slot < 0 || slot >= p.lv.n_slots) {
        if (threadIdx.x == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SLOT);
        return;
    }
    if (t0 < 0 || t1 < t0 || t1 > p.total_tokens || t1 - t0 > p.max_seqlen) {
        if (threadIdx.x == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SEQLENS);
        return;
    }
    int ck0 = 0;  // this sequence's first checkpoint id index
    if (p.ck.cu_ckpt) {
        ck0 = __ldg(p.ck.cu_ckpt + seq);
        if (ck0 < 0 || __ldg(p.ck.cu_ckpt + seq + 1) - ck0 != (t1 - t0) / 64) {
            if (threadIdx.x == 0 && h == 0) flag_status(p.lv.status, WKV7_DEV_BAD_SEQLENS);
            return;
        }
    }
    // element offset of this (slot, layer, head) state; elements are bf16 with SBF16
    const size_t s_off = static_cast<size_t>(slot) * p.lv.slot_stride + p.lv.layer_off +
                         static_cast<size_t>(h) * kHeadFloats;
    prefill_seq_unit<BF16, SBF16>(p, h, t0, t1, ck0, s_off, &stage);
}

}  // namespace

cudaError_t launch_prefill_sequential(const PrefillArgs &a, cudaStream_t s, int *launches) {
    if (a.n_seqs <= 0) return cudaSuccess;
    if (a.lv.n_heads > 65535) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(a.n_seqs), static_cast<unsigned>(a.lv.n_heads));
    void (*const kernels[4])(PrefillArgs) = {prefill_seq_kernel<false, false>, prefill_seq_kernel<false, true>,
                                             prefill_seq_kernel<true, false>, prefill_seq_kernel<true, true>};
    const cudaError_t e =
        launch_pdl(kernels[(a.in.bf16 ? 2 : 0) | (a.state_bf16 ? 1 : 0)], grid, dim3(256), 0, s, a);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace wkv7
