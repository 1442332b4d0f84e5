// Internal interface between the C-ABI layer (capi.cpp) and the kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace wkv7 {

constexpr int kHeadSize = 64;
constexpr int kHeadFloats = kHeadSize * kHeadSize;

// One layer of a pool, as the recurrence kernels see it.
struct LayerView {
    float *states;          // pool state base (slot 0, layer 0, head 0)
    long long slot_stride;  // floats per slot
    long long layer_off;    // floats from a slot's start to this layer
    int n_slots;
    int n_heads;
    int *status;            // sticky device status word
};

struct TokenInputs {
    const void *r, *w, *k, *v, *a, *b;
    bool bf16;
    void *o;      // float32, or bf16 when o_bf16
    bool o_bf16;  // the pool's out_dtype: o rounded to bf16 (nearest even)
};

struct DecodeArgs {
    LayerView lv;  // for a bf16-state pool, states/slot_stride/layer_off count bf16 elements
    const int *slot_ids;
    int n;
    TokenInputs in;
    bool state_bf16;
};

// K consecutive tokens per slot: inputs and o are [n][K][H][64]; with
// step_snap_ids ([n][K]) non-null, the state after token k of row b also goes
// to snapshot step_snap_ids[b*K + k] (this layer's slice).
struct DecodeMultiArgs {
    LayerView lv;  // for a bf16-state pool, states/slot_stride/layer_off count bf16 elements
    const int *slot_ids;
    int n;
    int n_tok;
    TokenInputs in;
    float *snaps;  // same element type and strides as the states
    int n_snaps;
    const int *step_snap_ids;
    bool state_bf16;
};

// Optional states at every 64-token boundary of each sequence: sequence s
// writes the state after its token 64*m (m = 1 .. len_s / 64) into snapshot
// ckpt_ids[cu_ckpt[s] + m - 1] (this layer's slice).  cu_ckpt == nullptr: none.
struct CheckpointArgs {
    float *snaps;          // snapshot store base (snapshot 0, layer 0, head 0)
    int n_snaps;
    const int *cu_ckpt;    // [n_seqs + 1]
    const int *ckpt_ids;
};

// On a bf16-state pool the start state is read as bf16 and the states written
// (the final one, checkpoints) are rounded to bf16; the carry inside a sequence
// stays float32 except at checkpoint boundaries, where it continues from the
// rounded checkpoint, so that resuming from a checkpoint reproduces the rest.
struct PrefillArgs {
    LayerView lv;  // for a bf16-state pool, states/slot_stride/layer_off count bf16 elements
    const int *slot_ids;
    const int *cu_seqlens;
    int n_seqs;
    int total_tokens;
    int max_seqlen;
    TokenInputs in;
    CheckpointArgs ck;  // snaps: same element type and strides as the states
    bool state_bf16;
    long long wait_cycles;      // bound of every wait in the chunked kernel (clock cycles)
    bool test_skip_first_load;  // test hook: the first input load is never issued
};

constexpr long long kWaitCycles = 4000000000LL;     // about 2 s at 2 GHz
constexpr long long kTestWaitCycles = 100000000LL;  // about 50 ms: the test hook's bound

// Whole-slot copies: dst[dst_ids[i]] <- src[src_ids[i]], slot_floats each; a
// null id array stands for the identity (the i-th slot of a packed buffer).
struct CopyArgs {
    float *dst;
    const float *src;
    const int *dst_ids;
    const int *src_ids;
    int n;
    int n_dst;
    int n_src;
    long long slot_floats;
    int *status;
};

constexpr int kZeroIdsPerLaunch = 512;
struct ZeroIds {
    int ids[kZeroIdsPerLaunch];
};

// Debug validation of two device id lists against a table of n_table ids
// (marks: a bitmap of (n_table + 31) / 32 words of scratch).
struct ValidateArgs {
    uint32_t *marks;
    int n_table;
    const int *ids_a;
    int n_a;
    const int *ids_b;
    int n_b;
    int *status;
};

// Launch counter and last-error text of the C-ABI layer, for entry points that
// live beside their kernels.
void note_launches(int launches);
void note_cuda_error(const char *what, cudaError_t e);

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_validate_ids(const ValidateArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_decode_multi(const DecodeMultiArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_prefill_sequential(const PrefillArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_slot_copy(const CopyArgs &a, cudaStream_t s, int *launches);
// Zero slots listed in a device id array.
cudaError_t launch_slot_zero_dev(float *states, int n_slots, long long slot_floats,
                                 const int *ids_dev, int n, int *status, cudaStream_t s,
                                 int *launches);
// Zero slots listed on the host (ids passed by value, in batches).
cudaError_t launch_slot_zero_host(float *states, int n_slots, long long slot_floats,
                                  const int *ids_host, int n, int *status, cudaStream_t s,
                                  int *launches);

}  // namespace wkv7
