/*
 * libwkv7 -- WKV-7 state-slot engine for one NVIDIA GB300 GPU (sm_103a).
 *
 * What it computes.  RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta
 * Rule)": per layer and head a [head_size x head_size] recurrent state S
 * ("State is a [head_size, head_size] matrix per head per RWKV-7 layer --
 * fixed size regardless of sequence length").  With S[i][j] (i = value index,
 * j = key index) every token does
 *
 *     h = S a;   S <- S diag(w) + h b^T + v k^T;   o = S r
 *
 * (decay, delta-rule term, key-value write, readout after the update).  The
 * delta term uses h = S a on the state before the decay and the vector b,
 * i.e. S <- S (diag(w) + a b^T) + v k^T.
 *
 * How state is held.  "wkvm: state-slot inference for RWKV, GDN and Mamba
 * hybrids", section "The allocation unit wkvm changes": the allocation unit is
 * a fixed-size per-request state slot, and the verbs are create, snapshot,
 * fork and resume (restore).  A pool owns n_slots live slots and n_snapshots
 * parked copies.  One slot holds the states of every layer and head:
 *
 *     slot layout  [layer][head][i][j]  float32 (or bf16, see state_dtype),
 *                  row-major, contiguous
 *     slot bytes   n_layers * n_heads * head_size^2 * 4 (2 for bf16 states)
 *     pool layout  a 256-byte header (the device status word), the slots
 *                  [slot][layer][head][i][j], the snapshots in the same
 *                  layout, then the id-validation bitmap (one bit per id of
 *                  the larger table, rounded up to 256 bytes)
 *
 * Token inputs are packed [rows][n_heads][head_size] (row = batch entry for
 * decode, token for prefill), contiguous, float32 or bf16; outputs o have
 * the same shape, float32 (or bf16, see out_dtype).
 *
 * Conventions for every call.
 *   - All pointers named *_dev and every tensor argument are device pointers
 *     owned by the caller; the library never frees them.  The pool owns its
 *     state buffer unless the caller supplied one at creation.
 *   - Calls that take a cudaStream_t are asynchronous on that stream and never
 *     synchronise, except wkv7_get_device_status.
 *   - Host-checkable faults (NULL pointers, counts, layer range, dtype, head
 *     size) return an error before anything is launched; the pool is left
 *     untouched.
 *   - Faults only the device can see (a slot id out of range inside a device
 *     array, inconsistent cu_seqlens) make the kernel skip that unit and
 *     record a code in the pool's sticky device status word (WKV7_DEV_*),
 *     read with wkv7_get_device_status.  Kernels never trap or assert.
 *   - Slot ids within one call must be distinct, and a call's source and
 *     destination sets must not overlap; violating this is a data race whose
 *     result is undefined.  The fast paths do not check it;
 *     wkv7_validate_ids is the debug pass that does.
 *   - Only head_size == 64 is implemented; other sizes return
 *     WKV7_ERR_UNSUPPORTED.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     begin launching while the previous one in its stream drains, but waits
 *     for all earlier work in the stream before it reads or writes anything
 *     that work may produce (before that, decode only reads its slot ids, which
 *     no library kernel writes, and prefetches state lines into L2), so stream
 *     order is kept exactly as with ordinary launches.
 */
#ifndef WKV7_H
#define WKV7_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WKV7_VERSION 1

typedef struct wkv7_pool wkv7_pool; /* opaque, owned by the library */

typedef enum {
    WKV7_OK = 0,
    WKV7_ERR_INVALID_ARG = 1,   /* NULL pointer, negative count, bad layer/dtype */
    WKV7_ERR_BAD_SLOT = 2,      /* host-side id not in range or not allocated */
    WKV7_ERR_DUP_SLOT = 3,      /* the same id twice in one host-side list */
    WKV7_ERR_POOL_FULL = 4,     /* fewer free slots/snapshots than requested */
    WKV7_ERR_BAD_SEQLENS = 5,   /* host-checkable sequence sizes are inconsistent */
    WKV7_ERR_CUDA = 6,          /* a CUDA runtime call failed; see wkv7_last_error */
    WKV7_ERR_UNSUPPORTED = 7,   /* head_size != 64, an input dtype the call does not
                                   take, or a misaligned input/output base */
    WKV7_ERR_DEVICE_STATUS = 8, /* a kernel recorded a fault; code in *code_out */
    WKV7_ERR_TIMEOUT = 9,       /* the stream did not finish within the limit */
    WKV7_ERR_NO_MEMORY = 10     /* host or device allocation failed */
} wkv7_status;

typedef enum { WKV7_F32 = 0, WKV7_BF16 = 1 } wkv7_dtype;

/* Codes of the sticky device status word (first fault wins). */
#define WKV7_DEV_OK 0
#define WKV7_DEV_BAD_SLOT 1     /* a device slot/snapshot id was out of range */
#define WKV7_DEV_BAD_SEQLENS 2  /* cu_seqlens not monotone, out of range or longer than max_seqlen */
#define WKV7_DEV_WAIT_TIMEOUT 3 /* a bounded in-kernel wait gave up; outputs of that unit are invalid */
#define WKV7_DEV_DECAY_RANGE 4  /* reserved: not recorded (the chunked prefill runs such units token by token) */
#define WKV7_DEV_DUP_SLOT 5     /* wkv7_validate_ids: an id listed twice (in one list or in both) */

/* Id tables for wkv7_validate_ids. */
#define WKV7_TABLE_SLOTS 0
#define WKV7_TABLE_SNAPSHOTS 1

typedef struct {
    int32_t n_layers;    /* >= 1 */
    int32_t n_heads;     /* >= 1 */
    int32_t head_size;   /* must be 64 */
    int32_t n_slots;     /* >= 1, live slots */
    int32_t n_snapshots; /* >= 0, parked copies */
    void *device_buffer; /* NULL: the library allocates (cudaMalloc) and frees.
                            Else a caller-owned device buffer of at least
                            wkv7_pool_required_bytes() bytes, 256-byte aligned,
                            that must outlive the pool. */
    size_t buffer_bytes; /* size of device_buffer (ignored when it is NULL) */
    int32_t state_dtype; /* WKV7_F32 (0, the default when zero-initialised): float32
                            states.  WKV7_BF16: states stored in bf16 -- half the
                            bytes per slot and per decode step; each decode step
                            is computed in float32 and rounds the new state to bf16
                            (nearest even), the readout coming from the unrounded
                            float32 state.  Every call works on a bf16-state pool,
                            computing in float32 and rounding what it stores:
                            wkv7_decode_multi is K such steps (rounded after every
                            token; its rollback snapshots hold the rounded states);
                            the prefill calls read the start state exactly, carry
                            float32 inside a sequence and round the final state
                            and every checkpoint, and at a checkpoint the carry
                            continues from the rounded value, so that resuming from
                            a checkpoint still reproduces the uninterrupted run. */
    int32_t out_dtype;   /* WKV7_F32 (0, the default when zero-initialised): every
                            recurrence call writes o in float32.  WKV7_BF16: o in
                            bf16, the float32 readout rounded to nearest even (the
                            states and everything else are unchanged; the method
                            fixes no output precision, and the float32 paths'
                            1e-4 contract holds only for float32 o). */
} wkv7_pool_desc;

/* ---------------------------------------------------------------- pool ---- */

/* Bytes of device memory a pool with this description needs: a 256-byte
 * header (the device status word), the slot and snapshot states, and the
 * bitmap that wkv7_validate_ids uses (max(n_slots, n_snapshots) bits rounded
 * up to 256 bytes).  Returns 0 for an invalid description. */
size_t wkv7_pool_required_bytes(const wkv7_pool_desc *desc);

/* Create a pool: the fixed-capacity store of state slots of "wkvm: state-slot
 * inference for RWKV, GDN and Mamba hybrids", section "The allocation unit wkvm
 * changes" (a request owns a fixed-size slot), with the capacity reserved up
 * front as "Virtual Memory for KV Cache and Model Weights" reserves hybrid
 * recurrent-state slots separately at admission; each slot holds the
 * per-layer, per-head [head_size, head_size] states of RWKV-X Architecture,
 * "WKV-7 Kernel (Generalized Delta Rule)".  With a caller buffer no CUDA call is made (slot contents are
 * whatever the buffer holds until wkv7_slot_create zeroes them) except that
 * the caller must have zeroed the first 256 bytes (the status word).  With
 * device_buffer == NULL the library allocates on the current device and zeroes
 * the status word.  Every slot and snapshot starts free.
 * Errors: INVALID_ARG, UNSUPPORTED (head_size), NO_MEMORY, CUDA. */
wkv7_status wkv7_pool_create(const wkv7_pool_desc *desc, wkv7_pool **out);

/* Destroy a pool (the opaque state's free of RWKV-X Architecture, "Adapter
 * API": new/free/reset of an opaque state); frees the device buffer only if
 * the library allocated it.
 * The caller must make sure no work using the pool is still in flight. */
wkv7_status wkv7_pool_destroy(wkv7_pool *pool);

/* Copy the pool's description (device_buffer = the buffer actually used). */
wkv7_status wkv7_pool_get_desc(const wkv7_pool *pool, wkv7_pool_desc *out);

/* Bytes of one slot (and of one snapshot): n_layers*n_heads*head_size^2*4
 * (*2 instead of *4 for a bf16-state pool). */
size_t wkv7_slot_bytes(const wkv7_pool *pool);

/* Device address of the float32 [n_heads][head_size][head_size] state of
 * (slot, layer) -- the per-head, per-layer state matrices of RWKV-X
 * Architecture, "WKV-7 Kernel (Generalized Delta Rule)" -- or of a snapshot (for a bf16-state pool the address of the
 * bf16 states, returned through the same float pointer type).  For tests and
 * for initialising states.
 * Errors: INVALID_ARG, BAD_SLOT (index out of range; allocation state is not
 * checked). */
wkv7_status wkv7_pool_state_ptr(wkv7_pool *pool, int32_t slot, int32_t layer, float **dev_ptr);
wkv7_status wkv7_pool_snapshot_ptr(wkv7_pool *pool, int32_t snap, int32_t layer, float **dev_ptr);

/* ------------------------------------------------ slot table (host only) -- */
/* The slot table is host bookkeeping: which ids are handed out.  These calls
 * launch nothing.  Recurrent-state slots are reserved up front, separately
 * from anything else ("Virtual Memory for KV Cache and Model Weights": hybrid
 * recurrent-state slots are reserved separately and must be available at
 * admission), so running out is reported, never grown. */

/* Hand out n free slot ids into ids_out[n] (host array).  All or nothing:
 * POOL_FULL if fewer than n are free. */
wkv7_status wkv7_slot_alloc(wkv7_pool *pool, int32_t n, int32_t *ids_out);
/* Return n slot ids.  All or nothing: BAD_SLOT if any id is out of range or
 * not allocated, DUP_SLOT if an id repeats. */
wkv7_status wkv7_slot_free(wkv7_pool *pool, int32_t n, const int32_t *ids);
wkv7_status wkv7_snapshot_alloc(wkv7_pool *pool, int32_t n, int32_t *ids_out);
wkv7_status wkv7_snapshot_free(wkv7_pool *pool, int32_t n, const int32_t *ids);
/* Number of free slots / snapshots (or -1 for a NULL pool). */
int32_t wkv7_slot_count_free(const wkv7_pool *pool);
int32_t wkv7_snapshot_count_free(const wkv7_pool *pool);
/* *out = 1 if the slot id is allocated, else 0.  BAD_SLOT if out of range. */
wkv7_status wkv7_slot_is_allocated(const wkv7_pool *pool, int32_t slot, int32_t *out);

/* ------------------------------------------------------------ verbs ----- */

/* create: hand out n free slots (ids_out, host array) and zero their state on
 * `stream` -- the verb "create" of the state-slot engine ("The allocation
 * unit wkvm changes"), with the zeroing of a fresh state as in RWKV-X
 * Architecture, "Dual State" (the reset zeros the recurrent state).
 * Errors: INVALID_ARG, POOL_FULL (nothing allocated), CUDA (ids are returned
 * to the free list). */
wkv7_status wkv7_slot_create(wkv7_pool *pool, int32_t n, int32_t *ids_out, cudaStream_t stream);

/* reset: zero the states of n slots given as a device id array (no table
 * change).  Out-of-range ids are skipped and flagged WKV7_DEV_BAD_SLOT. */
wkv7_status wkv7_slot_reset(wkv7_pool *pool, const int32_t *slot_ids_dev, int32_t n,
                            cudaStream_t stream);

/* snapshot: copy slot slot_ids_dev[i] -> snapshot snap_ids_dev[i], i < n, bit
 * for bit.  restore: snapshot -> slot (rolls the slot back to the snapshot).
 * fork: slot src_ids_dev[i] -> slot dst_ids_dev[i].  ("The allocation unit
 * wkvm changes": a fixed-size slot can be copied, parked and restored
 * cheaply; parking in host memory is wkv7_slot_hibernate / wkv7_slot_resume.)
 * Whole-slot copies of every layer and head; the id arrays are caller-owned
 * device int32 arrays of n entries.  Errors: INVALID_ARG (NULL pool or id
 * array with n > 0, n < 0, n larger than the destination table, snapshot or
 * restore on a pool without a snapshot store), CUDA.  Device: out-of-range ids
 * are skipped and flagged WKV7_DEV_BAD_SLOT.  n == 0 is a no-op. */
wkv7_status wkv7_slot_snapshot(wkv7_pool *pool, const int32_t *slot_ids_dev,
                               const int32_t *snap_ids_dev, int32_t n, cudaStream_t stream);
wkv7_status wkv7_slot_restore(wkv7_pool *pool, const int32_t *snap_ids_dev,
                              const int32_t *slot_ids_dev, int32_t n, cudaStream_t stream);
wkv7_status wkv7_slot_fork(wkv7_pool *pool, const int32_t *src_ids_dev,
                           const int32_t *dst_ids_dev, int32_t n, cudaStream_t stream);

/* hibernate: copy slot slot_ids_dev[i] -> bytes [i*slot_bytes, (i+1)*slot_bytes)
 * of host_dst, i < n, bit for bit; resume: those bytes of host_src -> slot
 * slot_ids_dev[i].  The verbs "hibernate" and "resume" of "wkvm: state-slot
 * inference for RWKV, GDN and Mamba hybrids", section "The allocation unit
 * wkvm changes": a fixed-size slot can be parked off the GPU and brought back.
 * host_dst / host_src is caller-owned page-locked host memory that the device
 * can address (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with the
 * mapped flag), 16-byte aligned, of host_bytes >= n * wkv7_slot_bytes(pool)
 * bytes, packed slot after slot.  One kernel gathers (or scatters) the slots
 * over the device's link to host memory; asynchronous on `stream` like every
 * verb, so the host must not read host_dst (or change host_src) before the
 * stream has passed the call.  The slot table is not changed: freeing a
 * hibernated slot's id, and taking one for its resume, are the caller's.
 * Errors: INVALID_ARG (NULL pointers, host_bytes too small, host memory that
 * is not page-locked and device-mapped or not 16-byte aligned), CUDA.  Device:
 * WKV7_DEV_BAD_SLOT for an out-of-range id (that slot is not copied).  n == 0
 * is a no-op. */
wkv7_status wkv7_slot_hibernate(wkv7_pool *pool, const int32_t *slot_ids_dev, int32_t n,
                                void *host_dst, size_t host_bytes, cudaStream_t stream);
wkv7_status wkv7_slot_resume(wkv7_pool *pool, const void *host_src, size_t host_bytes,
                             const int32_t *slot_ids_dev, int32_t n, cudaStream_t stream);

/* --------------------------------------------------------- recurrence ---- */

/* Every call in this section reads its inputs and writes o with vector loads
 * and stores, so the six input bases and o must be 16-byte aligned; a base
 * that is not is reported as UNSUPPORTED before any launch.  o holds float32
 * elements, or bf16 ones on a pool created with out_dtype = WKV7_BF16 (each
 * the float32 readout rounded to nearest even); the shapes below count
 * elements either way. */

/* decode: one token for each of n slots at one layer -- the per-token
 * recurrence of RWKV-X Architecture, "WKV-7 Kernel (Generalized Delta Rule)"
 * (decay, delta-rule term, key-value write, readout after the update), run as
 * one batched step over the state slots of "wkvm: state-slot inference for
 * RWKV, GDN and Mamba hybrids" ("The allocation unit wkvm changes").  For b < n and every
 * head h, the state at (slot_ids_dev[b], layer, h) takes one step of the
 * recurrence with inputs x[b][h][:] (x = r, w, k, v, a, b; [n][n_heads][64],
 * dtype in_dtype) and o[b][h][:] receives the readout.  The state is
 * read once and written once.  Errors: INVALID_ARG (including n > n_slots),
 * UNSUPPORTED (a misaligned base), CUDA.  Device: WKV7_DEV_BAD_SLOT for an out-of-range id (that
 * row's state and o are untouched). */
wkv7_status wkv7_decode_step(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                             int32_t n, wkv7_dtype in_dtype, const void *r, const void *w,
                             const void *k, const void *v, const void *a, const void *b,
                             void *o, cudaStream_t stream);

/* decode_multi: n_tokens (K >= 1) consecutive tokens for each of n slots at
 * one layer, the verify pass of speculative decoding on state slots (the
 * rvLLM README, "Speculative decoding (GPU, shipped)": K drafted tokens are
 * checked by one pass over K+1 tokens; with a recurrent state the pass must
 * also leave a state at every token so that the slot can be rolled back to
 * the last accepted one, the fork/restore verbs of "wkvm: state-slot
 * inference for RWKV, GDN and Mamba hybrids").  Inputs x[b][k][h][:] and
 * o[b][k][h][:] are [n][K][n_heads][64]; row b's state at
 * (slot_ids_dev[b], layer) takes the K steps in order, held on chip between
 * them (read once, written once), and o gets every token's readout.  With
 * step_snap_ids_dev ([n][K] device ids, or NULL for none) the state after
 * token k of row b is also written to this layer's slice of snapshot
 * step_snap_ids_dev[b*K + k]; restoring that snapshot rolls the slot back to
 * just after token k.  K == 1 without snapshots equals wkv7_decode_step bit
 * for bit.  Errors: INVALID_ARG (including n > n_slots, K < 1, snapshots
 * asked of a pool without a snapshot store), UNSUPPORTED, CUDA.  Device:
 * WKV7_DEV_BAD_SLOT for an out-of-range slot id (that row is untouched) or
 * snapshot id (that snapshot is not written). */
wkv7_status wkv7_decode_multi(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                              int32_t n, int32_t n_tokens, wkv7_dtype in_dtype, const void *r,
                              const void *w, const void *k, const void *v, const void *a,
                              const void *b, void *o, const int32_t *step_snap_ids_dev,
                              cudaStream_t stream);

/* prefill: n_seqs sequences packed back to back (RWKV-X Architecture, "What
 * Was Stripped": the batch forward is the prefill path).  Sequence s holds
 * tokens cu_seqlens_dev[s] .. cu_seqlens_dev[s+1]-1 of the packed inputs
 * [total_tokens][n_heads][64] (bf16) and starts from the state at
 * (slot_ids_dev[s], layer); the slot receives the state after its last token
 * and o[t][h][:] the readout of every token.  The result equals
 * the token-by-token recurrence up to rounding; it is computed in chunks of
 * 64 tokens anchored at each sequence's first token, with bf16 tensor-core
 * operands and a float32 state carried between chunks.  A (sequence, head)
 * whose decay over half a chunk (32 tokens) exceeds 2^120 in some channel --
 * beyond the float range of the chunk factorisation, e.g. w = 2^-8 for 32
 * tokens, or w = 0 -- is run token by token in float32 by the same call
 * instead (its results then equal wkv7_prefill_sequential's).  The test
 * takes every w in (0, 1], the range of the method's decay: it looks at the
 * factors at the ends of each 8-token run, between which they only fall (a
 * w above 1 may take a factor out of range unseen, losing precision there;
 * NaN, inf and 0 are always caught).  max_seqlen
 * bounds every sequence length.  Errors: INVALID_ARG, UNSUPPORTED (in_dtype
 * must be WKV7_BF16; a misaligned base), CUDA.  Device: WKV7_DEV_BAD_SLOT,
 * WKV7_DEV_BAD_SEQLENS (that sequence is skipped), WKV7_DEV_WAIT_TIMEOUT. */
wkv7_status wkv7_prefill(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                         const int32_t *cu_seqlens_dev, int32_t n_seqs, int32_t total_tokens,
                         int32_t max_seqlen, wkv7_dtype in_dtype, const void *r,
                         const void *w, const void *k, const void *v, const void *a,
                         const void *b, void *o, cudaStream_t stream);

/* prefill_sequential: the same contract as wkv7_prefill, computed token by
 * token in float32 on the CUDA cores (no chunking, no tensor cores; accepts
 * WKV7_F32 or WKV7_BF16 inputs).  Slower; exact to float32 rounding. */
wkv7_status wkv7_prefill_sequential(wkv7_pool *pool, int32_t layer,
                                    const int32_t *slot_ids_dev,
                                    const int32_t *cu_seqlens_dev, int32_t n_seqs,
                                    int32_t total_tokens, int32_t max_seqlen,
                                    wkv7_dtype in_dtype, const void *r, const void *w,
                                    const void *k, const void *v, const void *a,
                                    const void *b, void *o, cudaStream_t stream);

/* prefill_checkpointed: wkv7_prefill (sequential == 0) or
 * wkv7_prefill_sequential (sequential != 0) that also keeps the state at
 * every 64-token boundary of each sequence (xLLM, "Virtual Memory for KV
 * Cache and Model Weights", prefix caching: chunked prefill publishes whole
 * blocks only, and a hybrid model's linear-attention part can resume a
 * cached prefix only from a stored state).  Sequence s (length len_s) owns the ids
 * ckpt_snap_ids_dev[cu_ckpt_dev[s] .. cu_ckpt_dev[s+1]-1], which must number
 * len_s / 64 (rounded down); the m-th (m = 1, 2, ...) receives, in this
 * layer's slice of that snapshot, the float32 state after the sequence's
 * token 64*m, exactly as the next chunk starts from it, so restoring it and
 * prefilling the rest of the sequence reproduces the uninterrupted run's
 * later outputs and final state bit for bit on either path.  When a
 * length is a multiple of 64 the last checkpoint equals the final state.
 * cu_ckpt_dev ([n_seqs+1]) and ckpt_snap_ids_dev are caller-owned device
 * arrays.  Errors: those of the chosen path, and INVALID_ARG when either array
 * is missing or the pool has no snapshot store.  Device: WKV7_DEV_BAD_SEQLENS
 * for a count that does not match (that sequence is skipped),
 * WKV7_DEV_BAD_SLOT for an out-of-range snapshot id (that checkpoint is not
 * written). */
wkv7_status wkv7_prefill_checkpointed(wkv7_pool *pool, int32_t layer, const int32_t *slot_ids_dev,
                                      const int32_t *cu_seqlens_dev, int32_t n_seqs,
                                      int32_t total_tokens, int32_t max_seqlen,
                                      wkv7_dtype in_dtype, const void *r, const void *w,
                                      const void *k, const void *v, const void *a,
                                      const void *b, void *o, const int32_t *cu_ckpt_dev,
                                      const int32_t *ckpt_snap_ids_dev, int32_t sequential,
                                      cudaStream_t stream);

/* --------------------------------------------------------- validation ---- */

/* validate_ids: the debug pass over device id arrays that the fast paths skip.
 * Checks that every id of ids_a_dev[0..n_a) and ids_b_dev[0..n_b) lies in the
 * table (WKV7_TABLE_SLOTS: [0, n_slots); WKV7_TABLE_SNAPSHOTS: [0,
 * n_snapshots)) and that no id occurs twice, within either list or in both --
 * so it covers the repeated ids of one call (a = the call's ids, n_b = 0) and
 * the overlap of a mixed step's decode and prefill slot sets (a = decode ids,
 * b = prefill ids).  The state-slot engine's hard-error discipline (the rvLLM
 * README: no silent fallback; a request that breaks the contract is an
 * error, never repaired) applied to ids only the device holds.
 * Asynchronous on `stream` like every call: two kernels (clear the pool's
 * bitmap, then mark each id with an atomic OR).  A repeat records
 * WKV7_DEV_DUP_SLOT and an out-of-range id WKV7_DEV_BAD_SLOT in the device
 * status word (first fault wins); wkv7_get_device_status then returns
 * WKV7_ERR_DUP_SLOT (or WKV7_ERR_DEVICE_STATUS).  Reads only the id arrays;
 * writes only the pool's bitmap and status word, never a state.  Two
 * validate calls on one pool must not overlap in time (they share the
 * bitmap).  Id arrays are caller-owned device int32 arrays.  Errors:
 * INVALID_ARG (NULL pool, unknown table, n_a or n_b negative, a NULL array
 * with a positive count), CUDA.  n_a == n_b == 0 is a no-op. */
wkv7_status wkv7_validate_ids(wkv7_pool *pool, int32_t table, const int32_t *ids_a_dev, int32_t n_a,
                              const int32_t *ids_b_dev, int32_t n_b, cudaStream_t stream);

/* validate_ids_noalloc: the same check as wkv7_validate_ids for callers that
 * cannot allocate device memory -- a process whose device memory is already
 * handed out in full to another allocator (a framework's caching allocator
 * that reserved the device, say), or a serving loop that forbids allocation
 * after start-up because cudaMalloc synchronises the device at an unbounded
 * cost -- and that hold no pool to lend its scratch.  It takes no pool and
 * allocates nothing: its bitmap is a static device array built into the
 * library (1,048,576 bits = 128 KiB, held on every GPU that loads the library
 * until the process exits), and the verdict goes to the caller's word.  No
 * counterpart in the pages; it exists for such callers only.
 * n_table: the ids are valid in [0, n_table), at most 1,048,576 (larger is
 * WKV7_ERR_UNSUPPORTED).  ids_a_dev[n_a], ids_b_dev[n_b]: caller-owned device
 * int32 lists, as in wkv7_validate_ids.  result_dev: a caller-owned device
 * int32 that the call first sets to WKV7_DEV_OK and then, on a fault, to
 * WKV7_DEV_DUP_SLOT (an id twice, within a list or in both) or
 * WKV7_DEV_BAD_SLOT (an id out of range), the first fault winning; read it
 * once `stream` has passed the call.  The first call on a device (with that
 * device current) looks up the array's device address and keeps it; make that
 * first call before any stream capture.  Every call on a device uses the same
 * array, cleared by the call itself: calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race on it and may report
 * wrong results.  Errors: INVALID_ARG (negative sizes, NULL result_dev, a
 * NULL list with a positive count), UNSUPPORTED (n_table too large), CUDA. */
wkv7_status wkv7_validate_ids_noalloc(int32_t n_table, const int32_t *ids_a_dev, int32_t n_a,
                                      const int32_t *ids_b_dev, int32_t n_b, int32_t *result_dev,
                                      cudaStream_t stream);

/* ------------------------------------------------------------- status ---- */

/* Wait (at most timeout_ms, polling; <= 0 means 10000) for the work queued on
 * `stream`, then read and clear the pool's device status word into *code_out
 * (WKV7_DEV_*).  This is how the hard errors of the rvLLM README ("no
 * fallbacks": a fault is reported, never silently repaired) reach the host for
 * the faults that only a kernel sees.  Returns WKV7_ERR_DUP_SLOT when the code
 * is WKV7_DEV_DUP_SLOT, WKV7_ERR_DEVICE_STATUS for any other non-zero code,
 * WKV7_ERR_TIMEOUT when the stream did not finish in time (the word is left
 * as it is), WKV7_ERR_CUDA on a CUDA error. */
wkv7_status wkv7_get_device_status(wkv7_pool *pool, cudaStream_t stream, int32_t timeout_ms,
                                   int32_t *code_out);

/* Static text for a status code. */
const char *wkv7_status_string(wkv7_status status);
/* Text of the last CUDA error seen by this thread inside the library. */
const char *wkv7_last_error(void);
/* Number of kernels this process has launched through the library. */
uint64_t wkv7_launch_count(void);
int32_t wkv7_version(void);

/* Test hook for the bounded waits of the chunked prefill (process-wide, off by
 * default; for tests only).  While on != 0, every wkv7_prefill on the chunked
 * path skips its first input load, so the wait for it is never satisfied; each
 * wait then gives up after about 50 ms instead of about 2 s, the CTA releases
 * its tensor memory and exits, and the call reports WKV7_DEV_WAIT_TIMEOUT
 * through wkv7_get_device_status (its outputs and the slot's state are not
 * meaningful).  The context stays usable.  Returns WKV7_OK. */
wkv7_status wkv7_test_force_wait_timeout(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_H */
