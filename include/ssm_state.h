/*
 * ssm_state.h -- C ABI of libssmstate, the GB300 (sm_103a) library for the
 * Mamba-2 selective-state recurrence in its three serving forms.
 *
 * The recurrence (Mamba-2 structured state space duality: Mamba Streaming
 * State That Survives Chunking, section Separate Mamba-2 algebra from kernel
 * behavior; Why Speculative Decoding Slows Hybrid Mamba Models at Large Batch
 * Sizes, section The Fix: each token first decays the previous state and then
 * adds its own rank-one contribution), per request r, head h, row
 * p < headdim, column n < dstate:
 *
 *     dA_t      = exp(dt_t * A_h)
 *     h_t[p,n]  = dA_t * h_{t-1}[p,n] + dt_t * x_t[p] * B_t[g(h),n]
 *     y_t[p]    = sum_n C_t[g(h),n] * h_t[p,n] + D_h * x_t[p]
 *
 * with groups of contiguous heads, g(h) = h / (nheads / ngroups).  dt arrives
 * already positive (no softplus or bias is applied here); y reads the state
 * after the token.  The state is always fp32.
 *
 * Layouts (row-major, innermost last; every pointer below is a DEVICE pointer
 * unless it says host):
 *   state of a slot   float [nheads][headdim][dstate]
 *   x, y              [tokens][nheads][headdim]        input dtype
 *   dt                [tokens][nheads]                  dt dtype
 *   B, C              [tokens][ngroups][dstate]         input dtype
 *   A, D              float [nheads]
 * For a decode step "tokens" is the batch; for a verify step it is
 * [batch][n_tok]; for a scan it is the packed tokens of all sequences.
 *
 * Ownership.  The pool owns all state, snapshot, log and metadata memory
 * (allocated once by ssm_state_init, freed by ssm_state_destroy).  The caller
 * owns every input and output buffer and the stream.  All calls are
 * asynchronous on the given stream unless marked "synchronous".
 *
 * Errors.  Host-side checks (null pointers, shapes, slot range, duplicate or
 * released slots, chunk order) return an error before any work is queued:
 * nothing advances.  Errors found on the device (non-finite input, a
 * poisoned slot, an accept count out of range, a non-empty replay log where
 * none is allowed) do not stop the stream: the kernel skips the affected
 * (request, head) work, sets a sticky bit in the pool's device flag word,
 * and marks the slot poisoned; poisoned slots are skipped by every later
 * call until ssm_state_reset or ssm_state_restore.  ssm_pool_status reads
 * the flag word.  A pool is not thread safe.
 */
#ifndef SSM_STATE_H
#define SSM_STATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (0 = the legacy default stream). */
typedef struct CUstream_st *ssm_stream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,   /* bad pointer, size, shape, dtype, slot index */
    SSM_ERR_INVALID_CHUNK = 2, /* malformed chunk (Mamba Streaming State, runnable artifact: invalid_chunk) */
    SSM_ERR_INVALID_STATE = 3, /* slot released, or commit without a verify (same artifact: invalid_state) */
    SSM_ERR_SEQUENCE = 4,      /* chunk sequence number out of order (Let the full scan define legal chunking) */
    SSM_ERR_DUPLICATE = 5,     /* chunk sequence number already applied (same section: a chunk applied twice) */
    SSM_ERR_SCHEMA = 6,        /* restore of a state whose layout does not match the pool */
    SSM_ERR_CUDA = 7,          /* a CUDA runtime call failed */
    SSM_ERR_TIMEOUT = 8,       /* a bounded device wait gave up */
    SSM_ERR_NO_MEMORY = 9      /* device or host allocation failed */
} ssm_status;

/* dtype codes (those of the SSM.PREFIX state blob: 0 = fp32, 2 = bf16) */
enum { SSM_DTYPE_F32 = 0, SSM_DTYPE_BF16 = 2 };

/* speculative verify flavour of a pool */
enum {
    SSM_MODE_COPY = 0,   /* verify keeps a full state after every step token */
    SSM_MODE_REPLAY = 1  /* verify reads checkpoint + input log; commit appends or folds */
};

/* when a replay pool writes a full window into the checkpoint (The Fix: the
 * full state is written only when the window fills) */
enum {
    SSM_FOLD_AT_COMMIT = 0, /* the commit that fills the window folds it (a checkpoint read + write) */
    SSM_FOLD_IN_VERIFY = 1  /* the commit appends; the next verify, which reads the checkpoint anyway,
                               folds a log of W or more tokens and writes the checkpoint once */
};

/* sticky device flag bits (ssm_pool_status) */
enum {
    SSM_FLAG_NONFINITE_INPUT = 1u << 0, /* a NaN or Inf in x, dt, B or C */
    SSM_FLAG_POISONED_SLOT = 1u << 1,   /* work on a poisoned slot was skipped */
    SSM_FLAG_BAD_ACCEPT = 1u << 2,      /* accept count outside [0, n_tok - 1] */
    SSM_FLAG_LOG_NOT_EMPTY = 1u << 3,   /* in-place update on a replay slot whose log is not empty */
    SSM_FLAG_TIMEOUT = 1u << 4          /* a bounded device wait gave up */
};

typedef struct {
    int32_t nheads;      /* H */
    int32_t headdim;     /* P, 1..256 */
    int32_t dstate;      /* N, one of 16, 32, 64, 128, 256 */
    int32_t ngroups;     /* G, divides H */
    int32_t input_dtype; /* x, B, C and y: SSM_DTYPE_F32 or SSM_DTYPE_BF16 */
    int32_t dt_dtype;    /* dt: SSM_DTYPE_F32 or SSM_DTYPE_BF16 */
    int32_t mode;        /* SSM_MODE_COPY or SSM_MODE_REPLAY */
    int32_t window;      /* replay window W >= 1 (replay mode; ignored otherwise) */
    int32_t max_tokens;  /* largest n_tok (= T + 1) of one verify step, 1..64 */
    int32_t fold;        /* replay mode: SSM_FOLD_AT_COMMIT or SSM_FOLD_IN_VERIFY (0 otherwise) */
} ssm_config;

/* per-slot metadata (Make reset, checkpoint, and cancellation observable:
 * the absolute position and the chunk sequence travel with the state) */
typedef struct {
    int64_t position;   /* tokens applied since the last reset */
    int64_t next_chunk; /* chunk sequence number ssm_scan_chunk expects next */
    int64_t epoch;      /* number of resets of this slot */
    int32_t log_len;    /* replay mode: tokens in the input log (0..W-1; up to W - 1 + max_tokens
                           between a commit and the next verify with SSM_FOLD_IN_VERIFY) */
    uint32_t flags;     /* bit 0: poisoned; bit 1: released */
} ssm_slot_meta;

typedef struct ssm_pool_s *ssm_pool;

/* ---------------------------------------------------------------- lifecycle */

/*
 * Create a pool of n_slots fixed-size fp32 states on the current device,
 * each at position zero with a zero or caller-given initial state (Make
 * reset, checkpoint, and cancellation observable: initialization).
 * init_state: device float [n_slots][H][P][N] copied in, or NULL for zeros.
 * Copy mode also allocates 2 x max_tokens snapshot states per slot; replay
 * mode allocates a log of W - 1 + max_tokens entries per slot
 * (W - 1 + 2 max_tokens with SSM_FOLD_IN_VERIFY).  SSM_FOLD_IN_VERIFY needs
 * the tensor-core replay path: bf16 inputs, headdim 64, dstate 128, an even
 * number of heads per group, max_tokens <= 32 and W - 1 + 2 max_tokens <= 64
 * (SSM_ERR_INVALID_ARG otherwise).
 * Synchronous.  *out is set only on SSM_OK.
 */
ssm_status ssm_state_init(const ssm_config *cfg, int32_t n_slots, const float *init_state,
                          ssm_stream_t stream, ssm_pool *out);

/* Free every allocation of the pool (synchronous; the pool must be idle). */
ssm_status ssm_state_destroy(ssm_pool pool);

/*
 * Reset slots (host int32[n]): new sequence boundary, state := 0,
 * position := 0, next chunk := 0, log emptied, poison cleared, epoch += 1;
 * also re-opens a released slot (Make reset, checkpoint, and cancellation
 * observable: a reset cuts every tie to the previous stream).
 */
ssm_status ssm_state_reset(ssm_pool pool, const int32_t *slots, int32_t n, ssm_stream_t stream);

/*
 * Cancellation (host int32[n] slots): the slot stops advancing; every later
 * call naming it fails with SSM_ERR_INVALID_STATE until it is reset (Make
 * reset, checkpoint, and cancellation observable: cancellation ends
 * ownership and further advancement).
 */
ssm_status ssm_state_release(ssm_pool pool, const int32_t *slots, int32_t n);

/*
 * Checkpoint one slot: in replay mode first fold the input log into the
 * state (A: device float [H], the layer's A; may be NULL in copy mode), then
 * copy the state (float [H][P][N], H*P*N*4 bytes) into the host buffer and
 * its metadata into *meta (Make reset, checkpoint, and cancellation
 * observable: a checkpoint holds what resuming the same stream needs).
 * Synchronous.
 * SSM_ERR_INVALID_ARG if cap_bytes is too small.
 */
ssm_status ssm_state_checkpoint(ssm_pool pool, int32_t slot, const float *A, float *host_state,
                                size_t cap_bytes, ssm_slot_meta *meta, ssm_stream_t stream);

/*
 * Restore one slot from a checkpoint: host float [H][P][N] of exactly
 * H*P*N*4 bytes and the metadata it was saved with (position, next_chunk,
 * epoch).  The log is emptied and the poison cleared.  SSM_ERR_SCHEMA if
 * bytes does not match the pool's state size: an incompatible resume is
 * refused, never padded or truncated (Make reset, checkpoint, and
 * cancellation observable: checkpoint receipt).  Synchronous.
 */
ssm_status ssm_state_restore(ssm_pool pool, int32_t slot, const float *host_state, size_t bytes,
                             const ssm_slot_meta *meta, ssm_stream_t stream);

/* ---------------------------------------------------------------- checkpoint receipt */

/*
 * Whose state it is: given by the caller when it checkpoints and again when
 * it resumes (Treat Mamba streaming state as a stream-owned record: a state
 * belongs to one stream under one model, code revision and layer).  The
 * revisions are the caller's identifiers (for instance hashes of revision
 * strings); the library only compares them.
 */
typedef struct {
    uint64_t stream_id;
    uint64_t model_revision;
    uint64_t code_revision;
    int32_t layer;
    int32_t reserved; /* 0 */
} ssm_stream_identity;

#define SSM_STATE_SCHEMA_VERSION 1u /* layout of the state: fp32 [H][P][N], n fastest */

/*
 * A checkpoint receipt (Make reset, checkpoint, and cancellation
 * observable: checkpoint receipt): the identity, the state schema, dtypes,
 * layer and state dimensions, the absolute position, the chunk sequence and
 * a checksum of the state.
 */
typedef struct {
    ssm_stream_identity id;
    uint32_t schema_version; /* SSM_STATE_SCHEMA_VERSION */
    int32_t state_dtype;     /* SSM_DTYPE_F32 */
    int32_t input_dtype;     /* the pool's x / B / C dtype */
    int32_t dt_dtype;
    int32_t nheads, headdim, dstate, ngroups;
    int64_t position;        /* tokens applied since the stream began */
    int64_t next_chunk;      /* chunk sequence number expected next */
    uint64_t checksum;       /* FNV-1a 64 over the state blob */
} ssm_receipt;

/*
 * Serialized checkpoint, little-endian: "SSMR", uint32 format version 1,
 * then the receipt fields in the order above (uint64 x3, int32 layer,
 * uint32 schema, int32 x7, int64 x2), uint64 blob bytes, uint64 checksum,
 * then the state blob in the array format of the SSM.PREFIX state store:
 * uint32 version = 1, uint32 n_arrays = 1, uint32 ndim = 3, uint32 shape
 * {H, P, N}, uint32 dtype code 0 (fp32), H*P*N fp32 values.
 */
size_t ssm_receipt_bytes(int32_t nheads, int32_t headdim, int32_t dstate);

/*
 * Host only (no device work).  Serialize *r with the state (host float
 * [H][P][N] of r's dimensions); the checksum is computed here and written
 * back into r->checksum.  SSM_ERR_INVALID_ARG if cap is too small
 * (*written is then the size needed).
 */
ssm_status ssm_receipt_encode(ssm_receipt *r, const float *state, void *buf, size_t cap, size_t *written);

/*
 * Host only.  Parse and check a serialized checkpoint of len bytes: magic,
 * versions, the blob's array header against the receipt's dimensions, the
 * lengths and the checksum.  On SSM_OK fills *r and sets *state to the fp32
 * values inside buf (not necessarily 4-byte aligned).  SSM_ERR_SCHEMA for
 * anything that does not check.
 */
ssm_status ssm_receipt_decode(const void *buf, size_t len, ssm_receipt *r, const void **state);

/*
 * Checkpoint one slot as receipt + state blob (replay mode folds the log
 * first; A as for ssm_state_checkpoint).  Synchronous.
 */
ssm_status ssm_state_checkpoint_receipt(ssm_pool pool, int32_t slot, const float *A, const ssm_stream_identity *id,
                                        void *buf, size_t cap, size_t *written, ssm_stream_t stream);

/*
 * Resume one slot from a serialized checkpoint.  Refused with
 * SSM_ERR_SCHEMA, nothing changed, unless it decodes, its identity equals
 * *expect, and its schema, dtypes and dimensions equal the pool's: an
 * incompatible resume is rejected, never padded or truncated.  Then as
 * ssm_state_restore, with the position and chunk sequence of the receipt;
 * the slot's epoch counts the restore as a new occupancy.  Synchronous.
 */
ssm_status ssm_state_restore_receipt(ssm_pool pool, int32_t slot, const void *buf, size_t len,
                                     const ssm_stream_identity *expect, ssm_stream_t stream);

/* Read one slot's metadata (synchronous; no fold). */
ssm_status ssm_slot_info(ssm_pool pool, int32_t slot, ssm_slot_meta *meta, ssm_stream_t stream);

/*
 * Copy the current states of n slots (host int32[n]) into dst, device
 * float [n][H][P][N].  Copy mode resolves which snapshot is current; replay
 * mode copies the checkpoint as stored (logged tokens not folded in).
 */
ssm_status ssm_state_gather(ssm_pool pool, int32_t n, const int32_t *slots, float *dst,
                            ssm_stream_t stream);

/* ---------------------------------------------------------------- hot path */

/*
 * Chunked scan of n_seq packed sequences with state handoff ("Let the full
 * scan define legal chunking": scanning A + B equals scanning A, handing its
 * final state to B).  Sequence i owns tokens [cu_seqlens[i], cu_seqlens[i+1])
 * of x / dt / B / C / y and continues from slot slots[i]; its final state is
 * written back to that slot.  Lengths may be zero (an empty chunk consumes a
 * sequence number and changes nothing).
 *   cu_seqlens  host int32[n_seq + 1], non-decreasing, cu_seqlens[0] = 0
 *   slots       host int32[n_seq], distinct
 *   chunk_seq   host int64[n_seq]: must equal each slot's next chunk number;
 *               a smaller value is SSM_ERR_DUPLICATE, a larger one
 *               SSM_ERR_SEQUENCE (declared mismatch, nothing advances).
 * Replay pools require an empty log on each slot (device check).
 * bf16 pools with P = 64 and N = 128 take the tensor-core kernel when x, B,
 * C and y start on 16-byte boundaries, any other call the sequential one
 * (the same results within the tolerance).
 */
ssm_status ssm_scan_chunk(ssm_pool pool, int32_t n_seq, const int32_t *cu_seqlens, const int32_t *slots,
                          const int64_t *chunk_seq, const void *x, const void *dt, const void *B,
                          const void *C, const float *A, const float *D, void *y, ssm_stream_t stream);

/*
 * One decode token for each of `batch` requests, state updated in place
 * (batched single-token incremental update).  slots: host int32[batch],
 * distinct.  x [batch][H][P], dt [batch][H], B, C [batch][G][N],
 * y [batch][H][P].  position += 1.  Replay pools require an empty log.
 */
ssm_status ssm_decode_step(ssm_pool pool, int32_t batch, const int32_t *slots, const void *x,
                           const void *dt, const void *B, const void *C, const float *A,
                           const float *D, void *y, ssm_stream_t stream);

/*
 * n_steps decode tokens for the same `batch` requests with the token inputs
 * and outputs in page-locked host memory (cudaHostAlloc, cudaHostRegister):
 * step t is ssm_decode_step on row t of x [n_steps][batch][H][P],
 * dt [n_steps][batch][H], B, C [n_steps][batch][G][N] and
 * y [n_steps][batch][H][P] (dtypes as there); A and D stay device pointers.
 * The rows pass through two device staging sets owned by the pool: step
 * t + 1's inputs go up on one copy stream while step t decodes on `stream`
 * and step t - 1's output comes down on another, events ordering each reuse.
 * Copies start after the work queued on `stream` before the call.  The call
 * returns once everything is queued; `stream` is then ordered after the last
 * output copy, so y is complete once `stream` is synchronized, and the host
 * buffers must stay valid and unchanged until then.  Staging is allocated
 * the first time a call needs more than the pool holds (that call waits for
 * the previous staging to go idle).
 * SSM_ERR_INVALID_ARG: a null pointer, n_steps < 1, or x, dt, B, C or y not
 * page-locked host memory; slot errors as ssm_decode_step.  An error after
 * some steps were queued leaves those steps applied.
 */
ssm_status ssm_decode_steps_host(ssm_pool pool, int32_t batch, const int32_t *slots, int32_t n_steps,
                                 const void *x, const void *dt, const void *B, const void *C,
                                 const float *A, const float *D, void *y, ssm_stream_t stream);

/*
 * Speculative verify, copy flavour (copy pools only): each request walks its
 * n_tok = T + 1 tokens (the pending real token, then T drafts) from its
 * current state and keeps a full state copy after every token (Why
 * Speculative Decoding Slows Hybrid Mamba Models, The Problem: undo of a
 * rejected draft needs a saved state per draft).
 * x [batch][n_tok][H][P], dt [batch][n_tok][H], B, C [batch][n_tok][G][N],
 * y [batch][n_tok][H][P].  The current state is not modified.
 */
ssm_status ssm_verify_copy(ssm_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots,
                           const void *x, const void *dt, const void *B, const void *C,
                           const float *A, const float *D, void *y, ssm_stream_t stream);

/*
 * Speculative verify, ReplaySSM flavour (replay pools only): outputs come
 * from the checkpoint and the input log; no state is written in between
 * (The Fix: the unrolled update gives each output from the checkpoint and
 * the logged inputs):
 *   y_j[p] = exp(A * sum of all applied dt) * (C_j . h_ckpt[p,:])
 *          + sum_s exp(A * sum of dt applied after s) * dt_s * (C_j . B_s) * x_s[p]
 *          + D * x_j[p]
 * over the logged tokens and step tokens 0..j.  The step's x, dt and B are
 * staged after the log for the commit.  Arguments as ssm_verify_copy.
 * SSM_FOLD_IN_VERIFY pools: a request whose log holds W or more tokens has
 * them folded into its checkpoint here, in the same pass that reads the
 * checkpoint (one checkpoint read and one write instead of the commit's read
 * and write plus this call's read); its log then counts as empty and its
 * outputs come from the new checkpoint.  Such pools need x, B and C on
 * 16-byte boundaries (SSM_ERR_INVALID_ARG otherwise).
 */
ssm_status ssm_verify_replay(ssm_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots,
                             const void *x, const void *dt, const void *B, const void *C,
                             const float *A, const float *D, void *y, ssm_stream_t stream);

/*
 * Commit the last verify of each slot: c = 1 + accept[i] tokens (the real
 * token plus the drafts kept before the first miss).  accept: device
 * int32[batch] in [0, n_tok - 1] (outside: SSM_FLAG_BAD_ACCEPT, slot
 * skipped).  position += c.
 *   copy mode:   the state after token c - 1 becomes current (a pointer
 *                move into the snapshots; no state bytes are copied).
 *   replay mode: if log_len + c < W and !force_fold the c tokens are
 *                appended to the log; otherwise the log and the c tokens are
 *                folded into the checkpoint and the log empties (The Fix:
 *                the full state is written only when the window is full).
 *                SSM_FOLD_IN_VERIFY pools append the c tokens unless
 *                force_fold, and leave the fold of a full log to the next
 *                verify.  Rejected drafts never enter the log.
 * Every slot must have had a verify since its last commit or reset
 * (SSM_ERR_INVALID_STATE otherwise).  A is the same float [H] as the verify's.
 */
ssm_status ssm_state_commit(ssm_pool pool, int32_t batch, const int32_t *slots, const int32_t *accept,
                            int32_t force_fold, const float *A, ssm_stream_t stream);

/*
 * ssm_verify_replay without a pool and without any allocation.  The pages
 * have no counterpart to this entry point: it is for callers that cannot
 * call cudaMalloc -- a serving engine whose caching allocator owns all
 * device memory, or a plugin that is handed only the buffers its host
 * runtime manages -- and so cannot create a pool.  It runs the same kernels
 * as ssm_verify_replay.
 * The caller owns every buffer; request i uses row i of each (Wc = window - 1 + n_tok):
 *   ckpt     device float [batch][H][P][N], the checkpoints (read only)
 *   log_x    device [batch][Wc][H][P] (input dtype)
 *   log_dt   device float [batch][Wc][H]
 *   log_B    device [batch][Wc][G][N] (input dtype)
 *   log_len  device int32 [batch], logged tokens per request, each in [0, window - 1]
 *   x, dt, B, C, A, D, y   as ssm_verify_replay, [batch][n_tok][...]
 *   flags    device uint32: SSM_FLAG_* bits are ORed in, never cleared
 * Like ssm_verify_replay it writes the step's x, dt and B after each log
 * (entries log_len .. log_len + n_tok - 1), so appending c accepted tokens
 * is log_len += c; folding into ckpt is the caller's business.
 * Its scratch is a 4 MiB array inside the library, held by every GPU that
 * loads it until the process exits: batch <= 1024 and
 * batch * G * n_tok * Wc4 <= SSM_STATIC_SCRATCH_FLOATS, with Wc4 = Wc rounded
 * up to a multiple of 4, else
 * SSM_ERR_INVALID_ARG.  The first call on a device looks up the array's
 * device address (once per device, with that device current, and again if
 * the device's context has changed since, as after cudaDeviceReset); make
 * that first call before any stream capture.  All calls share the array,
 * which keeps the last call's contents: calls that overlap on the GPU race.
 * Launches are sized by the device's SM count, as the pool's are;
 * ssm_last_path(NULL) names the kernel path of the calling thread's last
 * call.  Asynchronous on stream.
 */
#define SSM_STATIC_SCRATCH_FLOATS 1047552
ssm_status ssm_verify_replay_static(int32_t batch, int32_t n_tok, int32_t nheads, int32_t headdim, int32_t dstate,
                                    int32_t ngroups, int32_t window, int32_t input_dtype, int32_t dt_dtype,
                                    const float *ckpt, void *log_x, float *log_dt, void *log_B,
                                    const int32_t *log_len, const void *x, const void *dt, const void *B,
                                    const void *C, const float *A, const float *D, void *y, uint32_t *flags,
                                    ssm_stream_t stream);

/* ------------------------------------------------------------- diagnostics */

/* Read (and if clear != 0, clear) the pool's sticky device flags.  Synchronous. */
ssm_status ssm_pool_status(ssm_pool pool, uint32_t *flags_out, int32_t clear, ssm_stream_t stream);

/* Name of the kernel path the last hot-path call used (static string); with
 * pool == NULL, that of the calling thread's last ssm_verify_replay_static. */
const char *ssm_last_path(ssm_pool pool);

/* Static text of a status code. */
const char *ssm_status_string(ssm_status s);

/* Bytes of device memory the pool holds. */
size_t ssm_pool_bytes(ssm_pool pool);

/*
 * For tests of the failure path: the pool's next replay verify on the tensor
 * cores withholds the per-item loads of one item in its first CTA, so that
 * the waits on them run out (each bounded at about a second).  That CTA's
 * roles then leave, the call's outputs for that item are not written, and
 * the pool's flags report SSM_FLAG_TIMEOUT; nothing faults and the pool stays
 * usable.  One-shot: the verify after it runs normally.  SSM_ERR_INVALID_ARG
 * without a pool.
 */
ssm_status ssm_debug_stall_next_verify(ssm_pool pool);

#ifdef __cplusplus
}
#endif

#endif /* SSM_STATE_H */
