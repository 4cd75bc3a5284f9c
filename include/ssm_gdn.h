/*
 * ssm_gdn.h -- the gated delta rule behind the same kind of C ABI: a pool of
 * per-slot fp32 states with a replay log, in-place decode, ReplaySSM verify
 * and commit ("Why Speculative Decoding Slows Hybrid Mamba Models", When the
 * layer is a different kind of recurrence: the replay trick needs an update
 * that unrolls as a decay plus a sum, and Gated DeltaNet's does; State
 * precision: keep the state in fp32).
 *
 * The recurrence, per value head h with key head g(h) = h / (H / G) (the
 * published gated delta rule; the pages name it without printing it):
 *   S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t = S_t q_t
 * S is fp32 [dv][dk].  q and k are used as given (normalizing them is the
 * caller's part).
 *
 * Layouts (row-major, innermost last; DEVICE pointers unless marked host):
 *   state of a slot   float [H][dv][dk]
 *   q, k              [tokens][G][dk]      input dtype
 *   v, y              [tokens][H][dv]      input dtype
 *   g, beta           float [tokens][H]    (g = log of the gate, <= 0)
 * "tokens" is the batch for a decode step and [batch][n_tok] for a verify.
 * q, k, v and y must start on 16-byte boundaries (else SSM_ERR_INVALID_ARG).
 *
 * Ownership, errors and asynchrony follow ssm_state.h: the pool owns its
 * memory; host-side checks return before any work is queued; device-side
 * errors (non-finite input, poisoned slot, accept out of range) set sticky
 * SSM_FLAG_* bits, poison the slot and skip its work; calls are
 * asynchronous on the given stream unless marked synchronous.  Supported
 * shapes: dk 64 or 128, dv a multiple of 4 up to 256, G dividing H,
 * max_tokens 1..32, window 1..32, and one key head's verify working set in
 * a CTA's shared memory: 4 * (L (dk + dv) + T dk + hpg L (T + 2)) bytes with
 * L = window - 1 + max_tokens, T = max_tokens, hpg = H / G (else
 * ssm_gdn_init returns SSM_ERR_INVALID_ARG).
 */
#ifndef SSM_GDN_H
#define SSM_GDN_H

#include "ssm_state.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t nheads;      /* H, value heads */
    int32_t nkheads;     /* G, key heads, divides H */
    int32_t dk;          /* key dimension: 64 or 128 */
    int32_t dv;          /* value dimension: multiple of 4, <= 256 */
    int32_t input_dtype; /* q, k, v and y: SSM_DTYPE_F32 or SSM_DTYPE_BF16 */
    int32_t window;      /* replay window W, 1..32 */
    int32_t max_tokens;  /* largest n_tok of one verify step, 1..32 */
} ssm_gdn_config;

typedef struct ssm_gdn_pool_s *ssm_gdn_pool;

/* n_slots states, zero or copied from init_state (device float
 * [n_slots][H][dv][dk]), each at position 0 with an empty log.  Allocates
 * the log (W - 1 + max_tokens entries a slot) and the verify scratch.
 * Synchronous.  *out is set only on SSM_OK. */
ssm_status ssm_gdn_init(const ssm_gdn_config *cfg, int32_t n_slots, const float *init_state, ssm_stream_t stream,
                        ssm_gdn_pool *out);
ssm_status ssm_gdn_destroy(ssm_gdn_pool pool);

/* Slots (host int32[n]): state := 0, log emptied, position := 0, poison cleared. */
ssm_status ssm_gdn_reset(ssm_gdn_pool pool, const int32_t *slots, int32_t n, ssm_stream_t stream);

/* One token per request, state updated in place (the log must be empty,
 * else SSM_FLAG_LOG_NOT_EMPTY).  slots: host int32[batch], distinct.
 * q, k [batch][G][dk], v [batch][H][dv], g, beta [batch][H], y [batch][H][dv]. */
ssm_status ssm_gdn_decode_step(ssm_gdn_pool pool, int32_t batch, const int32_t *slots, const void *q,
                               const void *k, const void *v, const float *g, const float *beta, void *y,
                               ssm_stream_t stream);

/* ReplaySSM verify: the outputs of n_tok step tokens from the checkpoint and
 * the log, with no state written (The Fix).  For the output at position m
 * (the log's K tokens, then the step tokens): start from u = q_m and walk
 * i = m .. 1, taking the weight beta_i (k_i . u) of v_i and then
 * u <- exp(g_i) (u - beta_i k_i (k_i . u)); the output is S_ckpt u plus the
 * weighted v_i.  The step's k, v, g and beta are staged after the log for
 * the commit.  Shapes as decode with [batch][n_tok] tokens.  bf16 pools with
 * dk = dv = 128 and 4 <= n_tok <= 32 take the checkpoint product S u on the tensor
 * cores (fp32 operands read as tf32: at most 2^-10 of each product) and add
 * the weighted logged values rounded to bf16 (2^-9 of that term), both below
 * the bf16 rounding of y; other pools the exact fp32 CUDA-core kernels. */
ssm_status ssm_gdn_verify_replay(ssm_gdn_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots,
                                 const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 void *y, ssm_stream_t stream);

/* Commit the last verify of each slot: c = 1 + accept[i] (device int32, in
 * [0, n_tok - 1]) tokens.  If log_len + c < W and !force_fold they join the
 * log; otherwise the log and they are applied to the checkpoint in order
 * and the log empties.  Rejected drafts never enter the log.  position += c.
 * bf16 pools with dk = dv = 128 and W - 1 + max_tokens <= 32 fold in the
 * chunked form on the tensor cores (Gated DeltaNet's WY form: the checkpoint
 * times the keys, then a rank-M update from a triangular solve; the
 * checkpoint's own decay is applied in fp32 and only the update takes tf32
 * operands, at most 2^-10 of each product); other pools fold token by token
 * in fp32 on the CUDA cores. */
ssm_status ssm_gdn_commit(ssm_gdn_pool pool, int32_t batch, const int32_t *slots, const int32_t *accept,
                          int32_t force_fold, ssm_stream_t stream);

/* Copy n checkpoints (host int32[n] slots) into dst, device float [n][H][dv][dk]. */
ssm_status ssm_gdn_gather(ssm_gdn_pool pool, int32_t n, const int32_t *slots, float *dst, ssm_stream_t stream);

/* Position, log length and flags (bit 0 poisoned) of one slot.  Synchronous. */
ssm_status ssm_gdn_slot_info(ssm_gdn_pool pool, int32_t slot, int64_t *position, int32_t *log_len,
                             uint32_t *flags, ssm_stream_t stream);

/* Read (and if clear != 0, clear) the pool's sticky device flags.  Synchronous. */
ssm_status ssm_gdn_status(ssm_gdn_pool pool, uint32_t *flags_out, int32_t clear, ssm_stream_t stream);

/* Kernel path of the pool's last verify: "gdn_verify_tc" (tensor cores),
 * "gdn_verify" (CUDA cores) or "none".  The string is static. */
const char *ssm_gdn_last_path(ssm_gdn_pool pool);

/* Fold path of the pool's last commit: "gdn_fold_tc" (tensor cores),
 * "gdn_fold" (CUDA cores) or "none".  The string is static. */
const char *ssm_gdn_last_commit_path(ssm_gdn_pool pool);

#ifdef __cplusplus
}
#endif

#endif /* SSM_GDN_H */
