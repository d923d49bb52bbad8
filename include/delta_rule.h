/*
 * delta_rule.h — the gated delta rule (GDN with one decay per value head, KDA with one decay
 * per key channel), forward and backward, on one NVIDIA GB300 (sm_103a).  Compiled into
 * librglru; the same status codes, dtypes and stream conventions as librglru.h.
 *
 * Source of the operation: [P3] "linear_attention.reference", entry
 * recurrent_delta_rule_reference: a token-by-token form of the rule whose decay is one number
 * per value head (GDN) or one per key channel (KDA); q, k [B, T, Hk, Dk],
 * v [B, T, Hv, Dv], beta [B, T, Hv], g [B, T, Hv] (GDN) or [B, T, Hv, Dk] (KDA); the state
 * [N, Hv, Dk, Dv] or, value first, [N, Hv, Dv, Dk]; output and final state returned, gradients
 * through the initial state; gates are natural logarithms; q, k, v, beta already normalised or
 * activated; packed sequences by cu_seqlens.  The page prints no formula; the reading taken
 * (per sequence, value head h reading key head h / (Hv / Hk), token t; S is [Dk, Dv]):
 *
 *   S' = D_t S,   D_t = exp(g_t) (GDN) or diag(exp(g_t)) (KDA)
 *   u  = beta_t (v_t - S'^T k_t)
 *   S  = S' + k_t u^T,   o_t = scale S^T q_t   (scale: given, usually Dk^-1/2)
 *
 * Conventions for every call:
 *   - Layout: q, k [B, T, Hk, Dk], v, o [B, T, Hv, Dv] row-major in shape.io (float32 or bf16);
 *     g, beta float32; states float32 [N, Hv, Dk, Dv] (state_v_first: [N, Hv, Dv, Dk]).
 *     Without cu_seqlens N = B and sequence n is batch row n; with it B must be 1 and sequence
 *     n is tokens [cu_seqlens[n], cu_seqlens[n+1]) of row 0 (device int32 [N + 1], from 0 to T,
 *     non-decreasing; a malformed array gives wrong results, never an out-of-bounds access).
 *   - Supported: Dk in {32, 64, 128}, 1 <= Dv <= 128 with Dv x sizeof(io) a multiple of 16
 *     bytes (rows of v come in by 16-byte copies), Hv a multiple of Hk, every pointer 16-byte
 *     aligned; else RGLRU_ERR_UNSUPPORTED (sizes) or RGLRU_ERR_INVALID_ARG.
 *   - Ownership: the caller allocates every buffer, `saved` and `workspace` sized by the
 *     queries below; the library never allocates or synchronises.  All work is enqueued on
 *     `stream`.  Argument checks run on the host before any launch; launch failures return
 *     RGLRU_ERR_CUDA.
 */
#ifndef DELTA_RULE_H
#define DELTA_RULE_H

#include <stddef.h>
#include <stdint.h>

#include "librglru.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int B, T, Hk, Hv, Dk, Dv;
  rglru_dtype io;     /* storage type of q, k, v, o (and of do) */
  int kda;            /* 0: g is [B, T, Hv] (GDN); 1: g is [B, T, Hv, Dk] (KDA) */
  int state_v_first;  /* 0: states [N, Hv, Dk, Dv]; 1: [N, Hv, Dv, Dk] */
} delta_shape;

/* Bytes of the `saved` buffer that delta_rule_forward fills for delta_rule_backward (the
 * float32 state entering every 16-token block of every sequence and head) for `num_seqs`
 * sequences; 0 for an unsupported shape. */
size_t delta_rule_saved_bytes(const delta_shape *shape, int32_t num_seqs);

/* Bytes of the backward's scratch (per-value-head dq, dk when Hv > Hk); may be 0. */
size_t delta_rule_workspace_bytes(const delta_shape *shape);

/* Forward: o (shape.io) and, if hT is not NULL, the final states (float32) from the initial
 * states h0 (NULL = zeros).  `saved` (delta_rule_saved_bytes, may be NULL when no backward
 * follows) receives the block states for the backward.  cu_seqlens NULL: num_seqs must be B.
 * hT may equal h0 (states carried in place), which with T = 1 is a decode step. */
rglru_status delta_rule_forward(const delta_shape *shape, const void *q, const void *k,
                                const void *v, const float *g, const float *beta, float scale,
                                const int32_t *cu_seqlens, int32_t num_seqs, const float *h0,
                                void *o, float *hT, void *saved, rglru_stream stream);

/* Backward: with do (shape.io) the gradient of o and dhT (float32, NULL = zeros) that of the
 * final states, writes dq, dk [B, T, Hk, Dk], dv [B, T, Hv, Dv], dg (the shape of g), dbeta
 * [B, T, Hv] and, if not NULL, dh0 (the shape of the states), all float32.  `saved` must come
 * from delta_rule_forward with the same inputs; workspace: delta_rule_workspace_bytes (may be
 * NULL when that is 0). */
rglru_status delta_rule_backward(const delta_shape *shape, const void *q, const void *k,
                                 const void *v, const float *g, const float *beta, float scale,
                                 const int32_t *cu_seqlens, int32_t num_seqs, const float *h0,
                                 const void *saved, const void *dout, const float *dhT,
                                 float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                 float *dh0, void *workspace, rglru_stream stream);

/* FP8 (E4M3) quantize-dequantize of float32 key-first states [n_states][Dk][Dv] [P3 "FP8
 * state" entry: dynamic E4M3 QDQ, one scale per [Dk, block_v] tile, an all-zero tile with
 * scale one, partial value tiles valid; its gradient is the identity]: per tile amax, scale =
 * amax / 448 (1 if amax is 0), each value replaced by code * scale with code the E4M3 value
 * nearest value / scale (ties to even, saturating at +-448), all in float32.  out may equal
 * state (in place).  Any n_states, Dk, Dv, block_v >= 1. */
rglru_status delta_rule_state_fp8_qdq(const float *state, float *out, int64_t n_states,
                                      int Dk, int Dv, int block_v, rglru_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* DELTA_RULE_H */
