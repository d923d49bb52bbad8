/*
 * librglru — the RG-LRU gated linear recurrence (the Hawk / Griffin recurrent layer),
 * forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operation (titles of the pages this library restates):
 *   [P1] "Fattori comparison" — the operator's inputs (recurrent input x, both raw gate
 *        logits, a_param = Lambda) and its fused steps: sigmoid gates, softplus(a_param) and
 *        the dynamic decay, the stationary square-root multiplier, the input-gated write,
 *        the state-stationary recurrence, and a backward of reverse recurrence plus pointwise
 *        derivatives; the block-diagonal gate projections that feed it (first paragraph);
 *        the "semantic limits" list that defines canonical resets (segment_pos / reset mask,
 *        m = 1 at reset tokens) and the nonzero initial state; and the closing paragraph
 *        (exact parallel chunked forward/backward with partial chunks).
 *   [P2] "public_fattori_h800.json" — the benchmark record: shape B4 T2048 W2048, BF16 with
 *        an FP32 recurrent carry, the restricted contract (zero initial state, no resets),
 *        and the gradients it checks (x, both gate logits, a_param).
 *   [P3] "linear_attention.reference" — small differentiable reference forms of other gated
 *        linear recurrences; their signatures pack variable-length sequences into one row by
 *        cu_seqlens offsets, with an initial state per sequence and the final states returned.
 *
 * Math (per batch row b, channel w, token t; c = 8 is fixed by the specification):
 *   r = sigmoid(lr), i = sigmoid(li), log a = -8 r softplus(Lambda_w), a = exp(log a)
 *   canonical mode: at a reset token abar = 0 and m = 1, else abar = a, m = sqrt(1 - a^2);
 *                   the state before token 0 is h0 (NULL = zeros)
 *   restricted mode: abar = a and m = sqrt(1 - a^2) on every token, zero initial state
 *   h_t = abar h_{t-1} + m i x,  y_t = h_t,  hT = h_{T-1}
 *   gate logits (block-diagonal, W = nblk * k, weights stored (in, out)):
 *     lr[., blk*k + j] = sum_i x[., blk*k + i] Wa[blk][i][j] + ba[blk*k + j]   (li: Wx, bx)
 *
 * Conventions for every call:
 *   - Layout: activations are [B, T, W] row-major (W contiguous); reset_mask (uint8) and
 *     segment_pos (int32) are [B, T]; h0, hT, dhT, dh0 are [B, W] float32; Lambda, ba, bx,
 *     dLambda, dba, dbx are [W] float32; Wa, Wx, dWa, dWx are [nblk, k, k] (in, out).
 *   - Dtypes: shape.io is the dtype of x, y, lr, li, dy and (bf16 I/O) of Wa/Wx; shape.grad is
 *     the dtype of dx, dlr, dli.  Everything else is float32.  The carry is always float32.
 *   - Ownership: the caller owns every buffer (device memory unless stated), including the
 *     `saved` and `workspace` scratch sized by rglru_saved_bytes / rglru_workspace_bytes.
 *     The library allocates nothing, never synchronises, and enqueues all work on `stream`.
 *   - Alignment: every pointer 16-byte aligned; W * sizeof(io) and W * sizeof(grad) must be
 *     multiples of 16 bytes.  W need not be a multiple of 64; T >= 1 need not be a multiple
 *     of any chunk size.
 *   - Resets: at most one of reset_mask (nonzero = reset) / segment_pos (== 0 = reset), and
 *     only in canonical mode; restricted mode takes neither and no h0.
 *   - Errors: arguments are validated on the host before any launch (RGLRU_ERR_INVALID_ARG,
 *     RGLRU_ERR_UNSUPPORTED); launch failures return RGLRU_ERR_CUDA.  The cross-chunk
 *     look-back waits are bounded; a wait that runs out sets a status word inside `saved`
 *     or `workspace`, which rglru_sync_status reports as RGLRU_ERR_TIMEOUT.
 *   - Gradient outputs are written, not accumulated, except rglru_gate_proj_backward's dx.
 */
#ifndef LIBRGLRU_H_
#define LIBRGLRU_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *rglru_stream;

typedef enum {
  RGLRU_OK = 0,
  RGLRU_ERR_INVALID_ARG = 1, /* null / misaligned pointer, inconsistent shape or mode */
  RGLRU_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement */
  RGLRU_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  RGLRU_ERR_TIMEOUT = 4      /* a bounded cross-chunk wait ran out (see rglru_sync_status) */
} rglru_status;

typedef enum { RGLRU_CANONICAL = 0, RGLRU_RESTRICTED = 1 } rglru_mode;
typedef enum { RGLRU_F32 = 0, RGLRU_BF16 = 1 } rglru_dtype;

typedef struct {
  int32_t B, T, W, nblk; /* batch, tokens, width, gate blocks (k = W / nblk) */
  int32_t io;            /* rglru_dtype of activations / logits / weights */
  int32_t grad;          /* rglru_dtype of dx, dlr, dli */
  int32_t mode;          /* rglru_mode */
} rglru_shape;

/* Human-readable name of a status code (static storage). */
const char *rglru_status_string(rglru_status s);

/* Bytes of the `saved` buffer a forward call fills and the matching backward reads
 * (float32 chunk-boundary states plus the forward's look-back scratch; for a fused call on a
 * shape the one-kernel fused path does not take, also the gate logits, as float32 or as bf16
 * hi + lo planes; for a packed-sequence call, also its token indices).  A buffer filled
 * by rglru_forward is read by rglru_backward; one filled by rglru_fused_forward by
 * rglru_fused_backward.  Sized for the current device.  0 on an invalid shape. */
size_t rglru_saved_bytes(const rglru_shape *shape);

/* Bytes of the `workspace` scratch taken by rglru_backward, rglru_gate_proj_backward,
 * rglru_fused_backward and rglru_fused_backward_varlen (the maximum over them).  Sized for the
 * current device.  0 on an invalid shape. */
size_t rglru_workspace_bytes(const rglru_shape *shape);

/* Block-diagonal gate projections [P1 first paragraph; P2 "protocol.scope"]:
 *   lr = x_blk @ Wa[blk] + ba,  li = x_blk @ Wx[blk] + bx   for every gate block.
 * x, Wa, Wx, lr, li in shape.io; ba, bx float32 (NULL = zero bias).  Float32 accumulation. */
rglru_status rglru_gate_proj(const rglru_shape *shape, const void *x, const void *Wa,
                             const float *ba, const void *Wx, const float *bx, void *lr,
                             void *li, rglru_stream stream);

/* Recurrence forward [P1 fused-steps list, semantic-limits list, closing paragraph]:
 * gates, decay, multiplier, write and an exact chunked scan (float32 carry).
 * Outputs y (shape.io), hT (float32, may be NULL) and `saved` (rglru_saved_bytes). */
rglru_status rglru_forward(const rglru_shape *shape, const void *x, const void *lr,
                           const void *li, const float *Lambda, const uint8_t *reset_mask,
                           const int32_t *segment_pos, const float *h0, void *y, float *hT,
                           void *saved, rglru_stream stream);

/* Recurrence backward [P1 "reverse recurrence and pointwise derivatives"; P2 checked
 * gradients]: recomputes the gates from the saved chunk states, runs the reverse scan of
 * g = dL/dh and writes dx (direct term only: g m i), dlr, dli (shape.grad), dLambda
 * (float32, reduced on device over batch and time) and dh0 (float32, may be NULL; zero in
 * restricted mode).  dhT may be NULL (zero).  `saved` must come from rglru_forward with the
 * same inputs; `workspace` holds rglru_workspace_bytes. */
rglru_status rglru_backward(const rglru_shape *shape, const void *dy, const float *dhT,
                            const void *x, const void *lr, const void *li, const float *Lambda,
                            const uint8_t *reset_mask, const int32_t *segment_pos,
                            const float *h0, const void *saved, void *dx, void *dlr, void *dli,
                            float *dLambda, float *dh0, void *workspace, rglru_stream stream);

/* Backward of the gate projections [P2 "protocol.scope" includes the projections]:
 *   dx += dlr Wa^T + dli Wx^T (per block; ACCUMULATES into dx, shape.grad),
 *   dWa = x^T dlr, dWx = x^T dli (float32 [nblk,k,k]), dba = sum dlr, dbx = sum dli.
 * dlr, dli in shape.grad; x, Wa, Wx in shape.io.  dba / dbx may be NULL. */
rglru_status rglru_gate_proj_backward(const rglru_shape *shape, const void *dlr,
                                      const void *dli, const void *x, const void *Wa,
                                      const void *Wx, void *dx, float *dWa, float *dba,
                                      float *dWx, float *dbx, void *workspace,
                                      rglru_stream stream);

/* Recurrence forward that allocates nothing and takes no `saved` buffer.  The pages have no
 * counterpart; it exists for callers that may not allocate device memory at all (code
 * running inside someone else's stream capture, under a fixed memory pool, in a real-time
 * loop that must not touch the allocator, or in a plugin handed only its inputs and
 * outputs).  Same arguments and outputs as rglru_forward minus `saved` (nothing is kept for
 * a backward).  The look-back scratch is a static device array of
 * RGLRU_NOALLOC_SCRATCH_BYTES per GPU, held from library load until process exit; a shape
 * needing more (about 0.75 * B*T*W bytes, e.g. B4 T2048 W2048 fits) returns
 * RGLRU_ERR_UNSUPPORTED.  The first call on each device finds the array's device address
 * (cudaGetSymbolAddress) and should come before any stream capture.  All calls share the
 * array; calls whose work overlaps on the GPU race on it.  A look-back wait that runs out
 * marks the status word inside the array (the results of that call are then wrong, and the
 * call itself still returns RGLRU_OK): read it with rglru_forward_noalloc_status before the
 * next call, which clears it. */
#define RGLRU_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
rglru_status rglru_forward_noalloc(const rglru_shape *shape, const void *x, const void *lr,
                                   const void *li, const float *Lambda,
                                   const uint8_t *reset_mask, const int32_t *segment_pos,
                                   const float *h0, void *y, float *hT, rglru_stream stream);

/* Status of the last rglru_forward_noalloc call on the current device (no counterpart on the
 * pages): synchronises `stream`, then reads the status word of the static scratch;
 * RGLRU_ERR_TIMEOUT if a bounded look-back wait of that call ran out, RGLRU_OK otherwise
 * (RGLRU_ERR_CUDA if the read fails).  Allocates nothing. */
rglru_status rglru_forward_noalloc_status(rglru_stream stream);

/* Fused forward: the projections folded into the recurrence [P1 closing paragraph credits
 * the fusion strategy; the logits are never rounded to the I/O dtype].  Same outputs as
 * rglru_gate_proj followed by rglru_forward, without writing the logits. */
rglru_status rglru_fused_forward(const rglru_shape *shape, const void *x, const void *Wa,
                                 const float *ba, const void *Wx, const float *bx,
                                 const float *Lambda, const uint8_t *reset_mask,
                                 const int32_t *segment_pos, const float *h0, void *y,
                                 float *hT, void *saved, rglru_stream stream);

/* Fused backward: all gradients of the fused layer — dx (direct term plus both projections,
 * shape.grad), dWa, dWx, dba, dbx, dLambda (float32), dh0 (may be NULL).  `saved` must come
 * from rglru_fused_forward with the same inputs. */
rglru_status rglru_fused_backward(const rglru_shape *shape, const void *dy, const float *dhT,
                                  const void *x, const void *Wa, const float *ba,
                                  const void *Wx, const float *bx, const float *Lambda,
                                  const uint8_t *reset_mask, const int32_t *segment_pos,
                                  const float *h0, const void *saved, void *dx, float *dWa,
                                  float *dba, float *dWx, float *dbx, float *dLambda,
                                  float *dh0, void *workspace, rglru_stream stream);

/* Packed variable-length sequences [the packing boundary of P3 "linear_attention.reference"
 * (cu_seqlens offsets, per-sequence initial and final states), applied to this layer]: one
 * row of shape.T tokens (shape.B must be 1, canonical mode) holds num_seqs sequences, sequence
 * s on tokens [cu_seqlens[s], cu_seqlens[s+1]) (device int32 [num_seqs + 1], non-decreasing
 * from 0 to T; a malformed array gives wrong results, never an out-of-bounds access).  Each
 * sequence is the layer on its own: its first token continues from h0[s] (float32
 * [num_seqs][W], NULL = zeros) without a reset, and hT[s] (may be NULL) is the state after its
 * last token; an empty sequence has hT[s] = h0[s].  Same computation as rglru_fused_forward on
 * each sequence as a row of its own.  bf16 I/O on the tensor cores (k a multiple of 16 up to
 * 160; k = 128 in one fused kernel, other k through the tensor-core projections), float32 I/O
 * on the CUDA cores (any k); other bf16 shapes give RGLRU_ERR_UNSUPPORTED.  `saved`
 * (rglru_saved_bytes of the shape) also keeps the token indices for the backward. */
rglru_status rglru_fused_forward_varlen(const rglru_shape *shape, const void *x, const void *Wa,
                                        const float *ba, const void *Wx, const float *bx,
                                        const float *Lambda, const int32_t *cu_seqlens,
                                        int32_t num_seqs, const float *h0, void *y, float *hT,
                                        void *saved, rglru_stream stream);

/* Gradients of rglru_fused_forward_varlen: dx, dWa, dba, dWx, dbx, dLambda as in
 * rglru_fused_backward; dhT (float32 [num_seqs][W], NULL = zeros) is the gradient arriving at
 * each sequence's final state; dh0 (may be NULL) receives each sequence's initial-state
 * gradient (dhT[s] for an empty one).  `saved` must come from rglru_fused_forward_varlen with
 * the same inputs and cu_seqlens. */
rglru_status rglru_fused_backward_varlen(const rglru_shape *shape, const void *dy,
                                         const float *dhT, const void *x, const void *Wa,
                                         const float *ba, const void *Wx, const float *bx,
                                         const float *Lambda, const int32_t *cu_seqlens,
                                         int32_t num_seqs, const float *h0, const void *saved,
                                         void *dx, float *dWa, float *dba, float *dWx,
                                         float *dbx, float *dLambda, float *dh0,
                                         void *workspace, rglru_stream stream);

/* One decode step with carried states [P1 semantic-limits list: an initial state and T = 1,
 * both of which the prior art rejects]: for every row b the layer's forward of one token from
 * the state h_in,
 *   lr = x_blk @ Wa[blk] + ba,  li = x_blk @ Wx[blk] + bx,  r = sigmoid(lr), i = sigmoid(li),
 *   a = exp(-8 r softplus(Lambda)),  h_out = abar h_in + m i x,  y = h_out,
 * with abar = 0 and m = 1 on a canonical reset row, abar = a and m = sqrt(1 - a^2) otherwise;
 * the same values as rglru_fused_forward with T = 1 and h0 = h_in.  shape.T must be 1.
 * x, y [B, W] and Wa, Wx in shape.io; h_in, h_out [B, W] float32 (h_in NULL = zeros; h_out
 * may be h_in, updated in place); reset uint8 [B] (nonzero = the token starts a segment; NULL
 * = none; canonical mode only); ba, bx may be NULL.  k = W / nblk <= 512 (else
 * RGLRU_ERR_UNSUPPORTED).  One kernel, no scratch, launched with programmatic stream
 * serialisation: its launch and set-up may overlap the end of the kernel before it on the
 * stream, but it reads and writes no memory before that kernel has completed, so stream order
 * holds for every argument. */
rglru_status rglru_step(const rglru_shape *shape, const void *x, const void *Wa,
                        const float *ba, const void *Wx, const float *bx, const float *Lambda,
                        const uint8_t *reset, const float *h_in, void *y, float *h_out,
                        rglru_stream stream);

/* Synchronises `stream`, then reads the status word at the start of a `saved` or
 * `workspace` buffer (device pointer) last used on it: RGLRU_ERR_TIMEOUT if a bounded
 * look-back wait ran out, RGLRU_OK otherwise (RGLRU_ERR_CUDA if the read fails). */
rglru_status rglru_sync_status(const void *saved_or_workspace, rglru_stream stream);

/* Test hook for failure detection (no counterpart on the pages): `spin_limit` > 0 replaces
 * the number of polls a look-back wait makes before it gives up (default ~2^22), and
 * `drop_tile` >= 0 makes the scan tile with that ticket skip publishing, so its successors'
 * waits run out.  (0, -1) restores the defaults.  Process-wide; not thread-safe. */
void rglru_debug_lookback(int32_t spin_limit, int32_t drop_tile);

/* Profiling hook (no counterpart on the pages): when `start` and `stop` (cudaEvent_t handles
 * owned by the caller) are both non-null, the next rglru_fused_forward or
 * rglru_fused_backward call that runs its tensor-core kernel records `start` on the call's
 * stream just before that kernel's launch and `stop` just after it, then forgets both; so a
 * caller can time that kernel alone with cudaEventElapsedTime.  (NULL, NULL) cancels.
 * Process-wide; not thread-safe. */
void rglru_debug_kernel_events(void *start, void *stop);

/* Which kernels rglru_fused_forward / rglru_fused_backward run for `shape` (no counterpart on
 * the pages): a short static description, "invalid shape" if the shape is rejected. */
const char *rglru_fused_path(const rglru_shape *shape);

/* Launch accounting (no counterpart on the pages): the number of CUDA kernels this library
 * has enqueued since the process started (memsets excluded).  Lets a caller count the
 * kernels behind a timed region.  Process-wide, atomic. */
uint64_t rglru_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* LIBRGLRU_H_ */
