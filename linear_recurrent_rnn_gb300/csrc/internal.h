// Internal interfaces between librglru's host layer and its kernel translation units:
// buffer layouts of `saved` / `workspace`, kernel argument blocks and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/librglru.h"

namespace rglru {

// Tokens per scan chunk of the SIMT scan kernels: a warp owns 32 channels x SC tokens,
// each lane two channels x SUB tokens.
constexpr int SC = 16;
constexpr int SUB = 8;
// Look-back of the SIMT scan kernels.  Chunks are counted in processing order (from the start
// in the forward, from the end in the backward); every STEP-th chunk publishes its
// chunk-boundary state, and a chunk q applies the aggregates of the chunks after its anchor
// to the anchor's state, the anchor being the nearest publishing chunk at least DIST
// chunks back (or, for q < DIST, the initial state).  Tiles are handed out in chunk order
// and about a dozen chunks' tiles are resident at once, so the anchor's state has normally
// been published before it is asked for.  The carry each tile sees is a fixed expression of
// the inputs, independent of timing: the scan is bitwise deterministic.
// The backward keeps fewer tiles resident (more registers per thread) than the forward, so
// each direction has its own distance and step.
template <bool BWD>
struct LbPlan {
  static constexpr int DIST = BWD ? 12 : 8;
  static constexpr int STEP = BWD ? 4 : 2;
  static constexpr int MAX = DIST + STEP - 2;  // aggregates composed at most
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Dims {
  int B, T, W, nblk, k;
  int nC;  // scan chunks per row: ceil(T / SC)
  int ng;  // 32-channel groups: ceil(W / 32)
  size_t N;
  int io, grad, mode;
};

// Scan scratch: [0, zero_bytes) is cleared before each launch (status word, ticket, flags).
//   header: u32 status, u32 ticket (256 bytes)
//   flags  u32 [B][nC][ng]
//   carry  f32 [B][nC+1][W]   forward: state entering chunk c (c = nC: hT)
//                             backward: carry passed from chunk c to chunk c-1
//   agg    float2 [B][nC][W]  per-chunk affine aggregate (A, B)
//   part   f32 [B*nC][W]      backward only: per-chunk dLambda partial sums
struct ScanLayout {
  size_t flags, zero_bytes, carry, agg, part, total;
};

inline ScanLayout scan_layout_n(int B, int nC, int ng, int W, bool backward) {
  ScanLayout L;
  const size_t nflags = (size_t)B * nC * ng;
  L.flags = 256;
  L.zero_bytes = align_up(L.flags + nflags * 4, 256);
  L.carry = L.zero_bytes;
  L.agg = align_up(L.carry + (size_t)B * (nC + 1) * W * 4, 256);
  L.part = align_up(L.agg + (size_t)B * nC * W * 8, 256);
  L.total = backward ? align_up(L.part + (size_t)B * nC * W * 4, 256) : L.part;
  return L;
}

inline ScanLayout scan_layout(const Dims& d, bool backward) {
  return scan_layout_n(d.B, d.nC, d.ng, d.W, backward);
}

// ---------------------------------------------------------------- fused tensor-core kernels
// Gate-block width and tokens per tile of the fused kernels (the tile's MMA is M = 128
// channels, N = 64 tokens, K = 128).
constexpr int FUSED_K = 128;
constexpr int FUSED_C = 64;

inline int fused_chunks(const Dims& d) { return (d.T + FUSED_C - 1) / FUSED_C; }

// Look-back of the fused kernels (lookback.cuh): at most LB_SLOTS aggregates per look-back.
// The anchor is at least `dist` chunks back, dist = ceil(P / B) with P CTAs sharing a gate
// block's B * nC tiles in chunk order, so that the anchor's tile came at least one round of
// the tile loop earlier; anchors are every 2^shift chunks, the largest power of two with
// dist + 2^shift - 2 <= LB_SLOTS.
constexpr int LB_SLOTS = 8;
struct LookbackPlan {
  int dist, shift;
};
inline LookbackPlan lookback_plan(int P, int B) {
  int dist = (P + B - 1) / B;
  if (dist < 1) dist = 1;
  if (dist > LB_SLOTS + 1) dist = LB_SLOTS + 1;
  int shift = 0;
  while (dist + (2 << shift) - 2 <= LB_SLOTS) ++shift;
  return {dist, shift};
}
inline ScanLayout fused_layout(const Dims& d, bool backward) {
  return scan_layout_n(d.B, fused_chunks(d), d.ng, d.W, backward);
}
// Fused forward `saved`: the look-back scratch (its chunk-boundary states are where the
// backward starts), then, for packed variable-length sequences, two int32 [T] token indices:
// the sequence that starts at each token and the one that ends there (-1: none).
struct FusedFwdLayout {
  ScanLayout L;
  size_t seq_start, seq_end, total;
};
inline FusedFwdLayout fused_fwd_layout(const Dims& d) {
  FusedFwdLayout F;
  F.L = fused_layout(d, false);
  F.seq_start = align_up(F.L.total, 256);
  F.seq_end = align_up(F.seq_start + (size_t)d.T * 4, 256);
  F.total = align_up(F.seq_end + (size_t)d.T * 4, 256);
  return F;
}

// Packed variable-length sequences (one row, sequence s on tokens [cu[s], cu[s+1])): the
// per-sequence states and the token indices in `saved`.
struct Varlen {
  const int32_t* cu_seqlens;  // device [S + 1]
  int S;
  const int32_t* seq_start;   // [T]: s if sequence s (non-empty) starts at the token, else -1
  const int32_t* seq_end;     // [T]: s if sequence s ends at the token, else -1
  const float* h0;            // [S][W] or null (zeros)
  float* hT;                  // [S][W] or null (forward)
  const float* dhT;           // [S][W] or null (backward)
  float* dh0;                 // [S][W] or null (backward)
};
// Forward: fills the token indices and, for empty sequences, hT = h0 (one launch).
cudaError_t launch_seq_index(const Varlen& v, int T, int W, int32_t* seq_start,
                             int32_t* seq_end, cudaStream_t s);
// Backward: dh0 = dhT for empty sequences (the token indices are the forward's).
cudaError_t launch_seq_empty_dh0(const Varlen& v, int W, cudaStream_t s);

// Fused backward workspace: the reverse look-back scratch, then per-CTA partial sums (the
// kernel runs at most FUSED_MAX_CTAS CTAs, each owning one gate block): dWa / dWx partials
// [cta][2][k][k] and per-channel partials [cta][part (4)][3][k] (dLambda before the sigmoid,
// dba, dbx).
constexpr int FUSED_MAX_CTAS = 256;
struct FusedBwdLayout {
  ScanLayout L;
  size_t dw_part, vec_part, total;
};
inline FusedBwdLayout fused_bwd_layout(const Dims& d) {
  FusedBwdLayout F;
  F.L = scan_layout_n(d.B, fused_chunks(d), d.ng, d.W, false);
  F.dw_part = align_up(F.L.total, 256);
  F.vec_part = align_up(F.dw_part + (size_t)FUSED_MAX_CTAS * 2 * FUSED_K * FUSED_K * 4, 256);
  F.total = align_up(F.vec_part + (size_t)FUSED_MAX_CTAS * 4 * 3 * FUSED_K * 4, 256);
  return F;
}

// Split-K layout of the SIMT projection-weight gradient.
inline int dw_splits(const Dims& d) {
  const int tiles = ((d.k + 63) / 64) * ((d.k + 63) / 64) * d.nblk * 2;
  const long BT = (long)d.B * d.T;
  long s = (600 + tiles - 1) / tiles;
  const long smax = (BT + 255) / 256;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return (int)s;
}

// Token splits of the bias-gradient partial sums: about 600 CTAs of 512 channels (two per
// thread) x one gate, each split at least 64 tokens.
inline int db_splits(const Dims& d) {
  const long cols = (long)((d.W + 511) / 512) * 2;
  const long BT = (long)d.B * d.T;
  long s = (600 + cols - 1) / cols;
  const long smax = (BT + 63) / 64;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  if (s > 256) s = 256;
  return (int)s;
}

struct GateBwdLayout {
  size_t dw_part, db_part, total;
};

// The partials start past a 256-byte header: the first word of a workspace is the status word
// that the scan backward sets and rglru_sync_status reads, so a projection backward run after
// it on the same workspace must leave that word alone.
inline GateBwdLayout gate_bwd_layout(const Dims& d) {
  GateBwdLayout L;
  const int S = dw_splits(d);
  L.dw_part = 256;
  L.db_part = align_up(L.dw_part + (size_t)S * 2 * d.nblk * d.k * d.k * 4, 256);
  L.total = align_up(L.db_part + (size_t)db_splits(d) * 2 * d.W * 4, 256);
  return L;
}

// ---------------------------------------------------------------- kernel arguments
struct ScanFwdArgs {
  int B, T, W, nC, ng;
  const void* x;
  const void* lr;
  const void* li;
  const float* Lambda;
  const uint8_t* reset_mask;
  const int32_t* segment_pos;
  const float* h0;
  void* y;
  float* hT;
  uint8_t* scratch;  // `saved`
  ScanLayout L;
  int spin_limit, drop_tile;
  // packed sequences (Varlen; null seq_start: none): token indices, per-sequence states
  const int32_t* seq_start = nullptr;
  const int32_t* seq_end = nullptr;
  const float* h0s = nullptr;
  float* hTs = nullptr;
};

struct ScanBwdArgs {
  int B, T, W, nC, ng;
  const void* dy;
  const float* dhT;
  const void* x;
  const void* lr;
  const void* li;
  const float* Lambda;
  const uint8_t* reset_mask;
  const int32_t* segment_pos;
  const float* h0;
  const float* fwd_carry;  // from `saved`: state entering each chunk
  void* dx;
  void* dlr;
  void* dli;
  size_t dl_plane;   // DT_SPLIT gradients: elements between the hi and lo planes
  float* dLambda;
  float* dh0;
  uint8_t* scratch;  // `workspace`
  ScanLayout L;
  int spin_limit, drop_tile;
  // packed sequences (Varlen; null seq_start: none)
  const int32_t* seq_start = nullptr;
  const int32_t* seq_end = nullptr;
  const float* h0s = nullptr;
  const float* dhTs = nullptr;
  float* dh0s = nullptr;
};

// Adds n to the process-wide count of kernels enqueued (rglru_kernel_launches).
void note_launches(unsigned n);
// The failure-injection settings of rglru_debug_lookback (look-back poll limit, dropped tile).
int debug_spin_limit();
int debug_drop_tile();

// rglru_debug_kernel_events: record the caller's events around the next tensor-core kernel.
extern cudaEvent_t g_kernel_events[2];
void kernel_event_before(cudaStream_t s);
void kernel_event_after(cudaStream_t s);

// Host-side validation shared by the entry points (defined in api.cu).
rglru_status make_dims(const rglru_shape* s, Dims* d);
bool req(const void* p);  // non-null and 16-byte aligned
bool opt(const void* p);  // null or 16-byte aligned
rglru_status check_resets(const Dims& d, const uint8_t* rm, const int32_t* sp, const float* h0);
rglru_status cuda_status(cudaError_t e);
ScanFwdArgs fwd_args(const Dims& d, const void* x, const void* lr, const void* li,
                     const float* Lambda, const uint8_t* rm, const int32_t* sp, const float* h0,
                     void* y, float* hT, void* saved);

// dtype codes used by the launchers (io of x/y/dy, of the logits, of dx, of dlr/dli);
// DT_SPLIT: float32 values written as bf16 hi and lo planes (SplitBf16)
enum { DT_F32 = RGLRU_F32, DT_BF16 = RGLRU_BF16, DT_SPLIT = 2 };

cudaError_t launch_scan_fwd(const ScanFwdArgs& a, int xt, int lt, bool canonical,
                            cudaStream_t s);
cudaError_t launch_scan_bwd(const ScanBwdArgs& a, int xt, int lt, int dxt, int dlt,
                            bool canonical, cudaStream_t s);

// Fused forward on tensor cores (bf16 I/O, k == FUSED_K).  Returns cudaErrorNotSupported
// when the shape is outside what the kernel covers (the caller then composes).
cudaError_t launch_fused_fwd(const Dims& d, const void* x, const void* Wa, const float* ba,
                             const void* Wx, const float* bx, const float* Lambda,
                             const uint8_t* rm, const int32_t* sp, const float* h0, void* y,
                             float* hT, void* saved, int spin_limit, int drop_tile,
                             cudaStream_t s, const Varlen* vl = nullptr);
bool fused_supported(const Dims& d);
int fused_ctas_per_block(const Dims& d);
// The same kernels with the logits given instead of projected (rglru_forward / rglru_backward
// and the composed layer, bf16 x): `nplanes` bf16 planes per logit (1, or 2 = hi + lo of a
// float32 value), `plane_elems` apart; 128-channel slices of W, the last one partial.
int logits_slices(const Dims& d);
int logits_ctas_per_slice(const Dims& d);
bool logits_scan_supported(const Dims& d);
// dx: the direct term only (dx_dt: DT_BF16 or DT_F32); dlr / dli in dl_dt (the dx dtype, or
// DT_SPLIT with a float32 dx: hi + lo planes dl_plane elements apart); dLambda, dh0 as in the
// fused backward.  `saved` comes from launch_logits_fwd with the same inputs.
cudaError_t launch_logits_bwd(const Dims& d, const void* dy, const float* dhT, const void* x,
                              const void* lr, const void* li, size_t plane_elems, int nplanes,
                              const float* Lambda, const uint8_t* rm, const int32_t* sp,
                              const void* saved, int dx_dt, void* dx, int dl_dt, void* dlr,
                              void* dli, size_t dl_plane, float* dLambda, float* dh0, void* ws,
                              int spin_limit, int drop_tile, cudaStream_t s,
                              const Varlen* vl = nullptr);
cudaError_t encode_logit_planes(const Dims& d, const void* base, size_t plane_elems, int nplanes,
                                CUtensorMap* m);
cudaError_t launch_logits_fwd(const Dims& d, const void* x, const void* lr, const void* li,
                              size_t plane_elems, int nplanes, const float* Lambda,
                              const uint8_t* rm, const int32_t* sp, const float* h0, void* y,
                              float* hT, void* saved, int spin_limit, int drop_tile,
                              cudaStream_t s, const Varlen* vl = nullptr);
// Clears the status word of a scan layout and marks every carry / aggregate slot empty.
cudaError_t clear_slots(void* buf, const ScanLayout& L, cudaStream_t s);

// Fused backward on tensor cores (same coverage as the fused forward; `saved` must come from
// launch_fused_fwd).  dx is written in shape.grad; dWa / dWx / dba / dbx / dLambda reduced
// deterministically on device; dh0 may be null.
cudaError_t launch_fused_bwd(const Dims& d, const void* dy, const float* dhT, const void* x,
                             const void* Wa, const float* ba, const void* Wx, const float* bx,
                             const float* Lambda, const uint8_t* rm, const int32_t* sp,
                             const float* h0, const void* saved, void* dx, float* dWa,
                             float* dba, float* dWx, float* dbx, float* dLambda, float* dh0,
                             void* ws, int spin_limit, int drop_tile, cudaStream_t s,
                             const Varlen* vl = nullptr);

// One decode step (T = 1) with carried states: projections, gates and the state update in one
// kernel (decode.cu); k <= STEP_KMAX.
constexpr int STEP_KMAX = 512;
// Batches from this size (bf16, k a multiple of 32 up to 256) take the tensor-core step.
constexpr int STEP_TC_MIN_B = 64;
bool step_tc_supported(const Dims& d);
cudaError_t launch_step(const Dims& d, const void* x, const void* Wa, const float* ba,
                        const void* Wx, const float* bx, const float* Lambda,
                        const uint8_t* reset, const float* h_in, void* y, float* h_out,
                        cudaStream_t s);

// Tensor-core projections (proj_tc.cu): bf16 operands, float32 accumulation, k a multiple of
// 16 up to PROJ_TC_KMAX.  The gradient operands dlr, dli are `nplanes` bf16 planes each
// ([plane][R][W], plane stride plane_elems elements): one plane, or hi + lo of a float32
// value.  dx = add + dl W^T (add float32 or bf16, may alias dx); dW / db through
// per-CTA partial sums (proj_dw_part_bytes) reduced in a fixed order.
constexpr int PROJ_TC_KMAX = 160;
bool proj_tc_supported(const Dims& d);
size_t proj_dw_part_bytes(const Dims& d);
// CTAs per gate block of the dx and dW kernels when the two run side by side (the dW kernel
// launched as a programmatic dependent of the dx one); {0, 0}: not on one wave, run them one
// after the other with the default P.
struct ProjBwdSplit {
  int P_dx, P_dw;
};
ProjBwdSplit proj_bwd_split(const Dims& d);
// float32 [N] -> bf16 hi plane [N] then lo plane [N] at `planes` (N = B T W).
cudaError_t launch_split_planes(const Dims& d, const float* src, void* planes, cudaStream_t s);
cudaError_t launch_proj_fwd(const Dims& d, int ot, const void* x, const void* Wa,
                            const float* ba, const void* Wx, const float* bx, void* lr, void* li,
                            cudaStream_t s);
cudaError_t launch_proj_dx(const Dims& d, int ot, const void* dlr, const void* dli,
                           size_t plane_elems, int nplanes, const void* Wa, const void* Wx,
                           const void* add, int add_f32, void* dx, cudaStream_t s, int P = 0);
cudaError_t launch_proj_dw(const Dims& d, const void* x, const void* dlr, const void* dli,
                           size_t plane_elems, int nplanes, float* part, float* dWa, float* dba,
                           float* dWx, float* dbx, cudaStream_t s, int P = 0);

// SIMT projections (float32 accumulation).
cudaError_t launch_gate_proj_simt(const Dims& d, int xt, int ot, const void* x, const void* Wa,
                                  const float* ba, const void* Wx, const float* bx, void* lr,
                                  void* li, cudaStream_t s);
cudaError_t launch_gate_dx_simt(const Dims& d, int wt, int gt, int dxt, const void* dlr,
                                const void* dli, const void* Wa, const void* Wx,
                                const float* dx_in, void* dx, cudaStream_t s);
cudaError_t launch_gate_dw_simt(const Dims& d, int xt, int gt, const void* x, const void* dlr,
                                const void* dli, float* dWa, float* dba, float* dWx, float* dbx,
                                uint8_t* ws, cudaStream_t s);

}  // namespace rglru
