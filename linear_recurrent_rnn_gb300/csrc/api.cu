// librglru host layer: argument validation, scratch layouts, and kernel launches on the
// caller's stream.  No allocation, no synchronisation (except rglru_sync_status, whose job
// it is).
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "internal.h"

using namespace rglru;

namespace {

std::atomic<uint64_t> g_launches{0};
int g_spin_limit = 1 << 22;
int g_drop_tile = -1;
size_t dsize(int dt) { return dt == RGLRU_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace rglru {

cudaEvent_t g_kernel_events[2] = {nullptr, nullptr};

void kernel_event_before(cudaStream_t s) {
  if (g_kernel_events[0] && g_kernel_events[1]) cudaEventRecord(g_kernel_events[0], s);
}
void kernel_event_after(cudaStream_t s) {
  if (g_kernel_events[0] && g_kernel_events[1]) {
    cudaEventRecord(g_kernel_events[1], s);
    g_kernel_events[0] = g_kernel_events[1] = nullptr;
  }
}

// Validates the shape and fills `d`.
rglru_status make_dims(const rglru_shape* s, Dims* d) {
  if (!s) return RGLRU_ERR_INVALID_ARG;
  if (s->B < 1 || s->T < 1 || s->W < 1 || s->nblk < 1) return RGLRU_ERR_INVALID_ARG;
  if (s->W % s->nblk) return RGLRU_ERR_INVALID_ARG;
  if ((s->io != RGLRU_F32 && s->io != RGLRU_BF16) || (s->grad != RGLRU_F32 && s->grad != RGLRU_BF16))
    return RGLRU_ERR_INVALID_ARG;
  if (s->mode != RGLRU_CANONICAL && s->mode != RGLRU_RESTRICTED) return RGLRU_ERR_INVALID_ARG;
  if (s->io == RGLRU_F32 && s->grad != RGLRU_F32) return RGLRU_ERR_UNSUPPORTED;
  if ((size_t)s->W * dsize(s->io) % 16 || (size_t)s->W * dsize(s->grad) % 16)
    return RGLRU_ERR_UNSUPPORTED;
  d->B = s->B;
  d->T = s->T;
  d->W = s->W;
  d->nblk = s->nblk;
  d->k = s->W / s->nblk;
  d->nC = (s->T + SC - 1) / SC;
  d->ng = (s->W + 31) / 32;
  d->N = (size_t)s->B * s->T * s->W;
  d->io = s->io;
  d->grad = s->grad;
  d->mode = s->mode;
  // ticket counters are 32-bit
  if ((double)d->B * d->nC * d->ng >= 4.0e9) return RGLRU_ERR_UNSUPPORTED;
  return RGLRU_OK;
}

// Required pointers: non-null and 16-byte aligned.  Optional: null or 16-byte aligned.
bool req(const void* p) { return p && aligned16(p); }
bool opt(const void* p) { return !p || aligned16(p); }

rglru_status check_resets(const Dims& d, const uint8_t* rm, const int32_t* sp, const float* h0) {
  if (!opt(rm) || !opt(sp) || !opt(h0)) return RGLRU_ERR_INVALID_ARG;
  if (rm && sp) return RGLRU_ERR_INVALID_ARG;
  if (d.mode == RGLRU_RESTRICTED && (rm || sp || h0)) return RGLRU_ERR_INVALID_ARG;
  return RGLRU_OK;
}

rglru_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RGLRU_OK;
  fprintf(stderr, "librglru: CUDA error %s\n", cudaGetErrorString(e));
  return RGLRU_ERR_CUDA;
}

// The fused layer through separate kernels: the logits are kept in `saved` (float32, or as bf16
// hi + lo planes on the tensor-core route: the same 4 bytes per element).
bool composed_tc(const Dims& d) { return proj_tc_supported(d) && logits_scan_supported(d); }

struct ComposedLayout {
  size_t lr, li, total;  // within `saved`, after the scan's own layout
};
ComposedLayout composed_saved(const Dims& d) {
  ComposedLayout C;
  size_t base = scan_layout(d, false).total;
  if (composed_tc(d) && fused_fwd_layout(d).total > base) base = fused_fwd_layout(d).total;
  C.lr = align_up(base, 256);
  C.li = align_up(C.lr + d.N * 4, 256);
  C.total = align_up(C.li + d.N * 4, 256);
  return C;
}
// Scratch of the projection backward inside a workspace: the SIMT kernels' partial sums, or
// the tensor-core kernels' per-CTA dW / db partials, both after a 256-byte header (a scan
// backward run on the same workspace keeps its status word there).
// With float32 gradients the tensor-core route first splits dlr and dli into bf16 hi + lo
// planes, kept after the partials.
constexpr size_t PROJ_PART_OFFSET = 256;
size_t gate_planes_offset(const Dims& d) {
  return align_up(PROJ_PART_OFFSET + proj_dw_part_bytes(d), 256);
}
size_t gate_bwd_ws_bytes(const Dims& d) {
  size_t a = gate_bwd_layout(d).total;
  if (proj_tc_supported(d)) {
    size_t b = PROJ_PART_OFFSET + proj_dw_part_bytes(d);
    if (d.grad == RGLRU_F32) b = gate_planes_offset(d) + 2 * (size_t)d.N * 4;
    if (b > a) a = b;
  }
  return a;
}

struct ComposedWs {
  size_t dxd, dlr, dli, gate, total;  // within `workspace`, after the backward scan layout
};
ComposedWs composed_ws(const Dims& d) {
  ComposedWs C;
  size_t base = scan_layout(d, true).total;
  if (composed_tc(d) && fused_bwd_layout(d).total > base) base = fused_bwd_layout(d).total;
  C.dxd = align_up(base, 256);
  C.dlr = align_up(C.dxd + d.N * 4, 256);
  C.dli = align_up(C.dlr + d.N * 4, 256);
  C.gate = align_up(C.dli + d.N * 4, 256);
  C.total = align_up(C.gate + gate_bwd_ws_bytes(d), 256);
  return C;
}

ScanFwdArgs fwd_args(const Dims& d, const void* x, const void* lr, const void* li,
                     const float* Lambda, const uint8_t* rm, const int32_t* sp, const float* h0,
                     void* y, float* hT, void* saved) {
  ScanFwdArgs a;
  a.B = d.B;
  a.T = d.T;
  a.W = d.W;
  a.nC = d.nC;
  a.ng = d.ng;
  a.x = x;
  a.lr = lr;
  a.li = li;
  a.Lambda = Lambda;
  a.reset_mask = rm;
  a.segment_pos = sp;
  a.h0 = h0;
  a.y = y;
  a.hT = hT;
  a.scratch = static_cast<uint8_t*>(saved);
  a.L = scan_layout(d, false);
  a.spin_limit = g_spin_limit;
  a.drop_tile = g_drop_tile;
  return a;
}

ScanBwdArgs bwd_args(const Dims& d, const void* dy, const float* dhT, const void* x,
                     const void* lr, const void* li, const float* Lambda, const uint8_t* rm,
                     const int32_t* sp, const float* h0, const void* saved, void* dx, void* dlr,
                     void* dli, float* dLambda, float* dh0, void* ws) {
  ScanBwdArgs a;
  a.B = d.B;
  a.T = d.T;
  a.W = d.W;
  a.nC = d.nC;
  a.ng = d.ng;
  a.dy = dy;
  a.dhT = dhT;
  a.x = x;
  a.lr = lr;
  a.li = li;
  a.Lambda = Lambda;
  a.reset_mask = rm;
  a.segment_pos = sp;
  a.h0 = h0;
  a.fwd_carry = reinterpret_cast<const float*>(static_cast<const uint8_t*>(saved) +
                                                scan_layout(d, false).carry);
  a.dx = dx;
  a.dlr = dlr;
  a.dli = dli;
  a.dl_plane = d.N;
  a.dLambda = dLambda;
  a.dh0 = dh0;
  a.scratch = static_cast<uint8_t*>(ws);
  a.L = scan_layout(d, true);
  a.spin_limit = g_spin_limit;
  a.drop_tile = g_drop_tile;
  return a;
}

}  // namespace rglru

namespace rglru {
void note_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
int debug_spin_limit() { return g_spin_limit; }
int debug_drop_tile() { return g_drop_tile; }
}  // namespace rglru

extern "C" {

const char* rglru_status_string(rglru_status s) {
  switch (s) {
    case RGLRU_OK: return "ok";
    case RGLRU_ERR_INVALID_ARG: return "invalid argument";
    case RGLRU_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case RGLRU_ERR_CUDA: return "CUDA error";
    case RGLRU_ERR_TIMEOUT: return "look-back wait timed out";
  }
  return "unknown status";
}

// Where a packed call keeps its token indices in `saved`: in the fused layout on the
// tensor-core routes, after the logits on the CUDA-core one (whose scan slots are wider).
struct VarlenIndex {
  size_t seq_start, seq_end, total;
};
static VarlenIndex varlen_index(const Dims& d) {
  VarlenIndex v;
  if (fused_supported(d) || composed_tc(d)) {
    const FusedFwdLayout FL = fused_fwd_layout(d);
    v.seq_start = FL.seq_start;
    v.seq_end = FL.seq_end;
    v.total = FL.total;
  } else {
    v.seq_start = composed_saved(d).total;
    v.seq_end = align_up(v.seq_start + (size_t)d.T * 4, 256);
    v.total = align_up(v.seq_end + (size_t)d.T * 4, 256);
  }
  return v;
}

size_t rglru_saved_bytes(const rglru_shape* shape) {
  Dims d;
  if (make_dims(shape, &d) != RGLRU_OK) return 0;
  // the unfused scan's layout, and the fused call's: the tensor-core kernels' own where they
  // take the shape, else the composed path's (which keeps float32 logits)
  size_t a = scan_layout(d, false).total;
  if (logits_scan_supported(d) && fused_fwd_layout(d).total > a) a = fused_fwd_layout(d).total;
  size_t f = fused_supported(d) ? fused_fwd_layout(d).total : composed_saved(d).total;
  if (d.B == 1 && varlen_index(d).total > f) f = varlen_index(d).total;  // packed calls
  return a > f ? a : f;
}

size_t rglru_workspace_bytes(const rglru_shape* shape) {
  Dims d;
  if (make_dims(shape, &d) != RGLRU_OK) return 0;
  size_t m = scan_layout(d, true).total;
  if (logits_scan_supported(d) && fused_bwd_layout(d).total > m) m = fused_bwd_layout(d).total;
  const size_t g = gate_bwd_ws_bytes(d);
  const size_t f = fused_supported(d) ? fused_bwd_layout(d).total : composed_ws(d).total;
  if (g > m) m = g;
  if (f > m) m = f;
  return m;
}

rglru_status rglru_gate_proj(const rglru_shape* shape, const void* x, const void* Wa,
                             const float* ba, const void* Wx, const float* bx, void* lr, void* li,
                             rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(x) || !req(Wa) || !req(Wx) || !req(lr) || !req(li) || !opt(ba) || !opt(bx))
    return RGLRU_ERR_INVALID_ARG;
  if (proj_tc_supported(d))
    return cuda_status(launch_proj_fwd(d, d.io, x, Wa, ba, Wx, bx, lr, li, stream));
  return cuda_status(launch_gate_proj_simt(d, d.io, d.io, x, Wa, ba, Wx, bx, lr, li, stream));
}

rglru_status rglru_forward(const rglru_shape* shape, const void* x, const void* lr,
                           const void* li, const float* Lambda, const uint8_t* reset_mask,
                           const int32_t* segment_pos, const float* h0, void* y, float* hT,
                           void* saved, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(x) || !req(lr) || !req(li) || !req(Lambda) || !req(y) || !opt(hT) || !req(saved))
    return RGLRU_ERR_INVALID_ARG;
  if ((st = check_resets(d, reset_mask, segment_pos, h0)) != RGLRU_OK) return st;
  if (logits_scan_supported(d))  // bf16: the fused scan kernel with the logits given
    return cuda_status(launch_logits_fwd(d, x, lr, li, d.N, 1, Lambda, reset_mask, segment_pos,
                                         h0, y, hT, saved, g_spin_limit, g_drop_tile, stream));
  const ScanFwdArgs a = fwd_args(d, x, lr, li, Lambda, reset_mask, segment_pos, h0, y, hT, saved);
  cudaError_t e = cudaMemsetAsync(saved, 0, a.L.zero_bytes, stream);
  if (e == cudaSuccess) e = launch_scan_fwd(a, d.io, d.io, d.mode == RGLRU_CANONICAL, stream);
  return cuda_status(e);
}

rglru_status rglru_backward(const rglru_shape* shape, const void* dy, const float* dhT,
                            const void* x, const void* lr, const void* li, const float* Lambda,
                            const uint8_t* reset_mask, const int32_t* segment_pos,
                            const float* h0, const void* saved, void* dx, void* dlr, void* dli,
                            float* dLambda, float* dh0, void* workspace, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(dy) || !opt(dhT) || !req(x) || !req(lr) || !req(li) || !req(Lambda) || !req(saved) ||
      !req(dx) || !req(dlr) || !req(dli) || !req(dLambda) || !opt(dh0) || !req(workspace))
    return RGLRU_ERR_INVALID_ARG;
  if ((st = check_resets(d, reset_mask, segment_pos, h0)) != RGLRU_OK) return st;
  if (logits_scan_supported(d))
    return cuda_status(launch_logits_bwd(d, dy, dhT, x, lr, li, d.N, 1, Lambda, reset_mask,
                                         segment_pos, saved, d.grad, dx, d.grad, dlr, dli, 0,
                                         dLambda, dh0, workspace, g_spin_limit, g_drop_tile,
                                         stream));
  const ScanBwdArgs a = bwd_args(d, dy, dhT, x, lr, li, Lambda, reset_mask, segment_pos, h0, saved,
                                 dx, dlr, dli, dLambda, dh0, workspace);
  cudaError_t e = cudaMemsetAsync(workspace, 0, a.L.zero_bytes, stream);
  if (e == cudaSuccess)
    e = launch_scan_bwd(a, d.io, d.io, d.grad, d.grad, d.mode == RGLRU_CANONICAL, stream);
  return cuda_status(e);
}

rglru_status rglru_gate_proj_backward(const rglru_shape* shape, const void* dlr, const void* dli,
                                      const void* x, const void* Wa, const void* Wx, void* dx,
                                      float* dWa, float* dba, float* dWx, float* dbx,
                                      void* workspace, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(dlr) || !req(dli) || !req(x) || !req(Wa) || !req(Wx) || !req(dx) || !req(dWa) ||
      !req(dWx) || !opt(dba) || !opt(dbx) || !req(workspace))
    return RGLRU_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (proj_tc_supported(d)) {
    // dx accumulates in place; dx and dW run side by side where one wave of CTAs holds both
    // grids.  bf16 gradients: one plane each; float32: split into bf16 hi + lo planes first.
    const ProjBwdSplit sp = proj_bwd_split(d);
    float* part = reinterpret_cast<float*>(ws + PROJ_PART_OFFSET);
    cudaError_t e = cudaSuccess;
    if (d.grad == RGLRU_BF16) {
      e = launch_proj_dx(d, DT_BF16, dlr, dli, d.N, 1, Wa, Wx, dx, 0, dx, stream, sp.P_dx);
      if (e == cudaSuccess)
        e = launch_proj_dw(d, x, dlr, dli, d.N, 1, part, dWa, dba, dWx, dbx, stream, sp.P_dw);
    } else {
      uint8_t* pr = ws + gate_planes_offset(d);  // dlr hi, lo, then dli hi, lo
      uint8_t* pi = pr + 4 * (size_t)d.N;
      e = launch_split_planes(d, static_cast<const float*>(dlr), pr, stream);
      if (e == cudaSuccess) e = launch_split_planes(d, static_cast<const float*>(dli), pi, stream);
      if (e == cudaSuccess)
        e = launch_proj_dx(d, DT_F32, pr, pi, d.N, 2, Wa, Wx, dx, 1, dx, stream, sp.P_dx);
      if (e == cudaSuccess)
        e = launch_proj_dw(d, x, pr, pi, d.N, 2, part, dWa, dba, dWx, dbx, stream, sp.P_dw);
    }
    return cuda_status(e);
  }
  cudaError_t e =
      launch_gate_dx_simt(d, d.io, d.grad, d.grad, dlr, dli, Wa, Wx, nullptr, dx, stream);
  if (e == cudaSuccess)
    e = launch_gate_dw_simt(d, d.io, d.grad, x, dlr, dli, dWa, dba, dWx, dbx, ws, stream);
  return cuda_status(e);
}

rglru_status rglru_fused_forward(const rglru_shape* shape, const void* x, const void* Wa,
                                 const float* ba, const void* Wx, const float* bx,
                                 const float* Lambda, const uint8_t* reset_mask,
                                 const int32_t* segment_pos, const float* h0, void* y, float* hT,
                                 void* saved, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(x) || !req(Wa) || !req(Wx) || !opt(ba) || !opt(bx) || !req(Lambda) || !req(y) ||
      !opt(hT) || !req(saved))
    return RGLRU_ERR_INVALID_ARG;
  if ((st = check_resets(d, reset_mask, segment_pos, h0)) != RGLRU_OK) return st;
  if (fused_supported(d))
    return cuda_status(launch_fused_fwd(d, x, Wa, ba, Wx, bx, Lambda, reset_mask, segment_pos,
                                        h0, y, hT, saved, g_spin_limit, g_drop_tile, stream));
  uint8_t* sv = static_cast<uint8_t*>(saved);
  const ComposedLayout C = composed_saved(d);
  if (composed_tc(d)) {
    // tensor-core projections to bf16 hi + lo logit planes, then the fused scan kernel on them
    cudaError_t e = launch_proj_fwd(d, DT_SPLIT, x, Wa, ba, Wx, bx, sv + C.lr, sv + C.li, stream);
    if (e == cudaSuccess)
      e = launch_logits_fwd(d, x, sv + C.lr, sv + C.li, d.N, 2, Lambda, reset_mask, segment_pos,
                            h0, y, hT, saved, g_spin_limit, g_drop_tile, stream);
    return cuda_status(e);
  }
  cudaError_t e = launch_gate_proj_simt(d, d.io, DT_F32, x, Wa, ba, Wx, bx, sv + C.lr, sv + C.li,
                                        stream);
  const ScanFwdArgs a = fwd_args(d, x, sv + C.lr, sv + C.li, Lambda, reset_mask, segment_pos, h0,
                                 y, hT, saved);
  if (e == cudaSuccess) e = cudaMemsetAsync(saved, 0, a.L.zero_bytes, stream);
  if (e == cudaSuccess) e = launch_scan_fwd(a, d.io, DT_F32, d.mode == RGLRU_CANONICAL, stream);
  return cuda_status(e);
}

rglru_status rglru_fused_backward(const rglru_shape* shape, const void* dy, const float* dhT,
                                  const void* x, const void* Wa, const float* ba, const void* Wx,
                                  const float* bx, const float* Lambda,
                                  const uint8_t* reset_mask, const int32_t* segment_pos,
                                  const float* h0, const void* saved, void* dx, float* dWa,
                                  float* dba, float* dWx, float* dbx, float* dLambda, float* dh0,
                                  void* workspace, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(dy) || !opt(dhT) || !req(x) || !req(Wa) || !req(Wx) || !opt(ba) || !opt(bx) ||
      !req(Lambda) || !req(saved) || !req(dx) || !req(dWa) || !req(dWx) || !opt(dba) ||
      !opt(dbx) || !req(dLambda) || !opt(dh0) || !req(workspace))
    return RGLRU_ERR_INVALID_ARG;
  if ((st = check_resets(d, reset_mask, segment_pos, h0)) != RGLRU_OK) return st;
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const ComposedLayout C = composed_saved(d);
  const ComposedWs CW = composed_ws(d);
  if (fused_supported(d))
    return cuda_status(launch_fused_bwd(d, dy, dhT, x, Wa, ba, Wx, bx, Lambda, reset_mask,
                                        segment_pos, h0, saved, dx, dWa, dba, dWx, dbx, dLambda,
                                        dh0, workspace, g_spin_limit, g_drop_tile, stream));
  const void* lr = sv + C.lr;
  const void* li = sv + C.li;
  const void* fsaved = saved;
  cudaError_t e = cudaSuccess;
  const ScanBwdArgs a = bwd_args(d, dy, dhT, x, lr, li, Lambda, reset_mask, segment_pos, h0,
                                 fsaved, ws + CW.dxd, ws + CW.dlr, ws + CW.dli, dLambda, dh0,
                                 workspace);
  // The direct term of dx stays float32 until the projections are added: one rounding.
  if (composed_tc(d)) {
    // the fused scan kernel on the saved hi + lo logit planes; dlr, dli out as bf16 hi + lo
    // planes (the same bytes as float32), the operands of the tensor-core products
    e = launch_logits_bwd(d, dy, dhT, x, lr, li, d.N, 2, Lambda, reset_mask, segment_pos, saved,
                          DT_F32, ws + CW.dxd, DT_SPLIT, ws + CW.dlr, ws + CW.dli, d.N, dLambda,
                          dh0, workspace, g_spin_limit, g_drop_tile, stream);
    if (e == cudaSuccess)
      e = launch_proj_dx(d, d.grad, ws + CW.dlr, ws + CW.dli, d.N, 2, Wa, Wx, ws + CW.dxd, 1,
                         dx, stream);
    if (e == cudaSuccess)
      e = launch_proj_dw(d, x, ws + CW.dlr, ws + CW.dli, d.N, 2,
                         reinterpret_cast<float*>(ws + CW.gate + PROJ_PART_OFFSET), dWa, dba,
                         dWx, dbx, stream);
    return cuda_status(e);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, a.L.zero_bytes, stream);
  if (e == cudaSuccess)
    e = launch_scan_bwd(a, d.io, DT_F32, DT_F32, DT_F32, d.mode == RGLRU_CANONICAL, stream);
  if (e == cudaSuccess)
    e = launch_gate_dx_simt(d, d.io, DT_F32, d.grad, ws + CW.dlr, ws + CW.dli, Wa, Wx,
                            reinterpret_cast<const float*>(ws + CW.dxd), dx, stream);
  if (e == cudaSuccess)
    e = launch_gate_dw_simt(d, d.io, DT_F32, x, ws + CW.dlr, ws + CW.dli, dWa, dba, dWx, dbx,
                            ws + CW.gate, stream);
  return cuda_status(e);
}

// Packed variable-length sequences: one row of T tokens, sequence s on [cu[s], cu[s+1]).
static rglru_status varlen_setup(const rglru_shape* shape, const int32_t* cu, int32_t S,
                                 const void* saved, Dims* d, Varlen* v) {
  rglru_status st = make_dims(shape, d);
  if (st != RGLRU_OK) return st;
  if (d->B != 1 || d->mode != RGLRU_CANONICAL || S < 1 || !req(cu) || !req(saved))
    return RGLRU_ERR_INVALID_ARG;
  const VarlenIndex VI = varlen_index(*d);
  v->cu_seqlens = cu;
  v->S = S;
  v->seq_start = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + VI.seq_start);
  v->seq_end = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + VI.seq_end);
  v->h0 = nullptr;
  v->hT = nullptr;
  v->dhT = nullptr;
  v->dh0 = nullptr;
  return RGLRU_OK;
}

rglru_status rglru_fused_forward_varlen(const rglru_shape* shape, const void* x, const void* Wa,
                                        const float* ba, const void* Wx, const float* bx,
                                        const float* Lambda, const int32_t* cu_seqlens,
                                        int32_t num_seqs, const float* h0, void* y, float* hT,
                                        void* saved, rglru_stream stream) {
  Dims d;
  Varlen v;
  rglru_status st = varlen_setup(shape, cu_seqlens, num_seqs, saved, &d, &v);
  if (st != RGLRU_OK) return st;
  if (!req(x) || !req(Wa) || !req(Wx) || !opt(ba) || !opt(bx) || !req(Lambda) || !opt(h0) ||
      !req(y) || !opt(hT))
    return RGLRU_ERR_INVALID_ARG;
  // the tensor-core routes (bf16 I/O, k a multiple of 16 up to 160), or float32 I/O on the
  // CUDA cores
  if (!fused_supported(d) && !composed_tc(d) && d.io != RGLRU_F32) return RGLRU_ERR_UNSUPPORTED;
  v.h0 = h0;
  v.hT = hT;
  cudaError_t e = launch_seq_index(v, d.T, d.W, const_cast<int32_t*>(v.seq_start),
                                   const_cast<int32_t*>(v.seq_end), stream);
  if (!fused_supported(d) && !composed_tc(d)) {
    // float32 I/O (and other shapes off the tensor cores): the SIMT projections, then the
    // CUDA-core scan over the packed sequences
    uint8_t* sv = static_cast<uint8_t*>(saved);
    const ComposedLayout C = composed_saved(d);
    if (e == cudaSuccess)
      e = launch_gate_proj_simt(d, d.io, DT_F32, x, Wa, ba, Wx, bx, sv + C.lr, sv + C.li, stream);
    ScanFwdArgs a = fwd_args(d, x, sv + C.lr, sv + C.li, Lambda, nullptr, nullptr, nullptr, y,
                             nullptr, saved);
    a.seq_start = v.seq_start;
    a.seq_end = v.seq_end;
    a.h0s = h0;
    a.hTs = hT;
    if (e == cudaSuccess) e = cudaMemsetAsync(saved, 0, a.L.zero_bytes, stream);
    if (e == cudaSuccess) e = launch_scan_fwd(a, d.io, DT_F32, true, stream);
    return cuda_status(e);
  }
  if (fused_supported(d)) {
    if (e == cudaSuccess)
      e = launch_fused_fwd(d, x, Wa, ba, Wx, bx, Lambda, nullptr, nullptr, nullptr, y, nullptr,
                           saved, g_spin_limit, g_drop_tile, stream, &v);
    return cuda_status(e);
  }
  // other gate blocks: tensor-core projections to hi + lo logit planes, then the packed scan
  uint8_t* sv = static_cast<uint8_t*>(saved);
  const ComposedLayout C = composed_saved(d);
  if (e == cudaSuccess)
    e = launch_proj_fwd(d, DT_SPLIT, x, Wa, ba, Wx, bx, sv + C.lr, sv + C.li, stream);
  if (e == cudaSuccess)
    e = launch_logits_fwd(d, x, sv + C.lr, sv + C.li, d.N, 2, Lambda, nullptr, nullptr, nullptr,
                          y, nullptr, saved, g_spin_limit, g_drop_tile, stream, &v);
  return cuda_status(e);
}

rglru_status rglru_fused_backward_varlen(const rglru_shape* shape, const void* dy,
                                         const float* dhT, const void* x, const void* Wa,
                                         const float* ba, const void* Wx, const float* bx,
                                         const float* Lambda, const int32_t* cu_seqlens,
                                         int32_t num_seqs, const float* h0, const void* saved,
                                         void* dx, float* dWa, float* dba, float* dWx,
                                         float* dbx, float* dLambda, float* dh0,
                                         void* workspace, rglru_stream stream) {
  Dims d;
  Varlen v;
  rglru_status st = varlen_setup(shape, cu_seqlens, num_seqs, saved, &d, &v);
  if (st != RGLRU_OK) return st;
  if (!req(dy) || !opt(dhT) || !req(x) || !req(Wa) || !req(Wx) || !opt(ba) || !opt(bx) ||
      !req(Lambda) || !opt(h0) || !req(dx) || !req(dWa) || !req(dWx) || !opt(dba) ||
      !opt(dbx) || !req(dLambda) || !opt(dh0) || !req(workspace))
    return RGLRU_ERR_INVALID_ARG;
  if (!fused_supported(d) && !composed_tc(d) && d.io != RGLRU_F32) return RGLRU_ERR_UNSUPPORTED;
  v.h0 = h0;
  v.dhT = dhT;
  v.dh0 = dh0;
  // the token indices were written by the forward into `saved`; empty sequences' dh0 here
  cudaError_t e = cudaSuccess;
  if (dh0) e = launch_seq_empty_dh0(v, d.W, stream);
  if (!fused_supported(d) && !composed_tc(d)) {
    // float32 I/O: the CUDA-core scan backward over the packed sequences on the saved float32
    // logits, then the SIMT projection backward
    const uint8_t* sv = static_cast<const uint8_t*>(saved);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const ComposedLayout C = composed_saved(d);
    const ComposedWs CW = composed_ws(d);
    ScanBwdArgs a = bwd_args(d, dy, nullptr, x, sv + C.lr, sv + C.li, Lambda, nullptr, nullptr,
                             nullptr, saved, ws + CW.dxd, ws + CW.dlr, ws + CW.dli, dLambda,
                             nullptr, workspace);
    a.seq_start = v.seq_start;
    a.seq_end = v.seq_end;
    a.h0s = h0;
    a.dhTs = dhT;
    a.dh0s = dh0;
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, a.L.zero_bytes, stream);
    if (e == cudaSuccess) e = launch_scan_bwd(a, d.io, DT_F32, DT_F32, DT_F32, true, stream);
    if (e == cudaSuccess)
      e = launch_gate_dx_simt(d, d.io, DT_F32, d.grad, ws + CW.dlr, ws + CW.dli, Wa, Wx,
                              reinterpret_cast<const float*>(ws + CW.dxd), dx, stream);
    if (e == cudaSuccess)
      e = launch_gate_dw_simt(d, d.io, DT_F32, x, ws + CW.dlr, ws + CW.dli, dWa, dba, dWx, dbx,
                              ws + CW.gate, stream);
    return cuda_status(e);
  }
  if (fused_supported(d)) {
    if (e == cudaSuccess)
      e = launch_fused_bwd(d, dy, nullptr, x, Wa, ba, Wx, bx, Lambda, nullptr, nullptr, nullptr,
                           saved, dx, dWa, dba, dWx, dbx, dLambda, nullptr, workspace,
                           g_spin_limit, g_drop_tile, stream, &v);
    return cuda_status(e);
  }
  // other gate blocks: the packed scan backward on the saved logit planes (float32 direct dx
  // term, dl as hi + lo planes), then the tensor-core projection backward
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const ComposedLayout C = composed_saved(d);
  const ComposedWs CW = composed_ws(d);
  if (e == cudaSuccess)
    e = launch_logits_bwd(d, dy, nullptr, x, sv + C.lr, sv + C.li, d.N, 2, Lambda, nullptr,
                          nullptr, saved, DT_F32, ws + CW.dxd, DT_SPLIT, ws + CW.dlr,
                          ws + CW.dli, d.N, dLambda, nullptr, workspace, g_spin_limit,
                          g_drop_tile, stream, &v);
  if (e == cudaSuccess)
    e = launch_proj_dx(d, d.grad, ws + CW.dlr, ws + CW.dli, d.N, 2, Wa, Wx, ws + CW.dxd, 1, dx,
                       stream);
  if (e == cudaSuccess)
    e = launch_proj_dw(d, x, ws + CW.dlr, ws + CW.dli, d.N, 2,
                       reinterpret_cast<float*>(ws + CW.gate + PROJ_PART_OFFSET), dWa, dba, dWx,
                       dbx, stream);
  return cuda_status(e);
}

rglru_status rglru_step(const rglru_shape* shape, const void* x, const void* Wa,
                        const float* ba, const void* Wx, const float* bx, const float* Lambda,
                        const uint8_t* reset, const float* h_in, void* y, float* h_out,
                        rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (d.T != 1) return RGLRU_ERR_INVALID_ARG;
  if (!req(x) || !req(Wa) || !req(Wx) || !opt(ba) || !opt(bx) || !req(Lambda) || !opt(reset) ||
      !opt(h_in) || !req(y) || !req(h_out))
    return RGLRU_ERR_INVALID_ARG;
  if (d.mode == RGLRU_RESTRICTED && reset) return RGLRU_ERR_INVALID_ARG;
  if (d.k > STEP_KMAX) return RGLRU_ERR_UNSUPPORTED;
  return cuda_status(launch_step(d, x, Wa, ba, Wx, bx, Lambda, reset, h_in, y, h_out, stream));
}

rglru_status rglru_sync_status(const void* buf, rglru_stream stream) {
  if (!buf) return RGLRU_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(&word, buf, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  return word ? RGLRU_ERR_TIMEOUT : RGLRU_OK;
}

const char* rglru_fused_path(const rglru_shape* shape) {
  Dims d;
  if (make_dims(shape, &d) != RGLRU_OK) return "invalid shape";
  if (fused_supported(d))
    return "fused: k_fused_fwd / k_fused_bwd (tcgen05 projections and CUDA-core scan in one "
           "kernel each)";
  if (composed_tc(d))
    return "composed: tcgen05 projections (k_proj_fwd, k_proj_dx, k_proj_dw) around the fused "
           "scan kernels with the logits given (kept as bf16 hi + lo planes)";
  return "composed: float32 SIMT projections, CUDA-core scan kernels (float32 logits kept)";
}

uint64_t rglru_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

void rglru_debug_kernel_events(void* start, void* stop) {
  rglru::g_kernel_events[0] = static_cast<cudaEvent_t>(start);
  rglru::g_kernel_events[1] = static_cast<cudaEvent_t>(stop);
}

void rglru_debug_lookback(int32_t spin_limit, int32_t drop_tile) {
  g_spin_limit = spin_limit > 0 ? spin_limit : (1 << 22);
  g_drop_tile = drop_tile;
}

}  // extern "C"
