// Exact chunked scan of the RG-LRU recurrence, forward and backward, on CUDA cores.
//
// Recurrence ("Fattori comparison" page, the operator's fused steps and the reset semantics
// of its "semantic limits" list): r = sigmoid(lr), i = sigmoid(li), log a = -8 r
// softplus(Lambda), m = sqrt(1 - a^2) (m = 1 and the previous state dropped at a reset token),
// h_t = a h_{t-1} + m i x.  The same page closes with an exact parallel chunked forward and
// backward with partial chunks; this file is that scan.
//
// Work split.  A warp owns one tile: 32 channels x SC = 16 tokens of one batch row.  Lane
// (pair p, half s) holds channels 2p, 2p+1 and tokens 8s .. 8s+7, so each token row is read
// as 64 contiguous bytes (bf16) or 128 bytes (float).  Within a lane the recurrence runs
// serially in float32 registers; the two halves are joined with one shuffle of their affine
// aggregates (A, B) (h -> A h + B, composed as (A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2)).
// Across tiles the carry travels by decoupled look-back: each tile publishes its aggregate and
// composes its predecessors' aggregates back to its anchor chunk (every STEP-th, at least
// DIST back, or the initial state; LbPlan), whose boundary state it applies them to; anchors then
// publish their own boundary state.  All of a look-back's flags are polled together and its
// aggregates loaded together.  Stopping at fixed anchors rather than at whichever state
// happens to be published first keeps the rounding, and so the result, independent of
// timing.  Tiles are handed out by an atomic ticket in dependency order, so every tile a warp
// waits on is held by a warp that is already running; waits are bounded.
#include "common.cuh"
#include "internal.h"

namespace rglru {

namespace {

struct Tile {
  int c, b, g;
  unsigned ticket;
  bool valid;
};

// Dependency-ordered tile of this warp.  Forward: chunk-major ascending; backward: descending.
__device__ __forceinline__ Tile grab_tile(uint32_t* ticket, int B, int nC, int ng, bool reverse) {
  const int lane = threadIdx.x & 31;
  unsigned t = 0;
  if (lane == 0) t = atomicAdd(ticket, 1u);
  t = __shfl_sync(0xffffffffu, t, 0);
  Tile r;
  r.ticket = t;
  const unsigned per_c = (unsigned)B * ng;
  r.valid = t < per_c * (unsigned)nC;
  const int cc = (int)(t / per_c);
  const int rem = (int)(t % per_c);
  r.c = reverse ? nC - 1 - cc : cc;
  r.b = rem / ng;
  r.g = rem % ng;
  return r;
}

// The look-back span of processing-order chunk q: `anchor` (-1: the initial state) and the
// n aggregates of chunks q-1 .. q-n composed onto it.
template <bool BWD>
__device__ __forceinline__ void lb_span(int q, int& anchor, int& n) {
  using LP = LbPlan<BWD>;
  if (q < LP::DIST) {
    anchor = -1;
    n = q;
  } else {
    anchor = ((q - LP::DIST) / LP::STEP) * LP::STEP;
    n = q - 1 - anchor;
  }
}

// Polls a tile's look-back flags together: bit k < n is the aggregate of processing-order
// chunk q-1-k (FLAG_AGG), bit n the anchor's boundary state (FLAG_INCL; none when anchor < 0).
// Each round issues one load per flag still short before testing any, so a round costs one
// L2 round trip however many flags are late.  Returns the mask of the flags seen set; after
// `limit` rounds the timeout is recorded in *status and the caller goes on without the
// missing ones.  fbase: the flag of (row, chunk 0, group); ng: the flag stride per chunk.
template <bool reverse>
__device__ __forceinline__ uint32_t poll_flags(const uint32_t* fbase, int ng, int q, int n,
                                               int anchor, int nC, int limit, uint32_t* status) {
  constexpr int LB_MAX = LbPlan<reverse>::MAX;
  const uint32_t all = anchor >= 0 ? (2u << n) - 1u : (1u << n) - 1u;
  uint32_t got = 0u;
  for (int round = 0;; ++round) {
    if (got == all) return got;
    if (round > limit) {
      atomicOr(status, STATUS_TIMEOUT);
      return got;
    }
    if (round > 0) __nanosleep(64);
    const uint32_t want = all & ~got;
    uint32_t f[LB_MAX + 1];
#pragma unroll
    for (int k = 0; k <= LB_MAX; ++k) {
      f[k] = 0u;
      if ((want >> k) & 1u) {
        const int pq = k < n ? q - 1 - k : anchor;
        f[k] = ld_acquire(fbase + (size_t)(reverse ? nC - 1 - pq : pq) * ng);
      }
    }
#pragma unroll
    for (int k = 0; k <= LB_MAX; ++k)
      if (((want >> k) & 1u) && f[k] >= (k < n ? FLAG_AGG : FLAG_INCL)) got |= 1u << k;
  }
}

// Composes the aggregates the poll found (chunk q-1-k for bit k, float4 = two channels'
// (A, B) at agg + (row_chunk0 + chunk) * W) newest first onto the state `hp`, in batches
// of seven loads.
template <bool reverse>
__device__ __forceinline__ void lb_compose(const float2* agg, size_t row_c0, int W, int w,
                                           int q, int n, uint32_t got, int nC, float2 hp,
                                           float (&out)[2]) {
  constexpr int LB_MAX = LbPlan<reverse>::MAX;
  float accA[2] = {1.0f, 1.0f}, accB[2] = {0.0f, 0.0f};
#pragma unroll
  for (int k0 = 0; k0 < LB_MAX; k0 += 7) {
    float4 ag[7];
#pragma unroll
    for (int u = 0; u < 7; ++u) {
      const int k = k0 + u;
      if (k < n && ((got >> k) & 1u)) {
        const int pq = q - 1 - k;
        ag[u] = __ldcg(reinterpret_cast<const float4*>(
            agg + (row_c0 + (size_t)(reverse ? nC - 1 - pq : pq)) * W + w));
      }
    }
#pragma unroll
    for (int u = 0; u < 7; ++u) {
      const int k = k0 + u;
      if (k < n && ((got >> k) & 1u)) {
        accB[0] = fmaf(accA[0], ag[u].y, accB[0]);
        accA[0] *= ag[u].x;
        accB[1] = fmaf(accA[1], ag[u].w, accB[1]);
        accA[1] *= ag[u].z;
      }
    }
  }
  out[0] = fmaf(accA[0], hp.x, accB[0]);
  out[1] = fmaf(accA[1], hp.y, accB[1]);
}

// The scan kernels are bound by the latency of short tiles, so resident warps matter more
// than a few spilled registers: 7 CTAs per SM (72 registers) for the forward, 4 (128) for
// the backward, each measured faster than the spill-free 5 and 3.
// VARLEN (packed sequences, one row): at the first token of sequence s the chain restarts from
// h0[s] (h -> abar h0[s] + m i x, the carry dropped), and the state after the last token of
// sequence s is its hT[s].
template <typename XT, typename LT, bool CANON, bool VARLEN>
__global__ void __launch_bounds__(128, 7) k_scan_fwd(ScanFwdArgs a) {
  uint32_t* status = reinterpret_cast<uint32_t*>(a.scratch);
  uint32_t* ticket = status + 1;
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.scratch + a.L.flags);
  float* carry = reinterpret_cast<float*>(a.scratch + a.L.carry);
  float2* agg = reinterpret_cast<float2*>(a.scratch + a.L.agg);

  const Tile tl = grab_tile(ticket, a.B, a.nC, a.ng, false);
  if (!tl.valid) return;
  const int lane = threadIdx.x & 31;
  const int pair = lane & 15, half = lane >> 4;
  const int w = tl.g * 32 + pair * 2;
  const bool wok = w < a.W;
  const int t0 = tl.c * SC + half * SUB;
  const XT* x = static_cast<const XT*>(a.x);
  const LT* lr = static_cast<const LT*>(a.lr);
  const LT* li = static_cast<const LT*>(a.li);

  float nk[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) nk[j] = wok ? -8.0f * softplus_f(a.Lambda[w + j]) : 0.0f;

  // Local scan from a zero carry: hl = state after each token, Ac = product of abar.
  float hl[2][SUB], Ac[2][SUB];
  float rh[2] = {0.0f, 0.0f}, rA[2] = {1.0f, 1.0f};
  int ens[SUB];  // VARLEN: the sequence ending at each token (-1: none)
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int t = t0 + s;
    const bool ok = wok && t < a.T;
    const size_t idx = ((size_t)tl.b * a.T + t) * a.W + w;
    float2 xv = make_float2(0.f, 0.f), rv = xv, iv = xv;
    bool rst = false;
    int st = -1;
    ens[s] = -1;
    if (ok) {
      xv = Pair<XT>::load(x + idx);
      rv = Pair<LT>::load(lr + idx);
      iv = Pair<LT>::load(li + idx);
      if (CANON) rst = is_reset(a.reset_mask, a.segment_pos, (size_t)tl.b * a.T + t);
      if (VARLEN) {
        st = a.seq_start[(size_t)tl.b * a.T + t];
        ens[s] = a.seq_end[(size_t)tl.b * a.T + t];
      }
    }
    const float xs[2] = {xv.x, xv.y}, rs[2] = {rv.x, rv.y}, is[2] = {iv.x, iv.y};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float r = sigmoid_f(rs[j]);
      const float i = sigmoid_f(is[j]);
      const float la = nk[j] * r;
      float abar = expf(la);
      float m = sqrtf(one_minus_a2(la));
      if (rst) {
        abar = 0.0f;
        m = 1.0f;
      }
      if (!ok) {
        abar = 1.0f;
        m = 0.0f;
      }
      float ach = abar, bv = m * (i * xs[j]);  // the chain's decay and input
      if (VARLEN && st >= 0) {
        bv = fmaf(abar, a.h0s ? a.h0s[(size_t)st * a.W + w + j] : 0.0f, bv);
        ach = 0.0f;
      }
      rh[j] = fmaf(ach, rh[j], bv);
      rA[j] *= ach;
      hl[j][s] = rh[j];
      Ac[j][s] = rA[j];
    }
  }

  // Join the two halves: (A1, B1) o (A0, B0).
  float A0[2], B0[2], At[2], Bt[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    A0[j] = __shfl_sync(0xffffffffu, rA[j], pair);
    B0[j] = __shfl_sync(0xffffffffu, rh[j], pair);
    const float A1 = __shfl_sync(0xffffffffu, rA[j], pair + 16);
    const float B1 = __shfl_sync(0xffffffffu, rh[j], pair + 16);
    At[j] = A1 * A0[j];
    Bt[j] = fmaf(A1, B0[j], B1);
  }

  const size_t cidx = ((size_t)tl.b * a.nC + tl.c);
  uint32_t* my_flag = flags + cidx * a.ng + tl.g;
  const bool publish = (int)tl.ticket != a.drop_tile;
  // Every chunk publishes its aggregate (the chunks before DIST compose back to chunk 0).
  if (half == 1 && wok)
    *reinterpret_cast<float4*>(agg + cidx * a.W + w) = make_float4(At[0], Bt[0], At[1], Bt[1]);
  __threadfence();
  __syncwarp();
  if (lane == 16 && publish) st_release(my_flag, FLAG_AGG);
  // Look-back: the aggregates of the chunks after the anchor, applied to the state after the
  // anchor (or to h0).
  float hin[2] = {0.0f, 0.0f};
  {
    int an, n;
    lb_span<false>(tl.c, an, n);
    const uint32_t got = poll_flags<false>(flags + (size_t)tl.b * a.nC * a.ng + tl.g, a.ng, tl.c,
                                           n, an, a.nC, a.spin_limit, status);
    if (wok) {
      float2 hp = make_float2(0.0f, 0.0f);
      if (an >= 0) {
        if ((got >> n) & 1u)
          hp = __ldcg(reinterpret_cast<const float2*>(
              carry + ((size_t)tl.b * (a.nC + 1) + an + 1) * a.W + w));
      } else if (CANON && a.h0) {
        hp = make_float2(a.h0[(size_t)tl.b * a.W + w], a.h0[(size_t)tl.b * a.W + w + 1]);
      }
      lb_compose<false>(agg, (size_t)tl.b * a.nC, a.W, w, tl.c, n, got, a.nC, hp, hin);
    }
  }

  // Publish this chunk's boundary state (and, for chunk 0, the state entering it).
  const float he0 = fmaf(At[0], hin[0], Bt[0]);
  const float he1 = fmaf(At[1], hin[1], Bt[1]);
  if (wok) {
    float* crow = carry + (size_t)tl.b * (a.nC + 1) * a.W;
    if (half == 1)
      *reinterpret_cast<float2*>(crow + (size_t)(tl.c + 1) * a.W + w) = make_float2(he0, he1);
    if (half == 0 && tl.c == 0) *reinterpret_cast<float2*>(crow + w) = make_float2(hin[0], hin[1]);
    if (half == 1 && tl.c == a.nC - 1 && a.hT)
      *reinterpret_cast<float2*>(a.hT + (size_t)tl.b * a.W + w) = make_float2(he0, he1);
  }
  if (tl.c % LbPlan<false>::STEP == 0) {  // only anchors publish their state (warp-uniform)
    __threadfence();
    __syncwarp();
    if (lane == 16 && publish) st_release(my_flag, FLAG_INCL);
  }

  // Outputs: y = local state + (product of abar) * state entering this half.
  float hs[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) hs[j] = half == 0 ? hin[j] : fmaf(A0[j], hin[j], B0[j]);
  XT* y = static_cast<XT*>(a.y);
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int t = t0 + s;
    if (wok && t < a.T) {
      const size_t idx = ((size_t)tl.b * a.T + t) * a.W + w;
      const float y0 = fmaf(Ac[0][s], hs[0], hl[0][s]), y1 = fmaf(Ac[1][s], hs[1], hl[1][s]);
      Pair<XT>::store(y + idx, y0, y1);
      if (VARLEN && ens[s] >= 0 && a.hTs)
        *reinterpret_cast<float2*>(a.hTs + (size_t)ens[s] * a.W + w) = make_float2(y0, y1);
    }
  }
}

// Backward.  g_t = dL/dh_t obeys g_t = dy_t + abar_{t+1} g_{t+1} (g_{T-1} = dy + dhT), an
// affine scan in reverse: a chunk maps the carry entering it from the right, c_in =
// abar_{t1} g_{t1}, to the carry it passes left, c_out = abar_{t0} g_{t0}.  With
// dla = abar g (h_{t-1} - u abar / m) (u = i x; zero at reset tokens):
//   dlr = dla (-8 softplus) r (1 - r),  dx = g m i,  dli = g m u (1 - i),
//   dLambda partial = sum dla (-8 r)   (times sigmoid(Lambda) in the reduction).
// VARLEN: at a sequence's first token the chain's decay is 0 (no gradient flows to the
// sequence before) while abar keeps its value for the derivatives, h_{t-1} is h0[s], and
// dh0[s] = abar g; at its last token dhT[s] joins dy.
template <typename XT, typename LT, typename DXT, typename DLT, bool CANON, bool VARLEN>
__global__ void __launch_bounds__(128, 4) k_scan_bwd(ScanBwdArgs a) {
  uint32_t* status = reinterpret_cast<uint32_t*>(a.scratch);
  uint32_t* ticket = status + 1;
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.scratch + a.L.flags);
  float* rcar = reinterpret_cast<float*>(a.scratch + a.L.carry);
  float2* agg = reinterpret_cast<float2*>(a.scratch + a.L.agg);
  float* part = reinterpret_cast<float*>(a.scratch + a.L.part);

  const Tile tl = grab_tile(ticket, a.B, a.nC, a.ng, true);
  if (!tl.valid) return;
  const int lane = threadIdx.x & 31;
  const int pair = lane & 15, half = lane >> 4;
  const int w = tl.g * 32 + pair * 2;
  const bool wok = w < a.W;
  const int t0 = tl.c * SC + half * SUB;
  const XT* x = static_cast<const XT*>(a.x);
  const XT* dy = static_cast<const XT*>(a.dy);
  const LT* lr = static_cast<const LT*>(a.lr);
  const LT* li = static_cast<const LT*>(a.li);

  float nk[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) nk[j] = wok ? -8.0f * softplus_f(a.Lambda[w + j]) : 0.0f;
  float hin_tile[2] = {0.0f, 0.0f};
  if (wok) {
    const float2 h = *reinterpret_cast<const float2*>(a.fwd_carry + ((size_t)tl.b * (a.nC + 1) + tl.c) * a.W + w);
    hin_tile[0] = h.x;
    hin_tile[1] = h.y;
  }

  // Phase A: recompute the gates and the local forward scan of this half.
  float hp[2][SUB], ab[2][SUB], uu[2][SUB], mm[2][SUB], rr[2][SUB], ii[2][SUB], gy[2][SUB];
  float rh[2] = {0.0f, 0.0f}, rA[2] = {1.0f, 1.0f};
  int sts[SUB];          // VARLEN: the sequence starting at each token (-1: none)
  uint32_t smask = 0u;   // VARLEN: bit s = a sequence starts at token s of this half
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int t = t0 + s;
    const bool ok = wok && t < a.T;
    const size_t idx = ((size_t)tl.b * a.T + t) * a.W + w;
    float2 xv = make_float2(0.f, 0.f), rv = xv, iv = xv, dv = xv;
    bool rst = false;
    sts[s] = -1;
    if (ok) {
      xv = Pair<XT>::load(x + idx);
      dv = Pair<XT>::load(dy + idx);
      rv = Pair<LT>::load(lr + idx);
      iv = Pair<LT>::load(li + idx);
      if (CANON) rst = is_reset(a.reset_mask, a.segment_pos, (size_t)tl.b * a.T + t);
      if (VARLEN) {
        sts[s] = a.seq_start[(size_t)tl.b * a.T + t];
        const int en = a.seq_end[(size_t)tl.b * a.T + t];
        if (en >= 0 && a.dhTs) {
          dv.x += a.dhTs[(size_t)en * a.W + w];
          dv.y += a.dhTs[(size_t)en * a.W + w + 1];
        }
        if (sts[s] >= 0) smask |= 1u << s;
      }
    }
    const float xs[2] = {xv.x, xv.y}, rs[2] = {rv.x, rv.y}, is[2] = {iv.x, iv.y},
                ds[2] = {dv.x, dv.y};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float r = sigmoid_f(rs[j]);
      const float i = sigmoid_f(is[j]);
      const float la = nk[j] * r;
      float abar = expf(la);
      float m = sqrtf(one_minus_a2(la));
      if (rst) {
        abar = 0.0f;
        m = 1.0f;
      }
      if (!ok) {
        abar = 1.0f;
        m = 0.0f;
      }
      const float u = i * xs[j];
      hp[j][s] = rh[j];  // local state before token s
      float ach = abar, bv = m * u;  // the chain's decay and input
      if (VARLEN && sts[s] >= 0) {
        const float h0v = a.h0s ? a.h0s[(size_t)sts[s] * a.W + w + j] : 0.0f;
        hp[j][s] = h0v;  // the true h_{t-1} of a sequence's first token
        bv = fmaf(abar, h0v, bv);
        ach = 0.0f;
      }
      rh[j] = fmaf(ach, rh[j], bv);
      rA[j] *= ach;
      ab[j][s] = abar;
      uu[j][s] = u;
      mm[j][s] = m;
      rr[j][s] = r;
      ii[j][s] = i;
      gy[j][s] = ok ? ds[j] : 0.0f;
    }
  }
  // State entering this half, then the true h_{t-1} of every token.
  float hs[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float A0 = __shfl_sync(0xffffffffu, rA[j], pair);
    const float B0 = __shfl_sync(0xffffffffu, rh[j], pair);
    hs[j] = half == 0 ? hin_tile[j] : fmaf(A0, hin_tile[j], B0);
  }

  // Phase B: coefficients (linear in g) and the local reverse scan.
  float gl[2][SUB], Q[2][SUB], cr[2][SUB], ci[2][SUB], cx[2][SUB], cs[2][SUB];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float P = 1.0f;
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      const bool start = VARLEN && ((smask >> s) & 1u);
      const float hprev = start ? hp[j][s] : fmaf(P, hs[j], hp[j][s]);
      P *= start ? 0.0f : ab[j][s];
      const float abar = ab[j][s], m = mm[j][s], u = uu[j][s], r = rr[j][s], i = ii[j][s];
      // dla / g = abar (h_{t-1} - u abar / m); zero at reset tokens since abar = 0 there.
      // (Tokens past T carry m = 0 and take no part.)
      const float alpha =
          (abar == 0.0f || m == 0.0f) ? 0.0f : abar * (hprev - __fdividef(u * abar, m));
      cr[j][s] = alpha * nk[j] * r * (1.0f - r);
      ci[j][s] = m * u * (1.0f - i);
      cx[j][s] = m * i;
      cs[j][s] = alpha * (-8.0f * r);
    }
    float g = 0.0f, q = 1.0f;
#pragma unroll
    for (int s = SUB - 1; s >= 0; --s) {
      if (s < SUB - 1) {
        const float ach = (VARLEN && ((smask >> (s + 1)) & 1u)) ? 0.0f : ab[j][s + 1];
        g *= ach;
        q *= ach;
      }
      g += gy[j][s];
      gl[j][s] = g;
      Q[j][s] = q;
    }
  }
  // Half aggregates: c_out = abar_first (gloc_first + Q_first c_in).
  float Ah[2], Bh[2], A1[2], B1[2], At[2], Bt[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float ach0 = (VARLEN && (smask & 1u)) ? 0.0f : ab[j][0];
    Ah[j] = ach0 * Q[j][0];
    Bh[j] = ach0 * gl[j][0];
    A1[j] = __shfl_sync(0xffffffffu, Ah[j], pair + 16);
    B1[j] = __shfl_sync(0xffffffffu, Bh[j], pair + 16);
    const float A0 = __shfl_sync(0xffffffffu, Ah[j], pair);
    const float B0 = __shfl_sync(0xffffffffu, Bh[j], pair);
    At[j] = A0 * A1[j];  // the later half is applied first
    Bt[j] = fmaf(A0, B1[j], B0);
  }

  const size_t cidx = ((size_t)tl.b * a.nC + tl.c);
  uint32_t* my_flag = flags + cidx * a.ng + tl.g;
  const bool publish = (int)tl.ticket != a.drop_tile;
  const int q = a.nC - 1 - tl.c;  // processing order: from the last chunk
  if (half == 0 && wok)
    *reinterpret_cast<float4*>(agg + cidx * a.W + w) = make_float4(At[0], Bt[0], At[1], Bt[1]);
  __threadfence();
  __syncwarp();
  if (lane == 0 && publish) st_release(my_flag, FLAG_AGG);
  // Look-back toward the end: the aggregates of the chunks between this one and the anchor,
  // applied to the carry the anchor passes left (or to dhT).
  float cin[2] = {0.0f, 0.0f};
  {
    int an, n;
    lb_span<true>(q, an, n);
    const uint32_t got = poll_flags<true>(flags + (size_t)tl.b * a.nC * a.ng + tl.g, a.ng, q, n,
                                          an, a.nC, a.spin_limit, status);
    if (wok) {
      float2 cv = make_float2(0.0f, 0.0f);
      if (an >= 0) {
        if ((got >> n) & 1u)
          cv = __ldcg(reinterpret_cast<const float2*>(
              rcar + ((size_t)tl.b * a.nC + (a.nC - 1 - an)) * a.W + w));
      } else if (a.dhT) {
        cv = make_float2(a.dhT[(size_t)tl.b * a.W + w], a.dhT[(size_t)tl.b * a.W + w + 1]);
      }
      lb_compose<true>(agg, (size_t)tl.b * a.nC, a.W, w, q, n, got, a.nC, cv, cin);
    }
  }
  const float co0 = fmaf(At[0], cin[0], Bt[0]);
  const float co1 = fmaf(At[1], cin[1], Bt[1]);
  if (wok && half == 0) {
    *reinterpret_cast<float2*>(rcar + cidx * a.W + w) = make_float2(co0, co1);
    if (tl.c == 0 && a.dh0) {
      // dh0 = abar_0 g_0 = the carry chunk 0 passes left (zero in restricted mode).
      *reinterpret_cast<float2*>(a.dh0 + (size_t)tl.b * a.W + w) =
          CANON ? make_float2(co0, co1) : make_float2(0.0f, 0.0f);
    }
  }
  if ((a.nC - 1 - tl.c) % LbPlan<true>::STEP == 0) {  // only anchors publish (warp-uniform)
    __threadfence();
    __syncwarp();
    if (lane == 0 && publish) st_release(my_flag, FLAG_INCL);
  }

  // Outputs.
  float ch[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) ch[j] = half == 1 ? cin[j] : fmaf(A1[j], cin[j], B1[j]);
  DXT* dx = static_cast<DXT*>(a.dx);
  using DLE = typename OutPair<DLT>::E;
  DLE* dlr = static_cast<DLE*>(a.dlr);
  DLE* dli = static_cast<DLE*>(a.dli);
  float dsp[2] = {0.0f, 0.0f};
#pragma unroll
  for (int s = 0; s < SUB; ++s) {
    const int t = t0 + s;
    float g[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      g[j] = fmaf(Q[j][s], ch[j], gl[j][s]);
      dsp[j] = fmaf(g[j], cs[j][s], dsp[j]);
    }
    if (wok && t < a.T) {
      const size_t idx = ((size_t)tl.b * a.T + t) * a.W + w;
      if (VARLEN && sts[s] >= 0 && a.dh0s)  // d h0[s] = abar g at the sequence's first token
        *reinterpret_cast<float2*>(a.dh0s + (size_t)sts[s] * a.W + w) =
            make_float2(ab[0][s] * g[0], ab[1][s] * g[1]);
      Pair<DXT>::store(dx + idx, g[0] * cx[0][s], g[1] * cx[1][s]);
      OutPair<DLT>::store(dlr + idx, a.dl_plane, g[0] * cr[0][s], g[1] * cr[1][s]);
      OutPair<DLT>::store(dli + idx, a.dl_plane, g[0] * ci[0][s], g[1] * ci[1][s]);
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) dsp[j] += __shfl_xor_sync(0xffffffffu, dsp[j], 16);
  if (wok && half == 0)
    *reinterpret_cast<float2*>(part + cidx * a.W + w) = make_float2(dsp[0], dsp[1]);
}

// dLambda_w = sigmoid(Lambda_w) * sum over (b, chunk) rows of the partials, in a fixed order
// (deterministic): 16 row-groups per channel, combined in group order.
__global__ void __launch_bounds__(512) k_reduce_dlambda(const float* part, int rows, int W,
                                                        const float* Lambda, float* dLambda) {
  __shared__ float acc[16][33];
  const int lx = threadIdx.x & 31, gy = threadIdx.x >> 5;
  const int w = blockIdx.x * 32 + lx;
  float s = 0.0f;
  if (w < W)
    for (int r = gy; r < rows; r += 16) s += part[(size_t)r * W + w];
  acc[gy][lx] = s;
  __syncthreads();
  if (gy == 0 && w < W) {
    float t = 0.0f;
#pragma unroll
    for (int q = 0; q < 16; ++q) t += acc[q][lx];
    const float L = Lambda[w];
    dLambda[w] = t * __fdividef(1.0f, 1.0f + expf(-L));
  }
}

template <typename XT, typename LT, bool WITH_VARLEN = false>
cudaError_t fwd_dispatch_mode(const ScanFwdArgs& a, bool canonical, cudaStream_t s) {
  const size_t ntiles = (size_t)a.B * a.nC * a.ng;
  const unsigned grid = (unsigned)((ntiles + 3) / 4);
  if (WITH_VARLEN && a.seq_start)  // packed sequences: canonical, one row
    k_scan_fwd<XT, LT, true, WITH_VARLEN><<<grid, 128, 0, s>>>(a);
  else if (canonical)
    k_scan_fwd<XT, LT, true, false><<<grid, 128, 0, s>>>(a);
  else
    k_scan_fwd<XT, LT, false, false><<<grid, 128, 0, s>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

template <typename XT, typename LT, typename DXT, typename DLT, bool WITH_VARLEN = false>
cudaError_t bwd_dispatch_mode(const ScanBwdArgs& a, bool canonical, cudaStream_t s) {
  const size_t ntiles = (size_t)a.B * a.nC * a.ng;
  const unsigned grid = (unsigned)((ntiles + 3) / 4);
  if (WITH_VARLEN && a.seq_start)
    k_scan_bwd<XT, LT, DXT, DLT, true, WITH_VARLEN><<<grid, 128, 0, s>>>(a);
  else if (canonical)
    k_scan_bwd<XT, LT, DXT, DLT, true, false><<<grid, 128, 0, s>>>(a);
  else
    k_scan_bwd<XT, LT, DXT, DLT, false, false><<<grid, 128, 0, s>>>(a);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float* part = reinterpret_cast<const float*>(a.scratch + a.L.part);
  k_reduce_dlambda<<<(a.W + 31) / 32, 512, 0, s>>>(part, a.B * a.nC, a.W, a.Lambda, a.dLambda);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_fwd(const ScanFwdArgs& a, int xt, int lt, bool canonical,
                            cudaStream_t s) {
  if (xt == DT_F32 && lt == DT_F32) return fwd_dispatch_mode<float, float, true>(a, canonical, s);
  if (a.seq_start) return cudaErrorInvalidValue;  // packed sequences: float32 only here
  if (xt == DT_BF16 && lt == DT_BF16) return fwd_dispatch_mode<bf16, bf16>(a, canonical, s);
  if (xt == DT_BF16 && lt == DT_F32) return fwd_dispatch_mode<bf16, float>(a, canonical, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, int xt, int lt, int dxt, int dlt,
                            bool canonical, cudaStream_t s) {
  if (xt == DT_F32 && lt == DT_F32 && dxt == DT_F32 && dlt == DT_F32)
    return bwd_dispatch_mode<float, float, float, float, true>(a, canonical, s);
  if (a.seq_start) return cudaErrorInvalidValue;  // packed sequences: float32 only here
  if (xt == DT_BF16 && lt == DT_BF16 && dxt == DT_BF16 && dlt == DT_BF16)
    return bwd_dispatch_mode<bf16, bf16, bf16, bf16>(a, canonical, s);
  if (xt == DT_BF16 && lt == DT_BF16 && dxt == DT_F32 && dlt == DT_F32)
    return bwd_dispatch_mode<bf16, bf16, float, float>(a, canonical, s);
  if (xt == DT_BF16 && lt == DT_F32 && dxt == DT_BF16 && dlt == DT_F32)
    return bwd_dispatch_mode<bf16, float, bf16, float>(a, canonical, s);
  if (xt == DT_BF16 && lt == DT_F32 && dxt == DT_F32 && dlt == DT_F32)
    return bwd_dispatch_mode<bf16, float, float, float>(a, canonical, s);
  if (xt == DT_BF16 && lt == DT_F32 && dxt == DT_F32 && dlt == DT_SPLIT)
    return bwd_dispatch_mode<bf16, float, float, SplitBf16>(a, canonical, s);
  return cudaErrorInvalidValue;
}

}  // namespace rglru
