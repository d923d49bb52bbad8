// Anchored look-back over value slots (see common.cuh), shared by the fused kernels.
//
// Chunks are counted in processing order (from the start in the forward, from the end in the
// backward): chunk q publishes its affine aggregate and, once it knows its carry-in, the carry
// it passes on.  Its own carry-in is compose(agg[q-1], ..., agg[a+1]) applied to the carry
// passed on by the anchor chunk a, the nearest multiple of 2^shift at least `dist` chunks
// back (or, for q < dist, to the initial value: h0 or dh_T).  Every carry is thus one fixed
// expression of the inputs, whatever the timing, so the scan is bitwise deterministic; and
// with dist = ceil(P / B) the anchor's tile sits at least one full round of the CTAs' tile
// loop earlier, so its carry is normally published well before it is read.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace rglru {

// The slots of one look-back are all requested at once (lookback_issue, which returns at
// once), consumed later (lookback_finish, which re-polls any slot that was still empty): the
// L2 round trip hides behind the work in between.
struct LookbackReq {
  uint64_t v[LB_SLOTS];
  uint32_t hv;
};

// Where chunk q (processing order) looks back to: n = aggregates to compose, anchor = the
// processing-order index of the anchor chunk (-1: the initial value).
struct LookbackSpan {
  int n, anchor;
};
__device__ __forceinline__ LookbackSpan lookback_span(int q, int dist, int shift) {
  LookbackSpan s;
  s.anchor = q >= dist ? ((q - dist) >> shift) << shift : -1;
  s.n = q - 1 - s.anchor;
  return s;
}

// first_agg: slot of chunk q-1 (processing order); agg_step: element offset to the next older
// chunk's slot; anchor_state: the anchor's carry slot, or null to use init (the initial value).
__device__ __forceinline__ void lookback_issue(LookbackReq& q, const float2* first_agg,
                                               long agg_step, int n, const float* anchor_state,
                                               float init) {
#pragma unroll
  for (int s = 0; s < LB_SLOTS; ++s)
    q.v[s] = s < n ? ld_relaxed_u64(first_agg + s * agg_step) : 0ull;
  q.hv = anchor_state ? ld_relaxed_u32(anchor_state) : slot_enc1(init);
}

// Re-requests every slot that was still empty when it was last read, and returns at once: a
// caller that knows when the missing aggregates are likely to have been published (the tiles
// processed alongside its own publish theirs at about the same point of their loop) requests
// them again there, so that the round trip overlaps its work before lookback_finish.
__device__ __forceinline__ void lookback_refresh(LookbackReq& q, const float2* first_agg,
                                                 long agg_step, int n, const float* anchor_state) {
#pragma unroll
  for (int s = 0; s < LB_SLOTS; ++s)
    if (s < n && q.v[s] == SLOT_EMPTY64) q.v[s] = ld_relaxed_u64(first_agg + s * agg_step);
  if (anchor_state != nullptr && q.hv == SLOT_EMPTY32) q.hv = ld_relaxed_u32(anchor_state);
}

// A slot that stays empty past `limit` polls counts as the identity (or a zero carry), and the
// timeout is recorded in *status.  Every slot still empty is re-requested in the same round,
// so a round costs one L2 round trip however many slots were late.
__device__ __forceinline__ float lookback_finish(LookbackReq& q, const float2* first_agg,
                                                 long agg_step, int n, const float* anchor_state,
                                                 int limit, uint32_t* status) {
  for (int round = 0;; ++round) {
    bool pending = anchor_state != nullptr && q.hv == SLOT_EMPTY32;
#pragma unroll
    for (int s = 0; s < LB_SLOTS; ++s) pending |= s < n && q.v[s] == SLOT_EMPTY64;
    if (!pending) break;
    if (round >= limit) {
      atomicOr(status, STATUS_TIMEOUT);
#pragma unroll
      for (int s = 0; s < LB_SLOTS; ++s)
        if (q.v[s] == SLOT_EMPTY64) q.v[s] = slot_enc2(1.0f, 0.0f);  // the identity map
      if (q.hv == SLOT_EMPTY32) q.hv = slot_enc1(0.0f);
      break;
    }
    __nanosleep(32);
#pragma unroll
    for (int s = 0; s < LB_SLOTS; ++s)
      if (s < n && q.v[s] == SLOT_EMPTY64) q.v[s] = ld_relaxed_u64(first_agg + s * agg_step);
    if (anchor_state != nullptr && q.hv == SLOT_EMPTY32) q.hv = ld_relaxed_u32(anchor_state);
  }
  // compose from the anchor's side: the oldest aggregate first
  float c = slot_dec1(q.hv);
#pragma unroll
  for (int s = LB_SLOTS - 1; s >= 0; --s) {
    if (s < n) {
      const float2 ab = slot_dec2(q.v[s]);
      c = fmaf(ab.x, c, ab.y);
    }
  }
  return c;
}

}  // namespace rglru
