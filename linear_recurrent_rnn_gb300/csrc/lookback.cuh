// Anchored look-back over value slots (see common.cuh), shared by the fused kernels.
//
// The carry entering a chunk is  compose(agg[k_1], ..., agg[k_n]) applied to the boundary
// state published by the nearest anchor chunk, where k_1 is the neighbouring chunk and k_n the
// one next to the anchor.  All n aggregate slots and the anchor's slot are requested at once
// (n <= ANCHOR - 1), so the wait costs about one L2 round trip when the slots are already
// filled; an empty slot is re-polled with a bounded spin.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace rglru {

// Split form: lookback_issue requests every slot at once (and returns immediately); the values
// are consumed later by lookback_finish, which re-polls the slots that were still empty.  A
// caller issues the requests, does other work, then finishes: the L2 round trip is hidden.
struct LookbackReq {
  uint64_t v[ANCHOR - 1];
  uint32_t hv;
};

__device__ __forceinline__ void lookback_issue(LookbackReq& q, const float2* first_agg,
                                               long agg_step, int n, const float* anchor_state) {
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s)
    q.v[s] = s < n ? ld_relaxed_u64(first_agg + s * agg_step) : 0ull;
  q.hv = ld_relaxed_u32(anchor_state);
}

__device__ __forceinline__ float lookback_finish(LookbackReq& q, const float2* first_agg,
                                                 long agg_step, int n, const float* anchor_state,
                                                 int limit, uint32_t* status) {
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s) {
    if (s < n) {
      int it = 0;
      while (q.v[s] == SLOT_EMPTY64) {
        if (++it > limit) {
          atomicOr(status, STATUS_TIMEOUT);
          q.v[s] = (uint64_t)__float_as_uint(1.0f);  // identity (A = 1, B = 0)
          break;
        }
        __nanosleep(64);
        q.v[s] = ld_relaxed_u64(first_agg + s * agg_step);
      }
    }
  }
  {
    int it = 0;
    while (q.hv == SLOT_EMPTY32) {
      if (++it > limit) {
        atomicOr(status, STATUS_TIMEOUT);
        q.hv = 0u;
        break;
      }
      __nanosleep(64);
      q.hv = ld_relaxed_u32(anchor_state);
    }
  }
  float accA = 1.0f, accB = 0.0f;
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s) {
    if (s < n) {
      const float A = __uint_as_float((uint32_t)(q.v[s] & 0xffffffffu));
      const float B = __uint_as_float((uint32_t)(q.v[s] >> 32));
      accB = fmaf(accA, B, accB);
      accA *= A;
    }
  }
  return fmaf(accA, __uint_as_float(q.hv), accB);
}

// first_agg: slot of k_1; agg_step: element offset from k_i to k_{i+1} (+-W); n: number of
// aggregates to compose; anchor_state: slot of the anchor's boundary state.  A slot that
// stays empty past `limit` polls counts as the identity (or a zero state), and the timeout is
// recorded in *status.
__device__ __forceinline__ float lookback_carry(const float2* first_agg, long agg_step, int n,
                                                const float* anchor_state, int limit,
                                                uint32_t* status) {
  uint64_t v[ANCHOR - 1];
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s)
    v[s] = s < n ? ld_relaxed_u64(first_agg + s * agg_step) : 0ull;
  uint32_t hv = ld_relaxed_u32(anchor_state);
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s) {
    if (s < n) {
      int it = 0;
      while (v[s] == SLOT_EMPTY64) {
        if (++it > limit) {
          atomicOr(status, STATUS_TIMEOUT);
          v[s] = (uint64_t)__float_as_uint(1.0f);  // identity (A = 1, B = 0)
          break;
        }
        __nanosleep(64);
        v[s] = ld_relaxed_u64(first_agg + s * agg_step);
      }
    }
  }
  {
    int it = 0;
    while (hv == SLOT_EMPTY32) {
      if (++it > limit) {
        atomicOr(status, STATUS_TIMEOUT);
        hv = 0u;
        break;
      }
      __nanosleep(64);
      hv = ld_relaxed_u32(anchor_state);
    }
  }
  float accA = 1.0f, accB = 0.0f;
#pragma unroll
  for (int s = 0; s < ANCHOR - 1; ++s) {
    if (s < n) {
      const float A = __uint_as_float((uint32_t)(v[s] & 0xffffffffu));
      const float B = __uint_as_float((uint32_t)(v[s] >> 32));
      accB = fmaf(accA, B, accB);
      accA *= A;
    }
  }
  return fmaf(accA, __uint_as_float(hv), accB);
}

}  // namespace rglru
