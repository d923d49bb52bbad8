// Packed variable-length sequences: the token indices the fused kernels read.  Sequence s of
// a packed row covers tokens [cu[s], cu[s+1]) and is the layer on its own: its first token
// continues from the sequence's initial state h0[s] (zeros when none is given) with no reset,
// its last token's state is hT[s].  The kernels see, per token, which non-empty sequence
// starts there and which ends there; an empty sequence has hT = h0 (and dh0 = dhT).
#include "common.cuh"
#include "internal.h"

namespace rglru {

namespace {

// The sequence holding token t: the largest s in [0, S) with cu[s] <= t (with non-decreasing
// offsets, the one non-empty sequence whose range contains t).  Reads cu[0 .. S] only, so a
// malformed array gives a wrong index but never an out-of-bounds one.
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int S, int t) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One thread per token (its start and end index) and per sequence (hT = h0 for an empty one),
// in a single launch.
__global__ void k_seq_index(Varlen v, int T, int W, int32_t* seq_start, int32_t* seq_end) {
  const int n = T > v.S ? T : v.S;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (i < T) {
      const int s = seq_of_token(v.cu_seqlens, v.S, i);
      seq_start[i] = v.cu_seqlens[s] == i ? s : -1;
      seq_end[i] = v.cu_seqlens[s + 1] == i + 1 ? s : -1;
    }
    if (i < v.S && v.hT && v.cu_seqlens[i] >= v.cu_seqlens[i + 1]) {
      for (int w = 0; w < W; ++w) v.hT[(size_t)i * W + w] = v.h0 ? v.h0[(size_t)i * W + w] : 0.0f;
    }
  }
}

// The backward's part: dh0 = dhT for every empty sequence (the token indices are the
// forward's, kept in `saved`).
__global__ void k_seq_empty_dh0(Varlen v, int W) {
  for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < v.S; q += gridDim.x * blockDim.x) {
    if (v.cu_seqlens[q] >= v.cu_seqlens[q + 1]) {
      for (int w = 0; w < W; ++w)
        v.dh0[(size_t)q * W + w] = v.dhT ? v.dhT[(size_t)q * W + w] : 0.0f;
    }
  }
}

}  // namespace

cudaError_t launch_seq_index(const Varlen& v, int T, int W, int32_t* seq_start,
                             int32_t* seq_end, cudaStream_t s) {
  const int thr = 256;
  const int n = T > v.S ? T : v.S;
  k_seq_index<<<(n + thr - 1) / thr, thr, 0, s>>>(v, T, W, seq_start, seq_end);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_seq_empty_dh0(const Varlen& v, int W, cudaStream_t s) {
  const int thr = 128;
  k_seq_empty_dh0<<<(v.S + thr - 1) / thr, thr, 0, s>>>(v, W);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rglru
