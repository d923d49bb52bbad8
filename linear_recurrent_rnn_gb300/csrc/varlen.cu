// Packed variable-length sequences: the token indices the fused kernels read.  Sequence s of
// a packed row covers tokens [cu[s], cu[s+1]) and is the layer on its own: its first token
// continues from the sequence's initial state h0[s] (zeros when none is given) with no reset,
// its last token's state is hT[s].  The kernels see, per token, which non-empty sequence
// starts there and which ends there; an empty sequence has hT = h0 (and dh0 = dhT).
#include "common.cuh"
#include "internal.h"

namespace rglru {

namespace {

__global__ void k_seq_clear(int32_t* seq_start, int32_t* seq_end, int T) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x)
    seq_start[t] = seq_end[t] = -1;
}

// One thread per sequence; entries outside [0, T) are ignored, so a malformed cu_seqlens
// gives wrong results but no out-of-bounds access.
__global__ void k_seq_mark(Varlen v, int T, int W, int32_t* seq_start, int32_t* seq_end,
                           bool backward) {
  for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < v.S; q += gridDim.x * blockDim.x) {
    const int a = v.cu_seqlens[q], b = v.cu_seqlens[q + 1];
    if (a < b) {
      if (a >= 0 && a < T) seq_start[a] = q;
      if (b - 1 >= 0 && b - 1 < T) seq_end[b - 1] = q;
    } else if (!backward && v.hT) {
      for (int w = 0; w < W; ++w) v.hT[(size_t)q * W + w] = v.h0 ? v.h0[(size_t)q * W + w] : 0.0f;
    } else if (backward && v.dh0) {
      for (int w = 0; w < W; ++w)
        v.dh0[(size_t)q * W + w] = v.dhT ? v.dhT[(size_t)q * W + w] : 0.0f;
    }
  }
}

}  // namespace

cudaError_t launch_seq_index(const Varlen& v, int T, int W, int32_t* seq_start,
                             int32_t* seq_end, bool backward, cudaStream_t s) {
  const int thr = 256;
  k_seq_clear<<<(T + thr - 1) / thr, thr, 0, s>>>(seq_start, seq_end, T);
  k_seq_mark<<<(v.S + thr - 1) / thr, thr, 0, s>>>(v, T, W, seq_start, seq_end, backward);
  note_launches(2);
  return cudaGetLastError();
}

}  // namespace rglru
