// One decode step of the RG-LRU layer: a single token per row, with the rows' states carried
// in and out, for inference loops that feed the layer one token at a time.
//
// Sources ("Fattori comparison" page): the semantic-limits list asks for an initial state and
// for T = 1 (the prior art rejects both); a step is the forward of one token from a carried
// state.  Per row b and channel w (gate block blk, k = W / nblk):
//   lr = x_blk Wa[blk] + ba,  li = x_blk Wx[blk] + bx       (the block-diagonal projections)
//   r = sigmoid(lr), i = sigmoid(li), la = -8 r softplus(Lambda), a = e^la
//   canonical reset row: abar = 0, m = 1; otherwise abar = a, m = sqrt(1 - a^2)
//   h_out = abar h_in + m i x,  y = h_out.
//
// Geometry: a CTA owns a 32-channel slice of one gate block (its Wa and Wx columns staged
// once in shared memory as float32) and up to 32 rows; each warp takes rows in turn, four at
// a time, lane = channel: the four rows' x segments go to shared memory and every lane runs
// its two dot products over the block's k inputs with the weights shared by the four rows.
// The gate arithmetic is the CUDA-core forward's (accurate exp / expm1 / log1p forms).
#include "common.cuh"
#include "internal.h"

namespace rglru {

namespace {

constexpr int DEC_WARPS = 8;  // warps per CTA
constexpr int DEC_ROWS = 32;  // rows per CTA
constexpr int DEC_RW = 4;     // rows a warp runs at once

struct DecArgs {
  int B, W, k, canonical;
  const void* x;
  const void* Wa;
  const float* ba;
  const void* Wx;
  const float* bx;
  const float* Lambda;
  const uint8_t* reset;
  const float* h_in;
  void* y;
  float* h_out;
};

template <typename T>
__device__ __forceinline__ float ld_elem(const void* p, size_t i) {
  return to_f32<T>(static_cast<const T*>(p)[i]);
}

template <typename T>
__global__ void __launch_bounds__(DEC_WARPS * 32) k_step(DecArgs a) {
  extern __shared__ float sm[];
  const int k = a.k;
  const int nsl = (k + 31) / 32;
  const int blk = blockIdx.x / nsl, j0 = (blockIdx.x % nsl) * 32;
  float* swa = sm;                 // [k][32] float32: Wa[blk][i][j0 + c]
  float* swx = sm + k * 32;        // [k][32]: Wx
  float* sxr = swx + k * 32;       // [warp][DEC_RW][k]: x segments of the warp's rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int jj = j0 + lane;  // the lane's channel within the block
  const bool live = jj < k;
  const int w = blk * k + jj;
  const int r0 = warp * DEC_RW;  // the warp's rows: row0 + r0 .. + DEC_RW - 1
  const int row0 = blockIdx.y * DEC_ROWS;
  float* xs = sxr + warp * DEC_RW * k;
  constexpr int V = 16 / sizeof(T);  // elements per vector
  const bool vec = (k * sizeof(T)) % 16 == 0;
  // Every independent global load of the step is issued before any is waited for (one memory
  // round trip): the weight slices, the warp's x rows, the lane's per-channel constants, and
  // the states and reset flags of the warp's rows.
  uint4 va[4], vx[4], xv[8];
  const bool wvec = vec && j0 + 32 <= k;
  constexpr int PR = 32 / V;  // vectors per row of a weight slice
  if (wvec) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = threadIdx.x + u * DEC_WARPS * 32;
      if (e < k * PR) {
        const size_t off = ((size_t)blk * k + e / PR) * k + j0 + (e % PR) * V;
        va[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wa) + off);
        vx[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wx) + off);
      }
    }
  }
  const int XPR = k / V;  // vectors per x row segment
  if (vec) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane + u * 32, rr = e / XPR, b = row0 + r0 + rr;
      xv[u] = (e < DEC_RW * XPR && b < a.B)
                  ? *reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + (size_t)b * a.W +
                                                    (size_t)blk * k + (e % XPR) * V)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const float lam = live ? a.Lambda[w] : 0.0f;
  const float bra = (live && a.ba) ? a.ba[w] : 0.0f;
  const float brx = (live && a.bx) ? a.bx[w] : 0.0f;
  float hp[DEC_RW];
  bool rst[DEC_RW];
#pragma unroll
  for (int rr = 0; rr < DEC_RW; ++rr) {
    const int b = row0 + r0 + rr;
    hp[rr] = (live && b < a.B && a.h_in) ? a.h_in[(size_t)b * a.W + w] : 0.0f;
    rst[rr] = (b < a.B && a.canonical && a.reset) ? a.reset[b] != 0 : false;
  }
  // the weight slices into shared memory as float32
  if (wvec) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = threadIdx.x + u * DEC_WARPS * 32;
      if (e < k * PR) {
        const T* pa = reinterpret_cast<const T*>(&va[u]);
        const T* px = reinterpret_cast<const T*>(&vx[u]);
        float* da = swa + (e / PR) * 32 + (e % PR) * V;
        float* dxw = swx + (e / PR) * 32 + (e % PR) * V;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          da[c] = to_f32<T>(pa[c]);
          dxw[c] = to_f32<T>(px[c]);
        }
      }
    }
    // slices wider than four vectors per thread (k > 512 / V ... not reached for k <= STEP_KMAX
    // at bf16: 4 x 256 threads x 8 elements = 8192 = 256 rows x 32 columns)
    for (int e = threadIdx.x + 4 * DEC_WARPS * 32; e < k * PR; e += DEC_WARPS * 32) {
      const size_t off = ((size_t)blk * k + e / PR) * k + j0 + (e % PR) * V;
      const uint4 ua = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wa) + off);
      const uint4 ux = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wx) + off);
      const T* pa = reinterpret_cast<const T*>(&ua);
      const T* px = reinterpret_cast<const T*>(&ux);
#pragma unroll
      for (int c = 0; c < V; ++c) {
        swa[(e / PR) * 32 + (e % PR) * V + c] = to_f32<T>(pa[c]);
        swx[(e / PR) * 32 + (e % PR) * V + c] = to_f32<T>(px[c]);
      }
    }
  } else {
    for (int e = threadIdx.x; e < k * 32; e += blockDim.x) {
      const int i = e >> 5, jc = j0 + (e & 31);
      const size_t wi = ((size_t)blk * k + i) * k + jc;
      swa[e] = jc < k ? ld_elem<T>(a.Wa, wi) : 0.0f;
      swx[e] = jc < k ? ld_elem<T>(a.Wx, wi) : 0.0f;
    }
  }
  // the warp's x rows into shared memory (zeros past B)
  if (vec) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = lane + u * 32;
      if (e < DEC_RW * XPR) {
        const T* pv = reinterpret_cast<const T*>(&xv[u]);
        float* dst = xs + (e / XPR) * k + (e % XPR) * V;
#pragma unroll
        for (int c = 0; c < V; ++c) dst[c] = to_f32<T>(pv[c]);
      }
    }
    for (int e = lane + 8 * 32; e < DEC_RW * XPR; e += 32) {  // x rows of more than 8 x 32 vectors
      const int rr = e / XPR, b = row0 + r0 + rr;
      uint4 u4 = make_uint4(0u, 0u, 0u, 0u);
      if (b < a.B)
        u4 = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + (size_t)b * a.W +
                                             (size_t)blk * k + (e % XPR) * V);
      const T* pv = reinterpret_cast<const T*>(&u4);
      float* dst = xs + rr * k + (e % XPR) * V;
#pragma unroll
      for (int c = 0; c < V; ++c) dst[c] = to_f32<T>(pv[c]);
    }
  } else {
    for (int e = lane; e < DEC_RW * k; e += 32) {
      const int rr = e / k, i = e - rr * k;
      const int b = row0 + r0 + rr;
      xs[e] = b < a.B ? ld_elem<T>(a.x, (size_t)b * a.W + (size_t)blk * k + i) : 0.0f;
    }
  }
  __syncthreads();
  if (row0 + r0 >= a.B) return;  // no rows for this warp (after the block-wide barrier)
  const float nk = -8.0f * softplus_f(lam);
  float lr[DEC_RW], li[DEC_RW];
#pragma unroll
  for (int rr = 0; rr < DEC_RW; ++rr) lr[rr] = bra, li[rr] = brx;
  for (int i = 0; i < k; ++i) {
    const float wa = swa[i * 32 + lane], wx = swx[i * 32 + lane];
#pragma unroll
    for (int rr = 0; rr < DEC_RW; ++rr) {
      const float xi = xs[rr * k + i];
      lr[rr] = fmaf(xi, wa, lr[rr]);
      li[rr] = fmaf(xi, wx, li[rr]);
    }
  }
#pragma unroll
  for (int rr = 0; rr < DEC_RW; ++rr) {
    const int b = row0 + r0 + rr;
    if (!live || b >= a.B) continue;
    const float rg = sigmoid_f(lr[rr]);
    const float ig = sigmoid_f(li[rr]);
    const float la = nk * rg;
    float abar = expf(la);
    float m = sqrtf(one_minus_a2(la));
    if (rst[rr]) {
      abar = 0.0f;
      m = 1.0f;
    }
    const size_t o = (size_t)b * a.W + w;
    const float h = fmaf(abar, hp[rr], m * (ig * xs[rr * k + jj]));
    static_cast<T*>(a.y)[o] = from_f32<T>(h);
    a.h_out[o] = h;
  }
}

}  // namespace

size_t step_smem_bytes(int k) { return (size_t)(2 * 32 + DEC_WARPS * DEC_RW) * k * 4; }

cudaError_t launch_step(const Dims& d, const void* x, const void* Wa, const float* ba,
                        const void* Wx, const float* bx, const float* Lambda,
                        const uint8_t* reset, const float* h_in, void* y, float* h_out,
                        cudaStream_t s) {
  DecArgs a;
  a.B = d.B;
  a.W = d.W;
  a.k = d.k;
  a.canonical = d.mode == RGLRU_CANONICAL;
  a.x = x;
  a.Wa = Wa;
  a.ba = ba;
  a.Wx = Wx;
  a.bx = bx;
  a.Lambda = Lambda;
  a.reset = reset;
  a.h_in = h_in;
  a.y = y;
  a.h_out = h_out;
  const size_t smem = step_smem_bytes(d.k);
  const dim3 grid((unsigned)(d.nblk * ((d.k + 31) / 32)), (unsigned)((d.B + DEC_ROWS - 1) / DEC_ROWS));
  cudaError_t e;
  if (d.io == RGLRU_BF16) {
    e = cudaFuncSetAttribute(k_step<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) k_step<bf16><<<grid, DEC_WARPS * 32, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(k_step<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) k_step<float><<<grid, DEC_WARPS * 32, smem, s>>>(a);
  }
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rglru
