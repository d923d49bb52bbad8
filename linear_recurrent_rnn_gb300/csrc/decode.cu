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
  // The weight slices: 16-byte vectors, a batch of loads in flight per thread before any is
  // stored (a whole slice and rows of whole vectors), else element by element.
  constexpr int V = 16 / sizeof(T);  // elements per vector
  if (j0 + 32 <= k && (k * sizeof(T)) % 16 == 0) {
    constexpr int PR = 32 / V;        // vectors per row of the slice
    const int nvec = k * PR;          // per matrix
    for (int e0 = threadIdx.x; e0 < nvec; e0 += 4 * DEC_WARPS * 32) {
      uint4 va[4], vx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * DEC_WARPS * 32;
        if (e < nvec) {
          const size_t off = ((size_t)blk * k + e / PR) * k + j0 + (e % PR) * V;
          va[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wa) + off);
          vx[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.Wx) + off);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * DEC_WARPS * 32;
        if (e < nvec) {
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
    }
  } else {
    for (int e = threadIdx.x; e < k * 32; e += blockDim.x) {
      const int i = e >> 5, jj = j0 + (e & 31);
      const size_t wi = ((size_t)blk * k + i) * k + jj;
      swa[e] = jj < k ? ld_elem<T>(a.Wa, wi) : 0.0f;
      swx[e] = jj < k ? ld_elem<T>(a.Wx, wi) : 0.0f;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int jj = j0 + lane;  // the lane's channel within the block
  const bool live = jj < k;
  const int w = blk * k + jj;
  const float nk = live ? -8.0f * softplus_f(a.Lambda[w]) : 0.0f;
  const float bra = (live && a.ba) ? a.ba[w] : 0.0f;
  const float brx = (live && a.bx) ? a.bx[w] : 0.0f;
  float* xs = sxr + warp * DEC_RW * k;
  const int row0 = blockIdx.y * DEC_ROWS;
  for (int r0 = warp * DEC_RW; r0 < DEC_ROWS; r0 += DEC_WARPS * DEC_RW) {
    if (row0 + r0 >= a.B) break;
    // the x segments of rows row0 + r0 .. + DEC_RW - 1 (zeros past B): 16-byte vectors,
    // all of a lane's in flight at once, when the rows split into whole vectors
    if ((k * sizeof(T)) % 16 == 0) {
      const int PR = k / V;  // vectors per row segment
      for (int e0 = lane; e0 < DEC_RW * PR; e0 += 8 * 32) {
        uint4 vv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + u * 32, rr = e / PR, b = row0 + r0 + rr;
          if (e < DEC_RW * PR && b < a.B)
            vv[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + (size_t)b * a.W +
                                                    (size_t)blk * k + (e % PR) * V);
          else
            vv[u] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + u * 32;
          if (e < DEC_RW * PR) {
            const T* pv = reinterpret_cast<const T*>(&vv[u]);
            float* dst = xs + (e / PR) * k + (e % PR) * V;
#pragma unroll
            for (int c = 0; c < V; ++c) dst[c] = to_f32<T>(pv[c]);
          }
        }
      }
    } else {
      for (int e = lane; e < DEC_RW * k; e += 32) {
        const int rr = e / k, i = e - rr * k;
        const int b = row0 + r0 + rr;
        xs[e] = b < a.B ? ld_elem<T>(a.x, (size_t)b * a.W + (size_t)blk * k + i) : 0.0f;
      }
    }
    __syncwarp();
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
      if (a.canonical && a.reset && a.reset[b]) {
        abar = 0.0f;
        m = 1.0f;
      }
      const size_t o = (size_t)b * a.W + w;
      const float hp = a.h_in ? a.h_in[o] : 0.0f;
      const float h = fmaf(abar, hp, m * (ig * xs[rr * k + jj]));
      static_cast<T*>(a.y)[o] = from_f32<T>(h);
      a.h_out[o] = h;
    }
    __syncwarp();
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
