// Block-diagonal gate projections and their backward on CUDA cores, float32 accumulation.
//
// Gate logits ("Fattori comparison" page, first paragraph: two block-diagonal projections of
// the recurrent input): for gate block blk of width k, lr[n, blk*k + j] =
// sum_i x[n, blk*k + i] Wa[blk][i][j] + ba[blk*k + j] (li likewise with Wx, bx).  The backward
// (the benchmark record scopes the projections into the measured layer): dx += dlr Wa^T +
// dli Wx^T, dW = x^T dl, db = sum_n dl.
//
// These kernels serve the shapes the tensor-core projections (proj_tc.cu) do not take: float32
// I/O, whose 1e-5 parity bound a bf16 tensor-core product cannot meet, and gate blocks that
// are not a multiple of 16 or wider than 160 channels.  Every kernel computes a 64 x 64 output
// tile per 256-thread block
// (4 x 4 per thread) through 16-deep shared-memory slabs; tails in k and in the token count
// are guarded.
#include "common.cuh"
#include "internal.h"

namespace rglru {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// OUT[n, blk*k + j] = sum_i X[n, blk*k + i] Wm[blk][i][j] + bias   (gate = blockIdx.z)
template <typename XT, typename OT>
__global__ void __launch_bounds__(256) k_proj(int BT, int W, int k, const XT* x, const XT* Wa,
                                              const float* ba, const XT* Wx, const float* bx,
                                              OT* lr, OT* li) {
  __shared__ float Xs[TK][TM + 4];
  __shared__ float Ws[TK][TN + 4];
  const int gate = blockIdx.z;
  const XT* Wm = gate ? Wx : Wa;
  const float* bias = gate ? bx : ba;
  OT* out = gate ? li : lr;
  const int ntile_n = (k + TN - 1) / TN;
  const int blk = blockIdx.y / ntile_n;
  const int j0 = (blockIdx.y % ntile_n) * TN;
  const int n0 = blockIdx.x * TM;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int i0 = 0; i0 < k; i0 += TK) {
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      const int r = e / TK, c = e % TK;  // token r, in-channel i0 + c
      const int n = n0 + r, i = i0 + c;
      Xs[c][r] = (n < BT && i < k) ? to_f32(x[(size_t)n * W + (size_t)blk * k + i]) : 0.0f;
    }
    for (int e = threadIdx.x; e < TK * TN; e += 256) {
      const int r = e / TN, c = e % TN;  // in-channel i0 + r, out-channel j0 + c
      const int i = i0 + r, j = j0 + c;
      Ws[r][c] = (i < k && j < k) ? to_f32(Wm[((size_t)blk * k + i) * k + j]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < TK; ++q) {
      float xa[4], wb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        xa[u] = Xs[q][ty * 4 + u];
        wb[u] = Ws[q][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(xa[u], wb[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int n = n0 + ty * 4 + u;
    if (n >= BT) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j < k) {
        const float b = bias ? bias[(size_t)blk * k + j] : 0.0f;
        out[(size_t)n * W + (size_t)blk * k + j] = from_f32<OT>(acc[u][v] + b);
      }
    }
  }
}

// DX[n, blk*k + i] = (dx_in ? dx_in : DX)[n, blk*k + i] + sum_j (Gr[n, blk*k+j] Wa[blk][i][j] + Gi[n, blk*k+j] Wx[blk][i][j])
template <typename WT, typename GT, typename DXT>
__global__ void __launch_bounds__(256) k_dx(int BT, int W, int k, const GT* gr, const GT* gi,
                                            const WT* Wa, const WT* Wx, const float* dx_in,
                                            DXT* dx) {
  __shared__ float Gs[TK][TM + 4];
  __shared__ float Ws[TK][TN + 4];
  const int ntile_n = (k + TN - 1) / TN;
  const int blk = blockIdx.y / ntile_n;
  const int i0t = (blockIdx.y % ntile_n) * TN;
  const int n0 = blockIdx.x * TM;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int gate = 0; gate < 2; ++gate) {
    const GT* g = gate ? gi : gr;
    const WT* Wm = gate ? Wx : Wa;
    for (int j0 = 0; j0 < k; j0 += TK) {
      for (int e = threadIdx.x; e < TM * TK; e += 256) {
        const int r = e / TK, c = e % TK;
        const int n = n0 + r, j = j0 + c;
        Gs[c][r] = (n < BT && j < k) ? to_f32(g[(size_t)n * W + (size_t)blk * k + j]) : 0.0f;
      }
      for (int e = threadIdx.x; e < TK * TN; e += 256) {
        const int c = e / TN, r = e % TN;  // j = j0 + c, i = i0t + r
        const int i = i0t + r, j = j0 + c;
        Ws[c][r] = (i < k && j < k) ? to_f32(Wm[((size_t)blk * k + i) * k + j]) : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < TK; ++q) {
        float ga[4], wb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ga[u] = Gs[q][ty * 4 + u];
          wb[u] = Ws[q][tx * 4 + u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(ga[u], wb[v], acc[u][v]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int n = n0 + ty * 4 + u;
    if (n >= BT) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = i0t + tx * 4 + v;
      if (i < k) {
        const size_t e = (size_t)n * W + (size_t)blk * k + i;
        const float base = dx_in ? dx_in[e] : to_f32(dx[e]);
        dx[e] = from_f32<DXT>(base + acc[u][v]);
      }
    }
  }
}

// Split-K partials of dW[gate][blk][i][j] = sum_{n in split} X[n, blk*k+i] G[n, blk*k+j].
template <typename XT, typename GT>
__global__ void __launch_bounds__(256) k_dw_part(int BT, int W, int k, int nblk, int splits,
                                                 const XT* x, const GT* gr, const GT* gi,
                                                 float* part) {
  __shared__ float Xs[TK][TM + 4];
  __shared__ float Gs[TK][TN + 4];
  const int nt = (k + 63) / 64;
  const int ti = blockIdx.x / nt, tj = blockIdx.x % nt;
  const int i0 = ti * 64, j0 = tj * 64;
  const int gate = blockIdx.y % 2, blk = blockIdx.y / 2;
  const int split = blockIdx.z;
  const GT* g = gate ? gi : gr;
  const long per = (BT + splits - 1) / splits;
  const long nb = split * per, ne = min((long)BT, nb + per);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // Each TK-row slab is summed on its own, then added to the running sums with a compensation
  // term (Kahan): a plain float32 running sum over a split's hundreds to thousands of rows
  // drifts by up to (rows x 2^-24) of the result where the products share a sign (the
  // diagonal of dW), beyond the float32 bound of 1e-5.
  float acc[4][4] = {}, cmp[4][4] = {};
  for (long nn = nb; nn < ne; nn += TK) {
    for (int e = threadIdx.x; e < TK * 64; e += 256) {
      const int r = e / 64, c = e % 64;
      const long n = nn + r;
      const int i = i0 + c, j = j0 + c;
      const bool okn = n < ne;
      Xs[r][c] = (okn && i < k) ? to_f32(x[(size_t)n * W + (size_t)blk * k + i]) : 0.0f;
      Gs[r][c] = (okn && j < k) ? to_f32(g[(size_t)n * W + (size_t)blk * k + j]) : 0.0f;
    }
    __syncthreads();
    float sl[4][4] = {};
#pragma unroll
    for (int q = 0; q < TK; ++q) {
      float xa[4], gb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        xa[u] = Xs[q][ty * 4 + u];
        gb[u] = Gs[q][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) sl[u][v] = fmaf(xa[u], gb[v], sl[u][v]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float yv = __fsub_rn(sl[u][v], cmp[u][v]);
        const float t = __fadd_rn(acc[u][v], yv);
        cmp[u][v] = __fsub_rn(__fsub_rn(t, acc[u][v]), yv);
        acc[u][v] = t;
      }
    __syncthreads();
  }
  float* P = part + (((size_t)split * 2 + gate) * nblk + blk) * (size_t)k * k;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= k) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j < k) P[(size_t)i * k + j] = acc[u][v];
    }
  }
}

// Split partials of the bias gradients: dbp[split][gate][w] = sum_{n in split} G[n, w].  A
// thread takes two channels (one 4- or 8-byte load per token) and four interleaved running
// sums, combined in a fixed order, so the result does not depend on timing.
template <typename GT>
__global__ void __launch_bounds__(256) k_db_part(int BT, int W, int splits, const GT* gr,
                                                 const GT* gi, float* dbp) {
  const int w = (blockIdx.x * 256 + threadIdx.x) * 2;
  const int gate = blockIdx.y, split = blockIdx.z;
  if (w >= W) return;
  const GT* g = gate ? gi : gr;
  const long per = (BT + splits - 1) / splits;
  const long nb = split * per, ne = min((long)BT, nb + per);
  float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  long n = nb;
  for (; n + 4 <= ne; n += 4) {
    float2 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = Pair<GT>::load(g + (size_t)(n + u) * W + w);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      s0[u] += v[u].x;
      s1[u] += v[u].y;
    }
  }
  for (; n < ne; ++n) {
    const float2 v = Pair<GT>::load(g + (size_t)n * W + w);
    s0[0] += v.x;
    s1[0] += v.y;
  }
  float* out = dbp + ((size_t)split * 2 + gate) * W + w;
  out[0] = (s0[0] + s0[1]) + (s0[2] + s0[3]);
  out[1] = (s1[0] + s1[1]) + (s1[2] + s1[3]);
}

// out[e] = sum over splits (in split order) of part[split][e], for `count` elements.
__global__ void k_sum_splits(const float* part, int splits, size_t count, size_t stride,
                             float* out) {
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= count) return;
  float s = 0.0f;
  for (int q = 0; q < splits; ++q) s += part[(size_t)q * stride + e];
  out[e] = s;
}

template <typename XT, typename OT>
cudaError_t proj(const Dims& d, const void* x, const void* Wa, const float* ba, const void* Wx,
                 const float* bx, void* lr, void* li, cudaStream_t s) {
  const int BT = d.B * d.T;
  dim3 grid((BT + TM - 1) / TM, d.nblk * ((d.k + TN - 1) / TN), 2);
  k_proj<XT, OT><<<grid, 256, 0, s>>>(BT, d.W, d.k, (const XT*)x, (const XT*)Wa, ba,
                                      (const XT*)Wx, bx, (OT*)lr, (OT*)li);
  note_launches(1);
  return cudaGetLastError();
}

template <typename WT, typename GT, typename DXT>
cudaError_t dxk(const Dims& d, const void* gr, const void* gi, const void* Wa, const void* Wx,
                const float* dx_in, void* dx, cudaStream_t s) {
  const int BT = d.B * d.T;
  dim3 grid((BT + TM - 1) / TM, d.nblk * ((d.k + TN - 1) / TN));
  k_dx<WT, GT, DXT><<<grid, 256, 0, s>>>(BT, d.W, d.k, (const GT*)gr, (const GT*)gi,
                                         (const WT*)Wa, (const WT*)Wx, dx_in, (DXT*)dx);
  note_launches(1);
  return cudaGetLastError();
}

template <typename XT, typename GT>
cudaError_t dwk(const Dims& d, const void* x, const void* gr, const void* gi, float* dWa,
                float* dba, float* dWx, float* dbx, uint8_t* ws, cudaStream_t s) {
  const int BT = d.B * d.T;
  const int S = dw_splits(d);
  const GateBwdLayout L = gate_bwd_layout(d);
  float* part = reinterpret_cast<float*>(ws + L.dw_part);
  float* dbp = reinterpret_cast<float*>(ws + L.db_part);
  const int nt = (d.k + 63) / 64;
  k_dw_part<XT, GT><<<dim3(nt * nt, d.nblk * 2, S), 256, 0, s>>>(
      BT, d.W, d.k, d.nblk, S, (const XT*)x, (const GT*)gr, (const GT*)gi, part);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t per_gate = (size_t)d.nblk * d.k * d.k;
  k_sum_splits<<<(unsigned)((per_gate + 255) / 256), 256, 0, s>>>(part, S, per_gate,
                                                                   2 * per_gate, dWa);
  note_launches(1);
  k_sum_splits<<<(unsigned)((per_gate + 255) / 256), 256, 0, s>>>(part + per_gate, S, per_gate,
                                                                   2 * per_gate, dWx);
  note_launches(1);
  if (dba || dbx) {
    const int SD = db_splits(d);
    k_db_part<GT><<<dim3((d.W + 511) / 512, 2, SD), 256, 0, s>>>(BT, d.W, SD, (const GT*)gr,
                                                                 (const GT*)gi, dbp);
    note_launches(1);
    if (dba) {
      k_sum_splits<<<(d.W + 255) / 256, 256, 0, s>>>(dbp, SD, (size_t)d.W, 2 * (size_t)d.W, dba);
      note_launches(1);
    }
    if (dbx) {
      k_sum_splits<<<(d.W + 255) / 256, 256, 0, s>>>(dbp + d.W, SD, (size_t)d.W, 2 * (size_t)d.W,
                                                     dbx);
      note_launches(1);
    }
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_proj_simt(const Dims& d, int xt, int ot, const void* x, const void* Wa,
                                  const float* ba, const void* Wx, const float* bx, void* lr,
                                  void* li, cudaStream_t s) {
  if (xt == DT_F32 && ot == DT_F32) return proj<float, float>(d, x, Wa, ba, Wx, bx, lr, li, s);
  if (xt == DT_BF16 && ot == DT_BF16) return proj<bf16, bf16>(d, x, Wa, ba, Wx, bx, lr, li, s);
  if (xt == DT_BF16 && ot == DT_F32) return proj<bf16, float>(d, x, Wa, ba, Wx, bx, lr, li, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gate_dx_simt(const Dims& d, int wt, int gt, int dxt, const void* dlr,
                                const void* dli, const void* Wa, const void* Wx,
                                const float* dx_in, void* dx, cudaStream_t s) {
  if (wt == DT_F32 && gt == DT_F32 && dxt == DT_F32)
    return dxk<float, float, float>(d, dlr, dli, Wa, Wx, dx_in, dx, s);
  if (wt == DT_BF16 && gt == DT_BF16 && dxt == DT_BF16)
    return dxk<bf16, bf16, bf16>(d, dlr, dli, Wa, Wx, dx_in, dx, s);
  if (wt == DT_BF16 && gt == DT_F32 && dxt == DT_F32)
    return dxk<bf16, float, float>(d, dlr, dli, Wa, Wx, dx_in, dx, s);
  if (wt == DT_BF16 && gt == DT_F32 && dxt == DT_BF16)
    return dxk<bf16, float, bf16>(d, dlr, dli, Wa, Wx, dx_in, dx, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gate_dw_simt(const Dims& d, int xt, int gt, const void* x, const void* dlr,
                                const void* dli, float* dWa, float* dba, float* dWx, float* dbx,
                                uint8_t* ws, cudaStream_t s) {
  if (xt == DT_F32 && gt == DT_F32)
    return dwk<float, float>(d, x, dlr, dli, dWa, dba, dWx, dbx, ws, s);
  if (xt == DT_BF16 && gt == DT_BF16)
    return dwk<bf16, bf16>(d, x, dlr, dli, dWa, dba, dWx, dbx, ws, s);
  if (xt == DT_BF16 && gt == DT_F32)
    return dwk<bf16, float>(d, x, dlr, dli, dWa, dba, dWx, dbx, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace rglru
