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
//
// Large batches (bf16, B >= STEP_TC_MIN_B, k a multiple of 32) take k_step_tc instead: the step
// is then a [B x k] x [k x k] product per gate block and matrix, which goes to the tcgen05
// tensor cores.  CTA = (128-row tile, gate block, 32-channel slice): TMA brings the x tile
// (16-channel slabs, 32-byte swizzle) and the two 32-column weight slices, issued by the thread
// that initialises the barriers before anything else; one thread issues the k / 16 MMAs of
// M = 128 rows x N = 32 channels per matrix into TMEM, and each of the eight warps then takes
// 32 rows (its TMEM lane quadrant) and 16 of the channels: lr, li from TMEM, x from the staged
// tile, the state row requested before the MMA wait, and the gate arithmetic of the fused bf16
// kernels (two ex2 and one rsqrt a channel, gates_any1).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_util.h"
#include "internal.h"
#include "tc.cuh"

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
  // launched with programmatic stream serialisation: the launch overlaps the end of the kernel
  // before it on the stream; every read and write of the step comes after the wait
  tc::griddep_wait();
  tc::griddep_launch_dependents();
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

// ---------------------------------------------------------------- tensor-core step
constexpr int STC_ROWS = 128;
constexpr int STC_N = 32;                     // channels per CTA
constexpr int STC_THREADS = 256;              // 8 warps: 4 lane quadrants x 2 channel halves
constexpr uint32_t STC_SLAB = STC_ROWS * 32;  // 16 channels x 128 rows of x

__global__ void __launch_bounds__(STC_THREADS, 1)
    k_step_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
              const __grid_constant__ CUtensorMap tm_wx, const __grid_constant__ DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = a.k;
  const int nsl = k / STC_N;
  const int blk = blockIdx.x / nsl, j0 = (blockIdx.x % nsl) * STC_N;
  const int row0 = blockIdx.y * STC_ROWS;
  const uint32_t XB = (uint32_t)(k / 16) * STC_SLAB;   // x tile
  const uint32_t WS = (uint32_t)k * 32;                // one 16-column weight slab
  uint8_t* s_x = smem;
  uint8_t* s_w[2] = {smem + XB, smem + XB + 2 * WS};
  GateK* s_c = reinterpret_cast<GateK*>(smem + XB + 4 * WS);  // per channel
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_c + STC_N);
  uint64_t* full = bars;
  uint64_t* done = bars + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launched with programmatic stream serialisation: up to griddep_wait nothing touches
  // global memory (barrier set-up, the TMEM allocation, the tensor-map prefetch), so this part
  // overlaps the end of the kernel before it on the stream; every read and write of the step's
  // operands comes after the wait.
  if (threadIdx.x == 0) {
    tc::mbar_init(full, 1);
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tm_x);
    tc::prefetch_tmap(&tm_wa);
    tc::prefetch_tmap(&tm_wx);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, 2 * STC_N);
    tc::tmem_relinquish();
  }
  tc::griddep_wait();
  tc::griddep_launch_dependents();
  // the operand loads go out first: thread 0 issues them at once
  if (threadIdx.x == 0) {
    tc::mbar_expect_tx(full, XB + 4 * WS);
    for (int s = 0; s < k / 16; ++s)
      tc::tma_load_2d(s_x + s * STC_SLAB, &tm_x, full, blk * k + 16 * s, row0);
    for (int m = 0; m < 2; ++m)
      for (int s = 0; s < 2; ++s)
        tc::tma_load_2d(s_w[m] + s * WS, m ? &tm_wx : &tm_wa, full, j0 + 16 * s, blk * k);
  }
  // this thread's row and 16 channels: state segment, reset flag, and (warp 2) the channel
  // constants, all requested before any wait
  const int q = warp & 3, hf = warp >> 2;
  const int row = row0 + 32 * q + lane;
  const bool live = row < a.B;
  const size_t o = (size_t)row * a.W + (size_t)blk * k + j0 + 16 * hf;
  float4 hp[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    hp[e] = (live && a.h_in) ? reinterpret_cast<const float4*>(a.h_in + o)[e]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
  const bool rst = live && a.canonical && a.reset && a.reset[row] != 0;
  if (warp == 2) {
    const int w = blk * k + j0 + lane;
    GateK g;
    g.nk = -8.0f * softplus_f(a.Lambda[w]);
    g.cm = sqrtf(-2.0f * g.nk);
    g.nbr = a.ba ? -a.ba[w] * LOG2E : 0.0f;  // the biases folded into the exponents
    g.nbi = a.bx ? -a.bx[w] * LOG2E : 0.0f;
    s_c[lane] = g;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (warp == 0) {
    const bool leader = tc::elect_one();
    const bool ok = tc::mbar_wait(full, 0, 2000000000ull);
    tc::tc_fence_after();
    if (leader && ok) {
      const uint32_t idesc = tc::idesc_bf16(STC_ROWS, STC_N, 0, 1);  // x K-major, W MN-major
      const uint32_t xs = tc::smem_u32(s_x);
      for (int m = 0; m < 2; ++m) {
        const uint32_t ws = tc::smem_u32(s_w[m]);
        for (int kk = 0; kk < k / 16; ++kk)
          tc::mma_bf16(tmem + m * STC_N, tc::smem_desc_sw32(xs + kk * STC_SLAB, 16, 256),
                       tc::smem_desc_sw32(ws + kk * 512, WS, 256), idesc, kk > 0);
      }
    }
    if (leader) tc::mma_commit(done);  // arrives once the MMAs (if any) are done
    __syncwarp();
  }
  const bool ok = tc::mbar_wait(done, 0, 2000000000ull);
  tc::tc_fence_after();
  float lr[16], li[16];
  {
    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + 16 * hf;
    tc::tmem_ld16(ta, lr);
    tc::tmem_ld16(ta + STC_N, li);
    tc::tmem_ld_wait();
    tc::reg_fence(lr);
    tc::reg_fence(li);
  }
  if (live && ok) {
    // x of the row's 16 channels from the staged tile: one slab, a 32-byte row whose 16-byte
    // halves are swapped on rows 4..7 of every 8
    const int r = 32 * q + lane;
    float xv[16];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint4 u = *reinterpret_cast<const uint4*>(
          s_x + (j0 / 16 + hf) * STC_SLAB + r * 32 + ((hh ^ ((r >> 2) & 1)) << 4));
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xv[8 * hh + 2 * e] = __uint_as_float(w4[e] << 16);
        xv[8 * hh + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
      }
    }
    const float* hpf = reinterpret_cast<const float*>(hp);
    float hn[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float abar, mi, ig;
      gates_any1(lr[c], li[c], s_c[16 * hf + c], abar, mi, ig);
      if (rst) {  // canonical reset row: abar = 0, m = 1
        abar = 0.0f;
        mi = ig;
      }
      hn[c] = fmaf(abar, hpf[c], mi * xv[c]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      reinterpret_cast<float4*>(a.h_out + o)[e] =
          make_float4(hn[4 * e], hn[4 * e + 1], hn[4 * e + 2], hn[4 * e + 3]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      uint4 u;
      uint32_t* pu = &u.x;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(hn[8 * e + 2 * h], hn[8 * e + 2 * h + 1]);
        pu[h] = *reinterpret_cast<const uint32_t*>(&v);
      }
      reinterpret_cast<uint4*>(static_cast<bf16*>(a.y) + o)[e] = u;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * STC_N);
  }
}

}  // namespace

bool step_tc_supported(const Dims& d) {
  return d.io == RGLRU_BF16 && d.B >= STEP_TC_MIN_B && d.k % STC_N == 0 && d.k <= 256 &&
         sm_count() > 0;
}

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
  if (step_tc_supported(d)) {
    // x [B][W] in 16-channel x 128-row boxes; W[nblk][k][k] as [nblk k rows][k columns] in
    // 16-column x k-row boxes (the 32-channel slice: two of them)
    CUtensorMap mx, mwa, mwx;
    const uint64_t dx[2] = {(uint64_t)d.W, (uint64_t)d.B};
    const uint64_t sx[1] = {(uint64_t)d.W * 2};
    const uint32_t bx_[2] = {16, STC_ROWS};
    cudaError_t e = encode_tmap(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dx, sx, bx_,
                                CU_TENSOR_MAP_SWIZZLE_32B);
    const uint64_t dw[2] = {(uint64_t)d.k, (uint64_t)d.nblk * d.k};
    const uint64_t sw[1] = {(uint64_t)d.k * 2};
    const uint32_t bw[2] = {16, (uint32_t)d.k};
    if (e == cudaSuccess)
      e = encode_tmap(&mwa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wa, dw, sw, bw,
                      CU_TENSOR_MAP_SWIZZLE_32B);
    if (e == cudaSuccess)
      e = encode_tmap(&mwx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wx, dw, sw, bw,
                      CU_TENSOR_MAP_SWIZZLE_32B);
    if (e != cudaSuccess) return e;
    const size_t smem = 1024 + (size_t)(d.k / 16) * STC_SLAB + 4 * (size_t)d.k * 32 +
                        STC_N * sizeof(GateK) + 64;
    e = cudaFuncSetAttribute(k_step_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(d.nblk * (d.k / STC_N)), (unsigned)((d.B + STC_ROWS - 1) / STC_ROWS));
    // programmatic stream serialisation: the kernel's set-up overlaps the end of the kernel
    // before it on the stream (a decode loop's previous step or layer)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(STC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_step_tc, mx, mwa, mwx, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
  }
  const size_t smem = step_smem_bytes(d.k);
  const dim3 grid((unsigned)(d.nblk * ((d.k + 31) / 32)), (unsigned)((d.B + DEC_ROWS - 1) / DEC_ROWS));
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(DEC_WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (d.io == RGLRU_BF16) {
    e = cudaFuncSetAttribute(k_step<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_step<bf16>, a);
  } else {
    e = cudaFuncSetAttribute(k_step<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_step<float>, a);
  }
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rglru
