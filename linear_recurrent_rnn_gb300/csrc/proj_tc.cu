// Block-diagonal gate projections and their gradients on the tcgen05 tensor cores: bf16
// operands staged by TMA, float32 accumulation in tensor memory, for gate blocks of
// k = 16 .. 160 channels (k a multiple of 16).
//
// Sources ("Fattori comparison" page, first paragraph: the two block-diagonal gate projections
// feed the recurrence; the benchmark record's protocol scope puts them inside the measured
// layer).  Rows r run over the B T tokens; per gate block blk:
//   forward   lr[r, blk k + j]  = sum_i x[r, blk k + i] Wa[blk][i][j] + ba[blk k + j]
//             li                = the same with Wx, bx
//   backward  dx[r, blk k + i]  = add[r, blk k + i] + sum_j dlr[r, blk k + j] Wa[blk][i][j]
//                                                   + sum_j dli[r, blk k + j] Wx[blk][i][j]
//             dWa[blk][i][j]    = sum_r x[r, blk k + i] dlr[r, blk k + j],  dba = sum_r dlr
//             dWx, dbx          = the same with dli
// The gradient operands dlr / dli come as one bf16 plane, or as two (hi + lo, v = hi + lo to
// ~2^-16) when they were float32: each plane is one more product into the same accumulator.
//
// Every operand tile is 128 rows of one gate block, loaded by TMA as 16-channel slabs with
// the 32-byte swizzle (128 rows x 32 bytes = 4 KB a slab): a slab is one K = 16 step of a
// K-major operand, and 16 consecutive M or N indices of an MN-major one.  One CTA per SM:
// warp 0 issues the TMA loads, warp 1 the MMAs (one elected lane), the other warps read the
// accumulators back (warp w reaches TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, so it owns those
// rows of a tile): one set of four in the dW kernel, which writes only its partial sums, and
// one or two sets (as shared memory allows their box rings) in the forward and dx kernels,
// whose epilogues write every output element.  Pipeline waits are bounded (2 s); a wait that runs out winds the CTA down.
#include <cudaTypedefs.h>

#include <algorithm>

#include "host_util.h"
#include "internal.h"
#include "tc.cuh"

namespace rglru {

namespace {

constexpr int TR = 128;                   // rows of a tile
constexpr uint32_t SLAB = TR * 32;        // one 16-channel slab of a tile
constexpr int NTHREADS = 192;             // TMA, MMA, one set of 4 epilogue warps
constexpr int NTHREADS_MAX = 320;         // TMA, MMA, two sets of 4 epilogue warps
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr size_t SMEM_MAX = 232448;       // 227 KB of dynamic shared memory per CTA
constexpr int NCMAX = PROJ_TC_KMAX / 16;   // 16-column chunks of a row, at most

// Bytes of one operand tile (128 rows x k bf16).
__host__ __device__ constexpr uint32_t tile_bytes(int k) { return (uint32_t)(k / 16) * SLAB; }
// Bytes of the addend's identity operand in the dx kernel: the 32 x 32 identity as two
// 16-column slabs (one per parity of the K step), see k_proj_dx.
constexpr uint32_t ID_BYTES = 2048;
// TMEM columns of a k-wide accumulator, rounded up to a multiple of 32.
__host__ __device__ constexpr uint32_t kcols(int k) { return (uint32_t)((k + 31) / 32 * 32); }
// TMEM columns of one matrix in the dW kernel: its dW accumulators and 32-column db ones.
__host__ __device__ constexpr uint32_t dw_mcols(int k) {
  return (uint32_t)((k + 127) / 128) * (kcols(k) + 32u);
}
// Bytes past the dW kernel's operand ring that an MN-major operand may read (see k_proj_dw).
__host__ __device__ constexpr uint32_t dw_pad(int k) {
  return (uint32_t)((k + 127) / 128) * 8 * SLAB - tile_bytes(k);
}

struct Abort {
  uint32_t* flag;  // shared: set once a wait has run out; every later wait returns at once
  __device__ bool wait(uint64_t* bar, uint32_t parity) const {
    if (*reinterpret_cast<volatile uint32_t*>(flag)) return false;
    if (tc::mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile uint32_t*>(flag) = 1u;
    return false;
  }
};

// ---------------------------------------------------------------- staged row stores
// An epilogue warp owns 32 rows of a tile, one a lane, and produces each row 16 columns at a
// time.  Stored straight to global memory, every 16-byte store of the warp would touch 32
// rows, and those stores run at a fraction of the copy bandwidth.  Instead the warp writes its
// chunks into shared-memory boxes of 32 rows x bi bytes (bi = 128, 64 or 32: the widest that
// divides a block row), in the layout the TMA swizzle of that width gives: 16-byte unit u of
// row r sits at unit u ^ ((r >> shift) & (bi / 16 - 1)), shift = 0, 1, 2 for bi = 128, 64,
// 32; the same XOR keeps the warp's writes free of bank conflicts.  One lane stores each
// completed box with a TMA tensor store; a ring of RING boxes (per output plane) lets the
// stores drain behind the next chunks.
constexpr int RING = 2;

template <typename OT>
struct BoxStore {
  static constexpr int UPC = (int)sizeof(OT);  // 16-byte units of a 16-column chunk
  uint8_t* ring;  // RING x planes boxes of 32 * bi bytes, 1024-byte aligned
  int bi, csh, cmask, sw, planes, lane, slot;  // chunks a box = 1 << csh (cmask = that - 1)

  __device__ BoxStore(uint8_t* r, int bi_, int planes_, int lane_)
      : ring(r), bi(bi_), planes(planes_), lane(lane_), slot(0) {
    // chunks a box: bi / (16 sizeof(OT)), a power of two; rows swizzled by lane >> shift
    csh = (bi_ == 128 ? 3 : (bi_ == 64 ? 2 : 1)) - (sizeof(OT) == 4 ? 2 : 1);
    cmask = (1 << csh) - 1;
    const int shift = bi_ == 128 ? 0 : (bi_ == 64 ? 1 : 2);
    sw = (lane_ >> shift) & (bi_ / 16 - 1);
  }
  __device__ uint8_t* box(int pl) const { return ring + (size_t)(slot * planes + pl) * 32 * bi; }
  // Before the first chunk of a box: the ring slot's earlier stores have finished reading it.
  __device__ void begin(int c) {
    if ((c & cmask) == 0) {
      if (lane == 0) tc::tma_store_wait_read_n<RING - 1>();
      __syncwarp();
    }
  }
  // Chunk c of this lane's row, plane pl.
  __device__ void put(int c, int pl, const float (&v)[16]) {
    uint8_t* row = box(pl) + lane * bi;
    const int u0 = (c & cmask) * UPC;
    if constexpr (sizeof(OT) == 2) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint4 q;
        uint32_t* w = &q.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(row + (((u0 + j) ^ sw) << 4)) = q;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float4*>(row + (((u0 + j) ^ sw) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  // After chunk c: a completed box goes out to columns x0 + (its first column), rows y0 .. y0 + 31
  // of planes z0, z0 + 1, ... (rows past the tensor are clipped by the store).
  __device__ void end(int c, const CUtensorMap* map, int x0, int y0, int z0 = 0) {
    if ((c & cmask) != cmask) return;
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int x = x0 + (c >> csh) * (bi / (int)sizeof(OT));
      for (int pl = 0; pl < planes; ++pl) tc::tma_store_3d(map, box(pl), x, y0, z0 + pl);
      tc::tma_store_commit();
    }
    slot ^= 1;  // RING = 2
  }
  __device__ void drain() const {
    if (lane == 0) tc::tma_store_wait0();
  }
};
static_assert(RING == 2, "BoxStore::end steps a two-slot ring");

// Bytes of one epilogue warp's box ring.
__host__ __device__ constexpr uint32_t ring_bytes(int bi, int planes) {
  return (uint32_t)(RING * planes * 32 * bi);
}

struct ProjParams {
  int R, k, nblk, P;     // rows, gate block, blocks, CTAs per (block, matrix group)
  const float* bias[2];  // forward: ba, bx (null = zero)
  const void* add;       // dx: the addend (float32 or bf16 [R][W]); may alias the output
  int add_f32;
  int W;
  int nplanes;           // gradient operand planes (1, or 2 for hi + lo)
  int nmat;              // dW: matrices per CTA (2: both; 1: CTA group m handles matrix m)
  float* part;           // dW: partial sums [blk][r][m][k * k + k]
  int bi;                // forward, dx: row bytes of an output box (128, 64 or 32)
  int nsets;             // forward, dx: sets of 4 epilogue warps (1 or 2)
};

// ================================================================ forward projection
// CTA (blk, r) keeps Wa[blk], Wx[blk] in shared memory and takes the row tiles r, r + P, ...
// Per tile the x tile feeds two accumulations, lr then li, each into the next slot of a ring
// of k-column TMEM buffers; the epilogue warps add the bias, convert, and stage each row into
// their box rings for TMA stores (BoxStore), the next chunk's TMEM load in flight meanwhile.
// SPLIT: the float32 logits go out as bf16 hi and lo planes (the output maps' second plane).
template <typename OT, bool SPLIT>
__global__ void __launch_bounds__(NTHREADS_MAX, 1)
    k_proj_fwd(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
               const __grid_constant__ CUtensorMap tm_wx, const __grid_constant__ CUtensorMap tm_lr,
               const __grid_constant__ CUtensorMap tm_li, const __grid_constant__ ProjParams p,
               int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = p.k;
  const uint32_t TB = tile_bytes(k);
  const uint32_t WB = (uint32_t)k * k * 2;
  const uint32_t KC = kcols(k);
  const int NS = 512 / (int)KC;  // TMEM ring slots
  constexpr int PLANES = SPLIT ? 2 : 1;
  uint8_t* s_w[2] = {smem, smem + WB};
  uint8_t* s_x = smem + 2 * WB;
  uint8_t* s_ring = s_x + stages * TB;  // the epilogue warps' box rings (1024-byte aligned)
  float* s_bias = reinterpret_cast<float*>(s_ring + 4 * p.nsets * ring_bytes(p.bi, PLANES));
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_bias + 2 * k);
  uint64_t* w_full = bars;
  uint64_t* x_full = bars + 1;
  uint64_t* x_empty = x_full + stages;
  uint64_t* acc_full = x_empty + stages;  // [NS]
  uint64_t* acc_empty = acc_full + NS;    // [NS]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + NS);
  uint32_t* abort_flag = tmem_holder + 1;
  const Abort ctl{abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x / p.P, rr = blockIdx.x % p.P;
  const int ntiles = (p.R + TR - 1) / TR;
  int my_tiles = 0;
  for (int n = rr; n < ntiles; n += p.P) ++my_tiles;

  if (threadIdx.x == 0) {
    tc::mbar_init(w_full, 1);
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&x_full[s], 1);
      tc::mbar_init(&x_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&acc_full[s], 1);
      tc::mbar_init(&acc_empty[s], 4);
    }
    *abort_flag = 0u;
    tc::fence_barrier_init();
  }
  for (int j = threadIdx.x; j < 2 * k; j += blockDim.x) {
    const float* b = p.bias[j >= k];
    s_bias[j] = b ? b[blk * k + (j % k)] : 0.0f;
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_holder, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_x);
      tc::mbar_expect_tx(w_full, 2 * WB);
      for (int s = 0; s < k / 16; ++s) {
        tc::tma_load_2d(s_w[0] + s * (k * 32), &tm_wa, w_full, 16 * s, blk * k);
        tc::tma_load_2d(s_w[1] + s * (k * 32), &tm_wx, w_full, 16 * s, blk * k);
      }
      for (int it = 0; it < my_tiles; ++it) {
        const int st = it % stages;
        if (!ctl.wait(&x_empty[st], ((it / stages) & 1) ^ 1u)) break;
        const int row0 = (rr + it * p.P) * TR;
        uint8_t* xs = s_x + st * TB;
        tc::mbar_expect_tx(&x_full[st], TB);
        for (int s = 0; s < k / 16; ++s)
          tc::tma_load_2d(xs + s * SLAB, &tm_x, &x_full[st], blk * k + 16 * s, row0);
      }
    }
  } else if (warp == 1) {
    const bool leader = tc::elect_one();
    const uint32_t idesc = tc::idesc_bf16(TR, k, 0, 1);  // A = x K-major, B = W MN-major
    ctl.wait(w_full, 0);
    for (int it = 0; it < my_tiles; ++it) {
      const int st = it % stages;
      if (!ctl.wait(&x_full[st], (it / stages) & 1)) break;
      const uint32_t xs = tc::smem_u32(s_x + st * TB);
#pragma unroll 1
      for (int m = 0; m < 2; ++m) {
        const int u = 2 * it + m, slot = u % NS;
        if (!ctl.wait(&acc_empty[slot], ((u / NS) & 1) ^ 1u)) break;
        tc::tc_fence_after();
        const uint32_t ws = tc::smem_u32(s_w[m]);
        if (leader) {
          for (int kk = 0; kk < k / 16; ++kk)
            tc::mma_bf16(tmem + slot * KC, tc::smem_desc_sw32(xs + kk * SLAB, 16, 256),
                         tc::smem_desc_sw32(ws + kk * 512, (uint32_t)k * 32, 256), idesc, kk > 0);
          tc::mma_commit(&acc_full[slot]);
        }
        __syncwarp();
      }
      if (leader) tc::mma_commit(&x_empty[st]);
      __syncwarp();
    }
  } else {
    const int q = warp & 3;  // TMEM lane quadrant = rows 32 q .. 32 q + 31 of a tile
    const int NC = k / 16;
    // one set: every warp writes lr then li; two sets: set 0 writes lr, set 1 li
    const int set = (warp - 2) >> 2;
    const int m0 = p.nsets == 2 ? set : 0, m1 = p.nsets == 2 ? set + 1 : 2;
    BoxStore<OT> bs(s_ring + (warp - 2) * ring_bytes(p.bi, PLANES), p.bi, PLANES, lane);
    for (int it = 0; it < my_tiles; ++it) {
      const int y0 = (rr + it * p.P) * TR + 32 * q;  // this warp's first row
#pragma unroll 1
      for (int m = m0; m < m1; ++m) {
        const int u = 2 * it + m, slot = u % NS;
        if (!ctl.wait(&acc_full[slot], (u / NS) & 1)) break;
        tc::tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + slot * KC;
        const CUtensorMap* om = m ? &tm_li : &tm_lr;
        const float4* b4 = reinterpret_cast<const float4*>(s_bias + m * k);
        // the next chunk's accumulator load is in flight while this one is staged
        float v[2][16];
        tc::tmem_ld16(ta, v[0]);
#pragma unroll
        for (int c = 0; c < NCMAX; ++c) {
          if (c >= NC) break;
          tc::tmem_ld_wait();
          tc::reg_fence(v[c & 1]);
          if (c + 1 < NC) tc::tmem_ld16(ta + 16 * (c + 1), v[(c + 1) & 1]);
          float (&vv)[16] = v[c & 1];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 b = b4[4 * c + e];
            vv[4 * e] += b.x;
            vv[4 * e + 1] += b.y;
            vv[4 * e + 2] += b.z;
            vv[4 * e + 3] += b.w;
          }
          bs.begin(c);
          bs.put(c, 0, vv);
          if (SPLIT) {  // lo = v - bf16(v), exact in float32, then rounded to bf16
#pragma unroll
            for (int e = 0; e < 16; ++e) vv[e] -= __bfloat162float(__float2bfloat16_rn(vv[e]));
            bs.put(c, 1, vv);
          }
          bs.end(c, om, blk * k, y0);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_empty[slot]);
      }
    }
    bs.drain();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dx of the projections
// CTA (blk, r) keeps Wa[blk], Wx[blk] in shared memory (the K-major B operand of dx = dl W^T)
// and takes the row tiles r, r + P, ...  Per tile the 2 x nplanes gradient operand tiles pass
// through a ring of `stages` buffers, each one K-loop into the tile's accumulator (one of two
// TMEM buffers); the epilogue adds the addend tile and stores dx through its box ring.
// Loads the 16 addend values of chunk c of this thread's row (zero past the rows).
template <typename AT>
struct AddChunk;
template <>
struct AddChunk<float> {
  float4 v[4];
  __device__ void load(const float* row, int c, bool in) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = in ? reinterpret_cast<const float4*>(row + 16 * c)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __device__ void add_to(float (&a)[16]) const {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[4 * e] += v[e].x;
      a[4 * e + 1] += v[e].y;
      a[4 * e + 2] += v[e].z;
      a[4 * e + 3] += v[e].w;
    }
  }
};
template <>
struct AddChunk<bf16> {
  uint4 v[2];
  __device__ void load(const bf16* row, int c, bool in) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      v[e] = in ? reinterpret_cast<const uint4*>(row + 16 * c)[e] : make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ void add_to(float (&a)[16]) const {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t w4[4] = {v[e].x, v[e].y, v[e].z, v[e].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        a[8 * e + 2 * h] += __uint_as_float(w4[h] << 16);
        a[8 * e + 2 * h + 1] += __uint_as_float(w4[h] & 0xffff0000u);
      }
    }
  }
};

template <typename OT, typename AT>
__global__ void __launch_bounds__(NTHREADS_MAX, 1)
    k_proj_dx(const __grid_constant__ CUtensorMap tm_dla, const __grid_constant__ CUtensorMap tm_dlx,
              const __grid_constant__ CUtensorMap tm_wa,
              const __grid_constant__ CUtensorMap tm_wx, const __grid_constant__ CUtensorMap tm_dx,
              const __grid_constant__ CUtensorMap tm_add, const __grid_constant__ ProjParams p,
              int stages) {
  // a bf16 addend is one more operand tile, added by MMAs against the identity: K step kk (input
  // channels 16 kk .. 16 kk + 15) adds into accumulator columns 32 (kk / 2) .. + 31 with N = 32,
  // B = slab kk % 2 of the 32 x 32 identity (ones at rows 16 (kk % 2) + c), so every element
  // gains one product with 1.0: the float32 sum of the two terms.  A float32 addend is read by
  // the epilogue warps.
  constexpr bool ADD_MMA = sizeof(AT) == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = p.k;
  const uint32_t TB = tile_bytes(k);
  const uint32_t WB = (uint32_t)k * k * 2;
  const uint32_t KC = kcols(k);
  const int NDL = 2 * p.nplanes;          // gradient operand tiles per row tile
  const int NOP = NDL + (ADD_MMA ? 1 : 0);  // operand tiles per row tile
  uint8_t* s_w[2] = {smem, smem + WB};
  uint8_t* s_id = smem + 2 * WB;  // the identity slabs (ADD_MMA)
  uint8_t* s_in = s_id + (ADD_MMA ? ID_BYTES : 0u);
  uint8_t* s_ring = s_in + stages * TB;  // the epilogue warps' box rings (1024-byte aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_ring + 4 * p.nsets * ring_bytes(p.bi, 1));
  uint64_t* w_full = bars;
  uint64_t* in_full = bars + 1;
  uint64_t* in_empty = in_full + stages;
  uint64_t* acc_full = in_empty + stages;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  uint32_t* abort_flag = tmem_holder + 1;
  const Abort ctl{abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x / p.P, rr = blockIdx.x % p.P;
  const int ntiles = (p.R + TR - 1) / TR;
  int my_tiles = 0;
  for (int n = rr; n < ntiles; n += p.P) ++my_tiles;

  // the dW kernel launched after this one reads none of its outputs: it may start at once on
  // the SMs this grid leaves free (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (ADD_MMA) tc::write_identity_sw32(s_id, 32);
  if (threadIdx.x == 0) {
    tc::mbar_init(w_full, 1);
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&in_full[s], 1);
      tc::mbar_init(&in_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&acc_full[s], 1);
      tc::mbar_init(&acc_empty[s], 4 * p.nsets);
    }
    *abort_flag = 0u;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_holder, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_dla);
      tc::prefetch_tmap(&tm_dlx);
      tc::mbar_expect_tx(w_full, 2 * WB);
      for (int s = 0; s < k / 16; ++s) {
        tc::tma_load_2d(s_w[0] + s * (k * 32), &tm_wa, w_full, 16 * s, blk * k);
        tc::tma_load_2d(s_w[1] + s * (k * 32), &tm_wx, w_full, 16 * s, blk * k);
      }
      // operand o of a row tile: matrix o / nplanes, plane o % nplanes; each matrix's gradient
      // tensor map is [nplanes][R][W], the plane its outermost coordinate
      int u = 0;
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int row0 = (rr + it * p.P) * TR;
        for (int o = 0; o < NOP; ++o, ++u) {
          const int st = u % stages;
          if (!(ok = ctl.wait(&in_empty[st], ((u / stages) & 1) ^ 1u))) break;
          uint8_t* buf = s_in + st * TB;
          tc::mbar_expect_tx(&in_full[st], TB);
          if (o < NDL) {
            const int m = o / p.nplanes, pl = o % p.nplanes;
            for (int s = 0; s < k / 16; ++s)
              tc::tma_load_3d(buf + s * SLAB, m ? &tm_dlx : &tm_dla, &in_full[st],
                              blk * k + 16 * s, row0, pl);
          } else {  // the addend tile
            for (int s = 0; s < k / 16; ++s)
              tc::tma_load_2d(buf + s * SLAB, &tm_add, &in_full[st], blk * k + 16 * s, row0);
          }
        }
      }
    }
  } else if (warp == 1) {
    const bool leader = tc::elect_one();
    const uint32_t idesc = tc::idesc_bf16(TR, k, 0, 0);  // A = dl K-major, B = W K-major
    const uint32_t idesc32 = tc::idesc_bf16(TR, 32, 0, 0);  // A = addend, B = identity slab
    ctl.wait(w_full, 0);
    int u = 0;
    for (int it = 0; it < my_tiles; ++it) {
      const int slot = it & 1;
      if (!ctl.wait(&acc_empty[slot], ((it >> 1) & 1) ^ 1u)) break;
      tc::tc_fence_after();
      bool ok = true;
      for (int o = 0; o < NOP; ++o, ++u) {
        const int st = u % stages;
        if (!ctl.wait(&in_full[st], (u / stages) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t a0 = tc::smem_u32(s_in + st * TB);
        if (leader) {
          if (o < NDL) {
            const uint32_t w0 = tc::smem_u32(s_w[o / p.nplanes]);
            for (int kk = 0; kk < k / 16; ++kk)
              tc::mma_bf16(tmem + slot * KC, tc::smem_desc_sw32(a0 + kk * SLAB, 16, 256),
                           tc::smem_desc_sw32(w0 + kk * (k * 32), 16, 256), idesc,
                           (o > 0 || kk > 0) ? 1u : 0u);
          } else {  // the addend tile
            const uint32_t i0 = tc::smem_u32(s_id);
            for (int kk = 0; kk < k / 16; ++kk)
              tc::mma_bf16(tmem + slot * KC + 32 * (kk >> 1),
                           tc::smem_desc_sw32(a0 + kk * SLAB, 16, 256),
                           tc::smem_desc_sw32(i0 + (kk & 1) * 1024, 16, 256), idesc32, 1u);
          }
          tc::mma_commit(&in_empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) tc::mma_commit(&acc_full[slot]);
      __syncwarp();
    }
  } else {
    const int q = warp & 3;
    const int NC = k / 16;
    // with two sets, set h writes the output boxes b = h mod 2 (the chunks c with
    // (c >> csh) mod 2 = h); the addend is loaded for those chunks only
    const int set = (warp - 2) >> 2;
    BoxStore<OT> bs(s_ring + (warp - 2) * ring_bytes(p.bi, 1), p.bi, 1, lane);
    // the warp's j-th chunk: c = j with one set; with two, chunk j mod (chunks a box) of the
    // warp's box j / (chunks a box), i.e. of box 2 (that) + set
    auto chunk = [&](int j) {
      return p.nsets == 1 ? j : ((((j >> bs.csh) << 1) + set) << bs.csh) | (j & bs.cmask);
    };
    for (int it = 0; it < my_tiles; ++it) {
      const int slot = it & 1;
      const int y0 = (rr + it * p.P) * TR + 32 * q;
      const int row = y0 + lane;
      const bool in = row < p.R;
      const AT* arow = static_cast<const AT*>(p.add) + (size_t)row * p.W + (size_t)blk * k;
      // the addend's first NA chunks of this warp are requested before the accumulator is
      // waited for, each later one NA chunks ahead of its use (a rolling window of registers)
      constexpr int NA = ADD_MMA ? 1 : 3;
      AddChunk<AT> add[NA];
#pragma unroll
      for (int j = 0; j < NA; ++j)
        if (!ADD_MMA && chunk(j) < NC) add[j].load(arow, chunk(j), in);
      if (!ctl.wait(&acc_full[slot], (it >> 1) & 1)) break;
      tc::tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + slot * KC;
      float v[2][16];
      if (chunk(0) < NC) tc::tmem_ld16(ta + 16 * chunk(0), v[0]);
#pragma unroll
      for (int j = 0; j < NCMAX; ++j) {
        const int c = chunk(j);
        if (c >= NC) break;
        tc::tmem_ld_wait();
        tc::reg_fence(v[j & 1]);
        if (chunk(j + 1) < NC) tc::tmem_ld16(ta + 16 * chunk(j + 1), v[(j + 1) & 1]);
        float (&vv)[16] = v[j & 1];
        if (!ADD_MMA) {
          add[j % NA].add_to(vv);
          if (chunk(j + NA) < NC) add[j % NA].load(arow, chunk(j + NA), in);
        }
        bs.begin(c);
        bs.put(c, 0, vv);
        bs.end(c, &tm_dx, blk * k, y0);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[slot]);
    }
    bs.drain();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dW, db of the projections
// CTA (blk, g, r): matrix group g (both matrices when nmat = 2, else matrix g) over the row
// tiles r, r + P, ...  Per tile the x tile and the group's gradient operand tiles pass through
// a ring of buffers; dW += x^T dl (M = input channel i in steps of 128, N = j) and db += dl^T 1
// (M = j in steps of 128, N = 16 columns of ones: column 0 of that accumulator holds the column
// sums of dl) accumulate in TMEM over the CTA's tiles; at the end the epilogue warps write the
// CTA's partial sums (dW through their box rings in the drained operand buffers), which
// k_proj_dw_reduce adds over the CTAs in a fixed order.
__global__ void __launch_bounds__(NTHREADS, 1)
    k_proj_dw(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dla,
              const __grid_constant__ CUtensorMap tm_dlx,
              const __grid_constant__ CUtensorMap tm_part, const __grid_constant__ ProjParams p,
              int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int k = p.k;
  const uint32_t TB = tile_bytes(k);
  const int MB = (k + 127) / 128;          // 128-channel row blocks of dW
  const uint32_t KC = kcols(k);
  const int NDL = p.nmat * p.nplanes;      // gradient operand tiles per row tile
  uint8_t* s_ones = smem;                  // 128 x 16 bf16 ones, one K-major slab
  // `stages` operand buffers of TB bytes, then a pad: an MN-major operand with M = 128 (x for
  // dW, dl for db) reads, for the last 128-channel block, MB * 8 slabs from its buffer's start,
  // past the k / 16 loaded ones (those lanes of the accumulator are never read), so every such
  // read stays in shared memory
  uint8_t* s_in = smem + SLAB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_in + stages * TB + dw_pad(k));
  uint64_t* in_full = bars;
  uint64_t* in_empty = in_full + stages;
  uint64_t* done = in_empty + stages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  uint32_t* abort_flag = tmem_holder + 1;
  const Abort ctl{abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = 2 / p.nmat;
  const int blk = blockIdx.x / (groups * p.P);
  const int g = (blockIdx.x / p.P) % groups;
  const int rr = blockIdx.x % p.P;
  const int ntiles = (p.R + TR - 1) / TR;
  int my_tiles = 0;
  for (int n = rr; n < ntiles; n += p.P) ++my_tiles;
  // TMEM per matrix of the group: MB dW accumulators (lanes = i - 128 mb), then MB db
  // accumulators of 32 columns (lanes = j - 128 mb, the sums in column 0)
  const uint32_t MCOLS = dw_mcols(k);

  for (int e = threadIdx.x; e < (int)(SLAB / 4); e += NTHREADS)
    reinterpret_cast<uint32_t*>(s_ones)[e] = 0x3F803F80u;  // bf16 1.0 pairs
  tc::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(&in_full[s], 1);
      tc::mbar_init(&in_empty[s], 1);
    }
    tc::mbar_init(done, 1);
    *abort_flag = 0u;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_holder, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_x);
      tc::prefetch_tmap(&tm_dla);
      tc::prefetch_tmap(&tm_dlx);
      int u = 0;
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int row0 = (rr + it * p.P) * TR;
        for (int o = 0; o <= NDL; ++o, ++u) {  // operand 0: x; then the gradient planes
          const int st = u % stages;
          if (!(ok = ctl.wait(&in_empty[st], ((u / stages) & 1) ^ 1u))) break;
          uint8_t* buf = s_in + st * TB;
          tc::mbar_expect_tx(&in_full[st], TB);
          if (o == 0) {
            for (int s = 0; s < k / 16; ++s)
              tc::tma_load_2d(buf + s * SLAB, &tm_x, &in_full[st], blk * k + 16 * s, row0);
          } else {
            const int m = p.nmat == 2 ? (o - 1) / p.nplanes : g;
            const int pl = (o - 1) % p.nplanes;
            for (int s = 0; s < k / 16; ++s)
              tc::tma_load_3d(buf + s * SLAB, m ? &tm_dlx : &tm_dla, &in_full[st],
                              blk * k + 16 * s, row0, pl);
          }
        }
      }
    }
  } else if (warp == 1) {
    const bool leader = tc::elect_one();
    const uint32_t id_dw = tc::idesc_bf16(TR, k, 1, 1);  // A = x MN-major, B = dl MN-major
    const uint32_t id_db = tc::idesc_bf16(TR, 16, 1, 0);  // A = dl MN-major, B = ones K-major
    const uint32_t ones = tc::smem_u32(s_ones);
    int u = 0;
    bool ok = true;
    for (int it = 0; it < my_tiles && ok; ++it) {
      const int sx = u % stages;
      if (!ctl.wait(&in_full[sx], (u / stages) & 1)) break;
      ++u;
      const uint32_t xs = tc::smem_u32(s_in + sx * TB);
      for (int o = 0; o < NDL; ++o, ++u) {
        const int st = u % stages;
        if (!ctl.wait(&in_full[st], (u / stages) & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const int mi = p.nmat == 2 ? o / p.nplanes : 0;  // matrix within the group
        const uint32_t dl = tc::smem_u32(s_in + st * TB);
        const uint32_t acc = tmem + mi * MCOLS;
        if (leader) {
          for (int kk = 0; kk < TR / 16; ++kk) {
            const uint32_t first = (it == 0 && o % p.nplanes == 0 && kk == 0) ? 0u : 1u;
            const uint64_t bdesc = tc::smem_desc_sw32(dl + kk * 512, SLAB, 256);
            const uint64_t odesc = tc::smem_desc_sw32(ones, 16, 256);
            for (int mb = 0; mb < MB; ++mb) {
              tc::mma_bf16(acc + mb * KC,
                           tc::smem_desc_sw32(xs + mb * 8 * SLAB + kk * 512, SLAB, 256), bdesc,
                           id_dw, first);
              tc::mma_bf16(acc + MB * KC + 32 * mb,
                           tc::smem_desc_sw32(dl + mb * 8 * SLAB + kk * 512, SLAB, 256), odesc,
                           id_db, first);
            }
          }
          tc::mma_commit(&in_empty[st]);
        }
        __syncwarp();
      }
      if (leader) tc::mma_commit(&in_empty[sx]);
      __syncwarp();
    }
    if (leader) tc::mma_commit(done);
    __syncwarp();
  } else {
    // partial sums of this CTA: dW rows i = 128 mb + 32 q + lane staged in box rings laid
    // over the drained operand buffers and stored by TMA (plane (blk P + r) 2 + m of the
    // partials map; rows past k are clipped), then db[j = 128 mb + 32 q + lane]
    const int q = warp & 3;
    const bool ok = my_tiles == 0 || ctl.wait(done, 0);
    tc::tc_fence_after();
    BoxStore<float> bs(s_in + (warp - 2) * ring_bytes(p.bi, 1), p.bi, 1, lane);
    const int NC = k / 16;
    for (int mi = 0; mi < p.nmat; ++mi) {
      const int m = p.nmat == 2 ? mi : g;
      const int z = (blk * p.P + rr) * 2 + m;
      float* dst = p.part + (size_t)z * ((size_t)k * k + k);
      for (int mb = 0; mb < MB; ++mb) {
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + mi * MCOLS + mb * KC;
        float v[2][16];
        if (my_tiles > 0 && ok) tc::tmem_ld16(ta, v[0]);
#pragma unroll 1
        for (int c = 0; c < NC; c += 2) {  // two chunks a step: the TMEM buffers stay static
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (c + h >= NC) break;
            if (my_tiles > 0 && ok) {
              tc::tmem_ld_wait();
              tc::reg_fence(v[h]);
              if (c + h + 1 < NC) tc::tmem_ld16(ta + 16 * (c + h + 1), v[h ^ 1]);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[h][e] = 0.0f;
            }
            bs.begin(c + h);
            bs.put(c + h, 0, v[h]);
            bs.end(c + h, &tm_part, 0, 128 * mb + 32 * q, z);
          }
        }
        const int j = 128 * mb + 32 * q + lane;
        float sb = 0.0f;
        if (my_tiles > 0 && ok) {
          float t[2];
          tc::tmem_ld2(tmem + ((uint32_t)(32 * q) << 16) + mi * MCOLS + MB * KC + 32 * mb, t);
          tc::tmem_ld_wait();
          tc::reg_fence(t);
          sb = t[0];
        }
        if (j < k) dst[(size_t)k * k + j] = sb;
      }
    }
    bs.drain();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// dW and db: the P partial sums of every (block, matrix) added in CTA order (deterministic).
// A thread takes four consecutive elements (k (k + 1) is a multiple of 4, and so is the
// dW / db boundary at k k): 16-byte loads, four partials requested at a time.
__global__ void k_proj_dw_reduce(const float* __restrict__ part, int nblk, int P, int k,
                                 float* dWa, float* dWx, float* dba, float* dbx) {
  const size_t per = (size_t)k * k + k;
  const size_t total4 = (size_t)nblk * 2 * per / 4;
  for (size_t e4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e4 < total4;
       e4 += (size_t)gridDim.x * blockDim.x) {
    const size_t e = 4 * e4;
    const size_t blk = e / (2 * per), rem = e % (2 * per);
    const int m = (int)(rem / per);
    const size_t off = rem % per;
    const float4* src = reinterpret_cast<const float4*>(part + (blk * P * 2 + m) * per + off);
    const size_t step = 2 * per / 4;  // float4s from one CTA's partials to the next
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](const float4& v) {
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    };
    int r = 0;
    for (; r + 4 <= P; r += 4) {
      const float4 a0 = src[r * step], a1 = src[(r + 1) * step];
      const float4 a2 = src[(r + 2) * step], a3 = src[(r + 3) * step];
      add(a0);
      add(a1);
      add(a2);
      add(a3);
    }
    for (; r < P; ++r) add(src[r * step]);
    if (off < (size_t)k * k) {
      *reinterpret_cast<float4*>((m ? dWx : dWa) + blk * k * k + off) = s;
    } else {
      float* db = m ? dbx : dba;
      if (db) *reinterpret_cast<float4*>(db + blk * k + (off - (size_t)k * k)) = s;
    }
  }
}

// float32 values as bf16 hi + lo planes (hi = bf16(v), lo = bf16(v - hi): v to ~2^-16), four
// values a thread: the gradient operands of the projection backward when the caller's
// gradients are float32.
__global__ void k_split_planes(const float4* __restrict__ src, uint2* hi, uint2* lo, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
    const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
    const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
    const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
    hi[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    lo[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
  }
}

// ---------------------------------------------------------------- host side
int ctas_per_group(int groups) {
  const int sms = sm_count();
  const int p = groups > 0 ? sms / groups : 0;
  return p < 1 ? 1 : p;
}

// Row tiles one dW accumulator takes at most.  The tensor core adds each K = 16 step into the
// float32 accumulator with a rounding that does not average out the way round-to-nearest sums
// do, so its error grows with the number of steps: measured at B8 T4096 with gate blocks of
// 160, 85 tiles (683 steps) per accumulator put two diagonal dW elements at E = 3.5e-3.  The
// row tiles are therefore split over enough CTAs that none accumulates more than this many;
// the per-CTA partials are then added on the CUDA cores in float32.
constexpr int DW_TILES_MAX = 16;

int dw_ctas_per_group(const Dims& d, int groups) {
  const int ntiles = (d.B * d.T + TR - 1) / TR;
  int P = ctas_per_group(groups);
  const int pmin = (ntiles + DW_TILES_MAX - 1) / DW_TILES_MAX;
  if (P < pmin) {  // whole waves of CTAs over the SMs
    const int sms = sm_count() > 0 ? sm_count() : 1;
    const long waves = ((long)groups * pmin + sms - 1) / sms;
    P = (int)std::max<long>(pmin, waves * sms / groups);
  }
  return std::max(1, std::min(P, ntiles));
}

int dw_nmat(const Dims& d) { return 2 * dw_mcols(d.k) <= 512 ? 2 : 1; }

cudaError_t weight_maps(const Dims& d, const void* Wa, const void* Wx, CUtensorMap* ma,
                        CUtensorMap* mx) {
  // W [nblk][k][k] viewed as [nblk * k rows (i)][k columns (j)]; box 16 columns x k rows
  const uint64_t dims[2] = {(uint64_t)d.k, (uint64_t)d.nblk * d.k};
  const uint64_t str[1] = {(uint64_t)d.k * 2};
  const uint32_t box[2] = {16, (uint32_t)d.k};
  cudaError_t e = encode_tmap(ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wa, dims, str, box,
                              CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  return encode_tmap(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wx, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_32B);
}

// An activation [R][W] bf16 as operand tiles: boxes of 16 channels x 128 rows.
cudaError_t act_map(const Dims& d, const void* base, CUtensorMap* m) {
  const uint64_t R = (uint64_t)d.B * d.T;
  const uint64_t dims[2] = {(uint64_t)d.W, R};
  const uint64_t str[1] = {(uint64_t)d.W * 2};
  const uint32_t box[2] = {16, TR};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_32B);
}

// The gradient operand of one matrix: nplanes planes [R][W] bf16, `plane_elems` apart.
cudaError_t planes_map(const Dims& d, const void* base, size_t plane_elems, int nplanes,
                       CUtensorMap* m) {
  const uint64_t R = (uint64_t)d.B * d.T;
  const uint64_t dims[3] = {(uint64_t)d.W, R, (uint64_t)nplanes};
  const uint64_t str[2] = {(uint64_t)d.W * 2, (uint64_t)plane_elems * 2};
  const uint32_t box[3] = {16, TR, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_32B);
}

// Row bytes of an output box: the widest of 128, 64, 32 that divides a block row of k elements.
int box_row_bytes(int k, int esize) {
  const int rb = k * esize;
  return rb % 128 == 0 ? 128 : (rb % 64 == 0 ? 64 : 32);
}

// An output [R][W] of element type et (planes of N elements apart: split hi + lo) in boxes of
// 32 rows x bi bytes, with the TMA swizzle of that width (the layout BoxStore writes).
cudaError_t out_map(const Dims& d, void* base, int et, int planes, int bi, CUtensorMap* m) {
  const int es = et == DT_F32 ? 4 : 2;
  const uint64_t dims[3] = {(uint64_t)d.W, (uint64_t)d.B * d.T, (uint64_t)planes};
  const uint64_t str[2] = {(uint64_t)d.W * es, (uint64_t)d.N * es};
  const uint32_t box[3] = {(uint32_t)(bi / es), 32, 1};
  const CUtensorMapSwizzle sw = bi == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                          : (bi == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_32B);
  return encode_tmap(m, et == DT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     3, base, dims, str, box, sw);
}

size_t bars_bytes(int n) { return 256 + (size_t)n * 8; }

}  // namespace

bool proj_tc_supported(const Dims& d) {
  return d.io == RGLRU_BF16 && d.k % 16 == 0 && d.k >= 16 && d.k <= PROJ_TC_KMAX &&
         sm_count() > 0;
}

ProjBwdSplit proj_bwd_split(const Dims& d) {
  // dx and dW side by side on one wave of CTAs: the P_dx + groups P_dw CTAs of a gate block fit
  // the SMs, dW's share near its share of the bytes moved (~45 %), and no dW accumulator takes
  // more than DW_TILES_MAX row tiles
  ProjBwdSplit sp = {0, 0};
  const int groups = 2 / dw_nmat(d);
  const int q = sm_count() / d.nblk;
  const int ntiles = (d.B * d.T + TR - 1) / TR;
  const int pmin = (ntiles + DW_TILES_MAX - 1) / DW_TILES_MAX;
  const int pdw = std::max(pmin, (int)(0.45 * q) / groups);
  const int pdx = q - groups * pdw;
  if (pdw >= 1 && pdx >= 1 && pdw <= dw_ctas_per_group(d, d.nblk * groups)) sp = {pdx, pdw};
  return sp;
}

size_t proj_dw_part_bytes(const Dims& d) {
  const int P = dw_ctas_per_group(d, d.nblk * (2 / dw_nmat(d)));
  return (size_t)d.nblk * P * 2 * ((size_t)d.k * d.k + d.k) * 4;
}

cudaError_t launch_split_planes(const Dims& d, const float* src, void* planes, cudaStream_t s) {
  const size_t n4 = (size_t)d.N / 4;  // W is a multiple of 16
  const int grid = (int)std::min<size_t>((n4 + 255) / 256, (size_t)8 * std::max(1, sm_count()));
  bf16* hi = static_cast<bf16*>(planes);
  k_split_planes<<<std::max(grid, 1), 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                                  reinterpret_cast<uint2*>(hi),
                                                  reinterpret_cast<uint2*>(hi + d.N), n4);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_proj_fwd(const Dims& d, int ot, const void* x, const void* Wa,
                            const float* ba, const void* Wx, const float* bx, void* lr, void* li,
                            cudaStream_t s) {
  if (!proj_tc_supported(d)) return cudaErrorNotSupported;
  const bool split = ot == DT_SPLIT;
  const int et = split ? DT_BF16 : ot;  // element type of each output plane
  CUtensorMap mx, mwa, mwx;
  cudaError_t e = act_map(d, x, &mx);
  if (e == cudaSuccess) e = weight_maps(d, Wa, Wx, &mwa, &mwx);
  if (e != cudaSuccess) return e;
  ProjParams p = {};
  p.R = d.B * d.T;
  p.k = d.k;
  p.nblk = d.nblk;
  p.W = d.W;
  p.P = ctas_per_group(d.nblk);
  p.bias[0] = ba;
  p.bias[1] = bx;
  // split: the lo planes follow the hi planes, N elements later (the maps' second plane)
  const int planes = split ? 2 : 1;
  p.bi = box_row_bytes(d.k, et == DT_F32 ? 4 : 2);
  CUtensorMap mlr, mli;
  e = out_map(d, lr, et, planes, p.bi, &mlr);
  if (e == cudaSuccess) e = out_map(d, li, et, planes, p.bi, &mli);
  if (e != cudaSuccess) return e;
  // two sets of epilogue warps where their box rings still leave two x stages
  const int NS = 512 / (int)kcols(d.k);
  const size_t TBs = tile_bytes(d.k);
  size_t smem = 0;
  int stages = 0;
  for (p.nsets = 2; p.nsets >= 1; --p.nsets) {
    const size_t fixed = 1024 + 2 * (size_t)d.k * d.k * 2 +
                         4 * (size_t)p.nsets * ring_bytes(p.bi, planes) + 2 * d.k * 4 +
                         bars_bytes(1 + 2 * NS);
    stages = fixed > SMEM_MAX ? 0 : (int)std::min<size_t>(6, (SMEM_MAX - fixed) / TBs);
    smem = fixed + stages * TBs;
    if (stages >= (p.nsets == 2 ? 2 : 1)) break;
  }
  if (p.nsets < 1 || stages < 1) return cudaErrorNotSupported;
  auto kern = split ? k_proj_fwd<bf16, true>
                    : (et == DT_F32 ? k_proj_fwd<float, false> : k_proj_fwd<bf16, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.P * d.nblk, 64 + 128 * p.nsets, smem, s>>>(mx, mwa, mwx, mlr, mli, p, stages);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_proj_dx(const Dims& d, int ot, const void* dlr, const void* dli,
                           size_t plane_elems, int nplanes, const void* Wa, const void* Wx,
                           const void* add, int add_f32, void* dx, cudaStream_t s, int P) {
  if (!proj_tc_supported(d)) return cudaErrorNotSupported;
  CUtensorMap mdla, mdlx, mwa, mwx;
  cudaError_t e = planes_map(d, dlr, plane_elems, nplanes, &mdla);
  if (e == cudaSuccess) e = planes_map(d, dli, plane_elems, nplanes, &mdlx);
  if (e == cudaSuccess) e = weight_maps(d, Wa, Wx, &mwa, &mwx);
  if (e != cudaSuccess) return e;
  ProjParams p = {};
  p.R = d.B * d.T;
  p.k = d.k;
  p.nblk = d.nblk;
  p.W = d.W;
  p.P = P > 0 ? P : ctas_per_group(d.nblk);
  p.add = add;
  p.add_f32 = add_f32;
  p.nplanes = nplanes;
  p.bi = box_row_bytes(d.k, ot == DT_F32 ? 4 : 2);
  CUtensorMap mdx, madd;
  e = out_map(d, dx, ot, 1, p.bi, &mdx);
  // a bf16 addend enters as an operand tile (the kernel's identity product); a float32 one
  // through the epilogue, and its map is unused
  if (e == cudaSuccess) e = act_map(d, add_f32 ? dx : add, &madd);
  if (e != cudaSuccess) return e;
  const size_t idb = add_f32 ? 0 : ID_BYTES;
  // two sets of epilogue warps where their box rings still leave three operand stages
  const size_t TBs = tile_bytes(d.k);
  size_t smem = 0;
  int stages = 0;
  for (p.nsets = 2; p.nsets >= 1; --p.nsets) {
    const size_t fixed = 1024 + 2 * (size_t)d.k * d.k * 2 + idb +
                         4 * (size_t)p.nsets * ring_bytes(p.bi, 1) + bars_bytes(5);
    stages = fixed > SMEM_MAX ? 0 : (int)std::min<size_t>(6, (SMEM_MAX - fixed) / TBs);
    smem = fixed + stages * TBs;
    if (stages >= (p.nsets == 2 ? 3 : 2)) break;
  }
  if (p.nsets < 1 || stages < 2) return cudaErrorNotSupported;
  auto kern = ot == DT_F32 ? (add_f32 ? k_proj_dx<float, float> : k_proj_dx<float, bf16>)
                           : (add_f32 ? k_proj_dx<bf16, float> : k_proj_dx<bf16, bf16>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.P * d.nblk, 64 + 128 * p.nsets, smem, s>>>(mdla, mdlx, mwa, mwx, mdx, madd, p, stages);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_proj_dw(const Dims& d, const void* x, const void* dlr, const void* dli,
                           size_t plane_elems, int nplanes, float* part, float* dWa, float* dba,
                           float* dWx, float* dbx, cudaStream_t s, int P) {
  if (!proj_tc_supported(d)) return cudaErrorNotSupported;
  CUtensorMap mx, mdla, mdlx;
  cudaError_t e = act_map(d, x, &mx);
  if (e == cudaSuccess) e = planes_map(d, dlr, plane_elems, nplanes, &mdla);
  if (e == cudaSuccess) e = planes_map(d, dli, plane_elems, nplanes, &mdlx);
  if (e != cudaSuccess) return e;
  ProjParams p = {};
  p.R = d.B * d.T;
  p.k = d.k;
  p.nblk = d.nblk;
  p.W = d.W;
  p.nplanes = nplanes;
  p.nmat = dw_nmat(d);
  const int groups = 2 / p.nmat;
  // P given: the split of proj_bwd_split, next to a running dx grid (programmatic launch)
  const bool beside = P > 0;
  p.P = beside ? P : dw_ctas_per_group(d, d.nblk * groups);
  p.part = part;
  // the partial sums [nblk P 2 planes][k + 1 rows][k]: dW in the first k rows of a plane,
  // stored in boxes of 32 rows (rows past k clipped); db in the last row, by plain stores
  p.bi = box_row_bytes(d.k, 4);
  CUtensorMap mpart;
  {
    const uint64_t dims[3] = {(uint64_t)d.k, (uint64_t)d.k, (uint64_t)d.nblk * p.P * 2};
    const uint64_t str[2] = {(uint64_t)d.k * 4, ((uint64_t)d.k * d.k + d.k) * 4};
    const uint32_t box[3] = {(uint32_t)(p.bi / 4), 32, 1};
    e = encode_tmap(&mpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part, dims, str, box,
                    p.bi == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (e != cudaSuccess) return e;
  }
  const size_t TB = tile_bytes(d.k);
  const size_t fixed = 1024 + SLAB + dw_pad(d.k) + bars_bytes(1);
  // all operands of one row tile (x and the group's gradient planes) are held at once
  const int need = p.nmat * nplanes + 1;
  int stages = 8;
  while (stages > need && fixed + stages * TB + 16 * stages > SMEM_MAX) --stages;
  const size_t smem = fixed + stages * TB + 16 * stages;
  if (smem > SMEM_MAX) return cudaErrorNotSupported;
  // the epilogue's box rings lie over the drained operand buffers
  if (4 * (size_t)ring_bytes(p.bi, 1) > stages * TB) return cudaErrorNotSupported;
  e = cudaFuncSetAttribute(k_proj_dw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (beside) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.P * d.nblk * groups);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_proj_dw, mx, mdla, mdlx, mpart, p, stages);
  } else {
    k_proj_dw<<<p.P * d.nblk * groups, NTHREADS, smem, s>>>(mx, mdla, mdlx, mpart, p, stages);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  note_launches(1);
  const size_t total4 = (size_t)d.nblk * 2 * ((size_t)d.k * d.k + d.k) / 4;
  const int rgrid = (int)std::min<size_t>((total4 + 255) / 256, 4096);
  k_proj_dw_reduce<<<rgrid, 256, 0, s>>>(part, d.nblk, p.P, d.k, dWa, dWx, dba, dbx);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rglru
