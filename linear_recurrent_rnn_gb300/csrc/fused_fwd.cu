// Fused RG-LRU forward on one GB300: block-diagonal gate projections on the tcgen05 tensor
// cores, gates / decay / multiplier / write and the exact chunked scan on the CUDA cores, in
// one persistent kernel.  The gate logits live only in tensor memory (float32), never in HBM.
//
// Sources ("Fattori comparison" page): the operator takes the recurrent input and both raw
// gate logits produced by two block-diagonal projections (first paragraph), fuses the sigmoid
// gates, softplus(a_param) with the dynamic decay, the square-root multiplier, the input-gated
// write and the recurrence (the fused-steps list), and the page closes by adopting that fusion
// and adding an exact parallel chunked scan with partial chunks.  Math: r = sigmoid(lr),
// i = sigmoid(li), log a = -8 r softplus(Lambda), m = sqrt(1 - a^2) (m = 1 and no carry at a
// reset token), h_t = a h_{t-1} + m i x.
//
// Tile = (batch row b, gate block blk, 64 tokens).  For the tile the MMA computes the
// transposed logits  lr^T[128 ch x 64 tok] = Wa[blk]^T (MN-major A, from W stored (in, out))
// x x_tile^T (K-major B, the x tile as TMA lands it), and li^T likewise, so TMEM lane =
// channel and column = token.  Two scan threads own each channel, one per 32-token part: each
// runs its part serially in registers from a zero state and parks the local states in TMEM;
// an output thread per channel joins the parts, and chunks through the anchored look-back over
// value slots in `saved` (lookback.cuh), which keeps the result bitwise deterministic.
//
// Roles (448 threads, one CTA per SM, launched cooperatively so that all CTAs are resident):
//   warp 0       TMA producer: Wa[blk], Wx[blk] once, then the x tile ring (7 stages)
//   warp 1       MMA issuer: 2 x 8 tcgen05.mma (K = 16 each) per tile into a 4-deep TMEM ring
//   warps 2..9   scan: warps 2+4p .. 5+4p take tokens 32p .. 32p+31 (lane quadrant warp % 4),
//                tile after tile, parking each over its own logits, with no barrier
//   warps 10..13 output: per parked tile, publish its aggregate, then finish the tile before
//                it (look-back, chunk-boundary state, y): each warp its 32 channels, through
//                its own double-buffered shared-memory strip and TMA store, with no barrier
// CTA (blk, r) of the P CTAs serving gate block blk takes the block's tiles n = r, r + P, ...
// in chunk-major order, so every tile it waits on is earlier in the same order.
#include <cudaTypedefs.h>

#include "host_util.h"
#include "internal.h"
#include "lookback.cuh"
#include "tc.cuh"

namespace rglru {

namespace {

constexpr int NPART = 2;              // token parts of a tile, one scan thread each per channel
constexpr int PT = FUSED_C / NPART;   // tokens per scan thread
constexpr int NSCAN = 4 * NPART;      // scan warps (4 lane quadrants per part)
constexpr int NOUT = 4;               // output warps, one per TMEM lane quadrant
constexpr int NTHREADS = 64 + (NSCAN + NOUT) * 32;
// The warps share the SM's four 16 K-register sub-partitions: registers per thread <= 16384 /
// (32 x warps per sub-partition), rounded down to a multiple of 8.
constexpr int MAXREG = (16384 / (((NSCAN + NOUT + 2 + 3) / 4) * 32)) / 8 * 8;
// x tiles in flight: the deepest ring the shared memory holds (the x reads of a tile wait on
// DRAM under the load of every SM; 3 -> 6 -> 7 stages took the forward call 41.1 -> 39.2 ->
// 38.6 us)
constexpr int XSTAGES = 7;
constexpr uint32_t W_BYTES = FUSED_K * FUSED_K * 2;  // one weight block, bf16
constexpr uint32_t X_BYTES = FUSED_C * FUSED_K * 2;  // one x tile, bf16
constexpr uint32_t YSTRIP_BYTES = FUSED_C * 32 * 2;  // y of 64 tokens x 32 channels, bf16
constexpr uint32_t Y_BYTES = NOUT * 2 * YSTRIP_BYTES;  // two strips per output warp
constexpr uint32_t SLAB_X = FUSED_C * 32;            // 16 channels x 64 tokens
constexpr uint32_t SLAB_W = FUSED_K * 32;            // 16 out-channels x 128 in-rows
// A ring of 4 tile buffers of 128 columns (lr 64 + li 64): the MMA writes a tile's logits,
// the scan threads overwrite them in place with the local states (over lr) and the decay
// products (over li), and the output threads read those out and release the buffer.
constexpr uint32_t TMEM_COLS = 512;
constexpr int NBUF = 4;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s: a pipeline wait never lasts this
constexpr uint32_t XCH_BYTES = NBUF * NPART * FUSED_K * 8;  // part maps, one set per buffer
constexpr size_t SMEM_BYTES =
    2 * W_BYTES + XSTAGES * X_BYTES + Y_BYTES + XCH_BYTES + 256 + 1024;
// Given-logits mode (the scan of rglru_forward and of the composed layer): no weights; each
// stage holds the x tile and up to two bf16 planes of each logit tile, and a 64 x 64 identity
// takes the place of W in the MMA that lays the logits out in TMEM.
// A stage holds x and the planes actually given, so one plane a logit (48 KB a stage) gets
// three stages in the region that two planes (80 KB a stage) fill with two.
constexpr int LG_PLANES = 2;
constexpr int LG_STAGES_MAX = 3;
__host__ __device__ constexpr uint32_t lg_stage_bytes(int nplanes) {
  return (1 + 2 * nplanes) * X_BYTES;
}
__host__ __device__ constexpr int lg_stages(int nplanes) { return nplanes == 1 ? 3 : 2; }
constexpr uint32_t LG_REGION = 2 * lg_stage_bytes(LG_PLANES);
static_assert(lg_stages(1) * lg_stage_bytes(1) <= LG_REGION, "one-plane stages fit the region");
static_assert(lg_stages(1) <= LG_STAGES_MAX && lg_stages(2) <= LG_STAGES_MAX, "barriers");
constexpr uint32_t ID_BYTES = FUSED_C * FUSED_C * 2;
constexpr size_t LG_SMEM_BYTES = ID_BYTES + LG_REGION + Y_BYTES + XCH_BYTES + 256 + 1024;
constexpr uint32_t STATUS_PIPE = 2u;

struct FwdParams {
  int B, T, W, nblk, nC, P, canonical;
  int nplanes;  // given-logits mode: bf16 planes per logit (1, or 2 = hi + lo)
  const float* Lambda;
  const float* ba;
  const float* bx;
  const uint8_t* reset_mask;
  const int32_t* segment_pos;
  const float* h0;
  float* hT;
  // packed variable-length sequences (null seq_start: none); one row
  const int32_t* seq_start;
  const int32_t* seq_end;
  const float* h0s;
  float* hTs;
  uint8_t* scratch;
  ScanLayout L;
  int spin_limit, drop_tile;
  int lb_dist, lb_shift;
};

struct Ctl {
  volatile uint32_t* abort;
  uint32_t* status;
  // Bounded wait; after any failure in the CTA every later wait returns at once, so the
  // kernel winds down in bounded time (with the failure recorded in the status word).
  __device__ bool wait(uint64_t* bar, uint32_t parity) const {
    if (*abort) return false;
    if (tc::mbar_wait(bar, parity, WAIT_LIMIT_NS)) return true;
    *abort = 1u;
    atomicOr(status, STATUS_PIPE);
    return false;
  }
};

// Local scan of one scan thread's PT tokens from a zero state.  The pointwise work runs on
// token pairs (u, u + 1) in the two lanes of f32x2 operations (adjacent TMEM columns land in
// adjacent registers); the recurrence itself is a scalar chain.  The state after each token
// (hl) and the product of abar up to it (Ac) are parked in TMEM as they are made, over the
// logits just read (hl over lr, Ac over li); (rA, rh) = the part's map.  This is the fast
// variant (chosen warp-uniformly): no reset, every token before T, every decay with la > -1/8;
// local_scan_gen below handles the others.
constexpr int GRP = 8;  // tokens per TMEM load / store group
// Sequence starts (smask): the token continues from its sequence's initial state instead of
// the carried one, h -> a h0[s] + m i x.
struct SeqStarts {
  uint32_t smask;         // tokens of the part where a sequence starts
  const int32_t* seq;     // sequence index of the part's tokens (valid where smask is set)
  const float* h0;        // h0[0][w] of the channel, rows W apart, or null (zeros)
  int W;
};
__device__ __forceinline__ float seq_h0(const SeqStarts& sq, int u) {
  return sq.h0 ? sq.h0[(size_t)sq.seq[u] * sq.W] : 0.0f;
}
__device__ __forceinline__ void local_scan(uint32_t t_lr, uint32_t t_li, uint32_t xb0,
                                           uint32_t xb1, const GateK& gk, float& rh, float& rA) {
  rh = 0.0f;
  rA = 1.0f;
  // the logits of group g + 1 are requested before group g is computed
  float vr[GRP], vi[GRP];
  tc::tmem_ld8(t_lr, vr);
  tc::tmem_ld8(t_li, vi);
  tc::tmem_ld_wait();
  tc::reg_fence(vr);
  tc::reg_fence(vi);
#pragma unroll
  for (int g = 0; g < PT / GRP; ++g) {
    float oh[GRP], oa[GRP], nr[GRP], ni[GRP];
    if (g + 1 < PT / GRP) {
      tc::tmem_ld8(t_lr + (g + 1) * GRP, nr);
      tc::tmem_ld8(t_li + (g + 1) * GRP, ni);
    }
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;  // tokens u, u + 1 of the part
      const float2 xv = make_float2(tok_elem(xb0, xb1, u), tok_elem(xb0, xb1, u + 1));
      const float2 lr = make_float2(vr[2 * q], vr[2 * q + 1]);
      const float2 li = make_float2(vi[2 * q], vi[2 * q + 1]);
      float2 abar, mi, r;
      gates_near2(lr, li, gk, abar, mi, r);
      const float2 bv = mul2(mi, xv);
      rh = fmaf(abar.x, rh, bv.x);
      rA *= abar.x;
      oh[2 * q] = rh;
      oa[2 * q] = rA;
      rh = fmaf(abar.y, rh, bv.y);
      rA *= abar.y;
      oh[2 * q + 1] = rh;
      oa[2 * q + 1] = rA;
    }
    tc::tmem_st8(t_lr + g * GRP, oh);
    tc::tmem_st8(t_li + g * GRP, oa);
    if (g + 1 < PT / GRP) {
      tc::tmem_ld_wait();
      tc::reg_fence(nr);
      tc::reg_fence(ni);
#pragma unroll
      for (int u = 0; u < GRP; ++u) {
        vr[u] = nr[u];
        vi[u] = ni[u];
      }
    }
  }
  tc::tmem_st_wait();
}

// The general variant of the local scan (resets, tokens past T, far decays, sequence starts),
// on a few tiles a launch: the same arithmetic, walking the token groups in a loop rather
// than unrolled, which keeps the kernel's code around the fast variant small.
template <bool VARLEN>
__device__ __forceinline__ void local_scan_gen(uint32_t t_lr, uint32_t t_li, uint32_t xb0,
                                               uint32_t xb1, const GateK& gk, uint32_t rmask,
                                               int valid, const SeqStarts& sq, float& rh,
                                               float& rA) {
  rh = 0.0f;
  rA = 1.0f;
#pragma unroll 1
  for (int g = 0; g < PT / GRP; ++g) {
    float vr[GRP], vi[GRP], oh[GRP], oa[GRP];
    tc::tmem_ld8(t_lr + g * GRP, vr);
    tc::tmem_ld8(t_li + g * GRP, vi);
    tc::tmem_ld_wait();
    tc::reg_fence(vr);
    tc::reg_fence(vi);
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;  // tokens u, u + 1 of the part
      const float2 xv = make_float2(tok_elem(xb0, xb1, u), tok_elem(xb0, xb1, u + 1));
      float2 abar, mi, r, i;
      gates_any2(make_float2(vr[2 * q], vr[2 * q + 1]), make_float2(vi[2 * q], vi[2 * q + 1]),
                 gk, abar, mi, r, i);
      if ((rmask >> u) & 1u) {
        abar.x = 0.0f;
        mi.x = i.x;
      }
      if ((rmask >> (u + 1)) & 1u) {
        abar.y = 0.0f;
        mi.y = i.y;
      }
      if (u >= valid) {
        abar.x = 1.0f;
        mi.x = 0.0f;
      }
      if (u + 1 >= valid) {
        abar.y = 1.0f;
        mi.y = 0.0f;
      }
      float2 bv = mul2(mi, xv);
      if (VARLEN && sq.smask) {
        if ((sq.smask >> u) & 1u) {
          bv.x = fmaf(abar.x, seq_h0(sq, u), bv.x);
          abar.x = 0.0f;
        }
        if ((sq.smask >> (u + 1)) & 1u) {
          bv.y = fmaf(abar.y, seq_h0(sq, u + 1), bv.y);
          abar.y = 0.0f;
        }
      }
      rh = fmaf(abar.x, rh, bv.x);
      rA *= abar.x;
      oh[2 * q] = rh;
      oa[2 * q] = rA;
      rh = fmaf(abar.y, rh, bv.y);
      rA *= abar.y;
      oh[2 * q + 1] = rh;
      oa[2 * q + 1] = rA;
    }
    tc::tmem_st8(t_lr + g * GRP, oh);
    tc::tmem_st8(t_li + g * GRP, oa);
  }
  tc::tmem_st_wait();
}

// LG: given-logits mode.  tm_wa / tm_wx then map the bf16 logit planes lr, li
// [plane][B][T][W]; blk is a 128-channel slice of W (the last one may be partial: its channels
// past W read zeros and write nothing).
template <bool VARLEN, bool LG>
__global__ void __maxnreg__(MAXREG)
    k_fused_fwd(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
                const __grid_constant__ CUtensorMap tm_wx, const __grid_constant__ CUtensorMap tm_y,
                FwdParams p) {
  const int XS = LG ? lg_stages(p.nplanes) : XSTAGES;           // stages in use
  const uint32_t STB = LG ? lg_stage_bytes(p.nplanes) : X_BYTES;  // bytes a stage
  constexpr int XSB = LG ? LG_STAGES_MAX : XSTAGES;               // stage barriers
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by pointer arithmetic so that it stays a shared pointer
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_wa = smem;            // LG: the identity
  uint8_t* s_wx = smem + W_BYTES;  // (unused in LG)
  uint8_t* s_x = smem + (LG ? ID_BYTES : 2 * W_BYTES);
  uint8_t* s_y = s_x + (LG ? LG_REGION : XSTAGES * X_BYTES);
  float2* s_agg = reinterpret_cast<float2*>(s_y + Y_BYTES);  // [buffer][part][channel]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_agg + NBUF * NPART * FUSED_K);
  uint64_t* w_full = bars;
  uint64_t* x_full = bars + 1;
  uint64_t* x_empty = bars + 1 + XSB;
  uint64_t* acc_full = bars + 1 + 2 * XSB;
  uint64_t* acc_empty = acc_full + NBUF;  // buffer read out by the output warps
  uint64_t* park_full = acc_empty + NBUF;  // a tile parked in its buffer (scan -> output)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(park_full + NBUF);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x / p.P, rr = blockIdx.x % p.P;
  const int ntiles = p.B * p.nC;
  uint32_t* status = reinterpret_cast<uint32_t*>(p.scratch);
  const Ctl ctl{abort_flag, status};

  if (threadIdx.x == 0) {
    tc::mbar_init(w_full, 1);
    for (int s = 0; s < XS; ++s) {
      tc::mbar_init(&x_full[s], 1);
      // LG: the stage also holds the logit planes, read by the MMA
      tc::mbar_init(&x_empty[s], NSCAN + (LG ? 1 : 0));
    }
    for (int a = 0; a < NBUF; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], NOUT);
      tc::mbar_init(&park_full[a], NSCAN);
    }
    *abort_flag = 0u;
    tc::fence_barrier_init();
  }
  if (LG) tc::write_identity_sw32(s_wa, FUSED_C);
  if (warp == 0) {
    tc::tmem_alloc(tmem_holder, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  int my_tiles = 0;
  for (int n = rr; n < ntiles; n += p.P) ++my_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_x);
      tc::prefetch_tmap(&tm_wa);
      tc::prefetch_tmap(&tm_wx);
      if (!LG) {
        tc::mbar_expect_tx(w_full, 2 * W_BYTES);
        for (int g = 0; g < FUSED_K / 16; ++g) {
          tc::tma_load_2d(s_wa + g * SLAB_W, &tm_wa, w_full, 16 * g, blk * FUSED_K);
          tc::tma_load_2d(s_wx + g * SLAB_W, &tm_wx, w_full, 16 * g, blk * FUSED_K);
        }
      } else {
        tc::mbar_arrive(w_full);  // the identity is in place (written before the CTA barrier)
      }
      int it = 0;
      TileWalk tw(rr, p.P, p.B);
      for (int n = rr; n < ntiles; n += p.P, ++it, tw.next()) {
        const int st = it % XS;
        const uint32_t ph = (it / XS) & 1;
        if (!ctl.wait(&x_empty[st], ph ^ 1u)) continue;
        uint8_t* sb = s_x + st * STB;
        tc::mbar_expect_tx(&x_full[st], LG ? (1 + 2 * p.nplanes) * X_BYTES : X_BYTES);
        for (int s = 0; s < FUSED_K / 16; ++s)
          tc::tma_load_3d(sb + s * SLAB_X, &tm_x, &x_full[st], blk * FUSED_K + 16 * s,
                          tw.c * FUSED_C, tw.b);
        if (LG) {
          for (int g = 0; g < 2; ++g)
            for (int pl = 0; pl < p.nplanes; ++pl)
              for (int s = 0; s < FUSED_K / 16; ++s)
                tc::tma_load_4d(sb + (1 + g * p.nplanes + pl) * X_BYTES + s * SLAB_X,
                                g ? &tm_wx : &tm_wa, &x_full[st], blk * FUSED_K + 16 * s,
                                tw.c * FUSED_C, tw.b, pl);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (the descriptor arithmetic stays warp-uniform); one elected
    // lane issues the MMAs and commits.
    const bool leader = tc::elect_one();
    {
      constexpr uint32_t idesc = tc::idesc_bf16(128, FUSED_C, /*A MN-major*/ 1, /*B K-major*/ 0);
      ctl.wait(w_full, 0);
      const uint32_t wa = tc::smem_u32(s_wa), wx = tc::smem_u32(s_wx);
      int it = 0;
      for (int n = rr; n < ntiles; n += p.P, ++it) {
        const int st = it % XS;
        const uint32_t ph = (it / XS) & 1;
        const int a = it % NBUF;
        const uint32_t aph = (it / NBUF) & 1;
        if (!ctl.wait(&acc_empty[a], aph ^ 1u)) continue;
        if (!ctl.wait(&x_full[st], ph)) continue;
        tc::tc_fence_after();
        const uint32_t xs = tc::smem_u32(s_x + st * STB);
        const uint32_t d_r = tmem + a * 128, d_i = d_r + 64;
        if (!LG) {
#pragma unroll
          for (int kk = 0; kk < FUSED_K / 16; ++kk) {
            // A: W^T, MN-major, 16-channel groups 4 KB apart (LBO), 8-row K groups 256 B (SBO);
            // B: x tile, K-major, one 16-channel slab per K step, 8-row groups 256 B apart.
            const uint64_t bdesc = tc::smem_desc_sw32(xs + kk * SLAB_X, 16, 256);
            if (leader) tc::mma_bf16(d_r, tc::smem_desc_sw32(wa + kk * 512, SLAB_W, 256), bdesc, idesc, kk > 0);
            if (leader) tc::mma_bf16(d_i, tc::smem_desc_sw32(wx + kk * 512, SLAB_W, 256), bdesc, idesc, kk > 0);
          }
        } else if (leader) {
          // lr^T = L_r^T I: A = the logit plane tile, MN-major (16-channel slabs 2 KB apart,
          // 16 tokens per K step); B = the identity, K-major; the planes accumulate (hi + lo)
          for (int g = 0; g < 2; ++g)
            for (int pl = 0; pl < p.nplanes; ++pl)
#pragma unroll
              for (int kk = 0; kk < FUSED_C / 16; ++kk)
                tc::mma_bf16(g ? d_i : d_r,
                             tc::smem_desc_sw32(xs + (1 + g * p.nplanes + pl) * X_BYTES + kk * 512,
                                                SLAB_X, 256),
                             tc::smem_desc_sw32(wa + kk * SLAB_X, 16, 256), idesc,
                             (pl > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) {
          tc::mma_commit(&acc_full[a]);
          if (LG) tc::mma_commit(&x_empty[st]);  // the logit planes are read
        }
        __syncwarp();
      }
    }
  } else if (warp < 2 + NSCAN) {
    // ------------------------------------------------------------ scan warps
    // Local scans back to back: each tile is parked in its TMEM buffer (with the parts' maps in
    // shared memory) and handed to the output warps; no barrier among the scan warps.
    const int part = (warp - 2) >> 2;  // token part of the tile
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int j = q * 32 + lane;
    // channels past W (LG only) compute, unstored
    const int w = LG ? min(blk * FUSED_K + j, p.W - 1) : blk * FUSED_K + j;
    const int tb = part * PT;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    GateK gk;
    gk.nk = -8.0f * softplus_f(p.Lambda[w]);  // log a = nk * r
    gk.cm = sqrtf(-2.0f * gk.nk);
    gk.nbr = p.ba ? -p.ba[w] * LOG2E : 0.0f;  // biases folded into the exponents
    gk.nbi = p.bx ? -p.bx[w] * LOG2E : 0.0f;
    // x[token tl, channel j] of a stage: 16-byte halves of the 32-byte row swap on rows 4..7
    // of every 8 (32-byte swizzle), so two base pointers cover both row parities.
    const int xoff0 = (j >> 4) * SLAB_X + (j & 7) * 2 + (((j & 15) >> 3) << 4);
    const int xoff1 = (j >> 4) * SLAB_X + (j & 7) * 2 + ((((j & 15) >> 3) ^ 1) << 4);
    // Warp-uniform: every channel of this warp has la > -1/8 on every token.
    const bool near_all = __all_sync(0xffffffffu, gk.nk > NEAR_LA);

    // this lane's token markers of a tile (lane < PT: one token of the part each)
    const int32_t* seq_start = VARLEN ? p.seq_start : nullptr;
    auto marks = [&](const TileWalk& tw) {
      const int t = tw.c * FUSED_C + tb + lane;
      return tok_marks_load(p.reset_mask, p.segment_pos, seq_start, nullptr,
                            (size_t)tw.b * p.T + t, lane < PT && t < p.T);
    };
    TileWalk cur(rr, p.P, p.B);
    TokMarks mk = marks(cur);  // tile it's, requested during tile it - 1
    for (int it = 0; it < my_tiles; ++it, cur.next()) {
      const int c = cur.c, b = cur.b;
      const int st = it % XS;
      const uint32_t ph = (it / XS) & 1;
      const int a = it % NBUF;
      const uint32_t aph = (it / NBUF) & 1;
      const TokMarks now = mk;
      if (it + 1 < my_tiles) {
        TileWalk nx = cur;
        nx.next();
        mk = marks(nx);
      }
      const uint32_t rmask =
          __ballot_sync(0xffffffffu, tok_marks_reset(now, p.reset_mask, p.segment_pos));
      const int valid = min(FUSED_C, p.T - c * FUSED_C) - tb;  // tokens of this part < T
      SeqStarts sq{0u, nullptr, nullptr, p.W};
      if (VARLEN) {
        sq.seq = p.seq_start + (size_t)b * p.T + c * FUSED_C + tb;
        sq.smask = __ballot_sync(0xffffffffu, now.st >= 0);
        sq.h0 = p.h0s ? p.h0s + w : nullptr;
      }
      ctl.wait(&acc_full[a], aph);
      ctl.wait(&x_full[st], ph);
      tc::tc_fence_after();
      const uint32_t xt = tc::smem_u32(s_x + st * STB + tb * 32);
      const uint32_t xb0 = xt + xoff0, xb1 = xt + xoff1;
      const uint32_t t_lr = tmem + lane_base + a * 128 + tb;
      float rh, rA;
      if (near_all && rmask == 0u && sq.smask == 0u && valid >= PT)
        local_scan(t_lr, t_lr + 64, xb0, xb1, gk, rh, rA);
      else
        local_scan_gen<VARLEN>(t_lr, t_lr + 64, xb0, xb1, gk, rmask, valid, sq, rh, rA);
      s_agg[(a * NPART + part) * FUSED_K + j] = make_float2(rA, rh);  // the part's map
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&x_empty[st]);
        tc::mbar_arrive(&park_full[a]);
      }
    }
  } else {
    // ------------------------------------------------------------ output warps
    // One thread per channel.  Iteration it publishes tile it's aggregate as soon as it is
    // parked, finishes tile it - 1 (look-back, carry, y), then requests tile it's look-back
    // slots, which have the next tile's scan to arrive.
    const int q = warp & 3;
    const int j = q * 32 + lane;
    // channels past W (LG only): nothing stored, their look-back reads a real channel's
    const bool wok = !LG || blk * FUSED_K + j < p.W;
    const int w = LG ? min(blk * FUSED_K + j, p.W - 1) : blk * FUSED_K + j;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* carry = reinterpret_cast<float*>(p.scratch + p.L.carry);
    float2* agg = reinterpret_cast<float2*>(p.scratch + p.L.agg);
    // y goes out per warp: 32 channels x 64 tokens through one of two shared-memory strips
    uint8_t* ystrip = s_y + (warp - 2 - NSCAN) * 2 * YSTRIP_BYTES;
    if (lane == 0) tc::prefetch_tmap(&tm_y);

    TileWalk cur(rr, p.P, p.B);
    int pc = 0, pb = 0;              // chunk and row of tile it - 1
    float Pa[NPART], Pb[NPART];      // tile it - 1: the map of the parts before each part
    float Ta = 1.0f, Tb = 0.0f;      // tile it - 1: the tile's map
    LookbackReq lbq;                 // tile it - 1's look-back
    int lb_n = 0;
    const float2* lb_agg = agg;
    const float* lb_anchor = nullptr;
    // packed sequences ending at the tile's tokens lane and 32 + lane: tile it - 1's, and tile
    // it's, requested an iteration ahead of their use
    int pe0 = -1, pe1 = -1;
#pragma unroll
    for (int pp = 0; pp < NPART; ++pp) Pa[pp] = 1.0f, Pb[pp] = 0.0f;
    for (int it = 0; it <= my_tiles; ++it) {
      // 1. tile it, parked: its map (the parts composed) and its aggregate, published at once
      float nPa[NPART], nPb[NPART], nTa = 1.0f, nTb = 0.0f;
      const int n = rr + it * p.P;
      int ce0 = -1, ce1 = -1;
      if (VARLEN && it < my_tiles) {
        const size_t tb0 = (size_t)cur.b * p.T + (size_t)cur.c * FUSED_C;
        if (cur.c * FUSED_C + lane < p.T) ce0 = p.seq_end[tb0 + lane];
        if (cur.c * FUSED_C + 32 + lane < p.T) ce1 = p.seq_end[tb0 + 32 + lane];
      }
      if (it < my_tiles) {
        const int a = it % NBUF;
        ctl.wait(&park_full[a], (it / NBUF) & 1);
        tc::tc_fence_after();
#pragma unroll
        for (int pp = 0; pp < NPART; ++pp) {
          const float2 g = s_agg[(a * NPART + pp) * FUSED_K + j];
          nPa[pp] = nTa;
          nPb[pp] = nTb;
          nTb = fmaf(g.x, nTb, g.y);
          nTa *= g.x;
        }
        if ((blk * ntiles + n) != p.drop_tile && wok)
          slot_put2(agg + ((size_t)cur.b * p.nC + cur.c) * p.W + w, nTa, nTb);
      }

      // 2. finish tile it - 1: its carry-in, the chunk-boundary state, y
      if (it > 0) {
        const int a = (it - 1) % NBUF;
        const float hin_t =
            lookback_finish(lbq, lb_agg, -(long)p.W, lb_n, lb_anchor, p.spin_limit, status);
        const float hend = fmaf(Ta, hin_t, Tb);
        float* crow = carry + (size_t)pb * (p.nC + 1) * p.W;
        if ((blk * ntiles + n - p.P) != p.drop_tile && wok)
          slot_put1(crow + (size_t)(pc + 1) * p.W + w, hend);
        if (pc == 0 && wok) slot_put1(crow + w, hin_t);
        if (pc == p.nC - 1 && p.hT && wok) p.hT[(size_t)pb * p.W + w] = hend;
        // packed sequences ending in the tile: their final state (warp-uniform masks)
        uint32_t em0 = 0u, em1 = 0u;
        const int e0 = pe0, e1 = pe1;
        if (VARLEN) {
          em0 = __ballot_sync(0xffffffffu, e0 >= 0);
          em1 = __ballot_sync(0xffffffffu, e1 >= 0);
        }
        uint8_t* yb = ystrip + ((it - 1) & 1) * YSTRIP_BYTES;
        if (lane == 0) tc::tma_store_wait_read1();  // the strip stored two tiles ago is free
        __syncwarp();
        // y strip: registers -> smem [token][32 channels] -> TMA store (clipped at T)
#pragma unroll
        for (int pp = 0; pp < NPART; ++pp) {
          const float hin = fmaf(Pa[pp], hin_t, Pb[pp]);
          const uint32_t park = tmem + lane_base + a * 128 + pp * PT;  // hl; Ac at + 64
#pragma unroll
          for (int c16 = 0; c16 < PT; c16 += 16) {
            float hl[16], Ac[16];
            tc::tmem_ld16(park + c16, hl);
            tc::tmem_ld16(park + 64 + c16, Ac);
            tc::tmem_ld_wait();
            tc::reg_fence(hl);
            tc::reg_fence(Ac);
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
              const float2 yv =
                  fma2(make_float2(Ac[u], Ac[u + 1]), bc2(hin), make_float2(hl[u], hl[u + 1]));
              const int tl = pp * PT + c16 + u;
              *reinterpret_cast<bf16*>(yb + tl * 64 + lane * 2) = __float2bfloat16_rn(yv.x);
              *reinterpret_cast<bf16*>(yb + (tl + 1) * 64 + lane * 2) = __float2bfloat16_rn(yv.y);
            }
          }
        }
        if (VARLEN && (em0 | em1) != 0u) {
          // the final state of each packed sequence ending in the tile: the float32 y of its
          // last token, taken again from the parked columns (off the loop above: rare)
          static_assert(NPART == 2 && PT == 32, "em0 / em1 are the two parts' tokens");
#pragma unroll
          for (int pp = 0; pp < NPART; ++pp) {
            uint32_t m = pp == 0 ? em0 : em1;
            const float hin = fmaf(Pa[pp], hin_t, Pb[pp]);
            const uint32_t park = tmem + lane_base + a * 128 + pp * PT;
            while (m != 0u) {
              const int u = __ffs(m) - 1;
              m &= m - 1u;
              float hl = tc::tmem_ld1(park + u);
              float Ac = tc::tmem_ld1(park + 64 + u);
              tc::tmem_ld_wait();
              tc::reg_fence(hl);
              tc::reg_fence(Ac);
              const int sidx = __shfl_sync(0xffffffffu, pp == 0 ? e0 : e1, u);
              if (p.hTs && wok) p.hTs[(size_t)sidx * p.W + w] = fmaf(Ac, hin, hl);
            }
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_empty[a]);  // the buffer and its maps are free
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_3d(&tm_y, yb, blk * FUSED_K + q * 32, pc * FUSED_C, pb);
          tc::tma_store_commit();
        }
      }

      // 3. request tile it's look-back slots; they are consumed in the next iteration
      if (it < my_tiles) {
        const int c = cur.c, b = cur.b;
        const LookbackSpan sp = lookback_span(c, p.lb_dist, p.lb_shift);
        lb_n = sp.n;
        lb_agg = c > 0 ? agg + ((size_t)b * p.nC + c - 1) * p.W + w : agg;
        // the anchor's boundary state (the state entering chunk anchor + 1), or h0
        lb_anchor = sp.anchor >= 0 ? carry + ((size_t)b * (p.nC + 1) + sp.anchor + 1) * p.W + w
                                   : nullptr;
        const float h0v = (p.canonical && p.h0) ? p.h0[(size_t)b * p.W + w] : 0.0f;
        lookback_issue(lbq, lb_agg, -(long)p.W, lb_n, lb_anchor, h0v);
#pragma unroll
        for (int pp = 0; pp < NPART; ++pp) Pa[pp] = nPa[pp], Pb[pp] = nPb[pp];
        Ta = nTa;
        Tb = nTb;
        pe0 = ce0;
        pe1 = ce1;
        pc = c;
        pb = b;
        cur.next();
      }
    }
    if (lane == 0) tc::tma_store_wait0();
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t make_maps(const Dims& d, const void* x, const void* Wa, const void* Wx,
                      const void* y, CUtensorMap* mx, CUtensorMap* mwa, CUtensorMap* mwx,
                      CUtensorMap* my) {
  const uint64_t W = d.W, T = d.T, B = d.B;
  const uint64_t dims3[3] = {W, T, B};
  const uint64_t str3[2] = {W * 2, T * W * 2};
  const uint32_t box_x[3] = {16, FUSED_C, 1};
  cudaError_t e = encode_tmap(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims3, str3, box_x,
                              CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  const uint32_t box_y[3] = {32, FUSED_C, 1};  // one output warp's strip
  e = encode_tmap(my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, dims3, str3, box_y,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  // W[nblk][k][k] viewed as [nblk*k rows][k columns]
  const uint64_t dimsw[2] = {(uint64_t)d.k, (uint64_t)d.nblk * d.k};
  const uint64_t strw[1] = {(uint64_t)d.k * 2};
  const uint32_t box_w[2] = {16, FUSED_K};
  e = encode_tmap(mwa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wa, dimsw, strw, box_w,
                  CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  return encode_tmap(mwx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wx, dimsw, strw, box_w,
                     CU_TENSOR_MAP_SWIZZLE_32B);
}

int ctas_per_block(const Dims& d) {
  const int sms = sm_count();
  return sms > 0 ? sms / d.nblk : 0;
}

}  // namespace

int fused_ctas_per_block(const Dims& d) {
  const int p = ctas_per_block(d);
  return p * d.nblk <= FUSED_MAX_CTAS ? p : FUSED_MAX_CTAS / d.nblk;
}

bool fused_supported(const Dims& d) {
  return d.io == RGLRU_BF16 && d.k == FUSED_K && fused_ctas_per_block(d) >= 1;
}

// Prepares a scan layout for slot-based look-back with one zero fill: the status word, any
// counters in the header and every slot (empty reads as zero).
cudaError_t clear_slots(void* buf, const ScanLayout& L, cudaStream_t s) {
  return cudaMemsetAsync(buf, 0, L.part, s);
}

cudaError_t launch_fused_fwd(const Dims& d, const void* x, const void* Wa, const float* ba,
                             const void* Wx, const float* bx, const float* Lambda,
                             const uint8_t* rm, const int32_t* sp, const float* h0, void* y,
                             float* hT, void* saved, int spin_limit, int drop_tile,
                             cudaStream_t s, const Varlen* vl) {
  if (!fused_supported(d)) return cudaErrorNotSupported;
  CUtensorMap mx, mwa, mwx, my;
  cudaError_t e = make_maps(d, x, Wa, Wx, y, &mx, &mwa, &mwx, &my);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.B = d.B;
  p.T = d.T;
  p.W = d.W;
  p.nblk = d.nblk;
  p.nC = fused_chunks(d);
  p.P = fused_ctas_per_block(d);
  p.canonical = d.mode == RGLRU_CANONICAL;
  p.Lambda = Lambda;
  p.ba = ba;
  p.bx = bx;
  p.reset_mask = p.canonical ? rm : nullptr;  // restricted mode has no resets
  p.segment_pos = p.canonical ? sp : nullptr;
  p.h0 = h0;
  p.hT = hT;
  p.seq_start = nullptr;
  p.seq_end = nullptr;
  p.h0s = nullptr;
  p.hTs = nullptr;
  if (vl) {
    const FusedFwdLayout FL = fused_fwd_layout(d);
    p.seq_start = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(saved) + FL.seq_start);
    p.seq_end = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(saved) + FL.seq_end);
    p.h0s = vl->h0;
    p.hTs = vl->hT;
  }
  p.scratch = static_cast<uint8_t*>(saved);
  p.L = fused_layout(d, false);
  p.spin_limit = spin_limit;
  p.drop_tile = drop_tile;
  const LookbackPlan lp = lookback_plan(p.P, d.B);
  p.lb_dist = lp.dist;
  p.lb_shift = lp.shift;
  auto kern = vl ? k_fused_fwd<true, false> : k_fused_fwd<false, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = clear_slots(saved, p.L, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P * d.nblk);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  kernel_event_before(s);
  e = cudaLaunchKernelEx(&cfg, kern, mx, mwa, mwx, my, p);
  kernel_event_after(s);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

int logits_slices(const Dims& d) { return (d.W + FUSED_K - 1) / FUSED_K; }

int logits_ctas_per_slice(const Dims& d) {
  const int sms = sm_count();
  const int n = logits_slices(d);
  if (sms <= 0 || n > sms || n > FUSED_MAX_CTAS) return 0;
  const int p = sms / n;
  return p * n <= FUSED_MAX_CTAS ? p : FUSED_MAX_CTAS / n;
}

bool logits_scan_supported(const Dims& d) {
  return d.io == RGLRU_BF16 && logits_ctas_per_slice(d) >= 1;
}

cudaError_t encode_logit_planes(const Dims& d, const void* base, size_t plane_elems, int nplanes,
                                CUtensorMap* m) {
  const uint64_t W = d.W, T = d.T, B = d.B;
  const uint64_t dims[4] = {W, T, B, (uint64_t)nplanes};
  const uint64_t str[3] = {W * 2, T * W * 2, (uint64_t)plane_elems * 2};
  const uint32_t box[4] = {16, FUSED_C, 1, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, str, box,
                     CU_TENSOR_MAP_SWIZZLE_32B);
}

cudaError_t launch_logits_fwd(const Dims& d, const void* x, const void* lr, const void* li,
                              size_t plane_elems, int nplanes, const float* Lambda,
                              const uint8_t* rm, const int32_t* sp, const float* h0, void* y,
                              float* hT, void* saved, int spin_limit, int drop_tile,
                              cudaStream_t s, const Varlen* vl) {
  if (!logits_scan_supported(d) || nplanes < 1 || nplanes > LG_PLANES)
    return cudaErrorNotSupported;
  const uint64_t W = d.W, T = d.T, B = d.B;
  const uint64_t dims3[3] = {W, T, B};
  const uint64_t str3[2] = {W * 2, T * W * 2};
  const uint32_t box_x[3] = {16, FUSED_C, 1};
  CUtensorMap mx, mlr, mli, my;
  cudaError_t e = encode_tmap(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims3, str3, box_x,
                              CU_TENSOR_MAP_SWIZZLE_32B);
  const uint32_t box_y[3] = {32, FUSED_C, 1};
  if (e == cudaSuccess)
    e = encode_tmap(&my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, dims3, str3, box_y,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess) e = encode_logit_planes(d, lr, plane_elems, nplanes, &mlr);
  if (e == cudaSuccess) e = encode_logit_planes(d, li, plane_elems, nplanes, &mli);
  if (e != cudaSuccess) return e;
  FwdParams p = {};
  p.B = d.B;
  p.T = d.T;
  p.W = d.W;
  p.nblk = logits_slices(d);
  p.nC = fused_chunks(d);
  p.P = logits_ctas_per_slice(d);
  p.canonical = d.mode == RGLRU_CANONICAL;
  p.nplanes = nplanes;
  p.Lambda = Lambda;
  p.ba = nullptr;
  p.bx = nullptr;
  p.reset_mask = p.canonical ? rm : nullptr;
  p.segment_pos = p.canonical ? sp : nullptr;
  p.h0 = h0;
  p.hT = hT;
  if (vl) {
    const FusedFwdLayout FL = fused_fwd_layout(d);
    p.seq_start = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(saved) + FL.seq_start);
    p.seq_end = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(saved) + FL.seq_end);
    p.h0s = vl->h0;
    p.hTs = vl->hT;
  }
  p.scratch = static_cast<uint8_t*>(saved);
  p.L = fused_layout(d, false);
  p.spin_limit = spin_limit;
  p.drop_tile = drop_tile;
  const LookbackPlan lp = lookback_plan(p.P, d.B);
  p.lb_dist = lp.dist;
  p.lb_shift = lp.shift;
  auto kern = vl ? k_fused_fwd<true, true> : k_fused_fwd<false, true>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)LG_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = clear_slots(saved, p.L, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P * p.nblk);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = LG_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mx, mlr, mli, my, p);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace rglru
