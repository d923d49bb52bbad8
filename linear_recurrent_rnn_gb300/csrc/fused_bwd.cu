// Fused RG-LRU backward on one GB300: the gate logits are recomputed on the tcgen05 tensor
// cores, the reverse scan and the pointwise derivatives run on the CUDA cores, and the
// projection gradients dx += dlr Wa^T + dli Wx^T and dW = x^T dl go back to the tensor
// cores, all in one persistent kernel, which also sums the per-CTA partials at its end.
//
// Sources ("Fattori comparison" page): the custom backward runs the reverse recurrence and the
// pointwise derivatives, recomputing the sigmoids, the transition and the multiplier rather
// than saving them; the a_param gradient is reduced over batch and time (done here on device,
// in a fixed order).  The benchmark record checks gradients of x, both gate logits and
// a_param, with the projections inside the measured layer.  Derivatives (loss
// L = sum y dy + sum hT dhT, g_t = dL/dh_t):
//   g_t = dy_t + abar_{t+1} g_{t+1}        (g_{T-1} = dy + dhT)
//   dla = abar g (h_{t-1} - u abar / m)    (u = i x; zero at reset tokens)
//   dlr = dla (-8 softplus) r (1 - r),  dli = g m u (1 - i),  dx_direct = g m i,
//   dsoftplus = sum dla (-8 r),  dLambda = sigmoid(Lambda) dsoftplus,  dh0 = abar_0 g_0.
//
// Tile = (b, blk, 64 tokens), visited in reverse chunk order; two scan threads per channel,
// one per 32-token part.  Per tile:
//   1. MMA: lr^T, li^T = W^T x^T into TMEM (as in the forward).
//   2. Pass 1 (tokens ascending): abar kept in registers, m i and r parked in TMEM over the
//      logits, i beside them; the part's forward aggregate (state map h -> A h + B) and reverse
//      aggregate (carry map c_in -> P c_in + S with P = prod abar, S = sum_t (prod_{s<=t}
//      abar_s) dy_t).
//   3. Parts exchange aggregates through shared memory; part 0 composes the tile's reverse
//      aggregate, publishes it, and runs the anchored look-back toward larger t (lookback.cuh)
//      for the carry from the right (its slots requested at the tile's start and again once the
//      tiles processed alongside have published); the forward entry state comes from the
//      chunk states the forward saved.
//   4. Pass 2: h_{t-1} forward through the part, then g exactly in reverse with the pointwise
//      gradients; dlr, dli go to shared memory as bf16 hi + lo pairs (v = hi + lo to ~2^-16),
//      the direct dx term into the TMEM dx accumulator.
//   5. MMA: dx^T += Wa (dlr_hi + dlr_lo)^T + Wx (dli_hi + dli_lo)^T on top of the direct term;
//      dWa += x^T (dlr_hi + dlr_lo), dWx += x^T (dli_hi + dli_lo) (both in one N = 256
//      product per 16 tokens) accumulated in TMEM over the CTA's tiles.  The lo halves keep both products at float32-like accuracy: dl can be O(1)
//      and a bf16-rounded dl alone would cost ~2^-9 |dl| in dx.
//   6. dx TMEM -> bf16/f32 -> smem -> TMA store, done after pass 1 of the next tile, so the
//      step-5 MMAs run while the scan warps work on that pass.
// Roles: warp 0 TMA (W once; x + dy tiles, 2 stages), warp 1 MMA, warps 2..9 scan.  CTA
// (blk, r) takes tiles r, r + P, ... of its block, so its partial sums cover a fixed set of
// tiles: the result is bitwise reproducible.
#include <cudaTypedefs.h>

#include "host_util.h"
#include "internal.h"
#include "lookback.cuh"
#include "tc.cuh"

namespace rglru {

namespace {

constexpr int NPART = 2;             // token parts of a tile, one scan thread each per channel
constexpr int PT = FUSED_C / NPART;  // tokens per scan thread
constexpr int NSCAN = 4 * NPART;     // scan warps (4 lane quadrants per part)
constexpr int NTHREADS = 64 + NSCAN * 32;
// The warps share the SM's four 16 K-register sub-partitions: registers per thread <= 16384 /
// (32 x warps per sub-partition), rounded down to a multiple of 8.
constexpr int MAXREG = (16384 / (((NSCAN + 2 + 3) / 4) * 32)) / 8 * 8;
constexpr int STAGES = 2;
constexpr uint32_t W_BYTES = FUSED_K * FUSED_K * 2;
constexpr uint32_t T_BYTES = FUSED_C * FUSED_K * 2;  // one 64 x 128 bf16 tile
constexpr uint32_t SLAB_X = FUSED_C * 32;            // 16 channels x 64 tokens
constexpr uint32_t SLAB_W = FUSED_K * 32;            // 16 out-channels x 128 in-rows
constexpr uint32_t SLAB_D = FUSED_K * 32;            // 16 tokens x 128 channels (dl buffers)
// The dl buffers (hi, then lo): per 16-token group the dlr slab, then the dli slab, so that a
// group's 256 rows are one K-major operand of the dW products (N = 256: dWa and dWx at once).
constexpr uint32_t DL_GSTR = 2 * SLAB_D;
constexpr uint32_t DY_ROW = FUSED_K * 2;             // dy tiles: [token][channel], unswizzled
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_LR = 0, COL_LI = 64, COL_DX = 128, COL_HP = 192, COL_DWA = 256,
                   COL_DWX = 384;
static_assert(COL_DWX == COL_DWA + FUSED_K, "the dW products write dWa and dWx as one N = 256");
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s: a pipeline wait never lasts this
constexpr uint32_t XCH_BYTES = NPART * FUSED_K * 16 + FUSED_K * 4;  // part aggregates + carry
// W (2) + x/dy stages (2 x 2) + dl buffers (4) + bf16 dx staging (1) tiles, exchange, barriers
constexpr size_t SMEM_BYTES =
    2 * W_BYTES + STAGES * 2 * T_BYTES + 4 * T_BYTES + T_BYTES + XCH_BYTES + 256 + 1024;
// Given-logits mode (the backward of rglru_backward and of the composed layer): no weights and
// no projection products; each stage holds x, dy and up to two bf16 planes of each logit tile,
// a 64 x 64 identity lays the logits out in TMEM, and dlr / dli go to global memory.
constexpr int LG_PLANES = 2;
constexpr uint32_t LG_STAGE_BYTES = (2 + 2 * LG_PLANES) * T_BYTES;
constexpr uint32_t ID_BYTES = FUSED_C * FUSED_C * 2;
constexpr size_t LG_SMEM_BYTES = ID_BYTES + STAGES * LG_STAGE_BYTES + T_BYTES + XCH_BYTES + 256 + 1024;
// Given-logits output of dlr, dli: LGM_SAME in the dx dtype, LGM_SPLIT as float32 values in
// bf16 hi + lo planes (the operands of the tensor-core projection backward).
constexpr int LGM_NONE = 0, LGM_SAME = 1, LGM_SPLIT = 2;
constexpr uint32_t STATUS_PIPE = 2u;
constexpr int BAR_SCAN = 1;  // named barrier of the scan warps
constexpr uint32_t DW_BOX_BYTES = FUSED_K * 128;  // 128 rows x 32 float32 columns
// Workspace offset of the per-gate-block counters of CTAs done with their partial sums
// (zeroed with the status word before every launch).
constexpr size_t BWD_COUNTERS = 256;

struct BwdParams {
  int B, T, W, nblk, nC, P, canonical;
  int nplanes;     // given logits: bf16 planes per logit
  void* dlr;       // given logits: outputs dlr, dli ([B][T][W]; split: lo plane dl_plane later)
  void* dli;
  size_t dl_plane;
  const float* Lambda;
  const float* ba;
  const float* bx;
  const uint8_t* reset_mask;
  const int32_t* segment_pos;
  const float* dhT;
  const float* fwd_carry;  // [B][nC+1][W], state entering each chunk (slot-encoded)
  // packed variable-length sequences (null seq_start: none); one row
  const int32_t* seq_start;
  const int32_t* seq_end;
  const float* h0s;
  const float* dhTs;
  float* dh0s;
  float* dh0;
  void* dx;                // written directly for float32 gradients
  float* dWa;
  float* dWx;
  float* dba;
  float* dbx;
  float* dLambda;
  uint8_t* scratch;        // workspace
  FusedBwdLayout F;
  int spin_limit, drop_tile;
  int lb_dist, lb_shift;
};

struct Ctl {
  volatile uint32_t* abort;
  uint32_t* status;
  __device__ bool wait(uint64_t* bar, uint32_t parity) const {
    if (*abort) return false;
    if (tc::mbar_wait(bar, parity, WAIT_LIMIT_NS)) return true;
    *abort = 1u;
    atomicOr(status, STATUS_PIPE);
    return false;
  }
};

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi) (v - hi is exact in float32), for two
// values at once; returns the bf16x2 bit patterns of (hi0, hi1) and (lo0, lo1).
__device__ __forceinline__ void split_hi_lo(float2 v, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  const float2 l = fma2(__bfloat1622float2(h), bc2(-1.0f), v);
  const __nv_bfloat162 lb = __floats2bfloat162_rn(l.x, l.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&lb);
}

// Writes 8 consecutive tokens u .. u + 7 of channel j (tu = their first token in the tile, a
// multiple of 8) as hi and lo bf16 parts, 16 bytes each: conflict-free, as the swizzle puts
// rows 4..7 of every 8 in the other half of the bank space.
__device__ __forceinline__ void store_dl8(uint8_t* hi_buf, uint8_t* lo_buf, int tu, int j,
                                          const float2 (&v)[4]) {
  uint4 hi, lo;
  split_hi_lo(v[0], hi.x, lo.x);
  split_hi_lo(v[1], hi.y, lo.y);
  split_hi_lo(v[2], hi.z, lo.z);
  split_hi_lo(v[3], hi.w, lo.w);
  const uint32_t at = (tu >> 4) * DL_GSTR + j * 32 + ((((tu >> 3) & 1) ^ ((j >> 2) & 1)) << 4);
  *reinterpret_cast<uint4*>(hi_buf + at) = hi;
  *reinterpret_cast<uint4*>(lo_buf + at) = lo;
}

// The passes of a scan thread over its part's 32 tokens do the pointwise work on token pairs
// (u, u + 1) in the two lanes of f32x2 operations (adjacent TMEM columns land in adjacent
// registers) and run the recurrences as scalar chains.  Per-token values parked in TMEM sit at
// column = token of the part; the thread's columns of each region start at tcol.
constexpr int GRP = 8;  // tokens per TMEM load / store group

// Pass 1, fast (tokens ascending; every token valid, no reset or packed-sequence boundary,
// every decay in the near regime, a warp-uniform condition): the gates once; abar stays in
// registers, m i -> COL_LR and r -> COL_LI (over the logits, already read), i -> COL_HP;
// returns the part's maps: forward h -> P h + fB and reverse c -> P c + S, with P = prod abar
// and S = sum_t (prod of abar up to t) dy_t.  The other tiles take the general passes below.
// Packed sequences in a part: at a start token (smask) the token continues from its
// sequence's initial state, h -> a h0[s] + m i x, so the recurrences take 0 for its decay while
// the derivatives keep the true a (and dh0[s] = a g); at an end token (emask) dhT[s] joins dy.
struct SeqB {
  const BwdParams& p;  // the sequence arrays (seq_start, seq_end, h0s, dhTs, dh0s)
  uint32_t smask, emask;
  int t0;  // row index of the part's first token (packed sequences: one row)
  int w;   // channel
  bool ok = true;  // the channel is stored (false: a lane past W of a partial slice)
};
__device__ __forceinline__ float seqb_h0(const SeqB& sq, int u) {
  return sq.p.h0s ? sq.p.h0s[(size_t)sq.p.seq_start[sq.t0 + u] * sq.p.W + sq.w] : 0.0f;
}
__device__ __forceinline__ float seqb_dhT(const SeqB& sq, int u) {
  return sq.p.dhTs ? sq.p.dhTs[(size_t)sq.p.seq_end[sq.t0 + u] * sq.p.W + sq.w] : 0.0f;
}
// The chains' decay of a token pair: 0 at sequence starts.
__device__ __forceinline__ float2 chain_decay(const SeqB& sq, int u, float2 a) {
  if ((sq.smask >> u) & 1u) a.x = 0.0f;
  if ((sq.smask >> (u + 1)) & 1u) a.y = 0.0f;
  return a;
}

__device__ __forceinline__ void bwd_pass1(uint32_t tcol, uint32_t xb0, uint32_t xb1, uint32_t dyb,
                                          const GateK& gk, float2 (&ab)[PT / 2],
                                          uint32_t (&xr)[PT / 2], float& P, float& fB, float& S) {
  P = 1.0f;
  fB = 0.0f;
  S = 0.0f;
  // the TMEM loads of group g + 1 are issued before group g is computed
  float vr[GRP], vi[GRP];
  tc::tmem_ld(tcol + COL_LR, vr);
  tc::tmem_ld(tcol + COL_LI, vi);
  tc::tmem_ld_wait();
  tc::reg_fence(vr);
  tc::reg_fence(vi);
#pragma unroll
  for (int g = 0; g < PT / GRP; ++g) {
    float m4[GRP], nr[GRP], ni[GRP];
    if (g + 1 < PT / GRP) {
      tc::tmem_ld(tcol + COL_LR + (g + 1) * GRP, nr);
      tc::tmem_ld(tcol + COL_LI + (g + 1) * GRP, ni);
    }
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;
      xr[u / 2] = tok_raw(xb0, xb1, u) | (tok_raw(xb0, xb1, u + 1) << 16);
      const float2 xv = bf16x2_unpack(xr[u / 2]);
      const float2 dyv =
          make_float2(lds_bf16(dyb + u * DY_ROW), lds_bf16(dyb + (u + 1) * DY_ROW));
      float2 abar, mi, r, i;
      gates_near2_i(make_float2(vr[2 * q], vr[2 * q + 1]), make_float2(vi[2 * q], vi[2 * q + 1]),
                    gk, abar, mi, r, i);
      const float2 bv = mul2(mi, xv);
      fB = fmaf(abar.x, fB, bv.x);
      P *= abar.x;
      S = fmaf(P, dyv.x, S);
      fB = fmaf(abar.y, fB, bv.y);
      P *= abar.y;
      S = fmaf(P, dyv.y, S);
      ab[u / 2] = abar;
      m4[2 * q] = mi.x;
      m4[2 * q + 1] = mi.y;
      vr[2 * q] = r.x;  // the logits are consumed: their registers take r and i
      vr[2 * q + 1] = r.y;
      vi[2 * q] = i.x;
      vi[2 * q + 1] = i.y;
    }
    tc::tmem_st(tcol + COL_LR + g * GRP, m4);
    tc::tmem_st(tcol + COL_LI + g * GRP, vr);
    tc::tmem_st(tcol + COL_HP + g * GRP, vi);
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

// Pass 2a, fast (tokens ascending): h_{t-1} of every token from the state h entering the part,
// parked in the dx columns (free once the previous tile's dx has been written out).
__device__ __forceinline__ void bwd_pass2a(uint32_t tcol, const uint32_t (&xr)[PT / 2],
                                           const float2 (&ab)[PT / 2], float h) {
  float m4[GRP];
  tc::tmem_ld(tcol + COL_LR, m4);
  tc::tmem_ld_wait();
  tc::reg_fence(m4);
#pragma unroll
  for (int g = 0; g < PT / GRP; ++g) {
    float h4[GRP], nm[GRP];
    if (g + 1 < PT / GRP) tc::tmem_ld(tcol + COL_LR + (g + 1) * GRP, nm);
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;
      const float2 xv = bf16x2_unpack(xr[u / 2]);
      const float2 bv = mul2(make_float2(m4[2 * q], m4[2 * q + 1]), xv);
      h4[2 * q] = h;
      h = fmaf(ab[u / 2].x, h, bv.x);
      h4[2 * q + 1] = h;
      h = fmaf(ab[u / 2].y, h, bv.y);
    }
    tc::tmem_st(tcol + COL_DX + g * GRP, h4);
    if (g + 1 < PT / GRP) {
      tc::tmem_ld_wait();
      tc::reg_fence(nm);
#pragma unroll
      for (int u = 0; u < GRP; ++u) m4[u] = nm[u];
    }
  }
  tc::tmem_st_wait();
}

// Pass 2b (tokens descending): g exactly from the carry `cin` entering the part's last token
// from the right, and the pointwise gradients; dlr, dli go to the dl operand buffers as bf16
// hi + lo pairs, the direct dx term g m i over h_{t-1} in the dx columns (the accumulator of
// the dx MMAs).  dsp sums dla r (the softplus gradient is -8 times the total).  The logits
// columns (COL_LR, COL_LI) are read for the last time by the loads of group 0; once those have
// landed the warp arrives on lg_free, so the next tile's logits MMAs overlap the rest of the
// pass.
// Given-logits output of one token pair of dlr / dli: token index t0 (row b) of channel w.
template <typename GT, int LGM>
__device__ __forceinline__ void store_dl_pair(void* base, size_t plane, size_t idx, int W,
                                              float2 v, bool ok0, bool ok1) {
  if (LGM == LGM_SPLIT) {
    bf16* p = static_cast<bf16*>(base) + idx;
    const bf16 h0 = __float2bfloat16_rn(v.x), h1 = __float2bfloat16_rn(v.y);
    if (ok0) {
      p[0] = h0;
      p[plane] = __float2bfloat16_rn(v.x - __bfloat162float(h0));
    }
    if (ok1) {
      p[W] = h1;
      p[plane + W] = __float2bfloat16_rn(v.y - __bfloat162float(h1));
    }
  } else {
    GT* p = static_cast<GT*>(base) + idx;
    if (ok0) p[0] = from_f32<GT>(v.x);
    if (ok1) p[W] = from_f32<GT>(v.y);
  }
}
struct DlOut {
  void* dlr;
  void* dli;
  size_t plane;
  size_t idx0;  // element index of (b, the part's first token, w)
  int W;
  int valid;    // tokens of the part before T (and a real channel: else 0)
};

template <typename GT = float, int LGM = LGM_NONE>
__device__ __forceinline__ void bwd_pass2b(uint32_t tcol, int tb, int j,
                                           const uint32_t (&xr)[PT / 2], uint32_t dyb, float nk,
                                           const float2 (&ab)[PT / 2], float cin,
                                           uint64_t* lg_free, uint8_t* s_dl, float2& dsp,
                                           float2& dba, float2& dbx, const DlOut& dlo = DlOut{}) {
  static_assert(PT / GRP >= 2, "the logits columns are released after the second-to-last group");
  float gnext = cin, anext = 1.0f;
  constexpr int G0 = PT / GRP - 1;
  float m4[GRP], r4[GRP], i4[GRP], h4[GRP];
  tc::tmem_ld(tcol + COL_LR + G0 * GRP, m4);
  tc::tmem_ld(tcol + COL_LI + G0 * GRP, r4);
  tc::tmem_ld(tcol + COL_HP + G0 * GRP, i4);
  tc::tmem_ld(tcol + COL_DX + G0 * GRP, h4);
  tc::tmem_ld_wait();
  tc::reg_fence(m4);
  tc::reg_fence(r4);
  tc::reg_fence(i4);
  tc::reg_fence(h4);
#pragma unroll
  for (int g = G0; g >= 0; --g) {
    float nm[GRP], nr[GRP], ni[GRP], nh[GRP];
    if (g > 0) {
      tc::tmem_ld(tcol + COL_LR + (g - 1) * GRP, nm);
      tc::tmem_ld(tcol + COL_LI + (g - 1) * GRP, nr);
      tc::tmem_ld(tcol + COL_HP + (g - 1) * GRP, ni);
      tc::tmem_ld(tcol + COL_DX + (g - 1) * GRP, nh);
    }
    float2 o_r[GRP / 2], o_i[GRP / 2];  // tokens (u, u + 1) of the two pairs
#pragma unroll
    for (int q = GRP / 2 - 1; q >= 0; --q) {
      const int u = g * GRP + 2 * q;
      const float2 xv = bf16x2_unpack(xr[u / 2]);
      const float2 dyv =
          make_float2(lds_bf16(dyb + u * DY_ROW), lds_bf16(dyb + (u + 1) * DY_ROW));
      const float2 abar = ab[u / 2];
      const float2 mi = make_float2(m4[2 * q], m4[2 * q + 1]);
      const float2 r = make_float2(r4[2 * q], r4[2 * q + 1]);
      const float2 i = make_float2(i4[2 * q], i4[2 * q + 1]);
      float2 gv;
      gv.y = fmaf(anext, gnext, dyv.y);
      gv.x = fmaf(abar.y, gv.y, dyv.x);
      gnext = gv.x;
      anext = abar.x;
      // d h_t / d la = abar (h_{t-1} - abar x i / m) with i / m = i^2 / (m i) (m i > 0 on the
      // fast path)
      const float2 nw = mul2(mul2(i, i), make_float2(rcp_approx(-mi.x), rcp_approx(-mi.y)));
      const float2 alpha =
          mul2(abar, fma2(mul2(abar, xv), nw, make_float2(h4[2 * q], h4[2 * q + 1])));
      const float2 dla = mul2(gv, alpha);
      const float2 dd = mul2(gv, mi);  // direct dx term
      o_r[q] = mul2(mul2(dla, bc2(nk)), mul2(r, fma2(r, bc2(-1.0f), bc2(1.0f))));
      o_i[q] = mul2(mul2(dd, xv), fma2(i, bc2(-1.0f), bc2(1.0f)));
      dsp = fma2(dla, r, dsp);
      dba = add2(dba, o_r[q]);
      dbx = add2(dbx, o_i[q]);
      h4[2 * q] = dd.x;
      h4[2 * q + 1] = dd.y;
    }
    static_assert(GRP == 8, "the dl stores take 8 tokens");
    if (LGM == LGM_NONE) {
      store_dl8(s_dl, s_dl + 2 * T_BYTES, tb + g * GRP, j, o_r);
      store_dl8(s_dl + SLAB_D, s_dl + 2 * T_BYTES + SLAB_D, tb + g * GRP, j, o_i);
    } else {
#pragma unroll
      for (int q = 0; q < GRP / 2; ++q) {
        const int u = g * GRP + 2 * q;
        const size_t idx = dlo.idx0 + (size_t)u * dlo.W;
        store_dl_pair<GT, LGM>(dlo.dlr, dlo.plane, idx, dlo.W, o_r[q], u < dlo.valid,
                               u + 1 < dlo.valid);
        store_dl_pair<GT, LGM>(dlo.dli, dlo.plane, idx, dlo.W, o_i[q], u < dlo.valid,
                               u + 1 < dlo.valid);
      }
    }
    tc::tmem_st(tcol + COL_DX + g * GRP, h4);
    if (g > 0) {
      tc::tmem_ld_wait();
      tc::reg_fence(nm);
      tc::reg_fence(nr);
      tc::reg_fence(ni);
      tc::reg_fence(nh);
#pragma unroll
      for (int u = 0; u < GRP; ++u) {
        m4[u] = nm[u];
        r4[u] = nr[u];
        i4[u] = ni[u];
        h4[u] = nh[u];
      }
      if (g == 1) {  // every read of the logits columns has landed
        tc::tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(lg_free);
      }
    }
  }
  tc::tmem_st_wait();
}

// The general passes: tiles with a reset, a packed-sequence start or end, tokens past T or a
// channel outside the near regime, a few tiles a launch.  They walk the part's token groups in
// a loop (not unrolled) and keep no per-token registers across passes: x comes from the
// staged tile and the decay is recomputed from the parked r (bitwise as pass 1 computed it),
// so their code stays small and leaves the fast passes' code compact (inlined fully unrolled,
// the packed-sequence variants alone slowed every tile of their kernel by a quarter).
// The decay of a token pair from its r, as gates_any2 computes it, then the token masks:
// 0 at a reset, 1 past T.
__device__ __forceinline__ float2 gen_decay(float2 r, const GateK& k, uint32_t rmask, int u,
                                            int valid) {
  const float2 la = mul2(bc2(k.nk), r);
  float2 p = fma2(la, bc2(DECAY_P3), bc2(DECAY_P2));
  p = fma2(la, p, bc2(DECAY_P1));
  p = fma2(la, p, bc2(1.0f));
  float2 a = fma2(la, p, bc2(1.0f));
  if (!(la.x > NEAR_LA)) a.x = ex2_approx(la.x * LOG2E);
  if (!(la.y > NEAR_LA)) a.y = ex2_approx(la.y * LOG2E);
  if ((rmask >> u) & 1u) a.x = 0.0f;
  if ((rmask >> (u + 1)) & 1u) a.y = 0.0f;
  if (u >= valid) a.x = 1.0f;
  if (u + 1 >= valid) a.y = 1.0f;
  return a;
}

// General pass 1: as the fast one (gates once, m i / r / i parked, the part's maps), with the
// token masks and packed-sequence starts and ends.
template <bool VARLEN>
__device__ __forceinline__ void bwd_pass1_gen(uint32_t tcol, uint32_t xb0, uint32_t xb1,
                                              uint32_t dyb, const GateK& gk, uint32_t rmask,
                                              int valid, const SeqB& sq, float& P, float& fB,
                                              float& S) {
  P = 1.0f;
  fB = 0.0f;
  S = 0.0f;
#pragma unroll 1
  for (int g = 0; g < PT / GRP; ++g) {
    float vr[GRP], vi[GRP], m4[GRP];
    tc::tmem_ld(tcol + COL_LR + g * GRP, vr);
    tc::tmem_ld(tcol + COL_LI + g * GRP, vi);
    tc::tmem_ld_wait();
    tc::reg_fence(vr);
    tc::reg_fence(vi);
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;
      const float2 xv =
          bf16x2_unpack(tok_raw(xb0, xb1, u) | (tok_raw(xb0, xb1, u + 1) << 16));
      float2 dyv = make_float2(lds_bf16(dyb + u * DY_ROW), lds_bf16(dyb + (u + 1) * DY_ROW));
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
        dyv.x = 0.0f;
      }
      if (u + 1 >= valid) {
        abar.y = 1.0f;
        mi.y = 0.0f;
        dyv.y = 0.0f;
      }
      float2 bv = mul2(mi, xv);
      float2 ach = abar;  // the chains' decay
      if (VARLEN && (sq.smask | sq.emask)) {
        if ((sq.smask >> u) & 1u) bv.x = fmaf(abar.x, seqb_h0(sq, u), bv.x);
        if ((sq.smask >> (u + 1)) & 1u) bv.y = fmaf(abar.y, seqb_h0(sq, u + 1), bv.y);
        ach = chain_decay(sq, u, abar);
        if ((sq.emask >> u) & 1u) dyv.x += seqb_dhT(sq, u);
        if ((sq.emask >> (u + 1)) & 1u) dyv.y += seqb_dhT(sq, u + 1);
      }
      fB = fmaf(ach.x, fB, bv.x);
      P *= ach.x;
      S = fmaf(P, dyv.x, S);
      fB = fmaf(ach.y, fB, bv.y);
      P *= ach.y;
      S = fmaf(P, dyv.y, S);
      m4[2 * q] = mi.x;
      m4[2 * q + 1] = mi.y;
      vr[2 * q] = r.x;
      vr[2 * q + 1] = r.y;
      vi[2 * q] = i.x;
      vi[2 * q + 1] = i.y;
    }
    tc::tmem_st(tcol + COL_LR + g * GRP, m4);
    tc::tmem_st(tcol + COL_LI + g * GRP, vr);
    tc::tmem_st(tcol + COL_HP + g * GRP, vi);
  }
  tc::tmem_st_wait();
}

// General pass 2a: h_{t-1} of every token, from the decay recomputed from r.
template <bool VARLEN>
__device__ __forceinline__ void bwd_pass2a_gen(uint32_t tcol, uint32_t xb0, uint32_t xb1,
                                               const GateK& gk, uint32_t rmask, int valid,
                                               const SeqB& sq, float h) {
#pragma unroll 1
  for (int g = 0; g < PT / GRP; ++g) {
    float m4[GRP], r4[GRP], h4[GRP];
    tc::tmem_ld(tcol + COL_LR + g * GRP, m4);
    tc::tmem_ld(tcol + COL_LI + g * GRP, r4);
    tc::tmem_ld_wait();
    tc::reg_fence(m4);
    tc::reg_fence(r4);
#pragma unroll
    for (int q = 0; q < GRP / 2; ++q) {
      const int u = g * GRP + 2 * q;
      const float2 xv =
          bf16x2_unpack(tok_raw(xb0, xb1, u) | (tok_raw(xb0, xb1, u + 1) << 16));
      const float2 ab = gen_decay(make_float2(r4[2 * q], r4[2 * q + 1]), gk, rmask, u, valid);
      const float2 bv = mul2(make_float2(m4[2 * q], m4[2 * q + 1]), xv);
      // at a sequence start the state before the token is the sequence's initial state
      if (VARLEN && ((sq.smask >> u) & 1u)) h = seqb_h0(sq, u);
      h4[2 * q] = h;
      h = fmaf(ab.x, h, bv.x);
      if (VARLEN && ((sq.smask >> (u + 1)) & 1u)) h = seqb_h0(sq, u + 1);
      h4[2 * q + 1] = h;
      h = fmaf(ab.y, h, bv.y);
    }
    tc::tmem_st(tcol + COL_DX + g * GRP, h4);
  }
  tc::tmem_st_wait();
}

// General pass 2b: as the fast one, the decay recomputed from r, with the token masks and the
// packed-sequence ends (dy += dhT) and starts (dh0 = a g).
template <bool VARLEN, typename GT, int LGM>
__device__ __forceinline__ void bwd_pass2b_gen(uint32_t tcol, int tb, int j, uint32_t xb0,
                                               uint32_t xb1, uint32_t dyb, const GateK& gk,
                                               uint32_t rmask, int valid, const SeqB& sq,
                                               float cin, uint64_t* lg_free, uint8_t* s_dl,
                                               float2& dsp, float2& dba, float2& dbx,
                                               const DlOut& dlo) {
  float gnext = cin, anext = 1.0f;
#pragma unroll 1
  for (int g = PT / GRP - 1; g >= 0; --g) {
    float m4[GRP], r4[GRP], i4[GRP], h4[GRP];
    tc::tmem_ld(tcol + COL_LR + g * GRP, m4);
    tc::tmem_ld(tcol + COL_LI + g * GRP, r4);
    tc::tmem_ld(tcol + COL_HP + g * GRP, i4);
    tc::tmem_ld(tcol + COL_DX + g * GRP, h4);
    tc::tmem_ld_wait();
    tc::reg_fence(m4);
    tc::reg_fence(r4);
    tc::reg_fence(i4);
    tc::reg_fence(h4);
    if (g == 0) {  // every read of the logits columns has landed
      tc::tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) tc::mbar_arrive(lg_free);
    }
    float2 o_r[GRP / 2], o_i[GRP / 2];
#pragma unroll
    for (int q = GRP / 2 - 1; q >= 0; --q) {
      const int u = g * GRP + 2 * q;
      const float2 xv =
          bf16x2_unpack(tok_raw(xb0, xb1, u) | (tok_raw(xb0, xb1, u + 1) << 16));
      float2 dyv = make_float2(lds_bf16(dyb + u * DY_ROW), lds_bf16(dyb + (u + 1) * DY_ROW));
      if (VARLEN) {
        if ((sq.emask >> u) & 1u) dyv.x += seqb_dhT(sq, u);
        if ((sq.emask >> (u + 1)) & 1u) dyv.y += seqb_dhT(sq, u + 1);
      }
      if (u >= valid) dyv.x = 0.0f;
      if (u + 1 >= valid) dyv.y = 0.0f;
      const float2 r = make_float2(r4[2 * q], r4[2 * q + 1]);
      const float2 abar = gen_decay(r, gk, rmask, u, valid);
      const float2 ach = VARLEN ? chain_decay(sq, u, abar) : abar;  // 0 at starts
      const float2 mi = make_float2(m4[2 * q], m4[2 * q + 1]);
      const float2 i = make_float2(i4[2 * q], i4[2 * q + 1]);
      float2 gv;
      gv.y = fmaf(anext, gnext, dyv.y);
      gv.x = fmaf(ach.y, gv.y, dyv.x);
      gnext = gv.x;
      anext = ach.x;
      if (VARLEN && sq.p.dh0s) {  // d h0[s] = a g at the sequence's first token
        float* dh0 = sq.p.dh0s + sq.w;
        const int32_t* st = sq.p.seq_start + sq.t0;
        if (((sq.smask >> u) & 1u) && sq.ok) dh0[(size_t)st[u] * sq.p.W] = abar.x * gv.x;
        if (((sq.smask >> (u + 1)) & 1u) && sq.ok) dh0[(size_t)st[u + 1] * sq.p.W] = abar.y * gv.y;
      }
      const float2 nw = mul2(mul2(i, i), make_float2(rcp_approx(-mi.x), rcp_approx(-mi.y)));
      float2 alpha = mul2(abar, fma2(mul2(abar, xv), nw, make_float2(h4[2 * q], h4[2 * q + 1])));
      if (abar.x == 0.0f || mi.x == 0.0f) alpha.x = 0.0f;
      if (abar.y == 0.0f || mi.y == 0.0f) alpha.y = 0.0f;
      const float2 dla = mul2(gv, alpha);
      const float2 dd = mul2(gv, mi);  // direct dx term
      o_r[q] = mul2(mul2(dla, bc2(gk.nk)), mul2(r, fma2(r, bc2(-1.0f), bc2(1.0f))));
      o_i[q] = mul2(mul2(dd, xv), fma2(i, bc2(-1.0f), bc2(1.0f)));
      dsp = fma2(dla, r, dsp);
      dba = add2(dba, o_r[q]);
      dbx = add2(dbx, o_i[q]);
      h4[2 * q] = dd.x;
      h4[2 * q + 1] = dd.y;
    }
    if (LGM == LGM_NONE) {
      store_dl8(s_dl, s_dl + 2 * T_BYTES, tb + g * GRP, j, o_r);
      store_dl8(s_dl + SLAB_D, s_dl + 2 * T_BYTES + SLAB_D, tb + g * GRP, j, o_i);
    } else {
#pragma unroll
      for (int q = 0; q < GRP / 2; ++q) {
        const int u = g * GRP + 2 * q;
        const size_t idx = dlo.idx0 + (size_t)u * dlo.W;
        store_dl_pair<GT, LGM>(dlo.dlr, dlo.plane, idx, dlo.W, o_r[q], u < dlo.valid,
                               u + 1 < dlo.valid);
        store_dl_pair<GT, LGM>(dlo.dli, dlo.plane, idx, dlo.W, o_i[q], u < dlo.valid,
                               u + 1 < dlo.valid);
      }
    }
    tc::tmem_st(tcol + COL_DX + g * GRP, h4);
  }
  tc::tmem_st_wait();
}

template <typename GT, bool VARLEN, int LGM>
__global__ void __maxnreg__(MAXREG)
    k_fused_bwd(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                const __grid_constant__ CUtensorMap tm_wa, const __grid_constant__ CUtensorMap tm_wx,
                const __grid_constant__ CUtensorMap tm_dx,
                const __grid_constant__ CUtensorMap tm_dwp, const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by pointer arithmetic so that it stays a shared pointer
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr bool LG = LGM != LGM_NONE;
  constexpr uint32_t STB = LG ? LG_STAGE_BYTES : 2 * T_BYTES;
  uint8_t* s_wa = smem;                             // LG: the identity
  uint8_t* s_wx = smem + W_BYTES;
  uint8_t* s_in = smem + (LG ? ID_BYTES : 2 * W_BYTES);  // stage s: x, dy (+ LG: logit planes)
  uint8_t* s_dl = s_in + STAGES * STB;              // dl hi, dl lo (none in LG)
  uint8_t* s_dx = s_dl + (LG ? 0 : 4 * T_BYTES);    // dx staging [token][channel]
  float4* s_agg = reinterpret_cast<float4*>(s_dx + T_BYTES);       // [part][k]
  float* s_cin = reinterpret_cast<float*>(s_agg + NPART * FUSED_K);  // [k]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_cin + FUSED_K);
  uint64_t* w_full = bars;
  uint64_t* in_full = bars + 1;
  uint64_t* in_empty = bars + 1 + STAGES;
  uint64_t* lg_full = bars + 1 + 2 * STAGES;
  uint64_t* lg_empty = lg_full + 1;
  uint64_t* dl_full = lg_full + 2;
  uint64_t* dl_empty = lg_full + 3;
  uint64_t* dx_full = lg_full + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(lg_full + 5);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x / p.P, rr = blockIdx.x % p.P;
  const int ntiles = p.B * p.nC;
  uint32_t* status = reinterpret_cast<uint32_t*>(p.scratch);
  const Ctl ctl{abort_flag, status};

  if (threadIdx.x == 0) {
    tc::mbar_init(w_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&in_full[s], 1);
      tc::mbar_init(&in_empty[s], NSCAN + 1);  // scan warps + the dW MMAs
    }
    tc::mbar_init(lg_full, 1);
    tc::mbar_init(lg_empty, NSCAN);
    tc::mbar_init(dl_full, NSCAN);
    tc::mbar_init(dl_empty, 1);
    tc::mbar_init(dx_full, 1);
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
      tc::prefetch_tmap(&tm_dy);
      if (!LG) {
        tc::mbar_expect_tx(w_full, 2 * W_BYTES);
        for (int g = 0; g < FUSED_K / 16; ++g) {
          tc::tma_load_2d(s_wa + g * SLAB_W, &tm_wa, w_full, 16 * g, blk * FUSED_K);
          tc::tma_load_2d(s_wx + g * SLAB_W, &tm_wx, w_full, 16 * g, blk * FUSED_K);
        }
      } else {
        tc::mbar_arrive(w_full);  // the identity is in place (written before the CTA barrier)
      }
      TileWalk tw(rr, p.P, p.B);  // tw.c counts chunks from the last one
      for (int it = 0; it < my_tiles; ++it, tw.next()) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!ctl.wait(&in_empty[st], ph ^ 1u)) continue;
        const int c = p.nC - 1 - tw.c, b = tw.b;
        uint8_t* xs = s_in + st * STB;
        tc::mbar_expect_tx(&in_full[st], LG ? (2 + 2 * p.nplanes) * T_BYTES : 2 * T_BYTES);
        for (int s = 0; s < FUSED_K / 16; ++s)
          tc::tma_load_3d(xs + s * SLAB_X, &tm_x, &in_full[st], blk * FUSED_K + 16 * s,
                          c * FUSED_C, b);
        tc::tma_load_3d(xs + T_BYTES, &tm_dy, &in_full[st], blk * FUSED_K, c * FUSED_C, b);
        if (LG) {  // tm_wa / tm_wx map the logit planes [plane][B][T][W]
          for (int g = 0; g < 2; ++g)
            for (int pl = 0; pl < p.nplanes; ++pl)
              for (int s = 0; s < FUSED_K / 16; ++s)
                tc::tma_load_4d(xs + (2 + g * LG_PLANES + pl) * T_BYTES + s * SLAB_X,
                                g ? &tm_wx : &tm_wa, &in_full[st], blk * FUSED_K + 16 * s,
                                c * FUSED_C, b, pl);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (the descriptor arithmetic stays warp-uniform); one elected
    // lane issues the MMAs and commits.
    const bool leader = tc::elect_one();
    constexpr uint32_t id_lg = tc::idesc_bf16(128, FUSED_C, 1, 0);  // W^T x^T
    constexpr uint32_t id_dx = tc::idesc_bf16(128, FUSED_C, 0, 1);  // W dl^T
    constexpr uint32_t id_dw = tc::idesc_bf16(128, 2 * FUSED_K, 1, 0);  // x^T [dlr dli]
    ctl.wait(w_full, 0);
    const uint32_t wa = tc::smem_u32(s_wa), wx = tc::smem_u32(s_wx);
    const uint32_t dl0 = tc::smem_u32(s_dl);
    auto logits = [&](int it) {
      const int st = it % STAGES;
      if (!ctl.wait(lg_empty, (it & 1) ^ 1u)) return;
      if (!ctl.wait(&in_full[st], (it / STAGES) & 1)) return;
      tc::tc_fence_after();
      const uint32_t xs = tc::smem_u32(s_in + st * STB);
      if (leader) {
        if (!LG) {
#pragma unroll
          for (int kk = 0; kk < FUSED_K / 16; ++kk) {
            const uint64_t bdesc = tc::smem_desc_sw32(xs + kk * SLAB_X, 16, 256);
            tc::mma_bf16(tmem + COL_LR, tc::smem_desc_sw32(wa + kk * 512, SLAB_W, 256), bdesc,
                         id_lg, kk > 0);
            tc::mma_bf16(tmem + COL_LI, tc::smem_desc_sw32(wx + kk * 512, SLAB_W, 256), bdesc,
                         id_lg, kk > 0);
          }
        } else {
          // l^T = L^T I: A = the logit plane tile MN-major, B = the identity K-major
          for (int g = 0; g < 2; ++g)
            for (int pl = 0; pl < p.nplanes; ++pl)
#pragma unroll
              for (int kk = 0; kk < FUSED_C / 16; ++kk)
                tc::mma_bf16(tmem + (g ? COL_LI : COL_LR),
                             tc::smem_desc_sw32(xs + (2 + g * LG_PLANES + pl) * T_BYTES + kk * 512,
                                                SLAB_X, 256),
                             tc::smem_desc_sw32(wa + kk * SLAB_X, 16, 256), id_lg,
                             (pl > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(lg_full);
        if (LG) tc::mma_commit(&in_empty[st]);  // the logit planes are read
      }
      __syncwarp();
    };
    if (LG) {
      for (int it = 0; it < my_tiles; ++it) logits(it);
    }
    if (!LG && my_tiles > 0) logits(0);
    for (int it = 0; it < my_tiles && !LG; ++it) {
      if (it + 1 < my_tiles) logits(it + 1);
      const int st = it % STAGES;
      if (!ctl.wait(dl_full, it & 1)) continue;
      tc::tc_fence_after();
      if (leader) {
        // dx^T[in][tok] += W[in][out] dl^T[out][tok]: A = W K-major (one 16-column slab per K
        // step), B = dl buffer MN-major (16-token groups 8 KB apart, 8-row groups 256 B).
#pragma unroll
        for (int kk = 0; kk < FUSED_K / 16; ++kk) {
          const uint64_t a_a = tc::smem_desc_sw32(wa + kk * SLAB_W, 16, 256);
          const uint64_t a_x = tc::smem_desc_sw32(wx + kk * SLAB_W, 16, 256);
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // hi, then lo halves of dl
            tc::mma_bf16(tmem + COL_DX, a_a,
                         tc::smem_desc_sw32(dl0 + 2 * h * T_BYTES + kk * 512, DL_GSTR, 256),
                         id_dx, 1);
            tc::mma_bf16(tmem + COL_DX, a_x,
                         tc::smem_desc_sw32(dl0 + 2 * h * T_BYTES + SLAB_D + kk * 512, DL_GSTR,
                                            256),
                         id_dx, 1);
          }
        }
        tc::mma_commit(dx_full);
        // [dWa dWx][in][out] += x^T[in][tok] [dlr dli][tok][out]: A = x tile MN-major
        // (16-channel slabs 2 KB apart), B = a 16-token group of the dl buffer K-major (dlr
        // rows, then dli rows), D = the 256 columns of dWa and dWx.
        const uint32_t xs = tc::smem_u32(s_in + st * 2 * T_BYTES);
#pragma unroll
        for (int kk = 0; kk < FUSED_C / 16; ++kk) {
          const uint64_t adesc = tc::smem_desc_sw32(xs + kk * 512, SLAB_X, 256);
          const uint32_t acc0 = (it > 0 || kk > 0) ? 1u : 0u;
          tc::mma_bf16(tmem + COL_DWA, adesc,
                       tc::smem_desc_sw32(dl0 + kk * DL_GSTR, 16, 256), id_dw, acc0);
          tc::mma_bf16(tmem + COL_DWA, adesc,
                       tc::smem_desc_sw32(dl0 + 2 * T_BYTES + kk * DL_GSTR, 16, 256), id_dw, 1);
        }
        tc::mma_commit(dl_empty);
        tc::mma_commit(&in_empty[st]);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ scan warps
    const int part = (warp - 2) >> 2;
    const int q = warp & 3;
    const int j = q * 32 + lane;
    // channels past W (LG only): nothing stored, their reads take a real channel's
    const bool wok = !LG || blk * FUSED_K + j < p.W;
    const int w = LG ? min(blk * FUSED_K + j, p.W - 1) : blk * FUSED_K + j;
    const int tb = part * PT;
    const uint32_t tcol = tmem + ((uint32_t)(q * 32) << 16) + tb;  // this thread's lane, part
    GateK gk;
    gk.nk = -8.0f * softplus_f(p.Lambda[w]);  // log a = nk * r
    gk.cm = sqrtf(-2.0f * gk.nk);
    gk.nbr = p.ba ? -p.ba[w] * LOG2E : 0.0f;  // biases folded into the exponents
    gk.nbi = p.bx ? -p.bx[w] * LOG2E : 0.0f;
    float* rcar = reinterpret_cast<float*>(p.scratch + p.F.L.carry);
    float2* agg = reinterpret_cast<float2*>(p.scratch + p.F.L.agg);
    const bool store_thread = (warp == 2 && lane == 0);
    if (store_thread) tc::prefetch_tmap(&tm_dx);
    float2 dsp = bc2(0.0f), dba = bc2(0.0f), dbx = bc2(0.0f);
    // The fast path needs every channel of the warp in the near regime and with a nonzero
    // multiplier constant: then m i > 0 on every token (the exponent clamps keep t > 0), so its
    // pass 2b needs no test for m = 0.
    const bool near_all = __all_sync(0xffffffffu, gk.nk > NEAR_LA && gk.cm > 0.0f);
    // Channel j of a token row in a stage: 16-channel slab, 2-byte column, and the 16-byte half
    // of the 32-byte row (swapped on rows 4..7 of every 8 by the swizzle).
    const int xoff0 = (j >> 4) * SLAB_X + (j & 7) * 2 + (((j & 15) >> 3) << 4);
    const int xoff1 = (j >> 4) * SLAB_X + (j & 7) * 2 + ((((j & 15) >> 3) ^ 1) << 4);

    // Software pipeline: iteration `it` runs pass 1 of tile it, then writes out the dx of tile
    // it - 1 (whose MMAs ran on the tensor cores during that pass 1), then the rest of tile it.
    // The last iteration only writes out the dx of the last tile.
    TileWalk cur(rr, p.P, p.B);  // tile it; cur.c counts chunks from the last one
    int pc = 0, pb = 0;          // chunk and row of tile it - 1
    // this lane's token markers of a tile (one token of the part each)
    const int32_t* seq_start = VARLEN ? p.seq_start : nullptr;
    const int32_t* seq_end = VARLEN ? p.seq_end : nullptr;
    auto marks = [&](const TileWalk& tw) {
      const int t = (p.nC - 1 - tw.c) * FUSED_C + tb + lane;
      return tok_marks_load(p.reset_mask, p.segment_pos, seq_start, seq_end,
                            (size_t)tw.b * p.T + t, t < p.T);
    };
    // The packed-sequence view of tile (b, c) for the general passes, built where it is used
    // so that its pointers are not live across the tile.
    auto seqb = [&](uint32_t sm, uint32_t em, int b_, int c_) {
      return SeqB{p, sm, em, b_ * p.T + c_ * FUSED_C + tb, w, wok};
    };
    for (int it = 0; it <= my_tiles; ++it) {
      const bool have = it < my_tiles;
      const int n = rr + it * p.P;
      const int c = p.nC - 1 - cur.c, b = cur.b;
      const int st = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      const uint32_t xt = tc::smem_u32(s_in + st * STB + tb * 32);
      const uint32_t xb0 = xt + xoff0, xb1 = xt + xoff1;
      const uint32_t dyb = tc::smem_u32(s_in + st * STB + T_BYTES + tb * DY_ROW + j * 2);
      float2 ab[PT / 2];
      uint32_t xr[PT / 2];  // x of the part's tokens, bf16 pairs
      float P = 1.0f, fB = 0.0f, S = 0.0f;
      float hin_tile = 0.0f;
      int valid = 0;
      bool fast = false;
      uint32_t rmask = 0, smask = 0, emask = 0;
      // Part 0 requests the look-back slots of this tile's carry from the right now; they are
      // read after pass 2a, so the L2 round trip hides behind passes 1 and 2a.
      const size_t cidx = (size_t)b * p.nC + c;
      LookbackReq lbq;
      int lb_n = 0;
      const float2* lb_agg = agg;
      const float* lb_anchor = nullptr;
      if (have && part == 0) {
        // chunks counted from the last one; the anchor passes on its carry to the left
        const LookbackSpan sp = lookback_span(p.nC - 1 - c, p.lb_dist, p.lb_shift);
        lb_n = sp.n;
        if (c < p.nC - 1) lb_agg = agg + (cidx + 1) * p.W + w;
        if (sp.anchor >= 0) lb_anchor = rcar + ((size_t)b * p.nC + (p.nC - 1 - sp.anchor)) * p.W + w;
        lookback_issue(lbq, lb_agg, (long)p.W, lb_n, lb_anchor,
                       p.dhT ? p.dhT[(size_t)b * p.W + w] : 0.0f);
      }
      if (have) {
        // the markers are requested before the waits for the tile's operands and read after
        const TokMarks now = marks(cur);
        hin_tile = slot_get1(p.fwd_carry + ((size_t)b * (p.nC + 1) + c) * p.W + w);
        ctl.wait(lg_full, it & 1);
        ctl.wait(&in_full[st], ph);
        tc::tc_fence_after();
        if (VARLEN) {
          smask = __ballot_sync(0xffffffffu, now.st >= 0);
          emask = __ballot_sync(0xffffffffu, now.en >= 0);
        }
        rmask = __ballot_sync(0xffffffffu, tok_marks_reset(now, p.reset_mask, p.segment_pos));
        valid = min(FUSED_C, p.T - c * FUSED_C) - tb;
        fast = near_all && rmask == 0u && (smask | emask) == 0u && valid >= PT;
        if (fast)
          bwd_pass1(tcol, xb0, xb1, dyb, gk, ab, xr, P, fB, S);
        else
          bwd_pass1_gen<VARLEN>(tcol, xb0, xb1, dyb, gk, rmask, valid, seqb(smask, emask, b, c),
                                P, fB, S);
      }

      if (have) s_agg[part * FUSED_K + j] = make_float4(P, fB, P, S);  // the part's maps
      if (store_thread) tc::tma_store_wait_read0();  // the dx staging is free again
      tc::named_bar(BAR_SCAN, NSCAN * 32);  // barrier A: the parts' maps, the dx staging
      const int cp = pc, bp = pb;           // tile it - 1
      float Fa = 1.0f, Fb = 0.0f, Rp = 1.0f, Rs = 0.0f, tP = 1.0f, tS = 0.0f;
      const bool publish = (blk * ntiles + n) != p.drop_tile;
      if (have) {
        pc = c;
        pb = b;
        cur.next();
        // The tiles processed alongside this one have published their aggregates by about now:
        // ask again for the slots that were empty at the tile's start.
        if (part == 0) lookback_refresh(lbq, lb_agg, (long)p.W, lb_n, lb_anchor);
        // Entry-state map of this part (earlier parts composed) and carry map from the tile's
        // right edge to this part (later parts composed).
#pragma unroll
        for (int pp = 0; pp < NPART; ++pp) {
          if (pp < part) {
            const float4 g = s_agg[pp * FUSED_K + j];
            Fb = fmaf(g.x, Fb, g.y);
            Fa *= g.x;
          }
        }
#pragma unroll
        for (int pp = NPART - 1; pp > 0; --pp) {
          if (pp > part) {
            const float4 g = s_agg[pp * FUSED_K + j];
            Rs = fmaf(g.z, Rs, g.w);
            Rp *= g.z;
          }
        }
        // Part 0 owns the chunk's reverse carry: its map after the later parts' is the tile's,
        // published at once.
        const float4 g0 = s_agg[j];
        tP = g0.z * Rp;
        tS = fmaf(g0.z, Rs, g0.w);
        if (part == 0 && publish && wok) slot_put2(agg + cidx * p.W + w, tP, tS);
      }

      // dx of tile it - 1: TMEM -> smem [token][channel] as bf16 (float32 goes straight to HBM),
      // here so that its MMAs have had pass 1 and the exchange to finish and the look-back round
      // trip has this to overlap; before pass 2a, which reuses the dx columns.
      if (it > 0) {
        const int validp = min(FUSED_C, p.T - cp * FUSED_C) - tb;
        if (!LG) ctl.wait(dx_full, (it - 1) & 1);  // LG: no products; the lane wrote it itself
        tc::tc_fence_after();
#pragma unroll
        for (int sub = 0; sub < PT / 8; ++sub) {
          float v[8];
          tc::tmem_ld8(tcol + COL_DX + sub * 8, v);
          tc::tmem_ld_wait();
          tc::reg_fence(v);  // no use of v moves above the wait
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int tl = tb + sub * 8 + u;
            if (sizeof(GT) == 2) {
              *reinterpret_cast<bf16*>(s_dx + tl * (FUSED_K * 2) + j * 2) =
                  __float2bfloat16_rn(v[u]);
            } else if (sub * 8 + u < validp && wok) {
              // 128 contiguous bytes per warp and token
              static_cast<float*>(p.dx)[((size_t)bp * p.T + cp * FUSED_C + tl) * p.W + w] = v[u];
            }
          }
        }
        tc::tc_fence_before();
        tc::fence_proxy_async_smem();  // the staging, for the TMA store after the next barrier
      }
      if (!have) {
        tc::named_bar(BAR_SCAN, NSCAN * 32);  // the last tile's dx staging is complete
        if (it > 0 && store_thread && sizeof(GT) == 2) {
          tc::tma_store_3d(&tm_dx, s_dx, blk * FUSED_K, cp * FUSED_C, bp);
          tc::tma_store_commit();
        }
        break;
      }

      // Pass 2a: h_{t-1} through the part, from the earlier parts' map applied to the tile's
      // entry state.
      if (!fast)
        bwd_pass2a_gen<VARLEN>(tcol, xb0, xb1, gk, rmask, valid, seqb(smask, emask, b, c),
                               fmaf(Fa, hin_tile, Fb));
      else
        bwd_pass2a(tcol, xr, ab, fmaf(Fa, hin_tile, Fb));

      if (part == 0) {
        const float cin =
            lookback_finish(lbq, lb_agg, (long)p.W, lb_n, lb_anchor, p.spin_limit, status);
        const float cout = fmaf(tP, cin, tS);
        if (publish && wok) slot_put1(rcar + cidx * p.W + w, cout);
        if (c == 0 && p.dh0 && wok) p.dh0[(size_t)b * p.W + w] = p.canonical ? cout : 0.0f;
        s_cin[j] = cin;
      }
      tc::named_bar(BAR_SCAN, NSCAN * 32);  // barrier B: the tile's right carry, the dx staging
      if (it > 0 && store_thread && sizeof(GT) == 2) {
        tc::tma_store_3d(&tm_dx, s_dx, blk * FUSED_K, cp * FUSED_C, bp);
        tc::tma_store_commit();
      }
      const float cin = fmaf(Rp, s_cin[j], Rs);  // carry into this part from the right

      // The dl buffers are free once the previous tile's MMAs are done.
      if (it > 0 && !LG) ctl.wait(dl_empty, (it - 1) & 1);
      tc::tc_fence_after();
      const DlOut dlo{p.dlr, p.dli, p.dl_plane,
                      ((size_t)b * p.T + (size_t)c * FUSED_C + tb) * p.W + w, p.W,
                      wok ? valid : 0};
      if (fast)
        bwd_pass2b<GT, LGM>(tcol, tb, j, xr, dyb, gk.nk, ab, cin, lg_empty, s_dl, dsp, dba, dbx,
                            dlo);
      else
        bwd_pass2b_gen<VARLEN, GT, LGM>(tcol, tb, j, xb0, xb1, dyb, gk, rmask, valid,
                                        seqb(smask, emask, b, c), cin, lg_empty, s_dl, dsp, dba,
                                        dbx, dlo);
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&in_empty[st]);
        tc::mbar_arrive(dl_full);
      }
    }
    if (store_thread) tc::tma_store_wait0();

    // Per-CTA, per-part partials of the per-channel sums.
    float* vp = reinterpret_cast<float*>(p.scratch + p.F.vec_part) +
                ((size_t)blockIdx.x * NPART + part) * 3 * FUSED_K;
    vp[j] = -8.0f * (dsp.x + dsp.y);  // d sp = sum dla (-8 r)
    vp[FUSED_K + j] = dba.x + dba.y;
    vp[2 * FUSED_K + j] = dbx.x + dbx.y;

    // Per-CTA dW partials: lane j of the accumulators is input channel j; each part takes
    // 128 / NPART of the output-channel columns.  TMEM -> shared memory (the x / dy stages and
    // the dl buffers are free now: row j of 128-byte-swizzled boxes of 32 columns, conflict-free
    // 16-byte stores) -> TMA store of 4 boxes per matrix.  (Given logits: no projections.)
    if (my_tiles > 0 && !LG) ctl.wait(dl_empty, (my_tiles - 1) & 1);
    tc::tc_fence_after();
#pragma unroll
    for (int mtx = 0; mtx < (LG ? 0 : 2); ++mtx) {
      uint8_t* stage = mtx ? s_dl : s_in;
#pragma unroll
      for (int sub = 0; sub < FUSED_K / NPART / 16; ++sub) {
        const int col = part * (FUSED_K / NPART) + sub * 16;
        float v[16];
        if (my_tiles > 0) {
          tc::tmem_ld16(tcol - tb + (mtx ? COL_DWX : COL_DWA) + col, v);
          tc::tmem_ld_wait();
          tc::reg_fence(v);
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) v[u] = 0.0f;
        }
        uint8_t* row = stage + (col >> 5) * DW_BOX_BYTES + j * 128;
        const int c0 = (col & 31) >> 2;  // the row's first 16-byte chunk
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<float4*>(row + (((c0 + u) ^ (j & 7)) << 4)) =
              make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      }
    }
    tc::fence_proxy_async_smem();
    tc::named_bar(BAR_SCAN, NSCAN * 32);
    if (store_thread && !LG) {
#pragma unroll
      for (int mtx = 0; mtx < 2; ++mtx)
#pragma unroll
        for (int bx = 0; bx < FUSED_K / 32; ++bx)
          tc::tma_store_2d(&tm_dwp, (mtx ? s_dl : s_in) + bx * DW_BOX_BYTES, bx * 32,
                           ((int)blockIdx.x * 2 + mtx) * FUSED_K);
      tc::tma_store_commit();
      tc::tma_store_wait0();  // the partials are in global memory before the block's counter
      tc::fence_proxy_async_global();
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }

  // Sum of the partials of the block's P CTAs, once all of them have written theirs; each CTA
  // sums a slice, every element in the same fixed order (deterministic): dWa, dWx [nblk][k][k];
  // dba, dbx [W]; dLambda = sigmoid(Lambda) * sum.  The counters start at zero every call.
  if (threadIdx.x == 0) {
    uint32_t* done = reinterpret_cast<uint32_t*>(p.scratch + BWD_COUNTERS) + blk;
    __threadfence();
    atomicAdd(done, 1u);
    const uint64_t t0 = tc::global_ns();
    while (ld_acquire(done) < (uint32_t)p.P) {
      if (tc::global_ns() - t0 > WAIT_LIMIT_NS) {
        atomicOr(status, STATUS_PIPE);
        break;
      }
      __nanosleep(256);
    }
  }
  __syncthreads();
  constexpr int KK = FUSED_K * FUSED_K;
  constexpr int NV = 2 * KK / 4;  // float4 vectors of the block's dWa, dWx
  const float4* dwp = reinterpret_cast<const float4*>(p.scratch + p.F.dw_part) +
                      (size_t)blk * p.P * NV;
  const int per = (NV + p.P - 1) / p.P;
  const int v0 = rr * per;
  const int nv = LG ? 0 : max(0, min(NV, v0 + per) - v0);
  // This CTA's slice of all P partials comes into shared memory (free now; at most
  // (NV + P) x 16 bytes) by bulk copies in one round trip, completing on w_full's second phase;
  // then each vector is summed over the partials in order.
  float4* sbuf = reinterpret_cast<float4*>(smem);
  if (nv > 0) {
    if (threadIdx.x == 0) {
      tc::fence_proxy_async_global();  // the partials were acquired through the counter
      tc::mbar_expect_tx(w_full, (uint32_t)(p.P * nv * 16));
      for (int r = 0; r < p.P; ++r)
        tc::bulk_load(sbuf + (size_t)r * nv, dwp + (size_t)r * NV + v0, (uint32_t)nv * 16, w_full);
    }
    // always waited for, so that no copy is in flight when the CTA exits
    if (!tc::mbar_wait(w_full, 1, WAIT_LIMIT_NS)) atomicOr(status, STATUS_PIPE);
    for (int v = threadIdx.x; v < nv; v += NTHREADS) {
      float4 t = sbuf[v];
      for (int r = 1; r < p.P; ++r) {
        const float4 a = sbuf[(size_t)r * nv + v];
        t.x += a.x, t.y += a.y, t.z += a.z, t.w += a.w;
      }
      const int vg = v0 + v;
      float* dst = vg < NV / 2 ? p.dWa + (size_t)blk * KK + vg * 4
                               : p.dWx + (size_t)blk * KK + (vg - NV / 2) * 4;
      *reinterpret_cast<float4*>(dst) = t;
    }
  }
  if (rr == 0 && threadIdx.x < FUSED_K && blk * FUSED_K + (int)threadIdx.x < p.W) {
    const int j = threadIdx.x, w = blk * FUSED_K + j;
    const float* vp = reinterpret_cast<const float*>(p.scratch + p.F.vec_part) +
                      (size_t)blk * p.P * NPART * 3 * FUSED_K;
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f;
    for (int r = 0; r < NPART * p.P; ++r) {
      s0 += vp[(size_t)r * 3 * FUSED_K + j];
      s1 += vp[(size_t)r * 3 * FUSED_K + FUSED_K + j];
      s2 += vp[(size_t)r * 3 * FUSED_K + 2 * FUSED_K + j];
    }
    p.dLambda[w] = s0 * __fdividef(1.0f, 1.0f + expf(-p.Lambda[w]));
    if (p.dba) p.dba[w] = s1;
    if (p.dbx) p.dbx[w] = s2;
  }
}

}  // namespace

cudaError_t launch_fused_bwd(const Dims& d, const void* dy, const float* dhT, const void* x,
                             const void* Wa, const float* ba, const void* Wx, const float* bx,
                             const float* Lambda, const uint8_t* rm, const int32_t* sp,
                             const float* h0, const void* saved, void* dx, float* dWa,
                             float* dba, float* dWx, float* dbx, float* dLambda, float* dh0,
                             void* ws, int spin_limit, int drop_tile, cudaStream_t s,
                             const Varlen* vl) {
  (void)h0;  // the chunk entry states saved by the forward already include h0
  if (!fused_supported(d)) return cudaErrorNotSupported;
  const uint64_t W = d.W, T = d.T, B = d.B;
  const uint64_t dims3[3] = {W, T, B};
  const uint64_t str3[2] = {W * 2, T * W * 2};
  const uint32_t box_in[3] = {16, FUSED_C, 1};
  CUtensorMap mx, mdy, mwa, mwx, mdx, mdwp;
  cudaError_t e = encode_tmap(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims3, str3, box_in,
                              CU_TENSOR_MAP_SWIZZLE_32B);
  const uint32_t box_dy[3] = {FUSED_K, FUSED_C, 1};  // one unswizzled [token][channel] tile
  if (e == cudaSuccess)
    e = encode_tmap(&mdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dy, dims3, str3, box_dy,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  const uint64_t dimsw[2] = {(uint64_t)d.k, (uint64_t)d.nblk * d.k};
  const uint64_t strw[1] = {(uint64_t)d.k * 2};
  const uint32_t box_w[2] = {16, FUSED_K};
  if (e == cudaSuccess)
    e = encode_tmap(&mwa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wa, dimsw, strw, box_w,
                    CU_TENSOR_MAP_SWIZZLE_32B);
  if (e == cudaSuccess)
    e = encode_tmap(&mwx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Wx, dimsw, strw, box_w,
                    CU_TENSOR_MAP_SWIZZLE_32B);
  const bool gf32 = d.grad == RGLRU_F32;
  const uint64_t gsz = gf32 ? 4 : 2;
  const uint64_t strg[2] = {W * gsz, T * W * gsz};
  const uint32_t box_dx[3] = {FUSED_K, FUSED_C, 1};
  if (e == cudaSuccess)
    e = encode_tmap(&mdx, gf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, dx, dims3, strg, box_dx, CU_TENSOR_MAP_SWIZZLE_NONE);
  const FusedBwdLayout F = fused_bwd_layout(d);
  const int grid = fused_ctas_per_block(d) * d.nblk;
  // per-CTA dW partials [cta][2][k][k] float32 viewed as [cta * 2 * k rows][k columns]
  const uint64_t dims_p[2] = {(uint64_t)FUSED_K, (uint64_t)grid * 2 * FUSED_K};
  const uint64_t str_p[1] = {(uint64_t)FUSED_K * 4};
  const uint32_t box_p[2] = {32, FUSED_K};
  if (e == cudaSuccess)
    e = encode_tmap(&mdwp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, static_cast<uint8_t*>(ws) + F.dw_part,
                    dims_p, str_p, box_p, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;

  BwdParams p = {};
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
  p.dhT = dhT;
  const FusedFwdLayout FL = fused_fwd_layout(d);
  p.fwd_carry = reinterpret_cast<const float*>(static_cast<const uint8_t*>(saved) + FL.L.carry);
  p.seq_start = vl ? reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + FL.seq_start)
                   : nullptr;
  p.seq_end = vl ? reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + FL.seq_end)
                 : nullptr;
  p.h0s = vl ? vl->h0 : nullptr;
  p.dhTs = vl ? vl->dhT : nullptr;
  p.dh0s = vl ? vl->dh0 : nullptr;
  p.dh0 = dh0;
  p.scratch = static_cast<uint8_t*>(ws);
  p.F = F;
  p.spin_limit = spin_limit;
  p.drop_tile = drop_tile;
  const LookbackPlan lp = lookback_plan(p.P, d.B);
  p.lb_dist = lp.dist;
  p.lb_shift = lp.shift;
  p.dx = dx;
  p.dWa = dWa;
  p.dWx = dWx;
  p.dba = dba;
  p.dbx = dbx;
  p.dLambda = dLambda;
  const size_t smem = SMEM_BYTES;
  auto kern = vl ? (gf32 ? k_fused_bwd<float, true, LGM_NONE> : k_fused_bwd<bf16, true, LGM_NONE>)
                 : (gf32 ? k_fused_bwd<float, false, LGM_NONE> : k_fused_bwd<bf16, false, LGM_NONE>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = clear_slots(ws, p.F.L, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  kernel_event_before(s);
  e = cudaLaunchKernelEx(&cfg, kern, mx, mdy, mwa, mwx, mdx, mdwp, p);
  kernel_event_after(s);
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_logits_bwd(const Dims& d, const void* dy, const float* dhT, const void* x,
                              const void* lr, const void* li, size_t plane_elems, int nplanes,
                              const float* Lambda, const uint8_t* rm, const int32_t* sp,
                              const void* saved, int dx_dt, void* dx, int dl_dt, void* dlr,
                              void* dli, size_t dl_plane, float* dLambda, float* dh0, void* ws,
                              int spin_limit, int drop_tile, cudaStream_t s, const Varlen* vl) {
  if (!logits_scan_supported(d) || nplanes < 1 || nplanes > LG_PLANES)
    return cudaErrorNotSupported;
  const uint64_t W = d.W, T = d.T, B = d.B;
  const uint64_t dims3[3] = {W, T, B};
  const uint64_t str3[2] = {W * 2, T * W * 2};
  const uint32_t box_in[3] = {16, FUSED_C, 1};
  CUtensorMap mx, mdy, mlr, mli, mdx, mdwp;
  cudaError_t e = encode_tmap(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims3, str3, box_in,
                              CU_TENSOR_MAP_SWIZZLE_32B);
  const uint32_t box_dy[3] = {FUSED_K, FUSED_C, 1};
  if (e == cudaSuccess)
    e = encode_tmap(&mdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dy, dims3, str3, box_dy,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess) e = encode_logit_planes(d, lr, plane_elems, nplanes, &mlr);
  if (e == cudaSuccess) e = encode_logit_planes(d, li, plane_elems, nplanes, &mli);
  const bool gf32 = dx_dt == DT_F32;
  const uint64_t gsz = gf32 ? 4 : 2;
  const uint64_t strg[2] = {W * gsz, T * W * gsz};
  const uint32_t box_dx[3] = {FUSED_K, FUSED_C, 1};
  if (e == cudaSuccess)
    e = encode_tmap(&mdx, gf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, dx, dims3, strg, box_dx, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  mdwp = mdx;  // unused without projections
  BwdParams p = {};
  p.B = d.B;
  p.T = d.T;
  p.W = d.W;
  p.nblk = logits_slices(d);
  p.nC = fused_chunks(d);
  p.P = logits_ctas_per_slice(d);
  p.canonical = d.mode == RGLRU_CANONICAL;
  p.nplanes = nplanes;
  p.dlr = dlr;
  p.dli = dli;
  p.dl_plane = dl_plane;
  p.Lambda = Lambda;
  p.reset_mask = p.canonical ? rm : nullptr;
  p.segment_pos = p.canonical ? sp : nullptr;
  p.dhT = dhT;
  const FusedFwdLayout FL = fused_fwd_layout(d);
  p.fwd_carry = reinterpret_cast<const float*>(static_cast<const uint8_t*>(saved) + FL.L.carry);
  if (vl) {
    p.seq_start = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + FL.seq_start);
    p.seq_end = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(saved) + FL.seq_end);
    p.h0s = vl->h0;
    p.dhTs = vl->dhT;
    p.dh0s = vl->dh0;
  }
  p.dh0 = dh0;
  p.scratch = static_cast<uint8_t*>(ws);
  p.F = fused_bwd_layout(d);
  p.spin_limit = spin_limit;
  p.drop_tile = drop_tile;
  const LookbackPlan lp = lookback_plan(p.P, d.B);
  p.lb_dist = lp.dist;
  p.lb_shift = lp.shift;
  p.dx = dx;
  p.dLambda = dLambda;
  decltype(&k_fused_bwd<float, false, LGM_SAME>) kern;
  if (dl_dt == DT_SPLIT) {
    if (!gf32) return cudaErrorNotSupported;
    kern = vl ? k_fused_bwd<float, true, LGM_SPLIT> : k_fused_bwd<float, false, LGM_SPLIT>;
  } else {
    if (vl) return cudaErrorNotSupported;
    if ((dl_dt == DT_F32) != gf32) return cudaErrorNotSupported;
    kern = gf32 ? k_fused_bwd<float, false, LGM_SAME> : k_fused_bwd<bf16, false, LGM_SAME>;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LG_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = clear_slots(ws, p.F.L, s);
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
  e = cudaLaunchKernelEx(&cfg, kern, mx, mdy, mlr, mli, mdx, mdwp, p);
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace rglru
