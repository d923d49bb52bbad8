// Device helpers shared by the librglru kernels: element access for the two I/O dtypes,
// the gate and decay arithmetic in float32, and the flag protocol of the cross-chunk
// look-back.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rglru {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- element pairs
// Two adjacent channels per access (4 bytes of bf16, 8 bytes of float).
template <typename T>
struct Pair;

template <>
struct Pair<float> {
  static __device__ __forceinline__ float2 load(const float* p) {
    return *reinterpret_cast<const float2*>(p);
  }
  static __device__ __forceinline__ void store(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
  }
  static __device__ __forceinline__ float load1(const float* p) { return *p; }
};

template <>
struct Pair<bf16> {
  static __device__ __forceinline__ float2 load(const bf16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  }
  static __device__ __forceinline__ void store(bf16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
  }
  static __device__ __forceinline__ float load1(const bf16* p) { return __bfloat162float(*p); }
};

// A float32 value stored as two bf16 planes `plane` elements apart: hi = bf16(v) and
// lo = bf16(v - hi) (v - hi is exact in float32), so hi + lo carries v to ~2^-16 relative and
// each plane can be an operand of a bf16 tensor-core product.
struct SplitBf16 {};
template <typename T>
struct OutPair {
  using E = T;
  static __device__ __forceinline__ void store(E* p, size_t, float a, float b) {
    Pair<T>::store(p, a, b);
  }
};
template <>
struct OutPair<SplitBf16> {
  using E = bf16;
  static __device__ __forceinline__ void store(bf16* p, size_t plane, float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(p) = h;
    *reinterpret_cast<__nv_bfloat162*>(p + plane) = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  }
};

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- gate arithmetic
// sigmoid(z) = 1 / (1 + e^-z); e^-z overflows to +inf for very negative z, giving 0.
__device__ __forceinline__ float sigmoid_f(float z) {
  return __fdividef(1.0f, 1.0f + __expf(-z));
}

// softplus(z) = log(1 + e^z) in the overflow-free form; once per channel, full precision.
__device__ __forceinline__ float softplus_f(float z) {
  return z > 0.0f ? z + log1pf(expf(-z)) : log1pf(expf(z));
}

// 1 - a^2 for a = e^la, la <= 0, without the cancellation of 1 - a*a as a -> 1.
__device__ __forceinline__ float one_minus_a2(float la) { return -expm1f(2.0f * la); }

// Single special-function-unit operations (PTX ex2.approx / rcp.approx, flush-to-zero).
constexpr float LOG2E = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sqrt(v) for v >= 0 (PTX sqrt.approx, 0 at 0).
__device__ __forceinline__ float sqrt_approx(float v) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(v));
  return y;
}

// ---------------------------------------------------------------- packed pairs
// Two independent float32 lanes per instruction (the f32x2 arithmetic of sm_100 and later):
// a scan thread runs two token chains side by side, one per lane.  Each lane rounds exactly as
// the scalar instruction would.
__device__ __forceinline__ float2 bc2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// ---------------------------------------------------------------- gates from one rsqrt
// The gates, the decay and the input multiplier of a token pair with two ex2 and one rsqrt per
// token (the special-function unit runs ex2 at twice the rate of the other operations).  With
// er = e^-(lr + ba), ei = e^-(li + bx), pr = 1 + er, pi = 1 + ei, so r = 1 / pr, i = 1 / pi:
//   t = (pr pi^2)^(-1/2),  s = t pi = sqrt(r),  r = s^2,  i = t s pr,  la = nk r  (nk = -8 sp).
// Near regime (la > -1/8): the decay and the multiplier come from two smooth factors,
//   a = e^la = 1 + la P(la),            P(la) = expm1(la) / la,
//   m = sqrt(1 - a^2) = sqrt(-2 la) Q(la),  Q(la) = sqrt((1 - e^(2 la)) / (-2 la)),
// each a degree-3 polynomial fitted on [-1/8, 0] (relative error below 3e-8 in float64).  The
// decay is multiplied over ~1 / (1 - a) tokens, so 1 - a = -la P(la) must carry no systematic
// error beyond float rounding, which the fit gives.  As sqrt(-2 la) = C s with the per-channel
// C = sqrt(-2 nk), the gated input weight is m i = C Q(la) s / pi = C Q(la) t: no sqrt and no
// reciprocal.  The exponents are clamped (er <= 2^48, ei <= 2^39) so that pr pi^2 < 2^127 never
// overflows: a gate that is clamped reads as 2^-48 (r) or 2^-39 (i) instead of something
// smaller still, which changes no result in float32.
constexpr float GATE_ZR_MAX = 48.0f, GATE_ZI_MAX = 39.0f;
constexpr float DECAY_P1 = 4.999970987e-01f, DECAY_P2 = 1.665260549e-01f,
                DECAY_P3 = 3.971588063e-02f;
constexpr float MULT_Q1 = 4.999952308e-01f, MULT_Q2 = 2.081021452e-01f,
                MULT_Q3 = 5.929165853e-02f;
constexpr float NEAR_LA = -0.125f;  // the near regime: la > NEAR_LA

// Per-channel constants of the gate arithmetic.
struct GateK {
  float nk;   // -8 softplus(Lambda): log a = nk r
  float cm;   // sqrt(-2 nk)
  float nbr;  // -ba log2(e)
  float nbi;  // -bx log2(e)
};

__device__ __forceinline__ float rsqrt_approx(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The shared front of the gate arithmetic: t, s and the two sums pr, pi of a token pair.
__device__ __forceinline__ void gate_front2(float2 lr, float2 li, const GateK& k, float2& t,
                                            float2& s, float2& pr, float2& pi) {
  float2 zr = fma2(lr, bc2(-LOG2E), bc2(k.nbr));
  float2 zi = fma2(li, bc2(-LOG2E), bc2(k.nbi));
  zr.x = fminf(zr.x, GATE_ZR_MAX);
  zr.y = fminf(zr.y, GATE_ZR_MAX);
  zi.x = fminf(zi.x, GATE_ZI_MAX);
  zi.y = fminf(zi.y, GATE_ZI_MAX);
  pr = add2(make_float2(ex2_approx(zr.x), ex2_approx(zr.y)), bc2(1.0f));
  pi = add2(make_float2(ex2_approx(zi.x), ex2_approx(zi.y)), bc2(1.0f));
  const float2 d = mul2(mul2(pr, pi), pi);
  t = make_float2(rsqrt_approx(d.x), rsqrt_approx(d.y));
  s = mul2(t, pi);
}

// Near-regime decay and gated input weight from la and t.
__device__ __forceinline__ void gate_near2(float2 la, float2 t, float cm, float2& a, float2& mi) {
  float2 p = fma2(la, bc2(DECAY_P3), bc2(DECAY_P2));
  p = fma2(la, p, bc2(DECAY_P1));
  p = fma2(la, p, bc2(1.0f));
  a = fma2(la, p, bc2(1.0f));
  float2 q = fma2(la, bc2(MULT_Q3), bc2(MULT_Q2));
  q = fma2(la, q, bc2(MULT_Q1));
  q = fma2(la, q, bc2(1.0f));
  mi = mul2(mul2(bc2(cm), t), q);
}

// A token pair, every token in the near regime: decay a, gated input weight m i, and r.
__device__ __forceinline__ void gates_near2(float2 lr, float2 li, const GateK& k, float2& a,
                                            float2& mi, float2& r) {
  float2 t, s, pr, pi;
  gate_front2(lr, li, k, t, s, pr, pi);
  r = mul2(s, s);
  gate_near2(mul2(bc2(k.nk), r), t, k.cm, a, mi);
}

// The same, with i as well.
__device__ __forceinline__ void gates_near2_i(float2 lr, float2 li, const GateK& k, float2& a,
                                              float2& mi, float2& r, float2& i) {
  float2 t, s, pr, pi;
  gate_front2(lr, li, k, t, s, pr, pi);
  r = mul2(s, s);
  i = mul2(mul2(t, s), pr);
  gate_near2(mul2(bc2(k.nk), r), t, k.cm, a, mi);
}

// Any token: the near-regime form where la > -1/8, else a = 2^(la log2 e) and m = sqrt(1 - a a)
// (a < 0.89: a memory of a few tokens, where the relative accuracy of 1 - a is not at stake).
// Also returns i.
__device__ __forceinline__ void gates_any2(float2 lr, float2 li, const GateK& k, float2& a,
                                           float2& mi, float2& r, float2& i) {
  float2 t, s, pr, pi;
  gate_front2(lr, li, k, t, s, pr, pi);
  r = mul2(s, s);
  i = mul2(mul2(t, s), pr);
  const float2 la = mul2(bc2(k.nk), r);
  gate_near2(la, t, k.cm, a, mi);
  if (!(la.x > NEAR_LA)) {
    a.x = ex2_approx(la.x * LOG2E);
    mi.x = sqrt_approx(fmaf(-a.x, a.x, 1.0f)) * i.x;
  }
  if (!(la.y > NEAR_LA)) {
    a.y = ex2_approx(la.y * LOG2E);
    mi.y = sqrt_approx(fmaf(-a.y, a.y, 1.0f)) * i.y;
  }
}

// One channel's gates by the same arithmetic, scalar (the decode step: one token a channel,
// each channel with its own constants).
__device__ __forceinline__ void gates_any1(float lr, float li, const GateK& k, float& a,
                                           float& mi, float& i) {
  const float zr = fminf(fmaf(lr, -LOG2E, k.nbr), GATE_ZR_MAX);
  const float zi = fminf(fmaf(li, -LOG2E, k.nbi), GATE_ZI_MAX);
  const float pr = ex2_approx(zr) + 1.0f, pi = ex2_approx(zi) + 1.0f;
  const float t = rsqrt_approx(pr * pi * pi);
  const float s = t * pi;
  const float r = s * s;
  i = t * s * pr;
  const float la = k.nk * r;
  if (la > NEAR_LA) {
    float p = fmaf(la, DECAY_P3, DECAY_P2);
    p = fmaf(la, p, DECAY_P1);
    p = fmaf(la, p, 1.0f);
    a = fmaf(la, p, 1.0f);
    float q = fmaf(la, MULT_Q3, MULT_Q2);
    q = fmaf(la, q, MULT_Q1);
    q = fmaf(la, q, 1.0f);
    mi = k.cm * t * q;
  } else {
    a = ex2_approx(la * LOG2E);
    mi = sqrt_approx(fmaf(-a, a, 1.0f)) * i;
  }
}

// ---------------------------------------------------------------- staged bf16 tiles
// A [token][channel] bf16 tile staged by TMA as slabs of 16 channels x 32-byte token rows with
// the 32-byte swizzle (the row's two 16-byte halves swap on rows 4..7 of every 8).  b0 / b1
// are the shared-memory addresses of one channel in row tb (a multiple of 8) for rows of
// swizzle parity 0 / 1; element (tb + tt, channel) is then at a compile-time offset from one
// of them for a compile-time tt.
__device__ __forceinline__ float lds_bf16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __uint_as_float((uint32_t)v << 16);
}
__device__ __forceinline__ float tok_elem(uint32_t b0, uint32_t b1, int tt) {
  return lds_bf16((((tt >> 2) & 1) ? b1 : b0) + tt * 32);
}
// The raw bf16 bits of the same element, and two of them packed (token u in the low half).
__device__ __forceinline__ uint32_t tok_raw(uint32_t b0, uint32_t b1, int tt) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"((((tt >> 2) & 1) ? b1 : b0) + tt * 32));
  return v;
}
__device__ __forceinline__ float2 bf16x2_unpack(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// ---------------------------------------------------------------- tile walks
// Chunk c and batch row b of the tiles n = r, r + P, r + 2P, ... of one gate block, with
// n = c * B + b, stepped without a division per tile.
struct TileWalk {
  int c, b, dc, db, B;
  __device__ TileWalk(int r, int P, int B_) : c(r / B_), b(r % B_), dc(P / B_), db(P % B_), B(B_) {}
  __device__ void next() {
    c += dc;
    b += db;
    if (b >= B) {
      b -= B;
      ++c;
    }
  }
};

// ---------------------------------------------------------------- value-as-flag slots
// Look-back slots of the fused kernels carry their own readiness: a value is stored bitwise
// inverted with a single-copy-atomic store, so a slot reads zero until it is written (zero is
// the inverse of the all-ones NaN, which float arithmetic never produces).  A reader polls the
// slot itself, so one L2 round trip delivers both the "ready" signal and the value; and one
// zero fill clears the slots together with the status word and counters before a call.
constexpr uint32_t SLOT_EMPTY32 = 0u;
constexpr uint64_t SLOT_EMPTY64 = 0ull;

__device__ __forceinline__ uint64_t ld_relaxed_u64(const void* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(void* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(void* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t slot_enc1(float a) { return ~__float_as_uint(a); }
__device__ __forceinline__ uint64_t slot_enc2(float a, float b) {
  return ~(((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(a));
}
__device__ __forceinline__ float slot_dec1(uint32_t v) { return __uint_as_float(~v); }
__device__ __forceinline__ float2 slot_dec2(uint64_t v) {
  return make_float2(__uint_as_float(~(uint32_t)v), __uint_as_float(~(uint32_t)(v >> 32)));
}
__device__ __forceinline__ void slot_put2(float2* p, float a, float b) {
  st_relaxed_u64(p, slot_enc2(a, b));
}
__device__ __forceinline__ void slot_put1(float* p, float a) { st_relaxed_u32(p, slot_enc1(a)); }
// A slot written before this kernel started (plain load).
__device__ __forceinline__ float slot_get1(const float* p) {
  return slot_dec1(*reinterpret_cast<const uint32_t*>(p));
}

// Reset flag of token (b, t) in canonical mode.
__device__ __forceinline__ bool is_reset(const uint8_t* reset_mask, const int32_t* segment_pos,
                                         size_t bt) {
  if (reset_mask) return reset_mask[bt] != 0;
  if (segment_pos) return segment_pos[bt] == 0;
  return false;
}

// The markers of one token that decide a fused tile's path, as stored: the reset-mask byte or
// the segment position (canonical mode), and the packed sequence that starts / ends at the
// token (-1: none).  The fused kernels request a tile's markers one tile ahead of their use,
// so that the load's round trip hides behind a tile of work.
struct TokMarks {
  int rs, st, en;
};
__device__ __forceinline__ TokMarks tok_marks_load(const uint8_t* reset_mask,
                                                   const int32_t* segment_pos,
                                                   const int32_t* seq_start,
                                                   const int32_t* seq_end, size_t bt, bool in) {
  TokMarks m{-1, -1, -1};
  if (in) {
    if (reset_mask) m.rs = reset_mask[bt];
    else if (segment_pos) m.rs = segment_pos[bt];
    if (seq_start) m.st = seq_start[bt];
    if (seq_end) m.en = seq_end[bt];
  }
  return m;
}
// Reset flag from the stored marker (-1: a token past T, never a reset).
__device__ __forceinline__ bool tok_marks_reset(const TokMarks& m, const uint8_t* reset_mask,
                                                const int32_t* segment_pos) {
  return reset_mask ? m.rs > 0 : (segment_pos ? m.rs == 0 : false);
}

// ---------------------------------------------------------------- look-back flags
// A scan tile publishes FLAG_AGG once its own affine aggregate (A, B) is stored, and
// FLAG_INCL once its chunk-boundary state (the "inclusive prefix") is stored.  Flags are
// zeroed before every launch.
constexpr uint32_t FLAG_AGG = 1u;
constexpr uint32_t FLAG_INCL = 2u;
constexpr uint32_t FLAG_TIMEOUT = 0xffffffffu;  // returned by spin_flag only
constexpr uint32_t STATUS_TIMEOUT = 1u;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Polls `flag` until it reaches `target` (FLAG_AGG or FLAG_INCL), at most `limit` times.  On
// running out it records the timeout in `status` and returns FLAG_TIMEOUT, so the caller
// carries on (with a zero carry) and the kernel always terminates.
__device__ __forceinline__ uint32_t spin_flag(const uint32_t* flag, uint32_t target, int limit,
                                              uint32_t* status) {
  uint32_t f = ld_acquire(flag);
  int it = 0;
  while (f < target) {
    if (++it > limit) {
      atomicOr(status, STATUS_TIMEOUT);
      return FLAG_TIMEOUT;
    }
    __nanosleep(64);
    f = ld_acquire(flag);
  }
  return f;
}

}  // namespace rglru
