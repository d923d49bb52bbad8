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

// The decay a = e^la and 1 - a^2 for la <= 0, from one short series.  The decay is multiplied
// over as many tokens as the memory is long (~1 / (1 - a), 10^4 for a = 0.9999), so a
// systematic relative error e in a grows to ~e / (1 - a) in the long-range products: a must
// be accurate to the rounding of a float, not just to a few ulp of an approximate exponential.
// For la > -1/8: e1 = expm1(la) from its Taylor series at 0 cut after la^7 (remainder below
// |la|^8 / 8! < 2e-12), a = 1 + e1, and 1 - a^2 = -e1 (e1 + 2) without cancellation.
// Otherwise (a < 0.89, memory of a few tokens) a = 2^(la log2 e) and 1 - a^2 = 1 - a a.
// The series branch alone, for callers that know la > -1/8 for every token (a channel whose
// softplus(Lambda) < 1/64, since r < 1).
__device__ __forceinline__ void decay_near(float la, float& a, float& om) {
  float p = fmaf(la, 1.0f / 5040.0f, 1.0f / 720.0f);
  p = fmaf(la, p, 1.0f / 120.0f);
  p = fmaf(la, p, 1.0f / 24.0f);
  p = fmaf(la, p, 1.0f / 6.0f);
  p = fmaf(la, p, 0.5f);
  p = fmaf(la, p, 1.0f);
  const float e1 = la * p;
  a = 1.0f + e1;
  om = -e1 * (e1 + 2.0f);
}

__device__ __forceinline__ void decay_fast(float la, float& a, float& om) {
  float p = fmaf(la, 1.0f / 5040.0f, 1.0f / 720.0f);
  p = fmaf(la, p, 1.0f / 120.0f);
  p = fmaf(la, p, 1.0f / 24.0f);
  p = fmaf(la, p, 1.0f / 6.0f);
  p = fmaf(la, p, 0.5f);
  p = fmaf(la, p, 1.0f);
  const float e1 = la * p;
  float ax;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ax) : "f"(la * 1.4426950408889634f));
  const bool near = la > -0.125f;
  a = near ? 1.0f + e1 : ax;
  om = near ? -e1 * (e1 + 2.0f) : fmaf(-ax, ax, 1.0f);
}

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
// sigmoid(z + bias) with nb = -bias * log2(e) precomputed: 1 / (1 + 2^(-(z + bias) log2 e)).
__device__ __forceinline__ float sigmoid_nb(float z, float nb) {
  return rcp_approx(1.0f + ex2_approx(fmaf(z, -LOG2E, nb)));
}

// sqrt(v) for v >= 0 as v * rsqrt(v) (one special-function op), 0 at v = 0.
__device__ __forceinline__ float sqrt_fast(float v) {
  return v > 0.0f ? v * rsqrtf(v) : 0.0f;
}

// ---------------------------------------------------------------- packed pairs
// Two independent float32 lanes per instruction (the f32x2 arithmetic of sm_100 and later):
// a scan thread runs two token chains side by side, one per lane.  Each lane rounds exactly as
// the scalar instruction would.
__device__ __forceinline__ float2 bc2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// sigmoid_nb on two logits.
__device__ __forceinline__ float2 sigmoid2_nb(float2 z, float nb) {
  const float2 s = fma2(z, bc2(-LOG2E), bc2(nb));
  const float2 d = add2(make_float2(ex2_approx(s.x), ex2_approx(s.y)), bc2(1.0f));
  return make_float2(rcp_approx(d.x), rcp_approx(d.y));
}

// decay_near / decay_fast on two lanes (same arithmetic, lane by lane).
__device__ __forceinline__ float2 expm1_series2(float2 la) {
  float2 p = fma2(la, bc2(1.0f / 5040.0f), bc2(1.0f / 720.0f));
  p = fma2(la, p, bc2(1.0f / 120.0f));
  p = fma2(la, p, bc2(1.0f / 24.0f));
  p = fma2(la, p, bc2(1.0f / 6.0f));
  p = fma2(la, p, bc2(0.5f));
  p = fma2(la, p, bc2(1.0f));
  return mul2(la, p);
}
__device__ __forceinline__ void decay_near2(float2 la, float2& a, float2& om) {
  const float2 e1 = expm1_series2(la);
  a = add2(e1, bc2(1.0f));
  om = mul2(e1, fma2(e1, bc2(-1.0f), bc2(-2.0f)));  // -e1 (e1 + 2)
}
__device__ __forceinline__ void decay_fast2(float2 la, float2& a, float2& om) {
  decay_near2(la, a, om);
  if (!(la.x > -0.125f)) {
    const float ax = ex2_approx(la.x * LOG2E);
    a.x = ax;
    om.x = fmaf(-ax, ax, 1.0f);
  }
  if (!(la.y > -0.125f)) {
    const float ax = ex2_approx(la.y * LOG2E);
    a.y = ax;
    om.y = fmaf(-ax, ax, 1.0f);
  }
}
// sqrt of two values >= 0, one special-function op each (PTX sqrt.approx, 0 at 0).
__device__ __forceinline__ float sqrt_approx(float v) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(v));
  return y;
}
__device__ __forceinline__ float2 sqrt_fast2(float2 v) {
  return make_float2(sqrt_approx(v.x), sqrt_approx(v.y));
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
// Look-back slots of the fused kernels carry their own readiness: a slot holds the all-ones
// bit pattern (a NaN that float arithmetic never produces) until its value is stored with a
// single-copy-atomic store.  A reader polls the slot itself, so one L2 round trip delivers
// both the "ready" signal and the value.
constexpr uint32_t SLOT_EMPTY32 = 0xffffffffu;
constexpr uint64_t SLOT_EMPTY64 = 0xffffffffffffffffull;

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
__device__ __forceinline__ void slot_put2(float2* p, float a, float b) {
  st_relaxed_u64(p, ((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(a));
}
__device__ __forceinline__ void slot_put1(float* p, float a) { st_relaxed_u32(p, __float_as_uint(a)); }

// Reset flag of token (b, t) in canonical mode.
__device__ __forceinline__ bool is_reset(const uint8_t* reset_mask, const int32_t* segment_pos,
                                         size_t bt) {
  if (reset_mask) return reset_mask[bt] != 0;
  if (segment_pos) return segment_pos[bt] == 0;
  return false;
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
