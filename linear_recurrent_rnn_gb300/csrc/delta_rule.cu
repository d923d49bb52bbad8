// Gated delta rule (GDN: one decay per value head and token; KDA: one per key channel) on the
// CUDA cores of one GB300, forward and backward.
//
// Source ("linear_attention.reference" page, the recurrent reference's entry): the exact token
// recurrence with scalar or per-key decay given as natural logarithms, grouped key heads,
// initial and final states, packed sequences.  Per sequence and value head (key head
// h / (Hv / Hk)), token t, S the [Dk, Dv] state:
//   S' = D_t S (D_t = exp(g_t), or diag(exp(g_t)) per key),  u = beta_t (v_t - S'^T k_t),
//   S = S' + k_t u^T,  o_t = scale S^T q_t.
//
// Geometry: the state lives in registers.  A thread owns 32 keys of one value column, so a
// column is shared by KG = Dk / 32 adjacent lanes (lane = column-in-warp * KG + key group) and
// S'^T k, S'^T q are 32-term dot products per thread plus log2(KG) shuffles.  Token data (k, q,
// decays, beta, v) comes in by asynchronous copies a block of 16 tokens ahead, is converted in
// shared memory to float32 rows with padded 32-key groups, and is read by every thread as
// broadcast 16-byte loads.
//   forward:  CTA = (sequence, value head, 2 x 4 x 32 / KG columns), 4 warps, two value
//             columns per thread (one at Dk = 32) sharing the k / q loads; the state entering
//             every 16-token block is saved (float32, [slot][Hv][Dv][Dk]) for the backward.
//   backward: a cluster of two CTAs per (sequence, value head), half of the Dv columns each;
//             per 16-token block in reverse it restores the block's entry state, runs the
//             block forward again keeping each token's state in thread-local memory, and then
//             runs the reverse recurrence.  The sums over value columns (dq, dk, KDA's dg) fold
//             the warp's columns with a halving butterfly of shuffles, the warps through shared
//             memory, and the two CTAs through distributed shared memory once per block.
//   k_state_qdq: the E4M3 quantize-dequantize of states, one scale per [Dk, block_v] tile.
#include <algorithm>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "delta_rule.h"

namespace rglru {

namespace {

constexpr int DR_TB = 16;                 // tokens per staged block = tokens per saved state
// float32 rows of keys are stored as groups of 32 keys 36 floats apart: the KG groups a warp
// reads at once then start 4 banks apart, so its broadcast 16-byte loads do not conflict
constexpr int KGS = 36;
// reduction rows: groups of 32 keys 33 floats apart (one bank apart)
constexpr int RGS = 33;
constexpr unsigned FULL = 0xffffffffu;

struct DrArgs {
  int B, T, Hk, Hv, Dk, Dv, kda, vfirst, N, nslices;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const int32_t* cu;
  const float* h0;
  void* o;
  float* hT;
  float* saved;  // [slot][Hv][Dv][Dk]
  // backward
  const void* dout;
  const float* dhT;
  float* dq;      // [B*T][Hk][Dk], or per value head [B*T][Hv][Dk] when Hv > Hk
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dh0;
};

// Sequence n: its batch row, first token within the row, length, and first saved-state slot.
// Slots are laid out so that sequences never share one: floor(flat start / 16) + 2 n.
struct Seq {
  int b, s, len;
  long slot0;
};
__device__ __forceinline__ Seq seq_of(const DrArgs& a, int n) {
  Seq q;
  if (a.cu) {
    q.b = 0;
    q.s = a.cu[n];
    const int e = a.cu[n + 1];
    q.len = max(0, min(e, a.T) - q.s);
    q.s = min(max(q.s, 0), a.T);
  } else {
    q.b = n;
    q.s = 0;
    q.len = a.T;
  }
  q.slot0 = ((long)q.b * a.T + q.s) / DR_TB + 2L * n;
  return q;
}

template <typename T>
__device__ __forceinline__ float ldf(const void* p, size_t i) {
  return to_f32<T>(static_cast<const T*>(p)[i]);
}

// ---- staging.  A block of DR_TB tokens comes in raw (storage dtype, as in global memory) by
// 16-byte asynchronous copies into one of two raw buffers, one block ahead of the compute;
// prepare_block then converts it in shared memory to float32 rows (and the decays, exp(g), and
// for KDA decay * k).  Tokens past the sequence are zero-filled, never read from global memory.
__device__ __forceinline__ void cp_async(void* dst, const void* src, uint32_t bytes, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
                 "r"(valid ? 16u : 0u) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
                 "r"(valid ? 4u : 0u) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// One raw stage: k, q [TB][DK], v (and do) [TB][NC] in the storage dtype; g [TB][DK] (KDA) or
// [TB] (GDN) and beta [TB] as float32.
template <typename T, int DK>
struct Raw {
  static constexpr size_t kq_bytes = (size_t)DR_TB * DK * sizeof(T);
  __host__ __device__ static size_t bytes(int NC, bool with_do) {
    return 2 * kq_bytes + (with_do ? 2 : 1) * (size_t)DR_TB * NC * sizeof(T) +
           (size_t)DR_TB * DK * 4 + DR_TB * 4;
  }
};

template <typename T, int DK>
__device__ void issue_block(const DrArgs& a, const Seq& sq, int hv, int t0, int nt, int c0,
                            int NC, uint8_t* raw, bool with_do) {
  constexpr int EV = 16 / sizeof(T);  // elements per 16-byte copy
  const int hk = hv / (a.Hv / a.Hk);
  T* rk = reinterpret_cast<T*>(raw);
  T* rq = rk + DR_TB * DK;
  T* rv = rq + DR_TB * DK;
  T* rdo = rv + DR_TB * NC;
  float* rg = reinterpret_cast<float*>(rv + (with_do ? 2 : 1) * DR_TB * NC);
  float* rb = rg + DR_TB * DK;
  const size_t row0 = (size_t)sq.b * a.T + sq.s + t0;  // first token of the block
  constexpr int VK = DK / EV;
  for (int e = threadIdx.x; e < DR_TB * VK; e += blockDim.x) {
    const int tt = e / VK, x = e % VK;
    const bool ok = tt < nt;
    const size_t src = ((row0 + (ok ? tt : 0)) * a.Hk + hk) * DK + x * EV;
    cp_async(rk + tt * DK + x * EV, static_cast<const T*>(a.k) + src, 16, ok);
    cp_async(rq + tt * DK + x * EV, static_cast<const T*>(a.q) + src, 16, ok);
  }
  const int VN = NC / EV;
  for (int e = threadIdx.x; e < DR_TB * VN; e += blockDim.x) {
    const int tt = e / VN, x = e % VN, j = c0 + x * EV;
    const bool ok = tt < nt && j < a.Dv;
    const size_t src = ((row0 + (ok ? tt : 0)) * a.Hv + hv) * a.Dv + (ok ? j : 0);
    cp_async(rv + tt * NC + x * EV, static_cast<const T*>(a.v) + src, 16, ok);
    if (with_do) cp_async(rdo + tt * NC + x * EV, static_cast<const T*>(a.dout) + src, 16, ok);
  }
  if (a.kda) {
    constexpr int VG = DK / 4;
    for (int e = threadIdx.x; e < DR_TB * VG; e += blockDim.x) {
      const int tt = e / VG, x = e % VG;
      const bool ok = tt < nt;
      const size_t src = ((row0 + (ok ? tt : 0)) * a.Hv + hv) * DK + x * 4;
      cp_async(rg + tt * DK + x * 4, a.g + src, 16, ok);
    }
  }
  if (threadIdx.x < DR_TB) {
    const int tt = threadIdx.x;
    const bool ok = tt < nt;
    const size_t src = (row0 + (ok ? tt : 0)) * a.Hv + hv;
    if (!a.kda) cp_async(rg + tt, a.g + src, 4, ok);
    cp_async(rb + tt, a.beta + src, 4, ok);
  }
}

template <typename T, int DK>
__device__ void prepare_block(const DrArgs& a, const uint8_t* raw, int NC, bool with_do,
                              float* s_k, float* s_q, float* s_a, float* s_ak, float* s_v,
                              float* s_do, float* s_b, float* s_ag, float* s_aq = nullptr,
                              float* s_kq = nullptr) {
  const T* rk = reinterpret_cast<const T*>(raw);
  const T* rq = rk + DR_TB * DK;
  const T* rv = rq + DR_TB * DK;
  const T* rdo = rv + DR_TB * NC;
  const float* rg = reinterpret_cast<const float*>(rv + (with_do ? 2 : 1) * DR_TB * NC);
  const float* rb = rg + DR_TB * DK;
  constexpr int DKP = DK / 32 * KGS;
  for (int e = threadIdx.x; e < DR_TB * DK; e += blockDim.x) {
    const int tt = e / DK, i = e % DK;
    const int d = tt * DKP + (i >> 5) * KGS + (i & 31);
    const float kv = to_f32<T>(rk[e]), qv = to_f32<T>(rq[e]);
    s_k[d] = kv;
    s_q[d] = qv;
    if (a.kda) {
      const float av = expf(rg[e]);
      s_a[d] = av;
      s_ak[d] = av * kv;
      if (s_aq) s_aq[d] = av * qv;
    }
  }
  if (s_kq) {  // k . q of every token, one warp per token
    const int nw = blockDim.x >> 5, lane = threadIdx.x & 31;
    for (int tt = threadIdx.x >> 5; tt < DR_TB; tt += nw) {
      float p = 0.0f;
      for (int i = lane; i < DK; i += 32)
        p = fmaf(to_f32<T>(rk[tt * DK + i]), to_f32<T>(rq[tt * DK + i]), p);
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) p += __shfl_xor_sync(FULL, p, m);
      if (lane == 0) s_kq[tt] = p;
    }
  }
  for (int e = threadIdx.x; e < DR_TB * NC; e += blockDim.x) {
    s_v[e] = to_f32<T>(rv[e]);
    if (with_do) s_do[e] = to_f32<T>(rdo[e]);
  }
  if (threadIdx.x < DR_TB) {
    s_b[threadIdx.x] = rb[threadIdx.x];
    s_ag[threadIdx.x] = a.kda ? 1.0f : expf(rg[threadIdx.x]);
  }
}

// 32 consecutive floats of a staged row (16-byte aligned) into registers.
__device__ __forceinline__ void ld32(const float* p, float (&r)[32]) {
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const float4 v = reinterpret_cast<const float4*>(p)[x];
    r[4 * x] = v.x, r[4 * x + 1] = v.y, r[4 * x + 2] = v.z, r[4 * x + 3] = v.w;
  }
}

// Sum over the KG lanes that share a column.
template <int KG>
__device__ __forceinline__ float kg_sum(float x) {
  if (KG >= 2) x += __shfl_xor_sync(FULL, x, 1);
  if (KG >= 4) x += __shfl_xor_sync(FULL, x, 2);
  return x;
}

// sum_x a[x] b[x] over 32 terms in four interleaved partial sums (a shorter dependent chain).
__device__ __forceinline__ float dot32(const float (&x)[32], const float (&y)[32]) {
  float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    p0 = fmaf(x[i], y[i], p0);
    p1 = fmaf(x[i + 1], y[i + 1], p1);
    p2 = fmaf(x[i + 2], y[i + 2], p2);
    p3 = fmaf(x[i + 3], y[i + 3], p3);
  }
  return (p0 + p1) + (p2 + p3);
}

// One token of the forward on a thread's 32 keys: S' = D S, w = S'^T k, u = beta (v - w),
// S = S' + k u; returns w and u (the column's, identical on its KG lanes).
template <int KG>
__device__ __forceinline__ void fwd_token(float (&S)[32], const float* kr, const float* ar,
                                          const float* akr, bool kda, float ag, float bt,
                                          float vj, float& w, float& u) {
  float kk[32];
  ld32(kr, kk);
  float part = 0.0f;
  if (kda) {
    float ak[32];
    ld32(akr, ak);
    part = dot32(S, ak);
    w = kg_sum<KG>(part);
    u = bt * (vj - w);
    float al[32];
    ld32(ar, al);
#pragma unroll
    for (int x = 0; x < 32; ++x) S[x] = fmaf(al[x], S[x], kk[x] * u);
  } else {
    part = dot32(S, kk);
    w = ag * kg_sum<KG>(part);
    u = bt * (vj - w);
#pragma unroll
    for (int x = 0; x < 32; ++x) S[x] = fmaf(ag, S[x], kk[x] * u);
  }
}

// Value columns per forward thread: two (sharing every shared-memory load of k and q, and
// giving the thread two independent chains) except at Dk = 32, where a CTA would span more
// columns than a head has.
constexpr int fwd_cpt(int KG) { return KG == 1 ? 1 : 2; }
// Columns of one forward CTA: 4 warps x (32 / KG) column slots x columns per thread.
constexpr int fwd_cols(int KG) { return 4 * (32 / KG) * fwd_cpt(KG); }

template <typename T, int KG>
__global__ void __launch_bounds__(128) k_dr_fwd(DrArgs a) {
  constexpr int DK = 32 * KG, CPW = 32 / KG, CPT = fwd_cpt(KG), NH = 4 * CPW;
  constexpr int NC = fwd_cols(KG), DKP = KG * KGS;
  extern __shared__ __align__(16) float sm[];
  float* s_k = sm;
  float* s_q = s_k + DR_TB * DKP;
  float* s_a = s_q + DR_TB * DKP;
  float* s_ak = s_a + DR_TB * DKP;
  float* s_aq = s_ak + DR_TB * DKP;
  float* s_v = s_aq + DR_TB * DKP;
  float* s_b = s_v + DR_TB * NC;
  float* s_ag = s_b + DR_TB;
  float* s_kq = s_ag + DR_TB;
  uint8_t* raw0 = reinterpret_cast<uint8_t*>(s_kq + DR_TB);
  const size_t rawb = Raw<T, DK>::bytes(NC, false);
  const int slice = blockIdx.x % a.nslices;
  const int hv = (blockIdx.x / a.nslices) % a.Hv;
  const int n = blockIdx.x / (a.nslices * a.Hv);
  const Seq sq = seq_of(a, n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kg = lane % KG, jc = warp * CPW + lane / KG;
  const int c0 = slice * NC;
  int j[CPT];
  bool live[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    j[c] = c0 + c * NH + jc;  // column c of this thread (c-th half of the CTA's columns)
    live[c] = j[c] < a.Dv;
  }
  const int key0 = kg * 32, kp0 = kg * KGS;  // first key, and its padded offset in a row
  const size_t base = (size_t)n * a.Hv + hv;

  float S[CPT][32];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
#pragma unroll
    for (int x = 0; x < 32; ++x) S[c][x] = 0.0f;
    if (a.h0 && live[c]) {
#pragma unroll
      for (int x = 0; x < 32; ++x)
        S[c][x] = a.vfirst ? a.h0[(base * a.Dv + j[c]) * DK + key0 + x]
                           : a.h0[(base * DK + key0 + x) * a.Dv + j[c]];
    }
  }
  const int nblk = (sq.len + DR_TB - 1) / DR_TB;
  if (nblk > 0) issue_block<T, DK>(a, sq, hv, 0, min(DR_TB, sq.len), c0, NC, raw0, false);
  cp_commit();
  for (int blk = 0; blk < nblk; ++blk) {
    const int t0 = blk * DR_TB, nt = min(DR_TB, sq.len - t0);
    if (blk + 1 < nblk)  // the next block's copies overlap this block's tokens
      issue_block<T, DK>(a, sq, hv, t0 + DR_TB, min(DR_TB, sq.len - t0 - DR_TB), c0, NC,
                         raw0 + ((blk + 1) & 1) * rawb, false);
    cp_commit();
    cp_wait1();
    __syncthreads();  // this block's copies have landed; the previous block is consumed
    prepare_block<T, DK>(a, raw0 + (blk & 1) * rawb, NC, false, s_k, s_q, s_a, s_ak, s_v,
                         nullptr, s_b, s_ag, s_aq, s_kq);
    __syncthreads();
    if (a.saved) {  // the state entering the block
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        if (!live[c]) continue;
        float* dst =
            a.saved + (((size_t)(sq.slot0 + t0 / DR_TB) * a.Hv + hv) * a.Dv + j[c]) * DK + key0;
#pragma unroll
        for (int x = 0; x < 8; ++x)
          reinterpret_cast<float4*>(dst)[x] =
              make_float4(S[c][4 * x], S[c][4 * x + 1], S[c][4 * x + 2], S[c][4 * x + 3]);
      }
    }
    for (int tt = 0; tt < nt; ++tt) {
      // Both products read the state before the token: with S' = D S,
      //   w = S'^T k,  u = beta (v - w),  S_t = S' + k u^T,
      //   o = scale S_t^T q = scale (S'^T q + (k . q) u),
      // so S'^T k and S'^T q of the thread's columns form one step of independent dot
      // products over the same k and q registers.
      const int r = tt * DKP + kp0;
      const float bt = s_b[tt], kq = s_kq[tt];
      float kk[32], pk[CPT], pq[CPT], ag = 1.0f;
      ld32(s_k + r, kk);
      if (a.kda) {
        float ak[32], aq[32];
        ld32(s_ak + r, ak);
        ld32(s_aq + r, aq);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          pk[c] = dot32(S[c], ak);
          pq[c] = dot32(S[c], aq);
        }
      } else {
        float qq[32];
        ld32(s_q + r, qq);
        ag = s_ag[tt];
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          pk[c] = ag * dot32(S[c], kk);
          pq[c] = ag * dot32(S[c], qq);
        }
      }
      float u[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        pk[c] = kg_sum<KG>(pk[c]);
        pq[c] = kg_sum<KG>(pq[c]);
        u[c] = bt * (s_v[tt * NC + c * NH + jc] - pk[c]);
      }
      if (a.kda) {
        float al[32];
        ld32(s_a + r, al);
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
          for (int x = 0; x < 32; ++x) S[c][x] = fmaf(al[x], S[c][x], kk[x] * u[c]);
      } else {
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
          for (int x = 0; x < 32; ++x) S[c][x] = fmaf(ag, S[c][x], kk[x] * u[c]);
      }
      if (kg == 0) {
        const size_t row = (size_t)sq.b * a.T + sq.s + t0 + tt;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
          if (live[c])
            static_cast<T*>(a.o)[(row * a.Hv + hv) * a.Dv + j[c]] =
                from_f32<T>(a.scale * fmaf(kq, u[c], pq[c]));
      }
    }
  }
  if (a.hT) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      if (!live[c]) continue;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        if (a.vfirst)
          a.hT[(base * a.Dv + j[c]) * DK + key0 + x] = S[c][x];
        else
          a.hT[(base * DK + key0 + x) * a.Dv + j[c]] = S[c][x];
      }
    }
  }
}

template <typename T>
size_t fwd_smem(int KG) {
  const int DK = 32 * KG, NC = fwd_cols(KG);
  const size_t raw = 2 * (size_t)DR_TB * DK * sizeof(T) + (size_t)DR_TB * NC * sizeof(T) +
                     (size_t)DR_TB * DK * 4 + DR_TB * 4;
  return (size_t)(5 * DR_TB * KG * KGS + DR_TB * NC + 3 * DR_TB) * sizeof(float) + 2 * raw;
}

// Sums 32 per-key values over the CPW columns of the warp with a halving butterfly: at level L
// the lanes that differ in lane bit KG << L swap halves, so after log2(CPW) levels each lane
// holds KG sums, of keys key0 + fold_key(lane) + x (x < KG).
template <int KG, int L>
__device__ __forceinline__ void fold(float (&v)[32], int lane) {
  constexpr int M = KG << L, H = 16 >> L;
  if constexpr (M < 32) {
    const bool hi = (lane & M) != 0;
#pragma unroll
    for (int x = 0; x < H; ++x) {
      const float send = hi ? v[x] : v[x + H];
      const float keep = hi ? v[x + H] : v[x];
      v[x] = keep + __shfl_xor_sync(FULL, send, M);
    }
    fold<KG, L + 1>(v, lane);
  }
}
template <int KG>
__device__ __forceinline__ int fold_key(int lane) {
  int off = 0;
#pragma unroll
  for (int L = 0; (KG << L) < 32; ++L)
    if (lane & (KG << L)) off += 16 >> L;
  return off;
}
// The CTA's rank in its cluster, a float from the same offset of another CTA's shared memory,
// and a barrier over the cluster (release / acquire).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ float ld_peer(const float* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(FULL, x, m);
  return x;
}

// Backward.  A cluster of two CTAs per (sequence n, value head hv), each with half of the value
// columns (blockDim = 32 x ceil(Dv / 2 / CPW)).  Per 16-token
// block, last block first: restore the block's entry state from `saved`, run the block forward
// keeping every token's state before its decay (thread-local), w and u; then for each token in
// reverse (dS the gradient of the state after the token):
//   dS += scale q do^T;  dq = scale (S' + k u^T) do;  du = dS^T k;  dw = -beta du
//   dk = dS u + S' dw;  dbeta = du . (v - w);  dv = beta du;  dS' = dS + k dw^T
//   dg = <dS', S'> (GDN) or its row sums (KDA);  dS = D dS'
// dq, dk (and KDA's dg) sum over the columns: warp butterfly, the warps through shared memory
// (one CTA barrier per token), and the CTAs of the cluster through distributed shared memory
// once per block: the sums feed only outputs, never the recurrence, so a block's per-token CTA
// sums are kept and each CTA writes its share of the outputs, the CTAs' sums added in rank
// order, after one cluster barrier.
template <typename T, int KG, int CL>
__global__ void __launch_bounds__(256, 1) k_dr_bwd(DrArgs a) {
  constexpr int DK = 32 * KG, CPW = 32 / KG, DKP = KG * KGS, DKR = KG * RGS;
  const int nwarps = blockDim.x >> 5, NC = nwarps * CPW;
  const int NV = a.kda ? 3 : 2;      // per-key vectors reduced per token: dq, dk (, dg)
  // a warp's reduction row: vectors, dbeta, GDN dg; a multiple of 4 floats, so that the raw
  // staging after the rows stays 16-byte aligned
  const int RS = (NV * DKR + 2 + 3) & ~3;
  extern __shared__ __align__(16) float sm[];
  float* s_k = sm;
  float* s_q = s_k + DR_TB * DKP;
  float* s_a = s_q + DR_TB * DKP;
  float* s_ak = s_a + DR_TB * DKP;
  float* s_v = s_ak + DR_TB * DKP;
  float* s_do = s_v + DR_TB * NC;
  float* s_b = s_do + DR_TB * NC;
  float* s_ag = s_b + DR_TB;
  float* s_red = s_ag + DR_TB;       // [2][nwarps][RS]
  const int NE = NV * DK + 2, XS = (NE + 3) & ~3;
  // [2 blocks][DR_TB tokens][XS]: this CTA's sums of a block, read by its peers too
  float* s_xp = s_red + 2 * nwarps * RS;
  uint8_t* raw0 = reinterpret_cast<uint8_t*>(s_xp + 2 * DR_TB * XS);
  const size_t rawb = Raw<T, DK>::bytes(NC, true);
  const uint32_t crank = cluster_rank();
  const int pid = blockIdx.x / CL;
  const int hv = pid % a.Hv, n = pid / a.Hv;
  const int hk = hv / (a.Hv / a.Hk);
  const Seq sq = seq_of(a, n);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = (int)crank * NC;  // this CTA's first value column
  const int kg = lane % KG, jc = warp * CPW + lane / KG, j = c0 + jc;
  const bool live = j < a.Dv;
  const int key0 = kg * 32, kp0 = kg * KGS;
  const int kf = kg * RGS + fold_key<KG>(lane);  // this lane's folded sums in a reduction row
  const size_t hbase = (size_t)n * a.Hv + hv;
  const bool per_vhead = a.Hv != a.Hk;  // dq, dk per value head, summed by a second kernel

  float dS[32];
#pragma unroll
  for (int x = 0; x < 32; ++x) dS[x] = 0.0f;
  if (a.dhT && live) {
#pragma unroll
    for (int x = 0; x < 32; ++x)
      dS[x] = a.vfirst ? a.dhT[(hbase * a.Dv + j) * DK + key0 + x]
                       : a.dhT[(hbase * DK + key0 + x) * a.Dv + j];
  }
  float hist[DR_TB][32];
  float wh[DR_TB], uh[DR_TB];
  const int nblk = (sq.len + DR_TB - 1) / DR_TB;
  if (nblk > 0) {
    const int tl = (nblk - 1) * DR_TB;
    issue_block<T, DK>(a, sq, hv, tl, sq.len - tl, c0, NC, raw0 + ((nblk - 1) & 1) * rawb, true);
  }
  cp_commit();
  for (int blk = nblk - 1; blk >= 0; --blk) {
    const int t0 = blk * DR_TB, nt = min(DR_TB, sq.len - t0);
    if (blk > 0)  // the previous block's copies overlap this block's work
      issue_block<T, DK>(a, sq, hv, t0 - DR_TB, DR_TB, c0, NC, raw0 + ((blk - 1) & 1) * rawb, true);
    cp_commit();
    cp_wait1();
    __syncthreads();
    prepare_block<T, DK>(a, raw0 + (blk & 1) * rawb, NC, true, s_k, s_q, s_a, s_ak, s_v, s_do,
                         s_b, s_ag);
    __syncthreads();
    float S[32];
    if (live) {
      const float* src = a.saved + (((size_t)(sq.slot0 + blk) * a.Hv + hv) * a.Dv + j) * DK + key0;
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float4 v = reinterpret_cast<const float4*>(src)[x];
        S[4 * x] = v.x, S[4 * x + 1] = v.y, S[4 * x + 2] = v.z, S[4 * x + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int x = 0; x < 32; ++x) S[x] = 0.0f;
    }
    for (int tt = 0; tt < nt; ++tt) {
#pragma unroll
      for (int x = 0; x < 32; ++x) hist[tt][x] = S[x];
      fwd_token<KG>(S, s_k + tt * DKP + kp0, s_a + tt * DKP + kp0, s_ak + tt * DKP + kp0,
                    a.kda != 0, s_ag[tt], s_b[tt], s_v[tt * NC + jc], wh[tt], uh[tt]);
    }
    for (int tt = nt - 1; tt >= 0; --tt) {
      const float ag = s_ag[tt], bt = s_b[tt], u = uh[tt], w = wh[tt];
      const float doj = s_do[tt * NC + jc], vj = s_v[tt * NC + jc];
      const float* kr = s_k + tt * DKP + kp0;
      const float* ar = s_a + tt * DKP + kp0;
      float Sp[32], vec[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) Sp[x] = hist[tt][x];
      if (a.kda) {
        float al[32];
        ld32(ar, al);
#pragma unroll
        for (int x = 0; x < 32; ++x) Sp[x] *= al[x];
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) Sp[x] *= ag;
      }
      // dS += scale q do;  dq = scale (S' + k u) do
      {
        float qq[32], kk[32];
        ld32(s_q + tt * DKP + kp0, qq);
        ld32(kr, kk);
        const float sd = a.scale * doj;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          dS[x] = fmaf(qq[x], sd, dS[x]);
          vec[x] = fmaf(kk[x], u, Sp[x]) * sd;
        }
      }
      const int buf = tt & 1;
      float* red = s_red + ((size_t)buf * nwarps + warp) * RS;
      fold<KG, 0>(vec, lane);
#pragma unroll
      for (int x = 0; x < KG; ++x) red[kf + x] = vec[x];
      // du = dS^T k;  dk = dS u + S' dw;  dS' = dS + k dw
      float du, dw;
      {
        float kk[32];
        ld32(kr, kk);
        du = kg_sum<KG>(dot32(dS, kk));
        dw = -bt * du;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          vec[x] = fmaf(dS[x], u, Sp[x] * dw);
          dS[x] = fmaf(kk[x], dw, dS[x]);
        }
      }
      fold<KG, 0>(vec, lane);
#pragma unroll
      for (int x = 0; x < KG; ++x) red[DKR + kf + x] = vec[x];
      // dg from dS' and S', then dS = D dS'
      float gpart = 0.0f;
      if (a.kda) {
        float al[32];
        ld32(ar, al);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          vec[x] = dS[x] * Sp[x];
          dS[x] *= al[x];
        }
        fold<KG, 0>(vec, lane);
#pragma unroll
        for (int x = 0; x < KG; ++x) red[2 * DKR + kf + x] = vec[x];
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          gpart = fmaf(dS[x], Sp[x], gpart);
          dS[x] *= ag;
        }
      }
      const float bpart = (kg == 0 && live) ? du * (vj - w) : 0.0f;
      const float bsum = warp_sum(bpart), gsum = warp_sum(live ? gpart : 0.0f);
      if (lane == 0) {
        red[NV * DKR] = bsum;
        red[NV * DKR + 1] = gsum;
      }
      const size_t row = (size_t)sq.b * a.T + sq.s + t0 + tt;
      if (kg == 0 && live) a.dv[(row * a.Hv + hv) * a.Dv + j] = bt * du;
      __syncthreads();
      // this CTA's columns: the sum over its warps, kept for the block's exchange
      const float* rb = s_red + (size_t)buf * nwarps * RS;
      float* xp = s_xp + ((size_t)(blk & 1) * DR_TB + tt) * XS;
      for (int e = threadIdx.x; e < NE; e += blockDim.x) {
        const int re = e < NV * DK
                           ? (e / DK) * DKR + ((e % DK) >> 5) * RGS + (e & 31)
                           : NV * DKR + (e - NV * DK);
        float s = 0.0f;
        for (int ww = 0; ww < nwarps; ++ww) s += rb[ww * RS + re];
        xp[e] = s;
      }
    }
    // The block's outputs: the CTAs' sums, added in rank order; the CTAs take outputs in turn.
    cluster_sync();
    const float* xb = s_xp + (size_t)(blk & 1) * DR_TB * XS;
    for (int f = CL * threadIdx.x + (int)crank; f < nt * NE; f += CL * blockDim.x) {
      const int tt = f / NE, e = f % NE;
      float s = 0.0f;
#pragma unroll
      for (int r = 0; r < CL; ++r)
        s += (uint32_t)r == crank ? xb[tt * XS + e] : ld_peer(xb + tt * XS + e, (uint32_t)r);
      const size_t row = (size_t)sq.b * a.T + sq.s + t0 + tt;
      if (e < NV * DK) {
        const int vsel = e / DK, i = e % DK;
        if (vsel == 0 || vsel == 1) {
          float* dst = vsel == 0 ? a.dq : a.dk;
          const size_t o = per_vhead ? (row * a.Hv + hv) * DK + i : (row * a.Hk + hk) * DK + i;
          dst[o] = s;
        } else {
          a.dg[(row * a.Hv + hv) * DK + i] = s;
        }
      } else if (e == NV * DK) {
        a.dbeta[row * a.Hv + hv] = s;
      } else if (!a.kda) {
        a.dg[row * a.Hv + hv] = s;
      }
    }
  }
  cluster_sync();  // the peer has read this CTA's last sums before either exits
  if (a.dh0 && live) {
#pragma unroll
    for (int x = 0; x < 32; ++x) {
      if (a.vfirst)
        a.dh0[(hbase * a.Dv + j) * DK + key0 + x] = dS[x];
      else
        a.dh0[(hbase * DK + key0 + x) * a.Dv + j] = dS[x];
    }
  }
}

// dq, dk of a key head: the sum over its Hv / Hk value heads (per-value-head values in ws).
__global__ void k_dr_group_sum(const float* ws, float* out, size_t rows, int Hk, int grp, int Dk) {
  const size_t total = rows * Hk * Dk;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e % Dk);
    const size_t rh = e / Dk;
    const int h = (int)(rh % Hk);
    const size_t row = rh / Hk;
    float s = 0.0f;
    for (int r = 0; r < grp; ++r) s += ws[((row * Hk + h) * grp + r) * Dk + i];
    out[e] = s;
  }
}

// FP8 (E4M3) quantize-dequantize of key-first states [n][Dk][Dv], one scale per [Dk, block_v]
// tile: amax over the tile, scale = amax / 448 (1 for an all-zero tile), each value replaced
// by its E4M3 code (nearest, ties to even, saturating at 448) of value / scale, times scale.
// The scale, the division and the product are IEEE float32 operations, so the codes are the
// ones a float32 reference picks.  CTA = (state, tile), 8 warps over the tile's rows, lanes
// over its columns (coalesced row segments); the second pass re-reads the tile from L2.
__device__ __forceinline__ float qdq_e4m3(float x, float scale) {
  const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3);
  const __half_raw h = __nv_cvt_fp8_to_halfraw(q, __NV_E4M3);
  return __fmul_rn(__half2float(__half(h)), scale);
}
__global__ void __launch_bounds__(256) k_state_qdq(const float* st, float* out, int Dk, int Dv,
                                                 int block_v, int ntiles) {
  __shared__ float s_amax[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t state = blockIdx.x / ntiles;
  const int v0 = (int)(blockIdx.x % ntiles) * block_v;
  const int bw = min(block_v, Dv - v0);
  const size_t base = state * (size_t)Dk * Dv + v0;
  float m = 0.0f;
  for (int i = warp; i < Dk; i += 8)
    for (int c = lane; c < bw; c += 32) m = fmaxf(m, fabsf(st[base + (size_t)i * Dv + c]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  if (lane == 0) s_amax[warp] = m;
  __syncthreads();
  float amax = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) amax = fmaxf(amax, s_amax[w]);
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  for (int i = warp; i < Dk; i += 8)
    for (int c = lane; c < bw; c += 32) {
      const size_t e = base + (size_t)i * Dv + c;
      out[e] = qdq_e4m3(st[e], scale);
    }
}

template <typename T>
size_t bwd_smem(int KG, int nwarps, int kda) {
  const int DK = 32 * KG, NC = nwarps * (32 / KG);
  const int RS = ((kda ? 3 : 2) * KG * RGS + 2 + 3) & ~3;
  const size_t raw = 2 * (size_t)DR_TB * DK * sizeof(T) + 2 * (size_t)DR_TB * NC * sizeof(T) +
                     (size_t)DR_TB * DK * 4 + DR_TB * 4;
  const int XS = ((kda ? 3 : 2) * DK + 2 + 3) & ~3;
  return (size_t)(4 * DR_TB * KG * KGS + 2 * DR_TB * NC + 2 * DR_TB + 2 * nwarps * RS +
                  2 * DR_TB * XS) * sizeof(float) + 2 * raw;
}

}  // namespace

// ------------------------------------------------------------------ host side

namespace {

bool dr_dims_ok(const delta_shape* s) {
  return s && s->B >= 1 && s->T >= 1 && s->Hk >= 1 && s->Hv >= 1 && s->Hv % s->Hk == 0 &&
         (s->io == RGLRU_F32 || s->io == RGLRU_BF16);
}
bool dr_supported(const delta_shape* s) {
  const int es = s->io == RGLRU_BF16 ? 2 : 4;
  return (s->Dk == 32 || s->Dk == 64 || s->Dk == 128) && s->Dv >= 1 && s->Dv <= 128 &&
         (s->Dv * es) % 16 == 0;
}
long dr_slots(const delta_shape* s, int N) { return (long)s->B * s->T / DR_TB + 2L * N + 1; }

DrArgs dr_args(const delta_shape* s, int N, float scale, const void* q, const void* k,
               const void* v, const float* g, const float* beta, const int32_t* cu,
               const float* h0) {
  DrArgs a{};
  a.B = s->B;
  a.T = s->T;
  a.Hk = s->Hk;
  a.Hv = s->Hv;
  a.Dk = s->Dk;
  a.Dv = s->Dv;
  a.kda = s->kda ? 1 : 0;
  a.vfirst = s->state_v_first ? 1 : 0;
  a.N = N;
  a.scale = scale;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.cu = cu;
  a.h0 = h0;
  return a;
}

template <typename T, int KG>
cudaError_t launch_fwd_t(DrArgs& a, cudaStream_t st) {
  const int NC = fwd_cols(KG);
  a.nslices = (a.Dv + NC - 1) / NC;
  const size_t smem = fwd_smem<T>(KG);
  cudaError_t e = cudaFuncSetAttribute(k_dr_fwd<T, KG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long grid = (long)a.N * a.Hv * a.nslices;
  if (grid < 1) return cudaSuccess;
  k_dr_fwd<T, KG><<<(unsigned)grid, 128, smem, st>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd_io(DrArgs& a, cudaStream_t st) {
  switch (a.Dk) {
    case 32: return launch_fwd_t<T, 1>(a, st);
    case 64: return launch_fwd_t<T, 2>(a, st);
    default: return launch_fwd_t<T, 4>(a, st);
  }
}

constexpr int DR_CL = 2;  // CTAs per (sequence, head) in the backward (4 measured slower)

template <typename T, int KG>
cudaError_t launch_bwd_t(DrArgs& a, float* ws, cudaStream_t st) {
  const int CPW = 32 / KG;
  const int part = (a.Dv + DR_CL - 1) / DR_CL;  // columns per CTA of the cluster
  const int nwarps = (part + CPW - 1) / CPW;
  const size_t smem = bwd_smem<T>(KG, nwarps, a.kda);
  cudaError_t e = cudaFuncSetAttribute(k_dr_bwd<T, KG, DR_CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  float* dq = a.dq;
  float* dk = a.dk;
  const size_t rows = (size_t)a.B * a.T;
  const size_t per = rows * a.Hv * a.Dk;
  if (a.Hv != a.Hk) {  // per value head first, then the group sums
    a.dq = ws;
    a.dk = ws + per;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long)DR_CL * a.N * a.Hv));
  cfg.blockDim = dim3(nwarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = DR_CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_dr_bwd<T, KG, DR_CL>, a);
  if (e != cudaSuccess) return e;
  note_launches(1);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.Hv == a.Hk) return e;
  const size_t total = rows * a.Hk * a.Dk;
  const unsigned blocks = (unsigned)std::min<size_t>((total + 255) / 256, 4096);
  k_dr_group_sum<<<blocks, 256, 0, st>>>(ws, dq, rows, a.Hk, a.Hv / a.Hk, a.Dk);
  k_dr_group_sum<<<blocks, 256, 0, st>>>(ws + per, dk, rows, a.Hk, a.Hv / a.Hk, a.Dk);
  note_launches(2);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_io(DrArgs& a, float* ws, cudaStream_t st) {
  switch (a.Dk) {
    case 32: return launch_bwd_t<T, 1>(a, ws, st);
    case 64: return launch_bwd_t<T, 2>(a, ws, st);
    default: return launch_bwd_t<T, 4>(a, ws, st);
  }
}

}  // namespace

}  // namespace rglru

using namespace rglru;

extern "C" size_t delta_rule_saved_bytes(const delta_shape* s, int32_t num_seqs) {
  if (!dr_dims_ok(s) || !dr_supported(s) || num_seqs < 1) return 0;
  return (size_t)dr_slots(s, num_seqs) * s->Hv * s->Dk * s->Dv * sizeof(float);
}

extern "C" rglru_status delta_rule_forward(const delta_shape* s, const void* q, const void* k,
                                           const void* v, const float* g, const float* beta,
                                           float scale, const int32_t* cu, int32_t num_seqs,
                                           const float* h0, void* o, float* hT, void* saved,
                                           rglru_stream stream) {
  if (!dr_dims_ok(s) || num_seqs < 1) return RGLRU_ERR_INVALID_ARG;
  if (cu ? (s->B != 1 || !req(cu)) : num_seqs != s->B) return RGLRU_ERR_INVALID_ARG;
  if (!req(q) || !req(k) || !req(v) || !req(g) || !req(beta) || !opt(h0) || !req(o) ||
      !opt(hT) || !opt(saved))
    return RGLRU_ERR_INVALID_ARG;
  if (!dr_supported(s)) return RGLRU_ERR_UNSUPPORTED;
  DrArgs a = dr_args(s, num_seqs, scale, q, k, v, g, beta, cu, h0);
  a.o = o;
  a.hT = hT;
  a.saved = static_cast<float*>(saved);
  const cudaError_t e = s->io == RGLRU_BF16 ? launch_fwd_io<bf16>(a, stream) : launch_fwd_io<float>(a, stream);
  return cuda_status(e);
}

extern "C" size_t delta_rule_workspace_bytes(const delta_shape* s) {
  if (!dr_dims_ok(s) || !dr_supported(s) || s->Hv == s->Hk) return 0;
  return 2 * (size_t)s->B * s->T * s->Hv * s->Dk * sizeof(float);
}

extern "C" rglru_status delta_rule_backward(const delta_shape* s, const void* q, const void* k,
                                            const void* v, const float* g, const float* beta,
                                            float scale, const int32_t* cu, int32_t num_seqs,
                                            const float* h0, const void* saved, const void* dout,
                                            const float* dhT, float* dq, float* dk, float* dv,
                                            float* dg, float* dbeta, float* dh0, void* workspace,
                                            rglru_stream stream) {
  (void)h0;  // the block states saved by the forward already include the initial states
  if (!dr_dims_ok(s) || num_seqs < 1) return RGLRU_ERR_INVALID_ARG;
  if (cu ? (s->B != 1 || !req(cu)) : num_seqs != s->B) return RGLRU_ERR_INVALID_ARG;
  if (!req(q) || !req(k) || !req(v) || !req(g) || !req(beta) || !opt(h0) || !req(saved) ||
      !req(dout) || !opt(dhT) || !req(dq) || !req(dk) || !req(dv) || !req(dg) || !req(dbeta) ||
      !opt(dh0))
    return RGLRU_ERR_INVALID_ARG;
  if (!dr_supported(s)) return RGLRU_ERR_UNSUPPORTED;
  if (s->Hv != s->Hk && !req(workspace)) return RGLRU_ERR_INVALID_ARG;
  DrArgs a = dr_args(s, num_seqs, scale, q, k, v, g, beta, cu, nullptr);
  a.saved = static_cast<float*>(const_cast<void*>(saved));
  a.dout = dout;
  a.dhT = dhT;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dg = dg;
  a.dbeta = dbeta;
  a.dh0 = dh0;
  float* ws = static_cast<float*>(workspace);
  const cudaError_t e = s->io == RGLRU_BF16 ? launch_bwd_io<bf16>(a, ws, stream)
                                            : launch_bwd_io<float>(a, ws, stream);
  return cuda_status(e);
}

extern "C" rglru_status delta_rule_state_fp8_qdq(const float* state, float* out,
                                                 int64_t n_states, int Dk, int Dv, int block_v,
                                                 rglru_stream stream) {
  if (n_states < 1 || Dk < 1 || Dv < 1 || block_v < 1 || !req(state) || !req(out))
    return RGLRU_ERR_INVALID_ARG;
  const long ntiles = (Dv + block_v - 1) / block_v;
  const long grid = n_states * ntiles;
  if (grid > 0x7fffffffL) return RGLRU_ERR_UNSUPPORTED;
  k_state_qdq<<<(unsigned)grid, 256, 0, stream>>>(state, out, Dk, Dv, block_v, (int)ntiles);
  note_launches(1);
  return cuda_status(cudaGetLastError());
}
